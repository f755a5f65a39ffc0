// la_api.cu -- the C ABI declared in include/la.h: argument validation, the
// packed-sequence table, and the mapping of la_fwd / la_bwd onto the two
// sweep shapes of la_internal.h.
//
// Backward by role swap (the gradient of the recurrence in the ejkernel
// `recurrent` custom VJP, `_recurrent_bwd`, written out per token):
//   dq_t = s * S_t do_t                  -> the forward-type sweep on
//                                           (q, k, v) := (do, v, k), state S^T
//   dv_u = sum_t ... (q_t . k_u) do_t + G^T k_u    -> backward-type sweep
//   dk_u = sum_t ... (do_t . v_u) q_t + G v_u      -> backward-type sweep on
//                                           (q, k, w) := (do, v, q), G^T
// so the kernels never see the words "query" or "gradient"; the host decides
// which tensors play which role.

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/la.h"
#include "la_internal.h"

namespace {
std::atomic<uint64_t> g_launches{0};
}

void la::note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

thread_local std::string g_msg;
thread_local int g_withhold = 0;   // la_debug_withhold_next_handoff

la_status fail(la_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_msg = buf;
    return st;
}

}  // namespace

void la::set_last_error(const char *msg) { g_msg = msg; }

namespace {

la_status cuda_fail(cudaError_t e, const char *where)
{
    return fail(LA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

struct Problem {
    int B, T, H, D, E, N;
    int Hkv, G;                     // key/value heads and query heads per key/value head
    const int64_t *k_st, *kv_v_st;  // strides of k, dk and of v, dv
    bool packed;
    std::vector<int32_t> cu_host;   // validated host copy of cu_seqlens (packed only)
};

// Sizes, dtype and the packed-sequence table; fills *P.
la_status check_dims(const la_dims *d, int32_t dtype, const int32_t *cu, const int32_t *cu_host,
                     cudaStream_t stream, Problem *P)
{
    if (!d)
        return fail(LA_ERR_INVALID_ARG, "dims is NULL");
    if (dtype != LA_DTYPE_BF16 && dtype != LA_DTYPE_F32)
        return fail(LA_ERR_INVALID_ARG, "dtype %d is neither LA_DTYPE_BF16 nor LA_DTYPE_F32",
                    dtype);
    if (d->batch < 0 || d->seq_len < 0)
        return fail(LA_ERR_INVALID_ARG, "negative batch (%d) or seq_len (%d)", d->batch,
                    d->seq_len);
    if (d->heads < 1 || d->heads > 65535)
        return fail(LA_ERR_INVALID_ARG, "heads = %d outside 1..65535", d->heads);
    if (d->dim_qk < 1 || d->dim_qk > 256 || d->dim_v < 1 || d->dim_v > 256)
        return fail(LA_ERR_UNSUPPORTED, "head dims D = %d, E = %d: supported range is 1..256",
                    d->dim_qk, d->dim_v);
    for (int i = 0; i < 3; ++i)
        if (d->qk_strides[i] < 0 || d->v_strides[i] < 0)
            return fail(LA_ERR_INVALID_ARG, "negative stride");
    if (d->reserved != 0)
        return fail(LA_ERR_INVALID_ARG, "la_dims.reserved = %d, must be 0", d->reserved);
    if (d->kv_heads < 0 || d->kv_heads > d->heads || (d->kv_heads && d->heads % d->kv_heads))
        return fail(LA_ERR_INVALID_ARG, "kv_heads = %d must be 0 or divide heads = %d",
                    d->kv_heads, d->heads);
    if (d->kv_heads)
        for (int i = 0; i < 3; ++i)
            if (d->k_strides[i] < 0 || d->kv_v_strides[i] < 0)
                return fail(LA_ERR_INVALID_ARG, "negative key/value stride");
    P->Hkv = d->kv_heads ? d->kv_heads : d->heads;
    P->G = d->heads / P->Hkv;
    P->k_st = d->kv_heads ? d->k_strides : d->qk_strides;
    P->kv_v_st = d->kv_heads ? d->kv_v_strides : d->v_strides;
    P->B = d->batch;
    P->T = d->seq_len;
    P->H = d->heads;
    P->D = d->dim_qk;
    P->E = d->dim_v;
    P->packed = cu != nullptr;
    if (!cu) {
        if (cu_host)
            return fail(LA_ERR_INVALID_ARG, "cu_seqlens_host given without cu_seqlens");
        if (d->batch > (1 << 30))
            return fail(LA_ERR_INVALID_ARG, "batch = %d", d->batch);
        P->N = d->batch;
        return LA_OK;
    }
    if (d->batch != 1)
        return fail(LA_ERR_INVALID_ARG,
                    "with cu_seqlens the sequences are packed in one batch row: "
                    "batch must be 1, got %d",
                    d->batch);
    if (d->num_seqs < 0 || d->num_seqs > (1 << 30))
        return fail(LA_ERR_INVALID_ARG, "num_seqs = %d", d->num_seqs);
    P->N = d->num_seqs;
    std::vector<int32_t> copy;
    if (!cu_host) {
        copy.resize((size_t)P->N + 1);
        cudaError_t e = cudaMemcpyAsync(copy.data(), cu, sizeof(int32_t) * copy.size(),
                                        cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "copying cu_seqlens to the host");
        cu_host = copy.data();
    }
    if (cu_host[0] != 0)
        return fail(LA_ERR_INVALID_ARG, "cu_seqlens[0] = %d, expected 0", cu_host[0]);
    for (int n = 0; n < P->N; ++n)
        if (cu_host[n + 1] < cu_host[n])
            return fail(LA_ERR_INVALID_ARG, "cu_seqlens decreases at %d (%d -> %d)", n,
                        cu_host[n], cu_host[n + 1]);
    if (cu_host[P->N] != d->seq_len)
        return fail(LA_ERR_INVALID_ARG, "cu_seqlens[%d] = %d but seq_len = %d", P->N,
                    cu_host[P->N], d->seq_len);
    P->cu_host.assign(cu_host, cu_host + P->N + 1);
    return LA_OK;
}

size_t schedule_bytes(int64_t num_seqs)
{
    return num_seqs <= 0 ? 0 : (size_t)((num_seqs * 4 + 255) / 256 * 256);
}

// Longest-first schedule of packed sequences: sequence indices sorted by
// length, longest first (ties keep index order), copied into the caller's
// workspace on `s`.  Returns the device array, or nullptr (index order) when
// nothing is packed, there is no workspace, or it is too small.
la_status make_schedule(const Problem &P, void *ws, size_t ws_bytes, cudaStream_t s,
                        const int32_t **order)
{
    *order = nullptr;
    if (!P.packed || P.N < 2 || !ws || ws_bytes < schedule_bytes(P.N))
        return LA_OK;
    if ((reinterpret_cast<uintptr_t>(ws) & 3) != 0)
        return fail(LA_ERR_INVALID_ARG, "workspace is not 4-byte aligned");
    std::vector<int32_t> idx((size_t)P.N);
    for (int n = 0; n < P.N; ++n)
        idx[(size_t)n] = n;
    const std::vector<int32_t> &cu = P.cu_host;
    std::stable_sort(idx.begin(), idx.end(), [&](int32_t x, int32_t y) {
        return cu[(size_t)x + 1] - cu[(size_t)x] > cu[(size_t)y + 1] - cu[(size_t)y];
    });
    // pageable source: the copy is staged before cudaMemcpyAsync returns
    cudaError_t e = cudaMemcpyAsync(ws, idx.data(), idx.size() * sizeof(int32_t),
                                    cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "copying the packed schedule");
    *order = static_cast<const int32_t *>(ws);
    return LA_OK;
}

// ---- sequence split -------------------------------------------------------
// Few (sequence, head) pairs leave most SMs idle while each CTA walks a long
// sequence.  Then every sequence is cut into segments of seg_len tokens (a
// multiple of the 128-token chunk) that run as packed sequences, in two
// passes around a state scan (la_split.cu): pass 1 from zero states gives
// each segment's own contribution, the scan turns those into each segment's
// initial state (and the sequence's final state), pass 2 produces the
// outputs.  Dense batches are viewed as one row of B*T tokens, which needs
// every token tensor's batch stride to be T times its token stride.

std::atomic<int> g_split_mode{1};            // 0 off, 1 when it pays
std::atomic<int> g_split_min_seg{0};         // shortest segment planned; 0 automatic

int sm_count()
{
    static std::mutex mu;
    static int cache[256] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256)
        return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            cache[dev] = n;
    }
    return cache[dev];
}

struct SplitPlan {
    int NS = 0;                       // segments; 0 = no split
    int64_t seg_len = 0;
    std::vector<int32_t> seg_cu;      // [NS + 1] token offsets of the one-row view
    std::vector<int32_t> seq_first;   // [N + 1] first segment of each sequence
    size_t bytes = 0;                 // workspace beyond the schedule
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

bool flat_rows(const Problem &P, const int64_t *st)
{
    return P.packed || P.B == 1 || st[0] == (int64_t)P.T * st[1];
}

// sms = 0: ask the current device.
SplitPlan plan_split(const Problem &P, const la_dims *d, int sms = 0)
{
    SplitPlan S;
    if (g_split_mode.load() == 0 || !flat_rows(P, d->qk_strides) || !flat_rows(P, d->v_strides) ||
        !flat_rows(P, P.k_st) || !flat_rows(P, P.kv_v_st))
        return S;
    if (sms <= 0)
        sms = sm_count();
    const int64_t items = (int64_t)P.N * P.H;
    const int64_t total = P.packed ? (int64_t)P.T : (int64_t)P.B * P.T;
    if (sms <= 0 || items == 0 || items * 2 > sms || total >= INT32_MAX)
        return S;
    int64_t max_len = 0;
    for (int n = 0; n < P.N; ++n) {
        const int64_t len = P.packed ? (int64_t)P.cu_host[(size_t)n + 1] - P.cu_host[(size_t)n]
                                     : (int64_t)P.T;
        max_len = std::max(max_len, len);
    }
    // Automatic segments, from measured calls (b2.h8.n2048 d=64, b2.h16.n4096
    // and b1.h16.n8192 d=128, b2.h12.n2048 d=192, fwd + bwd): at d <= 64
    // segments of 256 tokens already pay (154.7 -> 117.9 us); at d = 128 a
    // split pays from 4 segments of at least 1024 tokens (324 -> 288 us,
    // 623 -> 299 us) but not with 2 (348 us) or with 256-token segments; at
    // d > 128 the state pass has no state-only form and the split costs
    // (278 -> 399 us at 1024-token segments).
    int64_t min_seg = g_split_min_seg.load(), min_r = 2;
    if (min_seg == 0) {
        if (P.D > 128)
            return S;
        min_seg = P.D <= 64 ? 256 : 1024;
        min_r = P.D <= 64 ? 2 : 4;
    }
    const int64_t R = std::min<int64_t>(sms / items, max_len / min_seg);
    if (R < min_r)
        return S;
    const int64_t seg_len = ((max_len + R - 1) / R + 127) / 128 * 128;
    S.seq_first.push_back(0);
    S.seg_cu.push_back(0);
    for (int n = 0; n < P.N; ++n) {
        const int64_t start = P.packed ? (int64_t)P.cu_host[(size_t)n] : (int64_t)n * P.T;
        const int64_t len = P.packed ? (int64_t)P.cu_host[(size_t)n + 1] - start : (int64_t)P.T;
        for (int64_t t = 0; t < len; t += seg_len) {
            if (S.seg_cu.back() != start + t)   // a gap (never for these views)
                return SplitPlan{};
            S.seg_cu.push_back((int32_t)std::min(start + len, start + t + seg_len));
        }
        S.seq_first.push_back((int32_t)S.seg_cu.size() - 1);
    }
    S.NS = (int)S.seg_cu.size() - 1;
    S.seg_len = seg_len;
    S.bytes = round256(S.seg_cu.size() * 4) + round256(S.seq_first.size() * 4) +
              (size_t)S.NS * P.H * P.D * P.E * sizeof(float);
    return S;
}

// Device copies of the plan and the state buffer, carved from the workspace
// after the schedule.
struct SplitBufs {
    const int32_t *seg_cu, *seq_first;
    float *W;
};

la_status split_setup(const Problem &P, const SplitPlan &S, void *ws, size_t offset,
                      cudaStream_t s, SplitBufs *b)
{
    (void)P;
    uint8_t *p = static_cast<uint8_t *>(ws) + offset;
    int32_t *cu = reinterpret_cast<int32_t *>(p);
    int32_t *first = reinterpret_cast<int32_t *>(p + round256(S.seg_cu.size() * 4));
    b->W = reinterpret_cast<float *>(p + round256(S.seg_cu.size() * 4) +
                                     round256(S.seq_first.size() * 4));
    // pageable sources: each copy is staged before cudaMemcpyAsync returns
    cudaError_t e = cudaMemcpyAsync(cu, S.seg_cu.data(), S.seg_cu.size() * 4,
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(first, S.seq_first.data(), S.seq_first.size() * 4,
                            cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "copying the sequence split plan");
    b->seg_cu = cu;
    b->seq_first = first;
    return LA_OK;
}

// Whether this call runs split: a plan exists and the workspace holds it
// from `offset` on.
bool use_split(const Problem &P, const la_dims *d, void *ws, size_t ws_bytes, size_t offset,
               SplitPlan *S)
{
    *S = plan_split(P, d);
    if (S->NS == 0 || !ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 ||
        ws_bytes < offset + S->bytes) {
        *S = SplitPlan{};
        return false;
    }
    return true;
}

// ---- grouped key/value heads ---------------------------------------------------
// The backward sweeps give one dk / dv contribution per query head; they go
// to two dense [B, T, H, X] buffers of the token dtype in the workspace
// (after the schedule) and gqa_reduce sums each group into dk / dv.
struct GqaBufs {
    la::TokOut ck, cv;
};

size_t gqa_bytes(const Problem &P, int32_t dtype)
{
    if (P.G <= 1)
        return 0;
    const size_t elt = dtype == LA_DTYPE_BF16 ? 2 : 4;
    const size_t tokens = (size_t)(P.packed ? 1 : P.B) * P.T;
    return round256(tokens * P.H * P.D * elt) + round256(tokens * P.H * P.E * elt);
}

la_status gqa_setup(const Problem &P, int32_t dtype, void *ws, size_t ws_bytes, GqaBufs *g)
{
    const size_t need = schedule_bytes(P.N) + gqa_bytes(P, dtype);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 || ws_bytes < need)
        return fail(LA_ERR_INVALID_ARG,
                    "grouped key/value heads need a 256-byte aligned workspace of at least %zu "
                    "bytes for the backward (got %zu)",
                    need, ws ? ws_bytes : (size_t)0);
    const size_t elt = dtype == LA_DTYPE_BF16 ? 2 : 4;
    const size_t tokens = (size_t)(P.packed ? 1 : P.B) * P.T;
    uint8_t *p = static_cast<uint8_t *>(ws) + schedule_bytes(P.N);
    const int64_t T = P.T, H = P.H;
    g->ck = la::TokOut{p, T * H * P.D, H * P.D, P.D};
    g->cv = la::TokOut{p + round256(tokens * P.H * P.D * elt), T * H * P.E, H * P.E, P.E};
    return LA_OK;
}

// Sweep arguments of the segment view: one row of all tokens, the segments
// as packed sequences.
void to_segments(la::SweepArgs *a, const Problem &P, const SplitPlan &S, const SplitBufs &b)
{
    a->B = 1;
    a->T = P.packed ? P.T : P.B * P.T;
    a->N = S.NS;
    a->cu = b.seg_cu;
    a->order = nullptr;
    a->max_len = S.seg_len;
}

la::SplitScanArgs scan_args(const Problem &P, const SplitBufs &b, const float *g, int D, int E,
                            la::StateIn start, la::StateOut fin, bool descending)
{
    la::SplitScanArgs sc{};
    sc.N = P.N;
    sc.H = P.H;
    sc.D = D;
    sc.E = E;
    sc.seg_cu = b.seg_cu;
    sc.seq_first = b.seq_first;
    sc.g = g;
    sc.W = b.W;
    sc.start = start;
    sc.fin = fin;
    sc.descending = descending ? 1 : 0;
    return sc;
}

la_status scan(const la::SplitScanArgs &sc, cudaStream_t s)
{
    cudaError_t e = la::split_scan(sc, s);
    return e == cudaSuccess ? LA_OK : cuda_fail(e, "sequence split state scan");
}

bool has_tokens(const Problem &P) { return (int64_t)P.B * P.T > 0; }
bool has_states(const Problem &P) { return (int64_t)P.N * P.H > 0; }

la_status need(const void *p, const char *name)
{
    return p ? LA_OK : fail(LA_ERR_INVALID_ARG, "%s is NULL", name);
}

la::Tok tok(const void *p, const int64_t *st, int hdiv = 1)
{
    return la::Tok{p, st[0], st[1], st[2], hdiv};
}
la::TokOut tok_out(void *p, const int64_t *st) { return la::TokOut{p, st[0], st[1], st[2]}; }

la::SweepArgs base_args(const Problem &P, int32_t dtype, const int32_t *cu, const float *g,
                        float scale, int32_t reverse, const int32_t *order = nullptr)
{
    la::SweepArgs a{};
    a.B = P.B;
    a.T = P.T;
    a.H = P.H;
    a.N = P.N;
    a.cu = cu;
    a.order = order;
    a.g = g;
    a.scale = scale;
    a.reverse = reverse ? 1 : 0;
    a.bf16 = dtype == LA_DTYPE_BF16;
    a.max_len = P.T;
    if (P.packed) {
        a.max_len = 0;
        for (size_t n = 0; n < (size_t)P.N; ++n)
            a.max_len = std::max<int64_t>(a.max_len, P.cu_host[n + 1] - P.cu_host[n]);
    }
    return a;
}

la_status run_forward_type(const la::SweepArgs &a, cudaStream_t s)
{
    cudaError_t e = cudaErrorNotSupported;
    if (a.max_len <= la::SHORT_MAX_T) {
        la::SweepArgs b = a;
        b.withhold_handoff = g_withhold;
        bool streamed = false;
        e = la::short_forward_sweep(b, s, &streamed);
        if (streamed)   // the only token-by-token kernel with hand-offs to withhold
            g_withhold = 0;
    }
    if (e == cudaErrorNotSupported && la::tc_sweep_supported(a)) {
        la::SweepArgs b = a;
        b.withhold_handoff = g_withhold;
        g_withhold = 0;
        e = la::tc_forward_sweep(b, s);
    }
    // cudaErrorNotSupported: the tensor maps could not be encoded for this layout
    if (e == cudaErrorNotSupported)
        e = la::simt_forward_sweep(a, s);
    return e == cudaSuccess ? LA_OK : cuda_fail(e, "forward-type sweep launch");
}

la_status run_backward_type(const la::SweepArgs &a, cudaStream_t s)
{
    cudaError_t e = cudaErrorNotSupported;
    if (a.max_len <= la::SHORT_MAX_T)
        e = la::short_backward_sweep(a, s);
    if (e == cudaErrorNotSupported && la::tc_sweep_supported(a)) {
        la::SweepArgs b = a;
        b.withhold_handoff = g_withhold;
        g_withhold = 0;
        e = la::tc_backward_sweep(b, s);
    }
    if (e == cudaErrorNotSupported)
        e = la::simt_backward_sweep(a, s);
    return e == cudaSuccess ? LA_OK : cuda_fail(e, "backward-type sweep launch");
}

// The sweep's final states only (the sequence split's first pass): the
// tensor-core state-only mode where it applies, else the full sweep (whose
// outputs the second pass overwrites).
la_status run_states(const la::SweepArgs &a, bool bwd, cudaStream_t s)
{
    cudaError_t e = cudaErrorNotSupported;
    if (a.max_len > la::SHORT_MAX_T && la::tc_sweep_supported(a))
        e = la::tc_state_sweep(a, bwd, s);
    if (e == cudaErrorNotSupported)
        return bwd ? run_backward_type(a, s) : run_forward_type(a, s);
    return e == cudaSuccess ? LA_OK : cuda_fail(e, "state sweep launch");
}

la_status bwd_dq(const Problem &P, const la_dims *d, int32_t dtype, const void *k, const void *v,
                 const void *d_o, const float *g_gamma, float scale, const float *init,
                 int32_t reverse, const int32_t *cu, const int32_t *order, void *dq, cudaStream_t s,
                 const SplitPlan *S = nullptr, const SplitBufs *b = nullptr)
{
    // dq = forward-type sweep with (q, k, v) := (do, v, k); the state is S^T (E x D).
    la::SweepArgs a = base_args(P, dtype, cu, g_gamma, scale, reverse, order);
    a.D = P.E;
    a.E = P.D;
    a.q = tok(d_o, d->v_strides);
    a.k = tok(v, P.kv_v_st, P.G);
    a.v = tok(k, P.k_st, P.G);
    a.out = tok_out(dq, d->qk_strides);
    a.s_in = la::StateIn{init, 1, P.E};
    a.s_out = la::StateOut{nullptr, 0, 0};
    if (!S)
        return run_forward_type(a, s);
    // split: segment states from zero, scan from the initial state, outputs
    to_segments(&a, P, *S, *b);
    a.s_in = la::StateIn{nullptr, 0, 0};
    a.s_out = la::StateOut{b->W, P.D, 1};
    la_status st = run_states(a, false, s);
    if (st == LA_OK)
        st = scan(scan_args(P, *b, g_gamma, P.E, P.D, la::StateIn{init, 1, P.E},
                            la::StateOut{nullptr, 0, 0}, reverse != 0),
                  s);
    if (st != LA_OK)
        return st;
    a.s_in = la::StateIn{b->W, P.D, 1};
    a.s_out = la::StateOut{nullptr, 0, 0};
    return run_forward_type(a, s);
}

// dk and dv of grouped key/value heads: each group's per-query-head
// contributions (in the workspace) summed into dk and dv.
la_status gqa_sum(const Problem &P, const GqaBufs *gqa, void *dk, void *dv, int bf16,
                  cudaStream_t s)
{
    const int rows = P.packed ? 1 : P.B;
    cudaError_t e = la::gqa_reduce(gqa->ck.p, tok_out(dk, P.k_st), rows, P.T, P.Hkv, P.G, P.D,
                                   bf16, s);
    if (e == cudaSuccess)
        e = la::gqa_reduce(gqa->cv.p, tok_out(dv, P.kv_v_st), rows, P.T, P.Hkv, P.G, P.E, bf16,
                           s);
    return e == cudaSuccess ? LA_OK : cuda_fail(e, "grouped key/value gradient sum");
}

// The dv half of the backward: the fused dk/dv sweep (the tensor-core kernel
// of la_tc_dkdv.cu) when `fused` and its tensor maps can be built (*ran set),
// else the dv sweep alone (the dk sweep follows).
la_status run_dv(const la::SweepArgs &a, bool fused, const la::Tok &v, const la::TokOut &dk,
                 cudaStream_t s, bool *ran)
{
    *ran = false;
    if (fused) {
        la::SweepArgs b = a;
        b.withhold_handoff = g_withhold;
        cudaError_t e = la::tc_dkdv_sweep(b, v, dk, s);
        if (e != cudaErrorNotSupported) {
            g_withhold = 0;
            *ran = e == cudaSuccess;
            return e == cudaSuccess ? LA_OK : cuda_fail(e, "dk/dv sweep launch");
        }
    }
    return run_backward_type(a, s);
}

la_status bwd_dkdv(const Problem &P, const la_dims *d, int32_t dtype, const void *q,
                   const void *k, const void *v, const void *d_o, const float *g_gamma,
                   float scale, const float *dfinal, int32_t reverse, const int32_t *cu,
                   const int32_t *order, void *dk, void *dv, float *dinit, cudaStream_t s,
                   const SplitPlan *S = nullptr, const SplitBufs *b = nullptr,
                   const GqaBufs *gqa = nullptr)
{
    la::SweepArgs a = base_args(P, dtype, cu, g_gamma, scale, reverse, order);
    // dv: (q, k, w) as given, G = dL/dS (D x E)
    a.D = P.D;
    a.E = P.E;
    a.q = tok(q, d->qk_strides);
    a.k = tok(k, P.k_st, P.G);
    a.v = tok(d_o, d->v_strides);
    a.out = gqa ? gqa->cv : tok_out(dv, P.kv_v_st);
    a.s_in = la::StateIn{dfinal, P.E, 1};
    a.s_out = la::StateOut{dinit, P.E, 1};
    la::StateIn g_dk{dfinal, 1, P.E};   // G^T for the dk sweep
    const la::Tok vt = tok(v, P.kv_v_st, P.G);
    const la::TokOut dkt = gqa ? gqa->ck : tok_out(dk, P.k_st);
    // dk and dv in one sweep where the fused tensor-core kernel applies
    const bool fused = a.max_len > la::SHORT_MAX_T && la::tc_dkdv_supported(a, vt, dkt);
    la_status st;
    bool fused_ran = false;
    if (!S) {
        st = run_dv(a, fused, vt, dkt, s, &fused_ran);
    } else {
        // split: segment G from zero, scan from d_final (against processing
        // order), d_initial from the scan, then dv from each segment's G
        to_segments(&a, P, *S, *b);
        a.s_in = la::StateIn{nullptr, 0, 0};
        a.s_out = la::StateOut{b->W, P.E, 1};
        st = run_states(a, true, s);
        if (st == LA_OK)
            st = scan(scan_args(P, *b, g_gamma, P.D, P.E, la::StateIn{dfinal, P.E, 1},
                                la::StateOut{dinit, P.E, 1}, reverse == 0),
                      s);
        if (st == LA_OK) {
            a.s_in = la::StateIn{b->W, P.E, 1};
            a.s_out = la::StateOut{nullptr, 0, 0};
            st = run_dv(a, fused, vt, dkt, s, &fused_ran);
        }
        g_dk = la::StateIn{b->W, 1, P.E};
    }
    if (st != LA_OK)
        return st;
    if (fused_ran)
        return gqa ? gqa_sum(P, gqa, dk, dv, a.bf16, s) : LA_OK;
    // dk: (q, k, w) := (do, v, q), G^T (E x D)
    a.D = P.E;
    a.E = P.D;
    a.q = tok(d_o, d->v_strides);
    a.k = tok(v, P.kv_v_st, P.G);
    a.v = tok(q, d->qk_strides);
    a.out = gqa ? gqa->ck : tok_out(dk, P.k_st);
    a.s_in = g_dk;
    a.s_out = la::StateOut{nullptr, 0, 0};
    if ((st = run_backward_type(a, s)) != LA_OK || !gqa)
        return st;
    return gqa_sum(P, gqa, dk, dv, a.bf16, s);
}

}  // namespace

extern "C" {

la_status la_fwd(const la_dims *dims, int32_t dtype, const void *q, const void *k, const void *v,
                 const float *g_gamma, float scale, const float *initial_state, int32_t reverse,
                 const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, void *o,
                 float *final_state, void *workspace, size_t workspace_bytes, void *stream)
{
    g_msg.clear();
    cudaStream_t s = (cudaStream_t)stream;
    Problem P;
    la_status st = check_dims(dims, dtype, cu_seqlens, cu_seqlens_host, s, &P);
    if (st != LA_OK)
        return st;
    if (has_tokens(P)) {
        if ((st = need(q, "q")) || (st = need(k, "k")) || (st = need(v, "v")) ||
            (st = need(o, "o")))
            return st;
    }
    if (!has_states(P))
        return LA_OK;
    if ((st = need(g_gamma, "g_gamma")))
        return st;
    const int32_t *order = nullptr;
    if ((st = make_schedule(P, workspace, workspace_bytes, s, &order)))
        return st;
    la::SweepArgs a = base_args(P, dtype, cu_seqlens, g_gamma, scale, reverse, order);
    a.D = P.D;
    a.E = P.E;
    a.q = tok(q, dims->qk_strides);
    a.k = tok(k, P.k_st, P.G);
    a.v = tok(v, P.kv_v_st, P.G);
    a.out = tok_out(o, dims->v_strides);
    a.s_in = la::StateIn{initial_state, P.E, 1};
    a.s_out = la::StateOut{final_state, P.E, 1};
    SplitPlan S;
    const size_t off = schedule_bytes(P.N);
    if (!use_split(P, dims, workspace, workspace_bytes, off, &S))
        return run_forward_type(a, s);
    // split: segment states from zero, scan (which also writes the final
    // state), then every segment from its initial state
    SplitBufs b;
    if ((st = split_setup(P, S, workspace, off, s, &b)))
        return st;
    to_segments(&a, P, S, b);
    a.s_in = la::StateIn{nullptr, 0, 0};
    a.s_out = la::StateOut{b.W, P.E, 1};
    if ((st = run_states(a, false, s)))
        return st;
    if ((st = scan(scan_args(P, b, g_gamma, P.D, P.E, la::StateIn{initial_state, P.E, 1},
                             la::StateOut{final_state, P.E, 1}, reverse != 0),
                   s)))
        return st;
    a.s_in = la::StateIn{b.W, P.E, 1};
    a.s_out = la::StateOut{nullptr, 0, 0};
    return run_forward_type(a, s);
}

la_status la_bwd_dq(const la_dims *dims, int32_t dtype, const void *q, const void *k,
                    const void *v, const void *d_o, const float *g_gamma, float scale,
                    const float *initial_state, int32_t reverse, const int32_t *cu_seqlens,
                    const int32_t *cu_seqlens_host, void *dq, void *workspace,
                    size_t workspace_bytes, void *stream)
{
    (void)q;
    g_msg.clear();
    cudaStream_t s = (cudaStream_t)stream;
    Problem P;
    la_status st = check_dims(dims, dtype, cu_seqlens, cu_seqlens_host, s, &P);
    if (st != LA_OK)
        return st;
    if (has_tokens(P)) {
        if ((st = need(k, "k")) || (st = need(v, "v")) || (st = need(d_o, "d_o")) ||
            (st = need(dq, "dq")))
            return st;
    }
    if (!has_states(P))
        return LA_OK;
    if ((st = need(g_gamma, "g_gamma")))
        return st;
    const int32_t *order = nullptr;
    if ((st = make_schedule(P, workspace, workspace_bytes, s, &order)))
        return st;
    SplitPlan S;
    SplitBufs b;
    const size_t off = schedule_bytes(P.N);
    const bool split = use_split(P, dims, workspace, workspace_bytes, off, &S);
    if (split && (st = split_setup(P, S, workspace, off, s, &b)))
        return st;
    return bwd_dq(P, dims, dtype, k, v, d_o, g_gamma, scale, initial_state, reverse, cu_seqlens,
                  order, dq, s, split ? &S : nullptr, split ? &b : nullptr);
}

la_status la_bwd_dkdv(const la_dims *dims, int32_t dtype, const void *q, const void *k,
                      const void *v, const void *d_o, const float *g_gamma, float scale,
                      const float *d_final_state, int32_t reverse, const int32_t *cu_seqlens,
                      const int32_t *cu_seqlens_host, void *dk, void *dv,
                      float *d_initial_state, void *workspace, size_t workspace_bytes,
                      void *stream)
{
    g_msg.clear();
    cudaStream_t s = (cudaStream_t)stream;
    Problem P;
    la_status st = check_dims(dims, dtype, cu_seqlens, cu_seqlens_host, s, &P);
    if (st != LA_OK)
        return st;
    if (has_tokens(P)) {
        if ((st = need(q, "q")) || (st = need(k, "k")) || (st = need(v, "v")) ||
            (st = need(d_o, "d_o")) || (st = need(dk, "dk")) || (st = need(dv, "dv")))
            return st;
    }
    if (!has_states(P))
        return LA_OK;
    if ((st = need(g_gamma, "g_gamma")))
        return st;
    const int32_t *order = nullptr;
    if ((st = make_schedule(P, workspace, workspace_bytes, s, &order)))
        return st;
    GqaBufs gb;
    if (P.G > 1 && (st = gqa_setup(P, dtype, workspace, workspace_bytes, &gb)))
        return st;
    SplitPlan S;
    SplitBufs b;
    const size_t off = schedule_bytes(P.N) + gqa_bytes(P, dtype);
    const bool split = use_split(P, dims, workspace, workspace_bytes, off, &S);
    if (split && (st = split_setup(P, S, workspace, off, s, &b)))
        return st;
    return bwd_dkdv(P, dims, dtype, q, k, v, d_o, g_gamma, scale, d_final_state, reverse,
                    cu_seqlens, order, dk, dv, d_initial_state, s, split ? &S : nullptr,
                    split ? &b : nullptr, P.G > 1 ? &gb : nullptr);
}

la_status la_bwd(const la_dims *dims, int32_t dtype, const void *q, const void *k, const void *v,
                 const void *d_o, const float *g_gamma, float scale, const float *initial_state,
                 const float *d_final_state, int32_t reverse, const int32_t *cu_seqlens,
                 const int32_t *cu_seqlens_host, void *dq, void *dk, void *dv,
                 float *d_initial_state, void *workspace, size_t workspace_bytes, void *stream)
{
    g_msg.clear();
    cudaStream_t s = (cudaStream_t)stream;
    Problem P;
    la_status st = check_dims(dims, dtype, cu_seqlens, cu_seqlens_host, s, &P);
    if (st != LA_OK)
        return st;
    if (has_tokens(P)) {
        if ((st = need(q, "q")) || (st = need(k, "k")) || (st = need(v, "v")) ||
            (st = need(d_o, "d_o")) || (st = need(dq, "dq")) || (st = need(dk, "dk")) ||
            (st = need(dv, "dv")))
            return st;
    }
    if (!has_states(P))
        return LA_OK;
    if ((st = need(g_gamma, "g_gamma")))
        return st;
    const int32_t *order = nullptr;
    if ((st = make_schedule(P, workspace, workspace_bytes, s, &order)))
        return st;
    GqaBufs gb;
    if (P.G > 1 && (st = gqa_setup(P, dtype, workspace, workspace_bytes, &gb)))
        return st;
    SplitPlan S;
    SplitBufs b;
    const size_t off = schedule_bytes(P.N) + gqa_bytes(P, dtype);
    const bool split = use_split(P, dims, workspace, workspace_bytes, off, &S);
    if (split && (st = split_setup(P, S, workspace, off, s, &b)))
        return st;
    st = bwd_dq(P, dims, dtype, k, v, d_o, g_gamma, scale, initial_state, reverse, cu_seqlens,
                order, dq, s, split ? &S : nullptr, split ? &b : nullptr);
    if (st != LA_OK)
        return st;
    return bwd_dkdv(P, dims, dtype, q, k, v, d_o, g_gamma, scale, d_final_state, reverse,
                    cu_seqlens, order, dk, dv, d_initial_state, s, split ? &S : nullptr,
                    split ? &b : nullptr, P.G > 1 ? &gb : nullptr);
}

la_status la_get_device_error(void *stream)
{
    g_msg.clear();
    int err = 0;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e == cudaSuccess)
        e = la::tc_read_and_clear_error((cudaStream_t)stream, &err);
    int err2 = 0, err3 = 0, err4 = 0;
    if (e == cudaSuccess)
        e = la::token_read_and_clear_error((cudaStream_t)stream, &err2);
    if (e == cudaSuccess)
        e = la::tc_dkdv_read_and_clear_error((cudaStream_t)stream, &err3);
    if (e == cudaSuccess)
        e = la::decode_read_and_clear_error((cudaStream_t)stream, &err4);
    if (e != cudaSuccess)
        return cuda_fail(e, "la_get_device_error");
    if (!err)
        err = err2 ? err2 : err3 ? err3 : err4;
    else if ((err & 0xff) != LA_ERR_BOUNDS && (err3 & 0xff) == LA_ERR_BOUNDS)
        err = err3;
    if ((err & 0xff) == LA_ERR_BOUNDS)
        return fail(LA_ERR_BOUNDS, "an index check failed at site %d", err >> 8);
    if (err)
        return fail(LA_ERR_TIMEOUT, "an on-device wait ran out (code %d)", err);
    return LA_OK;
}

const char *la_strerror(int32_t status)
{
    switch (status) {
    case LA_OK: return "ok";
    case LA_ERR_INVALID_ARG: return "invalid argument";
    case LA_ERR_UNSUPPORTED: return "unsupported configuration";
    case LA_ERR_CUDA: return "CUDA error";
    case LA_ERR_TIMEOUT: return "on-device wait timed out";
    case LA_ERR_BOUNDS: return "on-device index check failed";
    default: return "unknown status";
    }
}

const char *la_last_error(void) { return g_msg.c_str(); }

int32_t la_kernel_family(const la_dims *dims, int32_t dtype)
{
    Problem P;
    std::string keep = g_msg;
    // The packed table does not change the kernel family.
    la_status st = check_dims(dims, dtype, nullptr, nullptr, nullptr, &P);
    g_msg = keep;
    if (st != LA_OK)
        return -1;
    la::SweepArgs a = base_args(P, dtype, nullptr, nullptr, 1.f, 0);
    a.D = P.D;
    a.E = P.E;
    a.q = tok(nullptr, dims->qk_strides);
    a.k = tok(nullptr, P.k_st, P.G);
    a.v = tok(nullptr, P.kv_v_st, P.G);
    a.out = tok_out(nullptr, dims->v_strides);
    if (a.max_len <= la::SHORT_MAX_T && P.D <= 256)
        return 2;
    return la::tc_sweep_supported(a) ? 1 : 0;
}

size_t la_workspace_size(int32_t num_seqs) { return schedule_bytes(num_seqs); }

size_t la_workspace_size_for(const la_dims *dims, int32_t dtype, const int32_t *cu_seqlens_host)
{
    Problem P;
    std::string keep = g_msg;
    // the host table stands in for the device one: check_dims reads only the host copy
    la_status st = check_dims(dims, dtype, cu_seqlens_host, cu_seqlens_host, nullptr, &P);
    g_msg = keep;
    if (st != LA_OK)
        return 0;
    const SplitPlan S = plan_split(P, dims);
    const size_t gqa = gqa_bytes(P, dtype);
    if (S.NS > 0 || gqa > 0)
        return schedule_bytes(P.N) + gqa + S.bytes;
    return P.packed ? schedule_bytes(P.N) : 0;
}

la_status la_set_sequence_split(int32_t mode, int32_t min_segment_tokens)
{
    if (mode < 0 || mode > 1 || (min_segment_tokens != 0 && min_segment_tokens < 128))
        return fail(LA_ERR_INVALID_ARG, "la_set_sequence_split: mode %d, min_segment_tokens %d",
                    mode, min_segment_tokens);
    g_split_mode.store(mode);
    g_split_min_seg.store(min_segment_tokens);
    return LA_OK;
}

int32_t la_debug_split_segments(const la_dims *dims, int32_t dtype,
                                const int32_t *cu_seqlens_host, int32_t sms)
{
    Problem P;
    std::string keep = g_msg;
    la_status st = check_dims(dims, dtype, cu_seqlens_host, cu_seqlens_host, nullptr, &P);
    g_msg = keep;
    if (st != LA_OK || sms < 1)
        return -1;
    return plan_split(P, dims, sms).NS;
}

la_status la_debug_withhold_next_handoff(int32_t on)
{
    g_withhold = on ? 1 : 0;
    return LA_OK;
}

uint64_t la_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int32_t la_version(void) { return (0 << 16) | 4; }

int32_t la_build_flags(void)
{
#ifdef LA_CHECK_BOUNDS
    return LA_BUILD_BOUNDS_CHECKED;
#else
    return 0;
#endif
}

}  // extern "C"

// ---- gated form (per-key gate, GLA) --------------------------------------------
namespace {

la_status gla_check(const Problem &P, const la_dims *d, const float *g, const int64_t *gs,
                    const float *g_gamma)
{
    (void)d;
    if (!has_states(P))
        return LA_OK;
    la_status st;
    if ((st = need(g_gamma, "g_gamma")))
        return st;
    if (has_tokens(P)) {
        if ((st = need(g, "g")) || (st = need(gs, "g_strides")))
            return st;
        for (int i = 0; i < 3; ++i)
            if (gs[i] < 0)
                return fail(LA_ERR_INVALID_ARG, "negative gate stride");
    }
    return LA_OK;
}

la::Gate gate_of(const float *g, const int64_t *gs, bool cols)
{
    la::Gate G;
    G.p = g;
    if (gs) {
        G.sb = gs[0];
        G.st = gs[1];
        G.sh = gs[2];
    }
    G.cols = cols ? 1 : 0;
    return G;
}

la_status short_run(const la::SweepArgs &a, bool bwd, cudaStream_t s)
{
    cudaError_t e = bwd ? la::short_backward_sweep(a, s) : la::short_forward_sweep(a, s);
    return e == cudaSuccess ? LA_OK : cuda_fail(e, "gated sweep launch");
}

int64_t gla_max_len(const Problem &P)
{
    int64_t m = P.packed ? 0 : P.T;
    for (size_t n = 0; P.packed && n < (size_t)P.N; ++n)
        m = std::max<int64_t>(m, P.cu_host[n + 1] - P.cu_host[n]);
    return m;
}

// Workspace of the chunked gated forward: q~, k~ (bf16, dense [rows][T][H][D]),
// exp(r) and exp(B - r) per chunk ([N][H][ncmax][D] fp32), one flag per
// (sequence, head).  0 when the chunked form does not apply to these sizes.
struct GlaFwdWs {
    size_t xq, yk, er, u, flags, total;
    int64_t ncmax;
};
// N sequences of at most maxlen tokens (the call's own, or the segments of
// the sequence split, whose tokens are the same).
GlaFwdWs gla_layout(const Problem &P, int32_t dtype, int64_t N, int64_t maxlen)
{
    GlaFwdWs w{};
    // 128 key channels; the backward's dq~ and dk~ sweeps put the 64 or 128
    // value channels on TMEM lanes
    if (dtype != LA_DTYPE_BF16 || P.D != 128 || (P.E != 64 && P.E != 128) ||
        maxlen <= la::SHORT_MAX_T || N > 65535 || P.H > 65535)
        return w;
    w.ncmax = (maxlen + 127) / 128;
    const int64_t rows = P.packed ? 1 : P.B;
    const size_t tok = round256((size_t)rows * P.T * P.H * P.D * 2);
    const size_t vec = round256((size_t)N * P.H * w.ncmax * P.D * 4);
    w.xq = 0;
    w.yk = tok;
    w.er = 2 * tok;
    w.u = 2 * tok + vec;
    w.flags = 2 * tok + 2 * vec;
    w.total = w.flags + round256((size_t)N * P.H * 4);
    return w;
}
GlaFwdWs gla_fwd_layout(const Problem &P, int32_t dtype)
{
    return gla_layout(P, dtype, P.N, gla_max_len(P));
}

// The gated forward's sequence split: the plan, its tables and per-segment
// states (split_setup, at offset 0), each segment's log-decays per key
// channel (lam, [NS][H][D] fp32), its chunks' totals (btot, [NS][H][ncmax][D]
// fp32, from the pre-pass) and the chunked form's buffers for the segments
// (prep).  total 0: no split.  gs: the gate's strides, which must allow the
// one-row token view (NULL: assume they do, for sizing).
struct GlaSplitWs {
    SplitPlan S;
    GlaFwdWs w;
    size_t lam = 0, btot = 0, prep = 0, total = 0;
};
GlaSplitWs gla_split_layout(const Problem &P, const la_dims *d, int32_t dtype, const int64_t *gs)
{
    GlaSplitWs x;
    if (gs && !(P.packed || P.B == 1 || gs[0] == (int64_t)P.T * gs[1]))
        return x;
    x.S = plan_split(P, d);
    if (x.S.NS == 0)
        return x;
    x.w = gla_layout(P, dtype, x.S.NS, x.S.seg_len);
    if (!x.w.total) {
        x.S = SplitPlan{};
        return x;
    }
    x.lam = round256(x.S.bytes);
    x.btot = x.lam + round256((size_t)x.S.NS * P.H * P.D * 4);
    x.prep = x.btot + round256((size_t)x.S.NS * P.H * x.w.ncmax * P.D * 4);
    x.total = x.prep + x.w.total;
    return x;
}

// The pre-pass's arguments for N sequences (or segments, cu their table) of
// the T-token rows; its buffers from the layout w at ws.
la::GlaPrepArgs gla_prep_args(const Problem &P, const la_dims *d, const void *q, const void *k,
                              const float *g, const int64_t *gs, const float *g_gamma,
                              int32_t reverse, uint8_t *ws, const GlaFwdWs &w, int N, int T,
                              const int32_t *cu)
{
    la::GlaPrepArgs pa{};
    pa.N = N;
    pa.H = P.H;
    pa.D = P.D;
    pa.T = T;
    pa.ncmax = w.ncmax;
    pa.cu = cu;
    pa.reverse = reverse ? 1 : 0;
    pa.bf16 = 1;
    pa.q = q;
    pa.k = k;
    pa.sb = d->qk_strides[0];
    pa.st = d->qk_strides[1];
    pa.sh = d->qk_strides[2];
    pa.ksb = P.k_st[0];
    pa.kst = P.k_st[1];
    pa.ksh = P.k_st[2];
    pa.khd = P.G;
    pa.g = g;
    pa.gsb = gs[0];
    pa.gst = gs[1];
    pa.gsh = gs[2];
    pa.g_gamma = g_gamma;
    pa.xq = ws + w.xq;
    pa.yk = ws + w.yk;
    pa.er = reinterpret_cast<float *>(ws + w.er);
    pa.u = reinterpret_cast<float *>(ws + w.u);
    pa.flags = reinterpret_cast<int *>(ws + w.flags);
    pa.lim = 72.f;
    return pa;
}

// The chunked form's forward sweep on the pre-pass's operands: X = q~,
// Y = k~ (dense [rows][T][H][D]), Z = v, the state's rows gated; pairs the
// pre-pass flagged are left to the token-by-token kernels.  so: the final
// states alone.
cudaError_t gla_chunked_sweep(const la::SweepArgs &a, const la::GlaPrepArgs &pa, int64_t ncmax,
                              cudaStream_t s, bool so = false)
{
    la::SweepArgs t = a;
    t.gate = la::Gate{};
    t.gla_er = pa.er;
    t.gla_u = pa.u;
    t.gla_ncmax = ncmax;
    t.gla_flags = pa.flags;
    t.gla_flag_run = 0;
    const int64_t dsh = a.D, dst = (int64_t)a.H * a.D, dsb = dst * a.T;
    return la::tc_gla_sweep(t, false, false, la::Tok{pa.xq, dsb, dst, dsh, 1},
                            la::Tok{pa.yk, dsb, dst, dsh, 1}, t.v, s, so);
}

// The gated forward split into segments (few long sequences): the pre-pass
// over the segments (also giving each chunk's total log-decay), the
// segments' log-decays from those, the sweep's state-only mode from zero states
// (chunked, flagged segments token by token) into the per-segment states,
// the scan with per-channel decays (which writes the final state), and the
// sweep again from the scanned states for the outputs.  The operands are
// laid out per segment, so they are not offered to the backward.
la_status gla_fwd_split(const Problem &P, const la_dims *d, const GlaSplitWs &sw, la::SweepArgs a,
                        const void *q, const void *k, const float *g, const int64_t *gs,
                        const float *g_gamma, const float *initial_state, float *final_state,
                        int32_t reverse, void *workspace, cudaStream_t s)
{
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    SplitBufs b;
    la_status st = split_setup(P, sw.S, workspace, 0, s, &b);
    if (st != LA_OK)
        return st;
    float *lam = reinterpret_cast<float *>(ws + sw.lam);
    uint8_t *pw = ws + sw.prep;
    cudaError_t e = cudaMemsetAsync(pw + sw.w.flags, 0, (size_t)sw.S.NS * P.H * 4, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "gated forward flags");
    to_segments(&a, P, sw.S, b);
    la::GlaPrepArgs pa = gla_prep_args(P, d, q, k, g, gs, g_gamma, reverse, pw, sw.w, sw.S.NS,
                                       a.T, b.seg_cu);
    pa.btot = reinterpret_cast<float *>(ws + sw.btot);
    if ((e = la::gla_prepare(pa, s)) != cudaSuccess)
        return cuda_fail(e, "gated forward operands");
    la::SegDecayArgs sd{};
    sd.NS = sw.S.NS;
    sd.H = P.H;
    sd.D = P.D;
    sd.seg_cu = b.seg_cu;
    sd.btot = pa.btot;
    sd.ncmax = sw.w.ncmax;
    sd.lam = lam;
    if ((e = la::gla_segment_decay(sd, s)) != cudaSuccess)
        return cuda_fail(e, "gated segment decays");
    // two passes: from zero states into W, then from the scanned W
    bool tc = true;
    for (int pass = 0; pass < 2; ++pass) {
        la::SweepArgs t = a;
        t.s_in = pass ? la::StateIn{b.W, P.E, 1} : la::StateIn{nullptr, 0, 0};
        t.s_out = pass ? la::StateOut{nullptr, 0, 0} : la::StateOut{b.W, P.E, 1};
        if (tc) {
            e = gla_chunked_sweep(t, pa, sw.w.ncmax, s, pass == 0);
            if (e == cudaErrorNotSupported && pass == 0)
                tc = false;   // every segment token by token, in both passes
            else if (e != cudaSuccess)
                return cuda_fail(e, "gated tensor-core sweep launch");
        }
        t.gla_flags = tc ? pa.flags : nullptr;
        t.gla_flag_run = 1;
        if ((st = short_run(t, false, s)))
            return st;
        if (pass == 0) {
            la::SplitScanArgs sc =
                scan_args(P, b, g_gamma, P.D, P.E, la::StateIn{initial_state, P.E, 1},
                          la::StateOut{final_state, P.E, 1}, reverse != 0);
            sc.lam = lam;   // the key channels are the state's rows
            if ((st = scan(sc, s)))
                return st;
        }
    }
    return LA_OK;
}

// dq and dk of the gated backward go through fp32 workspace rows (dense
// [rows][T][H][D], one row per query head) for bf16 tokens (the gate's
// gradient reads them unrounded before the bf16 copies are written) and
// whenever k has strides of its own (grouped key/value heads: the rows hold
// each query head's part of dk until the group is summed).
bool gla_f32_grads(const Problem &P, const la_dims *d, int32_t dtype)
{
    return dtype == LA_DTYPE_BF16 || P.G > 1 || P.k_st[0] != d->qk_strides[0] ||
           P.k_st[1] != d->qk_strides[1] || P.k_st[2] != d->qk_strides[2];
}

// Workspace of la_gla_bwd: the final state transposed, the block sums, the
// fp32 dq and dk rows (gla_f32_grads) and, with grouped key/value heads, each
// query head's part of dv (dense [rows][T][H][E], token dtype).
struct GlaBwdWs {
    size_t bsum, dqf, dkf, cv, total;
};
GlaBwdWs gla_bwd_layout(const Problem &P, const la_dims *d, int32_t dtype)
{
    GlaBwdWs w{};
    const int64_t nblk = (gla_max_len(P) + la::DG_TB - 1) / la::DG_TB;
    const int64_t rows = P.packed ? 1 : P.B;
    const size_t tokf =
        gla_f32_grads(P, d, dtype) ? round256((size_t)rows * P.T * P.H * P.D * 4) : 0;
    const size_t tokv =
        P.G > 1 ? round256((size_t)rows * P.T * P.H * P.E * (dtype == LA_DTYPE_BF16 ? 2 : 4))
                : 0;
    w.bsum = round256((size_t)P.N * P.H * P.D * P.E * 4);
    w.dqf = w.bsum + round256((size_t)P.N * P.H * nblk * P.D * 4);
    w.dkf = w.dqf + tokf;
    w.cv = w.dkf + tokf;
    w.total = w.cv + tokv;
    return w;
}

// Whether the gated backward's chunked form can take these tensors: 16-byte
// aligned token rows for its tensor maps and 8-byte gate pairs.
bool gla_bwd_chunkable(const Problem &P, const la_dims *d, const void *q, const void *k,
                       const void *v, const void *d_o, const void *dq, const void *dk,
                       const void *dv, const float *g, const int64_t *gs, const float *dg)
{
    auto al = [](const void *p, const int64_t *st) {
        return (reinterpret_cast<uintptr_t>(p) & 15) == 0 && st[0] % 8 == 0 && st[1] % 8 == 0 &&
               st[2] % 8 == 0;
    };
    const bool aligned = al(q, d->qk_strides) && al(k, P.k_st) && al(dq, d->qk_strides) &&
                         al(dk, P.k_st) && al(v, P.kv_v_st) && al(d_o, d->v_strides) &&
                         al(dv, P.kv_v_st);
    const bool gate_pairs = (reinterpret_cast<uintptr_t>(g) & 7) == 0 &&
                            (reinterpret_cast<uintptr_t>(dg) & 7) == 0 && gs[0] % 2 == 0 &&
                            gs[1] % 2 == 0 && gs[2] % 2 == 0;
    return aligned && gate_pairs;
}

// Workspace of the gated backward's split: the split tables and one state per
// (segment, head) (W: the dq~ sweep's, then dv's, whose transposes dk~ takes),
// the segments' log-decays, their chunks' totals, each segment's sum of dg's
// terms and its dg offset, the gate gradient's block sums per segment, the
// per-sequence part of la_gla_bwd's own layout (final state, fp32 dq, dk,
// grouped dv parts; base) and the pre-pass buffers for the segments (prep).
struct GlaBwdSplitWs {
    SplitPlan S;
    GlaFwdWs w;
    GlaBwdWs bw;
    int64_t nblk = 0;
    size_t lam = 0, btot = 0, segtot = 0, off = 0, bsum = 0, base = 0, prep = 0, total = 0;
};
GlaBwdSplitWs gla_bwd_split_layout(const Problem &P, const la_dims *d, int32_t dtype,
                                   const int64_t *gs)
{
    GlaBwdSplitWs x;
    if (gs && !(P.packed || P.B == 1 || gs[0] == (int64_t)P.T * gs[1]))
        return x;
    x.S = plan_split(P, d);
    if (x.S.NS == 0)
        return x;
    x.w = gla_layout(P, dtype, x.S.NS, x.S.seg_len);
    if (!x.w.total) {
        x.S = SplitPlan{};
        return x;
    }
    x.bw = gla_bwd_layout(P, d, dtype);
    x.nblk = (x.S.seg_len + la::DG_TB - 1) / la::DG_TB;
    const size_t vec = round256((size_t)x.S.NS * P.H * P.D * 4);
    x.lam = round256(x.S.bytes);
    x.btot = x.lam + vec;
    x.segtot = x.btot + round256((size_t)x.S.NS * P.H * x.w.ncmax * P.D * 4);
    x.off = x.segtot + vec;
    x.bsum = x.off + vec;
    x.base = x.bsum + round256((size_t)x.S.NS * P.H * x.nblk * P.D * 4);
    x.prep = x.base + x.bw.total;
    x.total = x.prep + x.w.total;
    return x;
}

// The gated backward split into segments: the pre-pass over the segments
// (with the chunk totals) and the segments' log-decays; dq~ in two passes
// around a scan with column decays (which gives the final state, transposed,
// for dg); dv in two passes around a scan against the processing order with
// row decays (which gives d_initial_state); dk~ in one pass from the scanned
// G, transposed; the rescaling pass per segment (dq, dk, and dg from the
// segment's own terms, with each segment's total); the flagged segments'
// dg from the block scan; then each segment's dg offset (the later
// segments' totals and the final state's term) added.  Flagged segments run
// token by token in every pass.
la_status gla_bwd_split(const Problem &P, const la_dims *d, int32_t dtype, const GlaBwdSplitWs &sx,
                        la::SweepArgs a, const void *q, const void *k, const void *v,
                        const void *d_o, const float *g, const int64_t *gs, const float *g_gamma,
                        const float *initial_state, const float *d_final_state, int32_t reverse,
                        void *dq, void *dk, void *dv, float *dg, float *d_initial_state,
                        uint8_t *ws, cudaStream_t s)
{
    SplitBufs b;
    la_status st = split_setup(P, sx.S, ws, 0, s, &b);
    if (st != LA_OK)
        return st;
    float *lam = reinterpret_cast<float *>(ws + sx.lam);
    uint8_t *base = ws + sx.base;
    float *Ft = reinterpret_cast<float *>(base);
    float *dqf = reinterpret_cast<float *>(base + sx.bw.dqf);
    float *dkf = reinterpret_cast<float *>(base + sx.bw.dkf);
    const bool grouped = P.G > 1;
    to_segments(&a, P, sx.S, b);   // the one-row view, segments as sequences
    const int64_t fsh = P.D, fst = (int64_t)P.H * P.D, fsb = fst * a.T;
    const int64_t vsh = P.E, vst = (int64_t)P.H * P.E, vsb = vst * a.T;
    const la::TokOut dvo =
        grouped ? la::TokOut{base + sx.bw.cv, vsb, vst, vsh} : tok_out(dv, P.kv_v_st);
    uint8_t *pw = ws + sx.prep;
    cudaError_t e = cudaMemsetAsync(pw + sx.w.flags, 0, (size_t)sx.S.NS * P.H * 4, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "gated backward flags");
    la::GlaPrepArgs pa = gla_prep_args(P, d, q, k, g, gs, g_gamma, reverse, pw, sx.w, sx.S.NS,
                                       a.T, b.seg_cu);
    pa.btot = reinterpret_cast<float *>(ws + sx.btot);
    if ((e = la::gla_prepare(pa, s)) != cudaSuccess)
        return cuda_fail(e, "gated backward operands");
    la::SegDecayArgs sd{};
    sd.NS = sx.S.NS;
    sd.H = P.H;
    sd.D = P.D;
    sd.seg_cu = b.seg_cu;
    sd.btot = pa.btot;
    sd.ncmax = sx.w.ncmax;
    sd.lam = lam;
    if ((e = la::gla_segment_decay(sd, s)) != cudaSuccess)
        return cuda_fail(e, "gated segment decays");
    const int64_t dsh = P.D, dst = (int64_t)P.H * P.D, dsb = dst * a.T;
    const la::Tok tq{pa.xq, dsb, dst, dsh, 1}, tk{pa.yk, dsb, dst, dsh, 1};
    const la::Tok tdo = tok(d_o, d->v_strides), tv = tok(v, P.kv_v_st, P.G);
    // one sweep: the chunked form (x, y, z tiles) for the pairs in range, the
    // token-by-token kernels (u's tiles and gate) for the flagged ones
    // (so: the tensor-core sweep's state-only mode, for the first passes)
    auto sweep = [&](la::SweepArgs t, la::SweepArgs u, bool bwd, bool cols, const la::Tok &x,
                     const la::Tok &y, const la::Tok &z, bool so) -> la_status {
        t.gate = la::Gate{};
        t.gla_er = pa.er;
        t.gla_u = pa.u;
        t.gla_ncmax = sx.w.ncmax;
        t.gla_flags = pa.flags;
        t.gla_flag_run = 0;
        cudaError_t err = la::tc_gla_sweep(t, bwd, cols, x, y, z, s, so);
        if (err != cudaSuccess)
            return cuda_fail(err, "gated tensor-core sweep launch");
        u.gla_flags = pa.flags;
        u.gla_flag_run = 1;
        return short_run(u, bwd, s);
    };
    la::SweepArgs t = a, u = a;
    // dq~ (fp32): forward-type (do, v, k~); S^T with gated columns
    t.D = u.D = P.E;
    t.E = u.E = P.D;
    t.out = u.out = la::TokOut{dqf, fsb, fst, fsh};
    u.out_f32 = 1;
    u.q = tdo;
    u.k = tv;
    u.v = tok(k, P.k_st, P.G);
    u.gate = gate_of(g, gs, true);
    for (int pass = 0; pass < 2; ++pass) {
        t.s_in = u.s_in = pass ? la::StateIn{b.W, P.D, 1} : la::StateIn{nullptr, 0, 0};
        t.s_out = u.s_out = pass ? la::StateOut{nullptr, 0, 0} : la::StateOut{b.W, P.D, 1};
        if ((st = sweep(t, u, false, true, tdo, tv, tk, pass == 0)))
            return st;
        if (pass == 0) {
            la::SplitScanArgs sc =
                scan_args(P, b, g_gamma, P.E, P.D, la::StateIn{initial_state, 1, P.E},
                          la::StateOut{Ft, P.D, 1}, reverse != 0);
            sc.lam = lam;
            sc.lam_cols = 1;   // the key channels are S^T's columns
            if ((st = scan(sc, s)))
                return st;
        }
    }
    // dv: backward-type (k~, q~, do); G with gated rows, scanned against the
    // processing order from d_final_state
    t = a;
    u = a;
    t.D = u.D = P.D;
    t.E = u.E = P.E;
    t.out = u.out = dvo;
    u.q = tok(q, d->qk_strides);
    u.k = tok(k, P.k_st, P.G);
    u.v = tdo;
    u.gate = gate_of(g, gs, false);
    for (int pass = 0; pass < 2; ++pass) {
        t.s_in = u.s_in = pass ? la::StateIn{b.W, P.E, 1} : la::StateIn{nullptr, 0, 0};
        t.s_out = u.s_out = pass ? la::StateOut{nullptr, 0, 0} : la::StateOut{b.W, P.E, 1};
        if ((st = sweep(t, u, true, false, tk, tq, tdo, pass == 0)))
            return st;
        if (pass == 0) {
            la::SplitScanArgs sc =
                scan_args(P, b, g_gamma, P.D, P.E, la::StateIn{d_final_state, P.E, 1},
                          la::StateOut{d_initial_state, P.E, 1}, reverse == 0);
            sc.lam = lam;   // the key channels are G's rows
            if ((st = scan(sc, s)))
                return st;
        }
    }
    // dk~ (fp32): backward-type (v, do, q~) from each segment's G, transposed
    t = a;
    u = a;
    t.D = u.D = P.E;
    t.E = u.E = P.D;
    t.out = u.out = la::TokOut{dkf, fsb, fst, fsh};
    u.out_f32 = 1;
    u.q = tdo;
    u.k = tv;
    u.v = tok(q, d->qk_strides);
    u.gate = gate_of(g, gs, true);
    t.s_in = u.s_in = la::StateIn{b.W, 1, P.E};
    t.s_out = u.s_out = la::StateOut{nullptr, 0, 0};
    if ((st = sweep(t, u, true, true, tv, tdo, tq, false)))
        return st;
    // dq, dk and each segment's own dg (no final-state term) with its total
    float *segtot = reinterpret_cast<float *>(ws + sx.segtot);
    pa.dq = dq;
    pa.dk = dk;
    pa.dk32 = grouped ? dkf : nullptr;
    pa.dqf = dqf;
    pa.dkf = dkf;
    pa.dg = dg;
    pa.Ft = nullptr;
    pa.dF = nullptr;
    pa.E = P.E;
    pa.segtot = segtot;
    if ((e = la::gla_undo(pa, s)) != cudaSuccess)
        return cuda_fail(e, "gated backward rescale");
    float *bsum = reinterpret_cast<float *>(ws + sx.bsum);
    la::GateGradArgs gg{};
    gg.N = sx.S.NS;
    gg.H = P.H;
    gg.D = P.D;
    gg.E = P.E;
    gg.T = a.T;
    gg.nblk = sx.nblk;
    gg.cu = b.seg_cu;
    gg.reverse = reverse ? 1 : 0;
    gg.bf16 = dtype == LA_DTYPE_BF16;
    gg.q = q;
    gg.k = k;
    gg.sb = d->qk_strides[0];
    gg.st = d->qk_strides[1];
    gg.sh = d->qk_strides[2];
    gg.ksb = P.k_st[0];
    gg.kst = P.k_st[1];
    gg.ksh = P.k_st[2];
    gg.khd = P.G;
    gg.dqf = dqf;
    gg.dkf = dkf;
    gg.fsb = fsb;
    gg.fst = fst;
    gg.fsh = fsh;
    gg.dq = dq;
    gg.dk = grouped ? nullptr : dk;
    gg.dg = dg;
    gg.gsb = gs[0];
    gg.gst = gs[1];
    gg.gsh = gs[2];
    gg.Ft = nullptr;
    gg.dF = nullptr;
    gg.bsum = bsum;
    gg.flags = pa.flags;
    if ((e = la::gate_grad(gg, s)) != cudaSuccess)
        return cuda_fail(e, "gate gradient");
    la::SplitDgArgs sg{};
    sg.N = P.N;
    sg.NS = sx.S.NS;
    sg.H = P.H;
    sg.D = P.D;
    sg.E = P.E;
    sg.seg_cu = b.seg_cu;
    sg.seq_first = b.seq_first;
    sg.reverse = reverse ? 1 : 0;
    sg.flags = pa.flags;
    sg.segtot = segtot;
    sg.bsum = bsum;
    sg.nblk = sx.nblk;
    sg.Ft = Ft;
    sg.dF = d_final_state;
    sg.off = reinterpret_cast<float *>(ws + sx.off);
    sg.dg = dg;
    sg.gst = gs[1];
    sg.gsh = gs[2];
    sg.max_seg_len = sx.S.seg_len;
    if ((e = la::split_dg(sg, s)) != cudaSuccess)
        return cuda_fail(e, "gate gradient of the split");
    if (grouped) {
        const int rows = P.packed ? 1 : P.B;
        const int bf16 = dtype == LA_DTYPE_BF16;
        e = la::gqa_reduce(dkf, tok_out(dk, P.k_st), rows, P.T, P.Hkv, P.G, P.D, bf16, s, true);
        if (e == cudaSuccess)
            e = la::gqa_reduce(dvo.p, tok_out(dv, P.kv_v_st), rows, P.T, P.Hkv, P.G, P.E, bf16,
                               s);
        if (e != cudaSuccess)
            return cuda_fail(e, "grouped key/value gradient sum");
    }
    return LA_OK;
}

}  // namespace

extern "C" {

size_t la_gla_fwd_workspace_size(const la_dims *dims, int32_t dtype,
                                 const int32_t *cu_seqlens_host)
{
    Problem P;
    std::string keep = g_msg;
    la_status st = check_dims(dims, dtype, cu_seqlens_host, cu_seqlens_host, nullptr, &P);
    g_msg = keep;
    if (st != LA_OK)
        return 0;
    return std::max(gla_fwd_layout(P, dtype).total,
                    gla_split_layout(P, dims, dtype, nullptr).total);
}

la_status la_gla_fwd(const la_dims *dims, int32_t dtype, const void *q, const void *k,
                     const void *v, const float *g, const int64_t *g_strides,
                     const float *g_gamma, float scale, const float *initial_state,
                     int32_t reverse, const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                     void *o, float *final_state, void *workspace, size_t workspace_bytes,
                     int32_t *operands_written, void *stream)
{
    if (operands_written)
        *operands_written = 0;
    g_msg.clear();
    cudaStream_t s = (cudaStream_t)stream;
    Problem P;
    la_status st = check_dims(dims, dtype, cu_seqlens, cu_seqlens_host, s, &P);
    if (st != LA_OK)
        return st;
    if (has_tokens(P)) {
        if ((st = need(q, "q")) || (st = need(k, "k")) || (st = need(v, "v")) ||
            (st = need(o, "o")))
            return st;
    }
    if ((st = gla_check(P, dims, g, g_strides, g_gamma)) || !has_states(P))
        return st;
    la::SweepArgs a = base_args(P, dtype, cu_seqlens, g_gamma, scale, reverse);
    a.D = P.D;
    a.E = P.E;
    a.q = tok(q, dims->qk_strides);
    a.k = tok(k, P.k_st, P.G);
    a.v = tok(v, P.kv_v_st, P.G);
    a.out = tok_out(o, dims->v_strides);
    a.s_in = la::StateIn{initial_state, P.E, 1};
    a.s_out = la::StateOut{final_state, P.E, 1};
    a.gate = gate_of(g, g_strides, false);   // state rows are key channels
    // the operands are prepared two channels at a time: 8-byte gate pairs
    const bool gate_pairs = (reinterpret_cast<uintptr_t>(g) & 7) == 0 && g_strides[0] % 2 == 0 &&
                            g_strides[1] % 2 == 0 && g_strides[2] % 2 == 0;
    const bool ws_ok = workspace && (reinterpret_cast<uintptr_t>(workspace) & 255) == 0;
    const bool chunked = ws_ok && gate_pairs && la::tc_sweep_supported(a);
    const GlaSplitWs sw = gla_split_layout(P, dims, dtype, g_strides);
    if (chunked && sw.total && workspace_bytes >= sw.total)
        return gla_fwd_split(P, dims, sw, a, q, k, g, g_strides, g_gamma, initial_state,
                             final_state, reverse, workspace, s);
    const GlaFwdWs w = gla_fwd_layout(P, dtype);
    if (chunked && w.total && workspace_bytes >= w.total) {
        // the chunked form on the tensor cores, for every (sequence, head)
        // whose gates stay in its range; the others token by token
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        cudaError_t e = cudaMemsetAsync(ws + w.flags, 0, (size_t)P.N * P.H * 4, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "gated forward flags");
        const la::GlaPrepArgs pa = gla_prep_args(P, dims, q, k, g, g_strides, g_gamma, reverse,
                                                 ws, w, P.N, P.T, cu_seqlens);
        if ((e = la::gla_prepare(pa, s)) != cudaSuccess)
            return cuda_fail(e, "gated forward operands");
        e = gla_chunked_sweep(a, pa, w.ncmax, s);
        if (e == cudaSuccess) {
            a.gla_flags = pa.flags;
            a.gla_flag_run = 1;
            if (operands_written)
                *operands_written = 1;
        } else if (e != cudaErrorNotSupported) {
            return cuda_fail(e, "gated tensor-core sweep launch");
        }
    }
    return short_run(a, false, s);
}

size_t la_gla_workspace_size(const la_dims *dims, int32_t dtype, const int32_t *cu_seqlens_host,
                             int32_t with_forward_operands)
{
    Problem P;
    std::string keep = g_msg;
    la_status st = check_dims(dims, dtype, cu_seqlens_host, cu_seqlens_host, nullptr, &P);
    g_msg = keep;
    if (st != LA_OK)
        return 0;
    const size_t t = gla_bwd_layout(P, dims, dtype).total +
                     (with_forward_operands ? 0 : gla_fwd_layout(P, dtype).total);
    // without the forward's operands, enough for the split where it applies
    return with_forward_operands ? t
                                 : std::max(t, gla_bwd_split_layout(P, dims, dtype, nullptr).total);
}

la_status la_gla_bwd(const la_dims *dims, int32_t dtype, const void *q, const void *k,
                     const void *v, const void *d_o, const float *g, const int64_t *g_strides,
                     const float *g_gamma, float scale, const float *initial_state,
                     const float *d_final_state, int32_t reverse, const int32_t *cu_seqlens,
                     const int32_t *cu_seqlens_host, void *dq, void *dk, void *dv, float *dg,
                     float *d_initial_state, void *workspace, size_t workspace_bytes,
                     void *fwd_workspace, size_t fwd_workspace_bytes, void *stream)
{
    g_msg.clear();
    cudaStream_t s = (cudaStream_t)stream;
    Problem P;
    la_status st = check_dims(dims, dtype, cu_seqlens, cu_seqlens_host, s, &P);
    if (st != LA_OK)
        return st;
    if (has_tokens(P)) {
        if ((st = need(q, "q")) || (st = need(k, "k")) || (st = need(v, "v")) ||
            (st = need(d_o, "d_o")) || (st = need(dq, "dq")) || (st = need(dk, "dk")) ||
            (st = need(dv, "dv")) || (st = need(dg, "dg")))
            return st;
    }
    if ((st = gla_check(P, dims, g, g_strides, g_gamma)) || !has_states(P))
        return st;
    const GlaBwdWs bw = gla_bwd_layout(P, dims, dtype);
    const size_t need_ws = bw.total;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 ||
        workspace_bytes < need_ws)
        return fail(LA_ERR_INVALID_ARG,
                    "la_gla_bwd needs a 256-byte aligned workspace of %zu bytes (got %zu)",
                    need_ws, workspace ? workspace_bytes : (size_t)0);
    uint8_t *wsb = static_cast<uint8_t *>(workspace);
    float *Ft = static_cast<float *>(workspace);
    float *bsum = reinterpret_cast<float *>(wsb + bw.bsum);
    // dq and dk in fp32 rows of the workspace, dense (token stride H D)
    const bool f32g = gla_f32_grads(P, dims, dtype);
    float *dqf = f32g ? reinterpret_cast<float *>(wsb + bw.dqf) : nullptr;
    float *dkf = f32g ? reinterpret_cast<float *>(wsb + bw.dkf) : nullptr;
    const int64_t fsh = P.D, fst = (int64_t)P.H * P.D, fsb = fst * P.T;
    // grouped key/value heads: every query head's part of dk (in dkf) and of
    // dv (below) first, each group summed at the end
    const bool grouped = P.G > 1;
    const int64_t vsh = P.E, vst = (int64_t)P.H * P.E, vsb = vst * P.T;
    const la::TokOut dvo =
        grouped ? la::TokOut{wsb + bw.cv, vsb, vst, vsh} : tok_out(dv, P.kv_v_st);
    la::SweepArgs a = base_args(P, dtype, cu_seqlens, g_gamma, scale, reverse);
    const bool chunkable = gla_bwd_chunkable(P, dims, q, k, v, d_o, dq, dk, dv, g, g_strides, dg);
    // Few long sequences: the split, when the chunked form applies and the
    // workspace holds it (the forward's operands, laid out per sequence, are
    // not used there).
    {
        const GlaBwdSplitWs sx = gla_bwd_split_layout(P, dims, dtype, g_strides);
        if (chunkable && sx.total && workspace_bytes >= sx.total)
            return gla_bwd_split(P, dims, dtype, sx, a, q, k, v, d_o, g, g_strides, g_gamma,
                                 initial_state, d_final_state, reverse, dq, dk, dv, dg,
                                 d_initial_state, wsb, s);
    }
    // The chunked form on the tensor cores, when it applies and the workspace
    // also holds its operands: the three sweeps on q~, k~ for the (sequence,
    // head) pairs in range (dq~, dk~ in fp32 into the workspace), then dq~,
    // dk~ rescaled into dq, dk with dg; the token-by-token sweeps below run
    // only the flagged pairs.
    const int *flags = nullptr;
    la::GlaPrepArgs pa{};
    {
        const GlaFwdWs w = gla_fwd_layout(P, dtype);
        // the forward's operands, when the caller kept them
        const bool ready = w.total && fwd_workspace &&
                           (reinterpret_cast<uintptr_t>(fwd_workspace) & 255) == 0 &&
                           fwd_workspace_bytes >= w.total;
        if (w.total && (ready || workspace_bytes >= need_ws + w.total) && chunkable) {
            uint8_t *ws = ready ? static_cast<uint8_t *>(fwd_workspace)
                                : static_cast<uint8_t *>(workspace) + need_ws;
            int *fl = reinterpret_cast<int *>(ws + w.flags);
            cudaError_t e = ready ? cudaSuccess : cudaMemsetAsync(fl, 0, (size_t)P.N * P.H * 4, s);
            if (e != cudaSuccess)
                return cuda_fail(e, "gated backward flags");
            pa = gla_prep_args(P, dims, q, k, g, g_strides, g_gamma, reverse, ws, w, P.N, P.T,
                               cu_seqlens);
            pa.dq = dq;
            pa.dk = dk;
            pa.dk32 = grouped ? dkf : nullptr;
            pa.dqf = dqf;
            pa.dkf = dkf;
            pa.dg = dg;
            pa.Ft = Ft;
            pa.dF = d_final_state;
            pa.E = P.E;
            if (!ready && (e = la::gla_prepare(pa, s)) != cudaSuccess)
                return cuda_fail(e, "gated backward operands");
            const int64_t dsh = P.D, dst = (int64_t)P.H * P.D, dsb = dst * P.T;
            const la::Tok tq{pa.xq, dsb, dst, dsh, 1}, tk{pa.yk, dsb, dst, dsh, 1};
            const la::Tok tdo = tok(d_o, dims->v_strides), tv = tok(v, P.kv_v_st, P.G);
            la::SweepArgs t = a;
            t.gla_er = pa.er;
            t.gla_u = pa.u;
            t.gla_ncmax = w.ncmax;
            t.gla_flags = fl;
            t.gla_flag_run = 0;
            // dq~ (fp32): forward-type (do, v, k~), state S^T with gated columns
            t.D = P.E;
            t.E = P.D;
            t.out = la::TokOut{dqf, fsb, fst, fsh};
            t.s_in = la::StateIn{initial_state, 1, P.E};
            t.s_out = la::StateOut{Ft, P.D, 1};
            e = la::tc_gla_sweep(t, false, true, tdo, tv, tk, s);
            if (e == cudaSuccess) {
                // dv: backward-type (k~, q~, do), G with gated rows
                t.D = P.D;
                t.E = P.E;
                t.out = dvo;
                t.s_in = la::StateIn{d_final_state, P.E, 1};
                t.s_out = la::StateOut{d_initial_state, P.E, 1};
                e = la::tc_gla_sweep(t, true, false, tk, tq, tdo, s);
            }
            if (e == cudaSuccess) {
                // dk~ (fp32): backward-type (v, do, q~), G^T with gated columns
                t.D = P.E;
                t.E = P.D;
                t.out = la::TokOut{dkf, fsb, fst, fsh};
                t.s_in = la::StateIn{d_final_state, 1, P.E};
                t.s_out = la::StateOut{nullptr, 0, 0};
                e = la::tc_gla_sweep(t, true, true, tv, tdo, tq, s);
            }
            if (e != cudaSuccess)
                return cuda_fail(e, "gated tensor-core sweep launch");
            flags = fl;
            a.gla_flags = fl;
            a.gla_flag_run = 1;
        }
    }
    // dq: forward-type with (q, k, v) := (do, v, k), state S^T (E x D): the
    // gated key channels are its columns; its final state F^T feeds dg
    a.D = P.E;
    a.E = P.D;
    a.q = tok(d_o, dims->v_strides);
    a.k = tok(v, P.kv_v_st, P.G);
    a.v = tok(k, P.k_st, P.G);
    a.out = f32g ? la::TokOut{dqf, fsb, fst, fsh} : tok_out(dq, dims->qk_strides);
    a.out_f32 = f32g ? 1 : 0;
    a.s_in = la::StateIn{initial_state, 1, P.E};
    a.s_out = la::StateOut{Ft, P.D, 1};
    a.gate = gate_of(g, g_strides, true);
    if ((st = short_run(a, false, s)))
        return st;
    // dv: backward-type (q, k, do), G = dL/dS (D x E): gated rows
    a.D = P.D;
    a.E = P.E;
    a.q = tok(q, dims->qk_strides);
    a.k = tok(k, P.k_st, P.G);
    a.v = tok(d_o, dims->v_strides);
    a.out = dvo;
    a.out_f32 = 0;
    a.s_in = la::StateIn{d_final_state, P.E, 1};
    a.s_out = la::StateOut{d_initial_state, P.E, 1};
    a.gate = gate_of(g, g_strides, false);
    if ((st = short_run(a, true, s)))
        return st;
    // dk: backward-type (do, v, q), G^T (E x D): gated columns
    a.D = P.E;
    a.E = P.D;
    a.q = tok(d_o, dims->v_strides);
    a.k = tok(v, P.kv_v_st, P.G);
    a.v = tok(q, dims->qk_strides);
    a.out = f32g ? la::TokOut{dkf, fsb, fst, fsh} : tok_out(dk, P.k_st);
    a.out_f32 = f32g ? 1 : 0;
    a.s_in = la::StateIn{d_final_state, 1, P.E};
    a.s_out = la::StateOut{nullptr, 0, 0};
    a.gate = gate_of(g, g_strides, true);
    if ((st = short_run(a, true, s)))
        return st;
    if (flags) {
        cudaError_t e = la::gla_undo(pa, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "gated backward rescale");
    }
    // dg from q dq - k dk and the final-state term
    la::GateGradArgs gg{};
    gg.N = P.N;
    gg.H = P.H;
    gg.D = P.D;
    gg.E = P.E;
    gg.T = P.T;
    gg.nblk = (gla_max_len(P) + la::DG_TB - 1) / la::DG_TB;
    gg.cu = cu_seqlens;
    gg.reverse = reverse ? 1 : 0;
    gg.bf16 = dtype == LA_DTYPE_BF16;
    gg.q = q;
    gg.k = k;
    gg.sb = dims->qk_strides[0];
    gg.st = dims->qk_strides[1];
    gg.sh = dims->qk_strides[2];
    gg.ksb = P.k_st[0];
    gg.kst = P.k_st[1];
    gg.ksh = P.k_st[2];
    gg.khd = P.G;
    if (f32g) {
        // fp32 gradients from the workspace; the kernels write the token-dtype
        // copies (dk: the group sums below, when grouped)
        gg.dqf = dqf;
        gg.dkf = dkf;
        gg.fsb = fsb;
        gg.fst = fst;
        gg.fsh = fsh;
        gg.dq = dq;
        gg.dk = grouped ? nullptr : dk;
    } else {
        gg.dqf = static_cast<const float *>(dq);
        gg.dkf = static_cast<const float *>(dk);
        gg.fsb = gg.sb;
        gg.fst = gg.st;
        gg.fsh = gg.sh;
    }
    gg.dg = dg;
    gg.gsb = g_strides[0];
    gg.gst = g_strides[1];
    gg.gsh = g_strides[2];
    gg.Ft = Ft;
    gg.dF = d_final_state;
    gg.bsum = bsum;
    gg.flags = flags;
    cudaError_t e = la::gate_grad(gg, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "gate gradient");
    if (grouped) {
        const int rows = P.packed ? 1 : P.B;
        const int bf16 = dtype == LA_DTYPE_BF16;
        e = la::gqa_reduce(dkf, tok_out(dk, P.k_st), rows, P.T, P.Hkv, P.G, P.D, bf16, s, true);
        if (e == cudaSuccess)
            e = la::gqa_reduce(dvo.p, tok_out(dv, P.kv_v_st), rows, P.T, P.Hkv, P.G, P.E, bf16,
                               s);
        if (e != cudaSuccess)
            return cuda_fail(e, "grouped key/value gradient sum");
    }
    return LA_OK;
}

}  // extern "C"

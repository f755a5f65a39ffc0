// la_internal.h -- kernel-launch interface shared by the translation units of
// the library (not part of the public ABI; include/la.h is that).
//
// Two kernel shapes cover the whole method:
//
//  * the "forward-type" sweep: per (sequence, head), chunks in processing order,
//        out_i = sum_{p(j)<=p(i)} s*gamma^(p(i)-p(j)) (q_i . k_j) v_j
//                + s*gamma^(p(i)+1) q_i^T S_in
//        S_out = gamma^Lc S_in + sum_j gamma^(Lc-1-p(j)) k_j v_j^T
//    (p = position in processing order inside the chunk, Lc = chunk length).
//    It is the forward pass, and, with q := do, k := v, v := k and the state
//    transposed, the dq half of the backward pass.
//
//  * the "backward-type" sweep: chunks against processing order, carrying
//    G = dL/dS,
//        out_j = sum_{p(i)>=p(j)} s*gamma^(p(i)-p(j)) (q_i . k_j) w_i
//                + gamma^(Lc-1-p(j)) G_in^T k_j
//        G_out = gamma^Lc G_in + s * sum_i gamma^(p(i)+1) q_i w_i^T
//    (w = do).  It is the dv half of the backward pass, and, with q := do,
//    k := v, w := q and G transposed, the dk half.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace la {

// A token tensor: element (row, token, head, c) lives at
// p + row*sb + token*st + (head / hdiv)*sh + c   (elements of the token dtype);
// hdiv > 1 for key/value tensors shared by groups of hdiv query heads.
struct Tok {
    const void *p;
    int64_t sb, st, sh;
    int hdiv = 1;
};
struct TokOut {
    void *p;
    int64_t sb, st, sh;
};
// A state tensor slice: element (a, b) of (sequence n, head h) lives at
// p + (n*H + h)*D*E + a*rs + b*cs   (fp32).  Transposed views swap rs/cs.
struct StateIn {
    const float *p;
    int64_t rs, cs;
};
struct StateOut {
    float *p;
    int64_t rs, cs;
};

// A per-key gate (fp32 log-decay added to g[h]): element (row, token, head,
// channel) at p + row*sb + token*st + head*sh + channel.  The gated channel is
// the state's row index (cols == 0) or its column index (cols == 1).
struct Gate {
    const float *p = nullptr;
    int64_t sb = 0, st = 0, sh = 0;
    int cols = 0;
};

struct SweepArgs {
    int B, T, H, D, E, N;     // D: width of q and k; E: width of v (w) and out
    const int32_t *cu;        // device [N+1] or nullptr (dense: N == B rows of T)
    const int32_t *order;     // device [N]: sequence processed at rank r, longest first;
                              // nullptr = natural order
    const float *g;           // [H] log-decay
    float scale;
    int reverse;
    int bf16;                 // token dtype: 1 bf16, 0 fp32
    Tok q, k, v;              // forward-type: q, k, v; backward-type: q, k, w
    TokOut out;               // forward-type: o (or dq); backward-type: dv (or dk)
    StateIn s_in;             // forward-type: initial state; backward-type: dL/dfinal
    StateOut s_out;           // forward-type: final state; backward-type: dL/dinitial
    int withhold_handoff;     // diagnostic: the tensor-core and streamed decode kernels skip one hand-off
    int64_t max_len;          // longest sequence (T when dense)
    Gate gate;                // per-key log-decay gate, or p == nullptr
    int64_t prefetch_ctas = 0;  // token-by-token kernels: L2 prefetch distance in CTAs
    // gated form on the tensor cores (la_gla_prep.cu): per chunk position and
    // state row, exp(r) and exp(B - r), [N][H][gla_ncmax][D]
    const float *gla_er = nullptr, *gla_u = nullptr;
    int64_t gla_ncmax = 0;
    // a CTA of (sequence n, head h) runs only if gla_flags is null or
    // gla_flags[n H + h] == gla_flag_run (1: gates out of the chunked form's
    // range, run token by token)
    const int *gla_flags = nullptr;
    int gla_flag_run = 0;
    // token-by-token kernels with bf16 tokens: out is fp32 (strides in floats)
    int out_f32 = 0;
};

// Operands of the chunked gated forward (la_gla_prep.cu).
struct GlaPrepArgs {
    int N, H, D, T;
    int64_t ncmax;            // chunks of the longest sequence
    const int32_t *cu;        // packed sequences, or nullptr
    int reverse, bf16;
    const void *q, *k;        // token dtype: q (and dq) at strides sb, st, sh; k
    int64_t sb, st, sh;       // (and dk) at ksb, kst, ksh, head h reading key
    int64_t ksb, kst, ksh;    // head h / khd (grouped key/value heads)
    int khd;
    const float *g;           // gate, strides gsb, gst, gsh
    int64_t gsb, gst, gsh;
    const float *g_gamma;
    void *xq, *yk;            // bf16 [rows][T][H][D]: q~ and k~
    float *er, *u;            // [N][H][ncmax][D]
    int *flags;               // [N H], zeroed beforehand
    float *btot = nullptr;    // gla_prepare, when set: each chunk's total log-decay
                              // per channel, [N][H][ncmax][D]
    float lim;                // largest |b - r| (and |r|) the chunked form takes
    void *dq, *dk;            // gla_undo: dq, dk out (token dtype, their strides)
    const float *dqf, *dkf;   // gla_undo: dq~, dk~ in (fp32, dense [rows][T][H][D])
    float *dk32;              // gla_undo: when set, dk goes there in fp32, in
                              // place of dk~ (per query head), not to dk
    float *segtot = nullptr;  // gla_undo, when set: each pair's sum of the terms
                              // (with the final state's, if dF), [N][H][D]
    float *dg;                // gla_undo: the gate's gradient (the gate's strides)
    const float *Ft, *dF;     // gla_undo: final state (transposed, [E][D] per
                              // pair) and its gradient ([D][E]), or dF null
    int E;
};
cudaError_t gla_prepare(const GlaPrepArgs &a, cudaStream_t s);
// dq~ -> dq, dk~ -> dk (fp32 in, token dtype out), and the gate's gradient
// dg from the rounded operands q~, k~ and their own gradients dq~, dk~, for
// the (sequence, head) pairs not flagged: one pass over each sequence against
// the processing order, the later chunks' terms carried in registers.
cudaError_t gla_undo(const GlaPrepArgs &a, cudaStream_t s);
// Each segment's total log-decay per key channel (the gated form's sequence
// split): lam[seg][h][c] = the sum over the segment's chunks of their totals
// btot[seg][h][chunk][c] (gla_prepare over the segments: len * g_gamma[h]
// plus the segment's gates).  D <= 256.
struct SegDecayArgs {
    int NS, H, D;
    const int32_t *seg_cu;
    const float *btot;
    int64_t ncmax;
    float *lam;
};
cudaError_t gla_segment_decay(const SegDecayArgs &a, cudaStream_t s);
// A tensor-core sweep of the gated form on rescaled operands (la_gla_prep.cu)
// with tile roles X, Y, Z given: forward-type or backward-type (bwd), the 128
// gated key channels being the state's rows (D = 128, E in {64, 128}) or its
// columns (cols: E = 128, D in {64, 128}); a.gla_* set, a.out the output:
// bf16 rows, or with cols (the sweeps giving dq~ and dk~) fp32 rows, 16-byte
// aligned.  so: the final states alone (the state-only mode; X and the output
// are not touched), for the sequence split's first pass.
// cudaErrorNotSupported when the tensor maps cannot be built.
cudaError_t tc_gla_sweep(const SweepArgs &a, bool bwd, bool cols, const Tok &x, const Tok &y,
                         const Tok &z, cudaStream_t s, bool so = false);
// The final states of a sweep alone (its outputs are not written; X is not
// read): the tensor-core kernel's state-only mode, for the sequence split's
// first pass.  Eligibility as tc_sweep_supported.
cudaError_t tc_state_sweep(const SweepArgs &a, bool bwd, cudaStream_t s);

// Calls whose longest sequence has at most this many tokens run the
// token-by-token kernels (la_token.cu) instead of the chunked ones.
constexpr int SHORT_MAX_T = 16;

// Host-side count of enqueued kernels (la_launch_count).
void note_launch();

// Sets the message la_last_error returns on this host thread.
void set_last_error(const char *msg);

// CUDA-core kernels: any D, E in 1..256, bf16 or fp32, every flag.
cudaError_t simt_forward_sweep(const SweepArgs &a, cudaStream_t s);
cudaError_t simt_backward_sweep(const SweepArgs &a, cudaStream_t s);

// Token-by-token kernels: any length (tokens pass through shared memory 16 at
// a time), any D in 1..256, any E, bf16 or fp32, every flag, and the only
// kernels that take a gate; cudaErrorNotSupported outside that range.  Used
// for every gated call and for ungated calls whose longest sequence has at
// most SHORT_MAX_T tokens.
// (*streamed, when given: whether the streamed decode kernel ran.)
cudaError_t short_forward_sweep(const SweepArgs &a, cudaStream_t s, bool *streamed = nullptr);
// Decoding up to 16 tokens as one chunk on the tensor cores (la_decode.cu):
// bf16, D = 128, E a multiple of 16 up to 128, forward-type, no gate,
// contiguous 16-byte aligned states, 16-byte aligned token rows;
// cudaErrorNotSupported otherwise.  (*streamed, when given: whether the
// streamed form, the one with ring hand-offs, ran.)
cudaError_t decode_chunk_sweep(const SweepArgs &a, cudaStream_t s, bool *streamed = nullptr);
// Reads (after synchronizing s) and clears the decode kernels' device error
// word (LA_ERR_TIMEOUT when a wait of the streamed form ran out).
cudaError_t decode_read_and_clear_error(cudaStream_t s, int *err);
cudaError_t short_backward_sweep(const SweepArgs &a, cudaStream_t s);
// Reads (after synchronizing s) and clears the token kernels' device error
// word (LA_ERR_TIMEOUT when a wait of the streamed decode kernel ran out).
cudaError_t token_read_and_clear_error(cudaStream_t s, int *err);

// Tensor-core (tcgen05) kernels for bf16, both sweep shapes; eligibility
// (dtype, widths, 16-byte alignment) is the same for both.
bool tc_sweep_supported(const SweepArgs &a);
cudaError_t tc_forward_sweep(const SweepArgs &a, cudaStream_t s);
cudaError_t tc_backward_sweep(const SweepArgs &a, cudaStream_t s);

// Sum of grouped contributions (la_gqa.cu): out[b, t, j, c] = sum over
// i < G of in[b, t, j*G + i, c] in fp32, for j < Hkv and c < X; `in` is dense
// [B, T, Hkv*G, X] of the token dtype (fp32 when in_f32), `out` strided like a
// TokOut, of the token dtype.
cudaError_t gqa_reduce(const void *in, const TokOut &out, int B, int T, int Hkv, int G, int X,
                       int bf16, cudaStream_t s, bool in_f32 = false);

// Gradient of the per-key gate (la_gla.cu) from q, k (token dtype) and the
// fp32 gradients dqf, dkf; dg is fp32 with the gate's strides.  With dq (dk)
// set, the kernels also write dqf (dkf) there in the token dtype.
// Ft: the final state transposed [N][H][E][D] (fp32), dF: its upstream
// gradient [N][H][D][E] (either may be null: no final-state term).  bsum:
// scratch [N][H][nblk][D] fp32, nblk = ceil(longest sequence / DG_TB).
constexpr int DG_TB = 256;
struct GateGradArgs {
    int N, H, D, E, T;
    int64_t nblk;
    const int32_t *cu;
    int reverse, bf16;
    const void *q, *k;        // token dtype: q (and dq) at strides sb, st, sh; k
    int64_t sb, st, sh;       // (and dk) at ksb, kst, ksh, head h reading key
    int64_t ksb, kst, ksh;    // head h / khd
    int khd;
    const float *dqf, *dkf;   // fp32 dq, dk (per query head), strides fsb, fst, fsh
    int64_t fsb, fst, fsh;
    void *dq, *dk;            // or null: token-dtype copies of dqf, dkf
    float *dg;
    int64_t gsb, gst, gsh;
    const float *Ft, *dF;
    float *bsum;
    // when set, only the (sequence, head) pairs whose flag is set are done
    // (gla_undo did the others)
    const int *flags = nullptr;
};
cudaError_t gate_grad(const GateGradArgs &a, cudaStream_t s);

// dg of the sequence split (gated backward): each segment's dg was formed
// from its own terms alone (gla_undo with segtot, or gate_grad's block sums
// for the flagged pairs); this adds to every token of segment s the sum of
// the terms of the segments processed after it, plus the final state's term
// sum_e F dF (Ft transposed [N][H][E][D], dF [N][H][D][E], either may be
// null).  Segments of sequence n: [seq_first[n], seq_first[n + 1]) over the
// one-row token view (seg_cu); dg strides gst, gsh.  off: scratch [NS][H][D].
struct SplitDgArgs {
    int N, NS, H, D, E;
    const int32_t *seg_cu, *seq_first;
    int reverse;
    const int *flags;          // [NS][H]: flagged pairs take their total from bsum
    const float *segtot;       // [NS][H][D]
    const float *bsum;         // [NS][H][nblk][D]
    int64_t nblk;
    const float *Ft, *dF;
    float *off;
    float *dg;
    int64_t gst, gsh;
    int64_t max_seg_len;       // the longest segment's tokens
};
cudaError_t split_dg(const SplitDgArgs &a, cudaStream_t s);

// State scan of the sequence split (la_split.cu).  W holds one D x E fp32
// state per (segment, head), [NS][H][D][E]; on entry the segments' results
// from a zero state, on return their initial states.  Sequence n owns the
// consecutive segments [seq_first[n], seq_first[n+1]), of lengths
// seg_cu[s+1] - seg_cu[s], visited in token order (or reversed).  start is the
// sequence's initial state (zero when null) and fin receives its final state
// (skipped when null), both with the StateIn / StateOut indexing.
// With lam set (the gated form) a segment's decay is per key channel:
// element (r, c) takes exp(lam[seg][h][r]) (lam_cols == 0: the key channels
// are the rows, lam [NS][H][D]) or exp(lam[seg][h][c]) (lam_cols: columns,
// lam [NS][H][E]) instead of gamma^L.
struct SplitScanArgs {
    int N, H, D, E;
    const int32_t *seg_cu;      // device [NS + 1]
    const int32_t *seq_first;   // device [N + 1]
    const float *g;             // [H]
    float *W;
    StateIn start;
    StateOut fin;
    int descending;
    const float *lam = nullptr;
    int lam_cols = 0;
};
cudaError_t split_scan(const SplitScanArgs &a, cudaStream_t s);

// Device error word of the tensor-core kernels (bounded waits that ran out).
cudaError_t tc_read_and_clear_error(cudaStream_t s, int *err);

// The backward's dk and dv in one tensor-core sweep (la_tc_dkdv.cu): bf16,
// D = E = 128, layouts TMA can describe.  Arguments as the dv sweep (a.q = q,
// a.k = k, a.v = do, a.out = dv, a.s_in = dL/dfinal as D x E, a.s_out =
// dL/dinitial) plus v and dk.  cudaErrorNotSupported when the tensor maps
// cannot be built.
bool tc_dkdv_supported(const SweepArgs &a, const Tok &v, const TokOut &dk);
cudaError_t tc_dkdv_sweep(const SweepArgs &a, const Tok &v, const TokOut &dk, cudaStream_t s);
cudaError_t tc_dkdv_read_and_clear_error(cudaStream_t s, int *err);

}  // namespace la

/*
 * la.h -- C ABI of the GB300 (sm_103a) library for causal linear attention
 * with a per-head scalar exponential decay (Lightning attention / the
 * `g_gamma` path of ejkernel's `recurrent`).
 *
 * The operation (ejkernel docs, kernels/_xla/recurrent/_interface, `recurrent`
 * docstring, its state-update formula, with the per-head `g_gamma` decay of
 * its Args and of the kernels/_triton/lightning_attn/_interface page), per
 * sequence n and head h, with gamma = exp(g_gamma[h]) and tokens t in
 * processing order:
 *
 *     S_t = gamma * S_{t-1} + k_t^T v_t          (S: d x e, fp32)
 *     o_t = (scale * q_t) S_t                    (an e-vector)
 *
 * S_0 = initial_state (or zeros); final_state = S after the last processed
 * token.  With reverse != 0 the tokens of every sequence are processed from
 * last to first (o is still written at each token's own position).  With
 * cu_seqlens the batch is one packed row of sequences [cu[n], cu[n+1]), each
 * with its own state.  The library evaluates this in the chunked form of
 * Lightning Attention-2 (OpenNLPLab/lightning-attention README): per chunk an
 * intra-chunk decay-masked (Q K^T) V product plus an inter-chunk carried state.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never frees, keeps or allocates them.  cu_seqlens_host is a HOST pointer.
 *   - Token tensors are indexed [batch, token, head, channel] through element
 *     strides (batch, token, head); the channel dimension must be contiguous.
 *     q, k, dq, dk share qk_strides; v, o, do, dv share v_strides (with
 *     grouped key/value heads k, dk and v, dv have their own, see la_dims).
 *     Both the token-major layout [B,T,H,X] (ejkernel) and the head-major
 *     layout [B,H,T,X] (Lightning-2's (b, h, n, d)) are expressible.  Outputs
 *     must not overlap inputs or each other, with one exception: the forward
 *     calls' final_state may be the very buffer passed as initial_state (an
 *     in-place state update, as in decoding).
 *   - State tensors (initial_state, final_state, d_final_state,
 *     d_initial_state) are dense fp32 [N, H, D, E], N = B, or num_seqs when
 *     cu_seqlens is given.
 *   - Workspace (optional, 256-byte aligned device memory, passed as
 *     (workspace, workspace_bytes)); la_workspace_size_for gives the bytes
 *     that enable everything below.  It holds, when it is large enough:
 *       * the longest-first schedule of packed sequences (la_workspace_size(N)
 *         bytes at its start);
 *       * the sequence split: when the (sequence, head) pairs would occupy at
 *         most half of the GPU's SMs, long sequences are cut into segments of
 *         whole 128-token chunks that run in parallel, in two passes around a
 *         scan of one fp32 state per (segment, head).  This needs every token
 *         tensor's batch stride to equal T times its token stride (or B = 1);
 *       * with grouped key/value heads, the backward's per-query-head dk and
 *         dv contributions (required there, see la_bwd).
 *     All of it is written there on `stream`, so the workspace must not be
 *     shared with another call in flight on another stream.  NULL (or too
 *     small a workspace) runs without the schedule and the split.  The
 *     schedule never changes results; the split changes the summation order
 *     of the states (fp32 rounding only).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) of the current device.  No entry point
 *     allocates device memory or synchronizes, except: when cu_seqlens is given
 *     without cu_seqlens_host the library copies cu_seqlens to the host and
 *     waits for that copy; and la_get_device_error synchronizes `stream`.
 *     Calls that use a workspace (or la_fwd_noalloc's array) for the
 *     schedule or the split -- packed calls, and sequences the split cuts --
 *     also copy host data into it during the call: the longest-first
 *     schedule and the sequence split's segment table are built on the host
 *     and sent with cudaMemcpyAsync from pageable memory.
 *   - CUDA graphs: those calls (and packed calls without cu_seqlens_host)
 *     cannot be captured.  Every other call -- no cu_seqlens, and no split
 *     (la_set_sequence_split(0, 0), or sizes it leaves whole) -- enqueues
 *     only kernels and memsets on `stream` (tensor maps travel as kernel
 *     parameters) and can be captured once and replayed with new contents
 *     in the same buffers; replays equal eager calls bit for bit.
 *     The tensor-core kernels are launched as programmatic dependents of
 *     the stream's previous kernel: they may start their set-up while it
 *     drains, but read and write global memory only after it has completed,
 *     so stream order holds as for any launch.
 *   - Every argument is validated before anything is enqueued.  A failed
 *     validation returns LA_ERR_INVALID_ARG or LA_ERR_UNSUPPORTED, launches
 *     nothing and leaves every output untouched; la_last_error() describes it.
 *   - Every output is fully overwritten (no accumulation into outputs).
 */
#ifndef LA_GB300_H
#define LA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum la_status {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,   /* bad pointer, size, stride or cu_seqlens        */
    LA_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels handle  */
    LA_ERR_CUDA = 3,          /* a CUDA runtime call or a launch failed         */
    LA_ERR_TIMEOUT = 4,       /* a bounded on-device wait ran out (device word) */
    LA_ERR_BOUNDS = 5         /* an index check of the bounds-checking build
                                 failed (device word; never in the normal build) */
} la_status;

/* Element type of the token tensors q, k, v, o, do, dq, dk, dv.  g_gamma and
 * every state tensor are always fp32. */
typedef enum la_dtype {
    LA_DTYPE_BF16 = 0,
    LA_DTYPE_F32 = 1
} la_dtype;

/* Problem sizes and layout.
 *   batch      B  >= 0; must be 1 when cu_seqlens is given (lightning_attn
 *                 docstring, Raises: batch must be 1 with cu_seqlens)
 *   seq_len    T  >= 0 tokens per batch row (total tokens when packed)
 *   heads      H  1..65535 query heads
 *   dim_qk     D  query/key channels, 1..256
 *   dim_v      E  value channels, 1..256
 *   num_seqs   N  number of packed sequences when cu_seqlens is given
 *                 (ignored otherwise; N = B)
 *   qk_strides element strides (batch, token, head) of q, dq (and of k, dk
 *                 when kv_heads is 0)
 *   v_strides  element strides (batch, token, head) of o, do (and of v, dv
 *                 when kv_heads is 0)
 *   kv_heads   0: keys and values have H heads (lightning_attn's Args give
 *                 them the queries' shape).  Else H_kv, a divisor of H: grouped
 *                 key/value heads (the num_kv_heads axis of ejkernel
 *                 `recurrent`'s key and value), query head h reading key and
 *                 value head h / (H / H_kv).  Decay, states and their
 *                 gradients stay per query head; dk and dv of a shared head
 *                 sum its query heads' contributions.
 *   reserved   must be 0
 *   k_strides  element strides of k, dk when kv_heads > 0 (k, dk: [B,T,H_kv,D])
 *   kv_v_strides element strides of v, dv when kv_heads > 0 ([B,T,H_kv,E]) */
typedef struct la_dims {
    int32_t batch;
    int32_t seq_len;
    int32_t heads;
    int32_t dim_qk;
    int32_t dim_v;
    int32_t num_seqs;
    int64_t qk_strides[3];
    int64_t v_strides[3];
    int32_t kv_heads;
    int32_t reserved;
    int64_t k_strides[3];
    int64_t kv_v_strides[3];
} la_dims;

/* Forward pass (ejkernel `recurrent` / `lightning_attn`: returns the output
 * and the final hidden state).
 *   q               [B,T,H,D] of `dtype`
 *   k               [B,T,H,D] of `dtype` ([B,T,H_kv,D] with kv_heads)
 *   v               [B,T,H,E] of `dtype` ([B,T,H_kv,E] with kv_heads)
 *   g_gamma         [H] fp32 log-decay per head (gamma = exp(g_gamma[h]);
 *                   values > 0 are accepted but grow the state)
 *   scale           multiplies q only (the pages' softmax_scale; callers apply
 *                   the default 1/sqrt(D) themselves)
 *   initial_state   [N,H,D,E] fp32, or NULL for zeros
 *   reverse         0: t = 0..L-1 per sequence; 1: t = L-1..0
 *   cu_seqlens      device int32 [N+1] with cu[0] = 0, non-decreasing,
 *                   cu[N] = T; or NULL for B independent rows of length T
 *   cu_seqlens_host host copy of cu_seqlens, or NULL (then copied, see above)
 *   o               [B,T,H,E] of `dtype` (output, v_strides)
 *   final_state     [N,H,D,E] fp32 output, or NULL to skip it
 *   workspace       device scratch for the schedule and the sequence split,
 *                   or NULL (above) */
la_status la_fwd(const la_dims *dims, int32_t dtype,
                 const void *q, const void *k, const void *v,
                 const float *g_gamma, float scale,
                 const float *initial_state, int32_t reverse,
                 const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                 void *o, float *final_state,
                 void *workspace, size_t workspace_bytes, void *stream);

/* Backward pass: gradients of  sum(o * d_o) + sum(final_state * d_final_state)
 * (the custom VJP of ejkernel `recurrent`, `_recurrent_bwd`, with upstream
 * grads (do, dfinal_state); g_gamma, scale, reverse and cu_seqlens are not
 * differentiated, as on that page).  Nothing from the forward pass is needed:
 * the states are recomputed.  Packed sequences are supported (the pages raise
 * NotImplementedError there; here each sequence gets its own gradient).
 *   q, k, v, g_gamma, scale, initial_state, reverse, cu_seqlens: as la_fwd
 *   d_o             [B,T,H,E] of `dtype` (v_strides)
 *   d_final_state   [N,H,D,E] fp32, or NULL for zeros
 *   dq              [B,T,H,D] of `dtype` output (qk_strides)
 *   dk, dv          [B,T,H,D], [B,T,H,E] of `dtype` outputs (qk_strides,
 *                   v_strides); with kv_heads: [B,T,H_kv,D], [B,T,H_kv,E]
 *                   (k_strides, kv_v_strides), each the fp32 sum of its
 *                   group's per-query-head contributions, which pass through
 *                   the workspace rounded to `dtype`.  Then the workspace is
 *                   required: la_workspace_size_for gives its size, and too
 *                   small a workspace is LA_ERR_INVALID_ARG.
 *   d_initial_state [N,H,D,E] fp32 output, or NULL to skip it
 * la_bwd is exactly la_bwd_dq followed by la_bwd_dkdv on the same stream.  */
la_status la_bwd(const la_dims *dims, int32_t dtype,
                 const void *q, const void *k, const void *v, const void *d_o,
                 const float *g_gamma, float scale,
                 const float *initial_state, const float *d_final_state,
                 int32_t reverse,
                 const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                 void *dq, void *dk, void *dv, float *d_initial_state,
                 void *workspace, size_t workspace_bytes, void *stream);

/* The first half of la_bwd: dq only (a sweep in processing order that
 * recomputes the states; q and d_final_state are not read).  Arguments as
 * la_bwd; q may be NULL. */
la_status la_bwd_dq(const la_dims *dims, int32_t dtype,
                    const void *q, const void *k, const void *v, const void *d_o,
                    const float *g_gamma, float scale,
                    const float *initial_state, int32_t reverse,
                    const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                    void *dq, void *workspace, size_t workspace_bytes, void *stream);

/* The second half of la_bwd: dk, dv and d_initial_state (a sweep against
 * the processing order carrying dL/dS; initial_state is not read).
 * Arguments as la_bwd; d_initial_state may be NULL. */
la_status la_bwd_dkdv(const la_dims *dims, int32_t dtype,
                      const void *q, const void *k, const void *v, const void *d_o,
                      const float *g_gamma, float scale,
                      const float *d_final_state, int32_t reverse,
                      const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                      void *dk, void *dv, float *d_initial_state,
                      void *workspace, size_t workspace_bytes, void *stream);

/* The forward pass without any device workspace, for callers that cannot
 * allocate device memory where they call it (their device memory belongs to
 * another allocator that hands out no scratch, or a cudaMalloc there would
 * synchronize the device).  The pages have no counterpart: this is an
 * interface for such callers.  Arguments, results and validation are those of
 * la_fwd; the packed-sequence schedule lives in an array compiled into the
 * library (LA_FWD_NOALLOC_MAX_SEQS int32 per GPU, held until exit) instead of
 * a caller workspace.  More than LA_FWD_NOALLOC_MAX_SEQS packed sequences is
 * rejected with LA_ERR_UNSUPPORTED before anything is enqueued.  The array
 * only ever holds the schedule (never the sequence split's states, so packed
 * calls here always run unsplit).  The first packed call on a device looks the
 * array's device address up (cudaGetSymbolAddress) with that device current
 * and keeps it for the rest of the process.  Packed calls copy the schedule
 * from pageable host memory into the array, so they cannot be captured in a
 * CUDA graph (dense calls never touch the array and capture as la_fwd
 * does).  The kept address does not survive a
 * cudaDeviceReset: do not use this entry point on a device after resetting
 * it.  Every call on a device shares the one array, which keeps the previous
 * call's schedule; each call overwrites the entries it uses.  Calls whose
 * work overlaps on the GPU (different streams, or host threads without
 * ordering between them) race on it and must be serialized by the caller. */
#define LA_FWD_NOALLOC_MAX_SEQS 16384
la_status la_fwd_noalloc(const la_dims *dims, int32_t dtype,
                         const void *q, const void *k, const void *v,
                         const float *g_gamma, float scale,
                         const float *initial_state, int32_t reverse,
                         const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                         void *o, float *final_state, void *stream);

/* Bytes of device workspace for the longest-first schedule of num_seqs packed
 * sequences (0 when num_seqs < 1).  Pure host function. */
size_t la_workspace_size(int32_t num_seqs);

/* Bytes of device workspace with which la_fwd, la_bwd, la_bwd_dq and
 * la_bwd_dkdv use the schedule and, when it applies, the sequence split for
 * these sizes (see Conventions, Workspace).  cu_seqlens_host: host copy of
 * cu_seqlens (num_seqs + 1 entries) for packed sequences, else NULL.  The
 * answer depends on the current device's SM count and on
 * la_set_sequence_split; 0 for invalid sizes.  Host function (reads one
 * device attribute, once per device). */
size_t la_workspace_size_for(const la_dims *dims, int32_t dtype, const int32_t *cu_seqlens_host);

/* Sequence split control, process-wide: mode 1 (default) splits when it
 * applies, 0 never.  min_segment_tokens 0 (default) chooses by head width:
 * segments of at least 256 tokens at D <= 64, at least 4 segments of at
 * least 1024 tokens at D <= 128, no split above; a value >= 128 is the
 * shortest segment planned, at any width.  The method's pages have no
 * counterpart: the split is a way of scheduling the same arithmetic.
 * LA_ERR_INVALID_ARG for other values. */
la_status la_set_sequence_split(int32_t mode, int32_t min_segment_tokens);

/* Gated form (GLA): ejkernel `recurrent` with its gate g (the GLA page's
 * `recurrent_gla` passes it on), a log-decay per key channel added to the
 * head's g_gamma:
 *     S_t[a, :] = exp(g_gamma[h] + g_t[a]) * S_{t-1}[a, :] + k_t[a] v_t,
 *     o_t = scale * q_t^T S_t
 * (the reading of the pages' "GLA-style gating"; the gate of token t decays
 * the state token t is added to, in either direction).
 *   g          [B,T,H,D] fp32 gate, channel-contiguous, element strides
 *              g_strides[3] = (batch, token, head)
 *   g_gamma    [H] fp32, required (zeros for no head decay)
 *   workspace  256-byte aligned device scratch of at least
 *              la_gla_fwd_workspace_size bytes, or NULL
 *   operands_written  host int32, or NULL: set to 1 when the call ran the
 *              chunked form, leaving its operands in the workspace (which
 *              la_gla_bwd can then reuse), else 0
 *   everything else as la_fwd, grouped key/value heads included: k and v
 *              with kv_heads heads (k_strides, kv_v_strides), query head h
 *              reading key/value head h / (H / kv_heads); the gate, the
 *              state and o are the query head's (ejkernel `recurrent`: key
 *              and value with num_kv_heads heads, g with num_heads).
 * With the workspace, bf16 calls with D = 128, E in {64, 128} and sequences
 * longer than 16 tokens run the chunked form on the tensor cores: per chunk
 * of 128 tokens the gate's running sums b are split around a reference r
 * (the middle of their range, raised to -72 if lower), q and k are rescaled
 * by exp(b - r) and exp(r - b) into the workspace, and the chunked sweep runs
 * on them.  Every (sequence, head) with a chunk where some |b - r| or r
 * exceeds 72 (gates stronger than the factors' bf16 range allows: a chunk's
 * total log-decay below about -144) runs the token-by-token kernels instead,
 * decided on the device.  All other calls, and calls without the
 * workspace, run the token-by-token kernels.  Not differentiated: g_gamma,
 * scale, reverse, cu_seqlens.
 * Sequence split (as la_fwd's, la_set_sequence_split): with few (sequence,
 * head) pairs and a gate whose strides allow the one-row token view, the
 * chunked form runs on segments of whole chunks in two passes around a
 * scan whose decay is per key channel, exp of the segment's summed
 * log-decays (len * g_gamma[h] + the gates), formed from the pre-pass's
 * chunk totals.  la_gla_fwd_workspace_size covers it.  Its operands are
 * laid out per segment: operands_written stays 0. */
la_status la_gla_fwd(const la_dims *dims, int32_t dtype,
                     const void *q, const void *k, const void *v,
                     const float *g, const int64_t *g_strides,
                     const float *g_gamma, float scale,
                     const float *initial_state, int32_t reverse,
                     const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                     void *o, float *final_state, void *workspace,
                     size_t workspace_bytes, int32_t *operands_written,
                     void *stream);

/* Bytes of workspace with which la_gla_fwd runs the chunked form for these
 * sizes (q~, k~ as bf16 [rows][T][H][D] each, two fp32 vectors per chunk and
 * (sequence, head), one flag per (sequence, head)); 0 when the chunked form
 * does not apply.  cu_seqlens_host as la_workspace_size_for.  Host only. */
size_t la_gla_fwd_workspace_size(const la_dims *dims, int32_t dtype,
                                 const int32_t *cu_seqlens_host);

/* Backward of la_gla_fwd: dq, dk, dv, d_initial_state as la_bwd, and
 * dg [B,T,H,D] fp32 (g_strides), the gradient of the gate:
 *     dg_w = sum over t at or after w (processing order) of
 *            q_t dq_t - k_t dk_t (+ sum_e F dF at the last token),
 * F the final state and dF = d_final_state.  Needs a 256-byte aligned device
 * workspace (LA_ERR_INVALID_ARG otherwise); la_gla_workspace_size gives the
 * bytes with which bf16 calls with D = 128, E in {64, 128}, sequences
 * longer than 16 tokens and 16-byte aligned token rows run the chunked form on the tensor
 * cores: the forward's rescaled q~, k~ (see la_gla_fwd), three sweeps on
 * them -- forward-type (do, v, k~) giving dq~ = dq exp(r - b), backward-
 * type (k~, q~, do) giving dv, backward-type (v, do, q~) giving dk~ =
 * dk exp(b - r), dq~ and dk~ in fp32 -- and a pass that rescales dq~, dk~
 * into dq, dk and forms dg, each term as q~ dq~ - k~ dk~ from the rounded
 * operands and their own gradients.  Pairs out of range, smaller workspaces
 * (down to the token-by-token part: the final state, dg's block sums and,
 * for bf16, dq and dk in fp32) and other shapes run the token-by-token
 * kernels.  dg never takes bf16-rounded gradients: rounding each of its T
 * terms would add errors that grow with T while dg does not.
 * Grouped key/value heads: dq and dg are per query head as without
 * grouping; dk and dv are the sums over each group's query heads, formed
 * from every query head's part (dk's in fp32, dv's in the token dtype, both
 * in the workspace) in fp32 and written in the token dtype.
 * Sequence split (as la_gla_fwd's; a workspace of la_gla_workspace_size(...,
 * 0) bytes): the operands are computed per segment (fwd_workspace is not
 * used), dq~ and dv run in two passes around scans with per-channel decays
 * (the latter giving d_initial_state), dk~ from the scanned gradients, and
 * dg per segment plus each segment's offset: the sum of the terms of the
 * segments processed after it and the final state's term.
 *   fwd_workspace  the workspace of a la_gla_fwd call on the same q, k, g,
 *              g_gamma, reverse and cu_seqlens that reported operands_written
 *              = 1, untouched since; or NULL.  The backward then uses the
 *              operands in it instead of computing them again (the main
 *              workspace needs only the token-by-token part) and uses the
 *              rest of it as scratch: it serves one backward. */
la_status la_gla_bwd(const la_dims *dims, int32_t dtype,
                     const void *q, const void *k, const void *v, const void *d_o,
                     const float *g, const int64_t *g_strides,
                     const float *g_gamma, float scale,
                     const float *initial_state, const float *d_final_state,
                     int32_t reverse,
                     const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                     void *dq, void *dk, void *dv, float *dg, float *d_initial_state,
                     void *workspace, size_t workspace_bytes,
                     void *fwd_workspace, size_t fwd_workspace_bytes, void *stream);

/* Workspace bytes of la_gla_bwd for these sizes (0 for invalid sizes): with
 * with_forward_operands = 0, enough to run the chunked form on its own where
 * it applies; nonzero, the part needed when the forward's operands are passed
 * as fwd_workspace.  That part: the final state, dg's block sums, dq and dk
 * in fp32 ([rows][T][H][D] each; for bf16 tokens, and for fp32 tokens when
 * kv_heads is set) and, with kv_heads < H, the query heads' parts of dv
 * ([rows][T][H][E], token dtype).  cu_seqlens_host: host copy of cu_seqlens for packed
 * sequences, else NULL.  Pure host function. */
size_t la_gla_workspace_size(const la_dims *dims, int32_t dtype,
                             const int32_t *cu_seqlens_host, int32_t with_forward_operands);

/* Reads and clears the device-side error words that bounded on-device waits
 * set when they run out (LA_ERR_TIMEOUT), after synchronizing `stream`.
 * Returns LA_OK when no wait ran out, LA_ERR_TIMEOUT when one did, or
 * LA_ERR_CUDA when the synchronization itself failed.  The words are shared
 * by every stream of the current device.
 * A library built with LA_CHECK_BOUNDS defined (build.py --checked) also
 * checks the tensor-core kernels' shared-memory, TMEM, descriptor, table and
 * global indices; a failed check skips the access and records the first
 * failing site here, reported as LA_ERR_BOUNDS with the site number in
 * la_last_error(). */
la_status la_get_device_error(void *stream);

/* Diagnostic, for testing error reporting: with on != 0, the next launch of
 * a kernel with internal hand-offs (the tensor-core sweeps, the streamed
 * decode kernel) made from this host thread withholds one of them -- between
 * its warps, or the copy of a state block -- so that a bounded on-device wait
 * runs out
 * (after about 2 s); the kernel then stops, frees what it holds and returns,
 * its outputs are undefined, and la_get_device_error reports LA_ERR_TIMEOUT.
 * The switch resets itself after that launch and is off by default. */
la_status la_debug_withhold_next_handoff(int32_t on);

/* Diagnostic, for testing the sequence split's planning without a device:
 * the number of segments la_fwd / la_bwd would cut these sizes into on a GPU
 * with `sms` multiprocessors under the current la_set_sequence_split
 * settings; 0 when they would run unsplit, -1 for invalid sizes.
 * cu_seqlens_host as la_workspace_size_for.  Pure host function. */
int32_t la_debug_split_segments(const la_dims *dims, int32_t dtype,
                                const int32_t *cu_seqlens_host, int32_t sms);

/* How this copy of the library was built: LA_BUILD_BOUNDS_CHECKED set when
 * the tensor-core kernels' index checks are compiled in (build.py --checked,
 * liblagb300_checked.so; see la_get_device_error).  Pure host function. */
#define LA_BUILD_BOUNDS_CHECKED 1
int32_t la_build_flags(void);

/* Static description of a status code (never NULL). */
const char *la_strerror(int32_t status);

/* Human-readable detail of the last failed call on this host thread (empty
 * string when none).  Valid until the next call on the same thread. */
const char *la_last_error(void);

/* Which kernel family la_fwd would launch for these sizes and dtype, assuming
 * 16-byte aligned base pointers: 2 = the short-call kernels (every sequence
 * at most 16 tokens long: decoding a few tokens against a carried state;
 * token by token, or for 5 to 16 tokens as one chunk -- on the tensor cores
 * for bf16 with D = 128 and E a multiple of 16),
 * 1 = tensor-core (tcgen05) chunked kernels, 0 = CUDA-core chunked kernels,
 * -1 = invalid or unsupported.  The sequence length is dims->seq_len; with
 * cu_seqlens the longest packed sequence decides, which this function does
 * not see.  Pure host function; launches nothing. */
int32_t la_kernel_family(const la_dims *dims, int32_t dtype);

/* Number of kernels this library has enqueued since it was loaded (all
 * devices, all host threads).  Pure host counter; lets a caller count the
 * launches inside a timed region. */
uint64_t la_launch_count(void);

/* ABI version, (major << 16) | minor. */
int32_t la_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LA_GB300_H */

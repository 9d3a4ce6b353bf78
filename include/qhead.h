/*
 * qhead.h -- C ABI of the GB300 fused quantized LM-head ("Flash Cut-Cross-
 * Entropy" over a frozen 4/8-bit affine-quantized head).
 *
 * The operation is the one described on the page "mlx-bun 0.0.4 -> 0.0.6"
 * (src/train/flash-cce.ts): for hidden states h[M,H] and a quantized head W
 * (FlashCceHead: packed uint32 codes, per-group scales and biases, bits,
 * group size, optional final-logit soft cap)
 *
 *     w[v,d]   = scale[v, d/group] * q[v,d] + bias[v, d/group]
 *     raw[m,v] = sum_d h[m,d] * w[v,d]
 *     z[m,v]   = cap * tanh(raw[m,v] / cap)      (z = raw when cap <= 0)
 *     lse[m]   = log sum_v exp(z[m,v])
 *     logp[m]  = z[m, target[m]] - lse[m]
 *
 * and, for the frozen head, the gradient of sum_m dlogp[m] * logp[m]:
 *
 *     dh[m,:]  = sum_v dlogp[m] * (1[v == target[m]] - exp(z[m,v] - lse[m]))
 *                              * sech2[m,v] * w[v,:]
 *     sech2    = 1 - tanh^2(raw / cap)           (1 when the cap is off)
 *
 * The vocab loop runs inside the kernels: neither the [M,V] logits nor a
 * dequantized [V,H] head is ever written to device memory.  The same call
 * with targets == NULL is the speculative-decode verify step of the page
 * "mlx-bun 0.0.8 -> 0.0.10" (src/spec/generate.ts, picksBatched): one head
 * pass over the gamma+1 window, then the argmax of every position (argmax of
 * the raw logits; the soft cap and the lse shift are monotone, so it is also
 * the argmax of z and of logp).
 *
 * Conventions shared by every entry point
 *   - All array arguments are DEVICE pointers unless stated otherwise.
 *   - The caller owns and allocates every input, output and workspace; the
 *     library allocates nothing and keeps no per-call state.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).  Nothing synchronizes.
 *   - Return value: QHEAD_OK or an error code; on error nothing was launched
 *     (argument errors) or a launch failed (QHEAD_ECUDA).  A message for the
 *     calling thread is available from qhead_last_error().
 *   - There is no fallback path: unsupported shapes are rejected.
 *   - Kernel time limits: every wait inside a pipelined kernel gives up after
 *     2 s (only a defect or a stalled device makes one that long).  The kernel
 *     then stops waiting, lets the copies and tensor-core operations it has
 *     issued complete, runs to its end and records the failure; qhead_fwd then
 *     writes logp = NaN, lse = NaN and argmax = -1 for every active row, and
 *     qhead_bwd writes NaN to every active row of dh (inactive rows keep their
 *     defined values).  The return value cannot report this, because the call
 *     returns before its kernels run.
 */
#ifndef QHEAD_H
#define QHEAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define QHEAD_OK 0
#define QHEAD_EINVAL 1        /* null required pointer, misalignment, bad size, small workspace */
#define QHEAD_EUNSUPPORTED 2  /* bits / group / H / sb_dtype the library does not implement */
#define QHEAD_ECUDA 3         /* a CUDA launch or runtime call failed */

/* Element type of scales and biases. */
#define QHEAD_SB_F16 0
#define QHEAD_SB_BF16 1
#define QHEAD_SB_F32 2

/*
 * The frozen quantized head (FlashCceHead on the page "mlx-bun 0.0.4 ->
 * 0.0.6", src/train/flash-cce.ts).
 *   wq       device, uint32 [V, H*bits/32], row-major.  Word j of row v holds
 *            elements j*(32/bits) + k, k = 0 .. 32/bits - 1, element k in bits
 *            bits*k .. bits*k + bits - 1 (least-significant field first).
 *            16-byte aligned.
 *   scales   device, [V, H/group] row-major, of type sb_dtype.  16-byte aligned.
 *   biases   device, [V, H/group] row-major, of type sb_dtype.  16-byte aligned.
 *   V        vocab rows, 1 <= V < 2^31.
 *   H        hidden size: a multiple of 128, 128 <= H <= 8192.
 *   bits     4 or 8.
 *   group    64 (the only group size implemented).
 *   sb_dtype QHEAD_SB_F16, QHEAD_SB_BF16 or QHEAD_SB_F32: the element type of
 *            scales and biases (the page casts any float type to f32).  The
 *            exact fp32 parts of the path (the target logit, the argmax
 *            recheck, the backward's one-hot term) widen the given values
 *            exactly.  The tensor-core and weight-streaming kernels take fp16
 *            operands: for a bf16 or fp32 head each call first rounds scales
 *            and biases to fp16 (nearest) into its workspace -- exact for bf16
 *            values of magnitude in [2^-17, 65504] or zero, one rounding for
 *            fp32 -- which costs a pass over 2 * V * H/64 elements and
 *            2 * 2 * V * H/64 bytes of workspace.  Magnitudes above 65504
 *            become infinite there (results NaN).
 *   softcap  final-logit soft cap; <= 0 turns it off.
 */
typedef struct qhead_head {
    const uint32_t* wq;
    const void* scales;
    const void* biases;
    int64_t V;
    int32_t H;
    int32_t bits;
    int32_t group;
    int32_t sb_dtype;
    float softcap;
} qhead_head;

/*
 * Workspace bytes qhead_fwd / qhead_bwd need for M rows with this head on the
 * current device (the plan depends on M, the head's shape and the SM count).
 * Returns 0 for M == 0 and (size_t)-1 if the arguments are invalid (see
 * qhead_last_error()).  Host-only; launches nothing.
 */
size_t qhead_fwd_workspace(const qhead_head* head, int64_t M);
size_t qhead_bwd_workspace(const qhead_head* head, int64_t M);

/*
 * Forward: logp, lse and argmax for every row of h.
 * Definition: flashCceForward on the page "mlx-bun 0.0.4 -> 0.0.6"
 * (src/train/flash-cce.ts, per-vocab-block partials merged into lse and
 * logp = target logit - lse); argmax as in picksBatched on the page
 * "mlx-bun 0.0.8 -> 0.0.10" (src/spec/generate.ts).
 *   h         device, bf16 [M, H] row-major, 16-byte aligned.  Every |h|
 *             must be below 65504: the kernels stage h as fp16 operands, so a
 *             larger magnitude becomes infinite there and the row's lse, logp
 *             (and dh) come out inf or NaN; no error is returned.
 *   M         rows, >= 0 (M == 0 returns QHEAD_OK and launches nothing).
 *   targets   device, int32 [M], or NULL (verify: no logp).  Each active
 *             row's target must lie in [0, V); a row whose target does not
 *             gets logp = NaN (no out-of-range read happens).
 *   mask      device, uint8 [M], or NULL (all rows active).  mask[m] != 0
 *             means row m is active; inactive rows are skipped and written as
 *             logp = 0, lse = 0, argmax = -1.
 *   logp      device, float [M], or NULL.  Requires targets.
 *   lse       device, float [M], or NULL.
 *   argmax    device, int32 [M], or NULL.  The lowest vocab index attaining
 *             the row's maximum logit (ties within float rounding of each
 *             other may resolve to either index).
 *   workspace device, >= qhead_fwd_workspace(head, M) bytes, 256-byte
 *             aligned; contents on entry are ignored.
 * Outputs may not alias inputs or each other.
 */
int qhead_fwd(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
              const uint8_t* mask, float* logp, float* lse, int32_t* argmax, void* workspace,
              size_t workspace_bytes, void* stream);

/*
 * Speculative-decode verify with the accept step fused on the device.
 * Definition: page "mlx-bun 0.0.8 -> 0.0.10" (src/spec/generate.ts): one head
 * pass over the gamma + 1 window, the argmax of every position (picksBatched),
 * then the longest prefix of the draft that the argmax reproduces.
 *   h         device, bf16 [B * W, H]: B windows of W = gamma + 1 rows each.
 *   B, W      B >= 0 windows (B == 0 returns QHEAD_OK), W in [1, 2^20].
 *   draft     device, int32 [B, W - 1]: the drafted tokens; required if W > 1.
 *   mask      as for qhead_fwd ([B * W] or NULL); a masked row's argmax is -1,
 *             so a draft token never matches it.
 *   lse       device, float [B * W], or NULL.
 *   argmax    device, int32 [B * W] (required): as for qhead_fwd.
 *   n_accept  device, int32 [B] (required): for window b, the first k < W - 1
 *             with draft[b, k] != argmax[b, k], or W - 1 if every draft token
 *             is accepted.
 *   next_token device, int32 [B], or NULL: argmax[b, n_accept[b]], the token
 *             the target model emits after the accepted prefix.
 *   workspace as for qhead_fwd with M = B * W (qhead_fwd_workspace(head, B * W)).
 * Outputs may not alias inputs or each other.
 */
int qhead_verify(const qhead_head* head, const void* h, int64_t B, int64_t W,
                 const int32_t* draft, const uint8_t* mask, float* lse, int32_t* argmax,
                 int32_t* n_accept, int32_t* next_token, void* workspace, size_t workspace_bytes,
                 void* stream);

/*
 * Backward of the frozen head: dh = d(sum_m dlogp[m] * logp[m]) / dh.
 * Definition: flashCceBackward on the page "mlx-bun 0.0.4 -> 0.0.6"
 * (src/train/flash-cce.ts: logits recomputed per vocab tile, coefficient
 * dlogp * (onehot - softmax) * sech2, dh accumulated over all vocab blocks),
 * with the forward's lse reused.
 *   h, M, targets, mask  as for qhead_fwd (including |h| < 65504); targets
 *             is required.
 *   lse       device, float [M]: the lse qhead_fwd returned for the same
 *             h / head / mask.
 *   dlogp     device, float [M]: the cotangent of each row's logp.
 *   dh        device, float [M, H] row-major, 16-byte aligned.  Every row is
 *             written; inactive rows are exactly 0.
 *   workspace device, >= qhead_bwd_workspace(head, M) bytes, 256-byte aligned.
 * The result is deterministic: fixed-order reductions; where vocab chunks add
 * into a partial buffer, each element receives one addition per chunk, in
 * chunk order.
 */
int qhead_bwd(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
              const uint8_t* mask, const float* lse, const float* dlogp, float* dh,
              void* workspace, size_t workspace_bytes, void* stream);

/*
 * The blockMax early exit (an approximate backward; page "mlx-bun 0.0.4 ->
 * 0.0.6", src/train/flash-cce.ts: the forward hands per-block logit maxima to
 * the backward, which skips a (token block, vocab block) program when every
 * token has exp(blockMax - lse) < eps and no target lies in the block).
 *
 * qhead_fwd_blockmax: qhead_fwd plus
 *   block_max device, float [M, ceil(V / 256)] row-major, 4-byte aligned: the
 *             maximum capped logit z of each active row over each 256-row
 *             vocab tile (rows with mask 0 are not written).
 *   workspace >= qhead_fwd_blockmax_workspace(head, M) bytes (every M takes
 *             the tensor-core path).
 *
 * qhead_bwd_blockskip: qhead_bwd, except that the (128 consecutive active
 * rows, 256-row vocab tile) blocks in which every row has
 * exp(block_max - lse) < eps and no row's target lies are left out of both
 * backward phases (their coefficients count as 0): dh then differs from the
 * exact one by at most |dlogp| * eps * sum_v |w_v| per row, and the skipped
 * blocks cost nothing.
 *   block_max the forward's block_max for the same h / head / mask.
 *   eps       in [0, 1]; 0 skips nothing (the exact backward).
 *   workspace >= qhead_bwd_blockskip_workspace(head, M) bytes.
 */
size_t qhead_fwd_blockmax_workspace(const qhead_head* head, int64_t M);
int qhead_fwd_blockmax(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
                       const uint8_t* mask, float* logp, float* lse, int32_t* argmax,
                       float* block_max, void* workspace, size_t workspace_bytes, void* stream);
size_t qhead_bwd_blockskip_workspace(const qhead_head* head, int64_t M);
int qhead_bwd_blockskip(const qhead_head* head, const void* h, int64_t M,
                        const int32_t* targets, const uint8_t* mask, const float* lse,
                        const float* dlogp, const float* block_max, float eps, float* dh,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * The coefficient filter (an approximate backward; page "mlx-bun 0.0.4 ->
 * 0.0.6", src/train/flash-cce.ts: the backward's near-zero coefficient filter
 * skips the dh contraction of a coefficient tile whose largest |coeff| is
 * below eps, since the softmax mass concentrates on a few vocab rows).
 *
 * qhead_bwd_filter: qhead_bwd, except that the blocks of 32 consecutive
 * active rows x 32 vocab rows (rows 32k .. 32k + 31) in which no row's target
 * lies and every softmax term |dlogp[m]| * softmax[m, v] * sech2[m, v] is
 * below eps are cold: their coefficients count as 0, and a dh step whose
 * blocks are all cold is skipped.  Blocks holding a target always stay warm
 * (the one-hot term is added whole).  dh then differs from the exact one by at
 * most eps * sum_v |w_v| per row.  The decision is taken in fp32 on the
 * kernel's logits, so a block whose largest term lies within a small relative
 * distance of eps may go either way.
 *   eps       >= 0 (+inf allowed); 0 makes nothing cold (the exact backward).
 *             NaN or a negative value is rejected (QHEAD_EINVAL).
 *   cold      device, uint8 [ceil(M / 32), ceil(V / 32)] row-major, or NULL:
 *             1 where the block of active rows 32j .. 32j + 31 (ascending
 *             order of the active rows) and vocab rows 32k .. 32k + 31 is
 *             cold, else 0; row blocks past the active rows are 1.
 *   workspace >= qhead_bwd_filter_workspace(head, M) bytes (every M takes
 *             the tensor-core path).
 */
size_t qhead_bwd_filter_workspace(const qhead_head* head, int64_t M);
int qhead_bwd_filter(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
                     const uint8_t* mask, const float* lse, const float* dlogp, float eps,
                     float* dh, uint8_t* cold, void* workspace, size_t workspace_bytes,
                     void* stream);

/*
 * Workspace bytes qhead_bwd_dw needs for M rows with this head ((size_t)-1 on
 * invalid arguments).
 */
size_t qhead_bwd_dw_workspace(const qhead_head* head, int64_t M);

/*
 * Backward with the head gradient: dw = d(sum_m dlogp[m] * logp[m]) / dW with
 * respect to the dequantized head W[v, d] = scale * q + bias, and optionally
 * dh as qhead_bwd computes it, from one pass of logit recomputation.
 * Definition: the classifier gradient (dC) of the Apple CCE reference that
 * the page "mlx-bun 0.0.4 -> 0.0.6" (src/train/flash-cce.ts) cites; the pages
 * compute none because their head is frozen:
 *     dw[v, :] = sum_m dlogp[m] * (1[v == target_m] - softmax[m, v]) * sech2[m, v] * h[m, :].
 * From it, d/dscale[v, g] = sum_{d in g} q[v, d] * dw[v, d] and
 * d/dbias[v, g] = sum_{d in g} dw[v, d] (the codes are not differentiable).
 *   h, M, targets, mask, lse, dlogp  as for qhead_bwd.
 *   dh        device, float [M, H], 16-byte aligned, or NULL (not computed).
 *   dw        device, float [V, H] row-major, 32-byte aligned; every element is
 *             written (M == 0 or no active row: all zeros).
 *   workspace device, >= qhead_bwd_dw_workspace(head, M) bytes, 256-byte aligned.
 * Every M takes the tensor-core path (dw reuses its per-chunk coefficient
 * blocks).  A row whose target lies outside [0, V) contributes its softmax
 * term but no one-hot term.  If a kernel wait expires, every element of dw is
 * NaN.  The result is deterministic: each dw element is written once, and the
 * rows that share a target are summed in row order.
 */
int qhead_bwd_dw(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
                 const uint8_t* mask, const float* lse, const float* dlogp, float* dh, float* dw,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward without a workspace argument, for callers that cannot allocate
 * device memory (no counterpart on the pages: it is an addition for this
 * library's users).  Engines that run the verify step inside a pre-sized
 * memory arena, plugins hosted by frameworks that forbid allocation after
 * start-up, and latency-critical loops that must not enter the allocator
 * cannot call cudaMalloc to provide qhead_fwd's workspace.  This call takes
 * the same arguments as qhead_fwd minus the workspace and computes the same
 * outputs, bit for bit, using instead a fixed scratch array of 8 MiB
 * (8388608 bytes) that lives in the library on every device that loads it,
 * until the process exits.  It allocates nothing and calls no allocating
 * routine.
 *   - The first call with a given device current looks up the array's device
 *     address (cudaGetSymbolAddress) and caches it by device ordinal; make
 *     that first call before any stream capture on the device.  The cached
 *     address belongs to the device's primary context as it was then: after
 *     cudaDeviceReset on that device, or with a non-primary context current
 *     on it, the cached address is stale and this call must not be used.
 *   - M rows whose workspace (qhead_fwd_workspace) exceeds the scratch size
 *     are rejected with QHEAD_EINVAL and a message; nothing is launched.
 *     In practice the scratch holds up to about 200 rows at H = 2560,
 *     V = 262144 (the weight-streaming path up to 16 rows needs a few hundred
 *     KB; the tensor-core path from 17 rows 32 bytes per row and 256-row
 *     vocab tile of partials); a bf16 or fp32 head's fp16 copies of scales
 *     and biases (4 * V * H/64 bytes, 42 MB at that shape) do not fit, so
 *     such heads are rejected.
 *   - Every call shares the one array.  No byte of it needs to start at zero
 *     (a call writes all scratch it reads), but calls whose kernels may
 *     overlap on the GPU (e.g. issued on different streams without ordering)
 *     race on it: order them on one stream or with events.
 *   - A call rejected by the size check disarms the thread's one-shot hooks
 *     (qhead_time_next_head_kernel, qhead_test_stall_next_call) as a forward
 *     call would.
 */
int qhead_fwd_noalloc(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
                      const uint8_t* mask, float* logp, float* lse, int32_t* argmax,
                      void* stream);

/* Message for the last error on the calling thread ("" if none).  The
 * pointer stays valid until the thread's next qhead_* call. */
const char* qhead_last_error(void);

/*
 * Instrumentation (no counterpart on the pages): arm a one-shot hook on the
 * calling thread.  The thread's next forward or backward call (qhead_fwd,
 * qhead_verify, qhead_fwd_noalloc, qhead_fwd_blockmax, qhead_bwd and the
 * other backward entry points) records the CUDA event `start` on its stream
 * immediately before its head kernel (the vocab-streaming contraction that
 * dominates the call; for a backward on the tensor-core path, the chain of
 * its per-chunk kernels) and `stop` immediately after it, then disarms the
 * hook.  A call rejected before it launches anything disarms it too.  start and stop are
 * cudaEvent_t handles passed as void*; passing NULL for both disarms.
 */
void qhead_time_next_head_kernel(void* start, void* stop);

/*
 * Test instrumentation (no counterpart on the pages): arm a one-shot switch
 * on the calling thread.  The thread's next forward or backward call (the
 * entry points listed for qhead_time_next_head_kernel) launches its
 * pipelined head kernel with the TMA producer issuing no loads,
 * so the consumers' bounded waits expire and the call ends as described under
 * "Kernel time limits" (about 2 s later, without a fault).  armed = 0
 * disarms.  Exists so that the time-limit path can be
 * tested.
 */
void qhead_test_stall_next_call(int armed);

/* Library version string, e.g. "qhead 0.1.0 sm_103a". */
const char* qhead_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QHEAD_H */

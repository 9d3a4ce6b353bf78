// qh_blockskip.cu -- the skip map of the approximate blockMax early exit.
//
// The vocab-parallel backward on the page "mlx-bun 0.0.4 -> 0.0.6"
// (src/train/flash-cce.ts) may skip a (token block, vocab block) program when
// every token's block maximum satisfies exp(blockMax - lse) < eps and no
// target lies in the block (the forward hands blockMax over).  Here the
// blocks are (128 consecutive active rows, 256-row vocab tile) pairs, the
// tensor-core kernels' tiles; the map marks the pairs both backward phases
// skip.  exp(bm - lse) < eps is evaluated as bm - lse < ln(eps) in fp32.
#include "qh_internal.cuh"

namespace qh {

namespace {

constexpr int kRowsPerTile = 128;

// One block per (row tile, vocab tile) pair: pair = mt * n_vt + vt.
__global__ void __launch_bounds__(kRowsPerTile) skip_map_kernel(
    const float* __restrict__ bmax, int64_t ld, const float* __restrict__ lse,
    const int32_t* __restrict__ targets, const int* __restrict__ rows,
    const int* __restrict__ count, int64_t n_vt, float log_eps, uint8_t* __restrict__ skip) {
    const int64_t pair = blockIdx.x;
    const int64_t mt = pair / n_vt, vt = pair - mt * n_vt;
    const int64_t i = mt * kRowsPerTile + threadIdx.x;
    bool ok = true;  // rows past the active ones do not hold the tile back
    if (i < *count) {
        const int r = rows[i];
        const int32_t t = targets[r];
        const bool holds_target = t >= 0 && ((int64_t)t >> 8) == vt;
        ok = !holds_target && bmax[(int64_t)r * ld + vt] - lse[r] < log_eps;
    }
    const int all = __syncthreads_and(ok);
    if (threadIdx.x == 0) skip[pair] = all ? 1 : 0;
}

}  // namespace

cudaError_t launch_skip_map(const float* bmax, int64_t ld, const float* lse,
                            const int32_t* targets, const int* rows, const int* count,
                            int64_t n_mt, int64_t n_vt, float eps, uint8_t* skip,
                            cudaStream_t st) {
    const int64_t pairs = n_mt * n_vt;
    if (pairs <= 0 || pairs > INT32_MAX) return cudaErrorInvalidValue;
    const float log_eps = eps > 0.f ? logf(eps) : -INFINITY;
    skip_map_kernel<<<(unsigned)pairs, kRowsPerTile, 0, st>>>(bmax, ld, lse, targets, rows, count,
                                                              n_vt, log_eps, skip);
    return cudaGetLastError();
}

}  // namespace qh

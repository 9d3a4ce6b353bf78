// qh_prologue.cu -- step a1 of the hot path: compact the active rows and stage
// h for the tensor-core kernels.
//
// The pages slice the response span out of h before the head runs (page
// "mlx-bun 0.0.9 -> 0.0.10", src/train/loss.ts, responseOnlyCe: the head is
// applied only at the supervised positions).  Here the same selection is a
// per-row mask, turned into an ascending list of active rows so the head
// kernels never spend work on masked rows.
#include "qh_internal.cuh"

namespace qh {

// One CTA of 1024 threads scans the mask in chunks of 1024 rows.
// rows[i] = original index of the i-th active row (ascending), rows[i] = -1 for
// i in [count, Mpad); pos[r] = compact index of row r, or -1 if r is masked.
// Must be called by all 1024 threads of the CTA; returns the active count.
__device__ int compact_rows(const uint8_t* __restrict__ mask, int64_t M, int64_t Mpad,
                            int* __restrict__ rows, int* __restrict__ pos, int* __restrict__ count) {
    __shared__ int warp_tot[32];
    __shared__ int base_sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) base_sh = 0;
    __syncthreads();
    for (int64_t c0 = 0; c0 < M; c0 += 1024) {
        const int64_t r = c0 + tid;
        const bool act = r < M && (mask == nullptr || mask[r] != 0);
        const unsigned bal = __ballot_sync(0xffffffffu, act);
        const int within = __popc(bal & ((1u << lane) - 1u));
        if (lane == 0) warp_tot[warp] = __popc(bal);
        __syncthreads();
        if (warp == 0) {
            const int v = warp_tot[lane];
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            warp_tot[lane] = incl - v;  // exclusive prefix of the warp totals
        }
        __syncthreads();
        const int base = base_sh;
        if (r < M) {
            const int idx = base + warp_tot[warp] + within;
            pos[r] = act ? idx : -1;
            if (act) rows[idx] = (int)r;
        }
        __syncthreads();
        if (tid == 1023) base_sh = base + warp_tot[31] + __popc(bal);
        __syncthreads();
    }
    const int n = base_sh;
    for (int64_t i = n + tid; i < Mpad; i += 1024) rows[i] = -1;
    if (tid == 0) *count = n;
    return n;
}

__global__ void __launch_bounds__(1024) compact_kernel(const uint8_t* __restrict__ mask, int64_t M,
                                                       int64_t Mpad, int* __restrict__ rows,
                                                       int* __restrict__ pos, int* __restrict__ count,
                                                       int* __restrict__ err) {
    if (err && threadIdx.x == 0) *err = 0;
    compact_rows(mask, M, Mpad, rows, pos, count);
}

// h16[i, :] = fp16(h[rows[i], :]) for i < count, zeros for count <= i < Mpad.
// For 4-bit heads every 8-element block is stored in the order
// (0,4,1,5,2,6,3,7): the order in which the tensor-core kernels' dequantizer
// yields (q_k, q_k+4) pairs out of one packed word, so both mma operands see
// the same permutation of the K axis.  8-bit heads keep the natural order.
__device__ __forceinline__ uint4 convert_unit(const __nv_bfloat16* __restrict__ src, int bits) {
    const uint4 in = *reinterpret_cast<const uint4*>(src);
    const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&in);
    __half y[8];
    if (bits == 4) {
        const int perm[8] = {0, 4, 1, 5, 2, 6, 3, 7};
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = __float2half_rn(__bfloat162float(x[perm[k]]));
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = __float2half_rn(__bfloat162float(x[k]));
    }
    return *reinterpret_cast<const uint4*>(y);
}

__global__ void convert_h_kernel(const __nv_bfloat16* __restrict__ h, int H, int bits,
                                 const int* __restrict__ rows, const int* __restrict__ count,
                                 __half* __restrict__ h16) {
    const int64_t i = blockIdx.x;
    const int u = threadIdx.x;  // 8-element unit
    if (u >= H / 8) return;
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (i < *count) out = convert_unit(h + (int64_t)rows[i] * H + 8 * u, bits);
    *reinterpret_cast<uint4*>(h16 + i * H + 8 * u) = out;
}

// Small M: one CTA compacts, then converts rows [0, nrows) (zeros past the
// active count): groups of 8 for the weight-streaming kernel, whole 128-row
// tiles for the tensor-core kernel.
__global__ void __launch_bounds__(1024) prologue_fused_kernel(
    const uint8_t* __restrict__ mask, const __nv_bfloat16* __restrict__ h, int64_t M, int64_t Mpad,
    int H, int bits, int* __restrict__ rows, int* __restrict__ pos, int* __restrict__ count,
    __half* __restrict__ h16, int64_t nrows, int* __restrict__ err) {
    if (err && threadIdx.x == 0) *err = 0;
    const int n = compact_rows(mask, M, Mpad, rows, pos, count);
    __syncthreads();  // rows[] written by other threads
    const int units = H / 8;
    for (int64_t idx = threadIdx.x; idx < nrows * units; idx += 1024) {
        const int64_t i = idx / units;
        const int u = (int)(idx - i * units);
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (i < n) out = convert_unit(h + (int64_t)rows[i] * H + 8 * u, bits);
        *reinterpret_cast<uint4*>(h16 + i * H + 8 * u) = out;
    }
}

cudaError_t launch_prologue_fused(const uint8_t* mask, const __nv_bfloat16* h, int64_t M,
                                  int64_t Mpad, int H, int bits, int* rows, int* pos, int* count,
                                  __half* h16, int64_t nrows, int* err, cudaStream_t st) {
    prologue_fused_kernel<<<1, 1024, 0, st>>>(mask, h, M, Mpad, H, bits, rows, pos, count, h16,
                                              nrows, err);
    return cudaGetLastError();
}

cudaError_t launch_compact(const uint8_t* mask, int64_t M, int64_t Mpad, int* rows, int* pos,
                           int* count, int* err, cudaStream_t st) {
    compact_kernel<<<1, 1024, 0, st>>>(mask, M, Mpad, rows, pos, count, err);
    return cudaGetLastError();
}

// Scales and biases of a bf16 or fp32 head rounded to fp16 (nearest, ties to
// even) for the kernels that read fp16 operands: exact for bf16 values in
// [2^-17, 65504] (bf16 has 8 significant bits, fp16 11), one rounding for fp32
// values.  Grid-stride over the n elements of each array.
__global__ void sb_to_f16_kernel(SbView sb, int64_t n, __half* __restrict__ s16,
                                 __half* __restrict__ b16) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        s16[i] = __float2half_rn(sb_elem(sb.s, i, sb.type));
        b16[i] = __float2half_rn(sb_elem(sb.b, i, sb.type));
    }
}

cudaError_t launch_sb_to_f16(SbView sb, int64_t n, __half* s16, __half* b16, cudaStream_t st) {
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)device_sms() * 8;
    if (blocks > cap && cap > 0) blocks = cap;
    if (blocks < 1) blocks = 1;
    sb_to_f16_kernel<<<(unsigned)blocks, 256, 0, st>>>(sb, n, s16, b16);
    return cudaGetLastError();
}

cudaError_t launch_convert_h(const __nv_bfloat16* h, int64_t Mpad, int H, int bits, const int* rows,
                             const int* count, __half* h16, cudaStream_t st) {
    const int threads = ((H / 8) + 31) / 32 * 32;
    convert_h_kernel<<<(unsigned)Mpad, threads, 0, st>>>(h, H, bits, rows, count, h16);
    return cudaGetLastError();
}

}  // namespace qh

// qh_bwd_simt.cu -- CUDA-core backward (steps a9-a10 of the hot path).
//
// The two-phase backward of the page "mlx-bun 0.0.4 -> 0.0.6"
// (src/train/flash-cce.ts, BWD_SOURCE): per block of vocab rows, phase 1
// recomputes each row's logit for a small group of tokens and forms
//   coeff = -dlogp * exp(z - lse) * sech2
// (the one-hot part of dlogp * (onehot - softmax) * sech2 is added exactly
// by the finalize kernel), then phase 2 accumulates dh[t, d] += coeff * w[v, d]
// with every thread owning a fixed set of output columns, so no two threads
// write the same output.  Instead of the page's float atomics across vocab
// blocks, each vocab split writes its own partial dh, summed in a fixed
// order by the finalize kernel (deterministic).  Arithmetic is fp32.
#include "qh_internal.cuh"

namespace qh {

namespace {

constexpr int kThreads = 256;

template <int TB, int DPT>
__global__ void __launch_bounds__(kThreads) bwd_simt_kernel(
    const uint32_t* __restrict__ wq, const __half* __restrict__ scales,
    const __half* __restrict__ biases, int64_t V, int H, int bits, float cap,
    const __nv_bfloat16* __restrict__ h, const int* __restrict__ rows,
    const int* __restrict__ count, const float* __restrict__ lse,
    const float* __restrict__ dlogp, float* __restrict__ dhp, int S, int64_t Mpad) {
    const int n_active = *count;
    const int tok0 = blockIdx.x * TB;
    if (tok0 >= n_active) return;
    const int split = blockIdx.y;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __nv_bfloat16* hs = reinterpret_cast<__nv_bfloat16*>(smem_raw);          // [TB][H]
    float* cs = reinterpret_cast<float*>(smem_raw + (size_t)TB * H * 2);     // [kThreads][TB]
    __shared__ float lse_sh[TB], g_sh[TB];

    const int tid = threadIdx.x;
    if (tid < TB) {
        const int i = tok0 + tid;
        if (i < n_active) {
            const int r = rows[i];
            lse_sh[tid] = lse[r];
            g_sh[tid] = dlogp[r];
        } else {
            lse_sh[tid] = 0.f;
            g_sh[tid] = 0.f;
        }
    }
    for (int idx = tid; idx < TB * (H / 8); idx += kThreads) {
        const int j = idx / (H / 8), u = idx % (H / 8);
        const int i = tok0 + j;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (i < n_active) v = *reinterpret_cast<const uint4*>(h + (int64_t)rows[i] * H + 8 * u);
        *reinterpret_cast<uint4*>(hs + j * H + 8 * u) = v;
    }
    __syncthreads();

    const int64_t v0 = V * split / S, v1 = V * (split + 1) / S;
    const int wpr = H * bits / 32;
    const int G = H / 64;
    const int per = 32 / bits;
    const uint32_t qmask = (1u << bits) - 1u;
    const int dpt = (H + kThreads - 1) / kThreads;

    float acc[DPT][TB];
#pragma unroll
    for (int k = 0; k < DPT; ++k)
#pragma unroll
        for (int j = 0; j < TB; ++j) acc[k][j] = 0.f;

    for (int64_t base = v0; base < v1; base += kThreads) {
        // Phase 1: row v = base + tid, logits for the TB tokens.
        const int64_t v = base + tid;
        float raw[TB];
#pragma unroll
        for (int j = 0; j < TB; ++j) raw[j] = 0.f;
        if (v < v1) {
            const uint32_t* wrow = wq + v * wpr;
            for (int gi = 0; gi < G; ++gi) {
                const float s = __half2float(scales[v * G + gi]);
                const float b = __half2float(biases[v * G + gi]);
                for (int wi = 0; wi < 64 / per; ++wi) {
                    const uint32_t word = wrow[gi * (64 / per) + wi];
                    const int d0 = gi * 64 + wi * per;
                    for (int k = 0; k < per; ++k) {
                        const float w = fmaf(s, (float)((word >> (bits * k)) & qmask), b);
#pragma unroll
                        for (int j = 0; j < TB; ++j)
                            raw[j] = fmaf(__bfloat162float(hs[j * H + d0 + k]), w, raw[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            float c = 0.f;
            if (v < v1) {
                float z = raw[j], sech2 = 1.f;
                if (cap > 0.f) {
                    const float th = tanhf(raw[j] / cap);
                    z = cap * th;
                    sech2 = 1.f - th * th;
                }
                c = -g_sh[j] * expf(z - lse_sh[j]) * sech2;
            }
            cs[tid * TB + j] = c;
        }
        __syncthreads();
        // Phase 2: dh[j, d] += coeff[row, j] * w[row, d] for this thread's columns.
        const int nrows = (int)min((int64_t)kThreads, v1 - base);
        for (int rr = 0; rr < nrows; ++rr) {
            const int64_t vv = base + rr;
            const uint32_t* wrow = wq + vv * wpr;
            float cj[TB];
#pragma unroll
            for (int j = 0; j < TB; ++j) cj[j] = cs[rr * TB + j];
#pragma unroll
            for (int k = 0; k < DPT; ++k) {
                const int d = tid + k * kThreads;
                if (k < dpt && d < H) {
                    const uint32_t word = wrow[d / per];
                    const float w = fmaf(__half2float(scales[vv * G + d / 64]),
                                         (float)((word >> (bits * (d % per))) & qmask),
                                         __half2float(biases[vv * G + d / 64]));
#pragma unroll
                    for (int j = 0; j < TB; ++j) acc[k][j] = fmaf(cj[j], w, acc[k][j]);
                }
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < DPT; ++k) {
        const int d = tid + k * kThreads;
        if (k < dpt && d < H) {
#pragma unroll
            for (int j = 0; j < TB; ++j) {
                const int i = tok0 + j;
                if (i < n_active) dhp[((int64_t)split * Mpad + i) * H + d] = acc[k][j];
            }
        }
    }
}

template <int TB, int DPT>
cudaError_t launch_t(const uint32_t* wq, const __half* scales, const __half* biases, int64_t V,
                     int H, int bits, float cap, const __nv_bfloat16* h, const int* rows,
                     const int* count, const float* lse, const float* dlogp, float* dhp, int S,
                     int64_t M, int64_t Mpad, cudaStream_t st) {
    const size_t smem = (size_t)TB * H * 2 + (size_t)kThreads * TB * sizeof(float);
    if (cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(bwd_simt_kernel<TB, DPT>),
                                          (int)smem))
        return e;
    dim3 grid((unsigned)((M + TB - 1) / TB), S);
    bwd_simt_kernel<TB, DPT><<<grid, kThreads, smem, st>>>(wq, scales, biases, V, H, bits, cap, h,
                                                            rows, count, lse, dlogp, dhp, S, Mpad);
    return cudaGetLastError();
}

}  // namespace

int bwd_simt_tokens(int H) { return H <= 4096 ? 8 : 4; }

cudaError_t launch_bwd_simt(const uint32_t* wq, const __half* scales, const __half* biases,
                            int64_t V, int H, int bits, float cap, const __nv_bfloat16* h,
                            const int* rows, const int* count, const float* lse,
                            const float* dlogp, float* dhp, int S, int64_t M, int64_t Mpad,
                            cudaStream_t st) {
    if (H <= 4096)
        return launch_t<8, 16>(wq, scales, biases, V, H, bits, cap, h, rows, count, lse, dlogp,
                               dhp, S, M, Mpad, st);
    return launch_t<4, 32>(wq, scales, biases, V, H, bits, cap, h, rows, count, lse, dlogp, dhp,
                           S, M, Mpad, st);
}

}  // namespace qh

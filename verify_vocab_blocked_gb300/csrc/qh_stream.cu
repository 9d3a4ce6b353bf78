// qh_stream.cu -- weight-streaming forward (steps a2-a5 and a8 of the hot path
// for small M; also the general path until the tcgen05 kernel takes large M).
//
// What it computes: for 8 compacted rows of h and a slice of the vocab, the
// per-row online-softmax partial (max z, sum exp(z - max)) and the two best
// raw logits with their indices -- the per-(token, vocab-block) partials of
// the vocab-parallel forward on the page "mlx-bun 0.0.4 -> 0.0.6"
// (src/train/flash-cce.ts, FWD_SOURCE: a bounded vocab slice per program,
// per-thread online softmax, merged inside the program), plus the argmax
// candidates the speculative-decode verify needs (page "mlx-bun 0.0.8 ->
// 0.0.10", src/spec/generate.ts, picksBatched).
//
// How (GB300): at M = gamma+1 the cost is reading the packed head once, but
// plain fp32 FMAs cannot keep up with HBM (10 FMA per packed byte at M = 5).
// So each warp streams 16 vocab rows at a time straight from HBM into
// registers, dequantizes them in registers into the A fragments of
// mma.sync.m16n8k16 (A = 16 vocab rows x 16 K, B = 16 K x 8 tokens, fp32
// accumulate), and never stages the dequantized head anywhere.  The K axis is
// permuted consistently in A and B so that one packed word yields A fragments
// with one shift + lop3 per pair of codes (4-bit), or one prmt per pair (8-bit):
//   4-bit: word j of a row holds d = 8j .. 8j+7; lop3((w >> 4k) & 0x000F000F |
//          0x64006400) = fp16 pair (1024 + q_k, 1024 + q_k+4); the staged h
//          rows store each 8-block as (0,4,1,5,2,6,3,7).
//   8-bit: prmt builds (1024 + q_0, 1024 + q_1) and (1024 + q_2, 1024 + q_3).
// then w = fma(q, scale, bias) in fp16 (one rounding) after an exact
// subtraction of 1024.  The row's logits never leave registers.
#include "qh_internal.cuh"

namespace qh {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
    return d;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 x) { return *reinterpret_cast<uint32_t*>(&x); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t x) { return *reinterpret_cast<__half2*>(&x); }

// (1024 + q_lo, 1024 + q_hi) -> (s*q_lo + b, s*q_hi + b), fp16, one rounding.
__device__ __forceinline__ uint32_t affine(uint32_t magic_pair, __half2 s, __half2 b) {
    const __half2 k1024 = __float2half2_rn(1024.f);
    const __half2 q = __hsub2(u32_as_h2(magic_pair), k1024);  // exact: integers < 2048
    return h2_as_u32(__hfma2(q, s, b));
}

__device__ __forceinline__ uint32_t deq4(uint32_t w, int k, __half2 s, __half2 b) {
    return affine(lop3_and_or(w >> (4 * k), 0x000F000Fu, 0x64006400u), s, b);
}

__device__ __forceinline__ uint32_t deq8(uint32_t w, uint32_t sel, __half2 s, __half2 b) {
    return affine(__byte_perm(w, 0x64646464u, sel), s, b);
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t u4_at(const uint4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// One chunk = 16 packed words of a row (128 elements at 4 bits, 64 at 8 bits).
// Thread (g, t) owns words 4t .. 4t+3 of the chunk for rows g and g+8.
template <int BITS>
__device__ __forceinline__ void chunk_mma(float (&acc)[4], const uint4& a0, const uint4& a1,
                                          __half2 s0, __half2 b0, __half2 s1, __half2 b1,
                                          const __half* hb) {
    if constexpr (BITS == 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 bq = *reinterpret_cast<const uint4*>(hb + 8 * j);
            const uint32_t w0 = u4_at(a0, j), w1 = u4_at(a1, j);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint32_t A0 = deq4(w0, 2 * e, s0, b0);
                const uint32_t A2 = deq4(w0, 2 * e + 1, s0, b0);
                const uint32_t A1 = deq4(w1, 2 * e, s1, b1);
                const uint32_t A3 = deq4(w1, 2 * e + 1, s1, b1);
                mma16816(acc, A0, A1, A2, A3, e ? bq.z : bq.x, e ? bq.w : bq.y);
            }
        }
    } else {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const uint4 bq = *reinterpret_cast<const uint4*>(hb + 8 * jj);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint32_t w0 = u4_at(a0, 2 * jj + e), w1 = u4_at(a1, 2 * jj + e);
                const uint32_t A0 = deq8(w0, 0x5140u, s0, b0);
                const uint32_t A2 = deq8(w0, 0x7362u, s0, b0);
                const uint32_t A1 = deq8(w1, 0x5140u, s1, b1);
                const uint32_t A3 = deq8(w1, 0x7362u, s1, b1);
                mma16816(acc, A0, A1, A2, A3, e ? bq.z : bq.x, e ? bq.w : bq.y);
            }
        }
    }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) stream_fwd_kernel(
    const uint32_t* __restrict__ wq, const __half* __restrict__ scales,
    const __half* __restrict__ biases, int64_t V, int H, float cap,
    const __half* __restrict__ h16, const int* __restrict__ count, Partial* __restrict__ part,
    int S) {
    const int n_active = *count;
    const int tok0 = blockIdx.x * kTokGroup;
    if (tok0 >= n_active) return;
    const int split = blockIdx.y;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    __half* hs = reinterpret_cast<__half*>(smem_raw);
    const int hstride = H + 8;  // halves; +16 bytes per row spreads the banks
    __shared__ Partial red[kWarps][kTokGroup];

    // Stage the group's 8 rows of h (fp16, K-permuted for 4-bit) in shared memory.
    const int units = H / 8;
    for (int idx = threadIdx.x; idx < kTokGroup * units; idx += kThreads) {
        const int r = idx / units, c = idx - r * units;
        const uint4 v = *reinterpret_cast<const uint4*>(h16 + (int64_t)(tok0 + r) * H + 8 * c);
        *reinterpret_cast<uint4*>(hs + r * hstride + 8 * c) = v;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int64_t cta_v0 = V * split / S, cta_v1 = V * (split + 1) / S;
    const int64_t len = cta_v1 - cta_v0;
    const int64_t wv0 = cta_v0 + len * warp / kWarps, wv1 = cta_v0 + len * (warp + 1) / kWarps;
    const int wpr = H * BITS / 32;
    const int G = H / 64;
    const int nchunks = wpr / 16;
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
    const __half* hrow = hs + g * hstride + (BITS == 4 ? 32 * t : 16 * t);

    RowState st[2];
    st[0].init();
    st[1].init();

    for (int64_t tile = wv0; tile < wv1; tile += 16) {
        const int64_t r0 = tile + g, r1 = tile + g + 8;
        const bool ok0 = r0 < wv1, ok1 = r1 < wv1;
        const uint4* p0 = reinterpret_cast<const uint4*>(wq + (ok0 ? r0 : wv0) * wpr) + t;
        const uint4* p1 = reinterpret_cast<const uint4*>(wq + (ok1 ? r1 : wv0) * wpr) + t;
        const __half* sc0 = scales + (ok0 ? r0 : wv0) * G;
        const __half* sc1 = scales + (ok1 ? r1 : wv0) * G;
        const __half* bi0 = biases + (ok0 ? r0 : wv0) * G;
        const __half* bi1 = biases + (ok1 ? r1 : wv0) * G;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};

        uint4 na0 = ok0 ? ld_stream(p0) : zero4;
        uint4 na1 = ok1 ? ld_stream(p1) : zero4;
        for (int c = 0; c < nchunks; ++c) {
            const uint4 a0 = na0, a1 = na1;
            if (c + 1 < nchunks) {
                na0 = ok0 ? ld_stream(p0 + 4 * (c + 1)) : zero4;
                na1 = ok1 ? ld_stream(p1 + 4 * (c + 1)) : zero4;
            }
            const int gi = BITS == 4 ? (2 * c + (t >> 1)) : c;
            const __half2 s0 = __half2half2(sc0[gi]), b0 = __half2half2(bi0[gi]);
            const __half2 s1 = __half2half2(sc1[gi]), b1 = __half2half2(bi1[gi]);
            chunk_mma<BITS>(acc, a0, a1, s0, b0, s1, b1, hrow + (BITS == 4 ? 128 : 64) * c);
        }
        // acc: (row g, token 2t), (row g, token 2t+1), (row g+8, token 2t), (row g+8, token 2t+1)
        if (ok0) {
            st[0].push(softcap_exact(acc[0], cap), acc[0], (int)r0);
            st[1].push(softcap_exact(acc[1], cap), acc[1], (int)r0);
        }
        if (ok1) {
            st[0].push(softcap_exact(acc[2], cap), acc[2], (int)r1);
            st[1].push(softcap_exact(acc[3], cap), acc[3], (int)r1);
        }
    }

    // Merge the 8 lanes that share t (lanes t, t+4, ..., t+28), then the warps.
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
        st[0].shfl_merge(o);
        st[1].shfl_merge(o);
    }
    if (g == 0) {
        red[warp][2 * t] = st[0].to_partial();
        red[warp][2 * t + 1] = st[1].to_partial();
    }
    __syncthreads();
    if (threadIdx.x < kTokGroup) {
        const int j = threadIdx.x;
        RowState acc;
        acc.init();
        for (int w = 0; w < kWarps; ++w) acc.merge(red[w][j]);
        part[(int64_t)(tok0 + j) * S + split] = acc.to_partial();
    }
}

}  // namespace

cudaError_t launch_stream_fwd(const uint32_t* wq, const __half* scales, const __half* biases,
                              int64_t V, int H, int bits, float cap, const __half* h16,
                              const int* count, int64_t M, Partial* part, int S, cudaStream_t st) {
    const int groups = (int)((M + kTokGroup - 1) / kTokGroup);
    const size_t smem = (size_t)kTokGroup * (H + 8) * sizeof(__half);
    dim3 grid(groups, S);
    if (bits == 4) {
        cudaFuncSetAttribute(stream_fwd_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        stream_fwd_kernel<4><<<grid, kThreads, smem, st>>>(wq, scales, biases, V, H, cap, h16,
                                                           count, part, S);
    } else {
        cudaFuncSetAttribute(stream_fwd_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        stream_fwd_kernel<8><<<grid, kThreads, smem, st>>>(wq, scales, biases, V, H, cap, h16,
                                                           count, part, S);
    }
    return cudaGetLastError();
}

}  // namespace qh

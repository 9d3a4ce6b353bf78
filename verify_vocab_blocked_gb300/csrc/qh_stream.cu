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
#include "qh_dequant.cuh"

namespace qh {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

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
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
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
            uint32_t p0[4], p1[4];
            deq4_word(u4_at(a0, j), s0, b0, p0);
            deq4_word(u4_at(a1, j), s1, b1, p1);
            // step e = 0 uses pairs (0,4) and (1,5); e = 1 uses (2,6) and (3,7)
            mma16816(acc, p0[0], p1[0], p0[1], p1[1], bq.x, bq.y);
            mma16816(acc, p0[2], p1[2], p0[3], p1[3], bq.z, bq.w);
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

// One packed chunk of a warp's work: A words of rows g and g+8 and their
// (scale, bias) pairs, packed as half2 (scale, bias).
struct Item {
    uint4 a0, a1;
    uint32_t sb0, sb1;
};

template <int BITS>
__global__ void __launch_bounds__(kThreads, 3) stream_fwd_kernel(
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

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int64_t cta_v0 = V * split / S, cta_v1 = V * (split + 1) / S;
    const int64_t len = cta_v1 - cta_v0;
    const int64_t wv0 = cta_v0 + len * warp / kWarps, wv1 = cta_v0 + len * (warp + 1) / kWarps;
    const int wpr = H * BITS / 32;
    const int G = H / 64;
    const int nchunks = wpr / 16;
    const int ntiles = (int)((wv1 - wv0 + 15) / 16);
    const int nitems = ntiles * nchunks;

    // Item loader.  Rows past the warp's range are clamped to its last row (a
    // valid address); their logits are discarded in the epilogue.  Only two
    // row indices are kept; addresses are formed at fetch time.
    int pf_c = 0;
    int64_t pf_r0 = wv0 + g;
    int rc0 = 0, rc1 = 0;
    const int wpr4 = wpr / 4;                      // uint4 per row
    const int go = BITS == 4 ? (t >> 1) : 0;      // group offset of this lane
    auto set_rows = [&]() {
        const int64_t last = wv1 - 1;
        rc0 = (int)min(pf_r0, last);
        rc1 = (int)min(pf_r0 + 8, last);
    };
    const uint4* wq4 = reinterpret_cast<const uint4*>(wq) + t;
    auto fetch = [&](Item& it) {
        it.a0 = ld_stream(wq4 + ((int64_t)rc0 * wpr4 + 4 * pf_c));
        it.a1 = ld_stream(wq4 + ((int64_t)rc1 * wpr4 + 4 * pf_c));
        const int gi = (BITS == 4 ? 2 * pf_c : pf_c) + go;
        const int64_t o0 = (int64_t)rc0 * G + gi, o1 = (int64_t)rc1 * G + gi;
        it.sb0 = h2_as_u32(__halves2half2(scales[o0], biases[o0]));
        it.sb1 = h2_as_u32(__halves2half2(scales[o1], biases[o1]));
        if (++pf_c == nchunks) {
            pf_c = 0;
            pf_r0 += 16;
            set_rows();
        }
    };

    Item A, B, C;
    if (nitems > 0) {
        set_rows();
        fetch(A);
    }
    if (nitems > 1) fetch(B);

    // Stage the group's 8 rows of h (fp16, K-permuted for 4-bit) in shared memory.
    const int units = H / 8;
    for (int idx = threadIdx.x; idx < kTokGroup * units; idx += kThreads) {
        const int r = idx / units, c = idx - r * units;
        const uint4 v = *reinterpret_cast<const uint4*>(h16 + (int64_t)(tok0 + r) * H + 8 * c);
        *reinterpret_cast<uint4*>(hs + r * hstride + 8 * c) = v;
    }
    __syncthreads();
    const __half* hrow = hs + g * hstride + (BITS == 4 ? 32 * t : 16 * t);
    constexpr int kChunkHalves = BITS == 4 ? 128 : 64;

    RowState st[2];
    st[0].init();
    st[1].init();
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int c = 0;
    int64_t tile_r0 = wv0 + g;
    auto compute = [&](const Item& it) {
        const __half2 sb0 = u32_as_h2(it.sb0), sb1 = u32_as_h2(it.sb1);
        chunk_mma<BITS>(acc, it.a0, it.a1, __low2half2(sb0), __high2half2(sb0), __low2half2(sb1),
                        __high2half2(sb1), hrow + kChunkHalves * c);
        if (++c == nchunks) {
            // acc: (row g, tok 2t), (row g, tok 2t+1), (row g+8, tok 2t), (row g+8, tok 2t+1)
            const int64_t r0 = tile_r0, r1 = tile_r0 + 8;
            if (r0 < wv1) {
                st[0].push(softcap_exact(acc[0], cap), acc[0], (int)r0);
                st[1].push(softcap_exact(acc[1], cap), acc[1], (int)r0);
            }
            if (r1 < wv1) {
                st[0].push(softcap_exact(acc[2], cap), acc[2], (int)r1);
                st[1].push(softcap_exact(acc[3], cap), acc[3], (int)r1);
            }
            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            c = 0;
            tile_r0 += 16;
        }
    };
    // Three-slot ring, unrolled so no slot is ever copied: item k is computed
    // while item k+2 is in flight.
    for (int k = 0; k < nitems; k += 3) {
        if (k + 2 < nitems) fetch(C);
        compute(A);
        if (k + 1 >= nitems) break;
        if (k + 3 < nitems) fetch(A);
        compute(B);
        if (k + 2 >= nitems) break;
        if (k + 4 < nitems) fetch(B);
        compute(C);
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

int stream_fwd_ctas_per_sm(int bits, int H) {
    const size_t smem = (size_t)kTokGroup * (H + 8) * sizeof(__half);
    int n = 0;
    cudaError_t e;
    if (bits == 4) {
        cudaFuncSetAttribute(stream_fwd_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, stream_fwd_kernel<4>, kThreads, smem);
    } else {
        cudaFuncSetAttribute(stream_fwd_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, stream_fwd_kernel<8>, kThreads, smem);
    }
    return (e == cudaSuccess && n > 0) ? n : 1;
}

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

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
// A producer warp streams the CTA's vocab range through shared memory with
// TMA (128 rows x 16 packed words per stage, 6 stages) and copies each
// stage's scales and biases with cp.async; eight consumer warps each take 16
// of the 128 rows, dequantize them in registers into the A fragments of
// mma.sync.m16n8k16 (A = 16 vocab rows x 16 K, B = 16 K x 8 tokens, fp32
// accumulate), and never stage the dequantized head anywhere.  The K axis is
// permuted consistently in A and B so that one packed word yields A fragments
// with one shift + lop3 per pair of codes (4-bit), or one prmt per pair (8-bit):
//   4-bit: word j of a row holds d = 8j .. 8j+7; lop3((w >> 4k) & 0x000F000F |
//          0x64006400) = fp16 pair (1024 + q_k, 1024 + q_k+4); the staged h
//          rows store each 8-block as (0,4,1,5,2,6,3,7).
//   8-bit: prmt builds (1024 + q_0, 1024 + q_1) and (1024 + q_2, 1024 + q_3).
// then w = fma(q, scale, bias) in fp16 (one rounding) after an exact
// subtraction of 1024.  The row's logits never leave registers.
#include <map>
#include <mutex>
#include <tuple>

#include "qh_dequant.cuh"
#include "qh_tc.cuh"
#include "qh_tmap.h"

namespace qh {

namespace {

constexpr int kConsumers = 8;                 // consumer warps, 16 rows each
constexpr int kThreads = 32 * (1 + kConsumers);
constexpr int kTile = 16 * kConsumers;        // vocab rows per stage
constexpr int kChunkWords = 16;               // packed words per row per stage
constexpr int kPBytes = kTile * kChunkWords * 4;
constexpr int kSBBytes = kTile * 2 * 4;       // per row: 2 scales + 2 biases (fp16)
constexpr int kStages = 6;

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t u4_at(const uint4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// One chunk = 16 packed words of a row (128 elements at 4 bits, 64 at 8 bits).
// Thread (g, t) owns words 4t .. 4t+3 of the chunk for rows g and g+8.
// hblk: the chunk's block of the staged h row of token g.  For 4-bit heads the
// staged rows are swizzled: 16-byte chunk k of each 128-element block sits at
// position k ^ (2 * (k >> 3)), so the four threads of a quad (reading at a
// 64-byte stride) hit distinct bank groups.
template <int BITS>
__device__ __forceinline__ void chunk_mma(float (&acc)[4], const uint4& a0, const uint4& a1,
                                          uint32_t s0, uint32_t b0, uint32_t s1, uint32_t b1,
                                          const __half* hblk, int t) {
    if constexpr (BITS == 4) {
        const int sw = 2 * (t >> 1);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 bq = *reinterpret_cast<const uint4*>(hblk + 8 * ((4 * t + j) ^ sw));
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
            const uint4 bq = *reinterpret_cast<const uint4*>(hblk + 16 * t + 8 * jj);
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

// Shared memory: [h rows: 8 x (H + 8) halves] [packed ring] [scale/bias ring] [barriers]
struct StreamSmem {
    int off_p, off_sb, off_bar, total;
    __host__ __device__ StreamSmem(int H) {
        const int hbytes = kTokGroup * (H + 8) * 2;
        off_p = (hbytes + 127) / 128 * 128;
        off_sb = off_p + kStages * kPBytes;
        off_bar = off_sb + kStages * kSBBytes;
        total = off_bar + 8 * 2 * kStages + 16;
    }
};

template <int BITS>
__global__ void __launch_bounds__(kThreads, 2) stream_fwd_kernel(
    const __grid_constant__ CUtensorMap tmap_w, const __half* __restrict__ scales,
    const __half* __restrict__ biases, int64_t V, int H, float cap,
    const __half* __restrict__ h16, const int* __restrict__ count, Partial* __restrict__ part,
    int S, int* __restrict__ err, int stall) {
    const int n_active = *count;
    const int tok0 = blockIdx.x * kTokGroup;
    if (tok0 >= n_active) return;
    const int split = blockIdx.y;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    const StreamSmem L(H);
    __half* hs = reinterpret_cast<__half*>(smem_raw);
    const int hstride = H + 8;  // halves; +16 bytes per row spreads the banks
    unsigned char* pring = smem_raw + L.off_p;
    unsigned char* sbring = smem_raw + L.off_sb;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + L.off_bar);
    uint64_t* empty = full + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);
    __shared__ Partial red[kConsumers][kTokGroup];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t cta_v0 = V * split / S, cta_v1 = V * (split + 1) / S;
    const int ntiles = (int)((cta_v1 - cta_v0 + kTile - 1) / kTile);
    const int wpr = H * BITS / 32;
    const int G = H / 64;
    const int nchunks = wpr / kChunkWords;
    const int nitems = ntiles * nchunks;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&full[i], 1 + 32);  // TMA (expect_tx) + 32 cp.async arrivals
            tc::mbar_init(&empty[i], kConsumers);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tmap_w);
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        int stage = 0;
        uint32_t phase = 0, fills = 0;
        bool ok = stall == 0;  // test switch: issue no loads, the consumers' waits expire
        for (int k = 0; k < nitems && ok; ++k) {
            const int tile = k / nchunks, c = k - tile * nchunks;
            const int64_t row0 = cta_v0 + (int64_t)tile * kTile;
            if (lane == 0)
                ok = tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag, err, tc::kErrTimeoutEmpty);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                tc::mbar_arrive_expect_tx(&full[stage], kPBytes);
                tc::tma_load_2d(pring + stage * kPBytes, &tmap_w, &full[stage], kChunkWords * c,
                                (int)row0);
            }
            // Scales and biases of the stage: 2 consecutive groups per row (the
            // chunk's two groups at 4 bits; chunks c and c^1 at 8 bits).
            const int g0 = BITS == 4 ? 2 * c : (c & ~1);
            unsigned char* sb = sbring + stage * kSBBytes;
#pragma unroll
            for (int i = 0; i < kTile / 32; ++i) {
                const int r = lane + 32 * i;
                const int64_t v = row0 + r;
                const int64_t gi = (v < V ? v : 0) * G + g0;
                const int nbytes = v < V ? 4 : 0;
                tc::cp_async_zfill<4>(sb + 4 * r, scales + gi, nbytes);
                tc::cp_async_zfill<4>(sb + 4 * (kTile + r), biases + gi, nbytes);
            }
            tc::cp_async_arrive(&full[stage]);
            ++fills;
            if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        // On the abort path the consumers stop waiting: let the copies in
        // flight land before the CTA exits.
        if (!ok && lane == 0) tc::drain_ring(full, kStages, fills, err);
    } else {
        // ---------------------------------------------------------------- consumers
        const int cw = warp - 1;
        const int g = lane >> 2, t = lane & 3;
        // Stage the group's 8 rows of h (fp16, K-permuted for 4-bit), consumers only.
        const int units = H / 8;
        for (int idx = threadIdx.x - 32; idx < kTokGroup * units; idx += 32 * kConsumers) {
            const int r = idx / units, cc = idx - r * units;
            const uint4 v = *reinterpret_cast<const uint4*>(h16 + (int64_t)(tok0 + r) * H + 8 * cc);
            int pos = cc;
            if (BITS == 4) {
                const int k = cc & 15;
                pos = (cc & ~15) | (k ^ (2 * (k >> 3)));
            }
            *reinterpret_cast<uint4*>(hs + r * hstride + 8 * pos) = v;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");
        const __half* hrow = hs + g * hstride;
        constexpr int kChunkHalves = BITS == 4 ? 128 : 64;
        const int ra = 16 * cw + g, rb = ra + 8;  // rows of this thread within a tile
        // which of the stage's two groups this thread uses
        const int gsel_fixed = t >> 1;

        RowState st[2];
        st[0].init();
        st[1].init();
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = 0; tile < ntiles; ++tile) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int c = 0; c < nchunks; ++c) {
                // Result ignored: the warp stays converged (see the abort policy).
                tc::mbar_wait(&full[stage], phase, abort_flag, err, tc::kErrTimeoutFull);
                const unsigned char* P = pring + stage * kPBytes;
                const uint4 a0 = *reinterpret_cast<const uint4*>(P + ra * 64 + 16 * t);
                const uint4 a1 = *reinterpret_cast<const uint4*>(P + rb * 64 + 16 * t);
                const __half* sbh = reinterpret_cast<const __half*>(sbring + stage * kSBBytes);
                const int gsel = BITS == 4 ? gsel_fixed : (c & 1);
                const uint32_t s0 = bcast_h(sbh[2 * ra + gsel]);
                const uint32_t s1 = bcast_h(sbh[2 * rb + gsel]);
                const uint32_t b0 = bcast_h(sbh[2 * (kTile + ra) + gsel]);
                const uint32_t b1 = bcast_h(sbh[2 * (kTile + rb) + gsel]);
                chunk_mma<BITS>(acc, a0, a1, s0, b0, s1, b1, hrow + kChunkHalves * c, t);
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&empty[stage]);
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
            // acc: (row ra, tok 2t), (row ra, tok 2t+1), (row rb, tok 2t), (row rb, tok 2t+1)
            const int64_t v0 = cta_v0 + (int64_t)tile * kTile + ra, v1 = v0 + 8;
            if (v0 < cta_v1) {
                st[0].push(softcap_exact(acc[0], cap), acc[0], (int)v0);
                st[1].push(softcap_exact(acc[1], cap), acc[1], (int)v0);
            }
            if (v1 < cta_v1) {
                st[0].push(softcap_exact(acc[2], cap), acc[2], (int)v1);
                st[1].push(softcap_exact(acc[3], cap), acc[3], (int)v1);
            }
        }
        // Merge the 8 lanes that share t (lanes t, t+4, ..., t+28).
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
            st[0].shfl_merge(o);
            st[1].shfl_merge(o);
        }
        if (g == 0) {
            red[cw][2 * t] = st[0].to_partial();
            red[cw][2 * t + 1] = st[1].to_partial();
        }
    }
    __syncthreads();
    if (threadIdx.x < kTokGroup) {
        const int j = threadIdx.x;
        RowState acc;
        acc.init();
        for (int w = 0; w < kConsumers; ++w) acc.merge(red[w][j]);
        part[(int64_t)(tok0 + j) * S + split] = acc.to_partial();
    }
}

}  // namespace

int stream_fwd_ctas_per_sm(int bits, int H) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, int> cache;  // (device, bits, H) -> CTAs per SM
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find({dev, bits, H});
        if (it != cache.end()) return it->second;
    }
    const int smem = StreamSmem(H).total;
    const void* fn = bits == 4 ? reinterpret_cast<const void*>(stream_fwd_kernel<4>)
                               : reinterpret_cast<const void*>(stream_fwd_kernel<8>);
    int n = 0;
    cudaError_t e = ensure_smem_limit(fn, smem);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem);
    n = (e == cudaSuccess && n > 0) ? n : 1;
    std::lock_guard<std::mutex> lock(mu);
    cache[{dev, bits, H}] = n;
    return n;
}

cudaError_t launch_stream_fwd(const uint32_t* wq, const __half* scales, const __half* biases,
                              int64_t V, int H, int bits, float cap, const __half* h16,
                              const int* count, int64_t M, Partial* part, int S, int* err,
                              int stall, cudaStream_t st) {
    CUtensorMap tw;
    if (!tmap_packed_rows(&tw, wq, (uint64_t)H * bits / 32, (uint64_t)V, kChunkWords, kTile))
        return cudaErrorInvalidValue;
    const int groups = (int)((M + kTokGroup - 1) / kTokGroup);
    const int smem = StreamSmem(H).total;
    dim3 grid(groups, S);
    if (bits == 4) {
        if (cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(stream_fwd_kernel<4>), smem))
            return e;
        stream_fwd_kernel<4><<<grid, kThreads, smem, st>>>(tw, scales, biases, V, H, cap, h16,
                                                           count, part, S, err, stall);
    } else {
        if (cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(stream_fwd_kernel<8>), smem))
            return e;
        stream_fwd_kernel<8><<<grid, kThreads, smem, st>>>(tw, scales, biases, V, H, cap, h16,
                                                           count, part, S, err, stall);
    }
    return cudaGetLastError();
}

}  // namespace qh

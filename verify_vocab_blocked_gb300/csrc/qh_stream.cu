// qh_stream.cu -- weight-streaming forward (steps a2-a5 and a8 of the hot path
// for small M, where the tensor-core kernel's 128-row tiles would be mostly
// empty).
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
// How (GB300): at M = gamma+1 the cost is reading the packed head once, and
// the limit is the instruction issue rate, not the arithmetic: a per-element
// dequantization (w = s q + b) costs more issue slots than HBM leaves.  So the
// affine map is factored out of the inner product, per 64-element group g:
//     sum_k (s q_k + b) h_k = s (sum_k (M_k + q_k) h_k - sum_k M_k h_k) + b sum_k h_k
// The tensor core multiplies the codes still carrying their magic-exponent
// offset M_k (one lop3 per code pair, nothing else per element), the group's
// fp32 accumulator starts at -sum_k M_k h_k so the offset cancels inside it,
// one FFMA per accumulator applies s, and b sum_k h_k is a small MMA per tile
// (fp16 biases x an fp16 hi/lo split of the group sums of h).  Each CTA
// compacts the mask, converts its 8 rows of h to fp16 in shared memory and
// takes the group sums from those values while the first stages load, so the
// verify call needs no separate prologue kernel.  w itself is never
// rounded to fp16.
//
// A producer warp streams the CTA's vocab range through shared memory with
// TMA (128 rows x 16 packed words per stage, 6 stages) and copies each
// stage's scales with cp.async; eight consumer warps each take 16 of the 128
// rows as the A operand of mma.sync.m16n8k16 (A = 16 vocab rows x 16 K,
// B = 16 K x 8 tokens, fp32 accumulate).  Every mma covers one group: a
// thread's codes for one mma come from one packed word, and the four threads
// of a quad take adjacent words of the same group.
//   4-bit: word j of a row holds d = 8j .. 8j+7; lop3((w >> 8i) & 0x000F000F |
//          0x64006400) = fp16 pair (1024 + q_k, 1024 + q_k+4) (k even) and
//          (w >> 8i) & 0x00F000F0 | 0x54005400 = (64 + q_k, 64 + q_k+4) (k odd);
//          the staged h rows store each 8-block as (0,4,1,5,2,6,3,7).
//   8-bit: prmt builds (1024 + q_0, 1024 + q_1) and (1024 + q_2, 1024 + q_3).
// The row's logits never leave registers.
#include <map>
#include <mutex>
#include <tuple>

#include "qh_dequant.cuh"
#include "qh_tc.cuh"
#include "qh_tmap.h"

namespace qh {

namespace {

constexpr int kConsumers = 16;                // consumer warps, 16 rows each
constexpr int kThreads = 32 * (1 + kConsumers);
constexpr int kTile = 16 * kConsumers;        // vocab rows per stage
constexpr int kStageWords = 32;               // packed words per row per stage (128 bytes)
constexpr int kPBytes = kTile * kStageWords * 4;
constexpr int kSBytes = kTile * 8;            // per row: the stage's group scales (up to 4, fp16)
constexpr int kMaxStages = 6;
// Dynamic shared memory of one CTA: 227 KB less the static reduction buffer.
constexpr int kSmemLimit = 227 * 1024 - kConsumers * kTokGroup * (int)sizeof(Partial);

// D = A B + C with C given separately (starts a group's accumulator).
__device__ __forceinline__ void mma16816_init(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1, float c0,
                                              float c1, float c2, float c3) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2),
          "f"(c3));
}

// C += A B.
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The eight 4-bit codes of one word with their magic offsets, as fp16 pairs:
// p[0] = (1024 + q0, 1024 + q4), p[1] = (64 + q1, 64 + q5),
// p[2] = (1024 + q2, 1024 + q6), p[3] = (64 + q3, 64 + q7).
__device__ __forceinline__ void codes4(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t w8 = w >> 8;
    p[0] = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
    p[1] = lop3_and_or(w, 0x00F000F0u, 0x54005400u);
    p[2] = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);
    p[3] = lop3_and_or(w8, 0x00F000F0u, 0x54005400u);
}

// Two 8-bit codes of w with offset 1024: sel 0x5140 -> bytes 0, 1; 0x7362 -> 2, 3.
__device__ __forceinline__ uint32_t codes8(uint32_t w, uint32_t sel) {
    return __byte_perm(w, 0x64646464u, sel);
}

// Groups per stage, padded hidden size (whole stages; the pad is zero) and
// padded group count of the shared-memory tables.
template <int BITS>
struct StreamShape {
    static constexpr int kGroupsPerStage = kStageWords * 32 / BITS / 64;  // 4 (4-bit) or 2 (8-bit)
    static constexpr int kStagesPerKb = 16 / kGroupsPerStage;             // stages per 16 groups
};

// TMA-staged scales (fast variant): one box of kSBoxGroups groups x 256 rows
// (16-byte rows, the TMA minimum) holds the scales of kPer consecutive stages
// of a tile; kSlots such boxes are in flight (at least the 5 stages of the
// packed ring, whatever the tile's remainder).
constexpr int kSBoxGroups = 8;
constexpr int kSSlotBytes = kTile * kSBoxGroups * 2;
template <int BITS>
struct ScaleRing {
    static constexpr int kPer = kSBoxGroups / StreamShape<BITS>::kGroupsPerStage;  // 2 or 4
    static constexpr int kSlots = BITS == 4 ? 3 : 2;
};

// Per-thread byte offsets (within a stage) of the packed words a thread reads
// for each of the stage's groups: its A-fragment rows ra, rb, the swizzled
// 16-byte chunk, and (4-bit) the 8-byte half of it.
template <int BITS>
struct StageOffsets {
    static constexpr int NG = StreamShape<BITS>::kGroupsPerStage;
    int a[NG], b[NG];
    __device__ __forceinline__ StageOffsets(int ra, int rb, int t) {
#pragma unroll
        for (int gm = 0; gm < NG; ++gm) {
            if constexpr (BITS == 4) {
                // words 8 gm + 2t, +1: chunk 2 gm + (t >> 1), half t & 1
                const int j = 2 * gm + (t >> 1);
                a[gm] = ra * 128 + ((j ^ (ra & 7)) << 4) + 8 * (t & 1);
                b[gm] = rb * 128 + ((j ^ (rb & 7)) << 4) + 8 * (t & 1);
            } else {
                // words 16 gm + 4t .. +3: chunk 4 gm + t
                const int j = 4 * gm + t;
                a[gm] = ra * 128 + ((j ^ (ra & 7)) << 4);
                b[gm] = rb * 128 + ((j ^ (rb & 7)) << 4);
            }
        }
    }
};

// One stage of one warp: for each group of the stage, the group-pure mma
// chain on the magic-offset codes (accumulator started at -sum M_k h_k), then
// tot += scale * acc.  P: the stage's packed tile; sa2 / sb2: the stage's
// fp16 scales of rows ra / rb; ncs: negc of the stage's first group at tokens
// 2t, 2t+1; hst: this thread's h fragment base for the stage.
template <int BITS, int UNROLL4>
__device__ __forceinline__ void stage_math(float (&tot)[4], const unsigned char* P,
                                           const StageOffsets<BITS>& off, uint2 sa2, uint2 sb2,
                                           const float* ncs, const __half* hst) {
    if constexpr (BITS == 4) {
        const float2 sa01 = __half22float2(u32_as_h2(sa2.x)), sa23 = __half22float2(u32_as_h2(sa2.y));
        const float2 sb01 = __half22float2(u32_as_h2(sb2.x)), sb23 = __half22float2(u32_as_h2(sb2.y));
#pragma unroll UNROLL4
        for (int gm = 0; gm < 4; ++gm) {  // the stage's four groups
            // (select chains: a run-time index into off.a would put it in local memory)
            const int oa = gm == 0 ? off.a[0] : gm == 1 ? off.a[1] : gm == 2 ? off.a[2] : off.a[3];
            const int ob = gm == 0 ? off.b[0] : gm == 1 ? off.b[1] : gm == 2 ? off.b[2] : off.b[3];
            const uint2 wa = *reinterpret_cast<const uint2*>(P + oa);
            const uint2 wb = *reinterpret_cast<const uint2*>(P + ob);
            const float2 nc = *reinterpret_cast<const float2*>(ncs + gm * kTokGroup);
            const uint4 q0 = *reinterpret_cast<const uint4*>(hst + 64 * gm);
            const uint4 q1 = *reinterpret_cast<const uint4*>(hst + 64 * gm + 8);
            uint32_t pa[4], pb[4];
            float acc[4];
            codes4(wa.x, pa);
            codes4(wb.x, pb);
            mma16816_init(acc, pa[0], pb[0], pa[1], pb[1], q0.x, q0.y, nc.x, nc.y, nc.x, nc.y);
            mma16816(acc, pa[2], pb[2], pa[3], pb[3], q0.z, q0.w);
            codes4(wa.y, pa);
            codes4(wb.y, pb);
            mma16816(acc, pa[0], pb[0], pa[1], pb[1], q1.x, q1.y);
            mma16816(acc, pa[2], pb[2], pa[3], pb[3], q1.z, q1.w);
            const float s_a = gm == 0 ? sa01.x : gm == 1 ? sa01.y : gm == 2 ? sa23.x : sa23.y;
            const float s_b = gm == 0 ? sb01.x : gm == 1 ? sb01.y : gm == 2 ? sb23.x : sb23.y;
            tot[0] = fmaf(s_a, acc[0], tot[0]);
            tot[1] = fmaf(s_a, acc[1], tot[1]);
            tot[2] = fmaf(s_b, acc[2], tot[2]);
            tot[3] = fmaf(s_b, acc[3], tot[3]);
        }
    } else {
        const float2 sa01 = __half22float2(u32_as_h2(sa2.x));
        const float2 sb01 = __half22float2(u32_as_h2(sb2.x));
#pragma unroll 1
        for (int gm = 0; gm < 2; ++gm) {  // the stage's two groups
            const uint4 wa = *reinterpret_cast<const uint4*>(P + (gm ? off.a[1] : off.a[0]));
            const uint4 wb = *reinterpret_cast<const uint4*>(P + (gm ? off.b[1] : off.b[0]));
            const float2 nc = *reinterpret_cast<const float2*>(ncs + gm * kTokGroup);
            const uint4 q0 = *reinterpret_cast<const uint4*>(hst + 64 * gm);
            const uint4 q1 = *reinterpret_cast<const uint4*>(hst + 64 * gm + 8);
            float acc[4];
            mma16816_init(acc, codes8(wa.x, 0x5140u), codes8(wb.x, 0x5140u), codes8(wa.x, 0x7362u),
                          codes8(wb.x, 0x7362u), q0.x, q0.y, nc.x, nc.y, nc.x, nc.y);
            mma16816(acc, codes8(wa.y, 0x5140u), codes8(wb.y, 0x5140u), codes8(wa.y, 0x7362u),
                     codes8(wb.y, 0x7362u), q0.z, q0.w);
            mma16816(acc, codes8(wa.z, 0x5140u), codes8(wb.z, 0x5140u), codes8(wa.z, 0x7362u),
                     codes8(wb.z, 0x7362u), q1.x, q1.y);
            mma16816(acc, codes8(wa.w, 0x5140u), codes8(wb.w, 0x5140u), codes8(wa.w, 0x7362u),
                     codes8(wb.w, 0x7362u), q1.z, q1.w);
            const float s_a = gm ? sa01.y : sa01.x, s_b = gm ? sb01.y : sb01.x;
            tot[0] = fmaf(s_a, acc[0], tot[0]);
            tot[1] = fmaf(s_a, acc[1], tot[1]);
            tot[2] = fmaf(s_b, acc[2], tot[2]);
            tot[3] = fmaf(s_b, acc[3], tot[3]);
        }
    }
}

// Shared memory (1024-byte aligned base): [packed ring: stages x 32 KB, 128B
// swizzle] [scale ring: per stage 256 x 8 bytes, or with TMA-staged scales
// kSlots boxes of 256 x 16 bytes] [h rows: 8 x (Hp + 8) halves] [negc: Gs x 8
// fp32] [hsum hi: 8 x gp fp16] [hsum lo: 8 x gp fp16] [barriers].  One CTA
// per SM: the stage count is the largest that fits (more bytes in flight).
struct StreamSmem {
    int stages, sslots, Hp, Gs, gp, off_s, off_h, off_negc, off_hs, off_bar, total;
    __host__ __device__ StreamSmem(int H, int bits, int n_stages, bool tma_scales) {
        const int per_stage = kStageWords * 32 / bits;      // hidden elements per stage
        Hp = (H + per_stage - 1) / per_stage * per_stage;
        Gs = Hp / 64;
        gp = (H / 64 + 15) / 16 * 16;  // groups padded to whole 16-wide k-blocks
        stages = n_stages;
        sslots = tma_scales ? (bits == 4 ? ScaleRing<4>::kSlots : ScaleRing<8>::kSlots) : 0;
        off_s = stages * kPBytes;
        off_h = off_s + (tma_scales ? sslots * kSSlotBytes : stages * kSBytes);
        off_negc = off_h + (kTokGroup * (Hp + 8) * 2 + 15) / 16 * 16;
        off_hs = off_negc + Gs * kTokGroup * 4;
        off_bar = (off_hs + 2 * kTokGroup * gp * 2 + 7) / 8 * 8;
        total = off_bar + 8 * 2 * (stages + sslots) + 16 + 1024;  // + alignment slack of the base
    }
};

// The deepest ring that fits next to the staged h rows (0 if not even two).
int stream_stages(int H, int bits) {
    for (int s = kMaxStages; s >= 2; --s)
        if (StreamSmem(H, bits, s, false).total <= kSmemLimit) return s;
    return 0;
}

// The per-tile push of a consumer thread's four logits: the soft cap and the
// online-softmax update in their approximate forms (ex2.approx, rcp.approx;
// relative error ~1e-7, far inside the lse tolerance), ~50 fewer instructions
// per push than tanhf / expf (the kernel is issue-bound: 80.0 -> 75.0 us per
// verify window).  The finalize recomputes the target logit and rechecks the
// argmax candidates with the accurate forms.
__device__ __forceinline__ float softcap_fast(float raw, float cap2l, float cap) {
    // cap * tanh(raw / cap) = cap - 2 cap / (exp(2 raw / cap) + 1)
    return cap > 0.f ? fmaf(-2.f * cap, tc::rcp_approx(tc::ex2_approx(raw * cap2l) + 1.f), cap)
                     : raw;
}

__device__ __forceinline__ void push_fast(RowState& st, float z, float raw, int idx) {
    constexpr float kL2e = 1.4426950408889634f;
    if (z > st.m) {
        st.s = fmaf(st.s, tc::ex2_approx((st.m - z) * kL2e), 1.f);
        st.m = z;
    } else {
        st.s += tc::ex2_approx((z - st.m) * kL2e);
    }
    if (better(raw, idx, st.v1, st.i1)) { st.v2 = st.v1; st.i2 = st.i1; st.v1 = raw; st.i1 = idx; }
    else if (better(raw, idx, st.v2, st.i2)) { st.v2 = raw; st.i2 = idx; }
}

// NST > 0: the ring has NST stages and NST divides the stages of a tile, so
// each round of NST stages uses compile-time ring slots (immediate shared
// offsets), and the scales arrive by TMA (tmap_s; the group count is a
// multiple of 8); NST == 0: n_stages at run time, any shape, scales copied
// with cp.async (tmap_s unused).
template <int BITS, int NST>
__global__ void __launch_bounds__(kThreads, 1) stream_fwd_kernel(
    const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
    const __half* __restrict__ scales,
    const __half* __restrict__ biases, int64_t V, int H, float cap,
    const __nv_bfloat16* __restrict__ h, const uint8_t* __restrict__ mask, int M,
    int* __restrict__ rows, int* __restrict__ pos, int* __restrict__ count,
    Partial* __restrict__ part, int S, int* __restrict__ err, int stall, int n_stages) {
    using Shape = StreamShape<BITS>;
    // Launched as a programmatic dependent: nothing in global memory is
    // touched before the preceding grid on the stream has completed; the
    // finalize that follows may then start its CTAs (they wait for this grid).
    tc::grid_dep_wait();
    tc::grid_dep_trigger();
    // Compaction of the (at most 63) rows, by every warp for itself: bit j of
    // (act1:act0) marks row j active; compact index = rank among active rows.
    const int lane_c = threadIdx.x & 31;
    const unsigned act0 =
        __ballot_sync(0xffffffffu, lane_c < M && (mask == nullptr || mask[lane_c] != 0));
    const unsigned act1 =
        __ballot_sync(0xffffffffu, lane_c + 32 < M && (mask == nullptr || mask[lane_c + 32] != 0));
    const int n_active = __popc(act0) + __popc(act1);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 32) {
        // One CTA publishes the maps and clears the error word for the finalize.
        for (int r = lane_c; r < kRowPad; r += 32) {
            if (r < M) {
                const bool a = r < 32 ? (act0 >> r) & 1u : (act1 >> (r - 32)) & 1u;
                const int idx = r < 32 ? __popc(act0 & ((1u << r) - 1u))
                                       : __popc(act0) + __popc(act1 & ((1u << (r - 32)) - 1u));
                pos[r] = a ? idx : -1;
                if (a) rows[idx] = r;
            }
            if (r >= n_active) rows[r] = -1;
        }
        if (lane_c == 0) {
            *count = n_active;
            *err = 0;
        }
    }
    const int tok0 = blockIdx.x * kTokGroup;
    if (tok0 >= n_active) return;
    const int split = blockIdx.y;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    // (offsetting the shared array itself keeps the accesses in the shared
    // address space; a round trip through an integer would make them generic)
    constexpr bool kTmaScales = NST > 0;
    constexpr int kSPer = ScaleRing<BITS>::kPer;
    constexpr int kSSlots = kTmaScales ? ScaleRing<BITS>::kSlots : 0;
    const StreamSmem L(H, BITS, NST > 0 ? NST : n_stages, kTmaScales);
    const int kStages = L.stages;
    unsigned char* pring = smem;
    unsigned char* sring = smem + L.off_s;
    __half* hs = reinterpret_cast<__half*>(smem + L.off_h);
    const int hstride = L.Hp + 8;  // halves; +16 bytes per row spreads the banks
    float* negc_s = reinterpret_cast<float*>(smem + L.off_negc);
    __half* hs_hi = reinterpret_cast<__half*>(smem + L.off_hs);
    __half* hs_lo = hs_hi + kTokGroup * L.gp;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_bar);
    uint64_t* empty = full + kStages;
    uint64_t* sfull = empty + kStages;  // TMA-staged scales: box landed
    uint64_t* sempty = sfull + kSSlots;  // box consumed by every consumer warp
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sempty + kSSlots);
    __shared__ Partial red[kConsumers][kTokGroup];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t cta_v0 = V * split / S, cta_v1 = V * (split + 1) / S;
    const int ntiles = (int)((cta_v1 - cta_v0 + kTile - 1) / kTile);
    const int G = H / 64;
    const int nst = L.Gs / Shape::kGroupsPerStage;  // stages per tile
    const int nitems = ntiles * nst;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            // TMA (expect_tx), plus 32 cp.async arrivals when the scales ride along
            tc::mbar_init(&full[i], kTmaScales ? 1 : 1 + 32);
            tc::mbar_init(&empty[i], kConsumers);
        }
        for (int i = 0; i < kSSlots; ++i) {
            tc::mbar_init(&sfull[i], 1);
            tc::mbar_init(&sempty[i], kConsumers);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tmap_w);
        if (kTmaScales) tc::prefetch_tmap(&tmap_s);
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        int stage = 0, sslot = 0;
        uint32_t phase = 0, fills = 0, sphase = 0, sfills = 0;
        bool ok = stall == 0;  // test switch: issue no loads, the consumers' waits expire
        for (int k = 0; k < nitems && ok; ++k) {
            const int tile = k / nst, c = k - tile * nst;
            const int64_t row0 = cta_v0 + (int64_t)tile * kTile;
            if (lane == 0)
                ok = tc::mbar_wait_cta(&empty[stage], phase ^ 1, abort_flag, err, tc::kErrTimeoutEmpty);
            if (kTmaScales && lane == 0 && ok && c % kSPer == 0) {
                // The scales of stages c .. c + kSPer - 1: groups kSBoxGroups * (c / kSPer)
                // onward of the tile's 256 rows (rows past V read as zero).
                ok = tc::mbar_wait_cta(&sempty[sslot], sphase ^ 1, abort_flag, err,
                                       tc::kErrTimeoutEmpty);
                if (ok) {
                    tc::mbar_arrive_expect_tx(&sfull[sslot], kSSlotBytes);
                    tc::tma_load_2d(sring + sslot * kSSlotBytes, &tmap_s, &sfull[sslot],
                                    kSBoxGroups * (c / kSPer), (int)row0);
                    ++sfills;
                    if (++sslot == kSSlots) { sslot = 0; sphase ^= 1; }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                // Words past the row end (4-bit, H not a multiple of 256) read as zero.
                tc::mbar_arrive_expect_tx(&full[stage], kPBytes);
                tc::tma_load_2d(pring + stage * kPBytes, &tmap_w, &full[stage], kStageWords * c,
                                (int)row0);
            }
            if constexpr (!kTmaScales) {
            // The stage's scales, two groups per 4-byte copy (zeros past G or V).
            const int g0 = Shape::kGroupsPerStage * c;
            unsigned char* sd = sring + stage * kSBytes;
#pragma unroll
            for (int i = 0; i < kTile / 32; ++i) {
                const int r = lane + 32 * i;
                const int64_t v = row0 + r;
                const int64_t vb = (v < V ? v : 0) * G;
#pragma unroll
                for (int q = 0; q < Shape::kGroupsPerStage / 2; ++q) {
                    const int gq = g0 + 2 * q;
                    tc::cp_async_zfill<4>(sd + 8 * r + 4 * q, scales + vb + (gq < G ? gq : 0),
                                          v < V && gq < G ? 4 : 0);
                }
            }
            tc::cp_async_arrive(&full[stage]);
            }
            ++fills;
            if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        // On the abort path the consumers stop waiting: let the copies in
        // flight land before the CTA exits.
        if (!ok && lane == 0) {
            tc::drain_ring(full, kStages, fills, err);
            if (kTmaScales) tc::drain_ring(sfull, kSSlots, sfills, err);
        }
    } else {
        // ---------------------------------------------------------------- consumers
        const int cw = warp - 1;
        const int g = lane >> 2, t = lane & 3;
        const int ct = threadIdx.x - 32;
        // Stage the group's 8 rows of h as fp16 (8-element blocks in the order
        // (0,4,1,5,2,6,3,7) for 4-bit heads, matching the pairs codes4 yields;
        // zeros past the active rows and in [H, Hp)), consumers only.
        __shared__ int orig_s[kTokGroup];
        if (ct < kTokGroup) {
            int row = -1, k = tok0 + ct;  // compact index -> original row
            if (k < n_active) {
                for (int r = 0; r < M; ++r) {
                    const bool a = r < 32 ? (act0 >> r) & 1u : (act1 >> (r - 32)) & 1u;
                    if (a && k-- == 0) { row = r; break; }
                }
            }
            orig_s[ct] = row;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");
        const int units = L.Hp / 8;
        for (int idx = ct; idx < kTokGroup * units; idx += 32 * kConsumers) {
            const int r = idx / units, cc = idx - r * units;
            const int row = orig_s[r];
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (row >= 0 && 8 * cc < H) {
                const uint4 in = *reinterpret_cast<const uint4*>(h + (int64_t)row * H + 8 * cc);
                const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&in);
                __half y[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    y[k] = __float2half_rn(__bfloat162float(x[BITS == 4 ? ((k & 1) * 4 + (k >> 1)) : k]));
                v = *reinterpret_cast<const uint4*>(y);
            }
            *reinterpret_cast<uint4*>(hs + r * hstride + 8 * cc) = v;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");
        // Group statistics of the staged fp16 rows (exactly what the mma sees):
        // negc = -sum_k M_k h_k (M_k = 1024 for even k, 64 for odd k at 4 bits,
        // 1024 at 8 bits) and hsum = sum_k h_k as an fp16 (hi, lo) pair.  Eight
        // lanes per (row, group), one 8-element block each, compensated sums
        // combined exactly across the lanes.
        {
            const int npair = kTokGroup * L.gp;
            const int ntask = npair * 8;
            for (int task0 = 0; task0 < ntask; task0 += 32 * kConsumers) {  // uniform trip count
                const int task = task0 + ct;
                const int pr = task >> 3, sub = task & 7;
                const int r = pr / L.gp, gg = pr - r * L.gp;
                float es = 0.f, ec = 0.f, os = 0.f, oc = 0.f;
                if (task < ntask && gg < L.Gs) {
                    const uint4 in = *reinterpret_cast<const uint4*>(hs + r * hstride + 64 * gg + 8 * sub);
                    const __half* y = reinterpret_cast<const __half*>(&in);
#pragma unroll
                    for (int p = 0; p < 8; ++p) {
                        // natural element index parity of staged position p
                        const bool even = BITS == 4 ? (p & 2) == 0 : (p & 1) == 0;
                        const float xv = __half2float(y[p]);
                        float e, sum;
                        if (even) { sum = es + xv; const float bb = sum - es; e = (es - (sum - bb)) + (xv - bb); es = sum; ec += e; }
                        else      { sum = os + xv; const float bb = sum - os; e = (os - (sum - bb)) + (xv - bb); os = sum; oc += e; }
                    }
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    const float es2 = __shfl_xor_sync(0xffffffffu, es, o);
                    const float ec2 = __shfl_xor_sync(0xffffffffu, ec, o);
                    const float os2 = __shfl_xor_sync(0xffffffffu, os, o);
                    const float oc2 = __shfl_xor_sync(0xffffffffu, oc, o);
                    float sum = es + es2, bb = sum - es;
                    ec += ec2 + ((es - (sum - bb)) + (es2 - bb));
                    es = sum;
                    sum = os + os2; bb = sum - os;
                    oc += oc2 + ((os - (sum - bb)) + (os2 - bb));
                    os = sum;
                }
                if (task < ntask && sub == 0) {
                    const float me = 1024.f, mo = BITS == 4 ? 64.f : 1024.f;
                    if (gg < L.Gs) negc_s[gg * kTokGroup + r] = -((me * es + mo * os) + (me * ec + mo * oc));
                    const float hsv = gg < G ? (es + os) + (ec + oc) : 0.f;
                    const __half hi = __float2half_rn(hsv);
                    hs_hi[pr] = hi;
                    hs_lo[pr] = __float2half_rn(hsv - __half2float(hi));
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");
        const __half* hrow = hs + g * hstride;
        // Physical rows of this thread's A-fragment rows g and g + 8, chosen so
        // that the packed loads of a quarter- (8-bit) or half-warp (4-bit) hit
        // distinct 16-byte chunks under the 128-byte swizzle.
        const int ra = BITS == 4 ? 16 * cw + 2 * g : 16 * cw + (g >> 1) + 4 * (g & 1);
        const int rb = BITS == 4 ? ra + 1 : ra + 8;
        const StageOffsets<BITS> off(ra, rb, t);
        const int nkb = L.gp / 16;
        constexpr int kPer = Shape::kStagesPerKb;
        constexpr int kNG = Shape::kGroupsPerStage;
        // This thread's h fragments of stage c start at half 32 c * (32 / BITS)
        // + 16 t of token g's row (words 2t.. of each 4-bit group, words 4t..
        // of each 8-bit group).
        const __half* hbase = hrow + 16 * t;

        RowState st[2];
        st[0].init();
        st[1].init();
        int stage = 0, cs = 0;  // packed ring slot; scale box slot (fast variant)
        uint32_t phase = 0, csphase = 0;
        for (int tile = 0; tile < ntiles; ++tile) {
            const int64_t va = cta_v0 + (int64_t)tile * kTile + ra;
            const int64_t vb = cta_v0 + (int64_t)tile * kTile + rb;
            // tot: (row ra, tok 2t), (row ra, tok 2t+1), (row rb, tok 2t), (row rb, tok 2t+1)
            float tot[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t bA[4] = {0u, 0u, 0u, 0u};  // biases of the pending k-block (A fragment)
            // sum_g b[v, g] hsum[tok, g] for k-block kb: fp16 biases x (hi + lo) sums.
            auto load_bias = [&](int kb) {
                const int k0 = 16 * kb + 2 * t;
                const bool oa = va < cta_v1, ob = vb < cta_v1;
                bA[0] = oa && k0 < G ? *reinterpret_cast<const uint32_t*>(biases + va * G + k0) : 0u;
                bA[1] = ob && k0 < G ? *reinterpret_cast<const uint32_t*>(biases + vb * G + k0) : 0u;
                bA[2] = oa && k0 + 8 < G ? *reinterpret_cast<const uint32_t*>(biases + va * G + k0 + 8) : 0u;
                bA[3] = ob && k0 + 8 < G ? *reinterpret_cast<const uint32_t*>(biases + vb * G + k0 + 8) : 0u;
            };
            auto bias_mma = [&](int kb) {
                const int k0 = g * L.gp + 16 * kb + 2 * t;
                mma16816(tot, bA[0], bA[1], bA[2], bA[3],
                         *reinterpret_cast<const uint32_t*>(hs_hi + k0),
                         *reinterpret_cast<const uint32_t*>(hs_hi + k0 + 8));
                mma16816(tot, bA[0], bA[1], bA[2], bA[3],
                         *reinterpret_cast<const uint32_t*>(hs_lo + k0),
                         *reinterpret_cast<const uint32_t*>(hs_lo + k0 + 8));
            };
            auto bias_step = [&](int c) {
                if ((c & (kPer - 1)) == 0) load_bias(c / kPer);
                if ((c & (kPer - 1)) == kPer / 2) bias_mma(c / kPer);
            };
            if constexpr (NST > 0) {
                // Rounds of NST stages: ring slot s of every round is stage s.
                for (int c0 = 0; c0 < nst; c0 += NST) {
#pragma unroll
                    for (int s = 0; s < NST; ++s) {
                        const int c = c0 + s;
                        bias_step(c);
                        const int cq = c % kSPer;  // this stage's part of the scale box
                        // Results ignored: the warp stays converged (see the abort policy).
                        if (cq == 0)
                            tc::mbar_wait_cta(&sfull[cs], csphase, abort_flag, err, tc::kErrTimeoutFull);
                        tc::mbar_wait_cta(&full[s], phase, abort_flag, err, tc::kErrTimeoutFull);
                        // Box row r: kSBoxGroups scales; this stage's kNG start at group kNG * cq.
                        const unsigned char* Sb = sring + cs * kSSlotBytes + 2 * kNG * cq;
                        uint2 sa, sb;
                        if constexpr (BITS == 4) {
                            sa = *reinterpret_cast<const uint2*>(Sb + 16 * ra);
                            sb = *reinterpret_cast<const uint2*>(Sb + 16 * rb);
                        } else {
                            sa = make_uint2(*reinterpret_cast<const uint32_t*>(Sb + 16 * ra), 0u);
                            sb = make_uint2(*reinterpret_cast<const uint32_t*>(Sb + 16 * rb), 0u);
                        }
                        stage_math<BITS, 4>(tot, pring + s * kPBytes, off, sa, sb,
                                         negc_s + kNG * c * kTokGroup + 2 * t,
                                         hbase + kStageWords * c * (32 / BITS));
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&empty[s]);
                        if (cq == kSPer - 1 || c == nst - 1) {
                            if (lane == 0) tc::mbar_arrive(&sempty[cs]);
                            if (++cs == kSSlots) { cs = 0; csphase ^= 1; }
                        }
                    }
                    phase ^= 1;
                }
            } else {
                for (int c = 0; c < nst; ++c) {
                    bias_step(c);
                    // Result ignored: the warp stays converged (see the abort policy).
                    tc::mbar_wait_cta(&full[stage], phase, abort_flag, err, tc::kErrTimeoutFull);
                    const unsigned char* Sst = sring + stage * kSBytes;
                    stage_math<BITS, 2>(tot, pring + stage * kPBytes, off,
                                     *reinterpret_cast<const uint2*>(Sst + 8 * ra),
                                     *reinterpret_cast<const uint2*>(Sst + 8 * rb),
                                     negc_s + kNG * c * kTokGroup + 2 * t,
                                     hbase + kStageWords * c * (32 / BITS));
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&empty[stage]);
                    if (++stage == kStages) { stage = 0; phase ^= 1; }
                }
            }
            // The last k-block's bias product, if its slot fell past the stages.
            if (kPer * (nkb - 1) + kPer / 2 >= nst) bias_mma(nkb - 1);
            // (computed here, not held across the tile loop: one register fewer)
            const float cap2l = cap > 0.f ? 2.f * 1.4426950408889634f / cap : 0.f;
            if (va < cta_v1) {
                push_fast(st[0], softcap_fast(tot[0], cap2l, cap), tot[0], (int)va);
                push_fast(st[1], softcap_fast(tot[1], cap2l, cap), tot[1], (int)va);
            }
            if (vb < cta_v1) {
                push_fast(st[0], softcap_fast(tot[2], cap2l, cap), tot[2], (int)vb);
                push_fast(st[1], softcap_fast(tot[3], cap2l, cap), tot[3], (int)vb);
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
        Partial p = acc.to_partial();
        p.status = *abort_flag;
        part[(int64_t)(tok0 + j) * S + split] = p;
    }
}

}  // namespace

namespace {

// Ring depth of the fast variant (compile-time ring slots).
constexpr int kFastStages = 5;

// Kernel variant for (bits, H): the fast one when its ring fits and divides
// the stages of a tile, else the run-time-depth one.
struct StreamVariant {
    const void* fn;
    int n_stages;
    bool tma_scales;
    int smem;
};

StreamVariant stream_variant(int bits, int H) {
    const int per_stage = kStageWords * 32 / bits;
    const int nst = (H + per_stage - 1) / per_stage;  // stages per tile
    StreamVariant v{};
    // The fast variant stages the scales by TMA: 16-byte rows of the scale
    // table (groups a multiple of 8).
    if (nst % kFastStages == 0 && (H / 64) % kSBoxGroups == 0 &&
        StreamSmem(H, bits, kFastStages, true).total <= kSmemLimit) {
        v.fn = bits == 4 ? reinterpret_cast<const void*>(stream_fwd_kernel<4, kFastStages>)
                         : reinterpret_cast<const void*>(stream_fwd_kernel<8, kFastStages>);
        v.n_stages = kFastStages;
        v.tma_scales = true;
    } else {
        v.fn = bits == 4 ? reinterpret_cast<const void*>(stream_fwd_kernel<4, 0>)
                         : reinterpret_cast<const void*>(stream_fwd_kernel<8, 0>);
        v.n_stages = stream_stages(H, bits);
    }
    v.smem = v.n_stages >= 2 ? StreamSmem(H, bits, v.n_stages, v.tma_scales).total : 0;
    return v;
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
    const StreamVariant v = stream_variant(bits, H);
    int n = 0;
    cudaError_t e = v.smem > 0 ? ensure_smem_limit(v.fn, v.smem) : cudaErrorInvalidValue;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, v.fn, kThreads, v.smem);
    n = (e == cudaSuccess && n > 0) ? n : 1;
    std::lock_guard<std::mutex> lock(mu);
    cache[{dev, bits, H}] = n;
    return n;
}

cudaError_t launch_stream_fwd(const uint32_t* wq, const __half* scales, const __half* biases,
                              int64_t V, int H, int bits, float cap, const __nv_bfloat16* h,
                              const uint8_t* mask, int64_t M, int* rows, int* pos, int* count,
                              Partial* part, int S, int* err, int stall, cudaStream_t st) {
    if (M >= 64) return cudaErrorInvalidValue;  // the in-kernel compaction covers 64 rows
    CUtensorMap tw;
    if (!tmap_packed_rows_sw128(&tw, wq, (uint64_t)H * bits / 32, (uint64_t)V, kTile))
        return cudaErrorInvalidValue;
    const int groups = (int)((M + kTokGroup - 1) / kTokGroup);
    const StreamVariant v = stream_variant(bits, H);
    if (v.n_stages < 2) return cudaErrorInvalidValue;
    CUtensorMap ts{};  // unused by the run-time-depth variant
    if (v.tma_scales &&
        !tmap_group_rows(&ts, scales, (uint64_t)H / 64, (uint64_t)V, kSBoxGroups, kTile))
        return cudaErrorInvalidValue;
    if (cudaError_t e = ensure_smem_limit(v.fn, v.smem)) return e;
    dim3 grid(groups, S);
    int n_stages = v.n_stages;
    int m32 = (int)M;
    void* args[] = {&tw,  &ts,   &scales, &biases, &V, &H,   &cap,   &h,       &mask,
                    &m32, &rows, &pos,    &count,  &part, &S, &err, &stall, &n_stages};
    return launch_dependent(v.fn, grid, dim3(kThreads), (size_t)v.smem, st, args);
}

}  // namespace qh

// qh_tc_dh.cu -- tensor-core backward contraction (step a10 of the hot path).
//
// For one vocab chunk [v_begin, v_begin + 64 * n_k):
//     dh_acc[i, :] (+)= (-dlogp[row_i] * 2^-14) * sum_k C[i, k] * w[v_begin + k, :]
// where C = p * sech2 * 2^14 (fp16) is the coefficient block phase 1 wrote.
// This is phase 2 of the backward on the page "mlx-bun 0.0.4 -> 0.0.6"
// (src/train/flash-cce.ts, BWD_STEEL_SOURCE: dh[8,H] += coeff[8,32] @ W[32,H]),
// as a tcgen05 GEMM: M = 128 token rows, N = 256 (or 128) hidden columns,
// K = the chunk's vocab rows.  The coefficient tile arrives by TMA (K-major,
// 128-byte swizzle); the weight tile is dequantized from its packed rows into
// the MN-major 128-byte-swizzled layout (hidden index contiguous), so the same
// packed rows the forward reads serve here without a transpose.  Each output
// tile is owned by one CTA and accumulated over the chunks in a fixed order:
// the result is deterministic.
//
// The approximate backwards skip K steps (64 vocab rows) whose coefficients
// all count as zero: by the blockMax early exit's map of (128-row tile, vocab
// tile) pairs, or by the coefficient filter's bits per (256-row unit, step)
// that phase 1 leaves set (the skip kind is a template parameter, so the
// exact backward carries no skip logic).
#include <type_traits>

#include "qh_dequant.cuh"
#include "qh_tc.cuh"
#include "qh_tmap.h"

namespace qh {

namespace {

constexpr int BM = 128;   // token rows per MMA (M); a unit covers two halves
constexpr int BMU = 2 * BM;
constexpr int BK = 64;    // vocab rows per stage
// Dequantized-tile stages: as many as input stages for 4-bit heads, so that
// the two rings are one (a stage's B slot is freed with its inputs: the
// dequant warps wait for the inputs alone and the MMA thread commits once per
// step); 8-bit heads, whose packed tiles are twice as large, keep a shorter
// B ring of their own.
template <int BITS, int BNH>
constexpr int dh_nb() { return BITS == 4 ? (BNH == 256 ? 3 : 4) : 2; }
constexpr int kDqWarps = 8;             // warps 2 .. 9 dequantize
constexpr int kDqThreads = 32 * kDqWarps;
constexpr int kEpiWarp0 = 2 + kDqWarps; // warps 10 .. 13 run the epilogue
constexpr int kThreads = 32 * (kEpiWarp0 + 4);

// Two rings: NS stages of TMA inputs (two 128-row coefficient tiles + packed
// tile), NB stages of dequantized weight tiles.  Each dequantized tile feeds
// the MMAs of both 128-row halves of the unit, so a weight tile is
// dequantized once per 256 token rows.
template <int BITS, int BNH>
struct DhLayout {
    static constexpr int NS = BNH == 256 ? 3 : 4;
    static constexpr int NB = dh_nb<BITS, BNH>();
    static constexpr bool ONE_RING = NB == NS;
    static constexpr int A_BYTES = 2 * BM * BK * 2;         // coeff tiles of both halves, K-major SW128
    static constexpr int A_HALF = BM * BK * 2;
    static constexpr int B_BYTES = BNH * BK * 2;            // weight tile, MN-major SW128
    static constexpr int P_ROW = BNH * BITS / 8;            // packed bytes per vocab row
    static constexpr int P_BYTES = BK * P_ROW;
    static constexpr int WORDS = BNH * BITS / 32;           // TMA box width (words)
    static constexpr int OFF_B = 0;                         // B first: descriptor reach stays inside
    static constexpr int NSB = BNH / 64;                     // groups of the N tile
    static constexpr int SB_BYTES = 2 * BK * NSB * 2;        // scales + biases per stage
    static constexpr int OFF_A = OFF_B + NB * B_BYTES;
    static constexpr int OFF_P = OFF_A + NS * A_BYTES;
    static constexpr int OFF_SB = OFF_P + NS * P_BYTES;
    static constexpr int OFF_BAR = OFF_SB + NS * SB_BYTES;
    static constexpr int BAR_BYTES = 8 * (2 * NS + 2 * NB + 4) + 16;
    static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static constexpr int TMEM_COLS = 2 * BNH;               // the two halves' accumulators
    // Dequant work split: a packed row is PIECES 16-byte pieces; thread t takes
    // piece t % PIECES of rows t / PIECES + RPP * pass.
    static constexpr int PIECES = P_ROW / 16;
    static constexpr int RPP = kDqThreads / PIECES;
    static constexpr int PASSES = BK / RPP;
    static constexpr int CPP = 128 / BITS;        // hidden columns per piece (32 or 16)
    static constexpr int CHUNKS = CPP / 8;        // 16-byte output chunks per piece
    // Packed rows of 128 or 256 bytes arrive as 128-byte-swizzled halves
    // [half][64 rows][128 B] (chunk j of row r at j ^ (r & 7)), and each 8-lane
    // phase of a dequant warp takes 8 consecutive vocab rows of one piece, so
    // that its 16-byte loads and its stores into the swizzled B tile hit 8
    // distinct bank groups; 64-byte rows keep the unswizzled layout with the
    // 8 pieces of one row per phase.
    static constexpr bool SWZ = P_ROW >= 128;
    static constexpr int HALVES = P_ROW / 128;
    static constexpr uint32_t IDESC = tc::idesc_f16_f32(BM, BNH, false, true);
};

// A 4-bit word dequantizes to the fp16 pairs (q0,q4), (q1,q5), (q2,q6),
// (q3,q7) (qh_dequant.cuh).  Here the hidden axis is the MMA's N axis, so the
// B tile keeps that order -- N position c of an 8-column block holds hidden
// column kPerm4[c] -- and the epilogue, which holds 32 consecutive N columns
// per thread in registers, writes column c to hidden offset kPerm4[c].  8-bit
// words dequantize in natural order.
__device__ __forceinline__ uint4 deq4_chunk(uint32_t w, __half2 s, __half2 b) {
    uint32_t p[4];
    deq4_word(w, s, b, p);
    return make_uint4(p[0], p[1], p[2], p[3]);
}

// SKIP: kSkipNone (no skip logic at all), kSkipTiles (the blockMax early
// exit's map of 128-row tiles x vocab tiles) or kSkipSteps (the coefficient
// filter's bits per 256-row unit and 64-row vocab step).
constexpr int kSkipNone = 0, kSkipTiles = 1, kSkipSteps = 2;
template <int BITS, int BNH, int SKIP>
__global__ void __launch_bounds__(kThreads, 1) tc_dh_kernel(
    const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_w,
    const TcDhArgs a) {
    using L = DhLayout<BITS, BNH>;
    constexpr int NS = L::NS;
    constexpr int NB = L::NB;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    // (offsetting the shared array itself keeps the accesses in the shared
    // address space; a round trip through an integer would make them generic)
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);  // TMA inputs landed
    uint64_t* empty = full + NS;  // inputs consumed (MMA commit + each dequant warp)
    uint64_t* dq = empty + NS;    // dequantized tile written
    uint64_t* bfree = dq + NB;    // dequantized tile consumed (MMA commit)
    uint64_t* accf = bfree + NB;  // [0]: the unit's accumulators are complete (MMA commit)
    uint64_t* acce = accf + 2;    // [h]: half h has been read out (epilogue warps)
    uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(acce + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_sh + 1);
    uint64_t* mdrain = acce + 3;  // MMA drain on the abort path
    int* err = a.err;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_active = *a.count;
    const int n_mt = (n_active + BMU - 1) / BMU;
    const int n_nt = a.H / BNH;
    const int KS = a.ks;                 // K slices per output tile
    const int units = n_mt * n_nt * KS;
    if (units == 0 || (int)blockIdx.x >= units) return;
    const int G = a.H / 64;
    // blockMax early exit: K step kk of 256-row unit mt is skipped when both
    // 128-row tiles skip its vocab tile.  Every role evaluates the same map.
    // Coefficient filter: K step kk is skipped when its bit is set (64 steps
    // share a word, so consecutive checks hit L1).
    auto kskip = [&](int mt, int kk) {
        if constexpr (SKIP == kSkipNone) return false;
        if constexpr (SKIP == kSkipSteps) {
            const int64_t k = (a.v_begin >> 6) + kk;
            return ((__ldg(a.kbits + mt * a.kbits_ld + (k >> 6)) >> (k & 63)) & 1ull) != 0;
        }
        const int64_t vt = (a.v_begin + (int64_t)kk * BK) >> 8;
        const int t0 = 2 * mt, t1 = 2 * mt + 1;
        return a.skip[(int64_t)t0 * a.skip_ld + vt] != 0 &&
               (t1 >= a.skip_rows || a.skip[(int64_t)t1 * a.skip_ld + vt] != 0);
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            tc::mbar_init(&full[i], 1 + 32);  // TMA (expect_tx) + 32 cp.async arrivals
            tc::mbar_init(&empty[i], 1 + kDqWarps);
        }
        for (int i = 0; i < NB; ++i) {
            tc::mbar_init(&dq[i], kDqWarps);
            tc::mbar_init(&bfree[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&accf[i], 1);
            tc::mbar_init(&acce[i], 4);
        }
        tc::mbar_init(mdrain, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tmap_c);
        tc::prefetch_tmap(&tmap_w);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_base_sh, L::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = *tmem_base_sh;

    if (warp == 0) {
        // Producer warp: lane 0 issues the TMA tiles; all 32 lanes copy the
        // stage's scales and biases (rows lane, lane + 32; the N tile's groups)
        // with cp.async, completing on the same barrier.
        int stage = 0;
        uint32_t phase = 0, fills = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const int mt = u / (n_nt * KS), nt = (u / KS) % n_nt, ks = u % KS;
            const int k0 = ks * a.n_k / KS, k1 = (ks + 1) * a.n_k / KS;
            for (int kk = k0; kk < k1; ++kk) {
                if (kskip(mt, kk)) continue;
                if (lane == 0)
                    ok = tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag, err,
                                       tc::kErrTimeoutEmpty);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    tc::mbar_arrive_expect_tx(&full[stage], L::A_BYTES + L::P_BYTES);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)  // rows past the block read as zero
                        tc::tma_load_2d(smem + L::OFF_A + stage * L::A_BYTES + hh * L::A_HALF,
                                        &tmap_c, &full[stage], kk * BK, mt * BMU + hh * BM);
                    if constexpr (L::SWZ) {
#pragma unroll
                        for (int hf = 0; hf < L::HALVES; ++hf)
                            tc::tma_load_2d(smem + L::OFF_P + stage * L::P_BYTES + hf * (BK * 128),
                                            &tmap_w, &full[stage], nt * L::WORDS + 32 * hf,
                                            (int)(a.v_begin + kk * BK));
                    } else {
                        tc::tma_load_2d(smem + L::OFF_P + stage * L::P_BYTES, &tmap_w, &full[stage],
                                        nt * L::WORDS, (int)(a.v_begin + kk * BK));
                    }
                }
                __half* sb = reinterpret_cast<__half*>(smem + L::OFF_SB + stage * L::SB_BYTES);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = lane + 32 * h;
                    const int64_t v = a.v_begin + (int64_t)kk * BK + r;
                    const int64_t gi = (v < a.V ? v : 0) * G + nt * L::NSB;
                    const int nbytes = v < a.V ? 2 * L::NSB : 0;
                    tc::cp_async_zfill<2 * L::NSB>(sb + r * L::NSB, a.scales + gi, nbytes);
                    tc::cp_async_zfill<2 * L::NSB>(sb + (BK + r) * L::NSB, a.biases + gi, nbytes);
                }
                tc::cp_async_arrive(&full[stage]);
                ++fills;
                if (++stage == NS) { stage = 0; phase ^= 1; }
            }
        }
        if (lane == 0) {
            // Drain: the last stages' copies landed and were consumed; on the
            // abort path only their landing is awaited.
            for (int i = 0; i < NS && ok; ++i) {
                ok = tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag, err, tc::kErrTimeoutEmpty);
                if (++stage == NS) { stage = 0; phase ^= 1; }
            }
            if (!ok) tc::drain_ring(full, NS, fills, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, bs = 0;
            uint32_t phase = 0, aphase = 0, bphase = 0;
            // The operand descriptors of ring slot 0: a slot's are these plus
            // its byte offset >> 4 in the 14-bit address field, which never
            // carries (shared addresses stay below 256 KB).  One thread issues
            // every MMA, so its per-stage instruction latency is on the
            // tensor pipe's critical path.
            const uint64_t ad_base = tc::sdesc_sw128(tc::smem_u32(smem + L::OFF_A), 16, 1024);
            const uint64_t bd_base =
                tc::sdesc_sw128(tc::smem_u32(smem + L::OFF_B), (BK / 8) * 1024, 1024);
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                const int mt = u / (n_nt * KS), ks = u % KS;
                const int k0 = ks * a.n_k / KS, k1 = (ks + 1) * a.n_k / KS;
                // Half h's accumulator may be overwritten once the epilogue has
                // read it out: half 0 before the unit starts, half 1 before its
                // first MMA (so reading out half 1 overlaps the next unit).
                if (!tc::mbar_wait(&acce[0], aphase ^ 1, abort_flag, err, tc::kErrTimeoutAccEmpty))
                    goto mma_abort;
                tc::tc_fence_after();
                bool first = true;  // no K step of this unit issued yet
                for (int kk = k0; kk < k1; ++kk) {
                    if (kskip(mt, kk)) continue;
                    if (!tc::mbar_wait(&full[stage], phase, abort_flag, err, tc::kErrTimeoutFull))
                        goto mma_abort;
                    if (!tc::mbar_wait(&dq[bs], bphase, abort_flag, err, tc::kErrTimeoutDequant))
                        goto mma_abort;
                    tc::tc_fence_after();
                    const uint64_t ad0 = ad_base + (uint32_t)(stage * (L::A_BYTES >> 4));
                    const uint64_t bd0 = bd_base + (uint32_t)(bs * (L::B_BYTES >> 4));
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        if (hh == 1 && first) {
                            if (!tc::mbar_wait(&acce[1], aphase ^ 1, abort_flag, err,
                                               tc::kErrTimeoutAccEmpty))
                                goto mma_abort;
                            tc::tc_fence_after();
                        }
#pragma unroll
                        for (int ks2 = 0; ks2 < BK / 16; ++ks2) {
                            // A: K-major, 32 bytes per 16-element K step inside the
                            // swizzle atom.  B: MN-major, two 8-row K groups (2 x 1024 B)
                            // per K step; 64-column blocks along N are BK/8 * 1024
                            // bytes apart (the leading offset).
                            tc::umma_f16(tmem_base + hh * BNH, ad0 + ((hh * L::A_HALF + 32 * ks2) >> 4),
                                         bd0 + ((2048 * ks2) >> 4), L::IDESC,
                                         (!first || ks2 > 0) ? 1u : 0u);
                        }
                    }
                    tc::umma_commit(&empty[stage]);
                    if constexpr (!L::ONE_RING) tc::umma_commit(&bfree[bs]);
                    if (++stage == NS) { stage = 0; phase ^= 1; }
                    if (++bs == NB) { bs = 0; bphase ^= 1; }
                    first = false;
                }
                tc::umma_commit(&accf[0]);
                aphase ^= 1;
            }
            goto mma_done;
        mma_abort:
            // Let every MMA issued so far finish before TMEM is released.
            tc::umma_commit(mdrain);
            tc::mbar_drain(mdrain, 0, err);
        mma_done:;
        }
    } else if (warp < kEpiWarp0) {
        // Dequant.  Swizzled rows (SWZ): in pass ps, dequant warp dw's lane
        // 8 a + b takes row 32 (ps & 1) + 8 (dw & 3) + b, piece
        // 8 (ps >> 1) + 4 (dw >> 2) + a.  Otherwise thread t takes piece
        // t % PIECES of rows t / PIECES + RPP * ps (a phase reads one 128-byte
        // span; its stores go to four 64-column blocks at one bank offset).
        const int t = threadIdx.x - 64;
        const int dw = t >> 5, qa = (t >> 3) & 3, qb = t & 7;
        int stage = 0, bs = 0;
        uint32_t phase = 0, bphase = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
            const int mt = u / (n_nt * KS), ks = u % KS;
            const int k0 = ks * a.n_k / KS, k1 = (ks + 1) * a.n_k / KS;
            for (int kk = k0; kk < k1; ++kk) {
                if (kskip(mt, kk)) continue;
                // Results ignored: the warp stays converged (see the abort policy).
                tc::mbar_wait(&full[stage], phase, abort_flag, err, tc::kErrTimeoutFull);
                if constexpr (!L::ONE_RING)
                    tc::mbar_wait(&bfree[bs], bphase ^ 1, abort_flag, err, tc::kErrTimeoutDequant);
                const unsigned char* P = smem + L::OFF_P + stage * L::P_BYTES;
                const __half* sb = reinterpret_cast<const __half*>(smem + L::OFF_SB + stage * L::SB_BYTES);
                unsigned char* Bs = smem + L::OFF_B + bs * L::B_BYTES;
#pragma unroll
                for (int ps = 0; ps < L::PASSES; ++ps) {
                    const int kr = L::SWZ ? 32 * (ps & 1) + 8 * (dw & 3) + qb
                                          : t / L::PIECES + L::RPP * ps;
                    const int pc = L::SWZ ? 8 * (ps >> 1) + 4 * (dw >> 2) + qa : t % L::PIECES;
                    const int krow = kr & 7;
                    const int ncol_piece = pc * L::CPP;     // first column of the piece in the N tile
                    const int nb = ncol_piece >> 6;         // 64-column block
                    const int j0 = (ncol_piece & 63) >> 3;  // first 16-byte chunk in the block
                    const uint4 wv = *reinterpret_cast<const uint4*>(
                        L::SWZ ? P + (pc >> 3) * (BK * 128) + kr * 128 + (((pc & 7) ^ krow) << 4)
                               : P + kr * L::P_ROW + pc * 16);
                    const __half2 s2 = __half2half2(sb[kr * L::NSB + nb]);
                    const __half2 b2 = __half2half2(sb[(BK + kr) * L::NSB + nb]);
                    unsigned char* dst_row = Bs + nb * (BK / 8) * 1024 + (kr >> 3) * 1024 + krow * 128;
                    // word i of the piece, selected without dynamic register indexing
                    auto word = [&](int i) {
                        return i == 0 ? wv.x : i == 1 ? wv.y : i == 2 ? wv.z : wv.w;
                    };
#pragma unroll
                    for (int q = 0; q < L::CHUNKS; ++q) {
                        const int qq = q;
                        uint4 out;
                        if constexpr (BITS == 4) {
                            out = deq4_chunk(word(qq), s2, b2);
                        } else {
                            const uint32_t w0 = word(2 * qq), w1 = word(2 * qq + 1);
                            out = make_uint4(deq8(w0, 0x5140u, s2, b2), deq8(w0, 0x7362u, s2, b2),
                                             deq8(w1, 0x5140u, s2, b2), deq8(w1, 0x7362u, s2, b2));
                        }
                        *reinterpret_cast<uint4*>(dst_row + (((j0 + qq) ^ krow) << 4)) = out;
                    }
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&dq[bs]);
                    tc::mbar_arrive(&empty[stage]);  // packed tile fully read
                }
                if (++stage == NS) { stage = 0; phase ^= 1; }
                if (++bs == NB) { bs = 0; bphase ^= 1; }
            }
        }
    } else {
        const int sub = warp & 3;
        const int row = sub * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(sub * 32) << 16;
        uint32_t aphase = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
            const int mt = u / (n_nt * KS), nt = (u / KS) % n_nt, ks = u % KS;
            // Whether any K step of the unit was issued (blockMax early exit:
            // otherwise the accumulators hold no sum of this unit).
            bool any_k = SKIP == kSkipNone;
            if (!any_k) {
                const int k0 = ks * a.n_k / KS, k1 = (ks + 1) * a.n_k / KS;
                for (int kk = k0; kk < k1 && !any_k; ++kk) any_k = !kskip(mt, kk);
            }
            // The rows' cotangents, fetched before the wait (a dependent pair
            // of global loads off the accumulators' critical path).
            float scale2[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = mt * BMU + hh * BM + row;
                scale2[hh] = i < n_active ? -a.dlogp[a.rows[i]] * (1.f / 16384.f) : 0.f;
            }
            // Result ignored: the warp stays converged (see the abort policy).
            tc::mbar_wait(&accf[0], aphase, abort_flag, err, tc::kErrTimeoutAccFull);
            tc::tc_fence_after();
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                const int i = mt * BMU + hh * BM + row;
                const bool row_ok = i < n_active;
                const float scale = hh ? scale2[1] : scale2[0];
                float* dst = a.dh_acc + (int64_t)ks * a.slice_stride + (int64_t)i * a.H + nt * BNH;
#pragma unroll 1
                for (int c = 0; c < BNH / 32; ++c) {
                    uint32_t r[32];
                    tc::tmem_ld32(tmem_base + lane_addr + hh * BNH + c * 32, r);
                    tc::tmem_wait_ld();
                    if (!any_k) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = 0u;  // an empty sum
                    }
                    if (row_ok && (any_k || !a.accumulate)) {
                        // N column j of this chunk is hidden offset (j & ~7) + perm[j & 7]
                        // for 4-bit heads (perm = 0,4,1,5,2,6,3,7), natural for 8-bit.
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            constexpr int inv4[8] = {0, 2, 4, 6, 1, 3, 5, 7};  // offset -> N column
                            const int src = BITS == 4 ? ((j & ~7) | inv4[j & 7]) : j;
                            v[j] = __uint_as_float(r[src]) * scale;
                        }
                        float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
                        // Later chunks add at L2 (one addition per element per
                        // launch, launches in chunk order: the sums of a
                        // read-modify-write in the same fixed order, subnormals
                        // flushed, without its round trip on the accumulators'
                        // critical path).
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 x = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                            if (a.accumulate) tc::red_add_v4(reinterpret_cast<float*>(d4 + q), x);
                            else d4[q] = x;
                        }
                    }
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&acce[hh]);
            }
            aphase ^= 1;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

template <int BITS, int BNH, int SKIP>
cudaError_t launch_t(const CUtensorMap& tc_map, const CUtensorMap& tw, const TcDhArgs& a, int grid,
                     cudaStream_t st) {
    using L = DhLayout<BITS, BNH>;
    if (cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(tc_dh_kernel<BITS, BNH, SKIP>),
                                          L::SMEM))
        return e;
    tc_dh_kernel<BITS, BNH, SKIP><<<grid, kThreads, L::SMEM, st>>>(tc_map, tw, a);
    return cudaGetLastError();
}

}  // namespace

int tc_dh_cols(int H) { return H % 256 == 0 ? 256 : 128; }

int tc_dh_words(int H, int bits) { return tc_dh_cols(H) * bits / 32; }

bool tc_dh_swizzled(int H, int bits) { return tc_dh_cols(H) * bits / 8 >= 128; }

cudaError_t launch_tc_dh(const CUtensorMap& tmap_c, const CUtensorMap& tmap_w, const TcDhArgs& a,
                         int bits, int grid, cudaStream_t st) {
    const int bnh = tc_dh_cols(a.H);
    const int skip = a.kbits != nullptr ? kSkipSteps : a.skip != nullptr ? kSkipTiles : kSkipNone;
    // One instantiation per (bits, columns, skip kind).
    auto go = [&](auto bits_c, auto bnh_c) {
        constexpr int B = decltype(bits_c)::value, N = decltype(bnh_c)::value;
        return skip == kSkipSteps   ? launch_t<B, N, kSkipSteps>(tmap_c, tmap_w, a, grid, st)
               : skip == kSkipTiles ? launch_t<B, N, kSkipTiles>(tmap_c, tmap_w, a, grid, st)
                                    : launch_t<B, N, kSkipNone>(tmap_c, tmap_w, a, grid, st);
    };
    using I4 = std::integral_constant<int, 4>;
    using I8 = std::integral_constant<int, 8>;
    using C256 = std::integral_constant<int, 256>;
    using C128 = std::integral_constant<int, 128>;
    if (bits == 4) return bnh == 256 ? go(I4{}, C256{}) : go(I4{}, C128{});
    return bnh == 256 ? go(I8{}, C256{}) : go(I8{}, C128{});
}

}  // namespace qh

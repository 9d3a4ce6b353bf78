// qh_tc_fwd.cu -- tensor-core forward for large M (steps a2-a5 of the hot path).
//
// Computes the same per-(row, vocab segment) partials as the vocab-parallel
// forward on the page "mlx-bun 0.0.4 -> 0.0.6" (src/train/flash-cce.ts,
// FWD_STEEL_SOURCE: a quantized block GEMM whose epilogue soft-caps each
// logit tile and folds it into a running max / sum-exp), re-designed for
// sm_103a around a pair of CTAs on two SMs (a cluster of two):
//
//   * the pair walks units (256 token rows x a segment of 256-row vocab
//     tiles), chosen on the device from the active-row count; the even CTA
//     holds token rows 0-127 of the unit and vocab rows 0-127 of each tile,
//     the odd CTA rows 128-255 of both;
//   * in each CTA a TMA warp streams its fp16 h tile (128 x 64, 128-byte
//     swizzle) and its half of the packed weight tile (128 rows x 64 codes);
//   * eight (4-bit heads) or sixteen (8-bit heads) dequant warps turn the
//     CTA's packed half-tile into fp16 in the tensor core's K-major
//     128-byte-swizzled layout (w = fma(q, scale, bias), one rounding), two
//     or four threads per vocab row so that the packed rows are read with
//     conflict-free 16-byte loads; the TMA warp also stages the half-tile's
//     scales and biases, eight groups per box, so that the dequant warps
//     hold no global loads in flight (a barrier arrival, a release, would
//     wait for them);
//   * one thread of the even CTA issues tcgen05.mma.cta_group::2 (M = 256
//     across the pair, N = 256, K = 16, fp32 accumulate) into one of two
//     256-column accumulators: each SM dequantizes only the half of every
//     weight tile its own B operand holds, half of what a one-CTA M = 128 MMA
//     would need per flop;
//   * four epilogue warps per CTA read their 128 accumulator rows with
//     tcgen05.ld (one row per thread), apply the soft cap, update the row's
//     online softmax and track the maxima of the two 32-column slices with
//     the largest raw logit, each with the lowest column holding it (argmax
//     candidates, rechecked exactly by the finalize kernel).
// The [M,V] logits and the dequantized head never leave the SMs.
//
// The same kernel is phase 1 of the backward: its coefficient epilogue writes
// p * sech2 * 2^14 as fp16 per logit into the chunk's [rows x chunk] block;
// with the coefficient filter (a separate instantiation) each warp also votes
// per 32 x 32 block whether any term reaches eps, writes a cold block as
// zeros and clears, for a warm one, the dh step's bit in the filter's map
// (the backward's near-zero coefficient filter on the same page).
//
// Synchronisation of the pair: each CTA's dequant warps, once their B half
// and (having waited for it) their TMA-loaded A tile are in place, arrive on
// their own CTA's dequant barrier (CTA scope: a cluster-scope release in every
// dequant warp at every stage would wait for the warp's prefetched scale
// loads); in the odd CTA one otherwise idle thread waits for that barrier and
// forwards a single cluster-scope arrival to the even CTA's, whose MMA thread
// thus waits for both CTAs.  Each commit of the MMAs is multicast to the
// barriers of both CTAs (stage free: its inputs and its B slot; accumulator
// full).
// Each CTA's epilogue warps arrive on the even CTA's accumulator-empty
// barrier (once per tile).
#include <stdio.h>

#include <map>
#include <mutex>
#include <utility>

#include "qh_dequant.cuh"
#include "qh_tc.cuh"
#include "qh_tmap.h"

namespace qh {

namespace {

constexpr int BM = 128;   // token rows per CTA per unit (the pair: 256, the MMA's M)
constexpr int BMU = 2 * BM;
constexpr int BN = kTcFwdTileRows;  // vocab rows per tile (MMA N); each CTA holds BN / 2
constexpr int BNH = BN / 2;
constexpr int BK = 64;    // K per stage (one quantization group, one swizzle atom)
// Warp roles: 0 TMA, 1 MMA (issues in the even CTA; allocates TMEM in both),
// 2 .. 2 + dequant warps - 1 dequantize, then four epilogue warps.
template <int BITS>
struct Warps {
    static constexpr int kDq = BITS == 4 ? 8 : 16;
    static constexpr int kTpr = kDq * 32 / BNH;  // dequant threads per vocab row (2 or 4)
    static constexpr int kEpi0 = 2 + kDq;        // first epilogue warp
    static constexpr int kThreads = 32 * (kEpi0 + 4);
    static_assert(kTpr * 16 == BK * BITS / 8, "one 16-byte part of the packed row per thread");
};
constexpr int kTmemCols = 512;  // two 256-column fp32 accumulators
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BNH * BK * 2;  // this CTA's half of the dequantized tile
constexpr uint32_t kIdesc = tc::idesc_f16_f32(BMU, BN, false, false);
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint16_t kPairMask = 0x3;

// One ring of NS stages, each the TMA inputs (h tile + packed half-tile) and
// the dequantized half-tile made from them: a stage's B slot is free again
// once its inputs are (the MMAs that read A also read B), so the dequant
// warps wait for the stage's inputs alone and the MMA thread commits once
// per stage (two rings, with a separate barrier for the B slots, were 2-5 %
// slower).
// Scales and biases: boxes of kSbGroups groups x BNH rows of fp16, one box
// of each per kSbGroups stages, in a ring of NSB slots.
constexpr int kSbGroups = 8;
constexpr int SB_BOX = kSbGroups * 2 * BNH;  // bytes of one box (16-byte rows)

template <int BITS>
struct Layout {
    static constexpr int NS = BITS == 4 ? 5 : 4;
    static constexpr int NSB = 2;
    static constexpr int P_ROW = BK * BITS / 8;  // packed bytes per row per stage
    static constexpr int P_BYTES = BNH * P_ROW;
    static constexpr int WORDS = BK * BITS / 32;
    static constexpr int OFF_B = 0;
    static constexpr int OFF_A = OFF_B + NS * B_BYTES;
    static constexpr int OFF_P = OFF_A + NS * A_BYTES;
    static constexpr int OFF_SB = OFF_P + NS * P_BYTES;  // slot i: scales, then biases
    static constexpr int OFF_BAR = OFF_SB + NSB * 2 * SB_BOX;
    static constexpr int BAR_BYTES = 8 * (3 * NS + 2 * NSB + 5) + 16;
    static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct Work {
    int n_mt, n_vt, n_seg, units;
};

// Units (256 rows x a segment of vocab tiles) per CTA pair: many small units
// keep the per-pair totals within a few percent of each other.
constexpr int kUnitsPerPair = 32;

__device__ __forceinline__ Work plan_work(int n_active, int n_vt, int n_pairs) {
    Work w;
    w.n_mt = (n_active + BMU - 1) / BMU;
    w.n_vt = n_vt;
    const int target = kUnitsPerPair * n_pairs;
    int seg = w.n_mt > 0 ? (target + w.n_mt - 1) / w.n_mt : 1;
    if (seg > w.n_vt) seg = w.n_vt;
    if (seg < 1) seg = 1;
    w.n_seg = seg;
    w.units = w.n_mt * w.n_seg;
    return w;
}

__device__ __forceinline__ void unit_coords(const Work& w, int vt_begin, int u, int& mt, int& seg,
                                            int& vt0, int& vt1) {
    seg = u / w.n_mt;
    mt = u - seg * w.n_mt;
    vt0 = vt_begin + (int)((int64_t)seg * w.n_vt / w.n_seg);
    vt1 = vt_begin + (int)((int64_t)(seg + 1) * w.n_vt / w.n_seg);
}

// EPI_SOFTMAX: per-row online softmax + argmax candidates -> partials (forward).
// EPI_COEFF: per logit c = exp(z - lse) * sech2 * 2^14 as fp16 into a
//            [rows x chunk] block (phase 1 of the backward).
// EPI_FILTER: EPI_COEFF plus the coefficient filter (blocks of 32 rows x 32
//             vocab rows below filter_eps are written as zeros; a.kbits).
constexpr int EPI_SOFTMAX = 0, EPI_COEFF = 1, EPI_FILTER = 2;

// The pair's sequence of (unit, vocab tile) steps, the tiles every role
// processes in the same order (skipped tiles left out).
struct TileIt {
    int u, mt, seg, vt, vt1;
    bool valid;
};

template <int BITS, int EPI>
__global__ void __launch_bounds__(Warps<BITS>::kThreads, 1) tc_fwd_kernel(
    const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
    const __grid_constant__ CUtensorMap tmap_s, const __grid_constant__ CUtensorMap tmap_b,
    const TcFwdArgs a) {
    using L = Layout<BITS>;
    using WR = Warps<BITS>;
    constexpr int NS = L::NS;
    constexpr int NSB = L::NSB;
    const __half* __restrict__ scales = a.scales;
    const __half* __restrict__ biases = a.biases;
    const int64_t V = a.V;
    const int H = a.H;
    const float cap = a.cap;
    int* __restrict__ err = a.err;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    // (offsetting the shared array itself keeps the accesses in the shared
    // address space; a round trip through an integer would make them generic)
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);  // own TMA inputs landed
    uint64_t* empty = full + NS;  // stage consumed (pair MMA commit + own dequant warps)
    uint64_t* dq = empty + NS;    // own dequant warps done (even CTA: and the odd CTA's relay)
    uint64_t* accf = dq + NS;     // accumulator full (pair MMA commit)
    uint64_t* acce = accf + 2;    // even CTA: both CTAs' epilogues drained the accumulator
    uint64_t* mdrain = acce + 2;  // MMA drain on the abort path
    uint64_t* sbf = mdrain + 1;   // scale / bias boxes landed
    uint64_t* sbe = sbf + NSB;    // scale / bias boxes consumed (own dequant warps)
    uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(sbe + NSB);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_sh + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = tc::cluster_ctarank();
    const int cid = (int)tc::cluster_id_x(), n_pairs = (int)tc::nclusters_x();
    const int n_active = *a.count;
    const Work W = plan_work(n_active, a.vt_end - a.vt_begin, n_pairs);
    if (EPI == EPI_SOFTMAX && blockIdx.x == 0 && threadIdx.x == 0) *a.S_out = W.n_seg;
    // (the same decision in both CTAs of the pair: nothing below has run yet)
    if (W.units == 0 || cid >= W.units) return;
    const int KSTEPS = H / BK;
    const int G = H / 64;
    // Scales and biases staged by TMA (rows of whole 16-byte blocks of 8
    // groups); otherwise each dequant thread loads its own, stage by stage.
    const bool sb_tma = a.sb_tma != 0;
    // Backward with the blockMax early exit: skip_half: the 128-row tile t of
    // the map skips vocab tile vt (tiles past the map's rows hold no row);
    // skipped: both 128-row tiles of 256-row unit mt do, and every role of
    // both CTAs leaves the vocab tile out (no loads, dequantization or MMAs).
    auto skip_half = [&](int t, int vt) {
        return t >= a.skip_rows || a.skip[(int64_t)t * a.skip_ld + vt] != 0;
    };
    auto skipped = [&](int mt, int vt) {
        return EPI != EPI_SOFTMAX && a.skip != nullptr && skip_half(2 * mt, vt) &&
               skip_half(2 * mt + 1, vt);
    };
    // Tile iteration shared by the roles that look ahead (dequant warps).
    auto tile_settle = [&](TileIt& t) {  // move to the first tile not skipped
        while (t.valid) {
            while (t.vt < t.vt1 && skipped(t.mt, t.vt)) ++t.vt;
            if (t.vt < t.vt1) return;
            t.u += n_pairs;
            if (t.u >= W.units) { t.valid = false; return; }
            int vt0;
            unit_coords(W, a.vt_begin, t.u, t.mt, t.seg, vt0, t.vt1);
            t.vt = vt0;
        }
    };
    auto tile_first = [&]() {
        TileIt t;
        t.u = cid;
        t.valid = true;
        unit_coords(W, a.vt_begin, t.u, t.mt, t.seg, t.vt, t.vt1);
        tile_settle(t);
        return t;
    };
    auto tile_next = [&](TileIt t) {
        ++t.vt;
        tile_settle(t);
        return t;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], 1 + WR::kDq);
            tc::mbar_init(&dq[i], WR::kDq + (rank == 0 ? 1 : 0));
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&accf[i], 1);
            tc::mbar_init(&acce[i], 2 * 4);
        }
        tc::mbar_init(mdrain, 1);
        for (int i = 0; i < NSB; ++i) {
            tc::mbar_init(&sbf[i], 1);
            tc::mbar_init(&sbe[i], WR::kDq);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tmap_h);
        tc::prefetch_tmap(&tmap_w);
        if (sb_tma) {
            tc::prefetch_tmap(&tmap_s);
            tc::prefetch_tmap(&tmap_b);
        }
    }
    if (warp == 1) {
        tc::tmem_alloc_pair(tmem_base_sh, kTmemCols);
        tc::tmem_relinquish_pair();
    }
    tc::tc_fence_before();
    tc::cluster_sync();  // barriers initialised in both CTAs before any remote arrival
    tc::tc_fence_after();
    const uint32_t tmem_base = *tmem_base_sh;
    // The even CTA's barriers, addressed from either CTA.
    const uint32_t dq_lead = tc::mapa_shared(dq, 0);
    const uint32_t acce_lead = tc::mapa_shared(acce, 0);
    // Tiles the pair processes, in order (every role walks the same ones).
    auto for_each_tile = [&](auto&& body) {
        for (int u = cid; u < W.units; u += n_pairs) {
            int mt, seg, vt0, vt1;
            unit_coords(W, a.vt_begin, u, mt, seg, vt0, vt1);
            for (int vt = vt0; vt < vt1; ++vt)
                if (!skipped(mt, vt) && !body(mt, vt)) return;
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0, sslot = 0;
            uint32_t phase = 0, fills = 0, sphase = 0, sfills = 0;
            if (a.stall) goto producer_abort;
            for (int u = cid; u < W.units; u += n_pairs) {
                int mt, seg, vt0, vt1;
                unit_coords(W, a.vt_begin, u, mt, seg, vt0, vt1);
                for (int vt = vt0; vt < vt1; ++vt) {
                    if (skipped(mt, vt)) continue;
                    for (int kk = 0; kk < KSTEPS; ++kk) {
                        if (sb_tma && kk % kSbGroups == 0) {
                            // the scales and biases of the next 8 stages
                            if (!tc::mbar_wait(&sbe[sslot], sphase ^ 1, abort_flag, err,
                                               tc::kErrTimeoutEmpty))
                                goto producer_abort;
                            unsigned char* sd = smem + L::OFF_SB + sslot * 2 * SB_BOX;
                            tc::mbar_arrive_expect_tx(&sbf[sslot], 2 * SB_BOX);
                            tc::tma_load_2d(sd, &tmap_s, &sbf[sslot], kk, vt * BN + (int)rank * BNH);
                            tc::tma_load_2d(sd + SB_BOX, &tmap_b, &sbf[sslot], kk,
                                            vt * BN + (int)rank * BNH);
                            ++sfills;
                            if (++sslot == NSB) { sslot = 0; sphase ^= 1; }
                        }
                        if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag, err,
                                           tc::kErrTimeoutEmpty))
                            goto producer_abort;
                        tc::mbar_arrive_expect_tx(&full[stage], A_BYTES + L::P_BYTES);
                        // rows past the tensor (h: the padded row count; the
                        // head: V) read as zeros
                        tc::tma_load_2d(smem + L::OFF_A + stage * A_BYTES, &tmap_h, &full[stage],
                                        kk * BK, mt * BMU + (int)rank * BM);
                        tc::tma_load_2d(smem + L::OFF_P + stage * L::P_BYTES, &tmap_w,
                                        &full[stage], kk * L::WORDS, vt * BN + (int)rank * BNH);
                        ++fills;
                        if (++stage == NS) { stage = 0; phase ^= 1; }
                    }
                }
            }
            // Drain: wait until the loads of the last stages have landed and
            // been consumed.
            for (int i = 0; i < NS; ++i) {
                if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag, err,
                                   tc::kErrTimeoutEmpty))
                    goto producer_abort;
                if (++stage == NS) { stage = 0; phase ^= 1; }
            }
            goto producer_done;
        producer_abort:
            tc::drain_ring(full, NS, fills, err);
            tc::drain_ring(sbf, NSB, sfills, err);
        producer_done:;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && rank == 0) {
            int stage = 0, buf = 0;
            uint32_t aphase = 0, phase = 0;
            // The operand descriptors of ring slot 0: a slot's are these plus
            // its byte offset >> 4 in the 14-bit address field, which never
            // carries (shared addresses stay below 256 KB).  One thread issues
            // every MMA, so its per-stage instruction latency is on the
            // tensor pipe's critical path.
            const uint64_t ad_base = tc::sdesc_sw128(tc::smem_u32(smem + L::OFF_A), 16, 1024);
            const uint64_t bd_base = tc::sdesc_sw128(tc::smem_u32(smem + L::OFF_B), 16, 1024);
            for (int u = cid; u < W.units; u += n_pairs) {
                int mt, seg, vt0, vt1;
                unit_coords(W, a.vt_begin, u, mt, seg, vt0, vt1);
                for (int vt = vt0; vt < vt1; ++vt) {
                    if (skipped(mt, vt)) continue;
                    if (!tc::mbar_wait_cluster(&acce[buf], aphase ^ 1, abort_flag, err,
                                               tc::kErrTimeoutAccEmpty))
                        goto mma_abort;
                    tc::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    for (int kk = 0; kk < KSTEPS; ++kk) {
                        // Both CTAs' dequant warps have arrived: their B halves
                        // are written and their A tiles have landed.
                        if (!tc::mbar_wait_cluster(&dq[stage], phase, abort_flag, err,
                                                   tc::kErrTimeoutDequant))
                            goto mma_abort;
                        tc::tc_fence_after();
                        const uint64_t ad = ad_base + (uint32_t)(stage * (A_BYTES >> 4));
                        const uint64_t bd = bd_base + (uint32_t)(stage * (B_BYTES >> 4));
#pragma unroll
                        for (int ks = 0; ks < BK / 16; ++ks)  // 32 bytes per 16-element K step
                            tc::umma_f16_pair(d_tmem, ad + 2 * ks, bd + 2 * ks, kIdesc, (kk | ks) != 0);
                        tc::umma_commit_pair(&empty[stage], kPairMask);  // A, P and B free
                        if (++stage == NS) { stage = 0; phase ^= 1; }
                    }
                    tc::umma_commit_pair(&accf[buf], kPairMask);
                    if (++buf == 2) { buf = 0; aphase ^= 1; }
                }
            }
            goto mma_done;
        mma_abort:
            // Let every MMA issued so far finish before TMEM is released.
            tc::umma_commit_pair(mdrain, 0x1);
            tc::mbar_drain(mdrain, 0, err);
        mma_done:;
        } else if (lane == 0) {
            // Odd CTA: forward each stage's "dequant done" to the even CTA.
            int stage = 0;
            uint32_t phase = 0;
            for_each_tile([&](int, int) {
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    if (!tc::mbar_wait(&dq[stage], phase, abort_flag, err, tc::kErrTimeoutDequant))
                        return false;
                    tc::mbar_arrive_cluster_relaxed(dq_lead + 8u * (uint32_t)stage);
                    if (++stage == NS) { stage = 0; phase ^= 1; }
                }
                return true;
            });
        }
    } else if (warp < WR::kEpi0) {
        // ------------------------------------------------------------ dequant warps
        // Thread: 16-byte part `pt` of vocab row r of this CTA's half-tile.
        const int t = threadIdx.x - 64;
        const int r = t / WR::kTpr, pt = t % WR::kTpr;
        int stage = 0;
        uint32_t phase = 0;
        // One stage: wait for its inputs (its B slot was freed with them),
        // dequantize this thread's part of row r with scale s2 / bias b2 (fp16
        // pairs), signal.
        auto stage_work = [&](uint32_t s2, uint32_t b2) {
            // Result ignored: the warp stays converged (see the abort policy).
            tc::mbar_wait(&full[stage], phase, abort_flag, err, tc::kErrTimeoutFull);
            const unsigned char* prow = smem + L::OFF_P + stage * L::P_BYTES + r * L::P_ROW;
            unsigned char* brow = smem + L::OFF_B + stage * B_BYTES + r * 128;
            const uint4 wv = *reinterpret_cast<const uint4*>(prow + 16 * pt);
            const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
            if constexpr (BITS == 4) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = 4 * pt + j;  // 16-byte chunk = one word of 8 codes
                    uint32_t p[4];
                    deq4_word(wd[j], s2, b2, p);
                    *reinterpret_cast<uint4*>(brow + ((c ^ (r & 7)) << 4)) =
                        make_uint4(p[0], p[1], p[2], p[3]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int c = 2 * pt + j;  // 16-byte chunk = two words of 4 codes
                    const uint32_t w0 = wd[2 * j], w1 = wd[2 * j + 1];
                    *reinterpret_cast<uint4*>(brow + ((c ^ (r & 7)) << 4)) =
                        make_uint4(deq8(w0, 0x5140u, s2, b2), deq8(w0, 0x7362u, s2, b2),
                                   deq8(w1, 0x5140u, s2, b2), deq8(w1, 0x7362u, s2, b2));
                }
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&dq[stage]);
                tc::mbar_arrive(&empty[stage]);  // packed half-tile fully read
            }
            if (++stage == NS) { stage = 0; phase ^= 1; }
        };
        // Vocab row of this thread in tile t (-1 past the head).
        auto vrow = [&](const TileIt& ti) -> int64_t {
            const int64_t v = (int64_t)ti.vt * BN + (int64_t)rank * BNH + r;
            return v < V ? v : -1;
        };
        if (sb_tma) {
            // Scales and biases of 8 groups per staged box: this row's 16-byte
            // rows of the scale box and the bias box.
            int sslot = 0;
            uint32_t sphase = 0;
            const int NKB = G / kSbGroups;
            for (TileIt ti = tile_first(); ti.valid; ti = tile_next(ti)) {
                for (int kb = 0; kb < NKB; ++kb) {
                    tc::mbar_wait(&sbf[sslot], sphase, abort_flag, err, tc::kErrTimeoutFull);
                    const unsigned char* sd = smem + L::OFF_SB + sslot * 2 * SB_BOX;
                    const uint4 sc = *reinterpret_cast<const uint4*>(sd + r * 16);
                    const uint4 bc = *reinterpret_cast<const uint4*>(sd + SB_BOX + r * 16);
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&sbe[sslot]);  // (values are in registers)
                    if (++sslot == NSB) { sslot = 0; sphase ^= 1; }
                    const uint32_t sw[4] = {sc.x, sc.y, sc.z, sc.w};
                    const uint32_t bw[4] = {bc.x, bc.y, bc.z, bc.w};
#pragma unroll
                    for (int k8 = 0; k8 < kSbGroups; ++k8) {
                        const uint32_t sel = (k8 & 1) ? 0x3232u : 0x1010u;
                        stage_work(__byte_perm(sw[k8 >> 1], sw[k8 >> 1], sel),
                                   __byte_perm(bw[k8 >> 1], bw[k8 >> 1], sel));
                    }
                }
            }
        } else {
            for (TileIt ti = tile_first(); ti.valid; ti = tile_next(ti)) {
                const int64_t v = vrow(ti);
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const __half z = __float2half(0.f);
                    const __half s0 = v >= 0 ? scales[v * G + kk] : z;
                    const __half b0 = v >= 0 ? biases[v * G + kk] : z;
                    stage_work(bcast_h(s0), bcast_h(b0));
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int sub = warp & 3;  // TMEM sub-partition of this warp
        const int row = (int)rank * BM + sub * 32 + lane;  // row of the pair's 256-row unit
        const uint32_t lane_addr = static_cast<uint32_t>(sub * 32) << 16;
        const float k2 = cap > 0.f ? 2.f * kLog2e / cap : 0.f;
        int buf = 0;
        uint32_t aphase = 0;
        for (int u = cid; u < W.units; u += n_pairs) {
            int mt, seg, vt0, vt1;
            unit_coords(W, a.vt_begin, u, mt, seg, vt0, vt1);
            const int i = mt * BMU + row;  // compact row of this thread
            float m = -INFINITY, s = 0.f, v1 = -INFINITY, v2 = -INFINITY;
            int i1 = INT32_MAX, i2 = INT32_MAX;
            // EPI_COEFF: log2(p * 2^14) = z * log2e - (lse * log2e - 14)
            float lsb = 0.f;
            bool row_ok = i < n_active;
            if (EPI != EPI_SOFTMAX && row_ok) lsb = a.lse[a.rows[i]] * kLog2e - 14.f;
            // Coefficient filter: |dlogp| and the valid target of this row.
            float fg = 0.f;
            int64_t ftgt = -1;
            if (EPI == EPI_FILTER && row_ok) {
                const int r = a.rows[i];
                fg = fabsf(a.dlogp[r]);
                const int32_t tg = a.targets[r];
                ftgt = tg >= 0 && (int64_t)tg < V ? (int64_t)tg : -1;
            }
            for (int vt = vt0; vt < vt1; ++vt) {
                // Both 128-row tiles of the unit skip the vocab tile: so does
                // the dh contraction's unit (the same pair of tiles), which
                // reads nothing of it.
                if (skipped(mt, vt)) continue;
                tc::mbar_wait(&accf[buf], aphase, abort_flag, err, tc::kErrTimeoutAccFull);
                tc::tc_fence_after();
                // blockMax exit: this CTA's 128-row tile skips the vocab tile
                // while the other one keeps it: its coefficients are written as
                // zeros (the dh contraction reads them).  Warp-uniform.
                const bool zero_half = EPI != EPI_SOFTMAX && a.skip != nullptr &&
                                       skip_half(2 * mt + (int)rank, vt);
                float tz = -INFINITY;  // the tile's maximum of z (blockMax)
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    const int64_t col0 = (int64_t)vt * BN + c * 32;
                    if (EPI != EPI_SOFTMAX && zero_half) {
                        if (i < a.coeff_rows) {
                            __half* dst = a.coeff + (int64_t)i * a.coeff_ld +
                                          (col0 - (int64_t)a.vt_begin * BN);
                            const uint32_t zero[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                            tc::st_global_v8(dst, zero);
                            tc::st_global_v8(dst + 16, zero);
                        }
                        continue;
                    }
                    uint32_t rr[32];
                    tc::tmem_ld32(tmem_base + lane_addr + buf * BN + c * 32, rr);
                    tc::tmem_wait_ld();
                    const int nvalid = (int)min((int64_t)32, V - col0);
                    float x[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(rr[j]);
                    if constexpr (EPI != EPI_SOFTMAX) {
                        // coefficient block column = col0 - first column of the chunk
                        __half* dst = a.coeff + (int64_t)i * a.coeff_ld + (col0 - (int64_t)a.vt_begin * BN);
                        uint32_t out[16];
                        float cmax = 0.f;  // the chunk's largest p * sech2 * 2^14 of this row
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            float cj[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float xv = x[j + e];
                                float lg2p, sech2 = 1.f;
                                if (cap > 0.f) {
                                    const float th = fmaf(-2.f, tc::rcp_approx(tc::ex2_approx(xv * k2) + 1.f), 1.f);
                                    lg2p = fmaf(cap * th, kLog2e, -lsb);
                                    sech2 = fmaf(-th, th, 1.f);
                                } else {
                                    lg2p = fmaf(xv, kLog2e, -lsb);
                                }
                                const bool ok = row_ok && (j + e) < nvalid;
                                cj[e] = ok ? tc::ex2_approx(lg2p) * sech2 : 0.f;
                            }
                            out[j / 2] = h2_as_u32(__floats2half2_rn(cj[0], cj[1]));
                            if constexpr (EPI == EPI_FILTER) cmax = fmaxf(cmax, fmaxf(cj[0], cj[1]));
                        }
                        if constexpr (EPI == EPI_FILTER) {
                            // The block of this warp's 32 rows x these 32 vocab rows is
                            // warm when a row has |dlogp| p sech2 >= eps there (both
                            // sides scaled by 2^14) or its target lies there.
                            const bool warm_row = row_ok && (fg * cmax >= a.filter_eps * 16384.f ||
                                                             (ftgt >> 5) == (col0 >> 5));
                            const bool warm = __any_sync(0xffffffffu, warm_row);
                            if (!warm) {
#pragma unroll
                                for (int q = 0; q < 16; ++q) out[q] = 0u;
                            }
                            if (lane == 0) {
                                const int64_t vc = col0 >> 5, rg = i >> 5, k = vc >> 1;
                                if (warm)  // the dh step of these rows is needed
                                    atomicAnd(a.kbits + (rg >> 3) * a.kbits_ld + (k >> 6),
                                              ~(1ull << (k & 63)));
                                if (a.cold_out != nullptr && rg < a.cold_out_rows && vc < a.cold_out_ld)
                                    a.cold_out[rg * a.cold_out_ld + vc] = warm ? 0 : 1;
                            }
                        }
                        if (i < a.coeff_rows) {
                            // 32-byte stores: every store fills whole sectors.
#pragma unroll
                            for (int q = 0; q < 2; ++q) tc::st_global_v8(dst + 16 * q, out + 8 * q);
                        }
                    } else {
                        if (nvalid <= 0) continue;
                        float rmax = -INFINITY;
                        if (nvalid == 32) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) rmax = fmaxf(rmax, x[j]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j < nvalid) rmax = fmaxf(rmax, x[j]);
                        }
                        // Lowest column of the slice holding its maximum.  No
                        // guard is needed: the column that set rmax is valid and
                        // lies below every padding column.
                        int jb = 31;
#pragma unroll
                        for (int j = 30; j >= 0; --j) jb = x[j] == rmax ? j : jb;
                        jb = min(jb, nvalid - 1);  // (no match at all: NaN logits)
                        // argmax candidates: the maxima of the two slices with the
                        // largest raw logit
                        const int ci = (int)col0 + jb;
                        if (better(rmax, ci, v1, i1)) { v2 = v1; i2 = i1; v1 = rmax; i1 = ci; }
                        else if (better(rmax, ci, v2, i2)) { v2 = rmax; i2 = ci; }
                        // soft cap z = cap * tanh(x / cap) = cap - 2 cap / (exp(2x/cap) + 1)
                        float zmax = rmax;
                        if (cap > 0.f) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                x[j] = fmaf(-2.f * cap, tc::rcp_approx(tc::ex2_approx(x[j] * k2) + 1.f), cap);
                            zmax = fmaf(-2.f * cap, tc::rcp_approx(tc::ex2_approx(rmax * k2) + 1.f), cap);
                        }
                        const float mn = fmaxf(m, zmax);
                        const float mb = mn * kLog2e;
                        float acc = 0.f;
                        if (nvalid == 32) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) acc += tc::ex2_approx(fmaf(x[j], kLog2e, -mb));
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j < nvalid) acc += tc::ex2_approx(fmaf(x[j], kLog2e, -mb));
                        }
                        s = s * tc::ex2_approx((m - mn) * kLog2e) + acc;
                        m = mn;
                        tz = fmaxf(tz, zmax);
                    }
                }
                if (EPI == EPI_SOFTMAX && a.bmax != nullptr && row_ok)
                    a.bmax[(int64_t)a.rows[i] * a.bmax_ld + vt] = tz;
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive_cluster(acce_lead + 8u * (uint32_t)buf);
                if (++buf == 2) { buf = 0; aphase ^= 1; }
            }
            if (EPI == EPI_SOFTMAX && row_ok) {
                Partial p;
                p.m = m; p.s = s; p.v1 = v1; p.v2 = v2; p.i1 = i1; p.i2 = i2; p.status = *abort_flag; p.pad1 = 0;
                a.part[(int64_t)i * W.n_seg + seg] = p;
            }
        }
    }

    // Neither CTA releases its tensor memory or shared memory (which the other
    // CTA's MMAs and arrivals use) before both are done.
    tc::tc_fence_before();
    tc::cluster_sync();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// Pairs that can be resident at once for a kernel on the current device
// (cluster scheduling can leave an SM of a GPC idle): cached per (kernel,
// device).
std::mutex g_pairs_mu;
std::map<std::pair<const void*, int>, int> g_pairs;

int resident_pairs(const void* fn, int threads, int smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_pairs_mu);
    auto it = g_pairs.find({fn, dev});
    if (it != g_pairs.end()) return it->second;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * 256);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
    g_pairs[{fn, dev}] = n;
    return n;
}

}  // namespace

int tc_fwd_smem_bytes(int bits) { return bits == 4 ? Layout<4>::SMEM : Layout<8>::SMEM; }

template <int BITS, int EPI>
static cudaError_t launch_t(const CUtensorMap& th, const CUtensorMap& tw, const CUtensorMap& ts,
                            const CUtensorMap& tb, const TcFwdArgs& a, int grid,
                            cudaStream_t st) {
    const void* fn = reinterpret_cast<const void*>(tc_fwd_kernel<BITS, EPI>);
    constexpr int kSmem = Layout<BITS>::SMEM;
    constexpr int kThreads = Warps<BITS>::kThreads;
    if (cudaError_t e = ensure_smem_limit(fn, kSmem)) return e;
    // One CTA per SM, as many pairs as fit (at most grid / 2).
    int pairs = resident_pairs(fn, kThreads, kSmem);
    if (pairs > grid / 2) pairs = grid / 2;
    if (pairs < 1) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_fwd_kernel<BITS, EPI>, th, tw, ts, tb, a);
}

cudaError_t launch_tc_fwd(const CUtensorMap& th, const CUtensorMap& tw, const TcFwdArgs& in,
                          int bits, bool coeff_epilogue, int grid, cudaStream_t st) {
    // Tensor maps of the scale and bias tables (boxes of 8 groups x the CTA's
    // 128 vocab rows) when their rows are whole 16-byte blocks.
    TcFwdArgs a = in;
    CUtensorMap ts{}, tb{};
    const uint64_t G = (uint64_t)a.H / 64;
    a.sb_tma = G % kSbGroups == 0 &&
               tmap_group_rows(&ts, a.scales, G, (uint64_t)a.V, kSbGroups, BNH) &&
               tmap_group_rows(&tb, a.biases, G, (uint64_t)a.V, kSbGroups, BNH);
    if (bits == 4)
        return !coeff_epilogue ? launch_t<4, EPI_SOFTMAX>(th, tw, ts, tb, a, grid, st)
               : a.kbits != nullptr ? launch_t<4, EPI_FILTER>(th, tw, ts, tb, a, grid, st)
                                    : launch_t<4, EPI_COEFF>(th, tw, ts, tb, a, grid, st);
    return !coeff_epilogue ? launch_t<8, EPI_SOFTMAX>(th, tw, ts, tb, a, grid, st)
           : a.kbits != nullptr ? launch_t<8, EPI_FILTER>(th, tw, ts, tb, a, grid, st)
                                : launch_t<8, EPI_COEFF>(th, tw, ts, tb, a, grid, st);
}

}  // namespace qh

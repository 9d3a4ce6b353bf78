// qh_tc_fwd.cu -- tensor-core forward for large M (steps a2-a5 of the hot path).
//
// Computes the same per-(row, vocab segment) partials as the vocab-parallel
// forward on the page "mlx-bun 0.0.4 -> 0.0.6" (src/train/flash-cce.ts,
// FWD_STEEL_SOURCE: a quantized block GEMM whose epilogue soft-caps each
// logit tile and folds it into a running max / sum-exp), re-designed for
// sm_103a:
//
//   * one persistent CTA per SM walks units (128 token rows x a segment of
//     256-row vocab tiles), chosen on the device from the active-row count;
//   * a TMA warp streams the fp16 h tile (128 x 64, 128-byte swizzle) and the
//     packed weight tile (256 rows x 64 codes) into a 3-stage ring;
//   * eight (4-bit heads) or sixteen (8-bit heads) dequant warps turn the
//     packed tile into fp16 in the tensor core's K-major 128-byte-swizzled
//     layout (w = fma(q, scale, bias), one rounding);
//   * one thread issues tcgen05.mma (M=128, N=256, K=16, fp32 accumulate) into
//     one of two 256-column TMEM accumulators;
//   * four epilogue warps read the accumulator with tcgen05.ld (one row per
//     thread), apply the soft cap, update the row's online softmax and track
//     the maxima of the two 32-column slices with the largest raw logit, each
//     with the lowest column holding it (argmax candidates, rechecked exactly
//     by the finalize kernel).
// The [M,V] logits and the dequantized head never leave the SM.
//
// The same kernel is phase 1 of the backward: its coefficient epilogue writes
// p * sech2 * 2^14 as fp16 per logit into the chunk's [rows x chunk] block;
// with the coefficient filter (a separate instantiation) each warp also votes
// per 32 x 32 block whether any term reaches eps, writes a cold block as
// zeros and clears, for a warm one, the dh step's bit in the filter's map
// (the backward's near-zero coefficient filter on the same page).
#include <stdio.h>

#include "qh_dequant.cuh"
#include "qh_tc.cuh"
#include "qh_tmap.h"

namespace qh {

namespace {

constexpr int BM = 128;   // token rows per tile (MMA M)
constexpr int BN = kTcFwdTileRows;  // vocab rows per tile (MMA N)
constexpr int BK = 64;    // K per stage (one quantization group, one swizzle atom)
constexpr int NB = 3;     // dequantized-tile stages
// Warp roles: 0 TMA, 1 MMA, 2 .. 2 + dequant warps - 1 dequantize, then four
// epilogue warps.  Dequant warps: one thread per vocab row at 4 bits; two per
// row at 8 bits (twice the words per row; measured faster).
template <int BITS>
struct Warps {
    static constexpr int kDq = BITS == 4 ? 8 : 16;
    static constexpr int kTpr = kDq * 32 / 256;  // dequant threads per vocab row
    static constexpr int kEpi0 = 2 + kDq;        // first epilogue warp
    static constexpr int kThreads = 32 * (kEpi0 + 4);
};
constexpr int kTmemCols = 512;  // two 256-column fp32 accumulators
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr uint32_t kIdesc = tc::idesc_f16_f32(BM, BN, false, false);
constexpr float kLog2e = 1.4426950408889634f;

// Two rings: NS stages of TMA inputs (h tile + packed tile, small, deep enough
// to cover HBM latency) and NB stages of dequantized tiles (large).
template <int BITS>
struct Layout {
    static constexpr int NS = BITS == 4 ? 5 : 4;
    static constexpr int P_ROW = BK * BITS / 8;  // packed bytes per row per stage
    static constexpr int P_BYTES = BN * P_ROW;
    static constexpr int WORDS = BK * BITS / 32;
    static constexpr int OFF_B = 0;
    static constexpr int OFF_A = OFF_B + NB * B_BYTES;
    static constexpr int OFF_P = OFF_A + NS * A_BYTES;
    static constexpr int OFF_BAR = OFF_P + NS * P_BYTES;
    static constexpr int BAR_BYTES = 8 * (2 * NS + 2 * NB + 4) + 16;
    static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
};

struct Work {
    int n_mt, n_vt, n_seg, units;
};

// Units (128 rows x a segment of vocab tiles) per CTA: many small units keep
// the per-CTA totals within a few percent of each other.
constexpr int kUnitsPerCta = 32;

__device__ __forceinline__ Work plan_work(int n_active, int n_vt) {
    Work w;
    w.n_mt = (n_active + BM - 1) / BM;
    w.n_vt = n_vt;
    const int target = kUnitsPerCta * (int)gridDim.x;
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

template <int BITS, int EPI>
__global__ void __launch_bounds__(Warps<BITS>::kThreads, 1) tc_fwd_kernel(
    const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
    const TcFwdArgs a) {
    using L = Layout<BITS>;
    using WR = Warps<BITS>;
    constexpr int NS = L::NS;
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
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);  // TMA inputs landed
    uint64_t* empty = full + NS;  // inputs consumed (MMA commit + each dequant warp)
    uint64_t* dq = empty + NS;    // dequantized tile written
    uint64_t* bfree = dq + NB;    // dequantized tile consumed (MMA commit)
    uint64_t* accf = bfree + NB;
    uint64_t* acce = accf + 2;
    uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(acce + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_sh + 1);
    uint64_t* mdrain = acce + 3;  // MMA drain on the abort path

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_active = *a.count;
    const Work W = plan_work(n_active, a.vt_end - a.vt_begin);
    if (EPI == EPI_SOFTMAX && blockIdx.x == 0 && threadIdx.x == 0) *a.S_out = W.n_seg;
    if (W.units == 0 || (int)blockIdx.x >= W.units) return;
    const int KSTEPS = H / BK;
    const int G = H / 64;
    // Backward with the blockMax early exit: every role skips the same
    // (row tile, vocab tile) pairs (no loads, dequantization or MMAs; the
    // epilogue writes the tile's coefficients as zeros).
    auto skipped = [&](int mt, int vt) {
        return EPI != EPI_SOFTMAX && a.skip != nullptr && a.skip[(int64_t)mt * a.skip_ld + vt] != 0;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], 1 + WR::kDq);
        }
        for (int i = 0; i < NB; ++i) {
            tc::mbar_init(&dq[i], WR::kDq);
            tc::mbar_init(&bfree[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&accf[i], 1);
            tc::mbar_init(&acce[i], 4);
        }
        tc::mbar_init(mdrain, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tmap_h);
        tc::prefetch_tmap(&tmap_w);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_base_sh, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = *tmem_base_sh;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, fills = 0;
            if (a.stall) goto producer_abort;
            for (int u = blockIdx.x; u < W.units; u += gridDim.x) {
                int mt, seg, vt0, vt1;
                unit_coords(W, a.vt_begin, u, mt, seg, vt0, vt1);
                for (int vt = vt0; vt < vt1; ++vt) {
                    if (skipped(mt, vt)) continue;
                    for (int kk = 0; kk < KSTEPS; ++kk) {
                        if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag, err,
                                           tc::kErrTimeoutEmpty))
                            goto producer_abort;
                        tc::mbar_arrive_expect_tx(&full[stage], A_BYTES + L::P_BYTES);
                        tc::tma_load_2d(smem + L::OFF_A + stage * A_BYTES, &tmap_h, &full[stage],
                                        kk * BK, mt * BM);
                        tc::tma_load_2d(smem + L::OFF_P + stage * L::P_BYTES, &tmap_w,
                                        &full[stage], kk * L::WORDS, vt * BN);
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
        producer_done:;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, buf = 0, bs = 0;
            uint32_t phase = 0, aphase = 0, bphase = 0;
            for (int u = blockIdx.x; u < W.units; u += gridDim.x) {
                int mt, seg, vt0, vt1;
                unit_coords(W, a.vt_begin, u, mt, seg, vt0, vt1);
                for (int vt = vt0; vt < vt1; ++vt) {
                    if (skipped(mt, vt)) continue;
                    if (!tc::mbar_wait(&acce[buf], aphase ^ 1, abort_flag, err,
                                       tc::kErrTimeoutAccEmpty))
                        goto mma_abort;
                    tc::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    for (int kk = 0; kk < KSTEPS; ++kk) {
                        if (!tc::mbar_wait(&full[stage], phase, abort_flag, err,
                                           tc::kErrTimeoutFull))
                            goto mma_abort;
                        if (!tc::mbar_wait(&dq[bs], bphase, abort_flag, err,
                                           tc::kErrTimeoutDequant))
                            goto mma_abort;
                        tc::tc_fence_after();
                        const uint32_t a0 = tc::smem_u32(smem + L::OFF_A + stage * A_BYTES);
                        const uint32_t b0 = tc::smem_u32(smem + L::OFF_B + bs * B_BYTES);
#pragma unroll
                        for (int ks = 0; ks < BK / 16; ++ks) {
                            const uint64_t ad = tc::sdesc_sw128(a0 + 32 * ks, 16, 1024);
                            const uint64_t bd = tc::sdesc_sw128(b0 + 32 * ks, 16, 1024);
                            tc::umma_f16(d_tmem, ad, bd, kIdesc, (kk | ks) != 0);
                        }
                        tc::umma_commit(&empty[stage]);
                        tc::umma_commit(&bfree[bs]);
                        if (++stage == NS) { stage = 0; phase ^= 1; }
                        if (++bs == NB) { bs = 0; bphase ^= 1; }
                    }
                    tc::umma_commit(&accf[buf]);
                    if (++buf == 2) { buf = 0; aphase ^= 1; }
                }
            }
            goto mma_done;
        mma_abort:
            // Let every MMA issued so far finish before TMEM is released.
            tc::umma_commit(mdrain);
            tc::mbar_drain(mdrain, 0, err);
        mma_done:;
        }
    } else if (warp < WR::kEpi0) {
        // ------------------------------------------------------------ dequant warps
        // Thread: part `pt` of vocab row t of the tile (kTpr parts per row).
        const int t = (threadIdx.x - 64) / WR::kTpr, pt = (threadIdx.x - 64) % WR::kTpr;
        int stage = 0, bs = 0;
        uint32_t phase = 0, bphase = 0;
        for (int u = blockIdx.x; u < W.units; u += gridDim.x) {
            int mt, seg, vt0, vt1;
            unit_coords(W, a.vt_begin, u, mt, seg, vt0, vt1);
            for (int vt = vt0; vt < vt1; ++vt) {
                if (skipped(mt, vt)) continue;
                const int64_t v0 = (int64_t)vt * BN + t;
                const bool ok0 = v0 < V;
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const __half z = __float2half(0.f);
                    const __half s0 = ok0 ? scales[v0 * G + kk] : z, b0 = ok0 ? biases[v0 * G + kk] : z;
                    // Results ignored: the warp stays converged (see the abort policy).
                    tc::mbar_wait(&full[stage], phase, abort_flag, err, tc::kErrTimeoutFull);
                    tc::mbar_wait(&bfree[bs], bphase ^ 1, abort_flag, err, tc::kErrTimeoutDequant);
                    const unsigned char* P = smem + L::OFF_P + stage * L::P_BYTES;
                    unsigned char* Bs = smem + L::OFF_B + bs * B_BYTES;
                    {
                        const int r = t;
                        const __half2 s2 = __half2half2(s0);
                        const __half2 b2 = __half2half2(b0);
                        // 8-bit packed tiles arrive with the 64-byte swizzle (16-byte
                        // part q of row r at q ^ ((r >> 1) & 3)), so an 8-lane phase
                        // of part loads hits 8 bank groups (measured -1.5 % at 8 bits;
                        // the 32-byte swizzle of 4-bit tiles was not faster).
                        const unsigned char* prow = P + r * L::P_ROW;
                        const int pswz = BITS == 8 ? (r >> 1) & 3 : 0;
                        unsigned char* brow = Bs + r * 128;
                        if constexpr (BITS == 4) {
                            static_assert(WR::kTpr == 1, "4-bit rows: one thread per row");
#pragma unroll
                            for (int hq = 0; hq < 2; ++hq) {
                                const uint4 wv = *reinterpret_cast<const uint4*>(prow + ((hq ^ pswz) << 4));
                                const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const int c = hq * 4 + j;  // 16-byte chunk = one word
                                    uint32_t p[4];
                                    deq4_word(wd[j], s2, b2, p);
                                    *reinterpret_cast<uint4*>(brow + ((c ^ (r & 7)) << 4)) =
                                        make_uint4(p[0], p[1], p[2], p[3]);
                                }
                            }
                        } else {
#pragma unroll
                            for (int hq0 = 0; hq0 < 4 / WR::kTpr; ++hq0) {
                                const int hq = pt * (4 / WR::kTpr) + hq0;  // this thread's 16-byte parts
                                const uint4 wv = *reinterpret_cast<const uint4*>(prow + ((hq ^ pswz) << 4));
                                const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                                for (int j = 0; j < 2; ++j) {
                                    const int c = hq * 2 + j;  // 16-byte chunk = two words
                                    const uint32_t w0 = wd[2 * j], w1 = wd[2 * j + 1];
                                    *reinterpret_cast<uint4*>(brow + ((c ^ (r & 7)) << 4)) =
                                        make_uint4(deq8(w0, 0x5140u, s2, b2),
                                                   deq8(w0, 0x7362u, s2, b2),
                                                   deq8(w1, 0x5140u, s2, b2),
                                                   deq8(w1, 0x7362u, s2, b2));
                                }
                            }
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
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int sub = warp & 3;  // TMEM sub-partition of this warp
        const int row = sub * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(sub * 32) << 16;
        const float k2 = cap > 0.f ? 2.f * kLog2e / cap : 0.f;
        int buf = 0;
        uint32_t aphase = 0;
        for (int u = blockIdx.x; u < W.units; u += gridDim.x) {
            int mt, seg, vt0, vt1;
            unit_coords(W, a.vt_begin, u, mt, seg, vt0, vt1);
            const int i = mt * BM + row;  // compact row of this thread
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
                if (skipped(mt, vt)) {
                    // The tile's coefficients of this row are written as zeros
                    // where the dh contraction reads them: when the other
                    // 128-row tile of its 256-row unit keeps the vocab tile.
                    const int pm = mt ^ 1;
                    const bool partner_skips =
                        pm >= a.skip_rows || a.skip[(int64_t)pm * a.skip_ld + vt] != 0;
                    if (EPI != EPI_SOFTMAX && !partner_skips && i < a.coeff_rows) {
                        __half* dst = a.coeff + (int64_t)i * a.coeff_ld +
                                      (int64_t)(vt - a.vt_begin) * BN;
                        const uint32_t zero[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll 1
                        for (int q = 0; q < BN / 16; ++q) tc::st_global_v8(dst + 16 * q, zero);
                    }
                    continue;
                }
                tc::mbar_wait(&accf[buf], aphase, abort_flag, err, tc::kErrTimeoutAccFull);
                tc::tc_fence_after();
                float tz = -INFINITY;  // the tile's maximum of z (blockMax)
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tc::tmem_ld32(tmem_base + lane_addr + buf * BN + c * 32, r);
                    tc::tmem_wait_ld();
                    const int64_t col0 = (int64_t)vt * BN + c * 32;
                    const int nvalid = (int)min((int64_t)32, V - col0);
                    float x[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
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
                                    const float t = fmaf(-2.f, tc::rcp_approx(tc::ex2_approx(xv * k2) + 1.f), 1.f);
                                    lg2p = fmaf(cap * t, kLog2e, -lsb);
                                    sech2 = fmaf(-t, t, 1.f);
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
                if (lane == 0) tc::mbar_arrive(&acce[buf]);
                if (++buf == 2) { buf = 0; aphase ^= 1; }
            }
            if (EPI == EPI_SOFTMAX && row_ok) {
                Partial p;
                p.m = m; p.s = s; p.v1 = v1; p.v2 = v2; p.i1 = i1; p.i2 = i2; p.status = *abort_flag; p.pad1 = 0;
                a.part[(int64_t)i * W.n_seg + seg] = p;
            }
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

int tc_fwd_smem_bytes(int bits) { return bits == 4 ? Layout<4>::SMEM : Layout<8>::SMEM; }

template <int BITS, int EPI>
static cudaError_t launch_t(const CUtensorMap& th, const CUtensorMap& tw, const TcFwdArgs& a,
                            int grid, cudaStream_t st) {
    if (cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(tc_fwd_kernel<BITS, EPI>),
                                          Layout<BITS>::SMEM))
        return e;
    tc_fwd_kernel<BITS, EPI><<<grid, Warps<BITS>::kThreads, Layout<BITS>::SMEM, st>>>(th, tw, a);
    return cudaGetLastError();
}

cudaError_t launch_tc_fwd(const CUtensorMap& th, const CUtensorMap& tw, const TcFwdArgs& a,
                          int bits, bool coeff_epilogue, int grid, cudaStream_t st) {
    if (bits == 4)
        return !coeff_epilogue ? launch_t<4, EPI_SOFTMAX>(th, tw, a, grid, st)
               : a.kbits != nullptr ? launch_t<4, EPI_FILTER>(th, tw, a, grid, st)
                                    : launch_t<4, EPI_COEFF>(th, tw, a, grid, st);
    return !coeff_epilogue ? launch_t<8, EPI_SOFTMAX>(th, tw, a, grid, st)
           : a.kbits != nullptr ? launch_t<8, EPI_FILTER>(th, tw, a, grid, st)
                                : launch_t<8, EPI_COEFF>(th, tw, a, grid, st);
}

}  // namespace qh

// qh_tc_dw.cu -- the head gradient dW (a variant the pages leave out: their
// head is frozen).
//
//     dW[v, :] = sum_m dlogp[m] * (1[v == t_m] - p[m, v]) * sech2[m, v] * h[m, :]
//
// the classifier gradient of the Apple CCE reference the pages cite next to
// flashCceBackward (page "mlx-bun 0.0.4 -> 0.0.6", src/train/flash-cce.ts).
// It reuses the backward's coefficient block C = p * sech2 * 2^14 (fp16,
// [tokens x chunk]) that the logit kernel writes per vocab chunk:
//
//     dW[v, :] = -(D * 2^-14) * sum_i C[i, v] * h'[i, :]  +  sum_{i : t_i = v} g_i * h[row_i, :]
//
// with h'[i, :] = fp16(h[row_i, :] * dlogp[row_i] / D), D = max |dlogp| over the
// active rows (so small cotangents stay clear of the fp16 subnormal range),
// and g_i = dlogp[row_i] * sech2(raw target logit of row i), the one-hot term,
// added exactly in fp32.
//
// The contraction runs on tcgen05 with both operands MN-major (the vocab index
// of C and the hidden index of h' are contiguous in memory) and no
// dequantization: M = 128 vocab rows per half of a 256-row unit, N = 256 or
// 128 hidden columns, K = 64 tokens per stage.  Every dW element of the chunk
// is written once, by one thread: the result is deterministic.
//
// The one-hot lists (rows i with t_i = v, ascending i) are built once per call
// by a counting sort whose placement step runs in one warp in row order, so
// rows that share a target are summed in a fixed order.
#include "qh_internal.cuh"
#include "qh_tc.cuh"
#include "qh_tmap.h"

namespace qh {

namespace {

constexpr int BMV = 128;          // vocab rows per MMA (M); a unit covers two halves
constexpr int BMU = 2 * BMV;
constexpr int BK = 64;            // tokens per stage (K)
constexpr int kThreads = 6 * 32;  // TMA warp, MMA warp, 4 epilogue warps
constexpr float kCoeffInvScale = 1.f / 16384.f;

template <int BN>
struct DwLayout {
    static constexpr int NS = 3;
    static constexpr int A_HALF = BMV * BK * 2;   // two 64-row MN blocks of 8 KB
    static constexpr int A_BYTES = 2 * A_HALF;
    static constexpr int B_BYTES = BN * BK * 2;   // BN / 64 MN blocks of 8 KB
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + NS * A_BYTES;
    static constexpr int OFF_BAR = OFF_B + NS * B_BYTES;
    static constexpr int BAR_BYTES = 8 * (2 * NS + 5) + 16;
    static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr uint32_t IDESC = tc::idesc_f16_f32(BMV, BN, true, true);
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) tc_dw_kernel(
    const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_hp,
    const TcDwArgs a) {
    using L = DwLayout<BN>;
    constexpr int NS = L::NS;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    // (offsetting the shared array itself keeps the accesses in the shared
    // address space; a round trip through an integer would make them generic)
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);  // TMA inputs landed
    uint64_t* empty = full + NS;  // inputs consumed (MMA commit)
    uint64_t* accf = empty + NS;  // the unit's accumulators are complete (MMA commit)
    uint64_t* acce = accf + 1;    // [h]: half h has been read out (epilogue warps)
    uint64_t* mdrain = acce + 2;  // MMA drain on the abort path
    uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(mdrain + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_sh + 1);
    int* err = a.err;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_active = *a.count;
    const int n_k = (n_active + BK - 1) / BK;
    const int n_vu = (a.chunk_rows + BMU - 1) / BMU;
    const int n_nt = a.H / BN;
    const int units = n_vu * n_nt;
    if (units == 0 || (int)blockIdx.x >= units) return;
    // No active rows: no MMAs; the epilogue writes the chunk's zeros.
    const bool no_k = n_k == 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], 1);
        }
        tc::mbar_init(accf, 1);
        tc::mbar_init(&acce[0], 4);
        tc::mbar_init(&acce[1], 4);
        tc::mbar_init(mdrain, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tmap_c);
        tc::prefetch_tmap(&tmap_hp);
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
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, fills = 0;
            bool ok = a.stall == 0;  // test switch: no loads, the waits expire
            for (int u = blockIdx.x; u < units && ok && !no_k; u += gridDim.x) {
                const int vu = u / n_nt, nt = u - vu * n_nt;
                for (int kk = 0; kk < n_k && ok; ++kk) {
                    ok = tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag, err,
                                       tc::kErrTimeoutEmpty);
                    if (!ok) break;
                    unsigned char* A = smem + L::OFF_A + stage * L::A_BYTES;
                    unsigned char* B = smem + L::OFF_B + stage * L::B_BYTES;
                    tc::mbar_arrive_expect_tx(&full[stage], L::A_BYTES + L::B_BYTES);
                    // A: coefficient columns (vocab) of the unit, 64 per box; rows = tokens.
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk)
                        tc::tma_load_2d(A + blk * (L::A_HALF / 2), &tmap_c, &full[stage],
                                        vu * BMU + 64 * blk, kk * BK);
                    // B: h' columns (hidden) of the N tile, 64 per box; rows = tokens.
#pragma unroll
                    for (int nb = 0; nb < BN / 64; ++nb)
                        tc::tma_load_2d(B + nb * 8192, &tmap_hp, &full[stage], nt * BN + 64 * nb,
                                        kk * BK);
                    ++fills;
                    if (++stage == NS) { stage = 0; phase ^= 1; }
                }
            }
            if (ok && !no_k) {
                // Drain: the last stages were consumed before the CTA exits.
                for (int i = 0; i < NS && ok; ++i) {
                    ok = tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag, err,
                                       tc::kErrTimeoutEmpty);
                    if (++stage == NS) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) tc::drain_ring(full, NS, fills, err);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, aphase = 0;
            // The operand descriptors of ring slot 0 (both MN-major: 64-element
            // MN blocks 8 KB apart); a slot's are these plus its byte offset
            // >> 4 in the 14-bit address field, which never carries (shared
            // addresses stay below 256 KB).
            const uint64_t ad_base = tc::sdesc_sw128(tc::smem_u32(smem + L::OFF_A), 8192, 1024);
            const uint64_t bd_base = tc::sdesc_sw128(tc::smem_u32(smem + L::OFF_B), 8192, 1024);
            for (int u = blockIdx.x; u < units && !no_k; u += gridDim.x) {
                // Half h's accumulator may be overwritten once the epilogue has
                // read it out: half 0 before the unit starts, half 1 before its
                // first MMA (so reading out half 1 overlaps the next unit).
                if (!tc::mbar_wait(&acce[0], aphase ^ 1, abort_flag, err, tc::kErrTimeoutAccEmpty))
                    goto mma_abort;
                tc::tc_fence_after();
                for (int kk = 0; kk < n_k; ++kk) {
                    if (!tc::mbar_wait(&full[stage], phase, abort_flag, err, tc::kErrTimeoutFull))
                        goto mma_abort;
                    tc::tc_fence_after();
                    const uint64_t ad0 = ad_base + (uint32_t)(stage * (L::A_BYTES >> 4));
                    const uint64_t bd0 = bd_base + (uint32_t)(stage * (L::B_BYTES >> 4));
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        if (hh == 1 && kk == 0) {
                            if (!tc::mbar_wait(&acce[1], aphase ^ 1, abort_flag, err,
                                               tc::kErrTimeoutAccEmpty))
                                goto mma_abort;
                            tc::tc_fence_after();
                        }
#pragma unroll
                        for (int ks2 = 0; ks2 < BK / 16; ++ks2)  // two 8-row K groups per K step
                            tc::umma_f16(tmem_base + hh * BN, ad0 + ((hh * L::A_HALF + 2048 * ks2) >> 4),
                                         bd0 + ((2048 * ks2) >> 4), L::IDESC,
                                         (kk > 0 || ks2 > 0) ? 1u : 0u);
                    }
                    tc::umma_commit(&empty[stage]);
                    if (++stage == NS) { stage = 0; phase ^= 1; }
                }
                tc::umma_commit(accf);
                aphase ^= 1;
            }
            goto mma_done;
        mma_abort:
            // Let every MMA issued so far finish before TMEM is released.
            tc::umma_commit(mdrain);
            tc::mbar_drain(mdrain, 0, err);
        mma_done:;
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int sub = warp & 3;  // TMEM lane quadrant of this warp
        const int row = sub * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(sub * 32) << 16;
        const float negscale = -(*a.dmax) * kCoeffInvScale;
        uint32_t aphase = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
            const int vu = u / n_nt, nt = u - vu * n_nt;
            // The rows' one-hot lists, fetched before the wait.
            int o0[2], o1[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int vc = vu * BMU + hh * BMV + row;  // column of the chunk
                const int64_t v = a.v_begin + vc;
                const bool ok = vc < a.chunk_rows && v < a.V;
                o0[hh] = ok ? a.offs[v] : 0;
                o1[hh] = ok ? a.offs[v + 1] : 0;
            }
            if (!no_k) {
                // Result ignored: the warp stays converged (see the abort policy).
                tc::mbar_wait(accf, aphase, abort_flag, err, tc::kErrTimeoutAccFull);
                tc::tc_fence_after();
            }
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                const int vc = vu * BMU + hh * BMV + row;
                const int64_t v = a.v_begin + vc;
                const bool row_ok = vc < a.chunk_rows && v < a.V;
                float* dst = a.dw + v * (int64_t)a.H + nt * BN;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    if (!no_k) {
                        tc::tmem_ld32(tmem_base + lane_addr + hh * BN + c * 32, r);
                        tc::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = 0u;
                    }
                    if (row_ok) {
                        float x[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]) * negscale;
                        // one-hot terms of the rows whose target is v, in row order
                        for (int e = o0[hh]; e < o1[hh]; ++e) {
                            const int i = a.idx[e];
                            const float gi = a.g[i];
                            const uint4* hp = reinterpret_cast<const uint4*>(
                                a.h + (int64_t)a.rows[i] * a.H + nt * BN + c * 32);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint4 hv = hp[q];
                                const __nv_bfloat16* hb = reinterpret_cast<const __nv_bfloat16*>(&hv);
#pragma unroll
                                for (int k = 0; k < 8; ++k)
                                    x[8 * q + k] = fmaf(gi, __bfloat162float(hb[k]), x[8 * q + k]);
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            tc::st_global_v8(dst + c * 32 + 8 * q,
                                             reinterpret_cast<const uint32_t*>(x + 8 * q));
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

template <int BN>
cudaError_t launch_dw_t(const CUtensorMap& tmap_c, const CUtensorMap& tmap_hp, const TcDwArgs& a,
                        int grid, cudaStream_t st) {
    using L = DwLayout<BN>;
    if (cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(tc_dw_kernel<BN>), L::SMEM))
        return e;
    tc_dw_kernel<BN><<<grid, kThreads, L::SMEM, st>>>(tmap_c, tmap_hp, a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- preparation

// D = max |dlogp| over the active rows (0 when there are none): one CTA.
__global__ void __launch_bounds__(1024) dw_dmax_kernel(const float* __restrict__ dlogp,
                                                       const int* __restrict__ rows,
                                                       const int* __restrict__ count,
                                                       float* __restrict__ dmax) {
    __shared__ float red[32];
    const int n = *count;
    float m = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, fabsf(dlogp[rows[i]]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < (int)(blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (threadIdx.x == 0) *dmax = m;
    }
}

// Compact row i: h'[i, :] = fp16(h[row_i, :] * dlogp[row_i] / D) (zeros past
// the active rows) and g[i] = dlogp[row_i] * sech2(exact raw target logit);
// rows whose target lies outside [0, V) get g = 0 (no one-hot term).
constexpr int kPrepThreads = 128;

__global__ void __launch_bounds__(kPrepThreads) dw_hprime_kernel(
    const uint32_t* __restrict__ wq, SbView sb, int64_t V, int H, int bits, float cap,
    const __nv_bfloat16* __restrict__ h, const int* __restrict__ rows,
    const int* __restrict__ count, const int32_t* __restrict__ targets,
    const float* __restrict__ dlogp, const float* __restrict__ dmax, __half* __restrict__ hp,
    float* __restrict__ g) {
    const int64_t i = blockIdx.x;
    const bool act = i < *count;
    const int r = act ? rows[i] : 0;
    const float D = *dmax;
    const float f = act && D > 0.f ? dlogp[r] / D : 0.f;
    for (int u = threadIdx.x; u < H / 8; u += kPrepThreads) {
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (act) {
            const uint4 in = *reinterpret_cast<const uint4*>(h + (int64_t)r * H + 8 * u);
            const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&in);
            __half y[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) y[k] = __float2half_rn(__bfloat162float(x[k]) * f);
            out = *reinterpret_cast<const uint4*>(y);
        }
        *reinterpret_cast<uint4*>(hp + i * H + 8 * u) = out;
    }
    if (threadIdx.x < 32) {
        float gi = 0.f;
        if (act) {
            const int32_t t = targets[r];
            if (t >= 0 && (int64_t)t < V) {
                const float raw =
                    warp_exact_logit<10>(h + (int64_t)r * H, wq, sb, t, H, bits);
                float sech2 = 1.f;
                if (cap > 0.f) {
                    const float th = tanhf(raw / cap);
                    sech2 = 1.f - th * th;
                }
                gi = dlogp[r] * sech2;
            }
        }
        if (threadIdx.x == 0) g[i] = gi;
    }
}

// cnt[v] = number of active rows whose target is v (cnt zeroed by the host).
__global__ void dw_count_kernel(const int* __restrict__ rows, const int* __restrict__ count,
                                const int32_t* __restrict__ targets, int64_t V,
                                int* __restrict__ cnt) {
    const int n = *count;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t t = targets[rows[i]];
        if (t >= 0 && (int64_t)t < V) atomicAdd(&cnt[t], 1);
    }
}

// offs = exclusive prefix sum of cnt (V + 1 entries); cursor = offs[0 .. V).
// One CTA: each thread scans a contiguous span, then the span totals.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) dw_scan_kernel(const int* __restrict__ cnt,
                                                               int64_t V, int* __restrict__ offs,
                                                               int* __restrict__ cursor) {
    __shared__ int tot[kScanThreads];
    const int64_t span = (V + kScanThreads - 1) / kScanThreads;
    const int64_t b = threadIdx.x * span, e = b + span < V ? b + span : V;
    int s = 0;
    for (int64_t v = b; v < e; ++v) s += cnt[v];
    tot[threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.x == 0) {  // 1024 sequential adds
        int run = 0;
        for (int k = 0; k < kScanThreads; ++k) {
            const int x = tot[k];
            tot[k] = run;
            run += x;
        }
        offs[V] = run;
    }
    __syncthreads();
    int run = tot[threadIdx.x];
    for (int64_t v = b; v < e; ++v) {
        offs[v] = run;
        cursor[v] = run;
        run += cnt[v];
    }
}

// Stable placement: one warp walks the active rows in order, 32 at a time;
// lanes with equal targets take consecutive slots in lane order
// (__match_any_sync), and the first of them advances the target's cursor.
__global__ void dw_place_kernel(const int* __restrict__ rows, const int* __restrict__ count,
                                const int32_t* __restrict__ targets, int64_t V,
                                int* __restrict__ cursor, int* __restrict__ idx) {
    const int lane = threadIdx.x & 31;
    const int n = *count;
    for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + lane;
        int32_t t = -1;
        if (i < n) {
            t = targets[rows[i]];
            if (t < 0 || (int64_t)t >= V) t = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, t);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int base = t >= 0 ? cursor[t] : 0;
        if (t >= 0) idx[base + rank] = i;
        __syncwarp();
        if (t >= 0 && rank == 0) cursor[t] = base + __popc(peers);
        __syncwarp();
    }
}

__global__ void dw_poison_kernel(const int* __restrict__ err, float* __restrict__ dw, int64_t n) {
    if (*err == 0) return;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n;
         k += (int64_t)gridDim.x * blockDim.x)
        dw[k] = __int_as_float(0x7fc00000);
}

}  // namespace

cudaError_t launch_dw_poison(const int* err, float* dw, int64_t n, cudaStream_t st) {
    dw_poison_kernel<<<1024, 256, 0, st>>>(err, dw, n);
    return cudaGetLastError();
}

int tc_dw_smem_bytes(int H) {
    return tc_dh_cols(H) == 256 ? DwLayout<256>::SMEM : DwLayout<128>::SMEM;
}

cudaError_t launch_dw_prep(const uint32_t* wq, SbView sb,
                           int64_t V, int H, int bits, float cap, const __nv_bfloat16* h,
                           const int* rows, const int* count, const int32_t* targets,
                           const float* dlogp, int64_t Mpad, float* dmax, __half* hp, float* g,
                           int* cnt, int* offs, int* cursor, int* idx, cudaStream_t st) {
    cudaError_t e;
    dw_dmax_kernel<<<1, 1024, 0, st>>>(dlogp, rows, count, dmax);
    if ((e = cudaGetLastError())) return e;
    dw_hprime_kernel<<<(unsigned)Mpad, kPrepThreads, 0, st>>>(wq, sb, V, H, bits, cap,
                                                              h, rows, count, targets, dlogp, dmax,
                                                              hp, g);
    if ((e = cudaGetLastError())) return e;
    if ((e = cudaMemsetAsync(cnt, 0, sizeof(int) * (size_t)V, st))) return e;
    const unsigned cgrid = (unsigned)((Mpad + 255) / 256);
    dw_count_kernel<<<cgrid, 256, 0, st>>>(rows, count, targets, V, cnt);
    if ((e = cudaGetLastError())) return e;
    dw_scan_kernel<<<1, kScanThreads, 0, st>>>(cnt, V, offs, cursor);
    if ((e = cudaGetLastError())) return e;
    dw_place_kernel<<<1, 32, 0, st>>>(rows, count, targets, V, cursor, idx);
    return cudaGetLastError();
}

cudaError_t launch_tc_dw(const CUtensorMap& tmap_c, const CUtensorMap& tmap_hp, const TcDwArgs& a,
                         int grid, cudaStream_t st) {
    return tc_dh_cols(a.H) == 256 ? launch_dw_t<256>(tmap_c, tmap_hp, a, grid, st)
                                  : launch_dw_t<128>(tmap_c, tmap_hp, a, grid, st);
}

}  // namespace qh

// qh_finalize.cu -- steps a6/a7 (forward) and a11 (backward) of the hot path.
//
// Forward: merge the per-(row, vocab split) partials in a fixed order,
//   gMax = max_b m_b;  lse = gMax + log(sum_b s_b * exp(m_b - gMax))
// (the cross-vocab-block merge of flashCceForward on the page "mlx-bun 0.0.4
// -> 0.0.6", src/train/flash-cce.ts, done here on device in a fixed order
// instead of in MLX ops), then
//   * the target logit is recomputed exactly in fp32 (h widened from bf16,
//     w = fmaf(scale, q, bias) from the caller's scales and biases in their
//     own type), so logp = softcap(raw_target) - lse carries no fp16 operand
//     rounding;
//   * the two argmax candidates (the best two raw logits over all splits)
//     are recomputed the same way and the better exact value wins, lowest index on ties (argmax over the raw logits, which
//     picksBatched on the page "mlx-bun 0.0.8 -> 0.0.10" notes is the argmax of
//     the capped, lse-shifted log-probs too);
//   * masked rows get logp = 0, lse = 0, argmax = -1.
// Backward: dh[r,:] = sum_s dh_partial[s, i, :] (fixed order) plus the one-hot
// term dlogp * sech2(raw_target) * w[target, :] added exactly in fp32; masked
// rows are written as exact zeros.
#include "qh_internal.cuh"
#include "qh_tc.cuh"

namespace qh {

namespace {

// Threads per row: 128 for small batches (the verify window: each row's
// latency is the call's), 64 from 1024 rows (twice the rows in flight; each
// row one more round of its exact dot products).
constexpr int kFwdFinRowsWide = 1024;

template <int kFinThreads>
__global__ void __launch_bounds__(kFinThreads) fwd_finalize_kernel(
    const uint32_t* __restrict__ wq, SbView sb, int64_t V, int H, int bits, float cap,
    const __nv_bfloat16* __restrict__ h, const int* __restrict__ pos,
    const int32_t* __restrict__ targets, const Partial* __restrict__ part, int S,
    const int* __restrict__ S_dev, const int* __restrict__ err,
    float* __restrict__ logp, float* __restrict__ lse, int32_t* __restrict__ argmax) {
    tc::grid_dep_wait();  // the head kernel's partials (programmatic dependent launch)
    tc::grid_dep_trigger();
    const int64_t r = blockIdx.x;
    const int i = pos[r];
    if (S_dev) S = *S_dev;
    if (err && *err != 0 && i >= 0) {
        // The head kernel gave up (a bounded wait expired): poison the row.
        if (threadIdx.x == 0) {
            if (logp) logp[r] = __int_as_float(0x7fc00000);
            if (lse) lse[r] = __int_as_float(0x7fc00000);
            if (argmax) argmax[r] = -1;
        }
        return;
    }
    if (i < 0) {
        if (threadIdx.x == 0) {
            if (logp) logp[r] = 0.f;
            if (lse) lse[r] = 0.f;
            if (argmax) argmax[r] = -1;
        }
        return;
    }
    __shared__ Partial red[kFinThreads / 32];
    __shared__ float exact[3 * (kFinThreads / 32)];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    RowState st;
    st.init();
    int bad = 0;  // some CTA that wrote a partial of this row gave up
    // Up to 4 partials per thread per round, loads issued before the merges.
    const Partial* prow = part + (int64_t)i * S;
    for (int s0 = threadIdx.x; s0 < S; s0 += 4 * kFinThreads) {
        Partial buf[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (s0 + k * kFinThreads < S) buf[k] = prow[s0 + k * kFinThreads];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (s0 + k * kFinThreads < S) {
                st.merge(buf[k]);
                bad |= buf[k].status;
            }
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) {
            if (logp) logp[r] = __int_as_float(0x7fc00000);
            if (lse) lse[r] = __int_as_float(0x7fc00000);
            if (argmax) argmax[r] = -1;
        }
        return;
    }
#pragma unroll
    for (int o = 1; o <= 16; o <<= 1) st.shfl_merge(o);
    if (lane == 0) red[warp] = st.to_partial();
    __syncthreads();
    RowState fin;
    fin.init();
    for (int w = 0; w < kFinThreads / 32; ++w) fin.merge(red[w]);

    const __nv_bfloat16* hrow = h + r * (int64_t)H;
    const int32_t t = targets ? targets[r] : -1;
    const bool t_ok = t >= 0 && (int64_t)t < V;
    // The exact logits of candidate 1, candidate 2 (if any) and the target,
    // shared by the whole block: each thread takes the 8-element units
    // u = threadIdx.x, + 128, ... of all three rows (one load of h per unit),
    // then the block sums them in a fixed order.
    const int n1 = fin.i1 < V ? 1 : 0;  // (an empty slot holds INT32_MAX)
    const int n2 = fin.i2 < V ? 1 : 0;
    const int64_t vr[3] = {n1 ? (int64_t)fin.i1 : -1, n2 ? (int64_t)fin.i2 : -1,
                           t_ok ? (int64_t)t : -1};
    const int units = H / 8, G = H / 64, wpr = H * bits / 32;
    float dot[3] = {0.f, 0.f, 0.f};
#pragma unroll 2
    for (int u = threadIdx.x; u < units; u += kFinThreads) {
        const uint4 hv = *reinterpret_cast<const uint4*>(hrow + 8 * u);
        const __nv_bfloat16* hp = reinterpret_cast<const __nv_bfloat16*>(&hv);
#pragma unroll
        for (int c = 0; c < 3; ++c) {
            if (vr[c] < 0) continue;
            const uint32_t* wrow = wq + vr[c] * wpr;
            const int64_t gi = vr[c] * G + u / 8;
            const float sc = sb_elem(sb.s, gi, sb.type), bi = sb_elem(sb.b, gi, sb.type);
            const uint32_t w0 = bits == 4 ? wrow[u] : wrow[2 * u];
            const uint32_t w1 = bits == 4 ? 0u : wrow[2 * u + 1];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t q = bits == 4 ? (w0 >> (4 * e)) & 15u
                                             : ((e < 4 ? w0 : w1) >> (8 * (e & 3))) & 255u;
                dot[c] = fmaf(__bfloat162float(hp[e]), fmaf(sc, (float)q, bi), dot[c]);
            }
        }
    }
#pragma unroll
    for (int c = 0; c < 3; ++c) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) dot[c] += __shfl_xor_sync(0xffffffffu, dot[c], o);
        if (lane == 0) exact[warp * 3 + c] = dot[c];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float x[3];
        for (int c = 0; c < 3; ++c) {
            x[c] = 0.f;
            for (int w = 0; w < kFinThreads / 32; ++w) x[c] += exact[w * 3 + c];
        }
        const float l = fin.m + logf(fin.s);
        float best = -INFINITY;
        int bi = INT32_MAX;
        for (int c = 0; c < 2; ++c) {
            const int v = c == 0 ? fin.i1 : fin.i2;
            if (vr[c] >= 0 && better(x[c], v, best, bi)) { best = x[c]; bi = v; }
        }
        if (lse) lse[r] = l;
        if (argmax) argmax[r] = bi == INT32_MAX ? -1 : bi;
        if (logp) logp[r] = t_ok ? softcap_exact(x[2], cap) - l : __int_as_float(0x7fc00000);
    }
}

// 8-element units of a row per thread (at most two): H <= kMaxH = 8192 is at
// most 1024 units, 512 threads; rows of H <= 4096 take 256 threads, so that
// twice as many rows (each a latency-bound round of loads) are in flight.
constexpr int kBwdFinUnits = 2;
constexpr int kBwdFinThreadsMax = kMaxH / 8 / kBwdFinUnits;

// One row per block.  Every thread takes the row's 8-element units u = t,
// t + THREADS: in one round of loads it reads, per unit, the S partial-dh
// slices (the sums it will write) and the target's weights and the hidden
// states (its part of the exact target logit), so the row costs one global
// latency, not a dot product by one warp followed by the sums.  The target
// logit is reduced over the block in a fixed order (deterministic), then
// dh = sum of slices + dlogp * sech2(target logit) * w_target, exactly in fp32.
template <int kBwdFinThreads>
__global__ void __launch_bounds__(kBwdFinThreads) bwd_finalize_kernel(
    const uint32_t* __restrict__ wq, SbView sb, int64_t V, int H, int bits, float cap,
    const __nv_bfloat16* __restrict__ h, const int* __restrict__ pos,
    const int32_t* __restrict__ targets, const float* __restrict__ dlogp,
    const float* __restrict__ dhp, int S, int64_t Mpad, const int* __restrict__ err,
    float* __restrict__ dh) {
    const int64_t r = blockIdx.x;
    const int i = pos[r];
    float* out = dh + r * (int64_t)H;
    if (i < 0) {
        for (int d = threadIdx.x; d < H; d += kBwdFinThreads) out[d] = 0.f;
        return;
    }
    if (*err != 0) {
        // A head kernel gave up (a bounded wait expired): poison the row.
        for (int d = threadIdx.x; d < H; d += kBwdFinThreads) out[d] = __int_as_float(0x7fc00000);
        return;
    }
    __shared__ float part_sh[kBwdFinThreads / 32];
    __shared__ float coef_sh;
    const int32_t t = targets[r];
    const bool t_ok = t >= 0 && (int64_t)t < V;
    const int units = H / 8, G = H / 64, wpr = H * bits / 32;
    const uint32_t* wrow = wq + (t_ok ? (int64_t)t : 0) * wpr;
    const __nv_bfloat16* hrow = h + r * (int64_t)H;
    float acc[kBwdFinUnits][8];  // the slice sums of this thread's units
    float wt[kBwdFinUnits][8];   // the target's weights of those units
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < kBwdFinUnits; ++k) {
        const int u = threadIdx.x + k * kBwdFinThreads;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[k][e] = wt[k][e] = 0.f;
        if (u >= units) continue;
        for (int sl = 0; sl < S; ++sl) {
            const float4* src = reinterpret_cast<const float4*>(dhp + ((int64_t)sl * Mpad + i) * H + 8 * u);
            const float4 a0 = src[0], a1 = src[1];
            acc[k][0] += a0.x; acc[k][1] += a0.y; acc[k][2] += a0.z; acc[k][3] += a0.w;
            acc[k][4] += a1.x; acc[k][5] += a1.y; acc[k][6] += a1.z; acc[k][7] += a1.w;
        }
        if (t_ok) {
            const int64_t gi = (int64_t)t * G + u / 8;
            const float sc = sb_elem(sb.s, gi, sb.type), bi = sb_elem(sb.b, gi, sb.type);
            const uint4 hv = *reinterpret_cast<const uint4*>(hrow + 8 * u);
            const __nv_bfloat16* hp = reinterpret_cast<const __nv_bfloat16*>(&hv);
            const uint32_t w0 = bits == 4 ? wrow[u] : wrow[2 * u];
            const uint32_t w1 = bits == 4 ? 0u : wrow[2 * u + 1];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t q = bits == 4 ? (w0 >> (4 * e)) & 15u
                                             : ((e < 4 ? w0 : w1) >> (8 * (e & 3))) & 255u;
                wt[k][e] = fmaf(sc, (float)q, bi);
                dot = fmaf(__bfloat162float(hp[e]), wt[k][e], dot);
            }
        }
    }
    // The target logit: warp sums, then the warps in order.
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if ((threadIdx.x & 31) == 0) part_sh[threadIdx.x >> 5] = dot;
    __syncthreads();
    if (threadIdx.x == 0) {
        float raw = 0.f;
        for (int w = 0; w < kBwdFinThreads / 32; ++w) raw += part_sh[w];
        float sech2 = 1.f;
        if (cap > 0.f) {
            const float th = tanhf(raw / cap);
            sech2 = 1.f - th * th;
        }
        coef_sh = t_ok ? dlogp[r] * sech2 : __int_as_float(0x7fc00000);
    }
    __syncthreads();
    const float coef = coef_sh;
#pragma unroll
    for (int k = 0; k < kBwdFinUnits; ++k) {
        const int u = threadIdx.x + k * kBwdFinThreads;
        if (u >= units) continue;
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = fmaf(coef, wt[k][e], acc[k][e]);
        float4* dst = reinterpret_cast<float4*>(out + 8 * u);
        dst[0] = make_float4(o[0], o[1], o[2], o[3]);
        dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    }
}

}  // namespace

cudaError_t launch_fwd_finalize(const uint32_t* wq, SbView sb,
                                int64_t V, int H, int bits, float cap, const __nv_bfloat16* h,
                                const int* pos, const int32_t* targets, const Partial* part, int S,
                                const int* S_dev, const int* err, float* logp,
                                float* lse, int32_t* argmax, int64_t M, cudaStream_t st) {
    void* args[] = {&wq, &sb, &V,     &H,   &bits,  &cap,   &h,      &pos,
                    &targets, &part, &S, &S_dev, &err, &logp, &lse, &argmax};
    if (M >= kFwdFinRowsWide)
        return launch_dependent(reinterpret_cast<const void*>(fwd_finalize_kernel<64>),
                                dim3((unsigned)M), dim3(64), 0, st, args);
    return launch_dependent(reinterpret_cast<const void*>(fwd_finalize_kernel<128>),
                            dim3((unsigned)M), dim3(128), 0, st, args);
}

// Longest accepted draft prefix per verify window (page "mlx-bun 0.0.8 ->
// 0.0.10", src/spec/generate.ts: the accept loop that follows picksBatched).
// Window b holds W = gamma + 1 consecutive rows of the forward's argmax;
// n_accept[b] = the first k < gamma with draft[b, k] != argmax[b, k] (gamma if
// there is none) and next_token[b] = argmax[b, n_accept[b]]: the target's own
// token at the first rejected position, or the bonus token after a fully
// accepted draft.  One warp per window.
__global__ void accept_prefix_kernel(const int32_t* __restrict__ argmax,
                                     const int32_t* __restrict__ draft, int64_t B, int W,
                                     int32_t* __restrict__ n_accept,
                                     int32_t* __restrict__ next_token) {
    const int64_t b = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (b >= B) return;
    const int gamma = W - 1;
    int n = gamma;
    for (int k0 = 0; k0 < gamma; k0 += 32) {
        const int k = k0 + lane;
        const bool miss = k < gamma && draft[b * gamma + k] != argmax[b * W + k];
        const unsigned bal = __ballot_sync(0xffffffffu, miss);
        if (bal) {  // the same for every lane
            n = k0 + __ffs(bal) - 1;
            break;
        }
    }
    if (lane == 0) {
        n_accept[b] = n;
        if (next_token) next_token[b] = argmax[b * W + n];
    }
}

cudaError_t launch_accept_prefix(const int32_t* argmax, const int32_t* draft, int64_t B, int W,
                                 int32_t* n_accept, int32_t* next_token, cudaStream_t st) {
    constexpr int kWarpsPerCta = 8;
    const unsigned grid = (unsigned)((B + kWarpsPerCta - 1) / kWarpsPerCta);
    accept_prefix_kernel<<<grid, 32 * kWarpsPerCta, 0, st>>>(argmax, draft, B, W, n_accept,
                                                             next_token);
    return cudaGetLastError();
}

cudaError_t launch_bwd_finalize(const uint32_t* wq, SbView sb,
                                int64_t V, int H, int bits, float cap, const __nv_bfloat16* h,
                                const int* pos, const int32_t* targets, const float* dlogp,
                                const float* dhp, int S, int64_t Mpad, const int* err, float* dh,
                                int64_t M, cudaStream_t st) {
    static_assert(kBwdFinThreadsMax == 512, "two units per thread cover kMaxH with 512 threads");
    if (H <= 4096)
        bwd_finalize_kernel<256><<<(unsigned)M, 256, 0, st>>>(wq, sb, V, H, bits, cap, h, pos,
                                                              targets, dlogp, dhp, S, Mpad, err, dh);
    else
        bwd_finalize_kernel<512><<<(unsigned)M, 512, 0, st>>>(wq, sb, V, H, bits, cap, h, pos,
                                                              targets, dlogp, dhp, S, Mpad, err, dh);
    return cudaGetLastError();
}

}  // namespace qh

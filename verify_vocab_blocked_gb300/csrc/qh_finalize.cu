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

constexpr int kFinThreads = 128;

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
    __shared__ float exact[2 * 32 + 1];
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
    // Work items: candidate 1, candidate 2 (if any), then the target.
    const int n1 = fin.i1 < V ? 1 : 0;  // (an empty slot holds INT32_MAX)
    const int n2 = fin.i2 < V ? 1 : 0;
    const int nitems = n1 + n2 + 1;
    for (int it = warp; it < nitems; it += kFinThreads / 32) {
        int64_t v;
        if (it < n1) v = fin.i1;
        else if (it < n1 + n2) v = fin.i2;
        else v = t_ok ? t : -1;
        float x = 0.f;
        if (v >= 0) x = warp_exact_logit<10>(hrow, wq, sb, v, H, bits);
        if (lane == 0) exact[it] = x;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const float l = fin.m + logf(fin.s);
        float best = -INFINITY;
        int bi = INT32_MAX;
        for (int it = 0; it < n1 + n2; ++it) {
            const int v = it < n1 ? fin.i1 : fin.i2;
            if (better(exact[it], v, best, bi)) { best = exact[it]; bi = v; }
        }
        if (lse) lse[r] = l;
        if (argmax) argmax[r] = bi == INT32_MAX ? -1 : bi;
        if (logp) logp[r] = t_ok ? softcap_exact(exact[n1 + n2], cap) - l : __int_as_float(0x7fc00000);
    }
}

constexpr int kBwdFinThreads = 256;

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
    __shared__ float coef_sh;
    const int32_t t = targets[r];
    const bool t_ok = t >= 0 && (int64_t)t < V;
    if (threadIdx.x < 32) {
        float raw = 0.f;
        if (t_ok) raw = warp_exact_logit(h + r * (int64_t)H, wq, sb, t, H, bits);
        if (threadIdx.x == 0) {
            float sech2 = 1.f;
            if (cap > 0.f) {
                const float th = tanhf(raw / cap);
                sech2 = 1.f - th * th;
            }
            coef_sh = t_ok ? dlogp[r] * sech2 : __int_as_float(0x7fc00000);
        }
    }
    __syncthreads();
    const float coef = coef_sh;
    for (int d = threadIdx.x; d < H; d += kBwdFinThreads) {
        float acc = 0.f;
        for (int s = 0; s < S; ++s) acc += dhp[((int64_t)s * Mpad + i) * H + d];
        const float wt = t_ok ? dequant_elem(wq, sb, t, d, H, bits) : 0.f;
        out[d] = fmaf(coef, wt, acc);
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
    return launch_dependent(reinterpret_cast<const void*>(fwd_finalize_kernel), dim3((unsigned)M),
                            dim3(kFinThreads), 0, st, args);
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
    bwd_finalize_kernel<<<(unsigned)M, kBwdFinThreads, 0, st>>>(wq, sb, V, H, bits,
                                                                 cap, h, pos, targets, dlogp, dhp,
                                                                 S, Mpad, err, dh);
    return cudaGetLastError();
}

}  // namespace qh

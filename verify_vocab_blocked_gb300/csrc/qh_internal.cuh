// qh_internal.cuh -- declarations shared by the translation units of libqhead.so.
// Not a public header: the public C ABI is include/qhead.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

namespace qh {

// Sets the calling thread's qhead_last_error() message.
void set_error(const std::string& msg);

// Per-(row, vocab split) partial of the forward: online-softmax state over the
// split's vocab rows (m = max z, s = sum exp(z - m)) and two argmax candidates
// with their vocab indices (the split's two best raw logits; the tensor-core
// kernel's are the maxima of its two best 32-column slices; empty entries hold
// v = -inf, i = INT32_MAX).  status: 0, or the code of a bounded wait that
// expired in the CTA that wrote the record (the finalize then poisons the row).
struct __align__(32) Partial {
    float m, s, v1, v2;
    int i1, i2, status, pad1;
};

// Element types of the head's scales and biases (the values of QHEAD_SB_* in
// the public header).
constexpr int kSbF16 = 0, kSbBf16 = 1, kSbF32 = 2;

// The caller's scales and biases, each [V, H/64], in their own element type.
// The exact fp32 parts of the path (target logit, argmax recheck, one-hot
// term) read them through sb_elem; the tensor-core and streaming kernels read
// an fp16 copy when the type is not fp16 (launch_sb_to_f16).
struct SbView {
    const void* s;
    const void* b;
    int type;
};

// Element i of a scale or bias array, widened to fp32 exactly.
__device__ __forceinline__ float sb_elem(const void* p, int64_t i, int type) {
    if (type == kSbF32) return static_cast<const float*>(p)[i];
    const unsigned short u = static_cast<const unsigned short*>(p)[i];
    if (type == kSbBf16) return __uint_as_float(static_cast<uint32_t>(u) << 16);
    return __half2float(__ushort_as_half(u));
}

constexpr int kTokGroup = 8;      // tokens per weight-streaming CTA (mma n = 8)
constexpr int kMaxH = 8192;
constexpr int kRowPad = 128;      // compacted row count is padded to this

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// Soft cap z = cap * tanh(raw / cap) (cap <= 0: identity), accurate tanhf.
__device__ __forceinline__ float softcap_exact(float raw, float cap) {
    return cap > 0.f ? cap * tanhf(raw / cap) : raw;
}

struct RowState {
    float m, s, v1, v2;
    int i1, i2;
    __device__ __forceinline__ void init() {
        m = -INFINITY; s = 0.f; v1 = -INFINITY; v2 = -INFINITY; i1 = INT32_MAX; i2 = INT32_MAX;
    }
    // One logit: z (capped) feeds the softmax state, raw feeds the top-2.
    __device__ __forceinline__ void push(float z, float raw, int idx) {
        if (z > m) { s = s * expf(m - z) + 1.f; m = z; }
        else       { s += expf(z - m); }
        if (better(raw, idx, v1, i1))      { v2 = v1; i2 = i1; v1 = raw; i1 = idx; }
        else if (better(raw, idx, v2, i2)) { v2 = raw; i2 = idx; }
    }
    __device__ __forceinline__ void merge(float om, float os, float ov1, int oi1, float ov2, int oi2) {
        const float nm = fmaxf(m, om);
        if (nm == -INFINITY) { s = 0.f; }
        else { s = s * expf(m - nm) + os * expf(om - nm); }
        m = nm;
        if (better(ov1, oi1, v1, i1)) {
            if (better(v1, i1, ov2, oi2)) { v2 = v1; i2 = i1; } else { v2 = ov2; i2 = oi2; }
            v1 = ov1; i1 = oi1;
        } else if (better(ov1, oi1, v2, i2)) {
            v2 = ov1; i2 = oi1;
        }
    }
    __device__ __forceinline__ void merge(const RowState& o) { merge(o.m, o.s, o.v1, o.i1, o.v2, o.i2); }
    __device__ __forceinline__ void merge(const Partial& o) { merge(o.m, o.s, o.v1, o.i1, o.v2, o.i2); }
    __device__ __forceinline__ void shfl_merge(int lane_mask) {
        RowState o;
        o.m = __shfl_xor_sync(0xffffffffu, m, lane_mask);
        o.s = __shfl_xor_sync(0xffffffffu, s, lane_mask);
        o.v1 = __shfl_xor_sync(0xffffffffu, v1, lane_mask);
        o.v2 = __shfl_xor_sync(0xffffffffu, v2, lane_mask);
        o.i1 = __shfl_xor_sync(0xffffffffu, i1, lane_mask);
        o.i2 = __shfl_xor_sync(0xffffffffu, i2, lane_mask);
        // Merge in a lane-order-independent way so both partners end equal:
        // the lower lane's state always comes first.
        const int lane = threadIdx.x & 31;
        if (lane & lane_mask) { RowState mine = *this; *this = o; merge(mine); }
        else { merge(o); }
    }
    __device__ __forceinline__ Partial to_partial() const {
        Partial p; p.m = m; p.s = s; p.v1 = v1; p.v2 = v2; p.i1 = i1; p.i2 = i2; p.status = 0; p.pad1 = 0;
        return p;
    }
};

// Exact fp32 logit of one (row of h, vocab row) pair, computed by one warp:
// h widened from bf16 exactly, w = fmaf(scale, q, bias) in fp32.  Every lane
// returns the same value (fixed butterfly order).  U: 8-element units per lane
// whose loads are issued together (one round trip per round).
template <int U = 4>
__device__ __forceinline__ float warp_exact_logit(const __nv_bfloat16* __restrict__ hrow,
                                                  const uint32_t* __restrict__ wq, SbView sb,
                                                  int64_t v, int H, int bits) {
    const int lane = threadIdx.x & 31;
    const int wpr = H * bits / 32;
    const int G = H / 64;
    const uint32_t* wrow = wq + v * (int64_t)wpr;
    const int64_t g0 = v * (int64_t)G;
    float acc = 0.f;
    // Units of 8 consecutive elements, U per lane per round, loads of a round
    // issued together.
    for (int u0 = lane; u0 < H / 8; u0 += U * 32) {
        uint4 hv[U];
        uint32_t w0[U], w1[U];
        float s[U], b[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int u = u0 + 32 * i;
            if (u < H / 8) {
                hv[i] = *reinterpret_cast<const uint4*>(hrow + 8 * u);
                s[i] = sb_elem(sb.s, g0 + u / 8, sb.type);
                b[i] = sb_elem(sb.b, g0 + u / 8, sb.type);
                if (bits == 4) { w0[i] = wrow[u]; w1[i] = 0u; }
                else { w0[i] = wrow[2 * u]; w1[i] = wrow[2 * u + 1]; }
            }
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            if (u0 + 32 * i < H / 8) {
                const __nv_bfloat16* hp = reinterpret_cast<const __nv_bfloat16*>(&hv[i]);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    uint32_t q;
                    if (bits == 4) q = (w0[i] >> (4 * k)) & 15u;
                    else q = ((k < 4 ? w0[i] : w1[i]) >> (8 * (k & 3))) & 255u;
                    acc = fmaf(__bfloat162float(hp[k]), fmaf(s[i], (float)q, b[i]), acc);
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

// fp32 dequantized element w[v,d].
__device__ __forceinline__ float dequant_elem(const uint32_t* __restrict__ wq, SbView sb,
                                              int64_t v, int d, int H, int bits) {
    const int per = 32 / bits;
    const uint32_t word = wq[v * (int64_t)(H * bits / 32) + d / per];
    const uint32_t q = (word >> (bits * (d % per))) & ((1u << bits) - 1u);
    const int64_t gi = v * (int64_t)(H / 64) + d / 64;
    return fmaf(sb_elem(sb.s, gi, sb.type), (float)q, sb_elem(sb.b, gi, sb.type));
}

// ------------------------------------------------------------- launchers
// Each returns the cudaError_t of its launch.

cudaError_t launch_compact(const uint8_t* mask, int64_t M, int64_t Mpad, int* rows, int* pos,
                           int* count, int* err, cudaStream_t st);
// Compaction and conversion in one single-CTA launch (small M only).
constexpr int64_t kFusedPrologueMaxM = 256;
cudaError_t launch_prologue_fused(const uint8_t* mask, const __nv_bfloat16* h, int64_t M,
                                  int64_t Mpad, int H, int bits, int* rows, int* pos, int* count,
                                  __half* h16, int64_t nrows, int* err, cudaStream_t st);
// Scales and biases of another element type rounded to fp16 (nearest, ties
// to even) for the tensor-core and streaming kernels: n elements of each.
cudaError_t launch_sb_to_f16(SbView sb, int64_t n, __half* s16, __half* b16, cudaStream_t st);
cudaError_t launch_convert_h(const __nv_bfloat16* h, int64_t Mpad, int H, int bits, const int* rows,
                             const int* count, __half* h16, cudaStream_t st);
// Launches `fn` with programmatic stream serialization: its CTAs may start
// while the preceding kernel on `st` finishes, and wait for it with
// tc::grid_dep_wait() before touching memory that kernel may write.
cudaError_t launch_dependent(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             void** args);
cudaError_t launch_stream_fwd(const uint32_t* wq, const __half* scales, const __half* biases,
                              int64_t V, int H, int bits, float cap, const __nv_bfloat16* h,
                              const uint8_t* mask, int64_t M, int* rows, int* pos, int* count,
                              Partial* part, int S, int* err, int stall, cudaStream_t st);
// Skip map of the blockMax early exit: skip[mt * n_vt + vt] = 1 when every
// active row of 128-row tile mt has bmax - lse < ln(eps) on vocab tile vt and
// none of them targets it.
cudaError_t launch_skip_map(const float* bmax, int64_t ld, const float* lse,
                            const int32_t* targets, const int* rows, const int* count,
                            int64_t n_mt, int64_t n_vt, float eps, uint8_t* skip,
                            cudaStream_t st);
cudaError_t launch_fwd_finalize(const uint32_t* wq, SbView sb,
                                int64_t V, int H, int bits, float cap, const __nv_bfloat16* h,
                                const int* pos, const int32_t* targets, const Partial* part, int S,
                                const int* S_dev, const int* err, float* logp,
                                float* lse, int32_t* argmax, int64_t M, cudaStream_t st);
cudaError_t launch_bwd_finalize(const uint32_t* wq, SbView sb,
                                int64_t V, int H, int bits, float cap, const __nv_bfloat16* h,
                                const int* pos, const int32_t* targets, const float* dlogp,
                                const float* dhp, int S, int64_t Mpad, const int* err, float* dh,
                                int64_t M, cudaStream_t st);

// Host-side caches (thread-safe).  ensure_smem_limit raises a kernel's dynamic
// shared-memory limit on the current device once, skipping the runtime call
// when the device already allows `bytes`; device_sms returns the current
// device's SM count (0 on error).
cudaError_t ensure_smem_limit(const void* func, int bytes);
int device_sms();

cudaError_t launch_accept_prefix(const int32_t* argmax, const int32_t* draft, int64_t B, int W,
                                 int32_t* n_accept, int32_t* next_token, cudaStream_t st);

int stream_fwd_ctas_per_sm(int bits, int H);  // occupancy of the weight-streaming kernel

}  // namespace qh

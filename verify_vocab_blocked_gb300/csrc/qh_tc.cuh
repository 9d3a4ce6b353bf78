// qh_tc.cuh -- sm_103a building blocks for the tensor-core kernels: mbarriers
// with bounded waits, TMA tile loads, tensor-memory (TMEM) allocation and
// loads, tcgen05.mma (kind::f16, one CTA) and its shared-memory / instruction
// descriptors.  Written directly in inline PTX; no library code.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the encoder is looked up at run time)

#include "qh_internal.cuh"

namespace qh {
namespace tc {

// Every wait gives up after this long (nanoseconds of %globaltimer), records an
// error code and lets the kernel wind down instead of hanging the GPU.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s

// Error codes written to the kernel's error word.
constexpr int kErrTimeoutFull = 1, kErrTimeoutEmpty = 2, kErrTimeoutDequant = 3,
              kErrTimeoutAccFull = 4, kErrTimeoutAccEmpty = 5, kErrTimeoutDrain = 6;

// Limit of a drain wait on the abort path (copies and MMAs already issued
// always complete; this only bounds the wait if the device misbehaves).
constexpr uint64_t kDrainTimeoutNs = 100000000ull;  // 0.1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Programmatic dependent launch.  grid_dep_wait: block until the grids this
// launch depends on have completed and their writes are visible (returns at
// once for a launch without programmatic dependencies).  grid_dep_trigger:
// allow the next programmatically dependent launch on the stream to start
// (its CTAs run up to their own grid_dep_wait).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// *p += v, four fp32 lanes, performed at L2 (fire-and-forget: no value comes
// back, so no round trip).  Each lane is one fp32 addition rounded to
// nearest; subnormal inputs and results are flushed to zero.
__device__ __forceinline__ void red_add_v4(float* p, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// 32-byte global store of 8 words (the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if the
// CTA has been told to abort, another CTA has set the kernel's error word, or
// the wait ran past the time limit (then the error word and the abort flag
// are set).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* err, int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag || *reinterpret_cast<volatile int*>(err) != 0) return false;
        if (globaltimer() - t0 > kWaitTimeoutNs) {
            atomicCAS(err, 0, code);
            *abort_flag = 1;
            return false;
        }
    }
}

// As mbar_wait, but only this CTA's abort flag ends the wait early: for a
// kernel that clears the error word itself, whose other CTAs must not read a
// value left there by an earlier call.
__device__ __forceinline__ bool mbar_wait_cta(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag, int* err, int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitTimeoutNs) {
            atomicCAS(err, 0, code);
            *abort_flag = code;
            return false;
        }
    }
}

// Abort-path policy.  A warp whose lanes all execute collective or .aligned
// instructions (mma.sync, tcgen05.ld, __syncwarp, bar.sync) never leaves its
// loop on a failed wait: it ignores the result and runs its remaining,
// uniform iterations on whatever shared memory holds (every address stays in
// bounds), each later wait returning at once because the abort flag is set.
// The error word makes the host-visible results NaN.  Warps driven by one
// thread (TMA producer, MMA issuer) do leave early, after draining their own
// in-flight operations with the waits below.

// Bounded wait that ignores the abort flag.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, int* err) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kDrainTimeoutNs) {
            atomicCAS(err, 0, kErrTimeoutDrain);
            return;
        }
    }
}

// Waits until the last min(fills, ns) fills of a ring of ns stages have landed;
// fill i completes phase i / ns of barrier full[i % ns].
__device__ __forceinline__ void drain_ring(uint64_t* full, int ns, uint32_t fills, int* err) {
    const uint32_t first = fills > (uint32_t)ns ? fills - (uint32_t)ns : 0u;
    for (uint32_t i = first; i < fills; ++i) mbar_drain(&full[i % ns], (i / ns) & 1u, err);
}

// ----------------------------------------------------------------------- TMA

// 2D tiled load global -> shared, completion counted in bytes on `bar`.
// x is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Asynchronous global -> shared copy of 4 or 8 bytes; src_bytes = 0 writes zeros
// without reading `src` (which must still be a valid address).
template <int BYTES>
__device__ __forceinline__ void cp_async_zfill(void* dst, const void* src, int src_bytes) {
    static_assert(BYTES == 4 || BYTES == 8, "cp.async size");
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(smem_u32(dst)), "l"(src),
                 "n"(BYTES), "r"(src_bytes)
                 : "memory");
}

// Arrive on `bar` when all of this thread's prior cp.async copies have landed
// (the arrival is counted in the barrier's initial count).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tensor core).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// -------------------------------------------------------------------- tcgen05

// Whole warp: allocate `ncols` TMEM columns (power of two >= 32); the base
// address is written to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, fp16 x fp16 -> fp32, issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every previously issued tcgen05.mma of this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Warp-wide: 32 lanes x 32 consecutive 32-bit columns of TMEM.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits  0-13 start address >> 4, 16-29 leading byte offset >> 4,
//   32-45 stride byte offset >> 4, 46-47 version (1), 61-63 layout (2 = 128B swizzle).
// K-major operand (rows of 64 fp16 = 128 B, 8-row atoms of 1024 B): the
// stride offset is the distance between 8-row groups; the leading offset is
// not used.  MN-major operand: leading offset = distance between 64-element
// blocks along M/N, stride offset = distance between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A and
// B fp16 (bits 7-9, 10-12 = 0), A/B major (bit 15, 16: 0 = K-major, 1 = MN-major),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------- CTA pairs (clusters of 2)
// The pair's two CTAs run one tcgen05.mma.cta_group::2 stream: the even CTA
// (rank 0) issues the MMAs, which read A and B from both CTAs' shared memory
// at the same offsets and write each CTA's half of the accumulator rows into
// its own tensor memory.

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t nclusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Every thread of both CTAs: arrive and wait (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// Arrive without ordering (relaxed, cluster scope) on an mbarrier given by
// its shared::cluster address.  For a thread that has just acquired, at CTA
// scope, the writes it forwards: the arrival is performed after that acquire
// and needs no cluster-wide fence, which a release would wait for.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// Arrive (release at cluster scope) on an mbarrier given by its
// shared::cluster address, in this CTA or the peer.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// mbar_wait for a barrier that the peer CTA arrives on (acquire at cluster
// scope, so the peer's writes before its arrival are visible).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, int* err, int code) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort_flag || *reinterpret_cast<volatile int*>(err) != 0) return false;
        if (globaltimer() - t0 > kWaitTimeoutNs) {
            atomicCAS(err, 0, code);
            *abort_flag = 1;
            return false;
        }
    }
}

// Tensor memory of a CTA pair: one warp in each of the two CTAs executes
// these together; the same columns are allocated in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D (+)= A * B^T across the pair, issued by one thread of the even CTA: A is
// M = 256 rows (rows 0-127 from the even CTA's shared memory, 128-255 from
// the odd CTA's, same descriptor), B is N columns (the first N/2 from the
// even CTA, the rest from the odd one); each CTA's tensor memory receives its
// 128 accumulator rows.
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at `bar`'s offset in every CTA of `cta_mask` once
// every previously issued pair MMA of this thread is done.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// fp32 exp2 / reciprocal (PTX approximations).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace tc
}  // namespace qh

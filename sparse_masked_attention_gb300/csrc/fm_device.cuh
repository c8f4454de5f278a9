// fm_device.cuh -- sm_103a building blocks written as inline PTX: mbarriers,
// TMA bulk-tensor copies, tcgen05 tensor-core MMAs with TMEM accumulators,
// TMEM loads/stores, and the bounded-wait discipline every kernel follows.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "fm_internal.h"

namespace fm {

// ------------------------------------------------------------------ basics
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_fp16(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);  // .x (low half) = lo
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
    return *reinterpret_cast<uint32_t *>(&h);
}

// --------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive without release semantics: the thread's earlier memory operations are
// not ordered before it, so the arrive does not wait for them (for instance
// for global reductions nobody in the CTA reads).  Execution order still
// holds, and tcgen05 operations are ordered by their own fences.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t *bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok;
}

// Non-blocking probe: has the phase of `bar` with this parity completed?
__device__ __forceinline__ uint32_t mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok;
}

// Bounded wait for the phase of `bar` with the given parity to complete.
// Returns false when `timeout_ns` elapsed or another role of the CTA already
// gave up (*abort != 0); in the first case it records the failure in *abort
// and in the kernel's device error word.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns,
                                          volatile int *abort, unsigned *err_word) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > timeout_ns) {
            *abort = 1;
            atomicExch(err_word, ERR_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait for this CTA's own asynchronous work on the way out (MMAs or
// TMA loads it issued, which must land before it frees TMEM or exits).
// Unlike mbar_wait it ignores the abort flag: after another role gave up, the
// work already in flight still completes, and the CTA waits for it.  On a
// timeout it records ERR_TIMEOUT and gives up.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity,
                                                uint64_t timeout_ns, unsigned *err_word) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > timeout_ns) {
            atomicExch(err_word, ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Waits (mbar_wait_drain) for the last loads a producer issued into a ring of
// `stages` stages: loads [0, issued), except the one numbered `skipped` (-1:
// none).  Each stage's latest load is the only one that can still be in
// flight, and its completion phase is load / stages.
__device__ __forceinline__ void drain_ring(uint64_t *full, int stages, int issued, int skipped,
                                           uint64_t timeout_ns, unsigned *err_word) {
    for (int j = issued > stages ? issued - stages : 0; j < issued; ++j)
        if (j != skipped) mbar_wait_drain(&full[j % stages], (j / stages) & 1, timeout_ns, err_word);
}

// -------------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Tiled 4-D prefetch of one box into L2 (coordinates innermost first); a hint,
// with no completion to wait for.
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap *map, int c0, int c1, int c2,
                                                   int c3) {
    asm volatile(
        "cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Tiled 4-D load (coordinates innermost first) completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar))
        : "memory");
}

// Tiled TMA store shared -> global of one box at coordinates (c0..c3); the
// source must have been made visible to the async proxy (fence_proxy_async_smem)
// and stay untouched until bulk_wait_read() returns.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, const void *src, int c0,
                                             int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
        : "memory");
}

// Closes the thread's outstanding bulk stores into a group and waits until
// every group has finished reading shared memory.
__device__ __forceinline__ void bulk_commit_wait_read() {
    asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream still
// runs; pdl_wait() blocks the calling thread until the grids it depends on
// have completed and their writes are visible.  pdl_trigger() lets the next
// kernel in the stream launch once every CTA of this grid has called it (or
// exited).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Fire-and-forget fp32 add of four consecutive floats in global memory (no
// value returned, so the issuing thread never waits for it); 16-byte aligned.
__device__ __forceinline__ void red_add_v4(float4 *p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a),
                 "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Bulk reduction shared -> global: fp32 add of `bytes` (a multiple of 16; both
// addresses 16-byte aligned) into global memory by the TMA engine, in the
// issuing thread's current bulk group.
__device__ __forceinline__ void bulk_reduce_add_f32(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                     gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
// Closes this thread's outstanding bulk operations into a group.
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every bulk group of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Plain bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy (MMA reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B): start address, leading/stride byte
// offsets, descriptor version 1, layout type 2 (SWIZZLE_128B).  Tiles must
// start on 1024-byte boundaries.
//   K-major operand:  SBO = 1024 (8-row group stride); LBO unused.
//   MN-major operand: LBO = stride between 64-element MN blocks,
//                     SBO = 1024 (8-row K group stride).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation; A and B are
// both bf16 (fp16 = false) or both fp16 (fp16 = true).  a_mn / b_mn select
// MN-major operands.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, bool a_mn, bool b_mn,
                                                     bool fp16) {
    return (1u << 4)                                  // D: f32
           | ((fp16 ? 0u : 1u) << 7)                  // A: f16 (0) / bf16 (1)
           | ((fp16 ? 0u : 1u) << 10)                 // B: f16 (0) / bf16 (1)
           | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return idesc_f16kind(M, N, a_mn, b_mn, false);
}
__host__ __device__ constexpr uint32_t idesc_fp16(int M, int N, bool a_mn, bool b_mn) {
    return idesc_f16kind(M, N, a_mn, b_mn, true);
}

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
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

// D[tmem] (+)= A[smem] * B[smem]^T
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 consecutive TMEM columns of this thread's lane -> registers, and wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 64 consecutive TMEM columns of this thread's lane -> 64 floats, and wait.
__device__ __forceinline__ void tmem_ld64f(uint32_t taddr, float *x) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]), "=f"(x[4]), "=f"(x[5]), "=f"(x[6]), "=f"(x[7]), "=f"(x[8]), "=f"(x[9]), "=f"(x[10]), "=f"(x[11]), "=f"(x[12]), "=f"(x[13]), "=f"(x[14]), "=f"(x[15]), "=f"(x[16]), "=f"(x[17]), "=f"(x[18]), "=f"(x[19]), "=f"(x[20]), "=f"(x[21]), "=f"(x[22]), "=f"(x[23]), "=f"(x[24]), "=f"(x[25]), "=f"(x[26]), "=f"(x[27]), "=f"(x[28]), "=f"(x[29]), "=f"(x[30]), "=f"(x[31]), "=f"(x[32]), "=f"(x[33]), "=f"(x[34]), "=f"(x[35]), "=f"(x[36]), "=f"(x[37]), "=f"(x[38]), "=f"(x[39]), "=f"(x[40]), "=f"(x[41]), "=f"(x[42]), "=f"(x[43]), "=f"(x[44]), "=f"(x[45]), "=f"(x[46]), "=f"(x[47]), "=f"(x[48]), "=f"(x[49]), "=f"(x[50]), "=f"(x[51]), "=f"(x[52]), "=f"(x[53]), "=f"(x[54]), "=f"(x[55]), "=f"(x[56]), "=f"(x[57]), "=f"(x[58]), "=f"(x[59]), "=f"(x[60]), "=f"(x[61]), "=f"(x[62]), "=f"(x[63])
        : "r"(taddr)
        : "memory");
}

// 128 consecutive TMEM columns of this thread's lane -> 128 floats, and wait.
__device__ __forceinline__ void tmem_ld128f(uint32_t taddr, float *x) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]), "=f"(x[4]), "=f"(x[5]), "=f"(x[6]), "=f"(x[7]), "=f"(x[8]), "=f"(x[9]), "=f"(x[10]), "=f"(x[11]), "=f"(x[12]), "=f"(x[13]), "=f"(x[14]), "=f"(x[15]), "=f"(x[16]), "=f"(x[17]), "=f"(x[18]), "=f"(x[19]), "=f"(x[20]), "=f"(x[21]), "=f"(x[22]), "=f"(x[23]), "=f"(x[24]), "=f"(x[25]), "=f"(x[26]), "=f"(x[27]), "=f"(x[28]), "=f"(x[29]), "=f"(x[30]), "=f"(x[31]), "=f"(x[32]), "=f"(x[33]), "=f"(x[34]), "=f"(x[35]), "=f"(x[36]), "=f"(x[37]), "=f"(x[38]), "=f"(x[39]), "=f"(x[40]), "=f"(x[41]), "=f"(x[42]), "=f"(x[43]), "=f"(x[44]), "=f"(x[45]), "=f"(x[46]), "=f"(x[47]), "=f"(x[48]), "=f"(x[49]), "=f"(x[50]), "=f"(x[51]), "=f"(x[52]), "=f"(x[53]), "=f"(x[54]), "=f"(x[55]), "=f"(x[56]), "=f"(x[57]), "=f"(x[58]), "=f"(x[59]), "=f"(x[60]), "=f"(x[61]), "=f"(x[62]), "=f"(x[63]), "=f"(x[64]), "=f"(x[65]), "=f"(x[66]), "=f"(x[67]), "=f"(x[68]), "=f"(x[69]), "=f"(x[70]), "=f"(x[71]), "=f"(x[72]), "=f"(x[73]), "=f"(x[74]), "=f"(x[75]), "=f"(x[76]), "=f"(x[77]), "=f"(x[78]), "=f"(x[79]), "=f"(x[80]), "=f"(x[81]), "=f"(x[82]), "=f"(x[83]), "=f"(x[84]), "=f"(x[85]), "=f"(x[86]), "=f"(x[87]), "=f"(x[88]), "=f"(x[89]), "=f"(x[90]), "=f"(x[91]), "=f"(x[92]), "=f"(x[93]), "=f"(x[94]), "=f"(x[95]), "=f"(x[96]), "=f"(x[97]), "=f"(x[98]), "=f"(x[99]), "=f"(x[100]), "=f"(x[101]), "=f"(x[102]), "=f"(x[103]), "=f"(x[104]), "=f"(x[105]), "=f"(x[106]), "=f"(x[107]), "=f"(x[108]), "=f"(x[109]), "=f"(x[110]), "=f"(x[111]), "=f"(x[112]), "=f"(x[113]), "=f"(x[114]), "=f"(x[115]), "=f"(x[116]), "=f"(x[117]), "=f"(x[118]), "=f"(x[119]), "=f"(x[120]), "=f"(x[121]), "=f"(x[122]), "=f"(x[123]), "=f"(x[124]), "=f"(x[125]), "=f"(x[126]), "=f"(x[127])
        : "r"(taddr)
        : "memory");
}

// Registers -> 32 consecutive TMEM columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
        "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
        "%27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Named barrier over `nthreads` threads (multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------- mask helper
// Bits [lo, hi) of a 32-bit word, lo and hi clamped to [0, 32].
__device__ __forceinline__ uint32_t bit_range(int lo, int hi) {
    lo = max(lo, 0);
    hi = min(hi, 32);
    if (hi <= lo) return 0u;
    const uint32_t below_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
    return below_hi & ~((1u << lo) - 1u);
}

// Rows R .. R+31 of key column j: bit r set <=> row R + r is masked.  The
// masked rows of one column are the union of at most three intervals: [0, j)
// under the causal flag, [LTS, LTE) and [UTS, UTE).
__device__ __forceinline__ uint32_t column_row_bits(int R, int j, int4 c, int causal) {
    uint32_t m = causal ? bit_range(-R, j - R) : 0u;
    m |= bit_range(c.x - R, c.y - R);
    m |= bit_range(c.z - R, c.w - R);
    return m;
}

// 32x32 bit transpose across a warp: on entry lane l holds row l of a bit
// matrix (bit b = element [l][b]); on exit lane l holds column l (bit b =
// element [b][l]).  Five exchange steps of halving block size.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
    const uint32_t keep[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const int s = 16 >> k;
        const uint32_t m = keep[k];
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, s);
        x = (lane & s) ? ((x & ~m) | ((y & ~m) >> s)) : ((x & m) | ((y & m) << s));
    }
    return x;
}

}  // namespace fm

// ck_device.cuh -- inline-PTX building blocks for sm_103a kernels: mbarriers with
// bounded waits, TMA (cp.async.bulk.tensor) loads/stores, and the tcgen05 tensor-core
// family (TMEM alloc, MMA, commit, loads, fences).  Everything here is a thin wrapper
// around one PTX instruction; the kernels that use them live in gemm.cu / quantize.cu.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace ck {

// Bits of the device error word (see ck_device_error in the C ABI).
enum : uint32_t {
    kErrWaitProducer = 1u << 0,  // TMA producer gave up waiting for a free stage
    kErrWaitMma = 1u << 1,       // MMA issuer gave up waiting for data / a free accumulator
    kErrWaitEpilogue = 1u << 2,  // epilogue gave up waiting for an accumulator
    kErrWaitDrain = 1u << 3,     // teardown gave up waiting for in-flight copies / MMAs
    kErrWaitSelfTest = 1u << 4,  // the wait self-test timed out (expected by that test)
    kErrWaitGrid = 1u << 5,      // a grid-wide barrier of a preparation kernel timed out
    kErrTailCount = 1u << 6,     // a K-split tail unit's arrival counter kept changing (not expected)
};

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- packed fp32 (two values per instruction)
// sm_100-family GPUs execute two fp32 adds, multiplies or fmas as one instruction, each
// lane rounded exactly like the scalar one.  The rounding mode is spelled out (.rn):
// an add or multiply with an explicit rounding modifier is never contracted into an fma
// with a neighbouring instruction, so a multiply followed by an add stays two roundings,
// as the scalar __fmul_rn / __fadd_rn would.
__device__ __forceinline__ float2 f2_add_rn(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "add.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 f2_mul_rn(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
        "mul.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// a * b + c, one rounding per lane
__device__ __forceinline__ float2 f2_fma_rn(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\tmov.b64 pc, {%6, %7};\n\t"
        "fma.rn.f32x2 pd, pa, pb, pc;\n\tmov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may start while its
// predecessor on the stream is still running; griddep_wait() blocks until that
// predecessor has completed and its memory is visible.  Every kernel here calls it
// before touching global memory.  griddep_launch_dependents() lets the successor launch
// early (it still waits for this grid's completion in its own griddep_wait()).
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
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

// Wait for the phase with the given parity to complete, but never forever: after
// timeout_ns of wall time (read every 256 polls) the waiter raises the CTA-wide abort
// flag, records `code` in the device error word and returns false.  A waiter also
// returns false as soon as another role of the CTA has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* err, uint32_t code, uint64_t timeout_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 255u) == 0) {
            if (*abort_flag)
                return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                atomicOr(err, code);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- register re-balancing
// Executed by every thread of a warpgroup (4 consecutive warps): release registers to,
// or claim them from, the block's pool.  An increase waits until the pool can serve it,
// so the caller must make sure the launch provides the sum of the final counts.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec()
{
    static_assert(N % 8 == 0 && N >= 24 && N <= 256, "register count");
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc()
{
    static_assert(N % 8 == 0 && N >= 24 && N <= 256, "register count");
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 2-D tiled load of box {c0 (innermost), c1} into shared memory; completion is
// signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0,
                                            int32_t c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 eviction-priority hint (an createpolicy value).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0,
                                                 int32_t c1, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2-D tiled store of a shared-memory box to global memory (rows/columns outside the
// tensor are clipped by the hardware).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t c0, int32_t c1)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map),
                 "r"(c0), "r"(c1), "r"(smem_u32(src))
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Load for a CTA pair (tcgen05 cta_group::2): the box lands in this CTA's shared memory
// and the completed bytes are counted on `bar_cluster`, a shared::cluster address that
// may name the barrier in the pair's leader CTA.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int32_t c0,
                                                 int32_t c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}

// shared::cluster address of the variable at `p` (this CTA's shared memory) in the CTA
// of the cluster with rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// Arrive once on a barrier given by its shared::cluster address (possibly another CTA's),
// with the default (release, CTA-scope) semantics.  The cluster-scope release form
// fences at cluster scope on every call and cost about 0.5 us per arrival on GB300.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of all CTAs of the cluster (also a barrier for this CTA's threads).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy (TMA store).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}


// Arrive (once) on `bar` when every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// ---- the same family for a CTA pair (cta_group::2).  Every tcgen05 instruction of a
// kernel uses one cta_group, so a pair kernel uses only these.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols)
{
    // issued by one warp in each CTA of the pair; both receive the same address
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}


// Arrive once on the barrier at the offset of `bar` in every CTA named in cta_mask when
// the pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T over one 64-deep k-block, kind::f16 (bf16
// or f16 inputs, fp32 accumulator): four MMAs in one statement, the A and B descriptors
// advancing by 32 bytes (2 in the address field) per 16-element K step.  The first MMA
// adds to D only if `accumulate`; the other three always do.  PAIR: cta_group::2, issued
// by one thread of the pair's leader CTA; D's rows are in both CTAs' TMEM, A's rows are
// split over both CTAs' shared memory and so are B's (N).
template <bool PAIR>
__device__ __forceinline__ void mma_bf16_kblock(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate)
{
    if (PAIR)
        asm volatile(
            "{\n\t.reg .pred p, t;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "setp.eq.b32 t, %4, %4;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %5, %6, %3, t;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %7, %8, %3, t;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %9, %10, %3, t;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "l"(a_desc + 2), "l"(b_desc + 2),
            "l"(a_desc + 4), "l"(b_desc + 4), "l"(a_desc + 6), "l"(b_desc + 6)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p, t;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "setp.eq.b32 t, %4, %4;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %3, t;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %3, t;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %3, t;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "l"(a_desc + 2), "l"(b_desc + 2),
            "l"(a_desc + 4), "l"(b_desc + 4), "l"(a_desc + 6), "l"(b_desc + 6)
            : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA with
// 128-byte swizzling: rows of 128 bytes (64 bf16 along K), 8-row swizzle atoms of
// 1024 bytes stacked along M/N.  Fields: start address >> 4 (bits 0-13), leading
// byte offset >> 4 (bits 16-29; unused for swizzled K-major), stride byte offset >> 4
// (bits 32-45: distance between 8-row atoms), descriptor version 1 (bits 46-47),
// swizzle mode 2 = 128B (bits 61-63).
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A and B, fp32 D, both operands
// K-major: D format (bits 4-5) = 1 (f32), A format (bits 7-9) = 1 (bf16), B format
// (bits 10-12) = 1 (bf16), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
template <int M_, int N_>
__host__ __device__ constexpr uint32_t idesc_bf16_f32()
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N_ >> 3) << 17) | ((uint32_t)(M_ >> 4) << 24);
}

}  // namespace ck

// idx_common.cuh -- small inline-PTX helpers for sm_103a: mbarriers with
// bounded waits, TMA tile loads, tcgen05 (TMEM alloc, MMA, commit, load, copy)
// and shared-memory matrix descriptors.  Device code only.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#define IDX_DEVFN __device__ __forceinline__

namespace idx {

constexpr unsigned kDevBadPage = 1u;
constexpr unsigned kDevTimeout = 4u;

IDX_DEVFN uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

IDX_DEVFN uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ----------------------------------------------------------------- mbarrier

IDX_DEVFN void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

IDX_DEVFN void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

IDX_DEVFN void mbar_arrive(uint64_t *bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}

// n arrivals at once (release semantics, as n single arrivals).
IDX_DEVFN void mbar_arrive_cnt(uint64_t *bar, uint32_t n)
{
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
                 "r"(n)
                 : "memory");
}

IDX_DEVFN void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

IDX_DEVFN bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Like mbar_try_wait, but the thread may sleep in hardware for up to
// `hint_ns` nanoseconds waiting for the phase instead of returning at once,
// so a waiting warp takes no issue slots from the warps that work.
IDX_DEVFN bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
                 : "memory");
    return ok != 0;
}

// Slow path of mbar_wait, kept out of line so every call site stays small.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t *bar, uint32_t parity, volatile int *abort,
                                            unsigned int *status, uint64_t limit_ns)
{
    uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u))
            return true;
        if (*abort)
            return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort = 1;
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

// Wait for a phase after an abort, regardless of the abort flag: the async
// copies and MMAs a role has issued finish on their own, and the role waits
// (at most limit_ns) for them before its CTA frees its shared and tensor
// memory.
static __device__ __noinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity,
                                                    uint64_t limit_ns = 20000000ull)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, parity, 20000u))
        if (globaltimer_ns() - t0 > limit_ns)
            return false;
    return true;
}

IDX_DEVFN bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                         unsigned int *status, uint64_t limit_ns = 2000000000ull)
{
    if (mbar_try_wait(bar, parity))
        return true;
    return mbar_wait_slow(bar, parity, abort, status, limit_ns);
}

// Order-preserving 32-bit key of a float: a larger float gives a larger key;
// non-finite values give 0, below the key of every finite value.  The
// top-k's radix digits and the logits kernel's digit-1 histograms both use
// it.
IDX_DEVFN uint32_t order_key(float v)
{
    const uint32_t b = __float_as_uint(v);
    if (!isfinite(v))
        return 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The float of a nonzero order_key (the inverse of order_key on finite
// values).
IDX_DEVFN float key_float(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Float max into memory holding a float (prefilled, e.g. with -inf): values
// with the sign bit clear order like their bits as signed integers and win by
// atomicMax; values with it set order inversely to their bits as unsigned
// integers and win by atomicMin, which never replaces a value whose sign bit
// is clear (those are smaller as unsigned integers).
IDX_DEVFN void atomic_max_float(float *addr, float v)
{
    if (__float_as_int(v) >= 0)
        atomicMax(reinterpret_cast<int *>(addr), __float_as_int(v));
    else
        atomicMin(reinterpret_cast<unsigned int *>(addr), __float_as_uint(v));
}

// Prefetch of a global line into L2.  It returns no data, so it may run
// before a programmatic wait: a later load after the wait still reads the
// coherent value, from L2.
IDX_DEVFN void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

// -------------------------------------------------------------------- TMA

IDX_DEVFN void tma_prefetch_desc(const void *desc)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(desc)) : "memory");
}

IDX_DEVFN void tma_load_1d(void *dst, const void *desc, uint64_t *bar, int x)
{
    asm volatile("cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3}], [%2];" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(desc)), "r"(smem_u32(bar)), "r"(x)
                 : "memory");
}

IDX_DEVFN void tma_load_2d(void *dst, const void *desc, uint64_t *bar, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(desc)), "r"(smem_u32(bar)), "r"(x), "r"(y)
                 : "memory");
}

IDX_DEVFN void tma_load_3d(void *dst, const void *desc, uint64_t *bar, int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(desc)), "r"(smem_u32(bar)), "r"(x), "r"(y),
                 "r"(z)
                 : "memory");
}

// Plain bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
IDX_DEVFN void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy
// (tensor core / TMA reads of shared memory).
IDX_DEVFN void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

IDX_DEVFN void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

IDX_DEVFN void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

IDX_DEVFN void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

IDX_DEVFN void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

IDX_DEVFN void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4 (fp8 operands, fp32 accumulate).
IDX_DEVFN void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                          uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Block-scaled fp4 MMA: one e8m0 scale per 32 elements of A rows / B rows,
// read from tensor memory at sfa_tmem / sfb_tmem.
IDX_DEVFN void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X"
                 " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem),
                 "r"(sfb_tmem)
                 : "memory");
}

// Copy a 32-row x 128-bit block of shared memory (described by a no-swizzle
// matrix descriptor) into 4 columns of TMEM, replicated into all four
// 32-lane sub-partitions.
IDX_DEVFN void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t src_desc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc)
                 : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05 async ops of this
// thread have completed.
IDX_DEVFN void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns; lane i of the warp gets TMEM lane
// (taddr.lane + i).
IDX_DEVFN void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32"
                 " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
                 " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
                 " [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}

// Four consecutive 32-bit columns of the warp's 32 TMEM lanes.
IDX_DEVFN void tmem_ld_32x32b_x4(uint32_t taddr, uint32_t (&r)[4])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}

IDX_DEVFN void tmem_st_32x32b_x4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
                 "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

IDX_DEVFN void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

IDX_DEVFN void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------- shared memory descriptors

// Layout types of the sm_100 family matrix descriptor (bits 61..63).
constexpr uint64_t kLayoutNone = 0;
constexpr uint64_t kLayoutSw128 = 2;
constexpr uint64_t kLayoutSw64 = 4;

// Matrix descriptor: start address (>>4) in bits 0..13, leading byte offset
// (>>4) in 16..29, stride byte offset (>>4) in 32..45, descriptor version 1 in
// bits 46..47, layout type in 61..63.
IDX_DEVFN uint64_t make_smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                  uint64_t layout)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= layout << 61;
    return d;
}

// ------------------------------------------------------------- misc helpers

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start before the previous kernel on its stream has
// finished; pdl_wait() blocks until that kernel has completed and its memory
// operations are visible, so everything a kernel reads or writes that an
// earlier kernel may touch comes after it.  pdl_launch_dependents() lets the
// next such kernel start launching.  Both are no-ops without the attribute.
IDX_DEVFN void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

IDX_DEVFN void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Two fp32 fused multiply-adds in one packed instruction: (a * b + c) per
// lane, each rounded to nearest like fmaf.  The compiler builtin (rather
// than inline assembly) leaves the choice of the register pairs to the
// register allocator, which then needs no moves to build them.
IDX_DEVFN float2 fma2(float2 a, float2 b, float2 c)
{
    return __ffma2_rn(a, b, c);
}

IDX_DEVFN void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

IDX_DEVFN int lane_id()
{
    return threadIdx.x & 31;
}

IDX_DEVFN bool elect_one()
{
    uint32_t pred = 0;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "elect.sync _|p, 0xffffffff;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(pred));
    return pred != 0;
}

} // namespace idx

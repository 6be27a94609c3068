// Inline-PTX helpers for sm_103a: shared-memory barriers (mbarrier), the
// tensor memory accelerator (cp.async.bulk.tensor), the 5th-generation
// tensor core (tcgen05: TMEM alloc, mma, commit, ld), and the E4M3 convert.
// Every wait here is bounded: it gives up after a time limit, records the
// failure and returns false instead of spinning forever.
#pragma once

#include <cstdint>
#include <cuda.h>   // CUtensorMap

namespace jetfp8 {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive once on `bar` from one lane of the (converged) warp, chosen by
// elect.sync; the other lanes skip it by predicate, without a branch.
__device__ __forceinline__ void mbar_arrive_elected(uint64_t *bar)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// One potentially blocking test of the phase with parity `parity`: the thread
// is suspended (issuing nothing) until the phase completes or about
// `suspend_ns` nanoseconds pass, whichever is first.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity, uint32_t suspend_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `bar` with parity `parity` to complete.
// Waiting threads sleep inside try_wait (so they take no issue slots from the
// warps that share their SM sub-partition) and wake when the phase completes.
// Gives up (returns false) when *abort becomes non-zero (another role gave
// up) or after timeout_ns; on a timeout it sets *abort and ORs `code` into
// the device error word so the host can see what happened.
constexpr uint32_t SUSPEND_NS = 200000;   // re-check abort / timeout every 0.2 ms at most

// Non-blocking probe of the phase with parity `parity` (about 20 cycles when
// the phase has already completed, against about 55 for a suspending try_wait).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          uint32_t *err_word, uint32_t code, uint64_t timeout_ns)
{
    if (mbar_test_wait(bar, parity))
        return true;
    if (mbar_try_wait(bar, parity, SUSPEND_NS))
        return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity, SUSPEND_NS))
            return true;
        if (abort != nullptr && *abort)
            return false;
        if (globaltimer() - t0 > timeout_ns) {
            if (abort != nullptr)
                *abort = 1;
            if (err_word != nullptr)
                atomicOr(err_word, code);
            return false;
        }
    }
}

// ------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled bulk tensor copy global -> shared, completion counted in bytes on
// `bar`.  c0 is the innermost (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// L2 eviction priorities for the copies below (createpolicy): a line loaded
// with evict_first is the first candidate for replacement, evict_normal is
// the default order.
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// As tma_load_2d, with an L2 eviction priority for the lines it brings in.
__device__ __forceinline__ void tma_load_2d_hint(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                                 int32_t c0, int32_t c1, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// Both addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load_1d(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// ------------------------------------------------------------ cp.async
// 16-byte asynchronous global -> shared copy (L2 only), grouped by commit.
__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// 4-byte asynchronous copy; with src_bytes == 0 nothing is read and the
// destination is zero-filled.
__device__ __forceinline__ void cp_async_4(void *smem_dst, const void *gmem_src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src),
                 "r"(src_bytes)
                 : "memory");
}

// 16-byte variant with the same zero-fill rule (src_bytes 0 or 16).
__device__ __forceinline__ void cp_async_16z(void *smem_dst, const void *gmem_src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src),
                 "r"(src_bytes)
                 : "memory");
}

// Arrive on `bar` once all of this thread's earlier cp.async copies have
// completed; the arrival counts towards the barrier's expected count.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Wait until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 2-D tiled bulk tensor copy shared -> global (a store), tracked by the
// issuing thread's bulk async-group.  Out-of-bound parts of the box are not
// written.  c0 is the innermost coordinate in elements.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *smem_src, int32_t c0, int32_t c1)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
                 : "memory");
}

// As tma_store_2d, with an L2 eviction priority for the written lines.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap *map, const void *smem_src, int32_t c0, int32_t c1,
                                                  uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all bulk groups of this thread have completed.
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA) before a bulk copy reads them.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *smem_holder, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(smem_holder)),
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

// D[tmem] (+)= A[smem] * B[smem]^T, both FP8 operands K-major, fp32 accumulate.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Loads that are waited for inside the same asm statement, their 32-bit
// results handed out as packed pairs of adjacent columns (64-bit registers):
// the register allocator then places each pair in an aligned register pair
// once, instead of moving two loose registers into one before every packed
// multiply-add (measured on the per-column Wgrad promotion: +7 %).
//
// Lanes 0-15 (a, at taddr) and 16-31 (b, at taddr + 16 lanes) of a 32-lane
// quarter, 16x256b.x4 each (32 columns): thread t receives, for each 8-column
// block j, lanes (base + t/4) and (base + 8 + t/4) at columns 8j + 2(t%4) and
// 8j + 2(t%4) + 1 -- pair 2j from the first lane, pair 2j + 1 from the second.
// A thread thus holds four rows of the quarter (t/4, 8 + t/4, 16 + t/4 and
// 24 + t/4) at a quarter of its columns.
__device__ __forceinline__ void tmem_ld_16x256b_x4_pair_packed(uint32_t taddr, uint64_t (&a)[8], uint64_t (&b)[8])
{
    asm volatile(
        "{\n\t"
        ".reg .b32 t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15;\n\t"
        ".reg .b32 u0, u1, u2, u3, u4, u5, u6, u7, u8, u9, u10, u11, u12, u13, u14, u15;\n\t"
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {u0, u1, u2, u3, u4, u5, u6, u7, u8, u9, u10, u11, u12, u13, u14, u15}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "mov.b64 %8, {u0, u1};\n\t"
        "mov.b64 %9, {u2, u3};\n\t"
        "mov.b64 %10, {u4, u5};\n\t"
        "mov.b64 %11, {u6, u7};\n\t"
        "mov.b64 %12, {u8, u9};\n\t"
        "mov.b64 %13, {u10, u11};\n\t"
        "mov.b64 %14, {u12, u13};\n\t"
        "mov.b64 %15, {u14, u15};\n\t"
        "}"
        : "=l"(a[0]), "=l"(a[1]), "=l"(a[2]), "=l"(a[3]), "=l"(a[4]), "=l"(a[5]), "=l"(a[6]), "=l"(a[7]),
          "=l"(b[0]), "=l"(b[1]), "=l"(b[2]), "=l"(b[3]), "=l"(b[4]), "=l"(b[5]), "=l"(b[6]), "=l"(b[7])
        : "r"(taddr), "r"(taddr + (16u << 16))
        : "memory");
}

// 32 lanes x 64 columns (32x32b.x64), waited for: thread i of the warp
// receives TMEM lane (base lane + i), pair k = columns 2k, 2k+1.
__device__ __forceinline__ void tmem_ld_32x32b_x64_packed(uint32_t taddr, uint64_t (&r)[32])
{
    asm volatile(
        "{\n\t"
        ".reg .b32 t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15,"
        " t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31,"
        " t32, t33, t34, t35, t36, t37, t38, t39, t40, t41, t42, t43, t44, t45, t46, t47,"
        " t48, t49, t50, t51, t52, t53, t54, t55, t56, t57, t58, t59, t60, t61, t62, t63;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15,"
        " t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31,"
        " t32, t33, t34, t35, t36, t37, t38, t39, t40, t41, t42, t43, t44, t45, t46, t47,"
        " t48, t49, t50, t51, t52, t53, t54, t55, t56, t57, t58, t59, t60, t61, t62, t63}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "mov.b64 %8, {t16, t17};\n\t"
        "mov.b64 %9, {t18, t19};\n\t"
        "mov.b64 %10, {t20, t21};\n\t"
        "mov.b64 %11, {t22, t23};\n\t"
        "mov.b64 %12, {t24, t25};\n\t"
        "mov.b64 %13, {t26, t27};\n\t"
        "mov.b64 %14, {t28, t29};\n\t"
        "mov.b64 %15, {t30, t31};\n\t"
        "mov.b64 %16, {t32, t33};\n\t"
        "mov.b64 %17, {t34, t35};\n\t"
        "mov.b64 %18, {t36, t37};\n\t"
        "mov.b64 %19, {t38, t39};\n\t"
        "mov.b64 %20, {t40, t41};\n\t"
        "mov.b64 %21, {t42, t43};\n\t"
        "mov.b64 %22, {t44, t45};\n\t"
        "mov.b64 %23, {t46, t47};\n\t"
        "mov.b64 %24, {t48, t49};\n\t"
        "mov.b64 %25, {t50, t51};\n\t"
        "mov.b64 %26, {t52, t53};\n\t"
        "mov.b64 %27, {t54, t55};\n\t"
        "mov.b64 %28, {t56, t57};\n\t"
        "mov.b64 %29, {t58, t59};\n\t"
        "mov.b64 %30, {t60, t61};\n\t"
        "mov.b64 %31, {t62, t63};\n\t"
        "}"
        : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]), "=l"(r[7]),
          "=l"(r[8]), "=l"(r[9]), "=l"(r[10]), "=l"(r[11]), "=l"(r[12]), "=l"(r[13]), "=l"(r[14]), "=l"(r[15]),
          "=l"(r[16]), "=l"(r[17]), "=l"(r[18]), "=l"(r[19]), "=l"(r[20]), "=l"(r[21]), "=l"(r[22]), "=l"(r[23]),
          "=l"(r[24]), "=l"(r[25]), "=l"(r[26]), "=l"(r[27]), "=l"(r[28]), "=l"(r[29]), "=l"(r[30]), "=l"(r[31])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 32 columns (32x32b.x32), waited for: thread i of the warp
// receives TMEM lane (base lane + i), pair k = columns 2k, 2k+1.
__device__ __forceinline__ void tmem_ld_32x32b_x32_packed(uint32_t taddr, uint64_t (&r)[16])
{
    asm volatile(
        "{\n\t"
        ".reg .b32 t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15,"
        " t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15,"
        " t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "mov.b64 %8, {t16, t17};\n\t"
        "mov.b64 %9, {t18, t19};\n\t"
        "mov.b64 %10, {t20, t21};\n\t"
        "mov.b64 %11, {t22, t23};\n\t"
        "mov.b64 %12, {t24, t25};\n\t"
        "mov.b64 %13, {t26, t27};\n\t"
        "mov.b64 %14, {t28, t29};\n\t"
        "mov.b64 %15, {t30, t31};\n\t"
        "}"
        : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]), "=l"(r[7]),
          "=l"(r[8]), "=l"(r[9]), "=l"(r[10]), "=l"(r[11]), "=l"(r[12]), "=l"(r[13]), "=l"(r[14]), "=l"(r[15])
        : "r"(taddr)
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row swizzle atoms of 1024 bytes laid
// out back to back (stride-dimension byte offset 1024).  The tile base must be
// 1024-byte aligned; the start address may then be advanced by 32-byte steps
// along K inside the 128-byte row.
__device__ __forceinline__ uint64_t smem_desc_sw128_kmajor(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version (tcgen05)
    d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f8f6f4, A and B E4M3, D fp32, both K-major,
// dense, shape M x N (K = 32 per instruction).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n)
{
    return (1u << 4)                                  // D format: fp32
           | (0u << 7) | (0u << 10)                   // A, B format: E4M3
           | (0u << 15) | (0u << 16)                  // A, B K-major
           | (static_cast<uint32_t>(n >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(m >> 4) << 24);   // M / 16
}

// ------------------------------------------------------------ dependent launch
// Wait until the grids this one depends on (the previous kernel of the stream,
// when launched as a programmatic dependent) have completed and their memory
// is visible; returns at once otherwise.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next programmatic dependent kernel of the stream to be scheduled.
__device__ __forceinline__ void launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ registers
// Per-warpgroup register rebalancing; all four warps of a warpgroup execute it.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------ packed fp32
// Two fp32 lanes in one 64-bit register (lo in bits 0..31).  The f32x2 forms
// round each half exactly like their scalar counterparts.
__device__ __forceinline__ uint64_t pack_f32x2(uint32_t lo, uint32_t hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}

__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi)
{
    return pack_f32x2(__float_as_uint(lo), __float_as_uint(hi));
}

__device__ __forceinline__ float lo_f32(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi_f32(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

// acc = p * w + acc, lane-wise
__device__ __forceinline__ void fma_f32x2(uint64_t &acc, uint64_t p, uint64_t w)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(p), "l"(w));
}

// a * b + c, lane-wise (each lane one correctly rounded fused multiply-add)
__device__ __forceinline__ uint64_t fma2_f32x2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// ------------------------------------------------------------ convert
// Two fp32 -> two E4M3 codes, round to nearest even, saturating to +-448.
// Returns lo's code in bits 0..7 and hi's code in bits 8..15.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace ptx
}  // namespace jetfp8

// qmv_device.cuh -- sm_103a device helpers: inline PTX for bulk copies, mbarriers,
// cache-hinted loads, element conversions and the m16n8k16 tensor-core op.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace qmv {

constexpr uint32_t kErrWaitTimeout = 1u;   // error-word bit: an mbarrier wait gave up

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier + bulk copy

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make initialized mbarriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Like mbar_try_wait, but the thread may sleep up to `suspend_ns` inside the
// instruction until the phase completes (no busy polling).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t suspend_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

// %globaltimer in ns; the memory clobber keeps the read in place relative to the
// barriers and waits around it.
__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t)::"memory");
    return t;
}

// Bounds of every mbarrier wait. A poll is one try_wait that may suspend the thread
// (hint: 1 ms) until the phase completes; an incomplete phase returns it after a few
// microseconds. The wait gives up once kWaitLimitNs of %globaltimer time AND
// kMinWaitPolls polls have passed -- a context switched off the GPU polls nothing,
// so elapsed time alone does not end a wait -- and after kMaxWaitPolls polls in any
// case (a clock that stood still). A weight copy lands within microseconds, even on
// a contended memory system, so the bound is far above any valid wait.
constexpr uint64_t kWaitLimitNs = 500ull * 1000ull * 1000ull;   // 0.5 s
constexpr uint32_t kMinWaitPolls = 1024u;
constexpr uint32_t kMaxWaitPolls = 1u << 21;

// Bounded wait on phase `parity` of `bar`: true when it completed, false when the
// bound ran out. The first poll reads no clock (the common case: the copy landed).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; i < kMaxWaitPolls; ++i) {
        if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
        if (i >= kMinWaitPolls && globaltimer_ns() - t0 >= limit_ns) return false;
    }
    return false;
}

// ---------------------------------------------------------------- giving up without a fault

// A warp whose bounded wait gave up does not leave the CTA on its own: the other warps
// may be on their way to a CTA-wide barrier, which would then wait for a thread that
// has exited. Instead the warp's lane 0 flags the error word and the CTA's abort word
// (shared memory, zeroed before the CTA's first barrier), the warp skips the rest of
// its work up to the CTA's next barrier, and after that barrier every warp reads the
// abort word, lets its own copies in flight land (drain_ring) and returns: all threads
// leave together and no copy writes into the memory of a CTA that has exited.
__device__ __forceinline__ void note_wait_timeout(uint32_t *err_word, volatile uint32_t *cta_abort)
{
    atomicOr(err_word, kErrWaitTimeout);
    if (cta_abort) *cta_abort = 1u;
}

// Lane 0: wait (bounded) for the `outstanding` copies of a warp's ring of S slots that
// were issued and not yet consumed, the first at ring position `slot`, phase `parity`
// (a completed wait consumes its copy; the one whose wait gave up is still counted).
__device__ __forceinline__ void drain_ring(uint64_t *bars, int S, int slot, uint32_t parity, int outstanding)
{
    for (int i = 0; i < outstanding; ++i) {
        (void)mbar_wait_bounded(&bars[slot], parity);
        if (++slot == S) {
            slot = 0;
            parity ^= 1u;
        }
    }
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

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 2-D tensor copy global -> shared of one box at coordinates (x bytes, y rows),
// completion counted on `bar`. The tensor map lives in kernel parameter space.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x, int y, uint64_t *bar,
                                            uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses (and, after a
// warp or CTA barrier, those of the threads it synchronized with) before its later
// async-proxy (bulk copy / TMA) accesses: a slot the warp has just read is refilled
// by a copy only after the reads are performed.
__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned), bypassing L1;
// cp_async_wait_all waits for all of this thread's outstanding copies.
__device__ __forceinline__ void cp_async_16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---------------------------------------------------------------- programmatic dependent launch

// Wait until the grid this launch depends on has completed and its writes are
// visible (no-op when the launch carries no programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next programmatically dependent grid to begin launching.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// ---------------------------------------------------------------- global loads

// Streamed once: skip L1, mark evict-first in L2.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p, uint64_t policy)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void *p, uint64_t policy)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(policy));
    return v;
}

// Re-read by many CTAs (activations): read-only path, cached in L1.
__device__ __forceinline__ uint4 ld_shared_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// ---------------------------------------------------------------- element conversions

// Two E2M1 codes (one byte: low nibble -> low half) to two exact fp16 values.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte)
{
    uint32_t out;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(out) : "r"(byte));
    return out;
}

// Eight E2M1 codes (one 32-bit word; byte i -> h[i], low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4])
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) to two exact fp16 values.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes)
{
    uint32_t out;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(static_cast<uint16_t>(two_bytes)));
    return out;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Replicate the low or high fp16 half of a word into both halves.
__device__ __forceinline__ uint32_t dup_lo16(uint32_t v) { return __byte_perm(v, 0, 0x1010); }
__device__ __forceinline__ uint32_t dup_hi16(uint32_t v) { return __byte_perm(v, 0, 0x3232); }

__device__ __forceinline__ float f16_bits_to_float(uint32_t bits16)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// ---------------------------------------------------------------- integer dot

// c + sum_{i<4} a.u8[i] * b.s8[i]
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---------------------------------------------------------------- tensor core (m16n8k16, f16 in, f32 acc)

// D(16x8) += A(16x16, row) * B(16x8, col). Fragment ownership per lane
// (gid = lane / 4, t = lane % 4):
//   a0: A[gid][2t..2t+1]   a1: A[gid+8][2t..2t+1]   a2: A[gid][2t+8..2t+9]   a3: A[gid+8][2t+8..2t+9]
//   b0: B[2t..2t+1][gid]   b1: B[2t+8..2t+9][gid]
//   d0,d1: D[gid][2t..2t+1]   d2,d3: D[gid+8][2t..2t+1]
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace qmv

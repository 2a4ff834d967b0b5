// qsa_sm100.cuh -- inline-PTX wrappers for the Blackwell (sm_100 family)
// features the tensor-core kernels use: mbarriers, bulk async copies,
// tensor memory (TMEM) allocation, tcgen05.mma / commit / ld, and the
// shared-memory and instruction descriptors of tcgen05.mma.
//
// Every wait is bounded: a spin that runs out of iterations returns false so
// the caller can record an error and leave instead of hanging the GPU.
#pragma once

#include <stdint.h>

namespace qsa {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}"
                 ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Test for completion of phase `parity`; a thread whose phase is not yet
// complete is suspended for up to `suspend_ns` (woken earlier when the phase
// completes), so waiting warps do not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity, uint32_t suspend_ns)
{
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n"
                 " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
                 " selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
                 : "memory");
    return ok != 0;
}

// Non-blocking test for completion of phase `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n"
                 " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 " selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Default bound of a device-side wait: 2^32 SM clock cycles, about two
// seconds at 2 GHz.
constexpr long long kWaitCycles = 1ll << 32;

// Bounded wait on phase `parity`: false once about `max_cycles` SM clock
// cycles have passed without completion.  Long bounds suspend the waiting
// thread between tests; short ones (below 2^24 cycles, used to exercise the
// time-out path) poll without suspending, so the bound holds from the first
// test on.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          long long max_cycles = kWaitCycles)
{
    if (max_cycles >= (1ll << 24)) {
        if (mbar_try_wait(bar, parity, 20000u)) return true;
        const long long t0 = clock64();
        while (!mbar_try_wait(bar, parity, 200000u))
            if (clock64() - t0 > max_cycles) return false;
        return true;
    }
    const long long t0 = clock64();
    while (!mbar_test_wait(bar, parity))
        if (clock64() - t0 > max_cycles) return false;
    return true;
}

// ------------------------------------------------------------- bulk copies

// Non-tensor bulk copy global -> shared, completion counted in bytes on
// `bar`.  dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy
// (tensor core reads through descriptors).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------- TMEM

// Warp-collective; writes the TMEM base address to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor of tcgen05.mma.
//   [0,14)  start address >> 4      [16,30) leading byte offset >> 4
//   [32,46) stride byte offset >> 4 [46,48) version (1)
//   [49,52) base offset (0: swizzle atoms 1024-byte aligned)
//   [61,64) layout: 0 none, 2 SWIZZLE_128B, 4 SWIZZLE_64B, 6 SWIZZLE_32B
constexpr uint64_t kLayoutSw128 = 2;

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint64_t layout = kLayoutSw128)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= layout << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with fp32 accumulation.
//   [4,6) D format (1 = f32)  [7,10) A format  [10,13) B format (0 f16, 1 bf16)
//   bit 15 A major, bit 16 B major (0 K-major, 1 MN-major)
//   [17,23) N >> 3            [24,29) M >> 4
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_bf16, bool b_bf16,
                                                 bool a_mn_major, bool b_mn_major)
{
    return (1u << 4) | ((a_bf16 ? 1u : 0u) << 7) | ((b_bf16 ? 1u : 0u) << 10) |
           ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------- MMA

// D[tmem] (+)= A[smem] x B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
                 ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// D[tmem] (+)= A[tmem] x B[smem]^T: A (M rows in M lanes, K packed two
// 16-bit values per 32-bit column) read from tensor memory at `a_tmem`.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Arrive on `bar` once every previously issued tcgen05.mma of this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

// ------------------------------------------------------------- TMEM -> registers

// 32 lanes x 32-bit, 8 consecutive columns per thread (thread i <- lane base+i).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float *v)
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float *v)
{
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v)
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 lanes x 256 bits per repetition, loaded: thread t gets lanes base + t/4
// (v[4k], v[4k+1]) and base + 8 + t/4 (v[4k+2], v[4k+3]) at columns
// 8k + 2(t%4) and 8k + 2(t%4) + 1 of repetition k.
__device__ __forceinline__ void tmem_ld_16x256b_x2(uint32_t taddr, float *v)
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, float *v)
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// NK repetitions (NK even, >= 2) starting at taddr's column.
template <int NK>
__device__ __forceinline__ void tmem_ld_16x256b(uint32_t taddr, float *v)
{
    static_assert(NK >= 2 && NK % 2 == 0, "16x256b repetitions");
    if constexpr (NK >= 4) {
        tmem_ld_16x256b_x4(taddr, v);
        if constexpr (NK > 4) tmem_ld_16x256b<NK - 4>(taddr + 32, v + 16);
    } else {
        tmem_ld_16x256b_x2(taddr, v);
    }
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// After tmem_wait_ld(): mark registers filled by tcgen05.ld as written here,
// so no use of them can be scheduled before the wait.
template <int K>
__device__ __forceinline__ void regs_after_wait(float *v)
{
#pragma unroll
    for (int i = 0; i < K; ++i) asm volatile("" : "+f"(v[i]));
}

// registers -> 32 lanes x 32-bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                   "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                   "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                   "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                   "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                   "r"(__float_as_uint(v[15]))
                 : "memory");
}

// registers -> 32 lanes x 32-bit, 16 consecutive columns per thread (raw bits).
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t *v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                   "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
                   "r"(v[14]), "r"(v[15])
                 : "memory");
}

// registers -> 16 lanes x 256 bits, four repetitions (32 columns).  Thread
// t writes lanes base + t/4 (v[4k], v[4k+1]) and base + 8 + t/4 (v[4k+2],
// v[4k+3]) at columns 8k + 2(t%4) and 8k + 2(t%4) + 1, k = 0..3.
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t *v)
{
    asm volatile("tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                   "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
                   "r"(v[14]), "r"(v[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------- misc

// True in exactly one lane of a converged warp (the lane that issues a
// single-thread operation such as tcgen05.mma while the others follow).
__device__ __forceinline__ bool elect_one()
{
    uint32_t r;
    asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}" : "=r"(r));
    return r != 0;
}

// Named barrier `id` over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier `id` over `count` threads that also ORs a predicate over
// them: every participant gets true if any passed true.  Orders memory like
// bar.sync.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t count, bool v)
{
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %3, 0;\n"
                 " barrier.cta.red.or.pred q, %1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
                 : "=r"(r)
                 : "r"(id), "r"(count), "r"(v ? 1u : 0u)
                 : "memory");
    return r != 0;
}

// 16-byte asynchronous copy global -> shared (L2 only), no registers held.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// 4-byte asynchronous copy global -> shared (through L1).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 32-byte read-only global load that does not allocate in L1 (streamed data).
__device__ __forceinline__ void ldg256_stream(const void *ptr, uint32_t *r)
{
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "l"(ptr));
}

// The same load, predicated: when `on` is false nothing is read and the
// registers keep their values.
__device__ __forceinline__ void ldg256_stream_if(const void *ptr, uint32_t *r, bool on)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %9, 0;\n"
                 " @p ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n}"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7])
                 : "l"(ptr), "r"(on ? 1u : 0u));
}

__device__ __forceinline__ void prefetch_l2(const void *ptr)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// ------------------------------------------------------------- layouts

// Byte offset of element (row, k) of a K-major, 128-byte-swizzled operand
// tile of 16-bit values with `rows` rows and K split in 64-element blocks:
// block kb = k/64 at kb*rows*128; 8-row groups 1024 B apart; inside a group,
// row r%8 at 128*(r%8) with its 16-byte chunks XOR-permuted by r%8.
__host__ __device__ __forceinline__ uint32_t kmajor_sw128_off(uint32_t row, uint32_t k, uint32_t rows)
{
    return (k >> 6) * rows * 128u + (row >> 3) * 1024u + (row & 7u) * 128u +
           ((((k & 63u) >> 3) ^ (row & 7u)) << 4) + (k & 7u) * 2u;
}

// Byte offset of element (mn, k) of an MN-major, 128-byte-swizzled operand
// tile of 16-bit values: 64-element MN blocks `mn_block_stride` bytes apart
// (the descriptor's leading byte offset); 8-k groups 1024 B apart (its
// stride byte offset); inside a group, k%8 selects the 128-byte row and the
// 16-byte chunks are XOR-permuted by k%8.
__host__ __device__ __forceinline__ uint32_t mnmajor_sw128_off(uint32_t mn, uint32_t k,
                                                               uint32_t mn_block_stride)
{
    return (mn >> 6) * mn_block_stride + (k >> 3) * 1024u + (k & 7u) * 128u +
           ((((mn & 63u) >> 3) ^ (k & 7u)) << 4) + (mn & 7u) * 2u;
}

} // namespace sm100
} // namespace qsa

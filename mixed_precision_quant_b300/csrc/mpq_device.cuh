// mpq_device.cuh -- sm_103a device helpers: mbarriers with bounded waits, TMA,
// tcgen05 (TMEM alloc / MMA / commit / load), packed FP32x2 arithmetic, E4M3
// conversion and the exact group-scale arithmetic shared by the quantizer and the
// fused decode path.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace mpq {

// Status codes written to the device status word (same values as mpq_status).
constexpr int kStatusTimeout = 6;

// ---------------------------------------------------------------- addresses

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Shared control block of one CTA: an abort flag every role polls, the caller's
// device status word and the wait limit.
struct WaitCtl {
    volatile int *abort;   // shared memory
    int *status;           // global: [0] = code, [1] = where (role << 8 | barrier id)
    uint64_t timeout_ns;
};

// Bounded wait on a barrier phase.  Returns false when the CTA is aborting, either
// because another role gave up or because this wait ran past the limit, in which
// case it records MPQ timeout status and the waiter's tag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl &c, int tag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (*c.abort)
            return false;
        if (globaltimer_ns() - t0 > c.timeout_ns) {
            *c.abort = 1;
            if (c.status != nullptr && atomicCAS(c.status, 0, kStatusTimeout) == 0)
                atomicExch(c.status + 1, tag);
            return false;
        }
    }
}

// The same bounded wait for a waiter with nothing else to do for a long time (e.g. an
// epilogue warp during a tile's main loop): each try_wait asks the hardware to suspend the
// thread until the phase completes or about 20 us pass, so the waiting warp takes no issue
// slots from the warps sharing its scheduler.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_sleepy(uint32_t bar, uint32_t parity, const WaitCtl &c, int tag)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_suspend(bar, parity)) {
        if (*c.abort)
            return false;
        if (globaltimer_ns() - t0 > c.timeout_ns) {
            *c.abort = 1;
            if (c.status != nullptr && atomicCAS(c.status, 0, kStatusTimeout) == 0)
                atomicExch(c.status + 1, tag);
            return false;
        }
    }
    return true;
}

// ---------------------------------------------------------------- TMA / cp.async

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// Plain bulk copy global -> shared (both addresses 16-byte aligned, size a multiple of 16),
// completing on an mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// 2-D tiled bulk tensor load into shared memory, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int32_t x, int32_t y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// 4- or 16-byte asynchronous global->shared copy; bytes past src_bytes are zero-filled.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// The barrier receives one arrival once every cp.async issued so far by this thread lands.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3 -> FP32, one CTA.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes,
// 8-row core-matrix groups 1024 bytes apart.  The tile base must be 1024-byte aligned; a
// K offset inside the 128-byte swizzle row is added to the start address.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address, bits 0-13
    d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;                    // swizzle mode: 128-byte
    return d;
}

// Instruction descriptor, kind::f8f6f4: D = F32, A = B = E4M3, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n)
{
    return (1u << 4)                                   // D format: F32
           | (0u << 7) | (0u << 10)                    // A, B format: E4M3
           | (static_cast<uint32_t>(n >> 3) << 17)     // N >> 3
           | (static_cast<uint32_t>(m >> 4) << 24);    // M >> 4
}

// 32 TMEM lanes x 32 consecutive 32-bit columns; thread i of the warp receives lane
// (warp's lane quadrant base + i).
#define MPQ_TMEM_LD32(taddr, r)                                                                   \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "                                        \
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"                        \
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"       \
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),        \
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),      \
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),  \
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),  \
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),  \
                   "=r"(r[30]), "=r"(r[31])                                                       \
                 : "r"(taddr))

// Wait for this thread's TMEM loads; the registers are tied in so no use moves above it.
#define MPQ_TMEM_WAIT_LD32(r)                                                                     \
    asm volatile("tcgen05.wait::ld.sync.aligned;"                                                 \
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),        \
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),      \
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),  \
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),  \
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),  \
                   "+r"(r[30]), "+r"(r[31])                                                       \
                 :                                                                                \
                 : "memory")

// ---------------------------------------------------------------- clusters / CTA pairs

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared::cluster address of the variable at shared::cta address `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Every thread of every CTA of the cluster; release/acquire ordering of shared memory.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in a peer CTA), with
// release semantics at CTA scope only: it orders nothing in memory for the peer, so use it
// where the protected resource is already drained (e.g. TMEM reads completed with
// tcgen05.wait::ld).  A cluster-scope release would fence all of the thread's prior memory
// traffic on every arrival.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// ---------------------------------------------------------------- CTA pairs (2-SM MMA)
//
// With cta_group::2 the even CTA of a cluster pair issues MMAs that read A and B from both
// CTAs' shared memory (each holds M/2 rows of A and N/2 rows of B at the same offsets) and
// write each CTA's TMEM (its M/2 rows, all N columns).  TMEM allocation is collective: one
// warp of each CTA of the pair executes the same alloc / relinquish / dealloc.

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
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

// D[tmem] (+)= A * B^T over both CTAs of the pair (issued by one thread of the even CTA).
__device__ __forceinline__ void umma_e4m3_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at the same offset in every CTA of `mask` when all prior
// pair MMAs of this thread have completed.
__device__ __forceinline__ void umma_commit_pair_mc(uint32_t bar, uint16_t mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// TMA 2-D load into this CTA's shared memory whose completion is counted on an mbarrier
// that may live in the peer CTA (`bar_cluster` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *m, uint32_t bar_cluster, int32_t x,
                                                 int32_t y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// ---------------------------------------------------------------- microscaling MMA
//
// kind::mxf8f6f4 with block scaling: the tensor cores multiply each 32-element K block of
// A row m by 2^(SFA(m) - 127) and of B column n by 2^(SFB(n) - 127) (UE8M0 scale factors,
// read from TMEM) while accumulating in FP32.  Scale-factor layout in TMEM used here (one
// 32-bit word per scale, its four bytes equal, so every K block of a 128-K slice takes the
// same scale and the byte selectors of the instruction descriptor stay 0): the word of A
// row m sits in column base + m/32 of lane m % 32, and the word of B column n in column
// base + 4 + n/32 of lane n % 32, repeated in all four 32-lane quadrants of TMEM.

// Instruction descriptor, kind::mxf8f6f4 block-scaled: D = F32, A = B = E4M3 (K-major),
// UE8M0 scale factors (bit 23), scale-factor byte selectors (bits 4-5 for B, 29-30 for A) 0.
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int m, int n)
{
    return (static_cast<uint32_t>(n >> 3) << 17)    // N >> 3
           | (1u << 23)                             // scale-factor type UE8M0
           | (static_cast<uint32_t>(m >> 4) << 24); // M >> 4
}

// D[tmem] (+)= (A * 2^SFA) (B * 2^SFB)^T over both CTAs of the pair (one thread of the even CTA).
__device__ __forceinline__ void umma_mx_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Shared-memory descriptor of a 32-row x 16-byte matrix stored row after row (no swizzle:
// 8-row core matrices of 128 bytes, 128 bytes apart), the source of tcgen05.cp 32x128b.
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(128 >> 4) << 16;             // leading byte offset (one 16-byte column)
    d |= static_cast<uint64_t>(128 >> 4) << 32;             // stride byte offset: 8 rows x 16 bytes
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version for tcgen05
    return d;                                               // swizzle mode 0: none
}

// Copy a 32-row x 16-byte shared-memory matrix into TMEM columns taddr .. taddr + 3, row r
// into lane r of each of the four 32-lane quadrants (both CTAs of the pair, each from its own
// shared memory).  Issued by one thread; ordered with that thread's MMAs.
__device__ __forceinline__ void tmem_cp_32x128b_x4_pair(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Stores of registers into TMEM: 32 lanes (the warp's quadrant) x 4 or 8 consecutive columns.
__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t (&v)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// Wait until this thread's TMEM stores have completed.
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// UE8M0 code of a power-of-2 scale: the binary32 exponent field of a positive normal power
// of 2 (2^-126 .. 2^127), or 0 for 2^-127; anything else is not representable and sets `bad`
// (the code 127, scale 1, is returned in its place).
__device__ __forceinline__ uint32_t ue8m0_of(float s, bool &bad)
{
    const uint32_t b = __float_as_uint(s);
    const uint32_t e = (b >> 23) & 0xFFu;
    if ((b & 0x807FFFFFu) == 0 && e >= 1 && e <= 254)
        return e;
    if (b == 0x00400000u)
        return 0;
    bad = true;
    return 127;
}

// ---------------------------------------------------------------- TMA stores

// 2-D tiled store of a shared-memory box to global memory (clipped at the tensor bounds),
// tracked by the executing thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, uint32_t src, int32_t x, int32_t y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until no committed bulk store of this thread still reads shared memory.
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Wait until at most the N most recent committed bulk stores of this thread (N = 1 or 3)
// still read shared memory.
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read3() { asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); }

// Wait until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Order this thread's generic-proxy shared-memory writes before later async-proxy reads.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------- packed FP32x2

__device__ __forceinline__ unsigned long long pack2(float lo, float hi)
{
    return (static_cast<unsigned long long>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}

__device__ __forceinline__ float lo_of(unsigned long long v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi_of(unsigned long long v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

// d = a * b + c on two lanes at once, each rounded once (round to nearest even).
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c)
{
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ unsigned long long fmul2(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ---------------------------------------------------------------- E4M3 conversion

// Two binary32 values -> two E4M3 codes, round to nearest even, saturating to +-448.
// Byte 0 of the result holds `first`, byte 1 holds `second`.
__device__ __forceinline__ uint32_t e4m3x2(float first, float second)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
    return r;
}

// Four binary32 values -> four E4M3 codes in one word, byte k holding value k (the two
// 16-bit halves joined by one vector move instead of a shift and an or).
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
    return r;
}

__device__ __forceinline__ uint32_t bf16x2_lo(uint32_t w) { return w << 16; }
__device__ __forceinline__ uint32_t bf16x2_hi(uint32_t w) { return w & 0xFFFF0000u; }

// ---------------------------------------------------------------- group scales
//
// A group's scale maps its max-abs value onto the largest E4M3 value 448: s = amax / 448
// (one IEEE binary32 division), or with power-of-2 scales s = 2^e, e the smallest integer
// with amax <= 448 * 2^e.  An all-zero group gets s = 1.  Every element becomes the
// correctly rounded binary32 quotient x / s, then E4M3 round-to-nearest-even.

// 2^e as binary32 for -149 <= e <= 127 (exact, subnormal below -126).
__device__ __forceinline__ float exp2_int(int e)
{
    return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                     : __uint_as_float(1u << (e + 149));
}

// Smallest e with amax <= 448 * 2^e, for finite amax > 0.  With amax = f * 2^E, f in [1, 2):
// 448 * 2^e = 1.75 * 2^(e + 8), so e = E - 8 when f <= 1.75 and E - 7 otherwise.
__device__ __forceinline__ int pow2_exponent(float amax)
{
    const uint32_t b = __float_as_uint(amax);
    int E = static_cast<int>((b >> 23) & 0xFF);
    uint32_t f = b & 0x7FFFFFu;
    if (E == 0) { // subnormal: normalise the 23-bit fraction
        const int p = 31 - __clz(f);                 // top set bit, 0..22
        f = (f << (23 - p)) & 0x7FFFFFu;
        E = p - 149;
    } else {
        E -= 127;
    }
    return E - 8 + (f > 0x600000u ? 1 : 0);
}

struct GroupScale {
    float s;     // the stored scale
    float r;     // RN(1 / s) (mode 0), or the exact reciprocal 2^-e of a power-of-2 scale (mode 1)
    int mode;    // 0: product plus one correction step, 1: exact product, 2: IEEE division
};

// Scales below this use the IEEE division: the correction step needs an exact remainder
// (see e4m3_pair), which holds when ulp(s) * 2^-33 >= 2^-149, i.e. s >= 2^-93.
constexpr float kMinCorrectedScale = 0x1p-80f;

// Scale of a group from its max-abs value.
__device__ __forceinline__ GroupScale make_group_scale(float amax, bool pow2)
{
    GroupScale g;
    if (amax == 0.0f) {
        g.s = 1.0f; g.r = 1.0f; g.mode = 1;
        return g;
    }
    // Floor: a positive max-abs never yields a zero scale; 2^-149, the smallest positive
    // binary32, replaces a power of 2 below it or a quotient amax / 448 that rounds to 0.
    // BF16 groups never reach it (max-abs >= 2^-133); dequantized FP8 values can.
    if (pow2) {
        const int e = max(pow2_exponent(amax), -149);
        g.s = exp2_int(e);
        if (e >= -126) { g.r = exp2_int(-e); g.mode = 1; }
        else { g.r = 0.0f; g.mode = 2; }
        return g;
    }
    // amax / 448 correctly rounded.  From 2^-100 up, the correction step below (the same
    // as the elements' quotients', with the constant r = RN(1/448)) yields the IEEE
    // quotient -- checked exhaustively on the CPU for every binary32 in [2^-100, max]
    // against IEEE division; smaller max-abs values take the division itself.
    if (amax >= 0x1p-100f) {
        constexpr float r448 = 0x1.24924ap-9f;   // RN(1/448)
        const float q0 = __fmul_rn(amax, r448);
        g.s = __fmaf_rn(__fmaf_rn(-q0, 448.0f, amax), r448, q0);
    } else {
        g.s = __fdiv_rn(amax, 448.0f);
    }
    if (g.s < kMinCorrectedScale) {
        g.s = fmaxf(g.s, 0x1p-149f);
        g.r = 0.0f; g.mode = 2;
        return g;
    }
    g.r = __frcp_rn(g.s);
    g.mode = 0;
    return g;
}

// IEEE binary32 division, kept out of line: it only runs for groups whose scale lies below
// kMinCorrectedScale (max-abs value below about 2^-71).
static __device__ __noinline__ float exact_quotient(float x, float s) { return __fdiv_rn(x, s); }

// Correctly rounded binary32 quotients x / s of a pair, negated, for mode 0.
//
// Method: the correction step of Markstein's division (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1),
// 1990).  With r = RN(1/s) and q0 = RN(x r) -- within one ulp of x / s -- the remainder
// x - q0 s is a binary32 number, so one fused multiply-add computes it exactly, and
// RN(q0 + (x - q0 s) r) = RN(x / s).  The remainder is exact when it cannot fall below the
// binary32 subnormal grid: for |q0| >= 2^-11 that needs s >= 2^-93 (kMinCorrectedScale keeps
// a margin), and a quotient below 2^-11 gives the code 0 whatever its last bits.
//
// The steps run on -r: nq0 = x (-r) = -q0, e = nq0 s + x = x - q0 s, t = e (-r) + nq0 =
// -RN(x / s).  Negated this way, t also carries the sign of x when x is a signed zero
// (t = -0 for x = +0 and +0 for x = -0), so the E4M3 code of x / s is the code of t with
// its sign bit flipped -- rounding to nearest even and saturation are symmetric in sign.
__device__ __forceinline__ unsigned long long neg_quotient2(unsigned long long x, unsigned long long nr,
                                                            unsigned long long s)
{
    const unsigned long long nq0 = fmul2(x, nr);
    const unsigned long long e = ffma2(nq0, s, x);
    return ffma2(e, nr, nq0);
}

// E4M3 codes of the correctly rounded binary32 quotients x0 / s and x1 / s, each then
// rounded to nearest even E4M3 with saturation; byte 0 = x0.  For power-of-2 scales
// x * 2^-e is the quotient itself (mode 1).
__device__ __forceinline__ uint32_t e4m3_pair(float x0, float x1, const GroupScale &g)
{
    if (g.mode == 2)
        return e4m3x2(exact_quotient(x0, g.s), exact_quotient(x1, g.s));
    const unsigned long long x = pack2(x0, x1);
    if (g.mode == 1) {
        const unsigned long long p = fmul2(x, pack2(g.r, g.r));
        return e4m3x2(lo_of(p), hi_of(p));
    }
    const unsigned long long t = neg_quotient2(x, pack2(-g.r, -g.r), pack2(g.s, g.s));
    return e4m3x2(lo_of(t), hi_of(t)) ^ 0x8080u;
}

// Single-value form (code in the low byte).
__device__ __forceinline__ uint32_t e4m3_one(float x, const GroupScale &g)
{
    return e4m3_pair(x, 0.0f, g) & 0xFFu;
}

} // namespace mpq

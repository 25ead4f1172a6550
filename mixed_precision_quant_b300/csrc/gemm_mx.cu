// gemm_mx.cu -- block-scaled FP8 GEMM for power-of-2 scales on the tensor cores'
// microscaling path (tcgen05.mma kind::mxf8f6f4.block_scale, UE8M0 scale factors).
//
// What it computes: the same sum as fp8_gemm_blockscaled (page 4, first paragraph: each
// 128-element slice of K carries its own scales, and the sum is kept in FP32),
//
//   C[m, n] = sum_kb ( sum_{k in slice kb} a[m,k] b[n,k] ) * sA[kb][m] * sB(n, kb),
//
// for scales that are integral powers of 2 (page 4, second paragraph), which the tensor
// cores of this GPU generation can apply themselves (page 3, first paragraph: microscaling
// formats with small quantization groups).  Each 128-K slice's scales are written as UE8M0
// scale factors of its four 32-K blocks, and the MMAs accumulate the scaled products of the
// whole K in FP32 in TMEM: the promotion of every slice into FP32, which the software path
// does with CUDA-core FMAs, happens inside the MMA.  A power-of-2 scale is exact in binary32,
// so the product a * b * 2^(ea + eb) is the term the software path scales in FP32.
//
// Design (B300, persistent, 2-CTA clusters computing 256 x 256 tiles with cta_group::2 MMAs,
// 16 warps per CTA):
//   warps 0-3   scale-factor writers: a slot of scale words covers up to four consecutive
//               slices of a tile, byte q of each word holding slice q's UE8M0 scale; warp w
//               takes every fourth slot-group, reads the group's row scales of A (this CTA's
//               rows) and 256 column scales of B and writes them into a shared-memory ring
//               in the layout tcgen05.cp takes (three 32-row x 16-byte matrices: row scales,
//               columns 0-127, 128-255);
//   warp 4      TMA producer: E4M3 slices into a 6-stage shared-memory ring;
//   warp 5      MMA issuer (even CTA): once per four slices three tcgen05.cp of a slot into
//               TMEM (in order with its MMAs, one group ahead); per slice four MMAs (K = 32
//               each) whose descriptor selects the slice's byte of the scale words, into one
//               256-column FP32 accumulator; one commit per slice (frees the operand stage),
//               one per group of four (frees the scale slot) and one per tile segment
//               (accumulator complete);
//   warps 8-15  epilogue: read the accumulator (32 lanes x 128 columns per warp) into
//               registers, release it to the MMA issuer (the next segment's MMAs start), then
//               write BF16 or FP32 through swizzled staging buffers and TMA stores.
// Work order: whole tiles (data-parallel), or stream-K when the last wave of tiles would be
// short -- the tile's later unit computes its last slices first and hands the FP32 partial
// over; the earlier one adds it before the store (sched_device.cuh).
// Every wait is bounded; a scale that is not a power of 2 in the UE8M0 range records
// MPQ_ERR_SCALE in the status word.
#include "mpq_internal.h"
#include "mpq_device.cuh"
#include "quant_device.cuh"
#include "sched_device.cuh"

namespace mpq {
namespace {

constexpr int BK = 128;
constexpr int BN = 256;
constexpr int STAGES = 6;
constexpr int WRITERS = 4;                      // scale-factor writer warps
constexpr int kThreads = 512;
constexpr uint32_t A_BYTES = 128 * BK;          // this CTA's 128 rows of A per slice
constexpr uint32_t B_BYTES = 128 * BK;          // this CTA's half of the tile's 256 B rows
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 512;             // accumulator 0..255, scale slots from 256
constexpr uint32_t SF_COL0 = 256;               // slot j: SFA at 256 + 16 j (4 columns), SFB at +4 (8)
constexpr uint32_t SF_SLOT_BYTES = 3 * 512;     // shared-memory scale words per slot: SFA, SFB 0-127, SFB 128-255
// Scale slots, each holding four slices' scales.  As many as writer warps: warp w fills slot w
// only, so a warp waiting for its slot's previous group is never two phases of the slot's
// barriers away from it (the parity waits stay unambiguous).
constexpr int SF_SLOTS = WRITERS;
constexpr uint32_t STAGE_OUT = 2048;            // output staging: one 2 KB buffer per epilogue warp
constexpr int ROWB = STAGE_OUT / 32;            // bytes per staged row piece (64-byte swizzle)
constexpr int PCS = ROWB / 16;                  // 16-byte pieces per row piece
constexpr int OUT_BUFS = 1;
constexpr int kStatusScale = 9;

constexpr int BAR_FULL = 0;
constexpr int BAR_DONE = BAR_FULL + STAGES;
constexpr int BAR_SFREADY = BAR_DONE + STAGES;
constexpr int BAR_SFDONE = BAR_SFREADY + SF_SLOTS;
constexpr int BAR_ACCFULL = BAR_SFDONE + SF_SLOTS;
constexpr int BAR_ACCEMPTY = BAR_ACCFULL + 1;
constexpr int BAR_DRAIN = BAR_ACCEMPTY + 1;
constexpr int NBARS = BAR_DRAIN + 1;

constexpr size_t kSmem = 1024 + STAGES * STAGE_BYTES + 8 * OUT_BUFS * STAGE_OUT + SF_SLOTS * SF_SLOT_BYTES +
                         NBARS * sizeof(uint64_t) + 32;

// Register split after the roles diverge: 8 x 32 x 88 + 8 x 32 x 168 = 65536 = 512 x 128.
constexpr int kRegsLow = 88, kRegsHigh = 168;

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > timeout_ns)
            return false;
    return true;
}

// Scales of B columns n0 + lane + 32 j (j = 0..7) for slice kb; columns past N take 1.
// With block scales, columns j < 4 lie in block n0 / 128 and j >= 4 in the next one.
template <int SCALE_B>
__device__ __forceinline__ void b_scales(const GemmArgs &p, int64_t n0, int lane, int kb, float (&fb)[8])
{
    if (SCALE_B == kScaleRowKN) {
        const float *row = p.sB + static_cast<int64_t>(kb) * p.ldsb + n0 + lane;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            fb[j] = n0 + lane + 32 * j < p.N ? row[32 * j] : 1.0f;
        return;
    }
    const int64_t nb = n0 / 128;
    float b0, b1;
    if (SCALE_B == kScaleBlockKN) {
        const float *row = p.sB + static_cast<int64_t>(kb) * p.ldsb + nb;
        b0 = row[0];
        b1 = n0 + 128 < p.N ? row[1] : 1.0f;
    } else {
        b0 = p.sB[nb * p.ldsb + kb];
        b1 = n0 + 128 < p.N ? p.sB[(nb + 1) * p.ldsb + kb] : 1.0f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
        fb[j] = j < 4 ? b0 : b1;
}

template <int SCALE_B, bool OUT_F32, bool SK>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *smA = base;
    uint8_t *smB = smA + STAGES * A_BYTES;
    uint8_t *smO = smB + STAGES * B_BYTES;
    uint8_t *smSF = smO + 8 * OUT_BUFS * STAGE_OUT;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smSF + SF_SLOTS * SF_SLOT_BYTES);
    uint32_t *misc = reinterpret_cast<uint32_t *>(bars + NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };
    const uint32_t rank = cluster_ctarank();
    const int unit = static_cast<int>(blockIdx.x >> 1);
    const int nunits = static_cast<int>(gridDim.x >> 1);
    const int64_t M = p.M, N = p.N;
    const int KB = static_cast<int>(p.K / BK);
    const int MT = static_cast<int>((M + 255) / 256);
    const int NT = static_cast<int>((N + BN - 1) / BN);
    const int T = MT * NT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(BAR_FULL + s), 1);
            mbar_init(bar(BAR_DONE + s), 1);
        }
        for (int j = 0; j < SF_SLOTS; ++j) {
            mbar_init(bar(BAR_SFREADY + j), 2);   // the writer warp of each CTA of the pair
            mbar_init(bar(BAR_SFDONE + j), 1);    // the MMAs that read the slot completed
        }
        mbar_init(bar(BAR_ACCFULL), 1);
        mbar_init(bar(BAR_ACCEMPTY), 16);        // 8 epilogue warps in each CTA
        mbar_init(bar(BAR_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
    }
    if (warp == 5) {
        tmem_alloc_pair(smem_u32(misc), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // the peer's barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = misc[0];
    WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

    if (warp < 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow) : "memory");
        if (warp < 4) {
            // ---------------------------------------------------------- scale-factor writers
            // The scale words of up to four consecutive slices of a tile share one slot: byte q
            // of each word is the UE8M0 scale of the group's slice q (its MMAs select byte q), so
            // the MMA issuer copies a slot into TMEM once per four slices.  Lane r writes row r of
            // the slot's three 32-row x 16-byte matrices: the words of A rows r + 32 j, B
            // columns r + 32 j and B columns 128 + r + 32 j (j = 0..3).  Warp w takes the groups
            // gc = w, w + 4, ... of the unit's sequence (slot gc % SF_SLOTS): four warps keep
            // their groups' scale loads in flight; warp w fills slot w.
            bool bad = false;
            uint32_t gc = 0;
            Sched sc = sched_init(SK, unit, nunits, T, KB);
            int t, kb0, kb1;
            while (sched_next(sc, t, kb0, kb1)) {
                const int mt = p.n_fastest ? t / NT : t % MT, nt = p.n_fastest ? t % NT : t / MT;
                const int64_t row0 = static_cast<int64_t>(mt) * 256 + rank * 128;
                const int64_t n0 = static_cast<int64_t>(nt) * BN;
                // the segment's groups of four slices (a stream-K segment may start or end
                // inside one; the group's other slices are written too and not used)
                for (int gi = kb0 >> 2; gi <= (kb1 - 1) >> 2; ++gi, ++gc) {
                    if ((gc & 3u) != static_cast<uint32_t>(warp))
                        continue;
                    const uint32_t slot = gc % SF_SLOTS, ph = (gc / SF_SLOTS) & 1;
                    float fa[4][4], fb[4][8];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {   // slices past the tile's K take scale 1 (unused)
                        const int kb = gi * 4 + q;
                        if (kb < KB) {
                            const float *sa_row = p.sA + static_cast<int64_t>(kb) * p.ldsa;
#pragma unroll
                            for (int j = 0; j < 4; ++j) {   // rows past M: scale 1 (zero products)
                                const int64_t r = row0 + lane + 32 * j;
                                fa[q][j] = r < M ? sa_row[r] : 1.0f;
                            }
                            b_scales<SCALE_B>(p, n0, lane, kb, fb[q]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                fa[q][j] = 1.0f;
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                fb[q][j] = 1.0f;
                        }
                    }
                    uint32_t w[12];
#pragma unroll
                    for (int j = 0; j < 12; ++j)
                        w[j] = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            w[j] |= ue8m0_of(fa[q][j], bad) << (8 * q);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            w[4 + j] |= ue8m0_of(fb[q][j], bad) << (8 * q);
                    }
                    // the slot is free once the MMAs that read its previous group completed
                    if (!mbar_wait(bar(BAR_SFDONE + slot), ph ^ 1, ctl, 0x0600 | slot))
                        goto writer_done;
                    const uint32_t dst = smem_u32(smSF + slot * SF_SLOT_BYTES) + lane * 16;
#pragma unroll
                    for (int q = 0; q < 3; ++q)
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst + q * 512),
                                     "r"(w[4 * q]), "r"(w[4 * q + 1]), "r"(w[4 * q + 2]), "r"(w[4 * q + 3])
                                     : "memory");
                    fence_proxy_async_smem();   // visible to tcgen05.cp
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_remote(mapa_shared(bar(BAR_SFREADY + slot), 0));
                }
            }
        writer_done:
            if (__any_sync(0xffffffffu, bad) && lane == 0 && p.status != nullptr &&
                atomicCAS(p.status, 0, kStatusScale) == 0)
                atomicExch(p.status + 1, 0x0680 | static_cast<int>(rank) << 2 | warp);
        } else if (warp == 4 && lane == 0) {
            // ---------------------------------------------------------- TMA producer
            uint32_t it = 0;
            Sched sc = sched_init(SK, unit, nunits, T, KB);
            int t, kb0, kb1;
            while (sched_next(sc, t, kb0, kb1)) {
                const int mt = p.n_fastest ? t / NT : t % MT, nt = p.n_fastest ? t % NT : t / MT;
                const int row0 = mt * 256 + static_cast<int>(rank) * 128;
                const int brow0 = nt * BN + static_cast<int>(rank) * 128;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (!mbar_wait(bar(BAR_DONE + s), ph ^ 1, ctl, 0x0700 | s))
                        goto producer_done;
                    const uint32_t full = mapa_shared(bar(BAR_FULL + s), 0);
                    if (rank == 0)
                        mbar_arrive_expect_tx(bar(BAR_FULL + s), 2 * STAGE_BYTES);
                    tma_load_2d_pair(smem_u32(smA + s * A_BYTES), &tmA, full, kb * BK, row0);
                    tma_load_2d_pair(smem_u32(smB + s * B_BYTES), &tmB, full, kb * BK, brow0);
                }
            }
        producer_done:
            if (rank == 0) {
                for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; ++j)
                    wait_drain(bar(BAR_FULL + j % STAGES), (j / STAGES) & 1, p.timeout_ns);
            } else if (*abort_flag) {
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
        } else if (warp == 5 && lane == 0 && rank == 0) {
            // ---------------------------------------------------------- MMA issuer
            const uint32_t idesc = idesc_mx_e4m3(256, BN);
            const uint64_t da0 = sdesc_kmajor_sw128(smem_u32(smA));
            const uint64_t db0 = sdesc_kmajor_sw128(smem_u32(smB));
            // a group's scale slot is copied into TMEM during the previous group, so the MMAs
            // never wait for a copy issued just ahead of them; the groups of all the unit's
            // segments, counted as the writers count them
            uint32_t ngroups = 0;
            {
                Sched sc = sched_init(SK, unit, nunits, T, KB);
                int t, kb0, kb1;
                while (sched_next(sc, t, kb0, kb1))
                    ngroups += static_cast<uint32_t>(((kb1 - 1) >> 2) - (kb0 >> 2) + 1);
            }
            auto copy_slot = [&](uint32_t g) -> bool {
                const uint32_t sl = g % SF_SLOTS;
                if (!mbar_wait(bar(BAR_SFREADY + sl), (g / SF_SLOTS) & 1, ctl, 0x0810 | sl))
                    return false;
                tc_fence_after();
                const uint32_t sfs = smem_u32(smSF + sl * SF_SLOT_BYTES);
                const uint32_t dst = tmem_base + SF_COL0 + 16 * sl;
#pragma unroll
                for (int c = 0; c < 3; ++c)   // SFA, SFB 0-127, SFB 128-255: columns +0, +4, +8
                    tmem_cp_32x128b_x4_pair(dst + 4 * c, sdesc_rows16(sfs + 512 * c));
                return true;
            };
            uint32_t s = 0, ph = 0, tc = 0, gc = 0;
            if (ngroups > 0 && !copy_slot(0))
                goto mma_done;
            for (Sched sc = sched_init(SK, unit, nunits, T, KB); ;) {
                int t, kb0, kb1;
                if (!sched_next(sc, t, kb0, kb1))
                    break;
                if (!mbar_wait(bar(BAR_ACCEMPTY), (tc & 1) ^ 1, ctl, 0x0800))
                    goto mma_done;
                tc_fence_after();
                for (int kb = kb0; kb < kb1; ++kb) {
                    const uint32_t q = static_cast<uint32_t>(kb & 3);
                    const uint32_t slot = gc % SF_SLOTS;
                    const uint32_t sfa = tmem_base + SF_COL0 + 16 * slot;
                    // a group's first slice (of the segment): copy the next group's slot
                    if ((q == 0 || kb == kb0) && gc + 1 < ngroups && !copy_slot(gc + 1))
                        goto mma_done;
                    if (!mbar_wait(bar(BAR_FULL + s), ph, ctl, 0x0820 | s))
                        goto mma_done;
                    tc_fence_after();
                    const uint64_t da = da0 + s * (A_BYTES >> 4), db = db0 + s * (B_BYTES >> 4);
                    // byte q of every scale word: this slice's scales (B: bits 4-5, A: bits 29-30)
                    const uint32_t id = idesc | (q << 4) | (q << 29);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        umma_mx_pair(tmem_base, da + 2 * k, db + 2 * k, id, sfa, sfa + 4, (kb > kb0 || k > 0) ? 1u : 0u);
                    umma_commit_pair_mc(bar(BAR_DONE + s), 0x3);
                    if (q == 3 || kb == kb1 - 1) {   // the group's last slice: its slot may be refilled
                        umma_commit_pair_mc(bar(BAR_SFDONE + slot), 0x3);
                        ++gc;
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                umma_commit_pair_mc(bar(BAR_ACCFULL), 0x3);
                ++tc;
            }
        mma_done:
            umma_commit_pair_mc(bar(BAR_DRAIN), 0x1);
            wait_drain(bar(BAR_DRAIN), 0, p.timeout_ns);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh) : "memory");
        // -------------------------------------------------------------- epilogue
        const int ew = warp - 8, quad = warp & 3, half = ew >> 2;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + half * 128;
        uint32_t tc = 0;
        Sched sc = sched_init(SK, unit, nunits, T, KB);
        int t, kb0, kb1;
        for (; sched_next(sc, t, kb0, kb1); ++tc) {
            const int mt = p.n_fastest ? t / NT : t % MT, nt = p.n_fastest ? t % NT : t / MT;
            if (!mbar_wait_sleepy(bar(BAR_ACCFULL), tc & 1, ctl, 0x0900))
                break;
            tc_fence_after();
            uint32_t v[128];
            {
                uint32_t *v0 = v, *v1 = v + 32, *v2 = v + 64, *v3 = v + 96;
                MPQ_TMEM_LD32(taddr, reinterpret_cast<uint32_t(&)[32]>(*v0));
                MPQ_TMEM_LD32(taddr + 32, reinterpret_cast<uint32_t(&)[32]>(*v1));
                MPQ_TMEM_LD32(taddr + 64, reinterpret_cast<uint32_t(&)[32]>(*v2));
                MPQ_TMEM_LD32(taddr + 96, reinterpret_cast<uint32_t(&)[32]>(*v3));
                MPQ_TMEM_WAIT_LD32(reinterpret_cast<uint32_t(&)[32]>(*v0));
                MPQ_TMEM_WAIT_LD32(reinterpret_cast<uint32_t(&)[32]>(*v1));
                MPQ_TMEM_WAIT_LD32(reinterpret_cast<uint32_t(&)[32]>(*v2));
                MPQ_TMEM_WAIT_LD32(reinterpret_cast<uint32_t(&)[32]>(*v3));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_remote(mapa_shared(bar(BAR_ACCEMPTY), 0));   // the next tile's MMAs may start
            if (SK && kb0 > 0) {
                // Tail of a tile the previous unit finishes: hand this warp's partial over
                // (layout [unit][rank][warp][i][lane], coalesced) and announce it.
                float4 *dst = p.sk_part + ((static_cast<int64_t>(unit) * 2 + rank) * 8 + ew) * 1024 + lane;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    dst[32 * i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                              __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p.sk_flags + (unit * 2 + rank) * 8 + ew),
                                 "r"(p.sk_epoch)
                                 : "memory");
                continue;
            }
            if (SK && kb1 < KB) {
                // Head of a tile: add the tail the next unit computed (final sum: head + tail).
                const int slot = ((unit + 1) * 2 + static_cast<int>(rank)) * 8 + ew;
                if (!wait_count(p.sk_flags + slot, p.sk_epoch, ctl, 0x0980))
                    break;
                const float4 *src = p.sk_part + static_cast<int64_t>(slot) * 1024 + lane;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float4 w4 = __ldcg(src + 32 * i);
                    v[4 * i] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * i]), w4.x));
                    v[4 * i + 1] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * i + 1]), w4.y));
                    v[4 * i + 2] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * i + 2]), w4.z));
                    v[4 * i + 3] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * i + 3]), w4.w));
                }
            }
            // rows [row0 + 32 quad, +32), columns [n0 + 128 half, +128) of this CTA's half tile
            const int wrow0 = mt * 256 + static_cast<int>(rank) * 128 + quad * 32;
            const int ncol0 = nt * BN + half * 128;
            if (ncol0 < N && wrow0 < M) {
                const uint32_t stg0 = smem_u32(smO + ew * OUT_BUFS * STAGE_OUT);
                constexpr int COLS = ROWB / (OUT_F32 ? 4 : 2);  // columns per row piece
#pragma unroll
                for (int ch = 0; ch < 128 / COLS; ++ch) {
                    const uint32_t stg = stg0 + (ch % OUT_BUFS) * STAGE_OUT;
                    if (lane == 0)
                        bulk_wait_read0();   // the buffer's previous piece has left shared memory
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < PCS; ++j) {   // 16-byte pieces of the row
                        uint4 w;
                        if (OUT_F32) {
                            const int a0 = ch * COLS + j * 4;
                            w = make_uint4(v[a0], v[a0 + 1], v[a0 + 2], v[a0 + 3]);
                        } else {
                            const int a0 = ch * COLS + j * 8;
                            uint32_t h[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[a0 + 2 * k]),
                                                                                __uint_as_float(v[a0 + 2 * k + 1]));
                                h[k] = *reinterpret_cast<const uint32_t *>(&b2);
                            }
                            w = make_uint4(h[0], h[1], h[2], h[3]);
                        }
                        // 64-byte swizzle: 16-byte piece j of row r at piece j ^ ((r >> 1) & 3)
                        const uint32_t off = lane * ROWB + ((j ^ ((lane >> 1) & 3)) << 4);
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(stg + off), "r"(w.x), "r"(w.y),
                                     "r"(w.z), "r"(w.w)
                                     : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, stg, ncol0 + ch * COLS, wrow0);
                        bulk_commit();
                    }
                }
            }
        }
        if (lane == 0)
            bulk_wait0();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // the pair's MMAs, copies and remote arrivals are all complete
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <int SB, bool F32, bool SK>
cudaError_t launch_mx_one(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC, const GemmArgs &a,
                          int grid, cudaStream_t st)
{
    auto kern = gemm_mx_kernel<SB, F32, SK>;
    static std::atomic<uint64_t> configured{0};
    if (cudaError_t e = ensure_max_dyn_smem(kern, kSmem, configured); e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, a);
}

} // namespace

cudaError_t launch_gemm_mx(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC, const GemmArgs &a,
                           int scale_b, bool out_fp32, int num_sms, cudaStream_t st)
{
    const int64_t tiles = ((a.M + 255) / 256) * ((a.N + BN - 1) / BN);
    if (tiles <= 0)
        return cudaSuccess;
    const int64_t pairs = tiles < num_sms / 2 ? tiles : num_sms / 2;
    const int grid = static_cast<int>(2 * (pairs < 1 ? 1 : pairs));
    const bool sk = a.sk_part != nullptr;
    if (sk && tiles < grid / 2)   // stream-K: at least one tile per pair
        return cudaErrorInvalidValue;
#define MPQ_MX(SB, F32)                                                                   \
    if (scale_b == SB && out_fp32 == F32)                                                 \
        return sk ? launch_mx_one<SB, F32, true>(tmA, tmB, tmC, a, grid, st)              \
                  : launch_mx_one<SB, F32, false>(tmA, tmB, tmC, a, grid, st);
    MPQ_MX(kScaleBlockNK, false)
    MPQ_MX(kScaleBlockNK, true)
    MPQ_MX(kScaleBlockKN, false)
    MPQ_MX(kScaleBlockKN, true)
    MPQ_MX(kScaleRowKN, false)
    MPQ_MX(kScaleRowKN, true)
#undef MPQ_MX
    return cudaErrorInvalidValue;
}

} // namespace mpq

// gemm.cu -- block-scaled FP8 GEMM with 128-element FP32 promotion on tcgen05.
//
// What it computes (source pages: page 1 second paragraph -- the GEMMs take FP8
// tensors and produce BF16 or FP32, the dequantization is folded into the
// increased-precision accumulation; page 4 first paragraph -- partial results are
// promoted every 128 elements of K and accumulated in full FP32; page 4 second
// paragraph -- Fprop, Dgrad and Wgrad all run in FP8):
//
//   C[m, n] = sum_kb ( sum_{k in slice kb} a[m,k] b[n,k] ) * sA[kb][m] * sB(n, kb)
//
// with A [M, K] and B [N, K] E4M3 codes (both K-major) and sB one of
//   block [N/128][K/128] (Fprop), block [K/128][N/128] (Dgrad through the
//   transposed weight), per-row [K/128][N] (Wgrad, 128x1 token tiles).
//
// Design (B300, persistent, one CTA per SM, 128 x 256 output tile per CTA).  Two modes:
//   pair   (default) a cluster of two CTAs on two SMs computes one 256 x 256 tile with
//          2-SM MMAs (cta_group::2, M = 256): each CTA stages its own 128 rows of A and
//          one half (128 rows) of B per 128-K slice -- 32 KB per stage instead of 48 KB,
//          so each SM's shared memory carries a third less operand traffic, the limit of
//          the single-SM form -- and the even CTA issues the MMAs, which write the
//          accumulators of both SMs.  Both CTAs' loads complete on the even CTA's stage
//          barrier; its commits release the stage and hand over the partial in both CTAs;
//          both CTAs' promotion warps release the partial buffer to it.
//   single one CTA loads all of its A and B slices itself (M = 128 MMAs).
// Roles in each CTA:
//   warp 0      TMA producer: E4M3 slices into a shared-memory ring (128-byte swizzle);
//   warp 1      MMA issuer: four MMAs (K = 32 each) per 128-K slice into one of two TMEM
//               partial buffers (2 x 256 columns), committed per slice;
//   warp 2      scale loader: cp.async of the slice's A and B scales into a 4-slot ring;
//   warps 4-11  promotion: tcgen05.ld the slice partial (two loads in flight), multiply
//               by its two scales and accumulate into FP32 registers with scalar FMAs;
//               promotion of slice k overlaps the MMAs of slice k+1.  The finished tile is
//               written as BF16 or FP32 through swizzled staging buffers (two of 4 KB per
//               warp in pair mode, so the stores drain while the next tile starts) and TMA
//               bulk-tensor stores (32 rows x 128 bytes per store; 64 bytes single-SM).
// Work order: whole tiles (data-parallel), or for dense GEMMs stream-K when the last wave of
// tiles would be short (sched_device.cuh): a tile's later unit computes its last slices
// first and hands the FP32 partial over, the earlier one adds it before the store.
// Every wait is bounded; on expiry the CTA records a timeout in the status word, drains
// its copies and MMAs, frees TMEM and exits.
#include "mpq_internal.h"
#include "mpq_device.cuh"
#include "quant_device.cuh"
#include "swiglu_device.cuh"
#include "sched_device.cuh"

namespace mpq {
namespace {

constexpr int BK = 128;              // K per promotion slice
constexpr int BN = 256;              // output columns per tile
constexpr int SSLOTS = 4;            // scale ring depth (slices)
constexpr int kThreads = 384;
// The SwiGLU epilogue runs in four more warps (12-15), which take each tile's BF16 gate / up
// values from a 64 KB hand-over area in shared memory while the promotion warps go on with
// the next tile.  Pair tiles use their output staging area for it; single-SM tiles make room
// with a 3-stage operand ring.
constexpr uint32_t kHandoffBytes = 128 * 128 * 4;   // 128 rows x 128 columns, gate | up words
__host__ __device__ constexpr int threads_of(bool swiglu) { return swiglu ? 512 : kThreads; }
constexpr uint32_t A_BYTES = 128 * BK;     // 128 rows of A per CTA per slice
constexpr uint32_t TMEM_COLS = 512;        // two 256-column partial buffers
constexpr int kMaxGroups = 1024;

template <bool PAIR>
struct Cfg {
    static constexpr int STAGES = 4;
    // Output staging per promotion warp: in pair mode two 4 KB buffers of 32 rows x 128 bytes
    // (8 KB, a whole warp tile in BF16), so a tile's TMA stores drain during the next tile's
    // main loop instead of holding the warp back -- the output is written in a burst, when
    // the write path is saturated.  128-byte rows halve the number of row pieces the TMA
    // unit writes against 64-byte rows (Dgrad 8192 x 7168 x 2048 +4%, Fprop +1%).  The
    // single-SM form has no room for more than one 2 KB buffer of 64-byte rows.
    static constexpr int OUT_BUFS = PAIR ? 2 : 1;
    static constexpr uint32_t STAGE_OUT = PAIR ? 4096 : 2048;
    static constexpr int ROWB = STAGE_OUT / 32;              // bytes per staged row piece
    static constexpr int B_ROWS = PAIR ? 128 : 256;          // B rows staged by one CTA per slice
    static constexpr uint32_t B_BYTES = B_ROWS * BK;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TILE_M = PAIR ? 256 : 128;          // rows per tile (both CTAs of a pair)
    static constexpr int BAR_FULL = 0;
    // DONE[s]: the MMAs of the slice held in stage s have completed -- the stage may be
    // refilled and the slice's partial may be promoted.  One commit per slice serves both
    // (every tcgen05.commit costs the tensor pipe a bubble).
    static constexpr int BAR_DONE = BAR_FULL + STAGES;
    static constexpr int BAR_TEMPTY = BAR_DONE + STAGES;
    static constexpr int BAR_SFULL = BAR_TEMPTY + 2;
    static constexpr int BAR_SEMPTY = BAR_SFULL + SSLOTS;
    static constexpr int BAR_DRAIN = BAR_SEMPTY + SSLOTS;
    // SwiGLU hand-over: a tile's gate / up values written (eight promotion warps) and
    // consumed (four epilogue warps)
    static constexpr int BAR_XFULL = BAR_DRAIN + 1;
    static constexpr int BAR_XEMPTY = BAR_XFULL + 1;
    static constexpr int NBARS = BAR_XEMPTY + 1;
    // Register split after the roles diverge (4 x 32 x low + 8 x 32 x high = 168 x 384, the
    // launch's allocation): for dense GEMMs with block B scales the producer, MMA and scale
    // warps run faster with 72 registers (Fprop +4%, Dgrad +1%); the per-column-scale
    // promotion (Wgrad) and the grouped kernels (3-5% slower at 72) keep 56 / 224.
    __host__ __device__ static constexpr bool wide_low(int scale_b, bool grouped)
    {
        return scale_b != kScaleRowKN && !grouped;
    }
    // SwiGLU (512 threads, 128 registers each at launch): eight warps at 40 (producer, MMA,
    // scale loader, idle, the four epilogue warps) and the eight promotion warps at 216.
    __host__ __device__ static constexpr int regs_low(int scale_b, bool grouped, bool swiglu = false)
    {
        return swiglu ? 40 : wide_low(scale_b, grouped) ? 72 : 56;
    }
    __host__ __device__ static constexpr int regs_high(int scale_b, bool grouped)
    {
        return wide_low(scale_b, grouped) ? 216 : 224;
    }
};

constexpr size_t kSmemGroups = (kMaxGroups + 1) * 2 * sizeof(int) + 16;

// Operand stages and output-staging bytes of an instantiation: the SwiGLU hand-over needs a
// 64 KB area, which pair tiles have as their staging area and single-SM tiles get by giving
// up one of their four 48 KB stages.
template <bool PAIR>
__host__ __device__ constexpr int stages_of(bool swiglu) { return swiglu && !PAIR ? 3 : Cfg<PAIR>::STAGES; }
template <bool PAIR>
__host__ __device__ constexpr size_t staging_of(bool swiglu)
{
    return swiglu ? kHandoffBytes : static_cast<size_t>(8 * Cfg<PAIR>::OUT_BUFS * Cfg<PAIR>::STAGE_OUT);
}
template <bool PAIR>
size_t smem_bytes(bool grouped, bool swiglu)
{
    using C = Cfg<PAIR>;
    const size_t main = stages_of<PAIR>(swiglu) * C::STAGE_BYTES + staging_of<PAIR>(swiglu) +
                        SSLOTS * (128 + BN) * sizeof(float) + C::NBARS * sizeof(uint64_t) + 16;
    return 1024 + main + (grouped ? kSmemGroups : 0);
}

// Sizes are validated on the host to stay below 2^31 rows / columns.
struct Tile {
    int g;            // expert (grouped), else 0
    int row0;         // first row of A / C handled by this CTA
    int row_end;      // one past the last valid row for this CTA
    int brow0;        // first row of B loaded by this CTA (TMA view [G*N, K] when grouped)
    int n0;           // first output column of the tile
    int64_t sb_base;  // offset of this expert's B scales
};

// Wait without abort polling (used to drain in-flight copies / MMAs before exit).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > timeout_ns)
            return false;
    return true;
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// acc[32 c + i] += partial column 32 c + i times its scales, for one 32-column chunk.
// Scalar FMAs on purpose: the packed FP32x2 form runs on one of the SM's two FP32 pipes
// only (four cycles per warp instruction), scalar FMAs use both -- half the pipe time for
// the same rounding (each lane of the packed form is an independent fma.rn).
template <int SCALE_B>
__device__ __forceinline__ void promote_chunk(float (&acc)[128], const uint32_t (&v)[32], int c, float sc, float sa,
                                              const float *sbcol)
{
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float x = __uint_as_float(v[i]);
        if (SCALE_B == kScaleRowKN)
            acc[c * 32 + i] = __fmaf_rn(x, __fmul_rn(sa, sbcol[c * 32 + i]), acc[c * 32 + i]);
        else
            acc[c * 32 + i] = __fmaf_rn(x, sc, acc[c * 32 + i]);
    }
}

template <int SCALE_B, bool OUT_F32, bool GROUPED, bool PAIR, bool FUSE, bool SK, bool SWIGLU>
__global__ void __launch_bounds__(threads_of(SWIGLU), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const GemmArgs p, const FuseArgs f)
{
    using C = Cfg<PAIR>;
    constexpr int STAGES = stages_of<PAIR>(SWIGLU);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *smA = base;
    uint8_t *smB = smA + STAGES * A_BYTES;
    uint8_t *smO = smB + STAGES * C::B_BYTES;                    // output staging (SwiGLU: the hand-over area)
    float *ssa = reinterpret_cast<float *>(smO + staging_of<PAIR>(SWIGLU));
    float *ssb = ssa + SSLOTS * 128;
    uint64_t *bars = reinterpret_cast<uint64_t *>(ssb + SSLOTS * BN);
    uint32_t *misc = reinterpret_cast<uint32_t *>(bars + C::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    int *goff = reinterpret_cast<int *>(misc + 4);                // grouped: clamped offsets [G+1]
    int *gtile = goff + kMaxGroups + 1;                           // grouped: first tile of expert

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };

    const uint32_t rank = PAIR ? cluster_ctarank() : 0;   // position in the CTA pair
    const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int nunits = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    const int64_t M = p.M, N = p.N;
    const int KB = static_cast<int>(p.K / BK);
    // SwiGLU tiles: 128 output columns, the matching gate and up weight rows side by side
    const int NT = SWIGLU ? p.sw_width / 128 : static_cast<int>((N + BN - 1) / BN);
    constexpr int TILE_N = SWIGLU ? 128 : BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(C::BAR_FULL + s), 1);
            mbar_init(bar(C::BAR_DONE + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::BAR_TEMPTY + b), PAIR ? 16 : 8);   // promotion warps of the pair
        }
        for (int j = 0; j < SSLOTS; ++j) {
            mbar_init(bar(C::BAR_SFULL + j), 32);
            mbar_init(bar(C::BAR_SEMPTY + j), 8);
        }
        mbar_init(bar(C::BAR_DRAIN), 1);
        mbar_init(bar(C::BAR_XFULL), 8);          // this CTA's promotion warps
        mbar_init(bar(C::BAR_XEMPTY), 4);         // the epilogue warps
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(misc), TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(misc), TMEM_COLS);
            tmem_relinquish();
        }
    }
    // m-tiles of an expert with `rows` token rows; experts outside [min_rows, max_rows) belong
    // to another launch and get none
    auto expert_mtiles = [&](int rows) -> int {
        return rows >= p.min_rows && rows < p.max_rows ? (rows + C::TILE_M - 1) / C::TILE_M : 0;
    };
    if (GROUPED && warp == 2) {
        // Expert schedule: offsets clamped into [0, M] and made monotone (running max),
        // then the exclusive prefix sum of (pair) m-tiles per expert, times the n-tiles.
        const int G = p.G;
        for (int g = lane; g <= G; g += 32) {
            const int64_t o = p.offsets[g];
            goff[g] = static_cast<int>(o < 0 ? 0 : (o > M ? M : o));
        }
        __syncwarp();
        const int per = (G + 1 + 31) / 32;
        const int c0 = lane * per, c1 = c0 + per < G + 1 ? c0 + per : G + 1;
        int mx = 0;
        for (int g = c0; g < c1; ++g)
            mx = goff[g] > mx ? goff[g] : mx;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, mx, o);
            if (lane >= o && v > mx)
                mx = v;
        }
        int run = __shfl_up_sync(0xffffffffu, mx, 1);
        if (lane == 0)
            run = 0;
        for (int g = c0; g < c1; ++g) {
            run = goff[g] > run ? goff[g] : run;
            goff[g] = run;
        }
        __syncwarp();
        const int perg = (G + 31) / 32;
        const int e0 = lane * perg, e1 = e0 + perg < G ? e0 + perg : G;
        int cnt = 0;
        for (int g = e0; g < e1; ++g)
            cnt += expert_mtiles(goff[g + 1] - goff[g]);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += v;
        }
        int ex = incl - cnt;
        for (int g = e0; g < e1; ++g) {
            gtile[g] = ex * NT;
            ex += expert_mtiles(goff[g + 1] - goff[g]);
        }
        if (lane == 31)
            gtile[G] = incl * NT;
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR)
        cluster_sync_all();  // the peer's barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = misc[0];

    // fused activation quantization: phase 1, all warps, before the roles split (SwiGLU: 512
    // threads at 128 registers each, one group a lane per batch)
    if (FUSE)
        quantize_rows_phase<SWIGLU ? 1 : 2>(goff, p.G, M, KB, p.K, f);

    const int MT = static_cast<int>((M + C::TILE_M - 1) / C::TILE_M);
    const int T = GROUPED ? gtile[p.G] : MT * NT;

    auto tile_of = [&](int t) -> Tile {
        Tile ti;
        int row0, rend;
        if (!GROUPED) {
            const int mt = p.n_fastest ? t / NT : t % MT, nt = p.n_fastest ? t % NT : t / MT;
            row0 = mt * C::TILE_M;
            rend = static_cast<int>(M);
            ti.g = 0;
            ti.n0 = nt * TILE_N;
            ti.brow0 = ti.n0;
            ti.sb_base = 0;
        } else {
            int lo = 0, hi = p.G - 1;  // last expert whose first tile is <= t
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (gtile[mid] <= t) lo = mid; else hi = mid - 1;
            }
            const int g = lo;
            ti.g = g;
            const int local = t - gtile[g];
            const int rows_g = goff[g + 1] - goff[g];
            const int mtg = expert_mtiles(rows_g);
            // an expert with more token rows than weight rows reads each row strip once and
            // keeps its (smaller) weight in L2; otherwise each weight strip is read once
            const bool nf = rows_g > N;
            const int nt = nf ? local % NT : local / mtg, mt = nf ? local / NT : local - nt * mtg;
            row0 = goff[g] + mt * C::TILE_M;
            rend = goff[g + 1];
            ti.n0 = nt * TILE_N;
            ti.brow0 = g * static_cast<int>(N) + ti.n0;
            ti.sb_base = static_cast<int64_t>(g) * p.sb_group_stride;
        }
        ti.row0 = row0 + static_cast<int>(rank) * 128;
        ti.row_end = ti.row0 + 128 < rend ? ti.row0 + 128 : rend;
        // pair mode: the odd CTA stages the second half of the tile's B rows (the up weights
        // of a SwiGLU tile)
        ti.brow0 += static_cast<int>(rank) * (SWIGLU ? p.sw_width : C::B_ROWS);
        return ti;
    };

    WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

    if (warp < 4 || warp >= 12) {   // warps 12-15: the SwiGLU hand-over's epilogue
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::regs_low(SCALE_B, GROUPED, SWIGLU)) : "memory");
        if (warp == 0 && lane == 0) {
            // ---------------------------------------------------------- TMA producer
            uint32_t it = 0;
            Sched sc = sched_init(SK, unit, nunits, T, KB);
            int t, kb0, kb1;
            while (sched_next(sc, t, kb0, kb1)) {
                const Tile ti = tile_of(t);
                if (FUSE) {   // the expert's token codes are complete (phase 1 of all CTAs)
                    if (!wait_count(f.ready + ti.g, goff[ti.g + 1] - goff[ti.g], ctl, 0x0180))
                        goto producer_done;
                    fence_proxy_async_global();
                }
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (!mbar_wait(bar(C::BAR_DONE + s), ph ^ 1, ctl, 0x0100 | s))
                        goto producer_done;
                    if (PAIR) {
                        // both CTAs' slices complete on the even CTA's stage barrier
                        const uint32_t full = mapa_shared(bar(C::BAR_FULL + s), 0);
                        if (rank == 0)
                            mbar_arrive_expect_tx(bar(C::BAR_FULL + s), 2 * C::STAGE_BYTES);
                        tma_load_2d_pair(smem_u32(smA + s * A_BYTES), &tmA, full, kb * BK, ti.row0);
                        tma_load_2d_pair(smem_u32(smB + s * C::B_BYTES), &tmB, full, kb * BK, ti.brow0);
                    } else {
                        mbar_arrive_expect_tx(bar(C::BAR_FULL + s), C::STAGE_BYTES);
                        tma_load_2d(smem_u32(smA + s * A_BYTES), &tmA, bar(C::BAR_FULL + s), kb * BK, ti.row0);
                        if (SWIGLU) {   // gate rows, then up rows (boxes of 128 rows)
                            tma_load_2d(smem_u32(smB + s * C::B_BYTES), &tmB, bar(C::BAR_FULL + s), kb * BK, ti.brow0);
                            tma_load_2d(smem_u32(smB + s * C::B_BYTES + 128 * BK), &tmB, bar(C::BAR_FULL + s), kb * BK,
                                        ti.brow0 + p.sw_width);
                        } else {
                            tma_load_2d(smem_u32(smB + s * C::B_BYTES), &tmB, bar(C::BAR_FULL + s), kb * BK, ti.brow0);
                        }
                    }
                }
            }
        producer_done:
            if (!PAIR || rank == 0) {
                for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; ++j)
                    mbar_wait_drain(bar(C::BAR_FULL + j % STAGES), (j / STAGES) & 1, p.timeout_ns);
            } else if (*abort_flag) {
                // The odd CTA's copies complete on the even CTA's barriers; after a timeout
                // give copies still in flight a grace period before this CTA exits.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 200000ull) {
                }
            }
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // ---------------------------------------------------------- MMA issuer
            // One lane issues for the CTA (or the pair) and shares its SMSP with two busy
            // promotion warps, so its loop is kept short: descriptors are a precomputed base
            // plus a small offset (the 14-bit start-address field cannot carry: shared
            // addresses stay below 2^18), and the ring positions advance incrementally.
            const uint32_t idesc = idesc_e4m3_f32(PAIR ? 256 : 128, BN);
            const uint64_t da0 = sdesc_kmajor_sw128(smem_u32(smA));
            const uint64_t db0 = sdesc_kmajor_sw128(smem_u32(smB));
            uint32_t s = 0, ph = 0, buf = 0, tph = 0;
            Sched sc = sched_init(SK, unit, nunits, T, KB);
            int t, kb0, kb1;
            while (sched_next(sc, t, kb0, kb1)) {
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(bar(C::BAR_TEMPTY + buf), tph ^ 1, ctl, 0x0200 | buf))
                        goto mma_done;
                    if (!mbar_wait(bar(C::BAR_FULL + s), ph, ctl, 0x0210 | s))
                        goto mma_done;
                    tc_fence_after();
                    const uint64_t da = da0 + s * (A_BYTES >> 4), db = db0 + s * (C::B_BYTES >> 4);
                    const uint32_t d = tmem_base + buf * BN;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k) {   // K = 32 per MMA: +32 bytes = +2 in the field
                        if (PAIR)
                            umma_e4m3_pair(d, da + 2 * k, db + 2 * k, idesc, k > 0 ? 1u : 0u);
                        else
                            umma_e4m3(d, da + 2 * k, db + 2 * k, idesc, k > 0 ? 1u : 0u);
                    }
                    if (PAIR)
                        umma_commit_pair_mc(bar(C::BAR_DONE + s), 0x3);   // in both CTAs
                    else
                        umma_commit(bar(C::BAR_DONE + s));
                    if (++s == static_cast<uint32_t>(STAGES)) {
                        s = 0;
                        ph ^= 1;
                    }
                    buf ^= 1;
                    tph ^= buf ^ 1;   // flips after every second slice
                }
            }
        mma_done:
            if (PAIR)
                umma_commit_pair_mc(bar(C::BAR_DRAIN), 0x1);
            else
                umma_commit(bar(C::BAR_DRAIN));
            mbar_wait_drain(bar(C::BAR_DRAIN), 0, p.timeout_ns);
        } else if (warp == 2) {
            // ---------------------------------------------------------- scale loader
            uint32_t it = 0;
            Sched sc = sched_init(SK, unit, nunits, T, KB);
            int t, kb0, kb1;
            while (sched_next(sc, t, kb0, kb1)) {
                const Tile ti = tile_of(t);
                if (FUSE && !wait_count(f.ready + ti.g, goff[ti.g + 1] - goff[ti.g], ctl, 0x0380))
                    goto scale_done;
                const float *sbg = p.sB + ti.sb_base;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const uint32_t j = it % SSLOTS, ph = (it / SSLOTS) & 1;
                    if (!mbar_wait(bar(C::BAR_SEMPTY + j), ph ^ 1, ctl, 0x0300 | j))
                        goto scale_done;
                    const float *sa_row = p.sA + static_cast<int64_t>(kb) * p.ldsa;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = ti.row0 + lane + 32 * i;
                        const bool ok = r < ti.row_end;
                        cp_async_4(smem_u32(ssa + j * 128 + lane + 32 * i), ok ? sa_row + r : p.sA, ok ? 4u : 0u);
                    }
                    if (SCALE_B == kScaleRowKN) {
                        const float *sb_row = sbg + static_cast<int64_t>(kb) * p.ldsb;
#pragma unroll
                        for (int i = 0; i < BN / 32; ++i) {
                            const int n = ti.n0 + lane + 32 * i;
                            const bool ok = n < N;
                            cp_async_4(smem_u32(ssb + j * BN + lane + 32 * i), ok ? sb_row + n : p.sB, ok ? 4u : 0u);
                        }
                    } else if (lane < BN / 128) {
                        // SwiGLU: lane 0 the gate rows' block, lane 1 the up rows'
                        const int nb = SWIGLU ? (ti.n0 + lane * p.sw_width) / 128 : ti.n0 / 128 + lane;
                        const bool ok = nb * 128 < N;
                        const float *src = SCALE_B == kScaleBlockNK ? sbg + nb * p.ldsb + kb
                                                                    : sbg + static_cast<int64_t>(kb) * p.ldsb + nb;
                        cp_async_4(smem_u32(ssb + j * BN + lane), ok ? src : p.sB, ok ? 4u : 0u);
                    }
                    cp_async_arrive_noinc(bar(C::BAR_SFULL + j));
                }
            }
        scale_done:
            cp_async_wait_all();
        } else if (SWIGLU && warp >= 12) {
            // ---------------------------------------------------------- SwiGLU epilogue
            // Thread er owns row er of this CTA's 128 tile rows and the tile's whole group of
            // 128 output columns [n0, n0 + 128): x = silu(gate) * up of the BF16 values the
            // promotion warps handed over, the group's max-abs and scale, 128 codes (and the
            // BF16 gate / up row when it is kept).  Hand-over layout: row r at r * 512 bytes,
            // the 16-byte chunk of columns 4j .. 4j+3 (a word per column, gate | up << 16) at
            // chunk j ^ (r mod 32); the first pass overwrites each word with x in binary32.
            const int er = (warp - 12) * 32 + lane;
            const uint32_t rowb = smem_u32(smO) + static_cast<uint32_t>(er) * 512;
            const uint32_t sw = static_cast<uint32_t>(er & 31);
            uint32_t ec = 0;
            Sched sc = sched_init(SK, unit, nunits, T, KB);
            int t, kb0, kb1;
            while (sched_next(sc, t, kb0, kb1)) {
                const Tile ti = tile_of(t);
                if (!mbar_wait_sleepy(bar(C::BAR_XFULL), ec & 1, ctl, 0x04E0))
                    break;
                const int m = ti.row0 + er;
                if (m < ti.row_end) {
                    __nv_bfloat16 *crow =
                        p.C != nullptr ? static_cast<__nv_bfloat16 *>(p.C) + static_cast<int64_t>(m) * p.ldc : nullptr;
                    float amax = 0.0f;
#pragma unroll 4
                    for (int j = 0; j < 32; ++j) {
                        const uint32_t addr = rowb + ((static_cast<uint32_t>(j) ^ sw) << 4);
                        const uint4 w = lds_v4(addr);
                        float x0, x1, x2, x3;
                        swiglu2(__uint_as_float(bf16x2_lo(w.x)), __uint_as_float(bf16x2_lo(w.y)),
                                __uint_as_float(bf16x2_hi(w.x)), __uint_as_float(bf16x2_hi(w.y)), x0, x1);
                        swiglu2(__uint_as_float(bf16x2_lo(w.z)), __uint_as_float(bf16x2_lo(w.w)),
                                __uint_as_float(bf16x2_hi(w.z)), __uint_as_float(bf16x2_hi(w.w)), x2, x3);
                        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3))));
                        if (crow != nullptr) {   // the cached SwiGLU input: gate | up, BF16
                            *reinterpret_cast<uint2 *>(crow + ti.n0 + 4 * j) =
                                make_uint2((w.x & 0xFFFFu) | (w.y << 16), (w.z & 0xFFFFu) | (w.w << 16));
                            *reinterpret_cast<uint2 *>(crow + p.sw_width + ti.n0 + 4 * j) =
                                make_uint2((w.x >> 16) | (w.y & 0xFFFF0000u), (w.z >> 16) | (w.w & 0xFFFF0000u));
                        }
                        sts_v4(addr, __float_as_uint(x0), __float_as_uint(x1), __float_as_uint(x2), __float_as_uint(x3));
                    }
                    const GroupScale gs = make_group_scale(amax, p.sw_pow2 != 0);
                    uint4 *qd = reinterpret_cast<uint4 *>(p.sw_q + static_cast<int64_t>(m) * p.sw_ldq + ti.n0);
#pragma unroll 2
                    for (int i = 0; i < 8; ++i) {   // sixteen codes per 16-byte store
                        float xs[16];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 v = lds_v4(rowb + ((static_cast<uint32_t>(4 * i + c) ^ sw) << 4));
                            xs[4 * c] = __uint_as_float(v.x);
                            xs[4 * c + 1] = __uint_as_float(v.y);
                            xs[4 * c + 2] = __uint_as_float(v.z);
                            xs[4 * c + 3] = __uint_as_float(v.w);
                        }
                        uint32_t w4[4];
                        codes_f32<16>(xs, gs, w4);
                        qd[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    p.sw_s[static_cast<int64_t>(ti.n0 / 128) * p.sw_lds + m] = gs.s;
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(C::BAR_XEMPTY));   // the hand-over area may be refilled
                ++ec;
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(SWIGLU ? 216 : C::regs_high(SCALE_B, GROUPED))
                     : "memory");
        // -------------------------------------------------------------- promotion
        const int ew = warp - 4, quad = warp & 3, half = ew >> 2;
        const int row_in = quad * 32 + lane;
        const uint32_t tm_lane = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t it = 0;
        bool ok = true;
        uint32_t xpar = 0;   // SwiGLU: tiles handed over
        Sched sc = sched_init(SK, unit, nunits, T, KB);
        int t, kb0, kb1;
        while (ok && sched_next(sc, t, kb0, kb1)) {
            const Tile ti = tile_of(t);
            // A warp whose 32 rows all lie past the expert's last row (a short expert's tile)
            // keeps every barrier wait and arrival but reads no TMEM and does no FMAs: less
            // TMEM traffic for the other warps (grouped prefill 3-4% faster).  Not in SwiGLU
            // tiles, whose promotion loop spills more with the branch and ran 9-12% slower.
            const bool live = !GROUPED || SWIGLU || ti.row0 + quad * 32 < ti.row_end;
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i)
                acc[i] = 0.0f;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const uint32_t j = it % SSLOTS, sph = (it / SSLOTS) & 1;
                const uint32_t buf = it & 1;
                const uint32_t ds = it % STAGES, dph = (it / STAGES) & 1;
                if (!mbar_wait(bar(C::BAR_SFULL + j), sph, ctl, 0x0400 | j) ||
                    !mbar_wait(bar(C::BAR_DONE + ds), dph, ctl, 0x0410 | ds)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (live) {
                    const float sa = ssa[j * 128 + row_in];
                    float sc = 0.0f, sc2 = 0.0f;
                    if (SCALE_B != kScaleRowKN)
                        sc = sa * ssb[j * BN + (SWIGLU ? 0 : half)];
                    if (SWIGLU)
                        sc2 = sa * ssb[j * BN + 1];
                    else
                        sc2 = sc;
                    const float *sbcol = ssb + j * BN + half * 128;
                    // chunk columns: half * 128 + {0, 32, 64, 96}; SwiGLU: gate half * 64 + {0, 32},
                    // up 128 + half * 64 + {0, 32} (acc[0, 64) gate, acc[64, 128) up, same columns)
                    const uint32_t taddr = tmem_base + tm_lane + buf * BN + (SWIGLU ? half * 64 : half * 128);
                    constexpr uint32_t O2 = SWIGLU ? 128 : 64, O3 = SWIGLU ? 160 : 96;
                    // two TMEM loads in flight: 0,1 | 2 while promoting 0 | 3 while promoting 1
                    uint32_t va[32], vb[32];
                    MPQ_TMEM_LD32(taddr, va);
                    MPQ_TMEM_LD32(taddr + 32, vb);
                    MPQ_TMEM_WAIT_LD32(va);
                    MPQ_TMEM_WAIT_LD32(vb);
                    promote_chunk<SCALE_B>(acc, va, 0, sc, sa, sbcol);
                    MPQ_TMEM_LD32(taddr + O2, va);
                    promote_chunk<SCALE_B>(acc, vb, 1, sc, sa, sbcol);
                    MPQ_TMEM_LD32(taddr + O3, vb);
                    MPQ_TMEM_WAIT_LD32(va);
                    promote_chunk<SCALE_B>(acc, va, 2, sc2, sa, sbcol);
                    MPQ_TMEM_WAIT_LD32(vb);
                    promote_chunk<SCALE_B>(acc, vb, 3, sc2, sa, sbcol);
                }
                // Release the partial buffer only after the last FMAs: releasing it as soon as
                // the loads land lets the next MMAs start earlier and measurably slows the
                // other warps' TMEM loads (about 25% on 4096 x 18432 x 7168).
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR)
                        mbar_arrive_remote(mapa_shared(bar(C::BAR_TEMPTY + buf), 0));   // the even CTA's
                    else
                        mbar_arrive(bar(C::BAR_TEMPTY + buf));
                    mbar_arrive(bar(C::BAR_SEMPTY + j));
                }
            }
            if (!ok)
                break;
            if (SK && kb0 > 0) {
                // Tail of a tile the previous unit finishes: hand this warp's partial over
                // (layout [unit][rank (pair mode)][warp][i][lane], coalesced) and announce it.
                float4 *dst = p.sk_part + ((static_cast<int64_t>(unit) * (PAIR ? 2 : 1) + rank) * 8 + ew) * 1024 + lane;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    dst[32 * i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    asm volatile("st.release.gpu.global.s32 [%0], %1;"
                                 ::"l"(p.sk_flags + (unit * (PAIR ? 2 : 1) + rank) * 8 + ew),
                                 "r"(p.sk_epoch)
                                 : "memory");
                continue;
            }
            if (SK && kb1 < KB) {
                // Head of a tile: add the tail the next unit computed (final sum: head + tail).
                const int slot = ((unit + 1) * (PAIR ? 2 : 1) + static_cast<int>(rank)) * 8 + ew;
                if (!wait_count(p.sk_flags + slot, p.sk_epoch, ctl, 0x0480)) {
                    ok = false;
                    break;
                }
                const float4 *src = p.sk_part + static_cast<int64_t>(slot) * 1024 + lane;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float4 v = __ldcg(src + 32 * i);
                    acc[4 * i] = __fadd_rn(acc[4 * i], v.x);
                    acc[4 * i + 1] = __fadd_rn(acc[4 * i + 1], v.y);
                    acc[4 * i + 2] = __fadd_rn(acc[4 * i + 2], v.z);
                    acc[4 * i + 3] = __fadd_rn(acc[4 * i + 3], v.w);
                }
            }
            if constexpr (SWIGLU) {
                // Hand the tile's gate and up values, rounded to BF16 (the values the plain
                // grouped GEMM writes), to the epilogue warps: this thread's row, columns
                // half * 64 .. +63 (chunks half * 16 .. +15 of the row's 32)
                if (!mbar_wait(bar(C::BAR_XEMPTY), (xpar & 1) ^ 1, ctl, 0x04D0)) {
                    ok = false;
                    break;
                }
                const uint32_t rowb = smem_u32(smO) + static_cast<uint32_t>(row_in) * 512;
#pragma unroll
                for (int c4 = 0; c4 < 16; ++c4) {
                    uint32_t w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const __nv_bfloat162 gu = __floats2bfloat162_rn(acc[4 * c4 + k], acc[64 + 4 * c4 + k]);
                        w[k] = *reinterpret_cast<const uint32_t *>(&gu);
                    }
                    const uint32_t j = static_cast<uint32_t>(half * 16 + c4);
                    sts_v4(rowb + ((j ^ static_cast<uint32_t>(row_in & 31)) << 4), w[0], w[1], w[2], w[3]);
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar(C::BAR_XFULL));
                ++xpar;
                continue;
            }
            // Output: rows [ti.row0 + 32 quad, +32), columns [ti.n0 + 128 half, +128).  A warp
            // whose 32 rows all belong to this tile stages row pieces (128 bytes in pair mode,
            // 64 single-SM) in its swizzled buffers and writes them with TMA stores (clipped at
            // the tensor bounds);
            // a warp on a ragged expert boundary stores its valid rows directly.
            const int wrow0 = ti.row0 + quad * 32;
            const int ncol0 = ti.n0 + half * 128;
            if (ncol0 < N) {
                const bool whole = GROUPED ? (wrow0 + 32 <= ti.row_end) : true;
                if (whole) {
                    const uint32_t stg0 = smem_u32(smO + ew * C::OUT_BUFS * C::STAGE_OUT);
                    constexpr int COLS = C::ROWB / (OUT_F32 ? 4 : 2);   // columns per row piece
                    constexpr int PCS = C::ROWB / 16;                   // 16-byte pieces per row piece
#pragma unroll
                    for (int ch = 0; ch < 128 / COLS; ++ch) {
                        const uint32_t stg_u32 = stg0 + (ch % C::OUT_BUFS) * C::STAGE_OUT;
                        if (lane == 0) {                                // the buffer's last piece has left smem
                            if (C::OUT_BUFS == 4)
                                bulk_wait_read3();
                            else if (C::OUT_BUFS == 2)
                                bulk_wait_read1();
                            else
                                bulk_wait_read0();
                        }
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < PCS; ++j) {                 // 16-byte pieces of the row
                            uint4 w;
                            if (OUT_F32) {
                                const int a0 = ch * COLS + j * 4;         // columns ch*16+4j..+3
                                w = make_uint4(__float_as_uint(acc[a0]), __float_as_uint(acc[a0 + 1]),
                                               __float_as_uint(acc[a0 + 2]), __float_as_uint(acc[a0 + 3]));
                            } else {
                                const int a0 = ch * COLS + j * 8;         // columns ch*32+8j..+7
                                uint32_t h[4];
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[a0 + 2 * k], acc[a0 + 2 * k + 1]);
                                    h[k] = *reinterpret_cast<const uint32_t *>(&b2);
                                }
                                w = make_uint4(h[0], h[1], h[2], h[3]);
                            }
                            // 128-byte swizzle: 16-byte piece j of row r sits at piece j ^ (r & 7);
                            // 64-byte swizzle: at piece j ^ ((r >> 1) & 3)
                            const uint32_t off = PCS == 8 ? lane * 128 + ((j ^ (lane & 7)) << 4)
                                                          : lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4);
                            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(stg_u32 + off), "r"(w.x),
                                         "r"(w.y), "r"(w.z), "r"(w.w)
                                         : "memory");
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmC, stg_u32, ncol0 + ch * COLS, wrow0);
                            bulk_commit();
                        }
                    }
                } else if (wrow0 + lane < ti.row_end) {
                    const int64_t m = wrow0 + lane;
                    const int64_t n = ncol0;
                    if (OUT_F32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.C) + m * p.ldc + n);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            dst[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.C) + m * p.ldc + n);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            uint32_t w[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const __nv_bfloat162 b2 =
                                    __floats2bfloat162_rn(acc[8 * i + 2 * k], acc[8 * i + 2 * k + 1]);
                                w[k] = *reinterpret_cast<const uint32_t *>(&b2);
                            }
                            dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            }
        }
        if (lane == 0)
            bulk_wait0();   // every TMA store of this warp has completed
    }

    tc_fence_before();
    __syncthreads();
    if (PAIR)
        cluster_sync_all();  // the pair's MMAs, copies and remote arrivals are all complete
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

__global__ void wait_selftest_kernel(int *status, uint64_t timeout_ns)
{
    __shared__ uint64_t b;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&b), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        WaitCtl c{&abort_flag, status, timeout_ns};
        // Nothing ever arrives on this barrier: the wait must give up and report.
        mbar_wait(smem_u32(&b), 0, c, 0x7F01);
    }
}

template <int SB, bool F32, bool GR, bool PAIR, bool FUSE, bool SK, bool SWIGLU = false>
cudaError_t launch_one(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC, const GemmArgs &a,
                       const FuseArgs &f, int grid, cudaStream_t st)
{
    auto kern = gemm_kernel<SB, F32, GR, PAIR, FUSE, SK, SWIGLU>;
    const size_t smem = smem_bytes<PAIR>(GR, SWIGLU);
    static std::atomic<uint64_t> configured{0};   // per instantiation: devices already set up
    if (cudaError_t e = ensure_max_dyn_smem(kern, smem, configured); e != cudaSuccess)
        return e;
    if (!PAIR && !FUSE) {
        kern<<<grid, threads_of(SWIGLU), smem, st>>>(tmA, tmB, tmC, a, f);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(threads_of(SWIGLU), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (PAIR) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
    } else {
        // Fused quantization: phase 2 waits on phase-1 work of every CTA, so all CTAs must be
        // resident at once -- a cooperative launch guarantees it (or fails).
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, a, f);
}

} // namespace

int gemm_b_box_rows(bool pair) { return pair ? Cfg<true>::B_ROWS : Cfg<false>::B_ROWS; }

cudaError_t launch_gemm(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC, const GemmArgs &a,
                        int scale_b, bool out_fp32, bool pair, int num_sms, cudaStream_t st, const FuseArgs *fuse)
{
    const bool grouped = a.offsets != nullptr;
    if (grouped && a.G > kMaxGroups)
        return cudaErrorInvalidValue;
    const int tile_m = pair ? 256 : 128;
    int64_t tiles;
    if (grouped)  // upper bound: every expert may add one partial m-tile
        tiles = ((a.M + tile_m - 1) / tile_m + a.G) * ((a.N + BN - 1) / BN);
    else
        tiles = ((a.M + tile_m - 1) / tile_m) * ((a.N + BN - 1) / BN);
    if (tiles <= 0)
        return cudaSuccess;
    int grid;
    if (pair) {
        const int64_t pairs = tiles < num_sms / 2 ? tiles : num_sms / 2;
        grid = static_cast<int>(2 * (pairs < 1 ? 1 : pairs));
    } else {
        grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    }
    const FuseArgs none{};
    if (fuse != nullptr) {   // grouped, single-SM tiles, weight block scales; one CTA per SM
        if (!grouped || pair || scale_b != kScaleBlockNK)
            return cudaErrorInvalidValue;
        cudaError_t e = cudaMemsetAsync(fuse->ready, 0, sizeof(int) * static_cast<size_t>(a.G), st);
        if (e != cudaSuccess)
            return e;
        return out_fp32 ? launch_one<kScaleBlockNK, true, true, false, true, false>(tmA, tmB, tmC, a, *fuse, num_sms, st)
                        : launch_one<kScaleBlockNK, false, true, false, true, false>(tmA, tmB, tmC, a, *fuse, num_sms, st);
    }
    const bool sk = a.sk_part != nullptr;
    if (sk && (grouped || tiles < (pair ? grid / 2 : grid)))   // stream-K: dense, at least one wave
        return cudaErrorInvalidValue;
#define MPQ_G(SB, F32, GR, PR, SKV)                                                        \
    if (scale_b == SB && out_fp32 == F32 && grouped == GR && pair == PR && sk == SKV)      \
        return launch_one<SB, F32, GR, PR, false, SKV>(tmA, tmB, tmC, a, none, grid, st);
#define MPQ_G2(SB, F32, GR, SKV) MPQ_G(SB, F32, GR, true, SKV) MPQ_G(SB, F32, GR, false, SKV)
    MPQ_G2(kScaleBlockNK, false, false, false)
    MPQ_G2(kScaleBlockNK, true, false, false)
    MPQ_G2(kScaleBlockKN, false, false, false)
    MPQ_G2(kScaleBlockKN, true, false, false)
    MPQ_G2(kScaleRowKN, false, false, false)
    MPQ_G2(kScaleRowKN, true, false, false)
    MPQ_G2(kScaleBlockNK, false, false, true)
    MPQ_G2(kScaleBlockNK, true, false, true)
    MPQ_G2(kScaleBlockKN, false, false, true)
    MPQ_G2(kScaleBlockKN, true, false, true)
    MPQ_G2(kScaleRowKN, false, false, true)
    MPQ_G2(kScaleRowKN, true, false, true)
    MPQ_G2(kScaleBlockNK, false, true, false)
    MPQ_G2(kScaleBlockNK, true, true, false)
#undef MPQ_G2
#undef MPQ_G
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_swiglu(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &a, bool pair,
                               int num_sms, cudaStream_t st, const FuseArgs *fuse)
{
    if (a.offsets == nullptr || a.G > kMaxGroups || a.sw_q == nullptr || a.sw_width <= 0 || a.sw_width % 128 != 0 ||
        a.N != 2 * static_cast<int64_t>(a.sw_width))
        return cudaErrorInvalidValue;
    const int tile_m = pair ? 256 : 128;
    // upper bound: every expert may add one partial m-tile
    const int64_t tiles = ((a.M + tile_m - 1) / tile_m + a.G) * (a.sw_width / 128);
    if (tiles <= 0)
        return cudaSuccess;
    // the output view is not used (no TMA stores): tmB stands in for it
    const FuseArgs none{};
    if (fuse != nullptr) {   // single-SM tiles, one cooperative CTA per SM
        if (pair)
            return cudaErrorInvalidValue;
        cudaError_t e = cudaMemsetAsync(fuse->ready, 0, sizeof(int) * static_cast<size_t>(a.G), st);
        if (e != cudaSuccess)
            return e;
        return launch_one<kScaleBlockNK, false, true, false, true, false, true>(tmA, tmB, tmB, a, *fuse, num_sms, st);
    }
    if (pair) {
        const int64_t pairs = tiles < num_sms / 2 ? tiles : num_sms / 2;
        return launch_one<kScaleBlockNK, false, true, true, false, false, true>(tmA, tmB, tmB, a, none,
                                                                               static_cast<int>(2 * (pairs < 1 ? 1 : pairs)), st);
    }
    const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    return launch_one<kScaleBlockNK, false, true, false, false, false, true>(tmA, tmB, tmB, a, none, grid, st);
}

cudaError_t launch_wait_selftest(int *status, uint64_t timeout_ns, cudaStream_t st)
{
    wait_selftest_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
    return cudaGetLastError();
}

} // namespace mpq

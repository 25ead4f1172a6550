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
// Design (B300, one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: A 128x128 and B 256x128 E4M3 slices into a 4-stage ring
//               (128-byte swizzle), one mbarrier per stage;
//   warp 1      MMA issuer: four tcgen05.mma (M=128, N=256, K=32) per 128-K slice into
//               one of two TMEM partial buffers (2 x 256 columns), committed per slice;
//   warp 2      scale loader: cp.async of the slice's A and B scales into an 8-slot ring;
//   warps 4-11  promotion: tcgen05.ld the slice partial, multiply by its two scales and
//               accumulate into FP32 registers with packed FP32x2 FMAs, then write the
//               tile as BF16 or FP32.  Promotion of slice k overlaps the MMAs of k+1.
// Every wait is bounded; on expiry the CTA records a timeout in the status word,
// drains its copies and MMAs, frees TMEM and exits.
#include "mpq_internal.h"
#include "mpq_device.cuh"

namespace mpq {
namespace {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int STAGES = 4;
constexpr int SSLOTS = 8;
constexpr int kThreads = 384;
constexpr uint32_t A_BYTES = BM * BK;
constexpr uint32_t B_BYTES = BN * BK;
constexpr uint32_t TMEM_COLS = 512;
constexpr int kMaxGroups = 1024;

// Barrier indices inside the barrier array.
constexpr int BAR_FULL = 0;
constexpr int BAR_EMPTY = BAR_FULL + STAGES;
constexpr int BAR_TFULL = BAR_EMPTY + STAGES;
constexpr int BAR_TEMPTY = BAR_TFULL + 2;
constexpr int BAR_SFULL = BAR_TEMPTY + 2;
constexpr int BAR_SEMPTY = BAR_SFULL + SSLOTS;
constexpr int BAR_DRAIN = BAR_SEMPTY + SSLOTS;
constexpr int NBARS = BAR_DRAIN + 1;

constexpr size_t kSmemMain = STAGES * (A_BYTES + B_BYTES) + SSLOTS * (BM + BN) * sizeof(float) +
                             NBARS * sizeof(uint64_t) + 16;
constexpr size_t kSmemGroups = (kMaxGroups + 1) * (sizeof(int64_t) + sizeof(int)) + 16;

size_t smem_bytes(bool grouped) { return 1024 + kSmemMain + (grouped ? kSmemGroups : 0); }

// Sizes are validated on the host to stay below 2^31 rows / columns.
struct Tile {
    int row0;         // first row of A / C
    int row_end;      // one past the last valid row of this tile
    int brow0;        // first row of B in the TMA view ([G*N, K] when grouped)
    int n0;           // first output column
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

template <int SCALE_B, bool OUT_F32, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *smA = base;
    uint8_t *smB = smA + STAGES * A_BYTES;
    float *ssa = reinterpret_cast<float *>(smB + STAGES * B_BYTES);
    float *ssb = ssa + SSLOTS * BM;
    uint64_t *bars = reinterpret_cast<uint64_t *>(ssb + SSLOTS * BN);
    uint32_t *misc = reinterpret_cast<uint32_t *>(bars + NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    int64_t *goff = reinterpret_cast<int64_t *>(misc + 4);   // grouped: clamped offsets [G+1]
    int *gtile = reinterpret_cast<int *>(goff + kMaxGroups + 1);  // grouped: first tile of expert

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };

    const int64_t M = p.M, N = p.N;
    const int KB = static_cast<int>(p.K / BK);
    const int NT = static_cast<int>((N + BN - 1) / BN);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(BAR_FULL + s), 1);
            mbar_init(bar(BAR_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(BAR_TFULL + b), 1);
            mbar_init(bar(BAR_TEMPTY + b), 8);
        }
        for (int j = 0; j < SSLOTS; ++j) {
            mbar_init(bar(BAR_SFULL + j), 32);
            mbar_init(bar(BAR_SEMPTY + j), 8);
        }
        mbar_init(bar(BAR_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), TMEM_COLS);
        tmem_relinquish();
    }
    if (GROUPED && warp == 2) {
        // Expert schedule: offsets clamped into [0, M] and made monotone (running max),
        // then the exclusive prefix sum of m-tiles per expert, times the n-tile count.
        const int G = p.G;
        for (int g = lane; g <= G; g += 32) {
            const int64_t o = p.offsets[g];
            goff[g] = o < 0 ? 0 : (o > M ? M : o);
        }
        __syncwarp();
        const int per = (G + 1 + 31) / 32;
        const int c0 = lane * per, c1 = c0 + per < G + 1 ? c0 + per : G + 1;
        int64_t mx = 0;
        for (int g = c0; g < c1; ++g)
            mx = goff[g] > mx ? goff[g] : mx;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t v = __shfl_up_sync(0xffffffffu, mx, o);
            if (lane >= o && v > mx)
                mx = v;
        }
        int64_t run = __shfl_up_sync(0xffffffffu, mx, 1);
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
            cnt += static_cast<int>((goff[g + 1] - goff[g] + BM - 1) / BM);
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
            ex += static_cast<int>((goff[g + 1] - goff[g] + BM - 1) / BM);
        }
        if (lane == 31)
            gtile[G] = incl * NT;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc[0];

    const int T = GROUPED ? gtile[p.G] : static_cast<int>(((M + BM - 1) / BM) * NT);
    const int MT = static_cast<int>((M + BM - 1) / BM);

    auto tile_of = [&](int t) -> Tile {
        Tile ti;
        if (!GROUPED) {
            const int mt = t % MT, nt = t / MT;
            ti.row0 = mt * BM;
            ti.row_end = ti.row0 + BM < M ? ti.row0 + BM : static_cast<int>(M);
            ti.n0 = nt * BN;
            ti.brow0 = ti.n0;
            ti.sb_base = 0;
        } else {
            int lo = 0, hi = p.G - 1;  // last expert whose first tile is <= t
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (gtile[mid] <= t) lo = mid; else hi = mid - 1;
            }
            const int g = lo;
            const int local = t - gtile[g];
            const int mtg = static_cast<int>((goff[g + 1] - goff[g] + BM - 1) / BM);
            const int nt = local / mtg, mt = local - nt * mtg;
            const int gend = static_cast<int>(goff[g + 1]);
            ti.row0 = static_cast<int>(goff[g]) + mt * BM;
            ti.row_end = ti.row0 + BM < gend ? ti.row0 + BM : gend;
            ti.n0 = nt * BN;
            ti.brow0 = g * static_cast<int>(N) + ti.n0;
            ti.sb_base = static_cast<int64_t>(g) * p.sb_group_stride;
        }
        return ti;
    };

    WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
        if (warp == 0 && lane == 0) {
            // ---------------------------------------------------------- TMA producer
            uint32_t it = 0;
            for (int t = blockIdx.x; t < T; t += gridDim.x) {
                const Tile ti = tile_of(t);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (!mbar_wait(bar(BAR_EMPTY + s), ph ^ 1, ctl, 0x0100 | s))
                        goto producer_done;
                    mbar_arrive_expect_tx(bar(BAR_FULL + s), A_BYTES + B_BYTES);
                    tma_load_2d(smem_u32(smA + s * A_BYTES), &tmA, bar(BAR_FULL + s), kb * BK, ti.row0);
                    tma_load_2d(smem_u32(smB + s * B_BYTES), &tmB, bar(BAR_FULL + s), kb * BK, ti.brow0);
                }
            }
        producer_done:
            for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; ++j)
                mbar_wait_drain(bar(BAR_FULL + j % STAGES), (j / STAGES) & 1, p.timeout_ns);
        } else if (warp == 1 && lane == 0) {
            // ---------------------------------------------------------- MMA issuer
            const uint32_t idesc = idesc_e4m3_f32(BM, BN);
            uint32_t it = 0;
            for (int t = blockIdx.x; t < T; t += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    const uint32_t buf = it & 1, tph = (it >> 1) & 1;
                    if (!mbar_wait(bar(BAR_TEMPTY + buf), tph ^ 1, ctl, 0x0200 | buf))
                        goto mma_done;
                    if (!mbar_wait(bar(BAR_FULL + s), ph, ctl, 0x0210 | s))
                        goto mma_done;
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smA + s * A_BYTES);
                    const uint32_t b0 = smem_u32(smB + s * B_BYTES);
                    const uint32_t d = tmem_base + buf * BN;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        umma_e4m3(d, sdesc_kmajor_sw128(a0 + k * 32), sdesc_kmajor_sw128(b0 + k * 32), idesc,
                                  k > 0 ? 1u : 0u);
                    umma_commit(bar(BAR_EMPTY + s));
                    umma_commit(bar(BAR_TFULL + buf));
                }
            }
        mma_done:
            umma_commit(bar(BAR_DRAIN));
            mbar_wait_drain(bar(BAR_DRAIN), 0, p.timeout_ns);
        } else if (warp == 2) {
            // ---------------------------------------------------------- scale loader
            uint32_t it = 0;
            for (int t = blockIdx.x; t < T; t += gridDim.x) {
                const Tile ti = tile_of(t);
                const float *sbg = p.sB + ti.sb_base;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t j = it % SSLOTS, ph = (it / SSLOTS) & 1;
                    if (!mbar_wait(bar(BAR_SEMPTY + j), ph ^ 1, ctl, 0x0300 | j))
                        goto scale_done;
                    const float *sa_row = p.sA + static_cast<int64_t>(kb) * p.ldsa;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = ti.row0 + lane + 32 * i;
                        const bool ok = r < ti.row_end;
                        cp_async_4(smem_u32(ssa + j * BM + lane + 32 * i), ok ? sa_row + r : p.sA, ok ? 4u : 0u);
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
                        const int nb = ti.n0 / 128 + lane;
                        const bool ok = nb * 128 < N;
                        const float *src = SCALE_B == kScaleBlockNK ? sbg + nb * p.ldsb + kb
                                                                    : sbg + static_cast<int64_t>(kb) * p.ldsb + nb;
                        cp_async_4(smem_u32(ssb + j * BN + lane), ok ? src : p.sB, ok ? 4u : 0u);
                    }
                    cp_async_arrive_noinc(bar(BAR_SFULL + j));
                }
            }
        scale_done:
            cp_async_wait_all();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 224;" ::: "memory");
        // -------------------------------------------------------------- promotion
        const int ew = warp - 4, quad = warp & 3, half = ew >> 2;
        const int row_in = quad * 32 + lane;
        const uint32_t tm_lane = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
            const Tile ti = tile_of(t);
            // decided before the K loop: keeps the tile bounds out of the loop's live registers
            const bool store_ok = (ti.row0 + row_in < ti.row_end) && (ti.n0 + half * 128 < N);
            unsigned long long acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i)
                acc[i] = 0ull;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const uint32_t j = it % SSLOTS, sph = (it / SSLOTS) & 1;
                const uint32_t buf = it & 1, tph = (it >> 1) & 1;
                if (!mbar_wait(bar(BAR_SFULL + j), sph, ctl, 0x0400 | j) ||
                    !mbar_wait(bar(BAR_TFULL + buf), tph, ctl, 0x0410 | buf)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float sa = ssa[j * BM + row_in];
                const unsigned long long sa2 = pack2(sa, sa);
                float sc = 0.0f;
                if (SCALE_B != kScaleRowKN)
                    sc = sa * ssb[j * BN + half];
                const unsigned long long sc2 = pack2(sc, sc);
                const uint32_t taddr = tmem_base + tm_lane + buf * BN + half * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    MPQ_TMEM_LD32(taddr + c * 32, v);
                    MPQ_TMEM_WAIT_LD32(v);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const unsigned long long pv =
                            (static_cast<unsigned long long>(v[2 * q + 1]) << 32) | v[2 * q];
                        if (SCALE_B == kScaleRowKN) {
                            const unsigned long long sb2 = *reinterpret_cast<const unsigned long long *>(
                                ssb + j * BN + half * 128 + c * 32 + 2 * q);
                            acc[c * 16 + q] = ffma2(fmul2(pv, sb2), sa2, acc[c * 16 + q]);
                        } else {
                            acc[c * 16 + q] = ffma2(pv, sc2, acc[c * 16 + q]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(BAR_TEMPTY + buf));
                    mbar_arrive(bar(BAR_SEMPTY + j));
                }
            }
            if (!ok)
                break;
            if (store_ok) {
                const int64_t m = ti.row0 + row_in;
                const int64_t n = ti.n0 + half * 128;
                if (OUT_F32) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.C) + m * p.ldc + n);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        dst[i] = make_float4(lo_of(acc[2 * i]), hi_of(acc[2 * i]), lo_of(acc[2 * i + 1]),
                                             hi_of(acc[2 * i + 1]));
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.C) + m * p.ldc + n);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        uint32_t w[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const __nv_bfloat162 b2 =
                                __floats2bfloat162_rn(lo_of(acc[4 * i + k]), hi_of(acc[4 * i + k]));
                            w[k] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
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

template <int SB, bool F32, bool GR>
cudaError_t launch_one(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &a, int grid,
                       cudaStream_t st)
{
    auto kern = gemm_kernel<SB, F32, GR>;
    const size_t smem = smem_bytes(GR);
    static bool configured = false;  // one attribute call per instantiation and process
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    kern<<<grid, kThreads, smem, st>>>(tmA, tmB, a);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_gemm(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &a, int scale_b,
                        bool out_fp32, int num_sms, cudaStream_t st)
{
    const bool grouped = a.offsets != nullptr;
    if (grouped && a.G > kMaxGroups)
        return cudaErrorInvalidValue;
    int64_t tiles;
    if (grouped) {
        // upper bound: every expert may add one partial m-tile
        tiles = ((a.M + BM - 1) / BM + a.G) * ((a.N + BN - 1) / BN);
    } else {
        tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
    }
    if (tiles <= 0)
        return cudaSuccess;
    const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
#define MPQ_G(SB, F32, GR)                                                     \
    if (scale_b == SB && out_fp32 == F32 && grouped == GR)                     \
        return launch_one<SB, F32, GR>(tmA, tmB, a, grid, st);
    MPQ_G(kScaleBlockNK, false, false)
    MPQ_G(kScaleBlockNK, true, false)
    MPQ_G(kScaleBlockKN, false, false)
    MPQ_G(kScaleBlockKN, true, false)
    MPQ_G(kScaleRowKN, false, false)
    MPQ_G(kScaleRowKN, true, false)
    MPQ_G(kScaleBlockNK, false, true)
    MPQ_G(kScaleBlockNK, true, true)
#undef MPQ_G
    return cudaErrorInvalidValue;
}

cudaError_t launch_wait_selftest(int *status, uint64_t timeout_ns, cudaStream_t st)
{
    wait_selftest_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
    return cudaGetLastError();
}

} // namespace mpq

// decode.cu -- grouped block-scaled FP8 GEMM for MoE experts with few tokens each.
//
// What it computes (source pages: page 1 second paragraph -- FP8 GEMMs with the
// dequantization folded into the FP32 accumulation; page 4 first paragraph -- promotion of
// the partial sums every 128 elements of K; page 2 "9 Amazing Deepseek Hacks" -- during
// decoding the experts' GEMMs are bound by memory access, not by arithmetic):
//
//   C[m, n] = sum_kb ( sum_{k in slice kb} x[m,k] w_g[n,k] ) * sX[kb][m] * sW_g[n/128][kb]
//
// for every token row m of expert g (rows offsets[g] .. offsets[g+1]), the same result as
// the row-tiled grouped GEMM.
//
// Design (B300, persistent, one CTA per SM).  With a few tokens per expert the row-tiled
// form spends a full 128- or 256-row MMA on each expert's handful of tokens, and the
// tensor cores, not the weight stream, set the pace.  Here the roles of the operands are
// swapped: a work item is one 128-row block of one expert's weight (the MMA's M = 128
// operand, streamed from HBM once) against that expert's tokens (the MMA's N operand,
// N = the token count rounded up to 16, at most 256 per item), so the tensor-core time of
// an item follows its token count.  TMEM then holds lanes = weight rows (output features),
// columns = tokens.
// The weights stream from HBM through a deep ring of their own (seven 16 KB slices in
// flight per SM), the tokens' codes -- read by every weight block of the expert, so mostly
// L2 hits -- through a shorter one.
// Roles in each CTA:
//   warp 0      TMA producer of the weight ring: the 128 x 128 weight tile of each slice;
//   warp 3      TMA producer of the token ring: the tokens' codes of each slice in 32-row
//               boxes (only as many boxes as the item has tokens);
//   warp 1      MMA issuer: four M128 x N x K32 MMAs per slice into one of two 256-column
//               TMEM buffers;
//   warp 2      scale loader: the product sX[kb][m] * sW[g][n/128][kb] per token column,
//               written to a shared-memory ring;
//   warps 4-11  promotion: tcgen05.ld of the item's valid 32-column chunks (shared evenly
//               by the two warps of each lane quarter, two loads in flight), one FMA per
//               element into FP32 registers, then direct stores of C (each warp writes 32
//               consecutive features of a token row per instruction).
// With fused activation quantization (page 2 "9 Amazing Deepseek Hacks", third
// paragraph after the title: the pages wish the FP8 cast to happen on the way into the
// GEMM), the launch runs in two phases.  Phase 1, all warps: the experts' BF16 token rows
// are quantized 1x128 (the arithmetic of the standalone quantizer, bit for bit) into a
// caller-provided workspace, 32 rows at a time; each finished block is published by a
// fence and an atomic add to a per-expert ready count.  Phase 2 is the GEMM above, whose
// token producer and scale loader first wait (bounded) until their expert's count is
// complete.  Every CTA finishes its phase-1 share before it waits on anything, and the
// launch is cooperative (all CTAs resident), so every wait is for work that is running.
// Every wait is bounded; on expiry the CTA records a timeout in the status word, drains
// its copies and MMAs, frees TMEM and exits.
#include "mpq_internal.h"
#include "mpq_device.cuh"
#include "quant_device.cuh"

namespace mpq {
namespace {

constexpr int DK = 128;                          // K per promotion slice
constexpr int WSTAGES = 7;                       // weight ring
constexpr int XSTAGES = 3;                       // token ring
constexpr int DTOK = 256;                        // tokens per work item at most (MMA N)
constexpr int kXBoxRows = 32;                    // token rows per TMA box
constexpr uint32_t DW_BYTES = 128 * DK;          // weight tile, 16 KB
constexpr uint32_t DX_BYTES = DTOK * DK;         // token tile, up to 32 KB
constexpr int DSSLOTS = 4;                       // scale ring depth
constexpr int kDThreads = 384;
constexpr uint32_t DTMEM_COLS = 512;             // two 256-column buffers
constexpr int kDMaxGroups = 1024;

// DONE[i % WSTAGES]: the MMAs of slice i have completed -- its weight and token stages may
// be refilled and its partial may be promoted.  One commit per slice serves all three
// (every tcgen05.commit costs the tensor pipe a bubble).  A waiter for slice i waits on
// DONE[i % WSTAGES] with parity (i / WSTAGES) & 1; no barrier can run two phases ahead of
// a waiter, because its next phase needs that waiter's own progress first.
constexpr int BAR_WFULL = 0;
constexpr int BAR_XFULL = BAR_WFULL + WSTAGES;
constexpr int BAR_DONE = BAR_XFULL + XSTAGES;
constexpr int BAR_TEMPTY = BAR_DONE + WSTAGES;
constexpr int BAR_SFULL = BAR_TEMPTY + 2;
constexpr int BAR_SEMPTY = BAR_SFULL + DSSLOTS;
constexpr int BAR_DRAIN = BAR_SEMPTY + DSSLOTS;
constexpr int NBARS = BAR_DRAIN + 1;

constexpr size_t kDSmem = 1024 + WSTAGES * DW_BYTES + XSTAGES * DX_BYTES + DSSLOTS * DTOK * sizeof(float) +
                          NBARS * 8 + 16 +
                          (kDMaxGroups + 1) * 2 * sizeof(int) + 16;

struct Item {
    int g;          // expert
    int row0;       // first token row of the item
    int ntok;       // tokens in the item, 1 .. 256
    int nb;         // 128-row block of the expert's weight
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > timeout_ns)
            return false;
    return true;
}

template <bool OUT_F32, bool FUSE>
__global__ void __launch_bounds__(kDThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const GemmArgs p,
                  const FuseArgs f)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *base = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *wring = base;                                           // [WSTAGES][16 KB]
    uint8_t *xring = wring + WSTAGES * DW_BYTES;                     // [XSTAGES][32 KB]
    float *ssc = reinterpret_cast<float *>(xring + XSTAGES * DX_BYTES);       // [DSSLOTS][256]
    uint64_t *bars = reinterpret_cast<uint64_t *>(ssc + DSSLOTS * DTOK);
    uint32_t *misc = reinterpret_cast<uint32_t *>(bars + NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    int *goff = reinterpret_cast<int *>(misc + 4);                   // clamped offsets [G+1]
    int *gitem = goff + kDMaxGroups + 1;                             // first item of expert [G+1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };
    const int64_t M = p.M;
    const int KB = static_cast<int>(p.K / DK);
    const int NB = static_cast<int>(p.N / 128);
    const int G = p.G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WSTAGES; ++s) {
            mbar_init(bar(BAR_WFULL + s), 1);
            mbar_init(bar(BAR_DONE + s), 1);
        }
        for (int s = 0; s < XSTAGES; ++s)
            mbar_init(bar(BAR_XFULL + s), 1);
        for (int b = 0; b < 2; ++b)
            mbar_init(bar(BAR_TEMPTY + b), 8);
        for (int j = 0; j < DSSLOTS; ++j) {
            mbar_init(bar(BAR_SFULL + j), 32);
            mbar_init(bar(BAR_SEMPTY + j), 8);
        }
        mbar_init(bar(BAR_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), DTMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 2) {
        // Expert schedule: offsets clamped into [0, M] and made monotone (running max); an
        // expert with t tokens contributes ceil(t / 256) token chunks x NB weight blocks.
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
            cnt += (goff[g + 1] - goff[g] + DTOK - 1) / DTOK;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += v;
        }
        int ex = incl - cnt;
        for (int g = e0; g < e1; ++g) {
            gitem[g] = ex * NB;
            ex += (goff[g + 1] - goff[g] + DTOK - 1) / DTOK;
        }
        if (lane == 31)
            gitem[G] = incl * NB;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc[0];
    const int T = gitem[G];

    if (FUSE)
        quantize_rows_phase(goff, G, M, KB, p.K, f);   // phase 1

    // Item t: expert g (last with gitem[g] <= t), then weight block fastest so that
    // neighbouring CTAs share the expert's tokens in L2 while streaming different weights.
    auto item_of = [&](int t) -> Item {
        int lo = 0, hi = G - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (gitem[mid] <= t) lo = mid; else hi = mid - 1;
        }
        Item it;
        it.g = lo;
        const int local = t - gitem[lo];
        const int chunk = local / NB;
        it.nb = local - chunk * NB;
        it.row0 = goff[lo] + chunk * DTOK;
        const int rest = goff[lo + 1] - it.row0;
        it.ntok = rest < DTOK ? rest : DTOK;
        return it;
    };

    WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
        if (warp == 0 && lane == 0) {
            // ---------------------------------------------------------- weight producer
            uint32_t it = 0;
            for (int t = blockIdx.x; t < T; t += gridDim.x) {
                const Item ti = item_of(t);
                const int wrow = ti.g * static_cast<int>(p.N) + ti.nb * 128;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t s = it % WSTAGES, ph = (it / WSTAGES) & 1;
                    if (!mbar_wait(bar(BAR_DONE + s), ph ^ 1, ctl, 0x0500 | s))   // slice it - WSTAGES
                        goto wproducer_done;
                    const uint32_t full = bar(BAR_WFULL + s);
                    mbar_arrive_expect_tx(full, DW_BYTES);
                    tma_load_2d(smem_u32(wring + s * DW_BYTES), &tmW, full, kb * DK, wrow);
                }
            }
        wproducer_done:
            for (uint32_t j = it > WSTAGES ? it - WSTAGES : 0; j < it; ++j)
                drain_wait(bar(BAR_WFULL + j % WSTAGES), (j / WSTAGES) & 1, p.timeout_ns);
        } else if (warp == 3 && lane == 0) {
            // ---------------------------------------------------------- token producer
            uint32_t it = 0;
            for (int t = blockIdx.x; t < T; t += gridDim.x) {
                const Item ti = item_of(t);
                const int nbox = (ti.ntok + kXBoxRows - 1) / kXBoxRows;
                if (FUSE) {   // the expert's token codes are complete (phase 1 of all CTAs)
                    if (!wait_count(f.ready + ti.g, goff[ti.g + 1] - goff[ti.g], ctl, 0x0590))
                        goto xproducer_done;
                    fence_proxy_async_global();
                }
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t s = it % XSTAGES;
                    if (it >= static_cast<uint32_t>(XSTAGES)) {   // slice it - XSTAGES is done
                        const uint32_t prev = it - XSTAGES;
                        if (!mbar_wait(bar(BAR_DONE + prev % WSTAGES), (prev / WSTAGES) & 1, ctl, 0x0580 | s))
                            goto xproducer_done;
                    }
                    const uint32_t full = bar(BAR_XFULL + s);
                    const uint32_t dst = smem_u32(xring + s * DX_BYTES);
                    mbar_arrive_expect_tx(full, nbox * (kXBoxRows * DK));
                    for (int b = 0; b < nbox; ++b)
                        tma_load_2d(dst + b * (kXBoxRows * DK), &tmX, full, kb * DK, ti.row0 + b * kXBoxRows);
                }
            }
        xproducer_done:
            for (uint32_t j = it > XSTAGES ? it - XSTAGES : 0; j < it; ++j)
                drain_wait(bar(BAR_XFULL + j % XSTAGES), (j / XSTAGES) & 1, p.timeout_ns);
        } else if (warp == 1 && lane == 0) {
            // ---------------------------------------------------------- MMA issuer
            uint32_t it = 0;
            for (int t = blockIdx.x; t < T; t += gridDim.x) {
                const Item ti = item_of(t);
                const int nmma = (ti.ntok + 15) & ~15;
                const uint32_t idesc = idesc_e4m3_f32(128, nmma);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t sw = it % WSTAGES, wph = (it / WSTAGES) & 1;
                    const uint32_t sx = it % XSTAGES, xph = (it / XSTAGES) & 1;
                    const uint32_t buf = it & 1, tph = (it >> 1) & 1;
                    if (!mbar_wait(bar(BAR_TEMPTY + buf), tph ^ 1, ctl, 0x0600 | buf))
                        goto mma_done;
                    if (!mbar_wait(bar(BAR_WFULL + sw), wph, ctl, 0x0610 | sw))
                        goto mma_done;
                    if (!mbar_wait(bar(BAR_XFULL + sx), xph, ctl, 0x0620 | sx))
                        goto mma_done;
                    tc_fence_after();
                    const uint32_t w0 = smem_u32(wring + sw * DW_BYTES);
                    const uint32_t x0 = smem_u32(xring + sx * DX_BYTES);
                    const uint32_t d = tmem_base + buf * 256;
#pragma unroll
                    for (int k = 0; k < DK / 32; ++k)
                        umma_e4m3(d, sdesc_kmajor_sw128(w0 + k * 32), sdesc_kmajor_sw128(x0 + k * 32), idesc,
                                  k > 0 ? 1u : 0u);
                    umma_commit(bar(BAR_DONE + sw));
                }
            }
        mma_done:
            umma_commit(bar(BAR_DRAIN));
            drain_wait(bar(BAR_DRAIN), 0, p.timeout_ns);
        } else if (warp == 2) {
            // ---------------------------------------------------------- scale loader
            // Lane l handles token columns l + 32 i.  The global loads of the next SPF slices
            // are kept in flight in registers (the loop is unrolled by SPF so that the
            // register arrays keep static indices), so the slices do not each pay a memory
            // latency in turn.
            constexpr int SPF = 4;
            uint32_t it = 0;
            for (int t = blockIdx.x; t < T; t += gridDim.x) {
                const Item ti = item_of(t);
                const float *sw = p.sB + static_cast<int64_t>(ti.g) * p.sb_group_stride +
                                  static_cast<int64_t>(ti.nb) * p.ldsb;
                if (FUSE && !wait_count(f.ready + ti.g, goff[ti.g + 1] - goff[ti.g], ctl, 0x0790))
                    goto scale_done;
                float px[SPF][DTOK / 32], pw[SPF];
                auto fetch = [&](int kb, float (&x)[DTOK / 32], float &w) {
                    if (kb < KB) {
                        w = sw[kb];
                        const float *sx = p.sA + static_cast<int64_t>(kb) * p.ldsa + ti.row0;
#pragma unroll
                        for (int i = 0; i < DTOK / 32; ++i) {
                            const int c = lane + 32 * i;
                            x[i] = c < ti.ntok ? sx[c] : 0.0f;
                        }
                    }
                };
#pragma unroll
                for (int d = 0; d < SPF; ++d)
                    fetch(d, px[d], pw[d]);
                for (int kb0 = 0; kb0 < KB; kb0 += SPF) {
#pragma unroll
                    for (int d = 0; d < SPF; ++d) {
                        const int kb = kb0 + d;
                        if (kb < KB) {
                            const uint32_t j = it % DSSLOTS, ph = (it / DSSLOTS) & 1;
                            if (!mbar_wait(bar(BAR_SEMPTY + j), ph ^ 1, ctl, 0x0700 | j))
                                goto scale_done;
#pragma unroll
                            for (int i = 0; i < DTOK / 32; ++i)
                                ssc[j * DTOK + lane + 32 * i] = __fmul_rn(px[d][i], pw[d]);
                            mbar_arrive(bar(BAR_SFULL + j));   // each lane releases its own stores
                            ++it;
                            fetch(kb + SPF, px[d], pw[d]);
                        }
                    }
                }
            }
        scale_done:;
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 224;" ::: "memory");
        // -------------------------------------------------------------- promotion
        // Warp (quad, half) owns TMEM lanes 32 quad .. +31 (weight rows) and the 32-column
        // token chunks 2 i + half, i = 0..3, so that the two warps of a quad share the
        // work evenly whatever the token count; two chunk loads are kept in flight.
        const int ew = warp - 4, quad = warp & 3, half = ew >> 2;
        const uint32_t tm_lane = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
            const Item ti = item_of(t);
            const int nct = (ti.ntok + 31) >> 5;           // chunks holding tokens, 1..8
            const int nmine = (nct - half + 1) >> 1;        // of them this warp's, 0..4
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i)
                acc[i] = 0.0f;
            auto fma_chunk = [&](int i, const uint32_t (&v)[32], const float *sc) {
                const float *s = sc + 32 * (2 * i + half);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 s4 = *reinterpret_cast<const float4 *>(s + 4 * q);
                    acc[32 * i + 4 * q + 0] = __fmaf_rn(__uint_as_float(v[4 * q + 0]), s4.x, acc[32 * i + 4 * q + 0]);
                    acc[32 * i + 4 * q + 1] = __fmaf_rn(__uint_as_float(v[4 * q + 1]), s4.y, acc[32 * i + 4 * q + 1]);
                    acc[32 * i + 4 * q + 2] = __fmaf_rn(__uint_as_float(v[4 * q + 2]), s4.z, acc[32 * i + 4 * q + 2]);
                    acc[32 * i + 4 * q + 3] = __fmaf_rn(__uint_as_float(v[4 * q + 3]), s4.w, acc[32 * i + 4 * q + 3]);
                }
            };
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const uint32_t j = it % DSSLOTS, sph = (it / DSSLOTS) & 1;
                const uint32_t buf = it & 1;
                const uint32_t ds = it % WSTAGES, dph = (it / WSTAGES) & 1;
                if (!mbar_wait(bar(BAR_SFULL + j), sph, ctl, 0x0800 | j) ||
                    !mbar_wait(bar(BAR_DONE + ds), dph, ctl, 0x0810 | ds)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float *sc = ssc + j * DTOK;
                const uint32_t taddr = tmem_base + tm_lane + buf * 256 + 32 * half;   // chunk i at + 64 i
                uint32_t va[32], vb[32];
                if (nmine > 0)
                    MPQ_TMEM_LD32(taddr, va);
                if (nmine > 1)
                    MPQ_TMEM_LD32(taddr + 64, vb);
                if (nmine > 0) {
                    MPQ_TMEM_WAIT_LD32(va);
                    fma_chunk(0, va, sc);
                }
                if (nmine > 2)
                    MPQ_TMEM_LD32(taddr + 128, va);
                if (nmine > 1) {
                    MPQ_TMEM_WAIT_LD32(vb);
                    fma_chunk(1, vb, sc);
                }
                if (nmine > 3)
                    MPQ_TMEM_LD32(taddr + 192, vb);
                if (nmine > 2) {
                    MPQ_TMEM_WAIT_LD32(va);
                    fma_chunk(2, va, sc);
                }
                if (nmine > 3) {
                    MPQ_TMEM_WAIT_LD32(vb);
                    fma_chunk(3, vb, sc);
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
            // C[row0 + col, n] for this lane's feature n and the item's valid token columns.
            const int64_t n = static_cast<int64_t>(ti.nb) * 128 + quad * 32 + lane;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (i < nmine) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int col = 32 * (2 * i + half) + q;
                        if (col < ti.ntok) {
                            const int64_t m = ti.row0 + col;
                            if (OUT_F32)
                                static_cast<float *>(p.C)[m * p.ldc + n] = acc[32 * i + q];
                            else
                                static_cast<__nv_bfloat16 *>(p.C)[m * p.ldc + n] = __float2bfloat16_rn(acc[32 * i + q]);
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, DTMEM_COLS);
    }
}

} // namespace

int decode_x_box_rows() { return kXBoxRows; }

cudaError_t launch_decode(const CUtensorMap &tmX, const CUtensorMap &tmW, const GemmArgs &a, bool out_fp32,
                          const FuseArgs *fuse, int num_sms, cudaStream_t st)
{
    if (a.G > kDMaxGroups)
        return cudaErrorInvalidValue;
    // upper bound on the items: every expert may add one partial token chunk
    const int64_t items = ((a.M + DTOK - 1) / DTOK + a.G) * (a.N / 128);
    if (items <= 0)
        return cudaSuccess;
    // the fused form quantizes on every SM first, so it always takes one CTA per SM
    const int grid = fuse != nullptr ? num_sms : static_cast<int>(items < num_sms ? items : num_sms);
    const int ki = (out_fp32 ? 1 : 0) + (fuse != nullptr ? 2 : 0);
    void (*kern)(CUtensorMap, CUtensorMap, GemmArgs, FuseArgs) =
        ki == 0 ? decode_kernel<false, false> : ki == 1 ? decode_kernel<true, false>
                : ki == 2 ? decode_kernel<false, true> : decode_kernel<true, true>;
    static std::atomic<uint64_t> configured[4];   // per variant: devices already set up
    if (cudaError_t e = ensure_max_dyn_smem(kern, kDSmem, configured[ki]); e != cudaSuccess)
        return e;
    const FuseArgs none{};
    if (fuse == nullptr) {
        kern<<<grid, kDThreads, kDSmem, st>>>(tmX, tmW, a, none);
        return cudaGetLastError();
    }
    // Phase 2 waits on phase-1 work of every CTA: a cooperative launch guarantees that all
    // CTAs are resident at once (or the launch fails).
    cudaError_t e = cudaMemsetAsync(fuse->ready, 0, sizeof(int) * static_cast<size_t>(a.G), st);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kDThreads, 1, 1);
    cfg.dynamicSmemBytes = kDSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmX, tmW, a, *fuse);
}

} // namespace mpq

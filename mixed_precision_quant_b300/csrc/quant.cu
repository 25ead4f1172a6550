// quant.cu -- online fine-grained FP8 (E4M3) quantizers.
//
// Method (source pages: page 1 second paragraph -- the scaling factor is derived from
// the online max-abs value and the activation or weight is quantized online into FP8;
// page 3 first paragraph -- the max-abs value is scaled to the largest FP8 value;
// page 2 "9 Amazing Deepseek Hacks" last paragraph -- groups of 128 activation values,
// and the backward pass re-quantizes into 128x1 tiles; page 4 second paragraph --
// integral power-of-2 scaling factors):
//   * 1x128 row groups (one scale per row per 128 columns),
//   * 128x1 column groups (one scale per column per 128 rows), written transposed,
//   * 128x128 blocks (one scale per block), optionally also written transposed.
//
// Design.  The three BF16 kernels are persistent and warp-specialised around tiles of
// 128 rows x 128 columns of BF16 (32 KB) in a four-slot ring:
//   * one producer lane loads a tile as two 128-row x 64-column TMA boxes with 128-byte
//     swizzle (completion counted on mbarriers);
//   * the two consumer warpgroups take alternate tiles of the CTA, each with its own
//     staging tiles and barrier; a thread owns one row group (rows, blocks: eight warps)
//     or half a row group and half a column group (dual: sixteen warps, the halves'
//     max-abs values meeting in one shuffle), reads its values with 16-byte (or, down a
//     column, transposing 8x8 matrix) shared loads, reduces the max-abs, derives the scale and converts
//     with the exact arithmetic of quant_device.cuh;
//   * codes are written into 128-byte-swizzled staging tiles and leave with TMA
//     bulk-tensor stores (coalesced, clipped at the tensor bounds).
// The re-quantization kernel streams FP8 code tiles the same way (below).
// Every wait is bounded.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "mpq_internal.h"
#include "mpq_device.cuh"
#include "quant_device.cuh"

namespace mpq {
namespace {

constexpr int kConsumers = 8;                       // consumer warps per CTA
constexpr int kQThreads = 32 * (kConsumers + 1);    // + one producer warp
constexpr uint32_t kBox = 128 * 128;                // one 128-row x 128-byte box (16 KB)

__device__ __forceinline__ uint4 lds_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts_u16(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(static_cast<uint16_t>(v)) : "memory");
}

// Four 8x8 matrices of 16-bit values, transposed on the way in: lane L names row L % 8 of
// matrix L / 8 (16 bytes); lane t receives in v[m] the two values of column t / 4 of
// matrix m at rows 2 (t % 4) (low half) and 2 (t % 4) + 1 (high half).
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t *v)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "r"(addr));
}

__device__ __forceinline__ void sts_v4(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Byte offset of 16-byte chunk j of row r in a 128-row box with 128-byte swizzle (the
// layout TMA writes and reads with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint32_t sw128(int r, int j) { return r * 128 + ((j ^ (r & 7)) << 4); }

// Bounded barrier among the four warps of one warpgroup (the mbarrier counts 4 warps):
// lane 0 of each warp arrives after the warp's own writes, every lane waits.
__device__ __forceinline__ bool wg_sync(uint32_t bar, uint32_t &k, const WaitCtl &ctl, int tag)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        mbar_arrive(bar);
    const bool ok = mbar_wait(bar, k & 1, ctl, tag);
    ++k;
    return ok;
}

// Row r (0..127) of the 128 x 128 BF16 tile at `tile` (two 128 x 64 boxes): its 128 values
// as 64 BF16x2 words, memory order.
__device__ __forceinline__ void load_row(uint32_t tile, int r, uint32_t (&w)[64])
{
#pragma unroll
    for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 v = lds_v4(tile + ch * kBox + sw128(r, j));
            w[ch * 32 + j * 4 + 0] = v.x;
            w[ch * 32 + j * 4 + 1] = v.y;
            w[ch * 32 + j * 4 + 2] = v.z;
            w[ch * 32 + j * 4 + 3] = v.w;
        }
}

// 128 values (64 words) -> 8 code chunks written to row `r` of a swizzled staging box.
__device__ __forceinline__ void write_codes(uint32_t box, int r, const uint32_t (&w)[64], const GroupScale &g)
{
#pragma unroll
    for (int q = 0; q < 8; ++q)
        sts_v4(box + sw128(r, q), codes16(&w[q * 8], g));
}

// Producer of the 128-row kernels: one lane streams tile `item` (128-row block rb, 128-column
// block cb) into a ring of `stages` 32 KB slots as two 128 x 64 boxes (rows past the tensor
// read as zero), then waits (bounded) until its last loads have landed.
__device__ __forceinline__ void produce128(uint32_t stage, uint32_t bars, int stages, const CUtensorMap *tm,
                                           int64_t items, int64_t ncb, const WaitCtl &ctl, uint64_t timeout_ns,
                                           int tag)
{
    uint32_t it = 0;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
        const uint32_t st = it % stages, ph = (it / stages) & 1;
        if (!mbar_wait(bars + 8 * (stages + st), ph ^ 1, ctl, tag | st))
            break;
        const int64_t rb = item / ncb, cb = item - rb * ncb;
        mbar_arrive_expect_tx(bars + 8 * st, 2 * kBox);
#pragma unroll
        for (int b = 0; b < 2; ++b)
            tma_load_2d(stage + st * 2 * kBox + b * kBox, tm, bars + 8 * st, static_cast<int32_t>(cb * 128 + b * 64),
                        static_cast<int32_t>(rb * 128));
    }
    for (uint32_t j = it > static_cast<uint32_t>(stages) ? it - stages : 0; j < it; ++j) {   // no load in flight
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bars + 8 * (j % stages), (j / stages) & 1))
            if (globaltimer_ns() - t0 > timeout_ns)
                break;
    }
}

// ------------------------------------------------------------------ 1x128 rows
//
// One 128-row x 128-column tile per ring slot (four slots); warpgroup h (warps 8h .. 8h+7,
// threads 256h .. +255) takes the CTA's tiles h, h+2, ..., with its own barrier and two
// staging boxes used in turn, so the two warpgroups run independently and a tile's store
// drains while the next tile is converted.  Thread u of a warpgroup owns half a row group:
// row u/2, columns 64 (u%2) .. +63 (one of the tile's two 128 x 64 boxes), and the two
// halves' max-abs values meet in one shuffle -- sixteen consumer warps where one thread per
// row (64 words of data) left room for eight (131072 x 7168: 6.08 against 5.95 TB/s; small
// tensors such as 4096 x 7168, twelve tiles per SM, are set by the first load and the last
// store rather than by the conversion).
constexpr int QR_STAGES = 4;
static_assert(QR_STAGES % 2 == 0, "a stage must belong to one of the two warpgroups");
constexpr int kRowsConsumers = 16;
constexpr int kRowsThreads = 32 * (kRowsConsumers + 1);
constexpr size_t kRowsSmem = 1024 + QR_STAGES * 2 * kBox + 4 * kBox + (2 * QR_STAGES + 2) * 8 + 16;

template <bool POW2>
__global__ void __launch_bounds__(kRowsThreads, 1)
    quant_rows_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmq,
                      const QuantArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base0 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (base0 & 1023u)) & 1023u;
    const uint32_t stage = base0 + pad, out_rows = stage + QR_STAGES * 2 * kBox;
    const uint32_t bars = out_rows + 4 * kBox;          // full[S], empty[S], warpgroup[2]
    volatile int *abort_flag =
        reinterpret_cast<volatile int *>(smem_raw + pad + QR_STAGES * 2 * kBox + 4 * kBox + (2 * QR_STAGES + 2) * 8);
    if (threadIdx.x == 0) {
        for (int i = 0; i < QR_STAGES; ++i) {
            mbar_init(bars + 8 * i, 1);
            mbar_init(bars + 8 * (QR_STAGES + i), 8);  // the eight warps of one warpgroup
        }
        mbar_init(bars + 8 * (2 * QR_STAGES), 8);
        mbar_init(bars + 8 * (2 * QR_STAGES + 1), 8);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
    const int64_t ncb = p.cols / 128, items = ((p.rows + 127) / 128) * ncb;
    const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    if (warp == kRowsConsumers) {
        if (lane == 0)
            produce128(stage, bars, QR_STAGES, &tmx, items, ncb, ctl, p.timeout_ns, 0x1100);
        return;
    }
    const int h = t >> 8, u = t & 255;
    const int rr = u >> 1, sub = u & 1;                 // row and column half
    const uint32_t wgbar = bars + 8 * (2 * QR_STAGES + h);
    const bool elected = u == 0;
    uint32_t cph = 0;
    uint32_t it = h;   // this warpgroup's tiles are the CTA's tiles h, h + 2, ...
    for (int64_t item = blockIdx.x + h * static_cast<int64_t>(gridDim.x); item < items;
         item += 2 * static_cast<int64_t>(gridDim.x), it += 2) {
        const uint32_t st = it % QR_STAGES, ph = (it / QR_STAGES) & 1;
        if (!mbar_wait(bars + 8 * st, ph, ctl, 0x1200 | st))
            break;
        const int64_t rb = item / ncb, kb = item - rb * ncb;
        const uint32_t out = out_rows + (2 * h + ((it >> 1) & 1)) * kBox;   // this tile's staging box
        uint32_t w[32];
        const uint32_t box = stage + st * 2 * kBox + sub * kBox;   // columns 64 sub .. +63
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 v = lds_v4(box + sw128(rr, j));
            w[4 * j + 0] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bars + 8 * (QR_STAGES + st));
        float a = amax_words(w);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        const GroupScale g = make_group_scale(a, POW2);
        const int64_t r = rb * 128 + rr;
        if (sub == 0 && r < p.rows)
            p.s[kb * p.lds + r] = g.s;
        if (elected)
            bulk_wait_read1();                 // the box's previous store has left it
        if (!wg_sync(wgbar, cph, ctl, 0x1210))
            break;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            sts_v4(out + sw128(rr, sub * 4 + q), codes16(&w[q * 8], g));
        fence_proxy_async_smem();
        if (!wg_sync(wgbar, cph, ctl, 0x1211))
            break;
        if (elected) {
            tma_store_2d(&tmq, out, static_cast<int32_t>(kb * 128), static_cast<int32_t>(rb * 128));
            bulk_commit();
        }
    }
    if (elected)
        bulk_wait0();
}

// --------------------------------------------------- fused 1x128 + 128x1 (dual)
//
// Row groups as in the row kernel, plus the 128x1 column groups written transposed (one
// read of the tile for both).  One thread per group would need 64 words of data in
// registers, which leaves room for eight consumer warps only, too few to hide the
// latencies of a pass (shared loads, the max-abs tree, the scale's division).  Here each
// thread owns half a group -- 64 values -- and the two halves' max-abs values meet in one
// shuffle, so sixteen consumer warps fit.  Tiles are 128 rows x 128 columns (32 KB of
// BF16, two 128 x 64 TMA boxes) in a four-stage ring; warpgroup h (warps 8h .. 8h+7) takes
// the CTA's tiles h, h+2, h+4, ..., so the two warpgroups run independently.  The stage count
// is even so that every stage belongs to one warpgroup: with an odd count a warpgroup could
// wait on a stage two phases ahead of its barrier, and a parity wait cannot tell those apart.
// Each warpgroup has its own barrier, one row-code staging tile and two transposed-code
// staging tiles used in turn; the row codes' store is committed as its own group ahead of
// the transposed codes', so a tile waits only for the previous tile's row store while the
// transposed store drains (8192 x 7168 +5% over one staging set).  Within a warpgroup
// thread u (0..255) holds
//   row pass:    row u/2, columns 64 (u%2) .. +63 (16-byte shared loads);
//   column pass: lane t of warp wl, for the two columns 16 wl + 8 b + t/4 (b = 0, 1), the
//                rows 8 rb + 2 (t%4), +1 (rb = 0..15) -- transposing 8x8 matrix loads
//                (ldmatrix .trans) deliver each as one BF16 pair, 128 bytes per shared
//                wavefront, so the four lanes of a column hold its 128 values and combine
//                max-abs values in two shuffles; codes leave as 2-byte shared stores.
constexpr int QD_STAGES = 4;
static_assert(QD_STAGES % 2 == 0, "a stage must belong to one of the two warpgroups");
constexpr uint32_t kDualTile = 2 * kBox;          // 128 x 128 BF16
constexpr int kDualConsumers = 16;
constexpr int kDualThreads = 32 * (kDualConsumers + 1);
constexpr size_t kDualSmem = 1024 + QD_STAGES * kDualTile + 6 * kBox + (2 * QD_STAGES + 2) * 8 + 16;

template <bool POW2, bool ROWS>
__global__ void __launch_bounds__(kDualThreads, 1)
    quant_dual16_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmq,
                        const __grid_constant__ CUtensorMap tmqT, const QuantArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base0 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (base0 & 1023u)) & 1023u;
    const uint32_t stage = base0 + pad;
    const uint32_t out_rows = stage + QD_STAGES * kDualTile, out_cols = out_rows + 2 * kBox;
    const uint32_t bars = out_cols + 4 * kBox;        // full[S], empty[S], warpgroup[2]
    volatile int *abort_flag =
        reinterpret_cast<volatile int *>(smem_raw + pad + QD_STAGES * kDualTile + 6 * kBox + (2 * QD_STAGES + 2) * 8);
    if (threadIdx.x == 0) {
        for (int i = 0; i < QD_STAGES; ++i) {
            mbar_init(bars + 8 * i, 1);
            mbar_init(bars + 8 * (QD_STAGES + i), 8);   // the eight warps of one warpgroup
        }
        mbar_init(bars + 8 * (2 * QD_STAGES), 8);
        mbar_init(bars + 8 * (2 * QD_STAGES + 1), 8);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
    const int64_t ncb = p.cols / 128, items = (p.rows / 128) * ncb;   // rows is a multiple of 128
    const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    if (warp == kDualConsumers) {   // producer: one 128-row tile as two 128 x 64 boxes
        if (lane == 0)
            produce128(stage, bars, QD_STAGES, &tmx, items, ncb, ctl, p.timeout_ns, 0x1400);
        return;
    }
    const int h = t >> 8, u = t & 255;
    const int g2 = u >> 1, sub = u & 1;                    // row pass: row and half
    const int wl = u >> 5;                                  // warp within the warpgroup
    const uint32_t wgbar = bars + 8 * (2 * QD_STAGES + h);
    const bool elected = u == 0;
    uint32_t cph = 0;
    uint32_t it = h;   // this warpgroup's tiles are the CTA's tiles h, h + 2, ...
    for (int64_t item = blockIdx.x + h * static_cast<int64_t>(gridDim.x); item < items;
         item += 2 * static_cast<int64_t>(gridDim.x), it += 2) {
        const uint32_t st = it % QD_STAGES, ph = (it / QD_STAGES) & 1;
        if (!mbar_wait(bars + 8 * st, ph, ctl, 0x1500 | st))
            break;
        const int64_t rb = item / ncb, cb = item - rb * ncb;
        const uint32_t tile = stage + st * kDualTile;
        const int64_t y = rb * 128;                         // first row of the tile
        const uint32_t sb = (it >> 1) & 1;                  // this warpgroup's staging set
        const uint32_t out_r = out_rows + h * kBox, out_c = out_cols + (2 * h + sb) * kBox;
        if (elected)
            bulk_wait_read1();                             // all but the newest group (the last transposed store) are read
        if (!wg_sync(wgbar, cph, ctl, 0x1510))
            break;
        if (ROWS) {
            uint32_t w[32];
            const uint32_t box = tile + sub * kBox;          // columns 64 sub .. +63
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 v = lds_v4(box + sw128(g2, j));
                w[4 * j + 0] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
            }
            float a = amax_words(w);
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            const GroupScale g = make_group_scale(a, POW2);
            if (sub == 0)
                p.s[cb * p.lds + y + g2] = g.s;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                sts_v4(out_r + sw128(g2, sub * 4 + q), codes16(&w[q * 8], g));
        }
        // Column pass: warp wl of the warpgroup owns columns 16 wl .. +15 as two 8-column
        // blocks; transposing 8x8 loads give lane t, for column 16 wl + 8 b + t / 4, the BF16
        // pair of rows 8 rb + 2 (t % 4), +1 in wc[b][rb] (rb = 0..15), so the four lanes
        // t / 4 = const hold the column's 128 values and meet in two shuffles.
        uint32_t wc[2][16];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int cbk = 2 * wl + b;                      // 8-column block, 0..15
            const uint32_t box = tile + (cbk >> 3) * kBox;
#pragma unroll
            for (int i = 0; i < 4; ++i)                      // row blocks 4i .. 4i+3: rows 32i + lane
                ldsm_x4_trans(box + sw128(32 * i + lane, cbk & 7), &wc[b][4 * i]);
        }
        float ac[2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            ac[b] = amax_words(wc[b]);
            ac[b] = fmaxf(ac[b], __shfl_xor_sync(0xffffffffu, ac[b], 1));
            ac[b] = fmaxf(ac[b], __shfl_xor_sync(0xffffffffu, ac[b], 2));
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bars + 8 * (QD_STAGES + st));      // this warp has read the tile
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            const int c = 16 * wl + 8 * b + (lane >> 2), k2 = (lane & 3) * 2;
            const GroupScale g = make_group_scale(ac[b], POW2);
            if (k2 == 0)
                p.sT[(y / 128) * p.ldsT + cb * 128 + c] = g.s;
            uint32_t o[8];                                   // o[j]: rows 16j + k2, +1 | 16j + 8 + k2, +1
            codes_words<16>(wc[b], g, o);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                sts_u16(out_c + sw128(c, j) + k2, o[j]);
                sts_u16(out_c + sw128(c, j) + 8 + k2, o[j] >> 16);
            }
        }
        fence_proxy_async_smem();
        if (!wg_sync(wgbar, cph, ctl, 0x1511))
            break;
        if (elected) {
            if (ROWS) {
                tma_store_2d(&tmq, out_r, static_cast<int32_t>(cb * 128), static_cast<int32_t>(y));
                bulk_commit();
            }
            tma_store_2d(&tmqT, out_c, static_cast<int32_t>(y), static_cast<int32_t>(cb * 128));
            bulk_commit();
        }
    }
    if (elected)
        bulk_wait0();
}

// ------------------------------------------------------------------ 128x128 blocks
//
// One 128 x 128 block per tile (two 128 x 64 TMA boxes, 32 KB) in a four-stage ring (even:
// each stage belongs to one warpgroup); warpgroup h (warps 4h .. 4h+3) takes the CTA's tiles
// h, h+2, ..., so the two warpgroups run independently.  Staging per warpgroup: two row-code
// boxes used in turn, or, when the transposed codes are written too, one row-code box and
// two transposed-code boxes, the row store committed as its own group first (a tile then
// waits only for the previous tile's row store; 2048 x 7168 +9%).
// Each thread owns one row of the block; the block max comes from warp shuffles and a
// 4-warp shared reduction.  Transposed codes are gathered column-wise from the row-code
// staging box.
template <bool TRANS>
__host__ __device__ constexpr int qb_stages() { return 4; }   // even: one owner warpgroup per stage
constexpr uint32_t kBlockTile = 2 * kBox;
template <bool TRANS>
constexpr size_t block_smem_bytes()
{
    return 1024 + qb_stages<TRANS>() * kBlockTile + (TRANS ? 6 : 4) * kBox + (2 * qb_stages<TRANS>() + 2) * 8 + 16 + 32;
}

template <bool POW2, bool TRANS>
__global__ void __launch_bounds__(kQThreads, 1)
    quant_block_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmq,
                       const __grid_constant__ CUtensorMap tmqT, const QuantArgs p)
{
    constexpr int QB_STAGES = qb_stages<TRANS>();
    static_assert(QB_STAGES % 2 == 0, "a stage must belong to one of the two warpgroups");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base0 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (base0 & 1023u)) & 1023u;
    const uint32_t stage = base0 + pad;
    const uint32_t out_rows = stage + QB_STAGES * kBlockTile, out_cols = out_rows + (TRANS ? 2 : 4) * kBox;
    const uint32_t bars = out_cols + (TRANS ? 4 * kBox : 0);   // full[S], empty[S], warpgroup[2]
    uint8_t *tail = smem_raw + pad + QB_STAGES * kBlockTile + (TRANS ? 6 : 4) * kBox + (2 * QB_STAGES + 2) * 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tail);
    float *red = reinterpret_cast<float *>(tail + 16);          // 8 per-warp partial maxima
    if (threadIdx.x == 0) {
        for (int i = 0; i < QB_STAGES; ++i) {
            mbar_init(bars + 8 * i, 1);
            mbar_init(bars + 8 * (QB_STAGES + i), 4);             // the four warps of one warpgroup
        }
        mbar_init(bars + 8 * (2 * QB_STAGES), 4);
        mbar_init(bars + 8 * (2 * QB_STAGES + 1), 4);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
    const int64_t ncb = p.cols / 128, items = (p.rows / 128) * ncb;   // rows is a multiple of 128
    const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    if (warp == kConsumers) {   // producer: one block per tile as two 128 x 64 boxes
        if (lane == 0)
            produce128(stage, bars, QB_STAGES, &tmx, items, ncb, ctl, p.timeout_ns, 0x1300);
        return;
    }
    const int h = t >> 7, rr = t & 127;
    const uint32_t wgbar = bars + 8 * (2 * QB_STAGES + h);
    const bool elected = rr == 0;
    uint32_t cph = 0;
    uint32_t it = h;   // this warpgroup's tiles are the CTA's tiles h, h + 2, ...
    for (int64_t item = blockIdx.x + h * static_cast<int64_t>(gridDim.x); item < items;
         item += 2 * static_cast<int64_t>(gridDim.x), it += 2) {
        const uint32_t st = it % QB_STAGES, ph = (it / QB_STAGES) & 1;
        if (!mbar_wait(bars + 8 * st, ph, ctl, 0x1400 | st))
            break;
        const int64_t rb = item / ncb, cb = item - rb * ncb;
        const int64_t y = rb * 128;                          // first row of the block
        const uint32_t sb = (it >> 1) & 1;                   // this warpgroup's staging set
        const uint32_t out_r = out_rows + (TRANS ? h : 2 * h + sb) * kBox, out_c = out_cols + (2 * h + sb) * kBox;
        uint32_t w[64];
        load_row(stage + st * kBlockTile, rr, w);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bars + 8 * (QB_STAGES + st));
        float a = amax_words(w);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (lane == 0)
            red[warp] = a;
        if (elected)
            bulk_wait_read1();                              // all but the newest store group are read
        if (!wg_sync(wgbar, cph, ctl, 0x1410))             // block max published
            break;
        a = fmaxf(fmaxf(red[h * 4], red[h * 4 + 1]), fmaxf(red[h * 4 + 2], red[h * 4 + 3]));
        const GroupScale g = make_group_scale(a, POW2);
        if (rr == 0)
            p.s[(y / 128) * p.lds + cb] = g.s;
        write_codes(out_r, rr, w, g);
        if (TRANS) {
            if (!wg_sync(wgbar, cph, ctl, 0x1411))         // row codes complete
                break;
            // column rr of the block: bytes (row i, col rr) of the staging box
            const int j = rr >> 4, e = rr & 15;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t wd[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = q * 16 + k * 4;
                    wd[k] = lds_u8(out_r + sw128(i, j) + e) | (lds_u8(out_r + sw128(i + 1, j) + e) << 8) |
                            (lds_u8(out_r + sw128(i + 2, j) + e) << 16) | (lds_u8(out_r + sw128(i + 3, j) + e) << 24);
                }
                sts_v4(out_c + sw128(rr, q), make_uint4(wd[0], wd[1], wd[2], wd[3]));
            }
        }
        fence_proxy_async_smem();
        if (!wg_sync(wgbar, cph, ctl, 0x1412))
            break;
        if (elected) {
            tma_store_2d(&tmq, out_r, static_cast<int32_t>(cb * 128), static_cast<int32_t>(y));
            bulk_commit();
            if (TRANS) {
                tma_store_2d(&tmqT, out_c, static_cast<int32_t>(y), static_cast<int32_t>(cb * 128));
                bulk_commit();
            }
        }
    }
    if (elected)
        bulk_wait0();
}

template <class K, class... Args>
cudaError_t launch_q(K kern, size_t smem, int64_t items, int num_sms, cudaStream_t st, int threads, Args... args)
{
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    const int64_t grid = items < num_sms ? items : num_sms;
    kern<<<static_cast<int>(grid), threads, smem, st>>>(args...);
    return cudaGetLastError();
}

// ------------------------------------ re-quantization of cached FP8 into 128x1 groups
//
// Page 2 ("9 Amazing Deepseek Hacks"), last paragraph: in the backward pass the cached FP8
// matrix is read out, dequantized, transposed and quantized again into 128x1 tiles.  Input:
// codes q[t, c] of a 1x128 quantization with scales s[(c/128) lds + t]; each element is
// dequantized to binary32 (dec(q) * s, one rounded product), and each column's 128 values
// of a 128-row block form one group, written transposed: qT[c, t], sT[(t/128) ldsT + c].
//
// Tiles of 128 rows x 128 columns of codes (16 KB) and their 128 row scales stream through
// a TMA ring.  Consumer thread (cp, qd) owns columns 2cp, 2cp+1 and rows 32qd .. +31 of the
// tile: it reads code pairs with 2-byte shared loads (the two columns of one row,
// conflict-free), keeps its 64 dequantized values in registers, and the four row quarters'
// max-abs values meet in shared memory (the partials double-buffered by tile parity).  The
// two column halves are independent: warps w, w+2, w+4, w+6 (w = 0, 1) own columns
// 64w .. +63 and meet only among themselves, once per tile; each column's 32 codes go to
// the swizzled staging tile as two 16-byte pieces of row c, and one thread per half waits
// for its four warps' rows and issues that half's TMA store while the others move on.  Two
// CTAs share an SM, so one's tile latency (barrier, conversion) overlaps the other's.
constexpr int RQ_STAGES = 4;
constexpr int kRqCtasPerSm = 2;
constexpr uint32_t kRqScales = 128 * 4;   // one tile's row scales
constexpr size_t kRqSmem =
    1024 + RQ_STAGES * kBox + 2 * kBox + RQ_STAGES * kRqScales + 2 * 4 * 128 * 4 + (2 * RQ_STAGES + 4) * 8 + 16;

template <bool POW2>
__global__ void __launch_bounds__(kQThreads, kRqCtasPerSm)
    requant_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmqT,
                   const RequantArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base0 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (base0 & 1023u)) & 1023u;
    const uint32_t stage = base0 + pad, out = stage + RQ_STAGES * kBox, scl = out + 2 * kBox;
    float *red = reinterpret_cast<float *>(smem_raw + pad + (RQ_STAGES + 2) * kBox + RQ_STAGES * kRqScales);
    // red: [2][4][128] partial max-abs values; then full[S], empty[S], syncA[2], ready[2], abort
    const uint32_t bars = smem_u32(red + 2 * 4 * 128);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(red + 2 * 4 * 128 + (2 * RQ_STAGES + 4) * 2);
    const uint32_t full = bars, empty = bars + 8 * RQ_STAGES, syncA0 = bars + 16 * RQ_STAGES, ready0 = syncA0 + 16;
    if (threadIdx.x == 0) {
        for (int i = 0; i < RQ_STAGES; ++i) {
            mbar_init(full + 8 * i, 1);
            mbar_init(empty + 8 * i, kConsumers);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(syncA0 + 8 * h, kConsumers / 2);
            mbar_init(ready0 + 8 * h, kConsumers / 2);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ncb = p.cols / 128, items = (p.rows / 128) * ncb;
    const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    if (warp == kConsumers) {   // producer: one 128 x 128 box of codes per tile
        if (lane == 0) {
            uint32_t it = 0;
            for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
                const uint32_t st = it % RQ_STAGES, ph = (it / RQ_STAGES) & 1;
                if (!mbar_wait(empty + 8 * st, ph ^ 1, ctl, 0x1800 | st))
                    break;
                const int64_t tb = item / ncb, cb = item - tb * ncb;
                mbar_arrive_expect_tx(full + 8 * st, kBox + kRqScales);
                tma_load_2d(stage + st * kBox, &tmq, full + 8 * st, static_cast<int32_t>(cb * 128),
                            static_cast<int32_t>(tb * 128));
                bulk_load(scl + st * kRqScales, p.s + cb * p.lds + tb * 128, kRqScales, full + 8 * st);
            }
            for (uint32_t j = it > RQ_STAGES ? it - RQ_STAGES : 0; j < it; ++j) {   // no load left in flight
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(full + 8 * (j % RQ_STAGES), (j / RQ_STAGES) & 1))
                    if (globaltimer_ns() - t0 > p.timeout_ns)
                        break;
            }
        }
        return;
    }
    const int half = warp & 1, cp = lane + 32 * half, qd = warp >> 1, c = 2 * cp;
    const bool elected = lane == 0 && warp < 2;   // one storing thread per column half
    const uint32_t syncA = syncA0 + 8 * half, ready = ready0 + 8 * half;
    // byte offset of this thread's code pair in a row r of a swizzled tile: chunk cp/8 sits
    // at chunk (cp/8) ^ (r % 8)
    const uint32_t chunk16 = (cp >> 3) << 4, byte_in = (2 * cp) & 15;
    uint32_t kA = 0, it = 0;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
        const int64_t tb = item / ncb, cb = item - tb * ncb;
        const uint32_t st = it % RQ_STAGES, ph = (it / RQ_STAGES) & 1;
        if (!mbar_wait(full + 8 * st, ph, ctl, 0x1810 | st))
            break;
        const uint32_t tile = stage + st * kBox + 32 * 128 * qd;   // row 32qd of the tile
        float sc[32];   // input scales of rows 32qd .. +31 (the same for every lane: broadcast)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 v = lds_v4(scl + st * kRqScales + (32 * qd + 4 * j) * 4);
            sc[4 * j] = __uint_as_float(v.x); sc[4 * j + 1] = __uint_as_float(v.y);
            sc[4 * j + 2] = __uint_as_float(v.z); sc[4 * j + 3] = __uint_as_float(v.w);
        }
        // P[i] = (column c, column c + 1) of row 32qd + i, dequantized: the pair's low and
        // high byte times the row's scale, kept packed for the pairwise arithmetic below
        unsigned long long P[32];
        float ma = 0.0f, mb = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {   // rows 32qd + k + 8m share the swizzle phase k
            const uint32_t rowk = tile + (chunk16 ^ (k << 4)) + byte_in + 128 * k;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int i = k + 8 * m;
                const uint32_t pair = lds_u16(rowk + 1024 * m);
                const __half2 h(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair), __NV_E4M3));
                const float2 d = __half22float2(h);   // exact: every E4M3 value is an FP16 value
                P[i] = fmul2(pack2(d.x, d.y), pack2(sc[i], sc[i]));
                ma = fmaxf(ma, fabsf(lo_of(P[i])));
                mb = fmaxf(mb, fabsf(hi_of(P[i])));
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty + 8 * st);
        float *redt = red + (it & 1) * 512;
        *reinterpret_cast<float2 *>(redt + qd * 128 + c) = make_float2(ma, mb);
        if (elected)
            bulk_wait_read1();   // the store of two tiles ago has left this tile's staging buffer
        if (!wg_sync(syncA, kA, ctl, 0x1820))
            break;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 v = *reinterpret_cast<const float2 *>(redt + q * 128 + c);
            ma = fmaxf(ma, v.x);
            mb = fmaxf(mb, v.y);
        }
        const GroupScale ga = make_group_scale(ma, POW2), gb = make_group_scale(mb, POW2);
        // Codes of both columns per row with per-lane scales; four rows' code pairs are then
        // regrouped by byte permutes into one word of column c and one of column c + 1.
        uint32_t wa[8], wb[8];
        if (POW2 ? (ga.mode == 1 && gb.mode == 1) : (ga.mode != 2 && gb.mode != 2)) {
            // amax/448 scales: the correction-step quotient (valid for the all-zero group's
            // s = r = 1 as well); power-of-2 scales: the exact product by 2^-e
            const unsigned long long nr = pack2(-ga.r, -gb.r), s2 = pack2(ga.s, gb.s), r2 = pack2(ga.r, gb.r);
            const uint32_t flip = POW2 ? 0u : 0x80808080u;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                unsigned long long t[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    t[u] = POW2 ? fmul2(P[4 * q + u], r2) : neg_quotient2(P[4 * q + u], nr, s2);
                // bytes: (c, c + 1) of row 4q, then of row 4q + 1 | rows 4q + 2, 4q + 3
                const uint32_t A = e4m3x4(lo_of(t[0]), hi_of(t[0]), lo_of(t[1]), hi_of(t[1]));
                const uint32_t B = e4m3x4(lo_of(t[2]), hi_of(t[2]), lo_of(t[3]), hi_of(t[3]));
                wa[q] = __byte_perm(A, B, 0x6420) ^ flip;
                wb[q] = __byte_perm(A, B, 0x7531) ^ flip;
            }
        } else {   // a tiny scale (IEEE division) in either column: element by element
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                wa[q] = e4m3_pair(lo_of(P[4 * q]), lo_of(P[4 * q + 1]), ga) |
                        (e4m3_pair(lo_of(P[4 * q + 2]), lo_of(P[4 * q + 3]), ga) << 16);
                wb[q] = e4m3_pair(hi_of(P[4 * q]), hi_of(P[4 * q + 1]), gb) |
                        (e4m3_pair(hi_of(P[4 * q + 2]), hi_of(P[4 * q + 3]), gb) << 16);
            }
        }
        const uint32_t stg = out + (it & 1) * kBox;
        sts_v4(stg + sw128(c, 2 * qd), make_uint4(wa[0], wa[1], wa[2], wa[3]));
        sts_v4(stg + sw128(c, 2 * qd + 1), make_uint4(wa[4], wa[5], wa[6], wa[7]));
        sts_v4(stg + sw128(c + 1, 2 * qd), make_uint4(wb[0], wb[1], wb[2], wb[3]));
        sts_v4(stg + sw128(c + 1, 2 * qd + 1), make_uint4(wb[4], wb[5], wb[6], wb[7]));
        fence_proxy_async_smem();
        if (qd == 0) {
            float *dst = p.sT + tb * p.ldsT + cb * 128 + c;
            dst[0] = ga.s;
            dst[1] = gb.s;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(ready);   // this warp's staging rows are written
        if (elected) {   // this half's 64 rows of the staging tile (rows of qT: columns of q)
            if (!mbar_wait(ready, it & 1, ctl, 0x1821))
                break;
            tma_store_2d(&tmqT, stg + half * 64 * 128, static_cast<int32_t>(tb * 128),
                         static_cast<int32_t>(cb * 128 + 64 * half));
            bulk_commit();
        }
    }
    if (elected)
        bulk_wait0();
}

} // namespace

cudaError_t launch_quant_rows(const CUtensorMap &tmx, const CUtensorMap &tmq, const QuantArgs &a, bool pow2,
                              int num_sms, cudaStream_t st)
{
    const int64_t items = ((a.rows + 127) / 128) * (a.cols / 128);
    if (items == 0)
        return cudaSuccess;
    constexpr size_t smem = kRowsSmem;
    return pow2 ? launch_q(quant_rows_kernel<true>, smem, items, num_sms, st, kRowsThreads, tmx, tmq, a)
                : launch_q(quant_rows_kernel<false>, smem, items, num_sms, st, kRowsThreads, tmx, tmq, a);
}

cudaError_t launch_quant_dual(const CUtensorMap &tmx, const CUtensorMap &tmq, const CUtensorMap &tmqT,
                              const QuantArgs &a, bool pow2, int num_sms, cudaStream_t st)
{
    const int64_t items = (a.rows / 128) * (a.cols / 128);   // rows is a multiple of 128 here
    if (items == 0)
        return cudaSuccess;
    constexpr size_t smem = kDualSmem;
    const bool rows_out = a.q != nullptr;
    if (pow2)
        return rows_out ? launch_q(quant_dual16_kernel<true, true>, smem, items, num_sms, st, kDualThreads, tmx, tmq,
                                   tmqT, a)
                        : launch_q(quant_dual16_kernel<true, false>, smem, items, num_sms, st, kDualThreads, tmx, tmq,
                                   tmqT, a);
    return rows_out ? launch_q(quant_dual16_kernel<false, true>, smem, items, num_sms, st, kDualThreads, tmx, tmq,
                               tmqT, a)
                    : launch_q(quant_dual16_kernel<false, false>, smem, items, num_sms, st, kDualThreads, tmx, tmq,
                               tmqT, a);
}

cudaError_t launch_quant_block(const CUtensorMap &tmx, const CUtensorMap &tmq, const CUtensorMap &tmqT,
                               const QuantArgs &a, bool pow2, int num_sms, cudaStream_t st)
{
    const int64_t items = (a.rows / 128) * (a.cols / 128);   // rows is a multiple of 128
    if (items == 0)
        return cudaSuccess;
    const bool tr = a.qT != nullptr;
    constexpr size_t smem_t = block_smem_bytes<true>();
    constexpr size_t smem_n = block_smem_bytes<false>();
    if (pow2)
        return tr ? launch_q(quant_block_kernel<true, true>, smem_t, items, num_sms, st, kQThreads, tmx, tmq, tmqT, a)
                  : launch_q(quant_block_kernel<true, false>, smem_n, items, num_sms, st, kQThreads, tmx, tmq, tmqT, a);
    return tr ? launch_q(quant_block_kernel<false, true>, smem_t, items, num_sms, st, kQThreads, tmx, tmq, tmqT, a)
              : launch_q(quant_block_kernel<false, false>, smem_n, items, num_sms, st, kQThreads, tmx, tmq, tmqT, a);
}

cudaError_t launch_requant(const CUtensorMap &tmq, const CUtensorMap &tmqT, const RequantArgs &a, bool pow2,
                           int num_sms, cudaStream_t st)
{
    const int64_t items = (a.rows / 128) * (a.cols / 128);
    if (items == 0)
        return cudaSuccess;
    const int ctas = kRqCtasPerSm * num_sms;
    return pow2 ? launch_q(requant_kernel<true>, kRqSmem, items, ctas, st, kQThreads, tmq, tmqT, a)
                : launch_q(requant_kernel<false>, kRqSmem, items, ctas, st, kQThreads, tmq, tmqT, a);
}

} // namespace mpq

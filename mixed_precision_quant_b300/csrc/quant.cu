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
// All three kernels are persistent and warp-specialised: one producer warp streams BF16
// tiles into a shared-memory ring with 2-D TMA loads (completion counted on mbarriers),
// eight consumer warps reduce group max-abs values with warp shuffles, convert with the
// exact scale arithmetic of mpq_device.cuh and write E4M3 codes with coalesced stores
// (transposed codes are staged through shared memory).  Every wait is bounded.
#include "mpq_internal.h"
#include "mpq_device.cuh"

namespace mpq {
namespace {

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

// Barrier among the consumer warps only (the producer warp does not take part), on an
// mbarrier so that the wait is bounded: lane 0 of each warp arrives after the warp's
// own shared-memory writes, every lane waits for the phase.  Returns false on abort.
__device__ __forceinline__ bool consumers_sync(uint32_t bar, uint32_t &k, const WaitCtl &ctl, int tag)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        mbar_arrive(bar);
    const bool ok = mbar_wait(bar, k & 1, ctl, tag);
    ++k;
    return ok;
}

// max |x| over eight BF16 values, in packed BF16x2 arithmetic (exact), as binary32.
__device__ __forceinline__ float amax8(const uint4 &v)
{
    uint32_t m;
    const uint32_t a0 = v.x & 0x7FFF7FFFu, a1 = v.y & 0x7FFF7FFFu, a2 = v.z & 0x7FFF7FFFu, a3 = v.w & 0x7FFF7FFFu;
    asm("{\n\t.reg .b32 t0, t1;\n\t"
        "max.bf16x2 t0, %1, %2;\n\t"
        "max.bf16x2 t1, %3, %4;\n\t"
        "max.bf16x2 %0, t0, t1;\n\t}"
        : "=r"(m) : "r"(a0), "r"(a1), "r"(a2), "r"(a3));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

__device__ __forceinline__ float half_warp_amax(float a)
{
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    return a;
}

// Eight BF16 values (one 16-byte chunk) -> eight E4M3 codes (8 bytes, memory order kept).
__device__ __forceinline__ uint2 codes8(const uint4 &v, const GroupScale &g)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        c[j] = e4m3_pair(__uint_as_float(bf16x2_lo(w[j])), __uint_as_float(bf16x2_hi(w[j])), g);
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// The group scale owned by lane `src` of the warp.
__device__ __forceinline__ GroupScale shfl_scale(const GroupScale &g, int src)
{
    GroupScale o;
    o.s = __shfl_sync(0xffffffffu, g.s, src);
    o.rlo = __shfl_sync(0xffffffffu, g.rlo, src);
    o.rhi = __shfl_sync(0xffffffffu, g.rhi, src);
    o.mode = __shfl_sync(0xffffffffu, g.mode, src);
    return o;
}

// Row groups held by a warp as row pairs: v[i] holds 8 values of row 2i + (lane >= 16).
// Lane l (l < 2P) computes the scale of row l once (returned); every row pair then takes
// its scale from the owner lane by shuffle and converts its values.
template <int P, bool POW2>
__device__ __forceinline__ GroupScale row_codes(const uint4 (&v)[P], uint2 (&out)[P])
{
    const int lane = threadIdx.x & 31, half = lane >> 4;
    float my_amax = 0.0f;
#pragma unroll
    for (int i = 0; i < P; ++i) {
        const float a = half_warp_amax(amax8(v[i]));
        const float other = __shfl_xor_sync(0xffffffffu, a, 16);
        if ((lane >> 1) == i)
            my_amax = ((lane & 1) == half) ? a : other;
    }
    const GroupScale mine = make_group_scale(my_amax, POW2);
#pragma unroll
    for (int i = 0; i < P; ++i)
        out[i] = codes8(v[i], shfl_scale(mine, 2 * i + half));
    return mine;
}

// ------------------------------------------------------------------ shared layout

constexpr int kConsumers = 8;                       // consumer warps per CTA
constexpr int kQThreads = 32 * (kConsumers + 1);    // + one producer warp
constexpr int kQtPitch = 144;                       // bytes per row of a transposed code tile

struct QuantSmem {
    uint8_t *stage;      // ring of tiles (BF16, rows of 256 bytes)
    uint64_t *bars;      // full[S], empty[S], consumer barrier
    volatile int *abort;
    uint8_t *extra;      // kernel-specific scratch (transposed tiles, reductions), 16-byte aligned
};

// Bytes of the fixed part: ring + barriers + abort flag, before the kernel's extra area.
template <int STAGES, int TILE_BYTES>
constexpr size_t ring_bytes() { return 128 + STAGES * TILE_BYTES + (2 * STAGES + 1) * 8 + 24; }

template <int STAGES, int TILE_BYTES>
__device__ __forceinline__ QuantSmem carve(uint8_t *raw)
{
    QuantSmem s;
    uint8_t *base = raw + ((128u - (smem_u32(raw) & 127u)) & 127u);
    s.stage = base;
    s.bars = reinterpret_cast<uint64_t *>(base + STAGES * TILE_BYTES);
    s.abort = reinterpret_cast<volatile int *>(s.bars + 2 * STAGES + 1);
    s.extra = base + ((STAGES * TILE_BYTES + (2 * STAGES + 1) * 8 + 8 + 15) & ~15);
    return s;
}

template <int STAGES>
__device__ __forceinline__ void init_ring(const QuantSmem &s)
{
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(smem_u32(s.bars + i), 1);
            mbar_init(smem_u32(s.bars + STAGES + i), kConsumers);
        }
        mbar_init(smem_u32(s.bars + 2 * STAGES), kConsumers);
        *s.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
}

// Producer: one lane streams tile `item` (row block, column block) into the ring.
template <int STAGES, int TILE_ROWS>
__device__ __forceinline__ void produce(const QuantSmem &s, const CUtensorMap *tm, int64_t items, int64_t ncb,
                                        const WaitCtl &ctl, uint64_t timeout_ns)
{
    constexpr uint32_t bytes = TILE_ROWS * 256;
    uint32_t it = 0;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
        const uint32_t st = it % STAGES, ph = (it / STAGES) & 1;
        if (!mbar_wait(smem_u32(s.bars + STAGES + st), ph ^ 1, ctl, 0x1100 | st))
            break;
        const int64_t rb = item / ncb, cb = item - rb * ncb;
        mbar_arrive_expect_tx(smem_u32(s.bars + st), bytes);
        tma_load_2d(smem_u32(s.stage + st * bytes), tm, smem_u32(s.bars + st), static_cast<int32_t>(cb * 128),
                    static_cast<int32_t>(rb * TILE_ROWS));
    }
    // drain: copies still in flight must land before the CTA exits
    for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; ++j) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(s.bars + j % STAGES), (j / STAGES) & 1))
            if (globaltimer_ns() - t0 > timeout_ns)
                break;
    }
}

// ------------------------------------------------------------------ 1x128 rows
//
// Tile = 64 rows x 128 columns (16 KB).  Consumer warp w owns rows 8w .. 8w+7 of the tile,
// a half-warp per row (16 lanes x 8 values); it copies its rows into registers, releases
// the stage, then writes 8 codes per lane (128 contiguous bytes per half-warp) and the
// 8 row scales with one store.
constexpr int QR_ROWS = 64, QR_STAGES = 4, QR_TILE = QR_ROWS * 256;
constexpr size_t QR_SMEM = ring_bytes<QR_STAGES, QR_TILE>();

template <bool POW2>
__global__ void __launch_bounds__(kQThreads, 3)
    quant_rows_kernel(const __grid_constant__ CUtensorMap tmx, const QuantArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    const QuantSmem sm = carve<QR_STAGES, QR_TILE>(smem_raw);
    init_ring<QR_STAGES>(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ncb = p.cols / 128, items = ((p.rows + QR_ROWS - 1) / QR_ROWS) * ncb;
    const WaitCtl ctl{sm.abort, p.status, p.timeout_ns};
    if (warp == kConsumers) {
        if (lane == 0)
            produce<QR_STAGES, QR_ROWS>(sm, &tmx, items, ncb, ctl, p.timeout_ns);
        return;
    }
    const int half = lane >> 4, hl = lane & 15;
    uint32_t it = 0;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
        const uint32_t st = it % QR_STAGES, ph = (it / QR_STAGES) & 1;
        if (!mbar_wait(smem_u32(sm.bars + st), ph, ctl, 0x1200 | st))
            break;
        const int64_t rb = item / ncb, kb = item - rb * ncb;
        const uint32_t tile = smem_u32(sm.stage + st * QR_TILE);
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[i] = lds_v4(tile + (warp * 8 + 2 * i + half) * 256 + hl * 16);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(sm.bars + QR_STAGES + st));
        uint2 cw[4];
        const GroupScale mine = row_codes<4, POW2>(v, cw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t r = rb * QR_ROWS + warp * 8 + 2 * i + half;
            if (r < p.rows)
                *reinterpret_cast<uint2 *>(p.q + r * p.ldq + kb * 128 + hl * 8) = cw[i];
        }
        const float my_s = mine.s;
        const int64_t r = rb * QR_ROWS + warp * 8 + lane;
        if (lane < 8 && r < p.rows)
            p.s[kb * p.lds + r] = my_s;
    }
}

// --------------------------------------------------- fused 1x128 + 128x1 (dual)
//
// Tile = 128 x 128 (32 KB).  Row groups: warp w owns rows 16w .. 16w+15 (half-warp per
// row).  Column groups: thread t owns column t % 128 over rows 64 (t / 128) .. +63; the
// two halves combine their max through shared memory.  After both passes have read the
// tile into registers the stage is released; the column codes are transposed through a
// padded shared tile and written as 128 contiguous bytes per output row.
constexpr int QD_STAGES = 2, QD_TILE = 128 * 256;
constexpr size_t QD_SMEM = ring_bytes<QD_STAGES, QD_TILE>() + 128 * kQtPitch + 2 * 128 * 4;

template <bool POW2, bool ROWS>
__global__ void __launch_bounds__(kQThreads, 2)
    quant_dual_kernel(const __grid_constant__ CUtensorMap tmx, const QuantArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    const QuantSmem sm = carve<QD_STAGES, QD_TILE>(smem_raw);
    uint8_t *qts = sm.extra;
    float *colmax = reinterpret_cast<float *>(sm.extra + 128 * kQtPitch);
    init_ring<QD_STAGES>(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
    const int64_t ncb = p.cols / 128, items = (p.rows / 128) * ncb;
    const WaitCtl ctl{sm.abort, p.status, p.timeout_ns};
    if (warp == kConsumers) {
        if (lane == 0)
            produce<QD_STAGES, 128>(sm, &tmx, items, ncb, ctl, p.timeout_ns);
        return;
    }
    const int half = lane >> 4, hl = lane & 15;
    const int c = t & 127, h = t >> 7;
    const uint32_t cbar = smem_u32(sm.bars + 2 * QD_STAGES);
    uint32_t cph = 0;  // consumer-barrier phase counter
    uint32_t it = 0;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
        const uint32_t st = it % QD_STAGES, ph = (it / QD_STAGES) & 1;
        if (!mbar_wait(smem_u32(sm.bars + st), ph, ctl, 0x1300 | st))
            break;
        const int64_t rb = item / ncb, cb = item - rb * ncb;
        const int64_t r0 = rb * 128, c0 = cb * 128;
        const uint32_t tile = smem_u32(sm.stage + st * QD_TILE);

        if (ROWS) {
            // row groups first, so their registers are free before the column pass
            uint4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = lds_v4(tile + (warp * 16 + 2 * i + half) * 256 + hl * 16);
            uint2 cw[8];
            const GroupScale mine = row_codes<8, POW2>(v, cw);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = warp * 16 + 2 * i + half;
                *reinterpret_cast<uint2 *>(p.q + (r0 + r) * p.ldq + c0 + hl * 8) = cw[i];
            }
            const float my_s = mine.s;
            if (lane < 16)
                p.s[cb * p.lds + r0 + warp * 16 + lane] = my_s;
        }
        float col[64];
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            col[i] = __uint_as_float(lds_u16(tile + (h * 64 + i) * 256 + c * 2) << 16);
            a = fmaxf(a, fabsf(col[i]));
        }
        colmax[h * 128 + c] = a;
        if (!consumers_sync(cbar, cph, ctl, 0x1310))  // tile fully read, column halves published
            break;
        if (lane == 0)
            mbar_arrive(smem_u32(sm.bars + QD_STAGES + st));

        a = fmaxf(colmax[c], colmax[128 + c]);
        const GroupScale g = make_group_scale(a, POW2);
        if (h == 0)
            p.sT[rb * p.ldsT + c0 + c] = g.s;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = j * 16 + 4 * k;
                w[k] = e4m3_pair(col[i], col[i + 1], g) | (e4m3_pair(col[i + 2], col[i + 3], g) << 16);
            }
            *reinterpret_cast<uint4 *>(qts + c * kQtPitch + h * 64 + j * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (!consumers_sync(cbar, cph, ctl, 0x1311))  // transposed tile complete
            break;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int id = t + k * 256;
            const int rr = id >> 3, part = id & 7;
            *reinterpret_cast<uint4 *>(p.qT + (c0 + rr) * p.ldqT + r0 + part * 16) =
                *reinterpret_cast<const uint4 *>(qts + rr * kQtPitch + part * 16);
        }
        if (!consumers_sync(cbar, cph, ctl, 0x1312))  // transposed tile and colmax free again
            break;
    }
}

// ------------------------------------------------------------------ 128x128 blocks
//
// Tile = one block (32 KB).  Each consumer thread copies its 64 values into registers;
// the block max goes through warp shuffles and one shared reduction; the stage is
// released before the codes are computed.  Optional transposed codes are gathered through
// two padded shared tiles.
constexpr int QB_STAGES = 2, QB_TILE = 128 * 256;
constexpr size_t QB_SMEM = ring_bytes<QB_STAGES, QB_TILE>() + 2 * 128 * kQtPitch + 64;

template <bool POW2, bool TRANS>
__global__ void __launch_bounds__(kQThreads, 2)
    quant_block_kernel(const __grid_constant__ CUtensorMap tmx, const QuantArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    const QuantSmem sm = carve<QB_STAGES, QB_TILE>(smem_raw);
    uint8_t *cs = sm.extra;
    uint8_t *qts = sm.extra + 128 * kQtPitch;
    float *red = reinterpret_cast<float *>(sm.extra + 2 * 128 * kQtPitch);
    init_ring<QB_STAGES>(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
    const int64_t ncb = p.cols / 128, items = (p.rows / 128) * ncb;
    const WaitCtl ctl{sm.abort, p.status, p.timeout_ns};
    if (warp == kConsumers) {
        if (lane == 0)
            produce<QB_STAGES, 128>(sm, &tmx, items, ncb, ctl, p.timeout_ns);
        return;
    }
    const int half = lane >> 4, hl = lane & 15;
    const uint32_t cbar = smem_u32(sm.bars + 2 * QB_STAGES);
    uint32_t cph = 0;  // consumer-barrier phase counter
    uint32_t it = 0;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x, ++it) {
        const uint32_t st = it % QB_STAGES, ph = (it / QB_STAGES) & 1;
        if (!mbar_wait(smem_u32(sm.bars + st), ph, ctl, 0x1400 | st))
            break;
        const int64_t bi = item / ncb, bj = item - bi * ncb;
        const int64_t r0 = bi * 128, c0 = bj * 128;
        const uint32_t tile = smem_u32(sm.stage + st * QB_TILE);
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = lds_v4(tile + (warp * 16 + 2 * i + half) * 256 + hl * 16);
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            a = fmaxf(a, amax8(v[i]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (lane == 0)
            red[warp] = a;
        if (!consumers_sync(cbar, cph, ctl, 0x1410))  // block max published, tile read
            break;
        if (lane == 0)
            mbar_arrive(smem_u32(sm.bars + QB_STAGES + st));
        a = red[0];
#pragma unroll
        for (int k = 1; k < kConsumers; ++k)
            a = fmaxf(a, red[k]);
        const GroupScale g = make_group_scale(a, POW2);
        if (t == 0)
            p.s[bi * p.lds + bj] = g.s;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = warp * 16 + 2 * i + half;
            const uint2 cw = codes8(v[i], g);
            *reinterpret_cast<uint2 *>(p.q + (r0 + r) * p.ldq + c0 + hl * 8) = cw;
            if (TRANS)
                *reinterpret_cast<uint2 *>(cs + r * kQtPitch + hl * 8) = cw;
        }
        if (TRANS) {
            if (!consumers_sync(cbar, cph, ctl, 0x1411))  // row-major codes complete
                break;
            const int c = t & 127, h = t >> 7;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t wd[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = h * 64 + j * 16 + k * 4;
                    wd[k] = static_cast<uint32_t>(cs[i * kQtPitch + c]) |
                            (static_cast<uint32_t>(cs[(i + 1) * kQtPitch + c]) << 8) |
                            (static_cast<uint32_t>(cs[(i + 2) * kQtPitch + c]) << 16) |
                            (static_cast<uint32_t>(cs[(i + 3) * kQtPitch + c]) << 24);
                }
                *reinterpret_cast<uint4 *>(qts + c * kQtPitch + h * 64 + j * 16) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            }
            if (!consumers_sync(cbar, cph, ctl, 0x1412))  // transposed tile complete
                break;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int id = t + k * 256;
                const int rr = id >> 3, part = id & 7;
                *reinterpret_cast<uint4 *>(p.qT + (c0 + rr) * p.ldqT + r0 + part * 16) =
                    *reinterpret_cast<const uint4 *>(qts + rr * kQtPitch + part * 16);
            }
        }
        if (!consumers_sync(cbar, cph, ctl, 0x1413))  // shared tiles and red[] free again
            break;
    }
}

template <class K>
cudaError_t launch_q(K kern, size_t smem, int per_sm, int64_t items, int num_sms, const CUtensorMap &tm,
                     const QuantArgs &a, cudaStream_t st)
{
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    int64_t grid = static_cast<int64_t>(num_sms) * per_sm;
    if (items < grid)
        grid = items;
    kern<<<static_cast<int>(grid), kQThreads, smem, st>>>(tm, a);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_quant_rows(const CUtensorMap &tm, const QuantArgs &a, bool pow2, int num_sms, cudaStream_t st)
{
    const int64_t items = ((a.rows + QR_ROWS - 1) / QR_ROWS) * (a.cols / 128);
    if (items == 0)
        return cudaSuccess;
    return pow2 ? launch_q(quant_rows_kernel<true>, QR_SMEM, 3, items, num_sms, tm, a, st)
                : launch_q(quant_rows_kernel<false>, QR_SMEM, 3, items, num_sms, tm, a, st);
}

cudaError_t launch_quant_dual(const CUtensorMap &tm, const QuantArgs &a, bool pow2, int num_sms, cudaStream_t st)
{
    const int64_t items = (a.rows / 128) * (a.cols / 128);
    if (items == 0)
        return cudaSuccess;
    const bool rows_out = a.q != nullptr;
    if (pow2)
        return rows_out ? launch_q(quant_dual_kernel<true, true>, QD_SMEM, 2, items, num_sms, tm, a, st)
                        : launch_q(quant_dual_kernel<true, false>, QD_SMEM, 2, items, num_sms, tm, a, st);
    return rows_out ? launch_q(quant_dual_kernel<false, true>, QD_SMEM, 2, items, num_sms, tm, a, st)
                    : launch_q(quant_dual_kernel<false, false>, QD_SMEM, 2, items, num_sms, tm, a, st);
}

cudaError_t launch_quant_block(const CUtensorMap &tm, const QuantArgs &a, bool pow2, int num_sms, cudaStream_t st)
{
    const int64_t items = (a.rows / 128) * (a.cols / 128);
    if (items == 0)
        return cudaSuccess;
    const bool tr = a.qT != nullptr;
    if (pow2)
        return tr ? launch_q(quant_block_kernel<true, true>, QB_SMEM, 2, items, num_sms, tm, a, st)
                  : launch_q(quant_block_kernel<true, false>, QB_SMEM, 2, items, num_sms, tm, a, st);
    return tr ? launch_q(quant_block_kernel<false, true>, QB_SMEM, 2, items, num_sms, tm, a, st)
              : launch_q(quant_block_kernel<false, false>, QB_SMEM, 2, items, num_sms, tm, a, st);
}

} // namespace mpq

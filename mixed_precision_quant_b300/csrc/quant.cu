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
// All kernels read BF16 once with 16-byte loads and write E4M3 codes with coalesced
// stores; group max-abs values are reduced with warp shuffles.
#include "mpq_internal.h"
#include "mpq_device.cuh"

namespace mpq {
namespace {

__device__ __forceinline__ uint4 ldg_v4(const uint16_t *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ float amax8(const uint4 &v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        a = fmaxf(a, fabsf(__uint_as_float(bf16x2_lo(w[j]))));
        a = fmaxf(a, fabsf(__uint_as_float(bf16x2_hi(w[j]))));
    }
    return a;
}

// Eight BF16 values (one 16-byte chunk) -> eight E4M3 codes (8 bytes, memory order kept).
__device__ __forceinline__ uint2 codes8(const uint4 &v, const GroupScale &g)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        c[j] = e4m3x2(scaled_value(__uint_as_float(bf16x2_lo(w[j])), g),
                      scaled_value(__uint_as_float(bf16x2_hi(w[j])), g));
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// ------------------------------------------------------------------ 1x128 rows
//
// One warp per item of 32 rows x 128 columns: each half-warp owns one row (16 lanes x 8
// values), 16 row pairs are loaded up front to keep 8 KB per warp in flight, and the 32
// row scales are written with one coalesced store.
template <bool POW2>
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                         int64_t ldx, uint8_t *__restrict__ q, int64_t ldq,
                                                         float *__restrict__ s, int64_t lds, int64_t nkb,
                                                         int64_t items)
{
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, hl = lane & 15;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * 8;
    for (int64_t item = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); item < items;
         item += nwarps) {
        const int64_t rb = item / nkb, kb = item - rb * nkb;
        const int64_t r0 = rb * 32;
        uint4 v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int64_t r = r0 + 2 * i + half;
            v[i] = r < rows ? ldg_v4(x + r * ldx + kb * 128 + hl * 8) : make_uint4(0, 0, 0, 0);
        }
        float my_s = 1.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float a = amax8(v[i]);
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            const GroupScale g = make_group_scale(a, POW2);
            const float other = __shfl_xor_sync(0xffffffffu, g.s, 16);
            if ((lane >> 1) == i)
                my_s = ((lane & 1) == half) ? g.s : other;
            const int64_t r = r0 + 2 * i + half;
            if (r < rows)
                *reinterpret_cast<uint2 *>(q + r * ldq + kb * 128 + hl * 8) = codes8(v[i], g);
        }
        if (r0 + lane < rows)
            s[kb * lds + r0 + lane] = my_s;
    }
}

// --------------------------------------------------- fused 1x128 + 128x1 (dual)
//
// One CTA per 128x128 tile per iteration: the tile is read once into registers and
// shared memory; the row groups are quantized from registers, the column groups from
// shared memory, and the column codes are transposed through shared memory so the
// transposed output is written with coalesced 16-byte stores.
constexpr int kQtPitch = 144; // bytes per row of the transposed code tile (bank spread)

template <bool POW2, bool ROWS>
__global__ void __launch_bounds__(256) quant_dual_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                         int64_t cols, int64_t ldx, uint8_t *__restrict__ q,
                                                         int64_t ldq, float *__restrict__ s, int64_t lds,
                                                         uint8_t *__restrict__ qT, int64_t ldqT,
                                                         float *__restrict__ sT, int64_t ldsT)
{
    // The BF16 tile and the transposed code tile share one buffer: the codes are written
    // only after every thread has read its column into registers.
    __shared__ __align__(16) uint8_t buf[128 * 128 * 2];
    __shared__ float colmax[2][128];
    auto xs = reinterpret_cast<uint16_t(*)[128]>(buf);
    auto qts = reinterpret_cast<uint8_t(*)[kQtPitch]>(buf);

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int half = lane >> 4, hl = lane & 15;
    const int64_t nrb = rows / 128, ncb = cols / 128, tiles = nrb * ncb;

    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t rb = tile / ncb, cb = tile - rb * ncb;
        const int64_t r0 = rb * 128, c0 = cb * 128;

        // 1. load rows 16*warp .. +15 (half-warp per row)
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = warp * 16 + 2 * i + half;
            v[i] = ldg_v4(x + (r0 + r) * ldx + c0 + hl * 8);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = warp * 16 + 2 * i + half;
            *reinterpret_cast<uint4 *>(&xs[r][hl * 8]) = v[i];
        }

        // 2. row groups (1x128)
        if (ROWS) {
            float my_s = 1.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float a = amax8(v[i]);
                a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
                a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
                a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
                a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
                const GroupScale g = make_group_scale(a, POW2);
                const float other = __shfl_xor_sync(0xffffffffu, g.s, 16);
                if ((lane >> 1) == i)
                    my_s = ((lane & 1) == half) ? g.s : other;
                const int r = warp * 16 + 2 * i + half;
                *reinterpret_cast<uint2 *>(q + (r0 + r) * ldq + c0 + hl * 8) = codes8(v[i], g);
            }
            if (lane < 16)
                s[cb * lds + r0 + warp * 16 + lane] = my_s;
        }
        __syncthreads();

        // 3. column groups (128x1): thread owns column c, rows h*64 .. h*64+63
        const int c = t & 127, h = t >> 7;
        float col[64];
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            col[i] = __uint_as_float(static_cast<uint32_t>(xs[h * 64 + i][c]) << 16);
            a = fmaxf(a, fabsf(col[i]));
        }
        colmax[h][c] = a;
        __syncthreads();
        a = fmaxf(colmax[0][c], colmax[1][c]);
        const GroupScale g = make_group_scale(a, POW2);
        if (h == 0)
            sT[rb * ldsT + c0 + c] = g.s;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = j * 16 + k * 4;
                w[k] = e4m3x2(scaled_value(col[i], g), scaled_value(col[i + 1], g)) |
                       (e4m3x2(scaled_value(col[i + 2], g), scaled_value(col[i + 3], g)) << 16);
            }
            *reinterpret_cast<uint4 *>(&qts[c][h * 64 + j * 16]) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncthreads();

        // 4. transposed codes out: 128 rows (columns of x) x 128 bytes
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int id = t + k * 256;
            const int rr = id >> 3, part = id & 7;
            *reinterpret_cast<uint4 *>(qT + (c0 + rr) * ldqT + r0 + part * 16) =
                *reinterpret_cast<const uint4 *>(&qts[rr][part * 16]);
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ 128x128 blocks
template <bool POW2, bool TRANS>
__global__ void __launch_bounds__(256) quant_block_kernel(const uint16_t *__restrict__ w, int64_t rows,
                                                          int64_t cols, int64_t ldw, uint8_t *__restrict__ q,
                                                          int64_t ldq, uint8_t *__restrict__ qT, int64_t ldqT,
                                                          float *__restrict__ s, int64_t lds)
{
    __shared__ __align__(16) uint8_t cs[TRANS ? 128 : 1][kQtPitch];
    __shared__ __align__(16) uint8_t qts[TRANS ? 128 : 1][kQtPitch];
    __shared__ float red[8];

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int half = lane >> 4, hl = lane & 15;
    const int64_t nbr = rows / 128, nbc = cols / 128, blocks = nbr * nbc;

    for (int64_t blk = blockIdx.x; blk < blocks; blk += gridDim.x) {
        const int64_t bi = blk / nbc, bj = blk - bi * nbc;
        const int64_t r0 = bi * 128, c0 = bj * 128;
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = warp * 16 + 2 * i + half;
            v[i] = ldg_v4(w + (r0 + r) * ldw + c0 + hl * 8);
        }
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            a = fmaxf(a, amax8(v[i]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (lane == 0)
            red[warp] = a;
        __syncthreads();
        a = red[0];
#pragma unroll
        for (int k = 1; k < 8; ++k)
            a = fmaxf(a, red[k]);
        const GroupScale g = make_group_scale(a, POW2);
        if (t == 0)
            s[bi * lds + bj] = g.s;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = warp * 16 + 2 * i + half;
            const uint2 cw = codes8(v[i], g);
            *reinterpret_cast<uint2 *>(q + (r0 + r) * ldq + c0 + hl * 8) = cw;
            if (TRANS)
                *reinterpret_cast<uint2 *>(&cs[r][hl * 8]) = cw;
        }
        if (TRANS) {
            __syncthreads();
            const int c = t & 127, h = t >> 7;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t wd[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = h * 64 + j * 16 + k * 4;
                    wd[k] = static_cast<uint32_t>(cs[i][c]) | (static_cast<uint32_t>(cs[i + 1][c]) << 8) |
                            (static_cast<uint32_t>(cs[i + 2][c]) << 16) |
                            (static_cast<uint32_t>(cs[i + 3][c]) << 24);
                }
                *reinterpret_cast<uint4 *>(&qts[c][h * 64 + j * 16]) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int id = t + k * 256;
                const int rr = id >> 3, part = id & 7;
                *reinterpret_cast<uint4 *>(qT + (c0 + rr) * ldqT + r0 + part * 16) =
                    *reinterpret_cast<const uint4 *>(&qts[rr][part * 16]);
            }
        }
        __syncthreads();
    }
}

int grid_for(int64_t work, int per_sm, int num_sms)
{
    int64_t g = static_cast<int64_t>(num_sms) * per_sm;
    if (work < g)
        g = work;
    return static_cast<int>(g < 1 ? 1 : g);
}

} // namespace

cudaError_t launch_quant_rows(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q,
                              int64_t ldq, float *s, int64_t lds, bool pow2, int num_sms, cudaStream_t st)
{
    const int64_t nkb = cols / 128;
    const int64_t items = ((rows + 31) / 32) * nkb;
    if (items == 0)
        return cudaSuccess;
    const int grid = grid_for((items + 7) / 8, 8, num_sms);
    if (pow2)
        quant_rows_kernel<true><<<grid, 256, 0, st>>>(x, rows, ldx, q, ldq, s, lds, nkb, items);
    else
        quant_rows_kernel<false><<<grid, 256, 0, st>>>(x, rows, ldx, q, ldq, s, lds, nkb, items);
    return cudaGetLastError();
}

cudaError_t launch_quant_dual(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q,
                              int64_t ldq, float *s, int64_t lds, uint8_t *qT, int64_t ldqT, float *sT,
                              int64_t ldsT, bool pow2, int num_sms, cudaStream_t st)
{
    const int64_t tiles = (rows / 128) * (cols / 128);
    if (tiles == 0)
        return cudaSuccess;
    const int grid = grid_for(tiles, 4, num_sms);
    const bool rows_out = q != nullptr;
#define MPQ_DUAL(P, R) \
    quant_dual_kernel<P, R><<<grid, 256, 0, st>>>(x, rows, cols, ldx, q, ldq, s, lds, qT, ldqT, sT, ldsT)
    if (pow2) {
        if (rows_out) MPQ_DUAL(true, true); else MPQ_DUAL(true, false);
    } else {
        if (rows_out) MPQ_DUAL(false, true); else MPQ_DUAL(false, false);
    }
#undef MPQ_DUAL
    return cudaGetLastError();
}

cudaError_t launch_quant_block(const uint16_t *w, int64_t rows, int64_t cols, int64_t ldw, uint8_t *q,
                               int64_t ldq, uint8_t *qT, int64_t ldqT, float *s, int64_t lds, bool pow2,
                               int num_sms, cudaStream_t st)
{
    const int64_t blocks = (rows / 128) * (cols / 128);
    if (blocks == 0)
        return cudaSuccess;
    const int grid = grid_for(blocks, 8, num_sms);
#define MPQ_BLK(P, T) \
    quant_block_kernel<P, T><<<grid, 256, 0, st>>>(w, rows, cols, ldw, q, ldq, qT, ldqT, s, lds)
    if (pow2) {
        if (qT) MPQ_BLK(true, true); else MPQ_BLK(true, false);
    } else {
        if (qT) MPQ_BLK(false, true); else MPQ_BLK(false, false);
    }
#undef MPQ_BLK
    return cudaGetLastError();
}

} // namespace mpq

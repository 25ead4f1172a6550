// swiglu.cu -- SwiGLU of the up-projection output fused with the 1x128 quantization of the
// result, the FP8 input of the MoE down projection.
//
// Method (source pages: page 1, first paragraph -- the SwiGLU operator's inputs are cached
// and its output recomputed in the backward pass; page 4, second paragraph -- the
// activation before the MoE down projection uses integral power-of-2 scaling factors):
//   x[r, c] = silu(gate[r, c]) * up[r, c],  silu(g) = g / (1 + e^-g),
// with the gate in the first W columns of each input row and the up value in the next W,
// all in binary32 with one rounding per operation; then the 1x128 groups of x are quantized
// with the arithmetic of the tile quantizer (quant_device.cuh).  e^x is a fixed sequence of
// binary32 operations: Cody and Waite's reduction (W. J. Cody, W. Waite, "Software Manual
// for the Elementary Functions", 1980) with a 15-bit head of ln 2, the degree-7 Taylor
// polynomial of e^r in Horner form with fused multiply-adds, and a scaling by 2^n with one
// rounding; every step uses an explicitly rounded intrinsic, so no contraction changes it.
//
// Design: memory-bound (4 bytes read, ~1 byte written per output value).  A grid-stride
// loop over (row, 128-column group) items, on one wave of resident blocks; four
// consecutive lanes share a group, each
// holding four 16-byte chunks of the gate and the matching four of the up half (coalesced
// 64-byte pieces per load instruction), the group's max-abs combined by two shuffles (eight
// or sixteen lanes per group were slower: the per-group scale work is repeated per lane).
// Each lane keeps the next batch's loads in flight while it converts the current one.
#include "mpq_internal.h"
#include "mpq_device.cuh"
#include "quant_device.cuh"
#include "swiglu_device.cuh"

namespace mpq {
namespace {

constexpr int kSwThreads = 128;
constexpr int kSwLpg = 4;                  // lanes per group
constexpr int kSwCpl = 16 / kSwLpg;        // 16-byte chunks per lane, per half
constexpr int kSwU = 1;                    // groups per lane and batch

template <bool POW2>
__global__ void __launch_bounds__(kSwThreads) swiglu_quant_kernel(const SwigluArgs p)
{
    const int KB = static_cast<int>(p.width / 128);
    const int64_t ngroups = p.rows * KB;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int lg = static_cast<int>(gtid % kSwLpg);
    const int64_t slot = gtid / kSwLpg, nslot = static_cast<int64_t>(gridDim.x) * blockDim.x / kSwLpg;
    const int64_t step = nslot * kSwU;
    // loads of batch `base`: per group u, the lane's chunks lg + c*LPG of the gate and up halves
    auto load = [&](int64_t base, uint4 (&gv)[kSwU][kSwCpl], uint4 (&uv)[kSwU][kSwCpl]) {
#pragma unroll
        for (int u = 0; u < kSwU; ++u) {
            const int64_t gi = base + u * nslot + slot;
            const bool ok = gi < ngroups;
            const int64_t r = ok ? gi / KB : 0;
            const int kb = ok ? static_cast<int>(gi - r * KB) : 0;
            const uint4 *gp = reinterpret_cast<const uint4 *>(p.h + r * p.ldh + kb * 128);
            const uint4 *up = reinterpret_cast<const uint4 *>(p.h + r * p.ldh + p.width + kb * 128);
#pragma unroll
            for (int c = 0; c < kSwCpl; ++c) {
                gv[u][c] = ok ? __ldg(gp + lg + c * kSwLpg) : make_uint4(0, 0, 0, 0);
                uv[u][c] = ok ? __ldg(up + lg + c * kSwLpg) : make_uint4(0, 0, 0, 0);
            }
        }
    };
    uint4 gv[kSwU][kSwCpl], uv[kSwU][kSwCpl];
    load(0, gv, uv);
    for (int64_t base = 0; base < ngroups; base += step) {   // trip count uniform over the grid
        uint4 gn[kSwU][kSwCpl], un[kSwU][kSwCpl];
        load(base + step, gn, un);
#pragma unroll
        for (int u = 0; u < kSwU; ++u) {
            const int64_t gi = base + u * nslot + slot;
            float x[8 * kSwCpl];
            float m = 0.0f;
#pragma unroll
            for (int c = 0; c < kSwCpl; ++c) {
                const uint32_t gw[4] = {gv[u][c].x, gv[u][c].y, gv[u][c].z, gv[u][c].w};
                const uint32_t uw[4] = {uv[u][c].x, uv[u][c].y, uv[u][c].z, uv[u][c].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float v0, v1;
                    swiglu2(__uint_as_float(bf16x2_lo(gw[j])), __uint_as_float(bf16x2_hi(gw[j])),
                            __uint_as_float(bf16x2_lo(uw[j])), __uint_as_float(bf16x2_hi(uw[j])), v0, v1);
                    x[8 * c + 2 * j] = v0;
                    x[8 * c + 2 * j + 1] = v1;
                    m = fmaxf(m, fmaxf(fabsf(v0), fabsf(v1)));
                }
            }
#pragma unroll
            for (int o = kSwLpg / 2; o > 0; o >>= 1)
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            if (gi < ngroups) {
                const int64_t r = gi / KB;
                const int kb = static_cast<int>(gi - r * KB);
                const GroupScale g = make_group_scale(m, POW2);
                uint8_t *dst = p.q + r * p.ldq + kb * 128;
#pragma unroll
                for (int c = 0; c < kSwCpl; ++c) {
                    uint32_t w[2];
                    codes_f32<8>(&x[8 * c], g, w);
                    *reinterpret_cast<uint2 *>(dst + (lg + c * kSwLpg) * 8) = make_uint2(w[0], w[1]);
                }
                if (lg == 0)
                    p.s[static_cast<int64_t>(kb) * p.lds + r] = g.s;
            }
        }
#pragma unroll
        for (int u = 0; u < kSwU; ++u)
#pragma unroll
            for (int c = 0; c < kSwCpl; ++c) {
                gv[u][c] = gn[u][c];
                uv[u][c] = un[u][c];
            }
    }
}

} // namespace

cudaError_t launch_swiglu_quant(const SwigluArgs &a, bool pow2, int num_sms, cudaStream_t st)
{
    const int64_t ngroups = a.rows * (a.width / 128);
    if (ngroups == 0)
        return cudaSuccess;
    // One wave: as many blocks as the SMs hold at once.  Every block runs the same number of
    // grid-stride iterations, so blocks beyond the resident ones would form a second, partial
    // wave that leaves SMs idle at the end.
    void (*kern)(const SwigluArgs) = pow2 ? swiglu_quant_kernel<true> : swiglu_quant_kernel<false>;
    static std::atomic<int> resident[2][64];   // blocks per SM, per variant and device (0: unknown)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    int per_sm = dev >= 0 && dev < 64 ? resident[pow2][dev].load(std::memory_order_relaxed) : 0;
    if (per_sm == 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSwThreads, 0);
        if (e != cudaSuccess)
            return e;
        per_sm = per_sm > 0 ? per_sm : 1;
        if (dev >= 0 && dev < 64)
            resident[pow2][dev].store(per_sm, std::memory_order_relaxed);
    }
    const int64_t want = (ngroups * kSwLpg + kSwThreads - 1) / kSwThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
    const int grid = static_cast<int>(want < cap ? want : cap);
    kern<<<grid, kSwThreads, 0, st>>>(a);
    return cudaGetLastError();
}

} // namespace mpq

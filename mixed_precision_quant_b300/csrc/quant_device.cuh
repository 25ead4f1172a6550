// quant_device.cuh -- the per-group arithmetic of the 1x128 / 128x1 / 128x128 quantizers,
// shared by the standalone quantizers and the grouped GEMM that quantizes its activations
// on the fly, so that both produce the same codes and scales bit for bit.
//
// A group's scale maps its max-abs value onto the largest E4M3 value (make_group_scale in
// mpq_device.cuh); each element becomes the E4M3 code of the correctly rounded binary32
// quotient x / s.
#pragma once
#include "mpq_device.cuh"
#include "mpq_internal.h"

namespace mpq {

// max |x| of the BF16 pairs in w[0..N), in packed BF16x2 arithmetic (exact), as binary32.
// max.xorsign.abs compares magnitudes (its result's sign is the XOR of the operands'
// signs, cleared once at the end), so no masking is needed per word.
template <int N>
__device__ __forceinline__ float amax_words(const uint32_t (&w)[N])
{
    uint32_t m[N];
#pragma unroll
    for (int i = 0; i < N; ++i)
        m[i] = w[i];
#pragma unroll
    for (int s = N / 2; s > 0; s >>= 1)
#pragma unroll
        for (int i = 0; i < s; ++i)
            asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[i]) : "r"(m[i]), "r"(m[i + s]));
    const uint32_t a = m[0] & 0x7FFF7FFFu;
    return fmaxf(__uint_as_float(a << 16), __uint_as_float(a & 0xFFFF0000u));
}

// Sixteen BF16 values (8 words, memory order) -> sixteen E4M3 codes (one 16-byte chunk),
// straight-line for the two common modes so that a thread's conversions overlap.
__device__ __forceinline__ uint4 codes16(const uint32_t *w, const GroupScale &g)
{
    uint32_t c[8];
    uint32_t flip = 0;
    if (g.mode == 0) {
        const unsigned long long nr = pack2(-g.r, -g.r), s2 = pack2(g.s, g.s);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const unsigned long long t =
                neg_quotient2(pack2(__uint_as_float(bf16x2_lo(w[j])), __uint_as_float(bf16x2_hi(w[j]))), nr, s2);
            c[j] = e4m3x2(lo_of(t), hi_of(t));
        }
        flip = 0x80808080u;
    } else if (g.mode == 1) {
        const unsigned long long r = pack2(g.r, g.r);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const unsigned long long p =
                fmul2(pack2(__uint_as_float(bf16x2_lo(w[j])), __uint_as_float(bf16x2_hi(w[j]))), r);
            c[j] = e4m3x2(lo_of(p), hi_of(p));
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            c[j] = e4m3_pair(__uint_as_float(bf16x2_lo(w[j])), __uint_as_float(bf16x2_hi(w[j])), g);
    }
    return make_uint4((c[0] | (c[1] << 16)) ^ flip, (c[2] | (c[3] << 16)) ^ flip, (c[4] | (c[5] << 16)) ^ flip,
                      (c[6] | (c[7] << 16)) ^ flip);
}

// Quantize one group of 128 consecutive BF16 values (64 words, memory order): returns the
// scale and writes the 128 codes as eight 16-byte chunks to out[0..7].
__device__ __forceinline__ float quantize_group128(const uint32_t (&w)[64], bool pow2, uint4 *out)
{
    const GroupScale g = make_group_scale(amax_words(w), pow2);
#pragma unroll
    for (int q = 0; q < 8; ++q)
        out[q] = codes16(&w[q * 8], g);
    return g.s;
}


// Wait until *count >= target (acquire at GPU scope), bounded like the mbarrier waits.
__device__ __forceinline__ bool wait_count(const int *count, int target, const WaitCtl &c, int tag)
{
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        int v;
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
        if (v >= target)
            return true;
        if (*c.abort)
            return false;
        if (globaltimer_ns() - t0 > c.timeout_ns) {
            *c.abort = 1;
            if (c.status != nullptr && atomicCAS(c.status, 0, kStatusTimeout) == 0)
                atomicExch(c.status + 1, tag);
            return false;
        }
        __nanosleep(128);
    }
}

__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Phase 1 of the grouped GEMMs with fused activation quantization (all threads of the CTA
// call it): the BF16 rows [goff[0], goff[G]) are quantized 1x128 -- the arithmetic of the
// standalone quantizer -- into f.xq [M, K] and f.sx [K/128][M], in blocks of 32 rows striped
// over the CTAs; each finished block is published by a fence and an atomic add to the
// ready count of every expert it overlaps.  Thread -> (row, 128-column group), consecutive
// threads on consecutive groups of a row (256 contiguous bytes each).
__device__ __forceinline__ void quantize_rows_phase(const int *goff, int G, int64_t M, int KB, int64_t K,
                                                    const FuseArgs &f)
{
    const int r_begin = goff[0], r_end = goff[G];
    const int nblk = (r_end - r_begin + 31) / 32;
    for (int b = blockIdx.x; b < nblk; b += gridDim.x) {
        const int r0 = r_begin + b * 32, r1 = r0 + 32 < r_end ? r0 + 32 : r_end;
        const int ngroups = (r1 - r0) * KB;
        for (int gi = threadIdx.x; gi < ngroups; gi += blockDim.x) {
            const int r = r0 + gi / KB, kb = gi - (gi / KB) * KB;
            const uint4 *src = reinterpret_cast<const uint4 *>(f.x + static_cast<int64_t>(r) * f.ldx + kb * 128);
            uint32_t w[64];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const uint4 v = __ldg(src + q);
                w[4 * q + 0] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
            }
            uint4 out[8];
            const float sc = quantize_group128(w, f.pow2 != 0, out);
            uint4 *dst = reinterpret_cast<uint4 *>(f.xq + static_cast<int64_t>(r) * K + kb * 128);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                dst[q] = out[q];
            f.sx[static_cast<int64_t>(kb) * M + r] = sc;
        }
        fence_proxy_async_global();   // the codes are read by TMA (async proxy)
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            int lo = 0, hi = G - 1;   // first expert whose rows end after r0
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (goff[mid + 1] > r0) hi = mid; else lo = mid + 1;
            }
            for (int g = lo; g < G && goff[g] < r1; ++g) {
                const int a = goff[g] > r0 ? goff[g] : r0, e = goff[g + 1] < r1 ? goff[g + 1] : r1;
                if (e > a)
                    atomicAdd(f.ready + g, e - a);
            }
        }
    }
}

} // namespace mpq

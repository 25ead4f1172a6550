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

// 2*NW BF16 values (NW words, memory order) -> 2*NW E4M3 codes (NW/2 words), straight-line
// for the two common modes so that a thread's conversions overlap.
template <int NW>
__device__ __forceinline__ void codes_words(const uint32_t *w, const GroupScale &g, uint32_t *out)
{
    if (g.mode == 0) {
        const unsigned long long nr = pack2(-g.r, -g.r), s2 = pack2(g.s, g.s);
#pragma unroll
        for (int j = 0; j < NW / 2; ++j) {
            const unsigned long long t0 = neg_quotient2(
                pack2(__uint_as_float(bf16x2_lo(w[2 * j])), __uint_as_float(bf16x2_hi(w[2 * j]))), nr, s2);
            const unsigned long long t1 = neg_quotient2(
                pack2(__uint_as_float(bf16x2_lo(w[2 * j + 1])), __uint_as_float(bf16x2_hi(w[2 * j + 1]))), nr, s2);
            out[j] = e4m3x4(lo_of(t0), hi_of(t0), lo_of(t1), hi_of(t1)) ^ 0x80808080u;
        }
    } else if (g.mode == 1) {
        const unsigned long long r = pack2(g.r, g.r);
#pragma unroll
        for (int j = 0; j < NW / 2; ++j) {
            const unsigned long long p0 =
                fmul2(pack2(__uint_as_float(bf16x2_lo(w[2 * j])), __uint_as_float(bf16x2_hi(w[2 * j]))), r);
            const unsigned long long p1 =
                fmul2(pack2(__uint_as_float(bf16x2_lo(w[2 * j + 1])), __uint_as_float(bf16x2_hi(w[2 * j + 1]))), r);
            out[j] = e4m3x4(lo_of(p0), hi_of(p0), lo_of(p1), hi_of(p1));
        }
    } else {
#pragma unroll
        for (int j = 0; j < NW / 2; ++j)
            out[j] = e4m3_pair(__uint_as_float(bf16x2_lo(w[2 * j])), __uint_as_float(bf16x2_hi(w[2 * j])), g) |
                     (e4m3_pair(__uint_as_float(bf16x2_lo(w[2 * j + 1])), __uint_as_float(bf16x2_hi(w[2 * j + 1])), g)
                      << 16);
    }
}

// N binary32 values (consecutive in the output row) -> N E4M3 codes (N/4 words), the
// same arithmetic as codes_words for values that are not BF16.
template <int N>
__device__ __forceinline__ void codes_f32(const float *x, const GroupScale &g, uint32_t *out)
{
    if (g.mode == 0) {
        const unsigned long long nr = pack2(-g.r, -g.r), s2 = pack2(g.s, g.s);
#pragma unroll
        for (int j = 0; j < N / 4; ++j) {
            const unsigned long long t0 = neg_quotient2(pack2(x[4 * j], x[4 * j + 1]), nr, s2);
            const unsigned long long t1 = neg_quotient2(pack2(x[4 * j + 2], x[4 * j + 3]), nr, s2);
            out[j] = e4m3x4(lo_of(t0), hi_of(t0), lo_of(t1), hi_of(t1)) ^ 0x80808080u;
        }
    } else if (g.mode == 1) {
        const unsigned long long r = pack2(g.r, g.r);
#pragma unroll
        for (int j = 0; j < N / 4; ++j) {
            const unsigned long long p0 = fmul2(pack2(x[4 * j], x[4 * j + 1]), r);
            const unsigned long long p1 = fmul2(pack2(x[4 * j + 2], x[4 * j + 3]), r);
            out[j] = e4m3x4(lo_of(p0), hi_of(p0), lo_of(p1), hi_of(p1));
        }
    } else {
#pragma unroll
        for (int j = 0; j < N / 4; ++j)
            out[j] = e4m3_pair(x[4 * j], x[4 * j + 1], g) | (e4m3_pair(x[4 * j + 2], x[4 * j + 3], g) << 16);
    }
}

// Sixteen BF16 values (8 words) -> sixteen E4M3 codes (one 16-byte chunk).
__device__ __forceinline__ uint4 codes16(const uint32_t *w, const GroupScale &g)
{
    uint32_t o[4];
    codes_words<8>(w, g, o);
    return make_uint4(o[0], o[1], o[2], o[3]);
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
// standalone quantizer -- into f.xq [M, K] and f.sx [K/128][M].  Each CTA takes one
// contiguous range of rows.  LPG consecutive lanes quantize one (row, 128-column group):
// the group's 16-byte chunks j = l + c * LPG go to lane l, so that each load instruction
// reads LPG * 16 contiguous bytes per group, and the group's max-abs is combined by
// shuffles across the LPG lanes.  Lanes handle U groups per batch and load the next batch
// before converting the current one.  When its range is done the CTA publishes it by a
// fence and an atomic add to the ready count of every expert the range overlaps.
template <int U = 2>
__device__ __forceinline__ void quantize_rows_phase(const int *goff, int G, int64_t M, int KB, int64_t K,
                                                    const FuseArgs &f)
{
    constexpr int LPG = 4, CPL = 16 / LPG;
    const int r_begin = goff[0], r_end = goff[G];
    const int per_cta = (r_end - r_begin + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
    const int r0 = min(r_end, r_begin + static_cast<int>(blockIdx.x) * per_cta);
    const int r1 = min(r_end, r0 + per_cta);
    const int lg = threadIdx.x % LPG, slot = threadIdx.x / LPG, nslot = blockDim.x / LPG;
    const bool pow2 = f.pow2 != 0;
    // Group index gi = (row - r0) * KB + kb; batch j, slot u holds gi = j * step + u * nslot + slot,
    // so gi < (r1 - r0) * KB exactly when row < r1.  (row, kb) advance by step per batch.
    const int step = nslot * U, step_r = step / KB, step_k = step - step_r * KB;
    int lr[U], lk[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int gi = u * nslot + slot;
        lr[u] = r0 + gi / KB;
        lk[u] = gi - (gi / KB) * KB;
    }
    auto load = [&](uint4 (&v)[U][CPL]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint4 *src = reinterpret_cast<const uint4 *>(f.x + static_cast<int64_t>(lr[u]) * f.ldx + lk[u] * 128);
#pragma unroll
            for (int c = 0; c < CPL; ++c)
                v[u][c] = lr[u] < r1 ? __ldg(src + lg + c * LPG) : make_uint4(0, 0, 0, 0);
        }
    };
    const int nbatch = ((r1 - r0) * KB + step - 1) / step;
    uint4 v[U][CPL];
    load(v);
    for (int j = 0; j < nbatch; ++j) {
        int cr[U], ck[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            cr[u] = lr[u]; ck[u] = lk[u];
            lk[u] += step_k; lr[u] += step_r;
            if (lk[u] >= KB) { lk[u] -= KB; ++lr[u]; }
        }
        uint4 nx[U][CPL];
        load(nx);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint32_t w[4 * CPL];
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                w[4 * c + 0] = v[u][c].x; w[4 * c + 1] = v[u][c].y; w[4 * c + 2] = v[u][c].z; w[4 * c + 3] = v[u][c].w;
            }
            uint32_t m[4 * CPL];
#pragma unroll
            for (int i = 0; i < 4 * CPL; ++i)
                m[i] = w[i];
#pragma unroll
            for (int h = 2 * CPL; h > 0; h >>= 1)
#pragma unroll
                for (int i = 0; i < h; ++i)
                    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[i]) : "r"(m[i]), "r"(m[i + h]));
#pragma unroll
            for (int o = LPG / 2; o > 0; o >>= 1) {
                const uint32_t t = __shfl_xor_sync(0xFFFFFFFFu, m[0], o);
                asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[0]) : "r"(m[0]), "r"(t));
            }
            if (cr[u] < r1) {
                const uint32_t a = m[0] & 0x7FFF7FFFu;
                const GroupScale g =
                    make_group_scale(fmaxf(__uint_as_float(a << 16), __uint_as_float(a & 0xFFFF0000u)), pow2);
                uint8_t *dst = f.xq + static_cast<int64_t>(cr[u]) * K + ck[u] * 128;
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    uint32_t q[2];
                    codes_words<4>(&w[4 * c], g, q);
                    *reinterpret_cast<uint2 *>(dst + (lg + c * LPG) * 8) = make_uint2(q[0], q[1]);
                }
                if (lg == 0)
                    f.sx[static_cast<int64_t>(ck[u]) * M + cr[u]] = g.s;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int c = 0; c < CPL; ++c)
                v[u][c] = nx[u][c];
    }
    fence_proxy_async_global();   // the codes are read by TMA (async proxy)
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0 && r1 > r0) {
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

} // namespace mpq

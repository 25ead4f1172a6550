// quant_device.cuh -- the per-group arithmetic of the 1x128 / 128x1 / 128x128 quantizers,
// shared by the standalone quantizers and the grouped GEMM that quantizes its activations
// on the fly, so that both produce the same codes and scales bit for bit.
//
// A group's scale maps its max-abs value onto the largest E4M3 value (make_group_scale in
// mpq_device.cuh); each element becomes the E4M3 code of the correctly rounded binary32
// quotient x / s.
#pragma once
#include "mpq_device.cuh"

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

} // namespace mpq

// swiglu_device.cuh -- the binary32 SwiGLU arithmetic shared by the standalone SwiGLU
// quantizer (swiglu.cu) and the grouped GEMM's fused SwiGLU epilogue (gemm.cu), so that
// both compute silu(gate) * up with the same operations, bit for bit.
//
// silu(g) = g / (1 + e^-g) and x = silu(g) * u, each operation rounded once to binary32.
// e^x is a fixed sequence of binary32 operations: Cody and Waite's reduction (W. J. Cody,
// W. Waite, "Software Manual for the Elementary Functions", 1980) with a 15-bit head of
// ln 2, the degree-7 Taylor polynomial of e^r in Horner form with fused multiply-adds, and
// a scaling by 2^n with one rounding; every step uses an explicitly rounded intrinsic, so
// no contraction changes it.
#pragma once

#include "mpq_device.cuh"

namespace mpq {

// e^x0 and e^x1: clamp to [-104, 89] (below, e^x rounds to 0; above, it overflows),
// n = rint(x log2 e) with ties to even, r = x - n ln2 with ln2 split into a 15-bit head
// (n * head is exact) and a tail, the degree-7 Taylor polynomial of e^r in Horner form,
// then p * 2^n with one rounding.  The multiply-adds run as packed FP32x2 operations, each
// lane rounded exactly like a scalar fused multiply-add.
__device__ __forceinline__ void exp_cw2(float x0, float x1, float &e0, float &e1)
{
    x0 = fminf(fmaxf(x0, -104.0f), 89.0f);
    x1 = fminf(fmaxf(x1, -104.0f), 89.0f);
    const unsigned long long x = pack2(x0, x1);
    const unsigned long long t = fmul2(x, pack2(0x1.715476p+0f, 0x1.715476p+0f));
    const float nf0 = rintf(lo_of(t)), nf1 = rintf(hi_of(t));
    const unsigned long long nn = pack2(-nf0, -nf1);
    unsigned long long r = ffma2(nn, pack2(0x1.62e4p-1f, 0x1.62e4p-1f), x);
    r = ffma2(nn, pack2(0x1.7f7d1cp-20f, 0x1.7f7d1cp-20f), r);
    unsigned long long p = pack2(0x1.a01a02p-13f, 0x1.a01a02p-13f);
    p = ffma2(p, r, pack2(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));
    p = ffma2(p, r, pack2(0x1.111112p-7f, 0x1.111112p-7f));
    p = ffma2(p, r, pack2(0x1.555556p-5f, 0x1.555556p-5f));
    p = ffma2(p, r, pack2(0x1.555556p-3f, 0x1.555556p-3f));
    p = ffma2(p, r, pack2(0.5f, 0.5f));
    p = ffma2(p, r, pack2(1.0f, 1.0f));
    p = ffma2(p, r, pack2(1.0f, 1.0f));
    const int n[2] = {static_cast<int>(nf0), static_cast<int>(nf1)};
    const float pv[2] = {lo_of(p), hi_of(p)};
    float e[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        if (n[i] > 127)
            e[i] = __fmul_rn(__fmul_rn(pv[i], 0x1p64f), exp2_int(n[i] - 64));
        else if (n[i] < -126)
            e[i] = __fmul_rn(__fmul_rn(pv[i], exp2_int(n[i] + 64)), 0x1p-64f);
        else
            e[i] = __fmul_rn(pv[i], exp2_int(n[i]));
    }
    e0 = e[0];
    e1 = e[1];
}

// silu(g0) u0 and silu(g1) u1.
__device__ __forceinline__ void swiglu2(float g0, float g1, float u0, float u1, float &v0, float &v1)
{
    float e0, e1;
    exp_cw2(-g0, -g1, e0, e1);
    v0 = __fmul_rn(__fdiv_rn(g0, __fadd_rn(1.0f, e0)), u0);
    v1 = __fmul_rn(__fdiv_rn(g1, __fadd_rn(1.0f, e1)), u1);
}

} // namespace mpq

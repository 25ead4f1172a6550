// mpq_internal.h -- launchers shared between the C-ABI layer and the kernel files.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mpq {

// Quantizer arguments.  Tensors are read and written through TMA views encoded by the
// caller: the BF16 source [rows, cols] in 128-row x 64-column boxes, and the E4M3 outputs
// q [rows, cols] / qT [cols, rows] in 128 x 128-byte boxes, all with 128-byte swizzle.
struct QuantArgs {
    int64_t rows, cols;
    uint8_t *q;         // row-wise (or block) codes [rows, cols] (may be null for the dual kernel)
    int64_t ldq;
    float *s;           // row-wise scales [cols/128][lds] or block scales [rows/128][lds]
    int64_t lds;
    uint8_t *qT;        // transposed codes [cols, rows] (optional)
    int64_t ldqT;
    float *sT;          // column-group scales [rows/128][ldsT]
    int64_t ldsT;
    int *status;        // device status word
    uint64_t timeout_ns;
};

// Re-quantization of a cached 1x128 quantization into 128x1 groups (codes travel by TMA).
struct RequantArgs {
    int64_t rows, cols;   // of the input codes [rows, cols]; both multiples of 128
    const float *s;       // input scales [cols/128][lds]
    int64_t lds;
    float *sT;            // output scales [rows/128][ldsT]
    int64_t ldsT;
    int *status;
    uint64_t timeout_ns;
};

cudaError_t launch_requant(const CUtensorMap &tmq, const CUtensorMap &tmqT, const RequantArgs &a, bool pow2,
                           int num_sms, cudaStream_t st);

// SwiGLU of [rows, 2*width] BF16 (gate | up) and the 1x128 quantization of the result.
struct SwigluArgs {
    const uint16_t *h;        // BF16 bits [rows][ldh]: gate in columns [0, width), up in [width, 2 width)
    int64_t rows, width, ldh;
    uint8_t *q;               // [rows][ldq]
    int64_t ldq;
    float *s;                 // [width/128][lds]
    int64_t lds;
};

cudaError_t launch_swiglu_quant(const SwigluArgs &a, bool pow2, int num_sms, cudaStream_t st);

cudaError_t launch_quant_rows(const CUtensorMap &tmx, const CUtensorMap &tmq, const QuantArgs &a, bool pow2,
                              int num_sms, cudaStream_t st);
cudaError_t launch_quant_dual(const CUtensorMap &tmx, const CUtensorMap &tmq, const CUtensorMap &tmqT,
                              const QuantArgs &a, bool pow2, int num_sms, cudaStream_t st);
cudaError_t launch_quant_block(const CUtensorMap &tmx, const CUtensorMap &tmq, const CUtensorMap &tmqT,
                               const QuantArgs &a, bool pow2, int num_sms, cudaStream_t st);

// Which B-side scale layout the GEMM reads (see fp8_gemm_blockscaled in mpq.h).
enum ScaleB : int { kScaleBlockNK = 0, kScaleBlockKN = 1, kScaleRowKN = 2 };

struct GemmArgs {
    int64_t M, N, K;            // rows of C, columns of C, reduction length
    const float *sA;            // [K/128][ldsa]
    int64_t ldsa;
    const float *sB;
    int64_t ldsb;
    int64_t sb_group_stride;    // elements between experts' B scales (grouped)
    void *C;
    int64_t ldc;
    const int64_t *offsets;     // grouped: device [G+1] row offsets, else null
    int G;                      // grouped: number of experts, else 1
    int *status;                // device status word (2 ints)
    uint64_t timeout_ns;
    // Stream-K schedule (dense GEMMs): when sk_part is set, the 128-K slices of all tiles
    // are split evenly over the CTAs (pairs); a tile begun by one and finished by the
    // previous one is completed with the partial the first wrote into sk_part, announced
    // by its sk_flags entries reaching sk_epoch.
    float4 *sk_part;            // [units][2][8 warps][32][32] float4
    int *sk_flags;              // [units][2][8 warps]
    int sk_epoch;
    // Tile order: with n_fastest the output tiles of one row strip follow each other (each
    // strip of A is read once while B stays in L2), else those of one column strip (each
    // strip of B read once).  Dense GEMMs take the smaller operand as the one re-read;
    // grouped GEMMs decide per expert (n-fastest when its rows outnumber its weight rows).
    int n_fastest;
    // Grouped GEMMs: only experts with min_rows <= rows < max_rows are computed by this launch
    // (the others' rows are left to another launch); 0 and INT32_MAX take every expert.
    int min_rows = 0, max_rows = 0x7FFFFFFF;
    // Fused SwiGLU epilogue (grouped up projection, the input of the down projection): B rows
    // [0, W) of each expert are the gate weights and [W, 2 W) the up weights (N = 2 W); an
    // output tile covers columns [n0, n0 + 128) of x = silu(gate) * up, staging gate and up
    // side by side in the MMA's 256 columns.  Written: the 1x128 quantization of x, codes
    // sw_q [M][sw_ldq] and scales sw_s [W/128][sw_lds] (power-of-2 scales when sw_pow2), and,
    // when C is not null, the BF16 gate and up values in C [M][ldc >= 2 W] (the cached
    // SwiGLU input).
    uint8_t *sw_q;
    int64_t sw_ldq;
    float *sw_s;
    int64_t sw_lds;
    int sw_width;
    int sw_pow2;
};

// Fused activation quantization: the token rows come as BF16 x [M, K] (ldx elements) and
// are quantized 1x128 into the workspace (xq [M, K] codes, sx [K/128][M] scales, ready[G]
// counts, cleared by the launcher) inside the same launch; tmX must then cover xq and
// GemmArgs.sA / ldsa must be sx / M.
struct FuseArgs {
    const uint16_t *x;
    int64_t ldx;
    uint8_t *xq;
    float *sx;
    int *ready;
    int pow2;
};

// Block-scaled FP8 GEMM on tcgen05: C[M,N] = sum over 128-wide K slices of
// (A_slice B_slice^T) * sA * sB, promoted into FP32 after every slice.
// tmA covers A [rows, K] E4M3, tmB covers B [rows, K] E4M3 (both K-major, 128B swizzle).
// `pair`: 2-CTA clusters computing 256 x 256 tiles with 2-SM MMAs (cta_group::2); each CTA
// loads its own 128 rows of A and half of the tile's B rows, in boxes of
// gemm_b_box_rows(true) = 128 rows, else 256.
// tmC: output view [rows, N] (BF16 or FP32), boxes of 32 rows x 128 bytes with 128-byte
// swizzle in pair mode, 32 rows x 64 bytes with 64-byte swizzle single-SM.
// fuse != null: grouped GEMM with fused 1x128 activation quantization (single-SM tiles,
// weight block scales): tmA must cover fuse->xq, a.sA / a.ldsa must be fuse->sx / M.
cudaError_t launch_gemm(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC, const GemmArgs &a,
                        int scale_b, bool out_fp32, bool pair, int num_sms, cudaStream_t st,
                        const FuseArgs *fuse = nullptr);
// The grouped GEMM with the SwiGLU epilogue (a.sw_q set): weight block scales, tmB in boxes of
// 128 rows, tmC unused (the BF16 gate / up values are stored directly when a.C is set).
cudaError_t launch_gemm_swiglu(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &a, bool pair,
                               int num_sms, cudaStream_t st, const FuseArgs *fuse = nullptr);
int gemm_b_box_rows(bool pair);

// The same GEMM for power-of-2 scales on the microscaling MMA (kind::mxf8f6f4.block_scale):
// 2-SM pair tiles of 256 x 256, tmA / tmB in boxes of 128 rows, tmC in boxes of 32 rows x
// 64 bytes with 64-byte swizzle.
cudaError_t launch_gemm_mx(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC, const GemmArgs &a,
                           int scale_b, bool out_fp32, int num_sms, cudaStream_t st);

// Grouped GEMM for few tokens per expert (weights as the MMA's M operand, tokens as N):
// tmX covers the token codes [M, K] in boxes of decode_x_box_rows() rows, tmW the expert
// weights [G*N, K] in boxes of 128 rows (both K-major, 128-byte swizzle).  Same GemmArgs as
// the grouped launch_gemm (sB block scales [G][N/128][ldsb]); C is written directly.
int decode_x_box_rows();
cudaError_t launch_decode(const CUtensorMap &tmX, const CUtensorMap &tmW, const GemmArgs &a, bool out_fp32,
                          const FuseArgs *fuse, int num_sms, cudaStream_t st);

// Self-test of the bounded wait: one CTA waits on a barrier nobody arrives on.
cudaError_t launch_wait_selftest(int *status, uint64_t timeout_ns, cudaStream_t st);

// Size of the fixed scratch area of fp8_grouped_gemm_fused_quant_noalloc (MPQ_NOALLOC_SCRATCH_BYTES),
// and its device address on the current device (looked up on first use, then cached).
constexpr size_t kNoallocScratchBytes = size_t(64) << 20;
cudaError_t noalloc_scratch(void **ptr);

// Dynamic shared memory above 48 KB is enabled per kernel and per device (the attribute
// belongs to the kernel's module in that device's context).  `done` caches, one bit per
// device (devices 0..63; others set the attribute on every call), that it has been set.
template <class Kern>
cudaError_t ensure_max_dyn_smem(Kern kern, size_t smem, std::atomic<uint64_t> &done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? uint64_t(1) << dev : 0;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0)
        return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess && bit != 0)
        done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

} // namespace mpq

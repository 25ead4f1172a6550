/*
 * mpq.h -- C ABI of libmpq: fine-grained FP8 (E4M3) quantization and block-scaled
 * FP8 GEMM for NVIDIA B300 (sm_103a), one GPU, one process.
 *
 * The method is the fine-grained FP8 mixed-precision scheme of an MoE transformer's
 * training framework as described by the source pages (scraped copies of its technical
 * report):
 *   - page 1 (second paragraph): the scaling factor is derived from the online max-abs
 *     value and activations or weights are quantized online into FP8; the FP8 GEMMs
 *     accept FP8 tensors and produce BF16 or FP32 outputs; activations are cached in FP8
 *     for the backward pass;
 *   - page 2, "9 Amazing Deepseek Hacks" (last paragraph): groups of 128 activation
 *     values; in the backward pass the matrix is read, transposed and re-quantized into
 *     128x1 tiles;
 *   - page 3 (first paragraph): the max-abs value is scaled to the largest FP8 value;
 *   - page 4 (first paragraph): partial sums are promoted every 128 elements of K and
 *     accumulated in full FP32; (second paragraph): Fprop, Dgrad and Wgrad all run in
 *     FP8, with integral power-of-2 scaling factors for some activations;
 *   - page 4 (third paragraph): during decoding the batch per expert is small (usually
 *     within 256 tokens) and the expert GEMM is bound by memory access.
 * E4M3 is the OCP FP8 format (bias 7, no infinities, largest finite value 448).
 *
 * Conventions for every call
 *   - Every pointer except the handle is a DEVICE pointer owned by the caller; the
 *     library never frees or retains it after the call returns.
 *   - Matrices are row-major; ld* is the row stride in ELEMENTS of that array.
 *   - BF16 inputs are passed as `const void *` (16-bit bfloat16 elements).
 *   - E4M3 codes are bytes; scales are float32.
 *   - `stream` is a cudaStream_t (passed as void *); every call only enqueues work on
 *     it and returns without synchronizing.  The device the handle was created on must be
 *     current (else MPQ_ERR_DEVICE, before any launch).
 *   - Arguments are validated on the host before anything is launched; a validation
 *     failure returns a status code and leaves all outputs untouched.
 *   - Device-side waits are bounded (about one second by default).  A wait that runs
 *     out records MPQ_ERR_TIMEOUT in the handle's device status word and the kernel
 *     exits cleanly; mpq_check_device_status() reports it.
 */
#ifndef MPQ_H
#define MPQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mpq_status {
    MPQ_OK = 0,
    MPQ_ERR_NULL = 1,        /* a required pointer is NULL                                */
    MPQ_ERR_SHAPE = 2,       /* a size or leading dimension is invalid                    */
    MPQ_ERR_ALIGN = 3,       /* a pointer or stride breaks the 16-byte (or 4-byte) rule    */
    MPQ_ERR_UNSUPPORTED = 4, /* unknown op, dtype or flag combination                     */
    MPQ_ERR_CUDA = 5,        /* a CUDA runtime / driver call failed                       */
    MPQ_ERR_TIMEOUT = 6,     /* a device-side wait ran out (reported by the status word)  */
    MPQ_ERR_WORKSPACE = 7,   /* no workspace set on the handle, or it is too small        */
    MPQ_ERR_DEVICE = 8,      /* the current CUDA device is not the one the handle was
                                created on (nothing was launched)                         */
    MPQ_ERR_SCALE = 9        /* a scale given to fp8_gemm_mx_pow2 is not a power of 2 in
                                2^-127 .. 2^127 (found on the device, reported by the
                                status word; that call's output is not valid)             */
} mpq_status;

typedef enum mpq_op {
    MPQ_OP_FPROP = 0, /* sB: 128x128 weight blocks, layout [N/128][ldsb >= K/128]        */
    MPQ_OP_DGRAD = 1, /* sB: 128x128 weight blocks seen through the transposed weight,
                         layout [K/128][ldsb >= N/128]                                   */
    MPQ_OP_WGRAD = 2  /* sB: 128x1 token tiles of B, layout [K/128][ldsb >= N]           */
} mpq_op;

typedef enum mpq_dtype {
    MPQ_OUT_BF16 = 0,
    MPQ_OUT_FP32 = 1
} mpq_dtype;

/* Flags */
#define MPQ_POW2 1u /* power-of-2 scales: s = 2^e, e the smallest integer with amax <= 448*2^e */
#define MPQ_GROUPED_ROW_TILES 2u    /* grouped GEMM: tiles of token rows (many tokens per expert) */
#define MPQ_GROUPED_WEIGHT_TILES 4u /* grouped GEMM: tiles of weight rows (few tokens per expert) */
#define MPQ_FUSE_QUANT_A 8u         /* grouped GEMM: A is BF16, quantized 1x128 inside the launch */

typedef struct mpq_handle_s *mpq_handle;

/* Library version string, e.g. "mpq 0.1.0 sm_103a". */
const char *mpq_version(void);

/* Human-readable text of a status code (static storage). */
const char *mpq_status_string(int status);

/* Create a handle bound to the current CUDA device.  Allocates (cudaMalloc, here and
 * nowhere else) the 8-byte device status word and the stream-K handover area of the dense
 * GEMM (128 KB per SM plus 32 bytes per SM of flags), and caches the SM count.  Not
 * thread-safe per handle; dense GEMMs that take the stream-K schedule through one handle
 * share its handover area and must not run concurrently (issue them on one stream). */
mpq_status mpq_create(mpq_handle *out);

/* Destroy a handle and free its device memory.  Synchronizes the handle's device first
 * (making it current for the call, then restoring the caller's current device). */
mpq_status mpq_destroy(mpq_handle h);

/* Limit for every device-side wait launched through this handle, in nanoseconds
 * (default 1e9).  0 restores the default. */
mpq_status mpq_set_wait_timeout(mpq_handle h, uint64_t timeout_ns);

/* Tiling of the row-tiled GEMMs issued through this handle.
 *   pair tiles: a 2-CTA cluster on two SMs computes a 256 x 256 tile with 2-SM MMAs (each
 *     SM stages its 128 A rows and half of the B rows);
 *   single-SM tiles: one CTA computes a 128 x 256 tile.
 * mode 1 (default): pair tiles for fp8_gemm_blockscaled; the row-tiled grouped GEMMs
 * (fp8_grouped_gemm_blockscaled, fp8_grouped_gemm_swiglu_quant) give pair tiles to the
 * experts with 1024 token rows or more and single-SM tiles to the others (each expert's rows
 * are rounded up to whole tiles, and a 256-row tile wastes more on a small expert): two
 * launches on the caller's stream, each computing only its experts' rows.
 * mode 0: single-SM tiles everywhere.  mode 2: pair tiles everywhere.  Other values:
 * MPQ_ERR_UNSUPPORTED.  The tilings give bit-identical results (with stream-K off). */
mpq_status mpq_set_gemm_cta_pair(mpq_handle h, int enable);

/* Schedule of fp8_gemm_blockscaled and fp8_gemm_mx_pow2 through this handle (a throughput
 * choice; the pages' method is the same).  Data-parallel: each CTA (pair) takes whole output tiles.  Stream-K:
 * the 128-K slices of all tiles are split evenly over the CTAs (pairs); a tile shared by
 * two of them is finished by the one holding its first slices, which adds the other's
 * partial sum (FP32, through the handle's handover area) before the store, so the last
 * wave has no idle SMs.  Results are deterministic for a given shape and device, and equal
 * the data-parallel ones up to the FP32 rounding of that one addition per shared tile.
 * mode 1 (default): stream-K when the tiles fill more than one wave and the last wave
 * would leave more than a tenth of the machine idle; mode 0: never; mode 2: whenever the
 * tiles fill more than one wave.  Other values: MPQ_ERR_UNSUPPORTED. */
mpq_status mpq_set_gemm_stream_k(mpq_handle h, int mode);

/*
 * mpq_set_workspace -- hands the handle a caller-owned device buffer for calls that need
 * scratch memory (today: fp8_grouped_gemm_blockscaled with MPQ_FUSE_QUANT_A, which keeps
 * the quantized activations there).  The library never allocates it, frees it or keeps
 * it past mpq_destroy; ptr must be 256-byte aligned and stay valid while calls that use it
 * are in flight.  Calls on one handle that use the workspace must not overlap (on
 * different streams) -- they share it.  ptr = NULL, bytes = 0 removes it.
 */
mpq_status mpq_set_workspace(mpq_handle h, void *ptr, size_t bytes);

/*
 * mpq_grouped_fused_workspace_bytes -- workspace bytes fp8_grouped_gemm_blockscaled needs
 * with MPQ_FUSE_QUANT_A for M_total token rows, reduction length K and G experts:
 * M_total*K codes + (K/128)*M_total scales + G counters, each part 256-byte aligned.
 */
mpq_status mpq_grouped_fused_workspace_bytes(int64_t M_total, int64_t K, int64_t G, size_t *bytes);

/* Synchronize `stream`, read and clear the device status word.  Returns MPQ_OK or the
 * recorded error (MPQ_ERR_TIMEOUT); *where_out (may be NULL) receives the tag of the
 * wait that gave up (role << 8 | barrier index), 0 if none. */
mpq_status mpq_check_device_status(mpq_handle h, void *stream, int *where_out);

/*
 * fp8_quant_tile_1x128 -- activation quantization in 1x128 tiles (page 1, second
 * paragraph; page 2, last paragraph; page 3, first paragraph), with an optional fused
 * 128x1 (along-rows) quantization written transposed for the Wgrad operand (page 2,
 * last paragraph: re-quantized into 128x1 tiles).
 *
 *   x    [rows, cols] BF16, ldx >= cols.
 *   Row-wise output (skipped when q == NULL; then s is ignored):
 *        q [rows, cols] E4M3, ldq >= cols;
 *        s [cols/128][lds] float32, lds >= rows: s[kb*lds + r] is the scale of
 *          x[r, kb*128 .. kb*128+127].
 *   Transposed output (only when qT != NULL):
 *        qT [cols, rows] E4M3, ldqT >= rows: qT[c, r] is the code of x[r, c] within the
 *          group x[rb*128 .. rb*128+127, c], rb = r/128;
 *        sT [rows/128][ldsT] float32, ldsT >= cols: sT[rb*ldsT + c].
 *   flags: 0 or MPQ_POW2.
 * Each group: amax = max |x|; s = amax/448 as one binary32 division (1.0 when amax is 0)
 * or the power of 2 above; code = E4M3 round-to-nearest-even of the binary32 quotient
 * x/s, saturating at +-448; zero keeps its sign.
 * Requirements: cols % 128 == 0; rows % 128 == 0 when qT != NULL; rows >= 0.
 * x, q, qT 16-byte aligned; ldx % 8 == 0; ldq and ldqT % 16 == 0; s, sT 4-byte aligned.
 * At least one of q, qT must be non-NULL.
 */
mpq_status fp8_quant_tile_1x128(mpq_handle h, const void *x, int64_t rows, int64_t cols, int64_t ldx,
                                uint8_t *q, int64_t ldq, float *s, int64_t lds,
                                uint8_t *qT, int64_t ldqT, float *sT, int64_t ldsT,
                                uint32_t flags, void *stream);

/*
 * fp8_requant_tile_128x1 -- re-quantization of a cached FP8 activation into 128x1 groups
 * (page 2, last paragraph: in the backward pass the FP8 matrix is read out, dequantized,
 * transposed and re-quantized into 128x1 tiles; page 1, second paragraph: activations are
 * cached in FP8 for the backward pass).  The input is what fp8_quant_tile_1x128 writes;
 * the output has the layout of its transposed part, so it feeds the Wgrad GEMM directly.
 *
 *   q  [rows, cols] E4M3, ldq >= cols (device, read only);
 *   s  [cols/128][lds] float32, lds >= rows: s[kb*lds + r] scales q[r, kb*128 .. +127];
 *   qT [cols, rows] E4M3, ldqT >= rows (device, written);
 *   sT [rows/128][ldsT] float32, ldsT >= cols (device, written).
 *   flags: 0 or MPQ_POW2 (the scale rule of the output groups).
 * Each element is dequantized to binary32 as dec(q) * s (one rounded product); the values
 * x[rb*128 .. rb*128+127, c] form one group, quantized as fp8_quant_tile_1x128 quantizes
 * its groups: qT[c, r] is the code of x[r, c], sT[rb*ldsT + c] the group's scale.  A
 * positive max-abs value never gives a scale below 2^-149 (the smallest positive
 * binary32): a smaller power of 2, or a quotient amax/448 that rounds to 0, is raised to
 * it (BF16 inputs never reach this; dequantized FP8 values can).  The dequantized values
 * must be finite, as they are for any codes and scales fp8_quant_tile_1x128 writes.
 * Requirements: rows % 128 == 0, cols % 128 == 0, rows >= 0; q, qT, s 16-byte aligned;
 * ldq, ldqT % 16 == 0; lds % 4 == 0; sT 4-byte aligned (pointers and alignment are not
 * checked when rows == 0: then nothing is read or written).  The input and output must not overlap.  Asynchronous on
 * `stream`; nothing is allocated.
 */
mpq_status fp8_requant_tile_128x1(mpq_handle h, const uint8_t *q, int64_t rows, int64_t cols, int64_t ldq,
                                  const float *s, int64_t lds, uint8_t *qT, int64_t ldqT, float *sT,
                                  int64_t ldsT, uint32_t flags, void *stream);

/*
 * fp8_swiglu_quant_1x128 -- SwiGLU of the MoE up-projection output fused with the 1x128
 * quantization of the result, the FP8 input of the down projection (page 1, first
 * paragraph: the SwiGLU output is recomputed from its cached inputs; page 4, second
 * paragraph: this activation uses integral power-of-2 scales, flag MPQ_POW2).
 *
 *   hcat [rows, 2*width] BF16, ldh >= 2*width: hcat[r, c] is the gate and hcat[r, width + c]
 *        the up value of output element (r, c) (device, read only);
 *   q    [rows, width] E4M3, ldq >= width (device, written);
 *   s    [width/128][lds] float32, lds >= rows: s[kb*lds + r] scales q[r, kb*128 .. +127].
 *   flags: MPQ_POW2 (the pages' rule for this activation) or 0 (amax/448).
 * x = silu(g) * u with silu(g) = g / (1 + e^-g), every operation in binary32 with one
 * rounding; e^x is a fixed operation sequence (Cody-Waite reduction, degree-7 Taylor
 * polynomial by fused multiply-adds, scaled by 2^n with one rounding; within 2 ulp of the
 * true exponential), so results are reproducible bit for bit.  Where e^-g overflows
 * (g below about -88.7) silu gives -0.  The groups of x are quantized as
 * fp8_quant_tile_1x128 quantizes its groups; every product x must be finite.
 * Requirements: width % 128 == 0, rows >= 0; hcat, q 16-byte aligned; ldh % 8 == 0;
 * ldq % 16 == 0; s 4-byte aligned.  Asynchronous on `stream`; nothing is allocated.
 */
mpq_status fp8_swiglu_quant_1x128(mpq_handle h, const void *hcat, int64_t rows, int64_t width, int64_t ldh,
                                  uint8_t *q, int64_t ldq, float *s, int64_t lds, uint32_t flags, void *stream);

/*
 * fp8_quant_block_128x128 -- weight quantization in 128x128 blocks (page 1, second
 * paragraph: weights are quantized online from their max-abs value), optionally also
 * writing the transposed codes (same scales) used as the Dgrad B operand.
 *
 *   w  [rows, cols] BF16, ldw >= cols;
 *   q  [rows, cols] E4M3, ldq >= cols;
 *   qT [cols, rows] E4M3 or NULL, ldqT >= rows: qT[c, r] == q[r, c];
 *   s  [rows/128][lds] float32, lds >= cols/128: s[i*lds + j] scales block (i, j).
 *   flags: 0 or MPQ_POW2.
 * Requirements: rows % 128 == 0, cols % 128 == 0; w, q, qT 16-byte aligned; ldw % 8 == 0;
 * ldq, ldqT % 16 == 0; s 4-byte aligned.
 */
mpq_status fp8_quant_block_128x128(mpq_handle h, const void *w, int64_t rows, int64_t cols, int64_t ldw,
                                   uint8_t *q, int64_t ldq, uint8_t *qT, int64_t ldqT,
                                   float *s, int64_t lds, uint32_t flags, void *stream);

/*
 * fp8_gemm_blockscaled -- block-scaled FP8 GEMM with 128-element FP32 promotion
 * (page 4, first paragraph; page 1, second paragraph; page 4, second paragraph: Fprop,
 * Dgrad and Wgrad in FP8):
 *
 *   C[m, n] = sum_kb ( sum_{k = 128 kb}^{128 kb + 127} A[m,k] B[n,k] ) * sA[kb*ldsa + m] * sB(n, kb)
 *
 *   A  [M, K] E4M3, lda >= K (K-major);   sA [K/128][ldsa] float32, ldsa >= M.
 *   B  [N, K] E4M3, ldb >= K (K-major);   sB per `op`:
 *        MPQ_OP_FPROP  sB[(n/128)*ldsb + kb]  (weight blocks; B = the quantized weight)
 *        MPQ_OP_DGRAD  sB[kb*ldsb + n/128]    (weight blocks of the weight whose
 *                                              transposed codes are B)
 *        MPQ_OP_WGRAD  sB[kb*ldsb + n]        (128x1 token tiles written transposed)
 *   C  [M, N] BF16 (out = MPQ_OUT_BF16, round to nearest even) or FP32, ldc >= N.
 * Within a 128-K slice the products are summed by the tensor cores in FP32; each slice
 * is then scaled and added into an FP32 accumulator.
 * Requirements: M >= 0, N % 128 == 0, K % 128 == 0, K > 0; A, B, C 16-byte aligned;
 * lda, ldb % 16 == 0; ldc * sizeof(out) % 16 == 0; sA, sB 4-byte aligned.
 */
mpq_status fp8_gemm_blockscaled(mpq_handle h, int op, int64_t M, int64_t N, int64_t K,
                                const uint8_t *A, int64_t lda, const float *sA, int64_t ldsa,
                                const uint8_t *B, int64_t ldb, const float *sB, int64_t ldsb,
                                void *C, int64_t ldc, int out_dtype, void *stream);

/*
 * fp8_gemm_mx_pow2 -- the block-scaled FP8 GEMM of fp8_gemm_blockscaled for operands whose
 * scales are all integral powers of 2 (page 4, second paragraph), with the scales applied
 * by the tensor cores' microscaling MMA (page 3, first paragraph: the tensor cores of this
 * GPU generation support microscaling formats with small quantization groups):
 * tcgen05.mma kind::mxf8f6f4.block_scale with UE8M0 scale factors, one per 32-element K
 * block (each 128-K slice's scale repeated over its four blocks).  The MMAs accumulate the
 * scaled products of the whole K in FP32 in TMEM, so no slice is promoted by CUDA-core
 * FMAs: with power-of-2 scales each scaled product is exact, and the per-slice promotion of
 * the software path becomes part of the tensor cores' FP32 accumulation.
 *
 *   Same arguments, layouts, ops (MPQ_OP_FPROP / DGRAD / WGRAD), output types and
 *   requirements as fp8_gemm_blockscaled, and the same sum.
 *   Every scale read (sA for rows < M, sB for columns < N) must be a power of 2 between
 *   2^-127 and 2^127 -- as the quantizers write with MPQ_POW2 for any group whose max-abs
 *   value is at least 2^-119 (smaller nonzero groups get smaller scales).  The kernel checks
 *   each scale; one that is not representable records MPQ_ERR_SCALE in the handle's status
 *   word (mpq_check_device_status) and the output of that call is not valid.
 * Tiling: 2-SM pair tiles of 256 x 256 (mpq_set_gemm_cta_pair does not apply); the
 * schedule follows mpq_set_gemm_stream_k as fp8_gemm_blockscaled does (stream-K when the
 * last wave of tiles would be short), sharing the handle's handover area.  Results agree with
 * fp8_gemm_blockscaled within the GEMM tolerance of the method, not bit for bit (the FP32
 * sums are rounded in another order).  Asynchronous on `stream`; nothing is allocated.
 */
mpq_status fp8_gemm_mx_pow2(mpq_handle h, int op, int64_t M, int64_t N, int64_t K,
                            const uint8_t *A, int64_t lda, const float *sA, int64_t ldsa,
                            const uint8_t *B, int64_t ldb, const float *sB, int64_t ldsb,
                            void *C, int64_t ldc, int out_dtype, void *stream);

/*
 * fp8_grouped_gemm_blockscaled -- MoE expert GEMMs (page 2, first paragraph: large
 * per-expert batches in training; page 4, third paragraph: small per-expert batches in
 * decoding), Fprop scaling per expert:
 *
 *   for g in [0, G): rows [off[g], off[g+1]) of A and C use weight B_g:
 *   C[m, n] = sum_kb (sum_k A[m,k] B_g[n,k]) * sA[kb*ldsa + m] * sB_g[(n/128)*ldsb + kb]
 *
 *   d_offsets  DEVICE int64 [G+1], non-decreasing, 0 <= off[g] <= M_total (the kernel
 *              clamps into this range; rows outside every expert are not written).
 *   A          [M_total, K] E4M3, lda >= K;  sA [K/128][ldsa] float32, ldsa >= M_total.
 *   B          [G][N][K] E4M3 (expert g at B + g*N*ldb), ldb >= K.
 *   sB         [G][N/128][ldsb] float32 (expert g at sB + g*(N/128)*ldsb), ldsb >= K/128.
 *   C          [M_total, N] BF16 or FP32, ldc >= N.
 *   flags      0, MPQ_GROUPED_ROW_TILES or MPQ_GROUPED_WEIGHT_TILES: the tiling (below);
 *              MPQ_FUSE_QUANT_A (optionally with MPQ_POW2): fused activation quantization
 *              (below).
 * Two tilings compute the same sums:
 *   row tiles     tiles of 256 (or 128) token rows x 256 features, for experts with many
 *                 tokens (prefill, training);
 *   weight tiles  one 128-row block of an expert's weight against all of the expert's
 *                 tokens (up to 256 per tile), the MMA sized to the token count.
 * With flags 0 the library takes row tiles: on single-SM tiles (see mpq_set_gemm_cta_pair)
 * they stream the weights at the HBM rate even for a few tokens per expert, faster than
 * weight tiles on this hardware.  The two tilings may differ in the last bits of the FP32
 * accumulation (both are within the GEMM tolerance of the method).
 * Fused activation quantization (MPQ_FUSE_QUANT_A; page 4, third paragraph: decoding;
 * page 2, third paragraph after the title: the FP8 cast on the way into the GEMM): A is
 * then BF16 [M_total, K] with lda >= K in elements (16-byte aligned rows), sA must be NULL
 * and ldsa is ignored.  One launch quantizes every expert row 1x128 exactly as
 * fp8_quant_tile_1x128 does (amax/448 scales, or power-of-2 with MPQ_POW2) into the
 * handle's workspace (mpq_set_workspace, mpq_grouped_fused_workspace_bytes), then runs
 * the row-tile GEMM (single-SM tiles) on those codes -- or the weight-tile GEMM with
 * MPQ_GROUPED_WEIGHT_TILES; the output equals fp8_quant_tile_1x128 followed by this call
 * on the same tiling, bit for bit.  The fused launch is cooperative: its GEMM phase waits
 * for the quantization phase of every CTA, so all of its CTAs (one per SM) must be
 * resident at once, and the call fails with MPQ_ERR_CUDA when the cooperative launch is
 * refused (e.g. other work occupies SMs).
 * Returns MPQ_ERR_WORKSPACE without a workspace of sufficient size.
 * Requirements: 1 <= G <= 1024; N % 128 == 0; K % 128 == 0; alignment as for
 * fp8_gemm_blockscaled.
 */
mpq_status fp8_grouped_gemm_blockscaled(mpq_handle h, int64_t G, const int64_t *d_offsets,
                                        int64_t M_total, int64_t N, int64_t K,
                                        const uint8_t *A, int64_t lda, const float *sA, int64_t ldsa,
                                        const uint8_t *B, int64_t ldb, const float *sB, int64_t ldsb,
                                        void *C, int64_t ldc, int out_dtype, uint32_t flags,
                                        void *stream);

/*
 * fp8_grouped_gemm_swiglu_quant -- the MoE up projection with SwiGLU and the quantization of
 * its result in the GEMM's epilogue: the FP8 input of the down projection leaves the GEMM
 * directly, without the BF16 round trip through HBM (page 2, "9 Amazing Deepseek Hacks",
 * the paragraphs on fusing the FP8 cast with the memory transfer: activations are read from
 * HBM for quantization and written back only to be read again; page 1, first paragraph:
 * the SwiGLU operator's inputs are cached and its output recomputed in the backward pass;
 * page 4, second paragraph: this activation uses integral power-of-2 scales).
 *
 *   for expert g, rows m in [off[g], off[g+1]):
 *     H[m, c]     = bf16( sum_kb (A_kb B_g[c]_kb^T) sA sB )        gate, c in [0, W)
 *     H[m, W + c] = bf16( same with B_g[W + c] )                    up
 *     x[m, c]     = silu(H[m, c]) * H[m, W + c]                     (as fp8_swiglu_quant_1x128)
 *     q, s        = the 1x128 quantization of x (MPQ_POW2: power-of-2 scales)
 *
 *   d_offsets, G, M_total, K, A, lda, sA, ldsa, B, ldb, sB, ldsb as for
 *              fp8_grouped_gemm_blockscaled with N = 2 W: B [G][2W][K] holds each expert's
 *              gate weight rows [0, W) and up weight rows [W, 2W); sB [G][2W/128][ldsb].
 *   H          BF16 [M_total, 2W], ldh >= 2W (device, written) or NULL: the SwiGLU input,
 *              the values fp8_grouped_gemm_blockscaled would write with BF16 output (cached
 *              for the backward pass's recomputation); not written when NULL.
 *   q          [M_total, W] E4M3, ldq >= W (device, written);
 *   s          [W/128][lds] float32, lds >= M_total (device, written).
 *   flags      MPQ_POW2: power-of-2 scales for x (the pages' rule), else amax/448;
 *              MPQ_FUSE_QUANT_A: A is BF16 [M_total, K] (lda in elements) quantized 1x128
 *              with amax/448 scales inside the launch, as with fp8_grouped_gemm_blockscaled
 *              (sA must be NULL; needs the handle's workspace; cooperative launch).
 * Rows outside every expert are not written.  The codes, scales and H equal those of
 * fp8_grouped_gemm_blockscaled (BF16 out, same tiling) followed by fp8_swiglu_quant_1x128,
 * bit for bit.  Tiling as for fp8_grouped_gemm_blockscaled's row tiles (see
 * mpq_set_gemm_cta_pair; single-SM tiles with MPQ_FUSE_QUANT_A).
 * Requirements: 1 <= G <= 1024; W % 128 == 0; K % 128 == 0; A, B, q, H 16-byte aligned;
 * lda, ldb, ldq % 16 == 0 (lda % 8 == 0 for BF16 A); ldh % 8 == 0; sA, sB, s 4-byte
 * aligned.  Asynchronous on `stream`; nothing is allocated.
 */
mpq_status fp8_grouped_gemm_swiglu_quant(mpq_handle h, int64_t G, const int64_t *d_offsets, int64_t M_total,
                                         int64_t W, int64_t K, const void *A, int64_t lda, const float *sA,
                                         int64_t ldsa, const uint8_t *B, int64_t ldb, const float *sB, int64_t ldsb,
                                         void *H, int64_t ldh, uint8_t *q, int64_t ldq, float *s, int64_t lds,
                                         uint32_t flags, void *stream);

/*
 * fp8_grouped_gemm_fused_quant_noalloc -- fp8_grouped_gemm_blockscaled with
 * MPQ_FUSE_QUANT_A (fused 1x128 quantization of BF16 token rows, row-tile GEMM) that
 * allocates no memory and needs no workspace.  The source pages have no counterpart; it
 * exists for callers that must not allocate device memory, or hand the library a
 * buffer, while they run -- e.g. a serving process that reserves all device memory at
 * start-up, or a latency-critical loop where an allocation (and the synchronisation it
 * can bring) is not acceptable.
 *
 * The quantized activations live in a fixed scratch area inside the library's device
 * code: MPQ_NOALLOC_SCRATCH_BYTES (64 MiB).  A call whose
 * mpq_grouped_fused_workspace_bytes(M_total, K, G) exceeds it is rejected with
 * MPQ_ERR_WORKSPACE before any launch (e.g. with K = 7168, up to about 9,000 token rows).
 *
 *   X       BF16 [M_total, K], ldx >= K elements, 16-byte aligned rows.
 *   flags   0 or MPQ_POW2 (power-of-2 activation scales).
 *   the other arguments as for fp8_grouped_gemm_blockscaled.
 * Results equal fp8_grouped_gemm_blockscaled with MPQ_FUSE_QUANT_A bit for bit.
 *
 * First call: the first call on each device (with that device current) looks up the
 * scratch area's address (cudaGetSymbolAddress, which may load the library's device code)
 * and caches it; make that first call before any stream capture.
 * Concurrency: there is one scratch area per device.  Calls that overlap in time -- on
 * different streams, or from several threads, including through several handles -- race
 * on it and corrupt each other's results; serialise them (calls on one stream are fine).
 * The per-expert counters in the scratch area are cleared on the call's stream before
 * the launch.
 */
#define MPQ_NOALLOC_SCRATCH_BYTES (64u << 20)
mpq_status fp8_grouped_gemm_fused_quant_noalloc(mpq_handle h, int64_t G, const int64_t *d_offsets,
                                                int64_t M_total, int64_t N, int64_t K,
                                                const void *X, int64_t ldx,
                                                const uint8_t *B, int64_t ldb, const float *sB, int64_t ldsb,
                                                void *C, int64_t ldc, int out_dtype, uint32_t flags,
                                                void *stream);

/*
 * mpq_selftest_wait_timeout -- launches one CTA that waits on a barrier nothing ever
 * arrives on, with the library's bounded wait and the given limit (nanoseconds).  The
 * wait must give up and record MPQ_ERR_TIMEOUT in the handle's status word; the
 * context stays usable.  Used to test device-side failure reporting without a fault.
 */
mpq_status mpq_selftest_wait_timeout(mpq_handle h, uint64_t timeout_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MPQ_H */

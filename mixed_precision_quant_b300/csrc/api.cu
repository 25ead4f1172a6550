// api.cu -- the C ABI of libmpq: handle, host-side validation, TMA descriptor
// encoding and launches.  See include/mpq.h for the contract of every entry point.
#include "mpq.h"
#include "mpq_internal.h"

#include <cstdint>
#include <cstring>
#include <new>
#include <cuda.h>
#include <cuda_runtime.h>

struct mpq_handle_s {
    int device;
    int num_sms;
    int *d_status;          // [0] code, [1] tag of the wait that gave up
    uint64_t timeout_ns;
    int pair_mode;          // 2-SM pair tiles: 0 never, 1 dense (+ grouped with large experts), 2 always
    void *workspace;        // caller-owned scratch (mpq_set_workspace), may be null
    size_t workspace_bytes;
    int sk_mode;            // stream-K for dense GEMMs: 0 never, 1 when the last wave is short, 2 always
    int sk_epoch;           // incremented per stream-K launch; flags equal to it are this launch's
    int *d_sk_flags;        // [num_sms][8] handover flags
    float4 *d_sk_part;      // [num_sms][8][32][32] handover partials (128 KB per SM)
};

namespace {

constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 2-D E4M3 operand view [rows, cols] (cols contiguous), box 128 (cols) x box_rows,
// 128-byte swizzle, out-of-bounds rows read as zero.
mpq_status encode_operand(CUtensorMap *m, const uint8_t *ptr, int64_t rows, int64_t cols, int64_t ld,
                          uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return MPQ_ERR_CUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MPQ_OK : MPQ_ERR_CUDA;
}

// 2-D BF16 source view [rows, cols] (cols contiguous), boxes of 128 rows x 64 columns
// (128 bytes) with 128-byte swizzle; out-of-bounds rows read as zero.
mpq_status encode_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int64_t ld)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return MPQ_ERR_CUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MPQ_OK : MPQ_ERR_CUDA;
}

// E4M3 code view [rows, cols] (cols contiguous), boxes of box_rows rows x 128 bytes with 128-byte
// swizzle (the quantizers' staging layout); stores are clipped at the tensor bounds.
mpq_status encode_codes(CUtensorMap *m, void *ptr, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows = 128)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return MPQ_ERR_CUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MPQ_OK : MPQ_ERR_CUDA;
}

// GEMM output view [rows, cols] (cols contiguous, BF16 or FP32), boxes of 32 rows x 128
// bytes with 128-byte swizzle (wide: the pair kernel's staging buffers) or 32 rows x 64
// bytes with 64-byte swizzle (the single-SM kernel's); stores are clipped at the tensor
// bounds.
mpq_status encode_output(CUtensorMap *m, void *ptr, int64_t rows, int64_t cols, int64_t ld, bool fp32, bool wide)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return MPQ_ERR_CUDA;
    const int64_t esz = fp32 ? 4 : 2;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * esz)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>((wide ? 128 : 64) / esz), 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MPQ_OK : MPQ_ERR_CUDA;
}

mpq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MPQ_OK : MPQ_ERR_CUDA; }

// Every buffer of a handle lives on the device that was current at mpq_create, and the
// kernels launch on the current device: a call made with another device current returns
// MPQ_ERR_DEVICE before anything is launched.
mpq_status device_ok(mpq_handle h)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MPQ_ERR_CUDA;
    return dev == h->device ? MPQ_OK : MPQ_ERR_DEVICE;
}

} // namespace

extern "C" {

const char *mpq_version(void) { return "mpq 0.1.0 sm_103a"; }

const char *mpq_status_string(int s)
{
    switch (s) {
    case MPQ_OK: return "ok";
    case MPQ_ERR_NULL: return "null pointer argument";
    case MPQ_ERR_SHAPE: return "invalid size or leading dimension";
    case MPQ_ERR_ALIGN: return "misaligned pointer or stride";
    case MPQ_ERR_UNSUPPORTED: return "unsupported op, dtype or flags";
    case MPQ_ERR_CUDA: return "CUDA call failed";
    case MPQ_ERR_TIMEOUT: return "device-side wait timed out";
    case MPQ_ERR_WORKSPACE: return "no workspace set, or too small";
    case MPQ_ERR_DEVICE: return "the current device is not the handle's device";
    case MPQ_ERR_SCALE: return "a scale is not a power of 2 in the UE8M0 range";
    default: return "unknown status";
    }
}

mpq_status mpq_create(mpq_handle *out)
{
    if (out == nullptr)
        return MPQ_ERR_NULL;
    *out = nullptr;
    mpq_handle h = new (std::nothrow) mpq_handle_s();
    if (h == nullptr)
        return MPQ_ERR_CUDA;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void **>(&h->d_status), 2 * sizeof(int)) != cudaSuccess) {
        delete h;
        return MPQ_ERR_CUDA;
    }
    const size_t flag_bytes = static_cast<size_t>(h->num_sms) * 8 * sizeof(int);
    const size_t part_bytes = static_cast<size_t>(h->num_sms) * 8 * 1024 * sizeof(float4);
    if (cudaMemset(h->d_status, 0, 2 * sizeof(int)) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void **>(&h->d_sk_flags), flag_bytes) != cudaSuccess) {
        cudaFree(h->d_status);
        delete h;
        return MPQ_ERR_CUDA;
    }
    if (cudaMemset(h->d_sk_flags, 0, flag_bytes) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void **>(&h->d_sk_part), part_bytes) != cudaSuccess) {
        cudaFree(h->d_sk_flags);
        cudaFree(h->d_status);
        delete h;
        return MPQ_ERR_CUDA;
    }
    h->sk_mode = 1;
    h->sk_epoch = 0;
    h->timeout_ns = kDefaultTimeoutNs;
    h->pair_mode = 1;
    h->workspace = nullptr;
    h->workspace_bytes = 0;
    *out = h;
    return MPQ_OK;
}

mpq_status mpq_destroy(mpq_handle h)
{
    if (h == nullptr)
        return MPQ_ERR_NULL;
    // Synchronize and free on the handle's device, then restore the caller's current device.
    int cur = -1;
    const bool switched = cudaGetDevice(&cur) == cudaSuccess && cur != h->device &&
                          cudaSetDevice(h->device) == cudaSuccess;
    cudaDeviceSynchronize();
    cudaError_t e = cudaFree(h->d_status);
    const cudaError_t e2 = cudaFree(h->d_sk_flags);
    const cudaError_t e3 = cudaFree(h->d_sk_part);
    if (switched)
        cudaSetDevice(cur);
    delete h;
    return from_cuda(e != cudaSuccess ? e : e2 != cudaSuccess ? e2 : e3);
}

mpq_status mpq_set_wait_timeout(mpq_handle h, uint64_t timeout_ns)
{
    if (h == nullptr)
        return MPQ_ERR_NULL;
    h->timeout_ns = timeout_ns == 0 ? kDefaultTimeoutNs : timeout_ns;
    return MPQ_OK;
}

mpq_status mpq_set_gemm_cta_pair(mpq_handle h, int enable)
{
    if (h == nullptr)
        return MPQ_ERR_NULL;
    if (enable < 0 || enable > 2)
        return MPQ_ERR_UNSUPPORTED;
    h->pair_mode = enable;
    return MPQ_OK;
}

mpq_status mpq_set_gemm_stream_k(mpq_handle h, int mode)
{
    if (h == nullptr)
        return MPQ_ERR_NULL;
    if (mode < 0 || mode > 2)
        return MPQ_ERR_UNSUPPORTED;
    h->sk_mode = mode;
    return MPQ_OK;
}

mpq_status mpq_set_workspace(mpq_handle h, void *ptr, size_t bytes)
{
    if (h == nullptr)
        return MPQ_ERR_NULL;
    if ((ptr == nullptr) != (bytes == 0))
        return MPQ_ERR_NULL;
    if (!aligned(ptr, 256))
        return MPQ_ERR_ALIGN;
    h->workspace = ptr;
    h->workspace_bytes = bytes;
    return MPQ_OK;
}

// Grouped row tiles: experts with at least this many token rows take 2-SM pair tiles.
constexpr int64_t kPairExpertRows = 1024;

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

mpq_status mpq_grouped_fused_workspace_bytes(int64_t M_total, int64_t K, int64_t G, size_t *bytes)
{
    if (bytes == nullptr)
        return MPQ_ERR_NULL;
    if (M_total < 0 || K <= 0 || K % 128 != 0 || G < 1)
        return MPQ_ERR_SHAPE;
    *bytes = align256(static_cast<size_t>(M_total) * static_cast<size_t>(K)) +
             align256(static_cast<size_t>(K / 128) * static_cast<size_t>(M_total) * sizeof(float)) +
             align256(static_cast<size_t>(G) * sizeof(int));
    return MPQ_OK;
}

mpq_status mpq_check_device_status(mpq_handle h, void *stream, int *where_out)
{
    if (h == nullptr)
        return MPQ_ERR_NULL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int hs[2] = {0, 0};
    if (cudaStreamSynchronize(st) != cudaSuccess ||
        cudaMemcpy(hs, h->d_status, sizeof(hs), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(h->d_status, 0, sizeof(hs)) != cudaSuccess)
        return MPQ_ERR_CUDA;
    if (where_out != nullptr)
        *where_out = hs[1];
    return hs[0] == 0 ? MPQ_OK : static_cast<mpq_status>(hs[0]);
}

mpq_status fp8_quant_tile_1x128(mpq_handle h, const void *x, int64_t rows, int64_t cols, int64_t ldx,
                                uint8_t *q, int64_t ldq, float *s, int64_t lds, uint8_t *qT, int64_t ldqT,
                                float *sT, int64_t ldsT, uint32_t flags, void *stream)
{
    if (h == nullptr || x == nullptr || (q == nullptr && qT == nullptr))
        return MPQ_ERR_NULL;
    if ((q != nullptr && s == nullptr) || (qT != nullptr && sT == nullptr))
        return MPQ_ERR_NULL;
    if (flags & ~MPQ_POW2)
        return MPQ_ERR_UNSUPPORTED;
    if (rows < 0 || cols <= 0 || cols % 128 != 0 || ldx < cols)
        return MPQ_ERR_SHAPE;
    if (q != nullptr && (ldq < cols || lds < rows))
        return MPQ_ERR_SHAPE;
    if (qT != nullptr && (rows % 128 != 0 || ldqT < rows || ldsT < cols))
        return MPQ_ERR_SHAPE;
    if (!aligned(x, 16) || ldx % 8 != 0)
        return MPQ_ERR_ALIGN;
    if (q != nullptr && (!aligned(q, 16) || ldq % 16 != 0 || !aligned(s, 4)))
        return MPQ_ERR_ALIGN;
    if (qT != nullptr && (!aligned(qT, 16) || ldqT % 16 != 0 || !aligned(sT, 4)))
        return MPQ_ERR_ALIGN;
    if (rows == 0)
        return MPQ_OK;
    if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31))
        return MPQ_ERR_SHAPE;
    if (mpq_status d = device_ok(h); d != MPQ_OK)
        return d;
    const bool pow2 = (flags & MPQ_POW2) != 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    mpq::QuantArgs a{};
    a.rows = rows; a.cols = cols;
    a.q = q; a.ldq = ldq; a.s = s; a.lds = lds;
    a.qT = qT; a.ldqT = ldqT; a.sT = sT; a.ldsT = ldsT;
    a.status = h->d_status; a.timeout_ns = h->timeout_ns;
    CUtensorMap tmx, tmq, tmqT;
    mpq_status e = encode_bf16(&tmx, x, rows, cols, ldx);
    if (e == MPQ_OK && q != nullptr)
        e = encode_codes(&tmq, q, rows, cols, ldq);
    if (e == MPQ_OK && qT != nullptr)
        e = encode_codes(&tmqT, qT, cols, rows, ldqT);
    if (e != MPQ_OK)
        return e;
    if (q == nullptr)
        tmq = tmqT;   // unused by the kernel
    if (qT == nullptr)
        return from_cuda(mpq::launch_quant_rows(tmx, tmq, a, pow2, h->num_sms, st));
    return from_cuda(mpq::launch_quant_dual(tmx, tmq, tmqT, a, pow2, h->num_sms, st));
}

mpq_status fp8_swiglu_quant_1x128(mpq_handle h, const void *hcat, int64_t rows, int64_t width, int64_t ldh,
                                  uint8_t *q, int64_t ldq, float *s, int64_t lds, uint32_t flags, void *stream)
{
    if (h == nullptr)
        return MPQ_ERR_NULL;
    if (flags & ~MPQ_POW2)
        return MPQ_ERR_UNSUPPORTED;
    if (rows < 0 || width <= 0 || width % 128 != 0 || ldh < 2 * width || ldq < width || lds < rows)
        return MPQ_ERR_SHAPE;
    if (rows == 0)   // nothing is read or written
        return MPQ_OK;
    if (hcat == nullptr || q == nullptr || s == nullptr)
        return MPQ_ERR_NULL;
    if (!aligned(hcat, 16) || ldh % 8 != 0 || !aligned(q, 16) || ldq % 16 != 0 || !aligned(s, 4))
        return MPQ_ERR_ALIGN;
    if (rows > (int64_t(1) << 31) || width > (int64_t(1) << 30))
        return MPQ_ERR_SHAPE;
    if (mpq_status d = device_ok(h); d != MPQ_OK)
        return d;
    mpq::SwigluArgs a{};
    a.h = static_cast<const uint16_t *>(hcat);
    a.rows = rows; a.width = width; a.ldh = ldh;
    a.q = q; a.ldq = ldq; a.s = s; a.lds = lds;
    return from_cuda(mpq::launch_swiglu_quant(a, (flags & MPQ_POW2) != 0, h->num_sms,
                                              static_cast<cudaStream_t>(stream)));
}

mpq_status fp8_requant_tile_128x1(mpq_handle h, const uint8_t *q, int64_t rows, int64_t cols, int64_t ldq,
                                  const float *s, int64_t lds, uint8_t *qT, int64_t ldqT, float *sT,
                                  int64_t ldsT, uint32_t flags, void *stream)
{
    if (h == nullptr)
        return MPQ_ERR_NULL;
    if (flags & ~MPQ_POW2)
        return MPQ_ERR_UNSUPPORTED;
    if (rows < 0 || cols <= 0 || rows % 128 != 0 || cols % 128 != 0 || ldq < cols || lds < rows ||
        ldqT < rows || ldsT < cols)
        return MPQ_ERR_SHAPE;
    if (rows == 0)   // nothing is read or written
        return MPQ_OK;
    if (q == nullptr || s == nullptr || qT == nullptr || sT == nullptr)
        return MPQ_ERR_NULL;
    if (!aligned(q, 16) || ldq % 16 != 0 || !aligned(s, 16) || lds % 4 != 0 || !aligned(qT, 16) ||
        ldqT % 16 != 0 || !aligned(sT, 4))
        return MPQ_ERR_ALIGN;
    if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31))
        return MPQ_ERR_SHAPE;
    if (mpq_status d = device_ok(h); d != MPQ_OK)
        return d;
    mpq::RequantArgs a{};
    a.rows = rows; a.cols = cols;
    a.s = s; a.lds = lds; a.sT = sT; a.ldsT = ldsT;
    a.status = h->d_status; a.timeout_ns = h->timeout_ns;
    CUtensorMap tmq, tmqT;
    mpq_status e = encode_codes(&tmq, const_cast<uint8_t *>(q), rows, cols, ldq);
    if (e == MPQ_OK)
        e = encode_codes(&tmqT, qT, cols, rows, ldqT, 64);   // stored in 64-row halves
    if (e != MPQ_OK)
        return e;
    return from_cuda(mpq::launch_requant(tmq, tmqT, a, (flags & MPQ_POW2) != 0, h->num_sms,
                                         static_cast<cudaStream_t>(stream)));
}

mpq_status fp8_quant_block_128x128(mpq_handle h, const void *w, int64_t rows, int64_t cols, int64_t ldw,
                                   uint8_t *q, int64_t ldq, uint8_t *qT, int64_t ldqT, float *s, int64_t lds,
                                   uint32_t flags, void *stream)
{
    if (h == nullptr || w == nullptr || q == nullptr || s == nullptr)
        return MPQ_ERR_NULL;
    if (flags & ~MPQ_POW2)
        return MPQ_ERR_UNSUPPORTED;
    if (rows < 0 || cols < 0 || rows % 128 != 0 || cols % 128 != 0 || ldw < cols || ldq < cols ||
        lds < cols / 128 || (qT != nullptr && ldqT < rows))
        return MPQ_ERR_SHAPE;
    if (!aligned(w, 16) || ldw % 8 != 0 || !aligned(q, 16) || ldq % 16 != 0 || !aligned(s, 4) ||
        (qT != nullptr && (!aligned(qT, 16) || ldqT % 16 != 0)))
        return MPQ_ERR_ALIGN;
    if (rows == 0 || cols == 0)
        return MPQ_OK;
    if (rows > (int64_t(1) << 31) || cols > (int64_t(1) << 31))
        return MPQ_ERR_SHAPE;
    if (mpq_status d = device_ok(h); d != MPQ_OK)
        return d;
    mpq::QuantArgs a{};
    a.rows = rows; a.cols = cols;
    a.q = q; a.ldq = ldq; a.s = s; a.lds = lds;
    a.qT = qT; a.ldqT = ldqT;
    a.status = h->d_status; a.timeout_ns = h->timeout_ns;
    CUtensorMap tmx, tmq, tmqT;
    mpq_status e = encode_bf16(&tmx, w, rows, cols, ldw);
    if (e == MPQ_OK)
        e = encode_codes(&tmq, q, rows, cols, ldq);
    if (e == MPQ_OK && qT != nullptr)
        e = encode_codes(&tmqT, qT, cols, rows, ldqT);
    if (e != MPQ_OK)
        return e;
    if (qT == nullptr)
        tmqT = tmq;   // unused by the kernel
    return from_cuda(mpq::launch_quant_block(tmx, tmq, tmqT, a, (flags & MPQ_POW2) != 0, h->num_sms,
                                             static_cast<cudaStream_t>(stream)));
}

static mpq_status check_gemm_common(int64_t N, int64_t K, const uint8_t *A, int64_t lda, const float *sA,
                                    const uint8_t *B, int64_t ldb, const float *sB, void *C, int64_t ldc,
                                    int out_dtype)
{
    if (A == nullptr || sA == nullptr || B == nullptr || sB == nullptr || C == nullptr)
        return MPQ_ERR_NULL;
    if (out_dtype != MPQ_OUT_BF16 && out_dtype != MPQ_OUT_FP32)
        return MPQ_ERR_UNSUPPORTED;
    if (N <= 0 || N % 128 != 0 || K <= 0 || K % 128 != 0 || lda < K || ldb < K || ldc < N)
        return MPQ_ERR_SHAPE;
    if (K > (int64_t(1) << 31) || N > (int64_t(1) << 31))
        return MPQ_ERR_SHAPE;
    const int64_t esz = out_dtype == MPQ_OUT_FP32 ? 4 : 2;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || lda % 16 != 0 || ldb % 16 != 0 ||
        (ldc * esz) % 16 != 0 || !aligned(sA, 4) || !aligned(sB, 4))
        return MPQ_ERR_ALIGN;
    return MPQ_OK;
}

// Stream-K for a dense GEMM of `tiles` output tiles on `units` CTAs (or CTA pairs): when the
// tiles fill more than one wave and, in the default mode, the last wave would leave more
// than a tenth of the machine's time idle, the launch gets the handle's handover area and a
// new epoch (a->sk_part stays null otherwise).
static mpq_status setup_stream_k(mpq_handle h, int64_t tiles, int64_t units, mpq::GemmArgs *a, void *stream)
{
    bool sk = false;
    if (h->sk_mode != 0 && tiles > units) {
        const int64_t waves = (tiles + units - 1) / units;
        sk = h->sk_mode == 2 || 10 * (waves * units - tiles) > waves * units;
    }
    if (!sk)
        return MPQ_OK;
    // The flags hold the epoch of the launch that last wrote them; a waiter accepts a flag
    // >= its own epoch.  Before the counter would overflow, the flags are cleared (in stream
    // order, ahead of the launch) and the count restarts.
    if (h->sk_epoch == INT32_MAX) {
        if (cudaMemsetAsync(h->d_sk_flags, 0, static_cast<size_t>(h->num_sms) * 8 * sizeof(int),
                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return MPQ_ERR_CUDA;
        h->sk_epoch = 0;
    }
    a->sk_part = h->d_sk_part;
    a->sk_flags = h->d_sk_flags;
    a->sk_epoch = ++h->sk_epoch;
    return MPQ_OK;
}

mpq_status fp8_gemm_blockscaled(mpq_handle h, int op, int64_t M, int64_t N, int64_t K, const uint8_t *A,
                                int64_t lda, const float *sA, int64_t ldsa, const uint8_t *B, int64_t ldb,
                                const float *sB, int64_t ldsb, void *C, int64_t ldc, int out_dtype,
                                void *stream)
{
    if (h == nullptr)
        return MPQ_ERR_NULL;
    if (op != MPQ_OP_FPROP && op != MPQ_OP_DGRAD && op != MPQ_OP_WGRAD)
        return MPQ_ERR_UNSUPPORTED;
    mpq_status st = check_gemm_common(N, K, A, lda, sA, B, ldb, sB, C, ldc, out_dtype);
    if (st != MPQ_OK)
        return st;
    if (M < 0 || M > (int64_t(1) << 31) || ldsa < M)
        return MPQ_ERR_SHAPE;
    if ((op == MPQ_OP_FPROP && ldsb < K / 128) || (op == MPQ_OP_DGRAD && ldsb < N / 128) ||
        (op == MPQ_OP_WGRAD && ldsb < N))
        return MPQ_ERR_SHAPE;
    if (M == 0)
        return MPQ_OK;
    if (mpq_status d = device_ok(h); d != MPQ_OK)
        return d;
    CUtensorMap tmA, tmB;
    if ((st = encode_operand(&tmA, A, M, K, lda, 128)) != MPQ_OK)
        return st;
    const bool pair = h->pair_mode != 0;
    if ((st = encode_operand(&tmB, B, N, K, ldb, mpq::gemm_b_box_rows(pair))) != MPQ_OK)
        return st;
    CUtensorMap tmC;
    if ((st = encode_output(&tmC, C, M, N, ldc, out_dtype == MPQ_OUT_FP32, pair)) != MPQ_OK)
        return st;
    mpq::GemmArgs a{};
    a.M = M; a.N = N; a.K = K;
    a.sA = sA; a.ldsa = ldsa;
    a.sB = sB; a.ldsb = ldsb; a.sb_group_stride = 0;
    a.C = C; a.ldc = ldc;
    a.offsets = nullptr; a.G = 1;
    a.status = h->d_status; a.timeout_ns = h->timeout_ns;
    const int sb = op == MPQ_OP_FPROP ? mpq::kScaleBlockNK : op == MPQ_OP_DGRAD ? mpq::kScaleBlockKN : mpq::kScaleRowKN;
    a.n_fastest = N < M ? 1 : 0;   // re-read the smaller operand (from L2)
    const int64_t tile_m = pair ? 256 : 128;
    const int64_t tiles = ((M + tile_m - 1) / tile_m) * ((N + 255) / 256);
    if ((st = setup_stream_k(h, tiles, pair ? h->num_sms / 2 : h->num_sms, &a, stream)) != MPQ_OK)
        return st;
    return from_cuda(mpq::launch_gemm(tmA, tmB, tmC, a, sb, out_dtype == MPQ_OUT_FP32, pair, h->num_sms,
                                      static_cast<cudaStream_t>(stream)));
}

mpq_status fp8_gemm_mx_pow2(mpq_handle h, int op, int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda,
                            const float *sA, int64_t ldsa, const uint8_t *B, int64_t ldb, const float *sB,
                            int64_t ldsb, void *C, int64_t ldc, int out_dtype, void *stream)
{
    if (h == nullptr)
        return MPQ_ERR_NULL;
    if (op != MPQ_OP_FPROP && op != MPQ_OP_DGRAD && op != MPQ_OP_WGRAD)
        return MPQ_ERR_UNSUPPORTED;
    mpq_status st = check_gemm_common(N, K, A, lda, sA, B, ldb, sB, C, ldc, out_dtype);
    if (st != MPQ_OK)
        return st;
    if (M < 0 || M > (int64_t(1) << 31) || ldsa < M)
        return MPQ_ERR_SHAPE;
    if ((op == MPQ_OP_FPROP && ldsb < K / 128) || (op == MPQ_OP_DGRAD && ldsb < N / 128) ||
        (op == MPQ_OP_WGRAD && ldsb < N))
        return MPQ_ERR_SHAPE;
    if (M == 0)
        return MPQ_OK;
    if (mpq_status d = device_ok(h); d != MPQ_OK)
        return d;
    CUtensorMap tmA, tmB, tmC;
    if ((st = encode_operand(&tmA, A, M, K, lda, 128)) != MPQ_OK)
        return st;
    if ((st = encode_operand(&tmB, B, N, K, ldb, 128)) != MPQ_OK)
        return st;
    if ((st = encode_output(&tmC, C, M, N, ldc, out_dtype == MPQ_OUT_FP32, false)) != MPQ_OK)
        return st;
    mpq::GemmArgs a{};
    a.M = M; a.N = N; a.K = K;
    a.sA = sA; a.ldsa = ldsa;
    a.sB = sB; a.ldsb = ldsb; a.sb_group_stride = 0;
    a.C = C; a.ldc = ldc;
    a.offsets = nullptr; a.G = 1;
    a.status = h->d_status; a.timeout_ns = h->timeout_ns;
    const int sb = op == MPQ_OP_FPROP ? mpq::kScaleBlockNK : op == MPQ_OP_DGRAD ? mpq::kScaleBlockKN : mpq::kScaleRowKN;
    a.n_fastest = N < M ? 1 : 0;   // re-read the smaller operand (from L2)
    // 256 x 256 pair tiles; stream-K under the same rule as fp8_gemm_blockscaled
    if ((st = setup_stream_k(h, ((M + 255) / 256) * ((N + 255) / 256), h->num_sms / 2, &a, stream)) != MPQ_OK)
        return st;
    return from_cuda(mpq::launch_gemm_mx(tmA, tmB, tmC, a, sb, out_dtype == MPQ_OUT_FP32, h->num_sms,
                                         static_cast<cudaStream_t>(stream)));
}

// Fused grouped GEMM after validation: carve the workspace (codes [M, K], scales [K/128][M],
// per-expert counts) and launch on row tiles (single-SM, cooperative) or, with
// MPQ_GROUPED_WEIGHT_TILES, on weight tiles.
static mpq_status launch_fused_grouped(mpq_handle h, void *workspace, int64_t G, const int64_t *d_offsets,
                                       int64_t M_total, int64_t N, int64_t K, const void *X, int64_t ldx,
                                       const uint8_t *B, int64_t ldb, const float *sB, int64_t ldsb, void *C,
                                       int64_t ldc, int out_dtype, uint32_t flags, void *stream)
{
    if (mpq_status d = device_ok(h); d != MPQ_OK)
        return d;
    uint8_t *xq = static_cast<uint8_t *>(workspace);
    float *sx = reinterpret_cast<float *>(xq + align256(static_cast<size_t>(M_total) * static_cast<size_t>(K)));
    int *ready = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(sx) +
                                         align256(static_cast<size_t>(K / 128) * static_cast<size_t>(M_total) *
                                                  sizeof(float)));
    mpq::GemmArgs a{};
    a.M = M_total; a.N = N; a.K = K;
    a.sA = sx; a.ldsa = M_total;
    a.sB = sB; a.ldsb = ldsb; a.sb_group_stride = (N / 128) * ldsb;
    a.C = C; a.ldc = ldc;
    a.offsets = d_offsets; a.G = static_cast<int>(G);
    a.status = h->d_status; a.timeout_ns = h->timeout_ns;
    mpq::FuseArgs f{};
    f.x = static_cast<const uint16_t *>(X);
    f.ldx = ldx;
    f.xq = xq; f.sx = sx; f.ready = ready;
    f.pow2 = (flags & MPQ_POW2) != 0 ? 1 : 0;
    const bool fp32 = out_dtype == MPQ_OUT_FP32;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    mpq_status e;
    if ((flags & MPQ_GROUPED_WEIGHT_TILES) != 0) {
        CUtensorMap tmX, tmW;
        if ((e = encode_operand(&tmX, xq, M_total, K, K, mpq::decode_x_box_rows())) != MPQ_OK)
            return e;
        if ((e = encode_operand(&tmW, B, G * N, K, ldb, 128)) != MPQ_OK)
            return e;
        return from_cuda(mpq::launch_decode(tmX, tmW, a, fp32, &f, h->num_sms, st));
    }
    CUtensorMap tmA, tmB, tmC;
    if ((e = encode_operand(&tmA, xq, M_total, K, K, 128)) != MPQ_OK)
        return e;
    if ((e = encode_operand(&tmB, B, G * N, K, ldb, mpq::gemm_b_box_rows(false))) != MPQ_OK)
        return e;
    if ((e = encode_output(&tmC, C, M_total, N, ldc, fp32, false)) != MPQ_OK)
        return e;
    return from_cuda(mpq::launch_gemm(tmA, tmB, tmC, a, mpq::kScaleBlockNK, fp32, false, h->num_sms, st, &f));
}

// Grouped GEMM with fused 1x128 quantization of the BF16 activations.
static mpq_status grouped_fused(mpq_handle h, int64_t G, const int64_t *d_offsets, int64_t M_total, int64_t N,
                                int64_t K, const uint8_t *A, int64_t lda, const float *sA, const uint8_t *B,
                                int64_t ldb, const float *sB, int64_t ldsb, void *C, int64_t ldc, int out_dtype,
                                uint32_t flags, void *stream)
{
    if ((flags & ~(MPQ_FUSE_QUANT_A | MPQ_POW2 | MPQ_GROUPED_WEIGHT_TILES)) != 0 || sA != nullptr)
        return MPQ_ERR_UNSUPPORTED;
    if (A == nullptr || B == nullptr || sB == nullptr || C == nullptr)
        return MPQ_ERR_NULL;
    if (out_dtype != MPQ_OUT_BF16 && out_dtype != MPQ_OUT_FP32)
        return MPQ_ERR_UNSUPPORTED;
    if (N <= 0 || N % 128 != 0 || K <= 0 || K % 128 != 0 || lda < K || ldb < K || ldc < N || ldsb < K / 128)
        return MPQ_ERR_SHAPE;
    if (G < 1 || G > 1024 || M_total < 0 || M_total > (int64_t(1) << 31) || K > (int64_t(1) << 31) ||
        G * N > (int64_t(1) << 31))
        return MPQ_ERR_SHAPE;
    const int64_t esz = out_dtype == MPQ_OUT_FP32 ? 4 : 2;
    if (!aligned(A, 16) || lda % 8 != 0 || !aligned(B, 16) || ldb % 16 != 0 || !aligned(C, 16) ||
        (ldc * esz) % 16 != 0 || !aligned(sB, 4) || !aligned(d_offsets, 8))
        return MPQ_ERR_ALIGN;
    if (M_total == 0)
        return MPQ_OK;
    size_t need = 0;
    mpq_status st = mpq_grouped_fused_workspace_bytes(M_total, K, G, &need);
    if (st != MPQ_OK)
        return st;
    if (h->workspace == nullptr || h->workspace_bytes < need)
        return MPQ_ERR_WORKSPACE;
    return launch_fused_grouped(h, h->workspace, G, d_offsets, M_total, N, K, A, lda, B, ldb, sB, ldsb, C, ldc,
                                out_dtype, flags, stream);
}

// The allocation-free form of the fused grouped GEMM: the same validation and launch as
// grouped_fused, with the library's fixed scratch area (noalloc.cu) as the workspace.
mpq_status fp8_grouped_gemm_fused_quant_noalloc(mpq_handle h, int64_t G, const int64_t *d_offsets,
                                                int64_t M_total, int64_t N, int64_t K, const void *X, int64_t ldx,
                                                const uint8_t *B, int64_t ldb, const float *sB, int64_t ldsb,
                                                void *C, int64_t ldc, int out_dtype, uint32_t flags, void *stream)
{
    static_assert(mpq::kNoallocScratchBytes == MPQ_NOALLOC_SCRATCH_BYTES, "scratch size");
    if (h == nullptr || d_offsets == nullptr || X == nullptr || B == nullptr || sB == nullptr || C == nullptr)
        return MPQ_ERR_NULL;
    if ((flags & ~MPQ_POW2) != 0 || (out_dtype != MPQ_OUT_BF16 && out_dtype != MPQ_OUT_FP32))
        return MPQ_ERR_UNSUPPORTED;
    if (N <= 0 || N % 128 != 0 || K <= 0 || K % 128 != 0 || ldx < K || ldb < K || ldc < N || ldsb < K / 128)
        return MPQ_ERR_SHAPE;
    if (G < 1 || G > 1024 || M_total < 0 || M_total > (int64_t(1) << 31) || K > (int64_t(1) << 31) ||
        G * N > (int64_t(1) << 31))
        return MPQ_ERR_SHAPE;
    const int64_t esz = out_dtype == MPQ_OUT_FP32 ? 4 : 2;
    if (!aligned(X, 16) || ldx % 8 != 0 || !aligned(B, 16) || ldb % 16 != 0 || !aligned(C, 16) ||
        (ldc * esz) % 16 != 0 || !aligned(sB, 4) || !aligned(d_offsets, 8))
        return MPQ_ERR_ALIGN;
    size_t need = 0;
    mpq_status st = mpq_grouped_fused_workspace_bytes(M_total, K, G, &need);
    if (st != MPQ_OK)
        return st;
    if (need > mpq::kNoallocScratchBytes)
        return MPQ_ERR_WORKSPACE;
    if (M_total == 0)
        return MPQ_OK;
    void *scratch = nullptr;
    if (mpq::noalloc_scratch(&scratch) != cudaSuccess)
        return MPQ_ERR_CUDA;
    return launch_fused_grouped(h, scratch, G, d_offsets, M_total, N, K, X, ldx, B, ldb, sB, ldsb, C, ldc, out_dtype,
                                flags, stream);
}

mpq_status fp8_grouped_gemm_swiglu_quant(mpq_handle h, int64_t G, const int64_t *d_offsets, int64_t M_total,
                                         int64_t W, int64_t K, const void *A, int64_t lda, const float *sA,
                                         int64_t ldsa, const uint8_t *B, int64_t ldb, const float *sB, int64_t ldsb,
                                         void *H, int64_t ldh, uint8_t *q, int64_t ldq, float *s, int64_t lds,
                                         uint32_t flags, void *stream)
{
    if (h == nullptr || d_offsets == nullptr || A == nullptr || B == nullptr || sB == nullptr || q == nullptr ||
        s == nullptr)
        return MPQ_ERR_NULL;
    if ((flags & ~(MPQ_POW2 | MPQ_FUSE_QUANT_A)) != 0)
        return MPQ_ERR_UNSUPPORTED;
    const bool fuse = (flags & MPQ_FUSE_QUANT_A) != 0;
    if (fuse ? sA != nullptr : sA == nullptr)
        return fuse ? MPQ_ERR_UNSUPPORTED : MPQ_ERR_NULL;
    const int64_t N = 2 * W;
    if (W <= 0 || W % 128 != 0 || K <= 0 || K % 128 != 0 || lda < K || ldb < K || ldsb < K / 128 || ldq < W)
        return MPQ_ERR_SHAPE;
    if (G < 1 || G > 1024 || M_total < 0 || M_total > (int64_t(1) << 31) || K > (int64_t(1) << 31) ||
        G * N > (int64_t(1) << 31) || lds < M_total || (!fuse && ldsa < M_total) || (H != nullptr && ldh < N))
        return MPQ_ERR_SHAPE;
    if (!aligned(A, 16) || (fuse ? lda % 8 != 0 : lda % 16 != 0) || !aligned(B, 16) || ldb % 16 != 0 ||
        !aligned(q, 16) || ldq % 16 != 0 || !aligned(s, 4) || !aligned(sB, 4) || !aligned(d_offsets, 8) ||
        (!fuse && !aligned(sA, 4)) || (H != nullptr && (!aligned(H, 16) || ldh % 8 != 0)))
        return MPQ_ERR_ALIGN;
    if (M_total == 0)
        return MPQ_OK;
    if (mpq_status d = device_ok(h); d != MPQ_OK)
        return d;
    mpq::GemmArgs a{};
    a.M = M_total; a.N = N; a.K = K;
    a.sB = sB; a.ldsb = ldsb; a.sb_group_stride = (N / 128) * ldsb;
    a.C = H; a.ldc = ldh;
    a.offsets = d_offsets; a.G = static_cast<int>(G);
    a.status = h->d_status; a.timeout_ns = h->timeout_ns;
    a.sw_q = q; a.sw_ldq = ldq; a.sw_s = s; a.sw_lds = lds;
    a.sw_width = static_cast<int>(W); a.sw_pow2 = (flags & MPQ_POW2) != 0 ? 1 : 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUtensorMap tmA, tmB;
    mpq_status e;
    if ((e = encode_operand(&tmB, B, G * N, K, ldb, 128)) != MPQ_OK)
        return e;
    if (fuse) {
        size_t need = 0;
        if ((e = mpq_grouped_fused_workspace_bytes(M_total, K, G, &need)) != MPQ_OK)
            return e;
        if (h->workspace == nullptr || h->workspace_bytes < need)
            return MPQ_ERR_WORKSPACE;
        uint8_t *xq = static_cast<uint8_t *>(h->workspace);
        float *sx = reinterpret_cast<float *>(xq + align256(static_cast<size_t>(M_total) * static_cast<size_t>(K)));
        int *ready = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(sx) +
                                             align256(static_cast<size_t>(K / 128) * static_cast<size_t>(M_total) *
                                                      sizeof(float)));
        a.sA = sx; a.ldsa = M_total;
        mpq::FuseArgs f{};
        f.x = static_cast<const uint16_t *>(A);
        f.ldx = lda;
        f.xq = xq; f.sx = sx; f.ready = ready;
        f.pow2 = 0;   // the up projection's input: amax/448 scales
        if ((e = encode_operand(&tmA, xq, M_total, K, K, 128)) != MPQ_OK)
            return e;
        return from_cuda(mpq::launch_gemm_swiglu(tmA, tmB, a, false, h->num_sms, st, &f));
    }
    a.sA = sA; a.ldsa = ldsa;
    if ((e = encode_operand(&tmA, static_cast<const uint8_t *>(A), M_total, K, lda, 128)) != MPQ_OK)
        return e;
    // tiling as fp8_grouped_gemm_blockscaled's row tiles (large experts on pair tiles)
    for (int pass = 0; pass < 2; ++pass) {
        const bool pair = pass == 0;
        mpq::GemmArgs ap = a;
        if (h->pair_mode == 1) {
            if (pair && M_total < kPairExpertRows)
                continue;
            ap.min_rows = pair ? kPairExpertRows : 0;
            ap.max_rows = pair ? 0x7FFFFFFF : kPairExpertRows;
        } else if (pair != (h->pair_mode == 2)) {
            continue;
        }
        if ((e = from_cuda(mpq::launch_gemm_swiglu(tmA, tmB, ap, pair, h->num_sms, st))) != MPQ_OK)
            return e;
    }
    return MPQ_OK;
}

mpq_status fp8_grouped_gemm_blockscaled(mpq_handle h, int64_t G, const int64_t *d_offsets, int64_t M_total,
                                        int64_t N, int64_t K, const uint8_t *A, int64_t lda, const float *sA,
                                        int64_t ldsa, const uint8_t *B, int64_t ldb, const float *sB,
                                        int64_t ldsb, void *C, int64_t ldc, int out_dtype, uint32_t flags,
                                        void *stream)
{
    if (h == nullptr || d_offsets == nullptr)
        return MPQ_ERR_NULL;
    if ((flags & MPQ_FUSE_QUANT_A) != 0)
        return grouped_fused(h, G, d_offsets, M_total, N, K, A, lda, sA, B, ldb, sB, ldsb, C, ldc, out_dtype, flags,
                             stream);
    if ((flags & ~(MPQ_GROUPED_ROW_TILES | MPQ_GROUPED_WEIGHT_TILES)) != 0 ||
        flags == (MPQ_GROUPED_ROW_TILES | MPQ_GROUPED_WEIGHT_TILES))
        return MPQ_ERR_UNSUPPORTED;
    mpq_status st = check_gemm_common(N, K, A, lda, sA, B, ldb, sB, C, ldc, out_dtype);
    if (st != MPQ_OK)
        return st;
    if (G < 1 || G > 1024 || M_total < 0 || M_total > (int64_t(1) << 31) || ldsa < M_total || ldsb < K / 128 ||
        G * N > (int64_t(1) << 31))
        return MPQ_ERR_SHAPE;
    if (!aligned(d_offsets, 8))
        return MPQ_ERR_ALIGN;
    if (M_total == 0)
        return MPQ_OK;
    if (mpq_status d = device_ok(h); d != MPQ_OK)
        return d;
    // Row tiles by default: on single-SM tiles they stream the weights at the HBM rate even
    // for a few tokens per expert; weight tiles only on request.
    const bool weight_tiles = (flags & MPQ_GROUPED_WEIGHT_TILES) != 0;
    mpq::GemmArgs a{};
    a.M = M_total; a.N = N; a.K = K;
    a.sA = sA; a.ldsa = ldsa;
    a.sB = sB; a.ldsb = ldsb; a.sb_group_stride = (N / 128) * ldsb;
    a.C = C; a.ldc = ldc;
    a.offsets = d_offsets; a.G = static_cast<int>(G);
    a.status = h->d_status; a.timeout_ns = h->timeout_ns;
    CUtensorMap tmA;
    if (weight_tiles) {
        CUtensorMap tmB;
        if ((st = encode_operand(&tmA, A, M_total, K, lda, mpq::decode_x_box_rows())) != MPQ_OK)
            return st;
        if ((st = encode_operand(&tmB, B, G * N, K, ldb, 128)) != MPQ_OK)
            return st;
        return from_cuda(mpq::launch_decode(tmA, tmB, a, out_dtype == MPQ_OUT_FP32, nullptr, h->num_sms,
                                            static_cast<cudaStream_t>(stream)));
    }
    if ((st = encode_operand(&tmA, A, M_total, K, lda, 128)) != MPQ_OK)
        return st;
    // Tiling: pair tiles round an expert's rows up to 256, single-SM tiles up to 128.  By
    // default experts with kPairExpertRows rows or more take pair tiles (faster per row, little
    // padding) and the others single-SM tiles, in two launches on the stream, each computing
    // only its experts' rows; mode 0 / 2: single-SM / pair tiles for every expert.
    const bool fp32 = out_dtype == MPQ_OUT_FP32;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    for (int pass = 0; pass < 2; ++pass) {
        const bool pair = pass == 0;
        mpq::GemmArgs ap = a;
        if (h->pair_mode == 1) {
            if (pair && M_total < kPairExpertRows)
                continue;   // no expert can be that large
            ap.min_rows = pair ? kPairExpertRows : 0;
            ap.max_rows = pair ? 0x7FFFFFFF : kPairExpertRows;
        } else if (pair != (h->pair_mode == 2)) {
            continue;
        }
        CUtensorMap tmB, tmC;
        if ((st = encode_operand(&tmB, B, G * N, K, ldb, mpq::gemm_b_box_rows(pair))) != MPQ_OK)
            return st;
        if ((st = encode_output(&tmC, C, M_total, N, ldc, fp32, pair)) != MPQ_OK)
            return st;
        if ((st = from_cuda(mpq::launch_gemm(tmA, tmB, tmC, ap, mpq::kScaleBlockNK, fp32, pair, h->num_sms, cs))) !=
            MPQ_OK)
            return st;
    }
    return MPQ_OK;
}

mpq_status mpq_selftest_wait_timeout(mpq_handle h, uint64_t timeout_ns, void *stream)
{
    if (h == nullptr)
        return MPQ_ERR_NULL;
    if (mpq_status d = device_ok(h); d != MPQ_OK)
        return d;
    return from_cuda(mpq::launch_wait_selftest(h->d_status, timeout_ns == 0 ? 1000000ull : timeout_ns,
                                               static_cast<cudaStream_t>(stream)));
}

} // extern "C"

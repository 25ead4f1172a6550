"""mixed_precision_quant_b300 -- Python binding of libmpq (fine-grained FP8 quantization
and block-scaled FP8 GEMM on B300 / sm_103a).

This module only marshals arguments: it turns torch tensors into device pointers,
leading dimensions and the current CUDA stream, calls the C ABI declared in
``include/mpq.h`` (same function names), and raises :class:`MPQError` on a non-zero
status.  PyTorch is used for device memory and streams only; every step of the path
runs in the library's own CUDA kernels.  There is no fallback: if ``libmpq.so`` is
missing or cannot be loaded, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmpq.so")

FPROP, DGRAD, WGRAD = 0, 1, 2
OUT_BF16, OUT_FP32 = 0, 1
POW2 = 1
GROUPED_ROW_TILES, GROUPED_WEIGHT_TILES = 2, 4
FUSE_QUANT_A = 8

_STATUS = {0: "ok", 1: "null pointer argument", 2: "invalid size or leading dimension",
           3: "misaligned pointer or stride", 4: "unsupported op, dtype or flags",
           5: "CUDA call failed", 6: "device-side wait timed out", 7: "no workspace set, or too small",
           8: "the current device is not the handle's device",
           9: "a scale is not a power of 2 in the UE8M0 range"}


class MPQError(RuntimeError):
    def __init__(self, fn: str, status: int, extra: str = ""):
        self.status = status
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)}{extra}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libmpq.so is not built ({LIB_PATH}); run `python -m mixed_precision_quant_b300._build` "
            "or __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, U32, U64, INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int
    sigs = {
        "mpq_version": (ctypes.c_char_p, []),
        "mpq_status_string": (ctypes.c_char_p, [INT]),
        "mpq_create": (INT, [ctypes.POINTER(P)]),
        "mpq_destroy": (INT, [P]),
        "mpq_set_wait_timeout": (INT, [P, U64]),
        "mpq_set_gemm_cta_pair": (INT, [P, INT]),
        "mpq_set_gemm_stream_k": (INT, [P, INT]),
        "mpq_check_device_status": (INT, [P, P, ctypes.POINTER(INT)]),
        "fp8_quant_tile_1x128": (INT, [P, P, I, I, I, P, I, P, I, P, I, P, I, U32, P]),
        "fp8_quant_block_128x128": (INT, [P, P, I, I, I, P, I, P, I, P, I, U32, P]),
        "fp8_requant_tile_128x1": (INT, [P, P, I, I, I, P, I, P, I, P, I, U32, P]),
        "fp8_swiglu_quant_1x128": (INT, [P, P, I, I, I, P, I, P, I, U32, P]),
        "fp8_gemm_blockscaled": (INT, [P, INT, I, I, I, P, I, P, I, P, I, P, I, P, I, INT, P]),
        "fp8_gemm_mx_pow2": (INT, [P, INT, I, I, I, P, I, P, I, P, I, P, I, P, I, INT, P]),
        "fp8_grouped_gemm_blockscaled": (INT, [P, I, P, I, I, I, P, I, P, I, P, I, P, I, P, I, INT, U32, P]),
        "mpq_selftest_wait_timeout": (INT, [P, U64, P]),
        "mpq_set_workspace": (INT, [P, P, ctypes.c_size_t]),
        "mpq_grouped_fused_workspace_bytes": (INT, [I, I, I, ctypes.POINTER(ctypes.c_size_t)]),
        "fp8_grouped_gemm_fused_quant_noalloc": (INT, [P, I, P, I, I, I, P, I, P, I, P, I, P, I, INT, U32, P]),
        "fp8_grouped_gemm_swiglu_quant": (INT, [P, I, P, I, I, I, P, I, P, I, P, I, P, I, P, I, P, I, P, I, U32, P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
_handles: dict = {}
_workspaces: dict = {}   # device index -> torch uint8 buffer handed to mpq_set_workspace
_hlock = threading.Lock()


def version() -> str:
    return _lib.mpq_version().decode()


def _handle(device: torch.device) -> ctypes.c_void_p:
    idx = device.index if device.index is not None else torch.cuda.current_device()
    with _hlock:
        h = _handles.get(idx)
        if h is None:
            with torch.cuda.device(idx):
                h = ctypes.c_void_p()
                st = _lib.mpq_create(ctypes.byref(h))
                if st != 0:
                    raise MPQError("mpq_create", st)
            _handles[idx] = h
        return h


def _stream(device: torch.device, stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _ld(t: Optional[torch.Tensor]) -> int:
    if t is None:
        return 0
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit column stride")
    return t.stride(0)


def _check(fn: str, st: int):
    if st != 0:
        raise MPQError(fn, st)


def _cuda2d(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda or t.dtype != dtype or t.dim() != 2:
        raise TypeError(f"{name}: expected a 2-D {dtype} CUDA tensor, got {t.dtype} {tuple(t.shape)} on {t.device}")


# ------------------------------------------------------------------- quantizers

def fp8_quant_tile_1x128(x: torch.Tensor, *, pow2: bool = False, rows_out: bool = True,
                         transposed: bool = False, q=None, s=None, qT=None, sT=None, stream=None):
    """1x128 activation quantization of BF16 ``x [rows, cols]``.

    Returns ``(q, s, qT, sT)``: row-wise codes ``q [rows, cols]`` uint8 with scales
    ``s [cols/128, rows]`` float32 (None when ``rows_out`` is False), and, when
    ``transposed``, the 128x1 (along rows) quantization stored transposed:
    ``qT [cols, rows]`` with ``sT [rows/128, cols]``."""
    _cuda2d(x, torch.bfloat16, "x")
    rows, cols = x.shape
    dev = x.device
    if rows_out:
        q = q if q is not None else torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        s = s if s is not None else torch.empty((cols // 128, rows), dtype=torch.float32, device=dev)
    else:
        q = s = None
    if transposed:
        qT = qT if qT is not None else torch.empty((cols, rows), dtype=torch.uint8, device=dev)
        sT = sT if sT is not None else torch.empty((rows // 128, cols), dtype=torch.float32, device=dev)
    else:
        qT = sT = None
    with torch.cuda.device(dev):   # the handle's device is current for the call
        st = _lib.fp8_quant_tile_1x128(_handle(dev), _ptr(x), rows, cols, _ld(x), _ptr(q), _ld(q), _ptr(s), _ld(s),
                                       _ptr(qT), _ld(qT), _ptr(sT), _ld(sT), POW2 if pow2 else 0,
                                       _stream(dev, stream))
    _check("fp8_quant_tile_1x128", st)
    return q, s, qT, sT


def fp8_swiglu_quant_1x128(hcat: torch.Tensor, *, pow2: bool = True, q=None, s=None, stream=None):
    """SwiGLU of the up-projection output ``hcat [rows, 2*width]`` BF16 (gate in the first
    ``width`` columns, up in the rest) fused with the 1x128 quantization of
    ``silu(gate) * up``.  Returns ``(q [rows, width] uint8, s [width/128, rows] float32)``;
    ``pow2`` selects power-of-2 scales (the pages' rule for this activation)."""
    _cuda2d(hcat, torch.bfloat16, "hcat")
    rows, w2 = hcat.shape
    width = w2 // 2
    dev = hcat.device
    q = q if q is not None else torch.empty((rows, width), dtype=torch.uint8, device=dev)
    s = s if s is not None else torch.empty((width // 128, rows), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):   # the handle's device is current for the call
        st = _lib.fp8_swiglu_quant_1x128(_handle(dev), _ptr(hcat), rows, width, _ld(hcat), _ptr(q), _ld(q), _ptr(s),
                                         _ld(s), POW2 if pow2 else 0, _stream(dev, stream))
    _check("fp8_swiglu_quant_1x128", st)
    return q, s


def fp8_requant_tile_128x1(q: torch.Tensor, s: torch.Tensor, *, pow2: bool = False, qT=None, sT=None,
                           stream=None):
    """Re-quantize a cached 1x128 quantization (codes ``q [rows, cols]`` uint8, scales
    ``s [cols/128, rows]`` float32, as written by :func:`fp8_quant_tile_1x128`) into 128x1
    groups along rows: each value is dequantized to binary32 (``dec(q) * s``) and the
    column groups are quantized again.  Returns ``(qT [cols, rows], sT [rows/128, cols])``,
    the layout of the transposed quantizer output."""
    _cuda2d(q, torch.uint8, "q")
    _cuda2d(s, torch.float32, "s")
    rows, cols = q.shape
    dev = q.device
    qT = qT if qT is not None else torch.empty((cols, rows), dtype=torch.uint8, device=dev)
    sT = sT if sT is not None else torch.empty((rows // 128, cols), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):   # the handle's device is current for the call
        st = _lib.fp8_requant_tile_128x1(_handle(dev), _ptr(q), rows, cols, _ld(q), _ptr(s), _ld(s), _ptr(qT), _ld(qT),
                                         _ptr(sT), _ld(sT), POW2 if pow2 else 0, _stream(dev, stream))
    _check("fp8_requant_tile_128x1", st)
    return qT, sT


def fp8_quant_block_128x128(w: torch.Tensor, *, pow2: bool = False, transposed: bool = False,
                            q=None, qT=None, s=None, stream=None):
    """128x128 block quantization of BF16 ``w [rows, cols]``.

    Returns ``(q [rows, cols], qT [cols, rows] or None, s [rows/128, cols/128])``."""
    _cuda2d(w, torch.bfloat16, "w")
    rows, cols = w.shape
    dev = w.device
    q = q if q is not None else torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    if transposed:
        qT = qT if qT is not None else torch.empty((cols, rows), dtype=torch.uint8, device=dev)
    else:
        qT = None
    s = s if s is not None else torch.empty((rows // 128, cols // 128), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):   # the handle's device is current for the call
        st = _lib.fp8_quant_block_128x128(_handle(dev), _ptr(w), rows, cols, _ld(w), _ptr(q), _ld(q), _ptr(qT),
                                          _ld(qT), _ptr(s), _ld(s), POW2 if pow2 else 0, _stream(dev, stream))
    _check("fp8_quant_block_128x128", st)
    return q, qT, s


# ------------------------------------------------------------------------ GEMMs

def _out(M, N, out_dtype, C, dev):
    if C is not None:
        _check_output(C, out_dtype, M, N, dev)
        return C
    dt = torch.float32 if out_dtype == OUT_FP32 else torch.bfloat16
    return torch.empty((M, N), dtype=dt, device=dev)


def fp8_gemm_blockscaled(op: int, A: torch.Tensor, sA: torch.Tensor, B: torch.Tensor, sB: torch.Tensor, *,
                         out_dtype: int = OUT_BF16, C: Optional[torch.Tensor] = None, stream=None):
    """Block-scaled FP8 GEMM ``C[M, N] = sum_kb (A_kb B_kb^T) sA sB`` (see mpq.h).

    ``A [M, K]`` and ``B [N, K]`` uint8 E4M3 codes, ``sA [K/128, M]`` float32, ``sB`` per op:
    FPROP ``[N/128, K/128]``, DGRAD ``[K/128, N/128]``, WGRAD ``[K/128, N]``."""
    _cuda2d(A, torch.uint8, "A"); _cuda2d(B, torch.uint8, "B")
    _cuda2d(sA, torch.float32, "sA"); _cuda2d(sB, torch.float32, "sB")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("A and B disagree on K")
    dev = A.device
    C = _out(M, N, out_dtype, C, dev)
    with torch.cuda.device(dev):   # the handle's device is current for the call
        st = _lib.fp8_gemm_blockscaled(_handle(dev), int(op), M, N, K, _ptr(A), _ld(A), _ptr(sA), _ld(sA), _ptr(B),
                                       _ld(B), _ptr(sB), _ld(sB), _ptr(C), _ld(C), int(out_dtype),
                                       _stream(dev, stream))
    _check("fp8_gemm_blockscaled", st)
    return C


def fp8_gemm_mx_pow2(op: int, A: torch.Tensor, sA: torch.Tensor, B: torch.Tensor, sB: torch.Tensor, *,
                     out_dtype: int = OUT_BF16, C: Optional[torch.Tensor] = None, stream=None):
    """The GEMM of :func:`fp8_gemm_blockscaled` for power-of-2 scales (2^-127 .. 2^127), with
    the scales applied by the tensor cores' microscaling MMA and the whole K accumulated in
    FP32 by the tensor cores.  Same arguments and layouts.  A scale outside that set is
    reported by :func:`mpq_check_device_status` (status 9)."""
    _cuda2d(A, torch.uint8, "A"); _cuda2d(B, torch.uint8, "B")
    _cuda2d(sA, torch.float32, "sA"); _cuda2d(sB, torch.float32, "sB")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("A and B disagree on K")
    dev = A.device
    C = _out(M, N, out_dtype, C, dev)
    with torch.cuda.device(dev):   # the handle's device is current for the call
        st = _lib.fp8_gemm_mx_pow2(_handle(dev), int(op), M, N, K, _ptr(A), _ld(A), _ptr(sA), _ld(sA), _ptr(B),
                                   _ld(B), _ptr(sB), _ld(sB), _ptr(C), _ld(C), int(out_dtype), _stream(dev, stream))
    _check("fp8_gemm_mx_pow2", st)
    return C


def fused_workspace_bytes(M_total: int, K: int, G: int) -> int:
    """Workspace bytes for ``fp8_grouped_gemm_blockscaled(..., fuse_quant=True)``."""
    n = ctypes.c_size_t()
    _check("mpq_grouped_fused_workspace_bytes", _lib.mpq_grouped_fused_workspace_bytes(M_total, K, G, ctypes.byref(n)))
    return n.value


def _ensure_workspace(device: torch.device, nbytes: int):
    """Give the device's handle a workspace of at least ``nbytes`` (a torch buffer kept by
    this module; the library itself allocates nothing)."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    h = _handle(device)
    with _hlock:
        buf = _workspaces.get(idx)
        if buf is None or buf.numel() < nbytes:
            # no call in flight, on any stream of the device, still uses the old buffer
            torch.cuda.synchronize(device)
            buf = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
            _workspaces[idx] = buf
            _check("mpq_set_workspace", _lib.mpq_set_workspace(h, _ptr(buf), buf.numel()))


def fp8_grouped_gemm_blockscaled(offsets: torch.Tensor, A: torch.Tensor, sA: Optional[torch.Tensor], B: torch.Tensor,
                                 sB: torch.Tensor, *, out_dtype: int = OUT_BF16, C: Optional[torch.Tensor] = None,
                                 tiles: str = "auto", fuse_quant: bool = False, pow2: bool = False, stream=None):
    """MoE grouped FP8 GEMM: rows ``[off[g], off[g+1])`` of ``A`` use expert ``g``'s weight.

    ``offsets`` int64 CUDA ``[G+1]``; ``A [M, K]`` codes, ``sA [K/128, M]``; ``B [G, N, K]`` codes;
    ``sB [G, N/128, K/128]``.  Rows outside every expert are left untouched in ``C``.
    ``tiles``: ``"rows"`` (token-row tiles, many tokens per expert), ``"weights"`` (weight-row
    tiles sized to each expert's tokens) or ``"auto"`` (rows: on single-SM tiles they stream
    the weights at the HBM rate even for a few tokens per expert)."""
    flags = {"auto": 0, "rows": GROUPED_ROW_TILES, "weights": GROUPED_WEIGHT_TILES}.get(tiles)
    if flags is None:
        raise ValueError("tiles: expected 'auto', 'rows' or 'weights'")
    _check_expert_args(offsets, B, sB)
    if fuse_quant:
        # A is BF16 [M, K], quantized 1x128 inside the launch (pow2: power-of-2 scales)
        _cuda2d(A, torch.bfloat16, "A")
        if sA is not None:
            raise ValueError("sA must be None with fuse_quant=True")
        flags |= FUSE_QUANT_A | (POW2 if pow2 else 0)
    else:
        if pow2:
            raise ValueError("pow2 applies to fuse_quant=True only")
        _cuda2d(A, torch.uint8, "A"); _cuda2d(sA, torch.float32, "sA")
    G, N, K = B.shape
    M = A.shape[0]
    if offsets.numel() != G + 1 or A.shape[1] != K:
        raise ValueError("shape mismatch between offsets, A and B")
    dev = A.device
    C = _out(M, N, out_dtype, C, dev)
    if fuse_quant:
        _ensure_workspace(dev, fused_workspace_bytes(M, K, G))
    with torch.cuda.device(dev):   # the handle's device is current for the call
        st = _lib.fp8_grouped_gemm_blockscaled(_handle(dev), G, _ptr(offsets), M, N, K, _ptr(A), _ld(A), _ptr(sA),
                                               _ld(sA), _ptr(B), K, _ptr(sB), sB.shape[2], _ptr(C), _ld(C),
                                               int(out_dtype), flags, _stream(dev, stream))
    _check("fp8_grouped_gemm_blockscaled", st)
    return C


def fp8_grouped_gemm_swiglu_quant(offsets: torch.Tensor, A: torch.Tensor, sA: Optional[torch.Tensor],
                                  B: torch.Tensor, sB: torch.Tensor, *, pow2: bool = True, fuse_quant: bool = False,
                                  H=False, q=None, s=None, stream=None):
    """MoE up projection with SwiGLU and the 1x128 quantization of its result in the GEMM's
    epilogue.  ``B [G, 2W, K]`` holds each expert's gate weight rows ``[0, W)`` and up weight
    rows ``[W, 2W)``; ``A``/``sA`` as for :func:`fp8_grouped_gemm_blockscaled` (or BF16 ``A``
    with ``fuse_quant=True``).  Returns ``(q [M, W] uint8, s [W/128, M] float32, H)`` where
    ``H [M, 2W]`` BF16 is the SwiGLU input (gate | up), written when ``H`` is True (allocated)
    or a tensor, else None.  ``pow2`` selects power-of-2 scales for the quantized result."""
    _check_expert_args(offsets, B, sB)
    G, N, K = B.shape
    if N % 2:
        raise ValueError("B: expected 2W rows per expert (gate then up)")
    W = N // 2
    if fuse_quant:
        _cuda2d(A, torch.bfloat16, "A")
        if sA is not None:
            raise ValueError("sA must be None with fuse_quant=True")
    else:
        _cuda2d(A, torch.uint8, "A"); _cuda2d(sA, torch.float32, "sA")
    M = A.shape[0]
    if offsets.numel() != G + 1 or A.shape[1] != K:
        raise ValueError("shape mismatch between offsets, A and B")
    dev = A.device
    q = q if q is not None else torch.empty((M, W), dtype=torch.uint8, device=dev)
    s = s if s is not None else torch.empty((W // 128, M), dtype=torch.float32, device=dev)
    if H is True:
        H = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    elif H is False:
        H = None
    elif H is not None:
        _check_output(H, OUT_BF16, M, N, dev)
    flags = (POW2 if pow2 else 0) | (FUSE_QUANT_A if fuse_quant else 0)
    if fuse_quant:
        _ensure_workspace(dev, fused_workspace_bytes(M, K, G))
    with torch.cuda.device(dev):   # the handle's device is current for the call
        st = _lib.fp8_grouped_gemm_swiglu_quant(_handle(dev), G, _ptr(offsets), M, W, K, _ptr(A), _ld(A), _ptr(sA),
                                                _ld(sA), _ptr(B), K, _ptr(sB), sB.shape[2], _ptr(H), _ld(H),
                                                _ptr(q), _ld(q), _ptr(s), _ld(s), flags, _stream(dev, stream))
    _check("fp8_grouped_gemm_swiglu_quant", st)
    return q, s, H


def _check_expert_args(offsets: torch.Tensor, B: torch.Tensor, sB: torch.Tensor, device: bool = True):
    """The expert ranges and weights of a grouped GEMM: dtype and layout, then (unless
    ``device`` is False) the device, so that a wrong dtype is reported as such wherever the
    tensor lives."""
    if offsets.dtype != torch.int64 or offsets.dim() != 1 or not offsets.is_contiguous():
        raise TypeError(f"offsets: expected a contiguous 1-D int64 tensor, got {offsets.dtype} {tuple(offsets.shape)}")
    if B.dtype != torch.uint8 or B.dim() != 3 or not B.is_contiguous():
        raise TypeError("B: expected a contiguous [G, N, K] uint8 tensor")
    if sB.dtype != torch.float32 or sB.dim() != 3 or not sB.is_contiguous():
        raise TypeError("sB: expected a contiguous [G, N/128, K/128] float32 tensor")
    if not device:
        return
    if not (offsets.is_cuda and B.is_cuda and sB.is_cuda):
        raise TypeError("offsets, B and sB must be CUDA tensors")
    if not (offsets.device == B.device == sB.device):
        raise ValueError("offsets, B and sB must be on one device")


def _check_output(C: torch.Tensor, out_dtype: int, M: int, N: int, device: torch.device):
    """A caller-given output: the dtype the kernel writes (float32 for OUT_FP32, bfloat16
    for OUT_BF16), [M, N] with unit column stride, on the inputs' device."""
    want = {OUT_FP32: torch.float32, OUT_BF16: torch.bfloat16}.get(out_dtype)
    if want is None:
        raise ValueError(f"out_dtype: expected OUT_BF16 or OUT_FP32, got {out_dtype}")
    if C.dtype != want:
        raise TypeError(f"C: out_dtype asks for {want}, got {C.dtype}")
    if C.dim() != 2 or tuple(C.shape) != (M, N):
        raise ValueError(f"C: expected shape {(M, N)}, got {tuple(C.shape)}")
    if not C.is_cuda or C.device != device:
        raise TypeError(f"C: expected a CUDA tensor on {device}, got {C.device}")


NOALLOC_SCRATCH_BYTES = 64 << 20


def fp8_grouped_gemm_fused_quant_noalloc(offsets: torch.Tensor, X: torch.Tensor, B: torch.Tensor, sB: torch.Tensor,
                                         C: torch.Tensor, *, out_dtype: int = OUT_BF16, pow2: bool = False,
                                         stream=None):
    """Fused 1x128 quantization + row-tile grouped GEMM that allocates nothing: the
    quantized activations stay in the library's fixed scratch area (NOALLOC_SCRATCH_BYTES),
    so the output ``C`` must be given (float32 for OUT_FP32, bfloat16 for OUT_BF16).  For
    callers that must not allocate device memory while they run.  Calls that overlap in
    time (other streams or threads) race on the one scratch area; the first call per device
    should come before any stream capture."""
    _check_expert_args(offsets, B, sB, device=False)
    if X.dtype != torch.bfloat16 or X.dim() != 2:
        raise TypeError(f"X: expected a 2-D bfloat16 tensor, got {X.dtype} {tuple(X.shape)}")
    G, N, K = B.shape
    M = X.shape[0]
    if offsets.numel() != G + 1 or X.shape[1] != K:
        raise ValueError("shape mismatch between offsets, X and B")
    _check_output(C, out_dtype, M, N, B.device)
    _check_expert_args(offsets, B, sB)
    _cuda2d(X, torch.bfloat16, "X")
    if X.device != B.device:
        raise ValueError("X must be on the device of B")
    dev = X.device
    with torch.cuda.device(dev):   # the handle's device is current for the call
        st = _lib.fp8_grouped_gemm_fused_quant_noalloc(_handle(dev), G, _ptr(offsets), M, N, K, _ptr(X), _ld(X), _ptr(B),
                                                       K, _ptr(sB), sB.shape[2], _ptr(C), _ld(C), int(out_dtype),
                                                       POW2 if pow2 else 0, _stream(dev, stream))
    _check("fp8_grouped_gemm_fused_quant_noalloc", st)
    return C


# --------------------------------------------------------------------- status

def mpq_check_device_status(device=None, stream=None):
    """Synchronize the stream and return (status, where) from the device status word."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    where = ctypes.c_int(0)
    with torch.cuda.device(dev):   # the handle's device is current for the call
        st = _lib.mpq_check_device_status(_handle(dev), _stream(dev, stream), ctypes.byref(where))
    return st, where.value


def mpq_set_wait_timeout(timeout_ns: int, device=None):
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    _check("mpq_set_wait_timeout", _lib.mpq_set_wait_timeout(_handle(dev), int(timeout_ns)))


def mpq_set_gemm_cta_pair(mode, device=None):
    """Tiling of the row-tiled GEMMs: 1 or True (default) -- 2-SM pair tiles for dense GEMMs,
    for grouped ones for the experts with 1024 rows or more (the others on single-SM tiles,
    in a second launch); 0 or False -- single-SM tiles everywhere; 2 -- pair tiles
    everywhere."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    _check("mpq_set_gemm_cta_pair", _lib.mpq_set_gemm_cta_pair(_handle(dev), int(mode)))


def mpq_set_gemm_stream_k(mode, device=None):
    """Schedule of the dense GEMM: 1 (default) -- stream-K when the last wave of tiles would
    leave more than a tenth of the SMs' time idle; 0 -- data-parallel whole tiles; 2 --
    stream-K whenever the tiles fill more than one wave."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    _check("mpq_set_gemm_stream_k", _lib.mpq_set_gemm_stream_k(_handle(dev), int(mode)))


def mpq_selftest_wait_timeout(timeout_ns: int = 1_000_000, device=None, stream=None):
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    with torch.cuda.device(dev):   # the handle's device is current for the call
        _check("mpq_selftest_wait_timeout", _lib.mpq_selftest_wait_timeout(_handle(dev), int(timeout_ns),
                                                                             _stream(dev, stream)))

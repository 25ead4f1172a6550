"""CPU oracle for fine-grained FP8 quantization and block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
leg of the benchmark may import this package.  The product path (the CUDA
library and its Python binding) never imports it, and it imports nothing from
the product path.

The arithmetic lives in ``mpq_oracle.c`` (plain single-threaded C, no SIMD, no
fast-math); this module only compiles it on first use and marshals numpy
arrays.  Every function cites, in the C source, the passage of the source pages
it follows.  Pins that tie it to something other than itself are in
``tests/test_oracle_pins.py``.

Parity status: every function here is pinned (see the tests).  The error-versus-K
study of the benchmark is a report against the unquantized inputs, computed there,
and is not a parity gate.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mpq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmpq_oracle.so")
_lock = threading.Lock()
_lib = None

FPROP, DGRAD, WGRAD = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, IEEE arithmetic)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off",
             "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int64
        lib.mpqo_e4m3_decode.restype = ctypes.c_double
        lib.mpqo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.mpqo_e4m3_encode.restype = ctypes.c_uint8
        lib.mpqo_e4m3_encode.argtypes = [ctypes.c_float]
        lib.mpqo_group_scale.restype = ctypes.c_float
        lib.mpqo_group_scale.argtypes = [ctypes.c_float, ctypes.c_int]
        lib.mpqo_quant_tile_1x128.restype = None
        lib.mpqo_quant_tile_1x128.argtypes = [P, I, I, I, P, I, P, I, ctypes.c_int]
        lib.mpqo_quant_tile_128x1.restype = None
        lib.mpqo_quant_tile_128x1.argtypes = [P, I, I, I, P, I, P, I, ctypes.c_int]
        lib.mpqo_quant_block_128x128.restype = None
        lib.mpqo_quant_block_128x128.argtypes = [P, I, I, I, P, I, P, I, P, I, ctypes.c_int]
        lib.mpqo_exp_f32.restype = ctypes.c_float
        lib.mpqo_exp_f32.argtypes = [ctypes.c_float]
        lib.mpqo_silu_f32.restype = ctypes.c_float
        lib.mpqo_silu_f32.argtypes = [ctypes.c_float]
        lib.mpqo_swiglu_quant_1x128.restype = None
        lib.mpqo_swiglu_quant_1x128.argtypes = [P, I, I, I, P, I, P, I, ctypes.c_int]
        lib.mpqo_requant_tile_128x1.restype = None
        lib.mpqo_requant_tile_128x1.argtypes = [P, I, I, I, P, I, P, I, P, I, ctypes.c_int]
        lib.mpqo_gemm_ref.restype = None
        lib.mpqo_gemm_ref.argtypes = [ctypes.c_int, I, I, I, P, I, P, I, P, I, P, I, P, P, I]
        lib.mpqo_gemm_ref_at.restype = None
        lib.mpqo_gemm_ref_at.argtypes = [ctypes.c_int, I, P, I, P, I, P, I, P, I, P, P, I, P, P]
        lib.mpqo_grouped_gemm_ref.restype = None
        lib.mpqo_grouped_gemm_ref.argtypes = [I, P, I, I, P, I, P, I, P, I, P, I, P, P, I]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


# ------------------------------------------------------------------ codec

def e4m3_decode(codes) -> np.ndarray:
    """Decode E4M3 byte codes to float64 (NaN for 0x7F / 0xFF)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    flat_c, flat_o = c.reshape(-1), out.reshape(-1)
    for i in range(flat_c.size):
        flat_o[i] = lib.mpqo_e4m3_decode(int(flat_c[i]))
    return out


def e4m3_encode(values) -> np.ndarray:
    """Encode binary32 values to E4M3 codes (RNE, saturating at +-448)."""
    lib = _load()
    v = np.asarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    flat_v, flat_o = v.reshape(-1), out.reshape(-1)
    for i in range(flat_v.size):
        flat_o[i] = lib.mpqo_e4m3_encode(float(flat_v[i]))
    return out


def group_scale(amax: float, pow2: bool = False) -> np.float32:
    """Scale of one group from its max-abs value (amax/448, or the power of 2)."""
    return np.float32(_load().mpqo_group_scale(float(np.float32(amax)), int(pow2)))


# ------------------------------------------------------------- quantizers

def quant_tile_1x128(x_bf16_bits: np.ndarray, pow2: bool = False):
    """Row-wise 1x128 quantization of a [rows, cols] BF16 matrix (given as uint16 bits).

    Returns (q uint8 [rows, cols], s float32 [cols/128, rows])."""
    x = _c(x_bf16_bits, np.uint16)
    rows, cols = x.shape
    assert cols % 128 == 0
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((cols // 128, rows), np.float32)
    _load().mpqo_quant_tile_1x128(_ptr(x), rows, cols, cols, _ptr(q), cols, _ptr(s), rows, int(pow2))
    return q, s


def quant_tile_128x1(x_bf16_bits: np.ndarray, pow2: bool = False):
    """Column-wise 128x1 quantization (groups of 128 along rows), stored transposed.

    Returns (qT uint8 [cols, rows], sT float32 [rows/128, cols])."""
    x = _c(x_bf16_bits, np.uint16)
    rows, cols = x.shape
    assert rows % 128 == 0
    qT = np.empty((cols, rows), np.uint8)
    sT = np.empty((rows // 128, cols), np.float32)
    _load().mpqo_quant_tile_128x1(_ptr(x), rows, cols, cols, _ptr(qT), rows, _ptr(sT), cols, int(pow2))
    return qT, sT


def exp_f32(x) -> np.ndarray:
    """The path's binary32 exponential (Cody-Waite reduction + degree-7 Taylor), elementwise."""
    lib = _load()
    x = np.asarray(x, np.float32)
    return np.array([lib.mpqo_exp_f32(float(v)) for v in x.ravel()], np.float32).reshape(x.shape)


def silu_f32(x) -> np.ndarray:
    lib = _load()
    x = np.asarray(x, np.float32)
    return np.array([lib.mpqo_silu_f32(float(v)) for v in x.ravel()], np.float32).reshape(x.shape)


def swiglu_quant_1x128(hcat_bf16_bits: np.ndarray, pow2: bool = True):
    """SwiGLU of [rows, 2W] BF16 (gate | up) and the 1x128 quantization of the result.

    Returns (q uint8 [rows, W], s float32 [W/128, rows])."""
    h = _c(hcat_bf16_bits, np.uint16)
    rows, w2 = h.shape
    assert w2 % 256 == 0
    w = w2 // 2
    q = np.empty((rows, w), np.uint8)
    s = np.empty((w // 128, rows), np.float32)
    _load().mpqo_swiglu_quant_1x128(_ptr(h), rows, w, w2, _ptr(q), w, _ptr(s), rows, int(pow2))
    return q, s


def requant_tile_128x1(q: np.ndarray, s: np.ndarray, pow2: bool = False):
    """Re-quantize a row-wise 1x128 quantization (codes q uint8 [rows, cols], scales s
    float32 [cols/128, rows]) into 128x1 groups along rows: dequantize to binary32
    (dec(q) * s), then quantize the column groups.  Returns (qT uint8 [cols, rows],
    sT float32 [rows/128, cols])."""
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    rows, cols = q.shape
    assert rows % 128 == 0 and cols % 128 == 0 and s.shape == (cols // 128, rows)
    qT = np.empty((cols, rows), np.uint8)
    sT = np.empty((rows // 128, cols), np.float32)
    _load().mpqo_requant_tile_128x1(_ptr(q), rows, cols, cols, _ptr(s), rows, _ptr(qT), rows, _ptr(sT), cols,
                                    int(pow2))
    return qT, sT


def quant_block_128x128(w_bf16_bits: np.ndarray, pow2: bool = False, transposed: bool = False):
    """128x128 block quantization of a [rows, cols] BF16 matrix.

    Returns (q [rows, cols], qT [cols, rows] or None, s float32 [rows/128, cols/128])."""
    w = _c(w_bf16_bits, np.uint16)
    rows, cols = w.shape
    assert rows % 128 == 0 and cols % 128 == 0
    q = np.empty((rows, cols), np.uint8)
    qT = np.empty((cols, rows), np.uint8) if transposed else None
    s = np.empty((rows // 128, cols // 128), np.float32)
    _load().mpqo_quant_block_128x128(
        _ptr(w), rows, cols, cols, _ptr(q), cols,
        _ptr(qT) if transposed else None, rows, _ptr(s), cols // 128, int(pow2))
    return q, qT, s


# ------------------------------------------------------------------- GEMM

def gemm_ref(op: int, qa: np.ndarray, sa: np.ndarray, qb: np.ndarray, sb: np.ndarray):
    """FP64 brute-force block-scaled GEMM, C[m, n] = sum_k A[m,k] B[n,k].

    qa [M, K] codes, sa [K/128, M]; qb [N, K] codes; sb laid out per ``op``
    (FPROP [N/128, K/128], DGRAD [K/128, N/128], WGRAD [K/128, N]).
    Returns (ref, absref) float64 [M, N]."""
    qa = _c(qa, np.uint8); qb = _c(qb, np.uint8)
    sa = _c(sa, np.float32); sb = _c(sb, np.float32)
    M, K = qa.shape
    N = qb.shape[0]
    ref = np.empty((M, N), np.float64)
    absref = np.empty((M, N), np.float64)
    _load().mpqo_gemm_ref(op, M, N, K, _ptr(qa), K, _ptr(sa), sa.shape[1],
                          _ptr(qb), K, _ptr(sb), sb.shape[1], _ptr(ref), _ptr(absref), N)
    return ref, absref


def gemm_ref_at(op: int, qa, sa, qb, sb, ms, ns):
    """``gemm_ref`` at the listed (m, n) positions only."""
    qa = _c(qa, np.uint8); qb = _c(qb, np.uint8)
    sa = _c(sa, np.float32); sb = _c(sb, np.float32)
    ms = _c(np.asarray(ms, np.int64), np.int64)
    ns = _c(np.asarray(ns, np.int64), np.int64)
    K = qa.shape[1]
    ref = np.empty(ms.size, np.float64)
    absref = np.empty(ms.size, np.float64)
    _load().mpqo_gemm_ref_at(op, K, _ptr(qa), K, _ptr(sa), sa.shape[1], _ptr(qb), qb.shape[1],
                             _ptr(sb), sb.shape[1], _ptr(ms), _ptr(ns), ms.size,
                             _ptr(ref), _ptr(absref))
    return ref, absref


def grouped_gemm_ref(offsets, qa, sa, qb, sb):
    """Grouped FPROP over experts: rows [off[g], off[g+1]) use weight qb[g] ([G, N, K])
    with block scales sb[g] ([G, N/128, K/128]).  Rows of no expert are left at 0."""
    off = _c(np.asarray(offsets, np.int64), np.int64)
    qa = _c(qa, np.uint8); qb = _c(qb, np.uint8)
    sa = _c(sa, np.float32); sb = _c(sb, np.float32)
    G, N, K = qb.shape
    M = qa.shape[0]
    ref = np.zeros((M, N), np.float64)
    absref = np.zeros((M, N), np.float64)
    _load().mpqo_grouped_gemm_ref(G, _ptr(off), N, K, _ptr(qa), K, _ptr(sa), sa.shape[1],
                                  _ptr(qb), K, _ptr(sb), sb.shape[2], _ptr(ref), _ptr(absref), N)
    return ref, absref

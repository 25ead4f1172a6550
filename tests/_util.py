"""Test helpers: host copies of device tensors and the GEMM parity bound."""
import numpy as np
import torch


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().float().numpy()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def gemm_within_tolerance(gpu, ref, absref):
    """Per-element parity bound for block-scaled GEMM outputs:
    |gpu - ref| <= 2^-7 |ref| + 1e-6 sum_k |a_k b_k|, with the GPU's BF16 or FP32 output
    taken as exact and ref the FP64 oracle."""
    gpu = np.asarray(gpu, np.float64)
    err = np.abs(gpu - ref)
    bound = 2.0 ** -7 * np.abs(ref) + 1e-6 * absref
    ok = err <= bound
    return ok, err, bound


def assert_gemm_close(gpu, ref, absref, what=""):
    ok, err, bound = gemm_within_tolerance(gpu, ref, absref)
    if not ok.all():
        idx = np.argwhere(~ok)[:8]
        details = [(tuple(int(v) for v in i), float(np.asarray(gpu, np.float64)[tuple(i)]), float(ref[tuple(i)]),
                    float(bound[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; first: {details}")

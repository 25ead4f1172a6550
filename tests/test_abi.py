"""Host-side checks (no GPU): the library builds, loads and exports every entry point
declared in include/mpq.h; argument validation happens before any device work."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mpq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z][a-z0-9_]*)\s*\(",
                                 src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["fp8_quant_tile_1x128", "fp8_quant_block_128x128", "fp8_requant_tile_128x1", "fp8_swiglu_quant_1x128",
              "fp8_gemm_blockscaled",
              "fp8_grouped_gemm_blockscaled", "mpq_version", "mpq_create", "mpq_destroy",
              "mpq_check_device_status"]:
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    lib.mpq_version.restype = ctypes.c_char_p
    assert b"sm_103a" in lib.mpq_version()
    lib.mpq_status_string.restype = ctypes.c_char_p
    assert lib.mpq_status_string(6) == b"device-side wait timed out"
    assert lib.mpq_status_string(8) == b"the current device is not the handle's device"
    assert lib.mpq_status_string(99) == b"unknown status"


def test_every_status_code_has_a_string_in_the_library_and_the_binding(lib):
    # the codes of the header's mpq_status enum, each with its own text on both sides
    src = open(os.path.join(ROOT, "include", "mpq.h")).read()
    codes = [int(v) for v in re.findall(r"MPQ_(?:OK|ERR_[A-Z]+)\s*=\s*(\d+)", src)]
    assert codes == list(range(len(codes)))
    lib.mpq_status_string.restype = ctypes.c_char_p
    texts = [lib.mpq_status_string(c) for c in codes]
    assert b"unknown status" not in texts and len(set(texts)) == len(texts)
    binding = open(os.path.join(ROOT, "mixed_precision_quant_b300", "__init__.py")).read()
    table = re.search(r"_STATUS = \{(.*?)\}", binding, flags=re.S).group(1)
    assert sorted(int(k) for k in re.findall(r"(\d+):", table)) == codes


def test_null_handle_rejected_before_any_cuda_call(lib):
    # every compute entry point validates its handle first and returns MPQ_ERR_NULL
    P = ctypes.c_void_p
    assert lib.mpq_check_device_status(P(0), P(0), P(0)) == 1
    assert lib.mpq_destroy(P(0)) == 1
    assert lib.mpq_create(P(0)) == 1
    I = ctypes.c_int64
    assert lib.fp8_requant_tile_128x1(P(0), P(0), I(128), I(128), I(128), P(0), I(128), P(0), I(128), P(0),
                                      I(128), ctypes.c_uint32(0), P(0)) == 1
    assert lib.fp8_swiglu_quant_1x128(P(0), P(0), I(128), I(128), I(256), P(0), I(128), P(0), I(128),
                                      ctypes.c_uint32(0), P(0)) == 1


def test_python_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib.util
    import shutil
    pkg = tmp_path / "mixed_precision_quant_b300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "mixed_precision_quant_b300", "__init__.py"), pkg / "__init__.py")
    spec = importlib.util.spec_from_file_location("mpq_copy", pkg / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)

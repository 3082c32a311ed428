"""The C-ABI library loads, exports every symbol include/ub.h declares, and validates
arguments on the host before any device work (no GPU needed)."""
import ctypes
import os
import re

import pytest
import torch

from gemm_overlap_gemms_gb300 import _build, ub

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ub.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ub.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ub_create", "ub_set_active_shape", "ag_gemm", "gemm_rs", "ub_destroy"):
        assert required in names
    assert sorted(ub.EXPORTS) == names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_no_cpu_fallback_when_library_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(ub, "_lib", None)
    monkeypatch.setattr(ub, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        ub.load()


C = ub.CODES


@pytest.mark.parametrize("shape,code", [
    ([4096, 1024], 0),
    ([8192, 1024], 0),
    ([4096], C["UB_ERR_RANK"]),
    ([4096, 1024, 1], C["UB_ERR_RANK"]),
    ([0, 1024], C["UB_ERR_ZERO"]),
    ([-4, 1024], C["UB_ERR_ZERO"]),
    ([4096, 0], C["UB_ERR_ZERO"]),
    ([8196, 1024], C["UB_ERR_CAPACITY"]),
    ([4096, 2048], C["UB_ERR_HIDDEN"]),
    ([4094, 1024], C["UB_ERR_DIVISIBLE"]),
    ([4, 1024], 0),
])
def test_validate_active_shape(lib, shape, code):
    assert ub.validate_active_shape(shape, 8192, 1024, 4) == code


def test_validate_matches_oracle_rule_order(lib):
    import oracle
    order = [0, C["UB_ERR_RANK"], C["UB_ERR_ZERO"], C["UB_ERR_CAPACITY"], C["UB_ERR_HIDDEN"],
             C["UB_ERR_DIVISIBLE"]]
    for shape in ([8, 16], [8], [0, 16], [40, 16], [8, 32], [6, 16], [0, 32], [40, 32], [6, 32]):
        assert ub.validate_active_shape(shape, 32, 16, 4) == order[
            oracle.check_active_shape(shape, 32, 16, 4)]


@pytest.mark.parametrize("args,code", [
    ((512, 256, 0), C["UB_ERR_ARG"]),
    ((512, 256, 9), C["UB_ERR_ARG"]),
    ((0, 256, 2), C["UB_ERR_ZERO"]),
    ((512, 0, 2), C["UB_ERR_ZERO"]),
    ((512, 250, 2), C["UB_ERR_ALIGN"]),
    ((511, 256, 2), C["UB_ERR_DIVISIBLE"]),
])
def test_create_rejects_bad_arguments_before_device_work(lib, args, code):
    h = ctypes.c_void_p()
    assert lib.ub_create(*args, 0, ctypes.byref(h)) == code
    assert h.value is None
    assert ub.last_error()


def test_create_rejects_other_dtypes(lib):
    h = ctypes.c_void_p()
    assert lib.ub_create(512, 256, 2, 1, ctypes.byref(h)) == C["UB_ERR_DTYPE"]


def test_null_handle_is_rejected(lib):
    assert lib.ub_set_active_shape(None, 8, 8) == C["UB_ERR_ARG"]
    assert lib.ag_gemm(None, None, None, 8, None, None) == C["UB_ERR_ARG"]
    assert lib.gemm_rs(None, None, None, 8, None, None) == C["UB_ERR_ARG"]
    assert lib.ub_destroy(None) == C["UB_ERR_ARG"]


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device error path")
def test_create_without_a_device_fails_cleanly(lib):
    h = ctypes.c_void_p()
    assert lib.ub_create(512, 256, 2, 0, ctypes.byref(h)) == C["UB_ERR_CUDA"]
    assert h.value is None
    assert "cuda" in ub.last_error().lower() or "driver" in ub.last_error().lower()


def _header_enum(prefix):
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return {name: int(val) for name, val in re.findall(r"\b(%s[A-Z_]*)\s*=\s*(-?\d+)" % prefix, text)}


def test_binding_constants_match_the_header():
    """Error codes, option keys and operation ids of the binding are the header's."""
    errs = _header_enum("UB_ERR_")
    assert errs == ub.CODES
    assert _header_enum("UB_OK") == {"UB_OK": ub.UB_OK}
    opts = {k[len("UB_OPT_"):].lower(): v for k, v in _header_enum("UB_OPT_").items()}
    assert opts == ub.OPTIONS
    ops = {k[len("UB_OP_"):].lower(): v for k, v in _header_enum("UB_OP_").items()}
    assert ops == ub.OPS
    m = re.search(r"#define UB_MAX_TP (\d+)", open(HEADER).read())
    assert int(m.group(1)) == ub.MAX_TP

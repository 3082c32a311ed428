"""The allocation-free AG-GEMM entry point, ag_gemm_noalloc.

Some callers cannot call cudaMalloc -- code running inside another framework's memory
pool or a custom allocator that owns the device, plugins whose device allocations are
audited, processes that must not grow their device footprint after start-up -- so they
cannot create a handle, whose user buffer is allocated. ag_gemm_noalloc runs the same
AG-GEMM with its scratch in a fixed file-scope device array instead.

This file is collected last on purpose, so that a run stopping at the first failure
has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gemm_overlap_gemms_gb300 import _build, synth, ub


def _lib():
    _build.build()
    return ub.load()


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    L = _lib()
    dummy = (ctypes.c_void_p * 2)(16, 16)
    T, H = 2 * 4096, 4096        # 2 * 16M elements: twice the fixed maximum
    rc = L.ag_gemm_noalloc(dummy, 2, T, H, ctypes.c_void_p(16), 256, ctypes.c_void_p(16), None)
    assert rc == ub.CODES["UB_ERR_CAPACITY"]
    assert "exceeds the fixed scratch" in ub.last_error()
    four = (ctypes.c_void_p * 4)(16, 16, 16, 16)
    # one chunk of 8 rows past the maximum is already rejected
    rc = L.ag_gemm_noalloc(four, 4, 4096 + 4, 4096, ctypes.c_void_p(16), 256, ctypes.c_void_p(16), None)
    assert rc == ub.CODES["UB_ERR_CAPACITY"]
    rc = L.ag_gemm_noalloc(four, 4, 6, 256, ctypes.c_void_p(16), 256, ctypes.c_void_p(16), None)
    assert rc == ub.CODES["UB_ERR_DIVISIBLE"]


@pytest.mark.gpu
def test_noalloc_binding_checks_shapes_before_the_call():
    """The C entry point cannot see tensor sizes, so the binding rejects a short Y or a
    weight of the wrong inner size before anything reaches the device."""
    _lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    shards = [torch.zeros((16, 64), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    Wt = torch.zeros((32, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError, match="Wt must be"):
        ub.ag_gemm_noalloc(shards, torch.zeros((32, 72), dtype=torch.bfloat16, device=dev))
    with pytest.raises(ValueError, match="Y must be"):
        ub.ag_gemm_noalloc(shards, Wt, torch.zeros((31, 32), dtype=torch.bfloat16, device=dev))
    with pytest.raises(ValueError, match="Y must be"):
        ub.ag_gemm_noalloc(shards, Wt, torch.zeros((32, 40), dtype=torch.bfloat16, device=dev))
    with pytest.raises(TypeError):          # host tensors are refused outright
        ub.ag_gemm_noalloc([s.cpu() for s in shards], Wt)


def _check(Y: torch.Tensor, T: int, G: np.ndarray, Yref: np.ndarray, Y_handle: torch.Tensor, what: str):
    y = Y[:T].float().cpu().numpy().astype(np.float64)
    lim = 2e-2 * np.maximum(1.0, np.abs(Yref))
    assert np.all(np.abs(y - Yref) <= lim), "%s: differs from the oracle" % what
    h = Y_handle[:T].float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(y - h) <= 2e-2 * np.maximum(1.0, np.abs(h))), "%s: differs from ag_gemm" % what
    tail = Y[T:].contiguous().view(torch.int16)
    assert bool((tail == -1).all().item()), "%s: rows >= T of Y were written" % what


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_handle_path_on_two_calls_in_a_row():
    _lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    g = synth.generator(seed=21)
    # (tp, T, hidden, N): the first call fills the fixed scratch exactly (T * hidden ==
    # NOALLOC_MAX_ELEMS, so the last chunk ends at the array's last byte); the second is
    # smaller, with a ragged chunk of 129 rows, and runs on the scratch the first left.
    cases = [(4, 4096, 4096, 256), (4, 4 * 129, 512, 384)]
    assert cases[0][1] * cases[0][2] == ub.NOALLOC_MAX_ELEMS
    for tp, T, H, N in cases:
        c = T // tp
        shards_cpu = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
        Wt_cpu = synth.normal_bf16((N, H), H ** -0.5, g)
        shards = [s.to(dev) for s in shards_cpu]
        Wt = Wt_cpu.to(dev)
        Y = torch.full((T + 7, N), -1, dtype=torch.int16, device=dev).view(torch.bfloat16)
        ub.ag_gemm_noalloc(shards, Wt, Y)
        torch.cuda.synchronize()
        with ub.UserBuffer([T, H], tp) as buf:
            buf.set_active_shape([T, H])
            Y_handle = buf.ag_gemm(shards, Wt)
            torch.cuda.synchronize()
            assert buf.query_status() == ub.UB_OK
        G, Yref = oracle.ag_gemm([synth.to_u16(s) for s in shards_cpu], synth.to_u16(Wt_cpu))
        _check(Y, T, G, Yref, Y_handle, "tp=%d T=%d hidden=%d N=%d" % (tp, T, H, N))

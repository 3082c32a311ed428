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
    rc = L.ag_gemm_noalloc(four, 4, 6, 256, ctypes.c_void_p(16), 256, ctypes.c_void_p(16), None)
    assert rc == ub.CODES["UB_ERR_DIVISIBLE"]


@pytest.mark.gpu
def test_noalloc_matches_handle_path_on_two_calls_in_a_row():
    _lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    tp, H, N = 4, 512, 384
    g = synth.generator(seed=21)
    Wt = synth.normal_bf16((N, H), H ** -0.5, g).to(dev)
    for T in (4 * 129, 4 * 64):   # two calls in a row; the second one smaller
        c = T // tp
        shards = [synth.normal_bf16((c, H), 1.0, g).to(dev) for _ in range(tp)]
        Y_free = ub.ag_gemm_noalloc(shards, Wt)
        with ub.UserBuffer([4 * 129, H], tp) as buf:
            buf.set_active_shape([T, H])
            Y_ref = buf.ag_gemm(shards, Wt)
            torch.cuda.synchronize()
            assert buf.query_status() == ub.UB_OK
        a = Y_free.float().cpu().numpy()
        b = Y_ref.float().cpu().numpy()
        assert np.all(np.abs(a - b) <= 2e-2 * np.maximum(1.0, np.abs(b))), "T=%d" % T

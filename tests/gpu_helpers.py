"""Shared helpers of the GPU parity tests: run the library, run the oracle, compare."""
import numpy as np
import torch

import oracle
from gemm_overlap_gemms_gb300 import synth, ub

SENTINEL_BITS = -1  # int16 view of 0xFFFF, a NaN pattern no result can produce
REL_TOL = 2e-2      # |gpu - oracle| <= REL_TOL * max(1, |oracle|), bf16 in, fp32 accumulate


def dev():
    return torch.device("cuda", torch.cuda.current_device())


def sentinel(shape, device=None):
    t = torch.full(tuple(shape), SENTINEL_BITS, dtype=torch.int16, device=device or dev())
    return t.view(torch.bfloat16)


def is_sentinel(t: torch.Tensor) -> bool:
    return bool((t.contiguous().view(torch.int16) == SENTINEL_BITS).all().item())


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what: str):
    g = gpu.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    err = np.abs(g - ref)
    lim = REL_TOL * np.maximum(1.0, np.abs(ref))
    bad = err > lim
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError("%s: %d of %d elements out of tolerance; first at %s: gpu %r oracle %r"
                             % (what, int(bad.sum()), bad.size, tuple(idx), g[tuple(idx)],
                                ref[tuple(idx)]))


def assert_exact(gpu: torch.Tensor, ref: np.ndarray, what: str):
    g = gpu.float().cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(g, ref, err_msg=what)


def run_ag(buf: "ub.UserBuffer", shards_cpu, Wt_cpu, y_rows=None):
    """AG-GEMM on the GPU with a sentinel-filled output of y_rows (>= T) rows."""
    T, H = buf.active_shape
    N = Wt_cpu.shape[0]
    shards = [s.to(dev()) for s in shards_cpu]
    Wt = Wt_cpu.to(dev())
    Y = sentinel((y_rows or T, N))
    buf.ag_gemm(shards, Wt, Y)
    torch.cuda.synchronize()
    return Y


def run_rs(buf: "ub.UserBuffer", A_cpu, Bt_cpu, pad=3):
    """GEMM-RS on the GPU; each output block is a view into one sentinel-filled buffer
    with `pad` guard rows after it. Returns (blocks, whole buffer)."""
    T, H = buf.active_shape
    tp = buf.tp
    c = T // tp
    A = [a.to(dev()) for a in A_cpu]
    Bt = [b.to(dev()) for b in Bt_cpu]
    big = sentinel((tp * (c + pad), H))
    Ys = [big[r * (c + pad): r * (c + pad) + c] for r in range(tp)]
    buf.gemm_rs(A, Bt, Ys)
    torch.cuda.synchronize()
    for r in range(tp):
        assert is_sentinel(big[r * (c + pad) + c: (r + 1) * (c + pad)]), "guard rows after block %d" % r
    return Ys, big


def oracle_ag(shards_cpu, Wt_cpu):
    return oracle.ag_gemm([synth.to_u16(s) for s in shards_cpu], synth.to_u16(Wt_cpu))


def oracle_rs(A_cpu, Bt_cpu):
    return oracle.gemm_rs([synth.to_u16(a) for a in A_cpu], [synth.to_u16(b) for b in Bt_cpu])

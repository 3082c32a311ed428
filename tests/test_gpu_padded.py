"""Padded-to-capacity comparator (the fallback the pages describe for varying token
counts: pad every microbatch to the configured maximum). Its real rows must agree with
the active-shape result and with the oracle; the benchmark times both."""
import numpy as np
import pytest
import torch

from gemm_overlap_gemms_gb300 import synth, ub
from gpu_helpers import assert_close, dev, oracle_ag, oracle_rs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [300, 1020])
def test_padded_matches_active_shape(T):
    tp, H, N, K, cap = 4, 256, 384, 512, 1024
    g = synth.generator(seed=31)
    shards, Wt = synth.ag_inputs(T, H, N, tp, g)
    A, Bt = synth.rs_inputs(T, K, H, tp, g)
    X = torch.cat(shards)
    d = dev()
    with ub.UserBuffer([cap, H], tp) as buf:
        buf.set_active_shape([T, H])
        Y_act = buf.ag_gemm([s.to(d) for s in shards], Wt.to(d))
        R_act = buf.gemm_rs([a.to(d) for a in A], [b.to(d) for b in Bt])
        # padded: real tokens first, zeros after, every microbatch at T = capacity
        Xp = torch.zeros((cap, H), dtype=torch.bfloat16, device=d)
        Xp[:T] = X.to(d)
        Ap = []
        for a in A:
            t = torch.zeros((cap, K), dtype=torch.bfloat16, device=d)
            t[:T] = a.to(d)
            Ap.append(t)
        buf.set_active_shape([cap, H])
        cc = cap // tp
        Y_pad = buf.ag_gemm([Xp[r * cc:(r + 1) * cc] for r in range(tp)], Wt.to(d))
        R_pad = buf.gemm_rs(Ap, [b.to(d) for b in Bt])
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    _, Yref = oracle_ag(shards, Wt)
    assert_close(Y_act, Yref, "active AG")
    assert_close(Y_pad[:T], Yref, "padded AG, real rows")
    assert torch.count_nonzero(Y_pad[T:].float()).item() == 0     # zero rows give zero outputs
    S_ref, _ = oracle_rs(A, Bt)
    assert_close(torch.cat(R_act), S_ref, "active RS")
    assert_close(torch.cat(R_pad)[:T], S_ref, "padded RS, real rows")

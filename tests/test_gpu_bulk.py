"""The "bulk" method: an all-gather or reduce-scatter run on its own, alone and beside an
unrelated GEMM on another stream, against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from gemm_overlap_gemms_gb300 import synth, ub
from gpu_helpers import assert_close, dev, is_sentinel, sentinel

pytestmark = pytest.mark.gpu


def _u16(t):
    return synth.to_u16(t)


@pytest.mark.parametrize("tp,c,H", [(4, 1, 256), (4, 127, 264), (2, 300, 512), (1, 33, 72),
                                    (8, 64, 4096)])
def test_reduce_scatter_matches_oracle(tp, c, H):
    T = c * tp
    g = synth.generator(seed=91)
    P = [synth.normal_bf16((T, H), 1.0, g) for _ in range(tp)]
    with ub.UserBuffer([T + 8 * tp, H], tp) as buf:
        buf.set_active_shape([T, H])
        pad = 2
        big = sentinel((tp * (c + pad), H))
        Ys = [big[r * (c + pad): r * (c + pad) + c] for r in range(tp)]
        buf.reduce_scatter([x.to(dev()) for x in P], Ys)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
        for r in range(tp):
            assert is_sentinel(big[r * (c + pad) + c:(r + 1) * (c + pad)])
    Yref = oracle.reduce_scatter([_u16(x) for x in P])
    for r in range(tp):
        assert_close(Ys[r], Yref[r], "RS block %d" % r)


def test_reduce_scatter_integer_inputs_are_exact():
    tp, c, H = 4, 70, 128
    T = c * tp
    g = synth.generator(seed=92)
    P = [synth.small_int_bf16((T, H), -20, 20, g) for _ in range(tp)]
    with ub.UserBuffer([T, H], tp) as buf:
        Ys = buf.reduce_scatter([x.to(dev()) for x in P])
        torch.cuda.synchronize()
    Yref = oracle.reduce_scatter([_u16(x) for x in P])
    for r in range(tp):
        np.testing.assert_array_equal(Ys[r].float().cpu().numpy(), Yref[r])


def test_allgather_then_wgrad():
    tp, c, H, M = 4, 129, 256, 192
    T = c * tp
    g = synth.generator(seed=93)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    D = synth.normal_bf16((T, M), 1.0, g)
    with ub.UserBuffer([T + 64, H], tp) as buf:
        buf.buffer().view(torch.int16).fill_(-1)
        buf.set_active_shape([T, H])
        buf.allgather([s.to(dev()) for s in shards])
        dW = buf.wgrad(D.to(dev()))
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
        Gall = buf.buffer().cpu()
    G = np.full((T + 64, H), 0xFFFF, dtype=np.uint16)
    oracle.allgather([_u16(s) for s in shards], G, T)
    np.testing.assert_array_equal(_u16(Gall), G)
    assert_close(dW, oracle.gemm_tn(_u16(D), G[:T]), "wgrad after bulk AG")


def test_bulk_collectives_beside_gemms_on_other_streams():
    """Column-parallel backward at hidden 2048: the input-gradient GEMM (gemm_rs_kn) on
    one stream while the bulk all-gather of the layer input runs on another; then the
    weight-gradient GEMM on one stream while a bulk reduce-scatter of other partials
    runs on another. Every result must match the oracle and the status stay clean."""
    tp, H, F, T = 4, 2048, 1024, 2048
    c = T // tp
    d = dev()
    g = synth.generator(d, seed=94)
    X = synth.normal_bf16((T, H), 1.0, g, d)
    dZ = [synth.normal_bf16((T, F), 1.0, g, d) for _ in range(tp)]
    Wt = [synth.normal_bf16((F, H), 1.0 / math.sqrt(H), g, d) for _ in range(tp)]
    P = [synth.normal_bf16((T, H), 1.0, g, d) for _ in range(tp)]
    s1, s2 = torch.cuda.Stream(d), torch.cuda.Stream(d)
    torch.cuda.synchronize()
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_active_shape([T, H])
        dX = buf.gemm_rs_kn(dZ, Wt, stream=s1)                              # GEMM on s1
        buf.allgather([X[r * c:(r + 1) * c] for r in range(tp)], stream=s2)  # bulk AG on s2
        s1.wait_stream(s2)
        dW = buf.wgrad(dZ[0], stream=s1)                                   # GEMM on s1 ...
        Ys = buf.reduce_scatter(P, stream=s2)                              # ... bulk RS on s2
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, c - 1, c, T - 1], rng.integers(0, T, 16)]))
    ridx = torch.as_tensor(rows, device=d)
    S = sum(oracle.gemm_xw_rows(_u16(dZ[j]), _u16(Wt[j]), rows) for j in range(tp))
    assert_close(torch.cat(dX)[ridx], S, "dgrad beside bulk AG")
    ms = np.array([0, 5, F // 2, F - 1])
    ref = oracle.gemm_tn(np.ascontiguousarray(_u16(dZ[0])[:, ms]), _u16(X))
    assert_close(dW[torch.as_tensor(ms, device=d)], ref, "wgrad beside bulk RS")
    Yref = oracle.reduce_scatter([_u16(x) for x in P])
    for r in range(tp):
        assert_close(Ys[r], Yref[r], "bulk RS block %d" % r)

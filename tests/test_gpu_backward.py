"""The backward-pass pair against the oracle: the weight read in its K x N layout
(MN-major for the tensor core) for both input gradients, and the weight gradient over
the active tokens from the gathered buffer.

* ag_gemm_kn  -- row-parallel input gradient dA = gather(dY) @ Bt (and forward AG with
                 W stored [hidden, N]);
* gemm_rs_kn  -- column-parallel input gradient dX_r = rows_r sum_j dY_j @ Wt_j;
* ub_wgrad    -- dWt = dY^T G (G = gathered input) and dBt = dS^T A (dS = gathered dY).
"""
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


@pytest.mark.parametrize("tp,c,H,N", [(4, 1, 256, 384), (4, 129, 256, 136), (2, 300, 512, 256),
                                      (1, 77, 256, 72), (4, 256, 2048, 512)])
def test_ag_gemm_kn_matches_oracle(tp, c, H, N):
    T = c * tp
    g = synth.generator(seed=71)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    W = synth.normal_bf16((H, N), 1.0 / math.sqrt(H), g)
    with ub.UserBuffer([T + 4 * tp, H], tp) as buf:
        buf.set_active_shape([T, H])
        Y = sentinel((T + 8, N))
        buf.ag_gemm_kn([s.to(dev()) for s in shards], W.to(dev()), Y)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
        G = buf.buffer()[:T].cpu()
    Gref = np.concatenate([_u16(s) for s in shards])
    np.testing.assert_array_equal(_u16(G), Gref)
    assert_close(Y[:T], oracle.gemm_xw_rows(Gref, _u16(W), np.arange(T)), "AG kn T=%d N=%d" % (T, N))
    assert is_sentinel(Y[T:])


@pytest.mark.parametrize("tp,c,H,K", [(4, 1, 256, 200), (4, 129, 320, 512), (2, 300, 256, 136),
                                      (4, 64, 2048, 1024)])
def test_gemm_rs_kn_matches_oracle(tp, c, H, K):
    T = c * tp
    g = synth.generator(seed=72)
    A = [synth.normal_bf16((T, K), 1.0, g) for _ in range(tp)]
    B = [synth.normal_bf16((K, H), 1.0 / math.sqrt(K), g) for _ in range(tp)]
    with ub.UserBuffer([T, H], tp) as buf:
        pad = 3
        big = sentinel((tp * (c + pad), H))
        Ys = [big[r * (c + pad): r * (c + pad) + c] for r in range(tp)]
        buf.gemm_rs_kn([a.to(dev()) for a in A], [b.to(dev()) for b in B], Ys)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
        for r in range(tp):
            assert is_sentinel(big[r * (c + pad) + c:(r + 1) * (c + pad)])
    # the pinned out-x-in GEMM-RS on the transposed weights (transposition is exact)
    _, Yref = oracle.gemm_rs([_u16(a) for a in A], [np.ascontiguousarray(_u16(b).T) for b in B])
    for r in range(tp):
        assert_close(Ys[r], Yref[r], "RS kn T=%d block %d" % (T, r))


@pytest.mark.parametrize("tp,c,H,M", [(4, 1, 256, 128), (4, 129, 256, 384), (2, 300, 512, 136),
                                      (4, 640, 512, 256)])
def test_wgrad_both_sides_match_oracle(tp, c, H, M):
    """T = 4, 516, 600, 2560: the contraction over T has a ragged tail in every case but
    the last (T % 64 != 0)."""
    T = c * tp
    g = synth.generator(seed=73)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    Wt = synth.normal_bf16((M, H), 1.0 / math.sqrt(H), g)
    D = synth.normal_bf16((T, M), 1.0, g)
    with ub.UserBuffer([T + 4 * tp, H], tp) as buf:
        buf.set_active_shape([T, H])
        buf.ag_gemm([s.to(dev()) for s in shards], Wt.to(dev()))     # leaves G in the buffer
        dW = buf.wgrad(D.to(dev()))                                   # [M, H] = D^T G
        dB = buf.wgrad(D.to(dev()), ub_is_a=True)                     # [H, M] = G^T D
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    G = np.concatenate([_u16(s) for s in shards])
    assert_close(dW, oracle.gemm_tn(_u16(D), G), "wgrad D^T G T=%d" % T)
    assert_close(dB, oracle.gemm_tn(G, _u16(D)), "wgrad G^T D T=%d" % T)


def test_backward_of_the_mlp_at_full_size():
    """Backward of the SwiGLU workload's two layers at hidden 4096 (tp=4, T=4640):
    fc2 input gradient (AG of dY, MN-major Bt), fc2 weight gradient from the gathered dY,
    fc1 input gradient (RS over dY_j Wt_j) -- sampled rows / columns against the oracle."""
    w = synth.WORKLOADS["swiglu"]
    T, H, F, tp = 4640, w.hidden, w.rs_k[0], w.tp
    c = T // tp
    g = synth.generator(dev(), seed=74)
    dY = synth.normal_bf16((T, H), 1.0, g, dev())              # gradient of fc2's output
    Bt = synth.normal_bf16((H, F), 1.0 / math.sqrt(F), g, dev())  # fc2 shard weight [H, K]
    A0 = synth.normal_bf16((T, F), 1.0, g, dev())              # fc2's saved input (rank 0)
    dZ = [synth.normal_bf16((T, F), 1.0, g, dev()) for _ in range(tp)]   # fc1 output grads
    Wt = [synth.normal_bf16((F, H), 1.0 / math.sqrt(H), g, dev()) for _ in range(tp)]
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, c - 1, c, 3 * c, T - 1], rng.integers(0, T, 24)]))
    ridx = torch.as_tensor(rows, device=dev())
    with ub.UserBuffer([w.max_tokens, H], tp) as buf:
        buf.set_active_shape([T, H])
        dA = buf.ag_gemm_kn([dY[r * c:(r + 1) * c] for r in range(tp)], Bt)    # [T, F]
        dBt = buf.wgrad(A0, ub_is_a=True)                                      # [H, F]
        dX = torch.cat(buf.gemm_rs_kn(dZ, Wt))                                  # [T, H]
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    dYu = _u16(dY)
    assert_close(dA[ridx], oracle.gemm_xw_rows(dYu, _u16(Bt), rows), "fc2 dgrad")
    # weight gradient: sampled rows h of dBt = dY^T A0 -> columns of the T contraction
    hs = np.array([0, 1, 777, 2048, H - 1])
    ref = oracle.gemm_tn(np.ascontiguousarray(dYu[:, hs]), _u16(A0))
    assert_close(dBt[torch.as_tensor(hs, device=dev())], ref, "fc2 wgrad")
    S = sum(oracle.gemm_xw_rows(_u16(dZ[j]), _u16(Wt[j]), rows) for j in range(tp))
    assert_close(dX[ridx], S, "fc1 dgrad")

"""AG-GEMM and GEMM-RS captured into a CUDA graph and replayed with new inputs: the
epoch of a captured call is a constant of the graph, so a replay must not find the
readiness or partial-tile flags already set by the replay before it (the library
clears them in stream order at the start of every captured call)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gemm_overlap_gemms_gb300 import synth, ub
from gpu_helpers import assert_close, dev

pytestmark = pytest.mark.gpu


def _u16(t):
    return synth.to_u16(t)


# T = 64: the few-token kernel with split pieces; T = 2048: CTA pairs, the gather
# overlapped with the GEMM (chunks of 512 rows that land while the self chunk computes);
# streamk = 1: the pairs' last wave cut into k-pieces, whose partial-tile flags a replay
# must not find set by the replay before (the captured call clears them).
@pytest.mark.parametrize("T,H,N,streamk", [(64, 1024, 768, -1), (2048, 1024, 768, -1), (1024, 2048, 512, 1)])
def test_captured_step_replays_with_new_inputs(T, H, N, streamk):
    tp, K = 4, 512
    c = T // tp
    d = dev()
    g = synth.generator(d, seed=121)
    X = torch.empty((T, H), dtype=torch.bfloat16, device=d)
    A = [torch.empty((T, K), dtype=torch.bfloat16, device=d) for _ in range(tp)]
    Wt = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g, d)
    Bt = [synth.normal_bf16((H, K), 1.0 / math.sqrt(K), g, d) for _ in range(tp)]
    Y = torch.empty((T, N), dtype=torch.bfloat16, device=d)
    Yrs = torch.empty((T, H), dtype=torch.bfloat16, device=d)
    shards = [X[r * c:(r + 1) * c] for r in range(tp)]
    outs = [Yrs[r * c:(r + 1) * c] for r in range(tp)]

    def refill():
        X.copy_(synth.normal_bf16((T, H), 1.0, g, d))
        for a in A:
            a.copy_(synth.normal_bf16((T, K), 1.0, g, d))

    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_active_shape([T, H])
        buf.set_option("streamk", streamk)
        s = torch.cuda.Stream(d)
        refill()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):  # warm-up outside the capture
            buf.ag_gemm(shards, Wt, Y, stream=s)
            if streamk == 1:
                assert buf.counters()["last_pieces"] > 1, "the AG call did not split its last wave"
            buf.gemm_rs(A, Bt, outs, stream=s)
            if streamk == 1:
                assert buf.counters()["last_pieces"] > 1, "the RS call did not split its last wave"
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            buf.ag_gemm(shards, Wt, Y, stream=s)
            buf.gemm_rs(A, Bt, outs, stream=s)
        rng = np.random.default_rng(4)
        rows = np.unique(np.concatenate([[0, c - 1, c, T - 1], rng.integers(0, T, 10)]))
        ridx = torch.as_tensor(rows, device=d)
        for rep in range(3):
            refill()
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            assert buf.query_status() == ub.UB_OK, "replay %d" % rep
            Xu = _u16(X)
            np.testing.assert_array_equal(_u16(buf.buffer()[:T]), Xu)  # the gather landed
            assert_close(Y[ridx], oracle.gemm_rows(Xu, _u16(Wt), rows), "AG replay %d T=%d" % (rep, T))
            S = sum(oracle.gemm_rows(_u16(A[j]), _u16(Bt[j]), rows) for j in range(tp))
            assert_close(Yrs[ridx], S, "RS replay %d T=%d" % (rep, T))
        del graph


# T = 64: few-token kernel (SwiGLU and RS); T = 512: single-CTA SwiGLU epilogue with the
# one-launch gather (chained on the call's stream, or on the side stream: chain 0);
# T = 2048 with the gather inside the GEMM (UB_OPT_GATHER_KERNEL = 2).
@pytest.mark.parametrize("T,gather,chain", [(64, -1, 1), (64, -1, 0), (512, -1, 1), (512, -1, 0), (2048, 2, 1)])
def test_captured_mlp_forward_and_backward_replay(T, gather, chain):
    """fc1 AG + SwiGLU, the K x N input-gradient GEMM-RS and the weight gradient from the
    gathered buffer, captured once and replayed with new activations."""
    tp, H, F = 4, 512, 256
    c = T // tp
    d = dev()
    g = synth.generator(d, seed=131)
    X = torch.empty((T, H), dtype=torch.bfloat16, device=d)
    dZ = [torch.empty((T, F), dtype=torch.bfloat16, device=d) for _ in range(tp)]
    W1 = synth.normal_bf16((2 * F, H), 1.0 / math.sqrt(H), g, d)
    Wt = [synth.normal_bf16((F, H), 1.0 / math.sqrt(F), g, d) for _ in range(tp)]
    Z = torch.empty((T, F), dtype=torch.bfloat16, device=d)
    dX = torch.empty((T, H), dtype=torch.bfloat16, device=d)
    dW = torch.empty((F, H), dtype=torch.bfloat16, device=d)
    shards = [X[r * c:(r + 1) * c] for r in range(tp)]
    outs = [dX[r * c:(r + 1) * c] for r in range(tp)]

    def refill():
        X.copy_(synth.normal_bf16((T, H), 1.0, g, d))
        for a in dZ:
            a.copy_(synth.normal_bf16((T, F), 1.0, g, d))

    def step(s):
        buf.ag_gemm_swiglu(shards, W1, Z, stream=s)
        buf.gemm_rs_kn(dZ, Wt, outs, stream=s)
        buf.wgrad(dZ[0], out=dW, stream=s)

    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_active_shape([T, H])
        buf.set_option("gather_kernel", gather)
        buf.set_option("gather_chain", chain)
        s = torch.cuda.Stream(d)
        refill()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            step(s)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step(s)
        rows = np.unique(np.array([0, c - 1, c, T // 2, T - 1]))
        ridx = torch.as_tensor(rows, device=d)
        for rep in range(2):
            refill()
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            assert buf.query_status() == ub.UB_OK, "replay %d" % rep
            Xu = _u16(X)
            ref_z = oracle.swiglu(oracle.gemm_rows(Xu, _u16(W1), rows))
            assert_close(Z[ridx], ref_z, "SwiGLU replay %d T=%d" % (rep, T))
            ref_dx = sum(oracle.gemm_xw_rows(_u16(dZ[j]), _u16(Wt[j]), rows) for j in range(tp))
            assert_close(dX[ridx], ref_dx, "dgrad replay %d T=%d" % (rep, T))
            ms = np.array([0, F // 2, F - 1])
            ref_w = oracle.gemm_tn(np.ascontiguousarray(_u16(dZ[0])[:, ms]), Xu)
            assert_close(dW[torch.as_tensor(ms, device=d)], ref_w, "wgrad replay %d T=%d" % (rep, T))
        del graph

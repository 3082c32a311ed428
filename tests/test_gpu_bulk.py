"""The "bulk" method: an all-gather or reduce-scatter run on its own, alone and beside an
unrelated GEMM (on another stream, or in beside mode on the GEMM's own stream), against
the oracle."""
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


# ---------------------------------------------------------------- beside mode (UB_OPT_BULK_BESIDE)

def test_bulk_collectives_in_beside_mode_on_the_gemms_stream():
    """The same column-parallel backward with every call on one stream, each collective
    launched beside the GEMM just before it: its inputs written just before that GEMM by
    another kernel, its results and the GEMM's read right after it by another kernel on
    the stream (ordering), all against the oracle."""
    tp, H, F, T = 4, 2048, 1024, 2048
    c = T // tp
    d = dev()
    g = synth.generator(d, seed=95)
    X = synth.normal_bf16((T, H), 1.0, g, d)
    dZ = [synth.normal_bf16((T, F), 1.0, g, d) for _ in range(tp)]
    Wt = [synth.normal_bf16((F, H), 1.0 / math.sqrt(H), g, d) for _ in range(tp)]
    P = [synth.normal_bf16((T, H), 1.0, g, d) for _ in range(tp)]
    s1 = torch.cuda.Stream(d)
    torch.cuda.synchronize()
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_active_shape([T, H])
        buf.set_option("bulk_beside", 1)
        assert buf.get_option("bulk_beside") == 1
        with torch.cuda.stream(s1):
            Xs = torch.empty_like(X)
            Xs.copy_(X)                       # the gather's input, written just before the GEMM
            Pn = [torch.empty_like(x) for x in P]
            for j in range(tp):
                torch.add(P[j], 0.0, out=Pn[j])   # the reduce-scatter's inputs, likewise
        dX = buf.gemm_rs_kn(dZ, Wt, stream=s1)                                # GEMM ...
        buf.allgather([Xs[r * c:(r + 1) * c] for r in range(tp)], stream=s1)  # ... beside it
        dW = buf.wgrad(dZ[0], stream=s1)     # reads the gathered buffer: after the gather
        Ys = buf.reduce_scatter(Pn, stream=s1)                              # beside the wgrad
        with torch.cuda.stream(s1):
            dW_after = dW.clone()             # read by the next kernel on the stream
            Y_after = [y.clone() for y in Ys]
            G_after = buf.buffer()[:T].clone()
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([[0, c - 1, c, T - 1], rng.integers(0, T, 16)]))
    ridx = torch.as_tensor(rows, device=d)
    S = sum(oracle.gemm_xw_rows(_u16(dZ[j]), _u16(Wt[j]), rows) for j in range(tp))
    assert_close(torch.cat(dX)[ridx], S, "dgrad with the gather beside it")
    np.testing.assert_array_equal(_u16(G_after), _u16(X))
    ms = np.array([0, 5, F // 2, F - 1])
    ref = oracle.gemm_tn(np.ascontiguousarray(_u16(dZ[0])[:, ms]), _u16(X))
    assert_close(dW_after[torch.as_tensor(ms, device=d)], ref, "wgrad with the reduce-scatter beside it")
    Yref = oracle.reduce_scatter([_u16(x) for x in P])
    for r in range(tp):
        assert_close(Y_after[r], Yref[r], "beside RS block %d" % r)


def test_beside_mode_integer_inputs_exact_alone_and_after_a_gemm():
    """Beside mode with nothing before it on a fresh stream (runs as a plain launch) and
    directly after a GEMM: bit-exact sums of small integers, and every row past c of the
    output blocks untouched."""
    tp, c, H, M = 4, 96, 512, 256
    T = c * tp
    g = synth.generator(seed=96)
    P = [synth.small_int_bf16((T, H), -20, 20, g).to(dev()) for _ in range(tp)]
    D = synth.normal_bf16((T, M), 1.0, g).to(dev())
    Yref = oracle.reduce_scatter([_u16(x) for x in P])
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_active_shape([T, H])
        buf.buffer().zero_()
        assert buf.get_option("bulk_beside") == 0           # off by default
        with pytest.raises(ub.UbError) as ei:
            buf.set_option("bulk_beside", 2)
        assert ei.value.name == "UB_ERR_ARG"
        buf.set_option("bulk_beside", 1)
        for after_gemm in (False, True):
            st = torch.cuda.Stream()
            pad = 3
            big = sentinel((tp * (c + pad), H))
            Ys = [big[r * (c + pad): r * (c + pad) + c] for r in range(tp)]
            torch.cuda.synchronize()
            if after_gemm:
                buf.wgrad(D, stream=st)
            buf.reduce_scatter(P, Ys, stream=st)
            torch.cuda.synchronize()
            assert buf.query_status() == ub.UB_OK
            for r in range(tp):
                np.testing.assert_array_equal(Ys[r].float().cpu().numpy(), Yref[r])
                assert is_sentinel(big[r * (c + pad) + c:(r + 1) * (c + pad)])


def test_beside_mode_replays_from_a_cuda_graph():
    """A weight-gradient GEMM with the reduce-scatter beside it, captured once and
    replayed: the programmatic edge holds in the graph, and each replay gives the
    oracle's values for new inputs copied in before it."""
    tp, c, H, M = 4, 256, 1024, 512
    T = c * tp
    g = synth.generator(dev(), seed=97)
    D = synth.normal_bf16((T, M), 1.0, g, dev())
    X = synth.normal_bf16((T, H), 1.0, g, dev())
    P = [torch.empty((T, H), dtype=torch.bfloat16, device=dev()) for _ in range(tp)]
    dW = torch.empty((M, H), dtype=torch.bfloat16, device=dev())
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_active_shape([T, H])
        buf.allgather([X[r * c:(r + 1) * c] for r in range(tp)])
        buf.set_option("bulk_beside", 1)
        st = torch.cuda.Stream()
        Ys = [torch.empty((c, H), dtype=torch.bfloat16, device=dev()) for _ in range(tp)]
        for x in P:
            x.zero_()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            buf.wgrad(D, out=dW, stream=st)
            buf.reduce_scatter(P, Ys, stream=st)
        for rep in range(2):
            src = [synth.normal_bf16((T, H), 1.0, synth.generator(seed=200 + 10 * rep + j)) for j in range(tp)]
            for x, y in zip(P, src):
                x.copy_(y)
            graph.replay()
            torch.cuda.synchronize()
            assert buf.query_status() == ub.UB_OK
            Yref = oracle.reduce_scatter([_u16(x) for x in src])
            for r in range(tp):
                assert_close(Ys[r], Yref[r], "graph replay %d block %d" % (rep, r))
        ms = np.array([0, 7, M - 1])
        ref = oracle.gemm_tn(np.ascontiguousarray(_u16(D)[:, ms]), _u16(X))
        assert_close(dW[torch.as_tensor(ms, device=dev())], ref, "wgrad in the graph")


# ---------------------------------------------------------------- gather ahead, GEMM from the buffer

@pytest.mark.parametrize("swiglu", [False, True])
@pytest.mark.parametrize("T", [4 * 300, 4 * 64, 2048])
def test_ag_gemm_from_buffer_after_allgather(T, swiglu):
    """ub_allgather lands the chunks; ag_gemm_from_buffer then computes the AG-GEMM (or
    AG + SwiGLU) over the buffer as it stands: the same values as the oracle."""
    tp, H, N = 4, 1024, 896
    g = synth.generator(seed=141)
    shards, Wt = synth.ag_inputs(T, H, N, tp, g)
    Gref = np.concatenate([synth.to_u16(s) for s in shards])
    with ub.UserBuffer([T + 64, H], tp) as buf:
        buf.set_active_shape([T, H])
        buf.allgather([s.to(dev()) for s in shards])
        n_out = N // 2 if swiglu else N
        Y = sentinel((T + 5, n_out))
        buf.ag_gemm_from_buffer(Wt.to(dev()), Y[:T], swiglu=swiglu)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
        np.testing.assert_array_equal(synth.to_u16(buf.buffer()[:T]), Gref)
    ref = oracle.gemm_rows(Gref, synth.to_u16(Wt), np.arange(T))
    if swiglu:
        ref = oracle.swiglu(ref)
    assert_close(Y[:T], ref, "from buffer T=%d swiglu=%s" % (T, swiglu))
    assert is_sentinel(Y[T:]), "rows past T touched"


@pytest.mark.parametrize("beside", [False, True])
def test_gather_ahead_pipeline_matches_the_oracle(beside):
    """Three microbatches of different T: each all-gather beside the previous GEMM-RS --
    on a second stream once the previous fc1 has read the buffer, or (beside mode) on the
    main stream right after the GEMM-RS; fc1 (AG + SwiGLU) on the gathered buffer, fc2
    GEMM-RS on the main stream. Every output against the oracle on sampled rows."""
    tp, H, F, K = 4, 1024, 256, 512
    Ts = [4 * 260, 4 * 96, 4 * 400]
    g = synth.generator(dev(), seed=142)
    W1 = synth.normal_bf16((2 * F, H), H ** -0.5, g, dev())
    Bt = [synth.normal_bf16((H, K), K ** -0.5, g, dev()) for _ in range(tp)]
    X = [synth.normal_bf16((T, H), 1.0, g, dev()) for T in Ts]
    A = [[synth.normal_bf16((T, K), 1.0, g, dev()) for _ in range(tp)] for T in Ts]
    Z = [torch.empty((T, F), dtype=torch.bfloat16, device=dev()) for T in Ts]
    R = [torch.empty((T, H), dtype=torch.bfloat16, device=dev()) for T in Ts]
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    ev_read = [torch.cuda.Event() for _ in Ts]
    ev_landed = [torch.cuda.Event() for _ in Ts]

    def shards(i):
        c = Ts[i] // tp
        return [X[i][r * c:(r + 1) * c] for r in range(tp)]

    with ub.UserBuffer([max(Ts), H], tp) as buf:
        buf.set_active_shape([Ts[0], H])
        buf.allgather(shards(0), stream=main)
        for i, T in enumerate(Ts):
            buf.set_active_shape([T, H])
            if i > 0:
                main.wait_event(ev_landed[i])
            buf.ag_gemm_from_buffer(W1, Z[i], swiglu=True, stream=main)
            ev_read[i].record(main)
            if i + 1 < len(Ts) and not beside:
                buf.set_active_shape([Ts[i + 1], H])
                side.wait_event(ev_read[i])
                buf.allgather(shards(i + 1), stream=side)
                ev_landed[i + 1].record(side)
                buf.set_active_shape([T, H])
            c = T // tp
            buf.gemm_rs(A[i], Bt, [R[i][r * c:(r + 1) * c] for r in range(tp)], stream=main)
            if i + 1 < len(Ts) and beside:
                buf.set_active_shape([Ts[i + 1], H])
                buf.set_option("bulk_beside", 1)
                buf.allgather(shards(i + 1), stream=main)   # beside the GEMM-RS just issued
                buf.set_option("bulk_beside", 0)
                ev_landed[i + 1].record(main)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    for i, T in enumerate(Ts):
        c = T // tp
        rows = np.unique(np.array([0, c - 1, c, T // 2, T - 1]))
        ridx = torch.as_tensor(rows, device=dev())
        Xu = synth.to_u16(X[i])
        assert_close(Z[i][ridx], oracle.swiglu(oracle.gemm_rows(Xu, synth.to_u16(W1), rows)), "fc1 mb %d" % i)
        ref = sum(oracle.gemm_rows(synth.to_u16(A[i][j]), synth.to_u16(Bt[j]), rows) for j in range(tp))
        assert_close(R[i][ridx], ref, "fc2 mb %d" % i)


def test_beside_reduce_scatter_after_a_chained_ag_gemm():
    """A few-token AG-GEMM whose gather kernel runs chained on the stream (the GEMM its
    programmatic dependent, letting the next grid launch at entry), then a reduce-scatter
    in beside mode on the same stream: the collective starts while the AG call may still
    be running. Its inputs were written before the AG call, so both results must match
    the oracle, and a kernel after the pair must see both."""
    tp, H, N, T = 4, 1024, 512, 64
    c = T // tp
    g = synth.generator(seed=98)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    Wt = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g)
    P = [synth.small_int_bf16((T, H), -20, 20, g).to(dev()) for _ in range(tp)]
    st = torch.cuda.Stream()
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_active_shape([T, H])
        torch.cuda.synchronize()
        Y = buf.ag_gemm([s.to(dev()) for s in shards], Wt.to(dev()), stream=st)
        assert ub.GATHERS[buf.counters()["last_gather"]] == "gather_kernel"
        buf.set_option("bulk_beside", 1)
        Ys = buf.reduce_scatter(P, stream=st)
        with torch.cuda.stream(st):
            Y_after = Y.clone()
            Ys_after = [y.clone() for y in Ys]
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    Gref, Yref = oracle.ag_gemm([_u16(s) for s in shards], _u16(Wt))
    assert_close(Y_after, Yref, "AG before the beside reduce-scatter")
    Rref = oracle.reduce_scatter([_u16(x) for x in P])
    for r in range(tp):
        np.testing.assert_array_equal(Ys_after[r].float().cpu().numpy(), Rref[r])

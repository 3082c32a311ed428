"""The few-token kernel (weight rows on the tensor core's M dimension, tokens on its N
dimension) against the oracle: AG-GEMM, AG-GEMM + SwiGLU, GEMM-RS and the K x N weight
variants, for T from tp up to the largest token tile it takes, with ragged chunks,
split k-pieces, untouched output tails, determinism and the bounded flag wait."""
import math

import numpy as np
import pytest
import torch

import oracle
from gemm_overlap_gemms_gb300 import synth, ub
from gpu_helpers import assert_close, dev, is_sentinel, oracle_ag, run_ag, run_rs, sentinel

pytestmark = pytest.mark.gpu


def _u16(t):
    return synth.to_u16(t)


def _make_buf(T, H, tp, skinny=1, extra=8):
    buf = ub.UserBuffer([T + extra * tp, H], tp)
    buf.set_option("skinny", skinny)
    buf.set_active_shape([T, H])
    return buf


# (tp, c, H, N): chunks of 1..64 rows (token sub-tiles of 16..64 columns), one or many
# weight tiles, N not a multiple of 128, K of 2..64 k-blocks (split into pieces or not).
@pytest.mark.parametrize("gather", [-1, 2, 3])
@pytest.mark.parametrize("tp,c,H,N", [(4, 1, 256, 384), (4, 16, 256, 136), (4, 63, 512, 264),
                                      (2, 100, 256, 392), (1, 200, 320, 128), (8, 32, 1024, 1000),
                                      (4, 64, 4096, 3072), (1, 1, 72, 8)])
def test_skinny_ag_matches_oracle(tp, c, H, N, gather):
    """gather -1: the one-launch gather kernel, chained on the call's stream; 3: the same
    kernel on the handle's side stream; 2: the kernel's epilogue warps gather, each chunk
    by its own group of CTAs (N tiles fewer than the chunks included)."""
    T = c * tp
    g = synth.generator(seed=101)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    Wt = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g)
    with _make_buf(T, H, tp) as buf:
        buf.set_option("gather_kernel", -1 if gather == 3 else gather)
        buf.set_option("gather_chain", 0 if gather == 3 else 1)
        Y = run_ag(buf, shards, Wt, y_rows=T + 5)
        assert buf.query_status() == ub.UB_OK
        G = buf.buffer()[:T].cpu()
    Gref, Yref = oracle_ag(shards, Wt)
    np.testing.assert_array_equal(_u16(G), Gref)
    assert_close(Y[:T], Yref, "skinny AG tp=%d c=%d N=%d" % (tp, c, N))
    assert is_sentinel(Y[T:]), "Y rows >= T touched"


@pytest.mark.parametrize("tp,T,H,K", [(4, 4, 256, 512), (4, 100, 256, 200), (2, 256, 512, 136),
                                      (8, 64, 1024, 1024), (1, 17, 256, 64), (4, 240, 1024, 3584)])
def test_skinny_rs_matches_oracle(tp, T, H, K):
    g = synth.generator(seed=102)
    A = [synth.normal_bf16((T, K), 1.0, g) for _ in range(tp)]
    Bt = [synth.normal_bf16((H, K), 1.0 / math.sqrt(K), g) for _ in range(tp)]
    with _make_buf(T, H, tp) as buf:
        Ys, _ = run_rs(buf, A, Bt)
        assert buf.query_status() == ub.UB_OK
    _, Yref = oracle.gemm_rs([_u16(a) for a in A], [_u16(b) for b in Bt])
    for r in range(tp):
        assert_close(Ys[r], Yref[r], "skinny RS T=%d block %d" % (T, r))


def test_skinny_rs_integer_inputs_are_exact():
    """Small integers: every product and partial sum is exact in fp32, so the split
    pieces' fix-up must give the oracle's exact sum, rounded once to bf16 (to nearest
    even, as the output conversion does)."""
    tp, T, H, K = 4, 36, 512, 2048
    g = synth.generator(seed=103)
    A = [synth.small_int_bf16((T, K), -3, 3, g) for _ in range(tp)]
    Bt = [synth.small_int_bf16((H, K), -3, 3, g) for _ in range(tp)]
    with _make_buf(T, H, tp) as buf:
        Ys, _ = run_rs(buf, A, Bt)
    _, Yref = oracle.gemm_rs([_u16(a) for a in A], [_u16(b) for b in Bt])
    for r in range(tp):
        assert np.abs(Yref[r]).max() < 2 ** 24  # exact in fp32
        want = torch.from_numpy(Yref[r]).to(torch.bfloat16).float().numpy()
        np.testing.assert_array_equal(Ys[r].float().cpu().numpy(), want)


@pytest.mark.parametrize("tp,c,F,H", [(4, 1, 128, 256), (4, 16, 136, 256), (2, 100, 384, 512),
                                      (4, 64, 3584, 4096)])
def test_skinny_swiglu_matches_oracle(tp, c, F, H):
    T = c * tp
    g = synth.generator(seed=104)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    Wt = synth.normal_bf16((2 * F, H), 1.0 / math.sqrt(H), g)
    with _make_buf(T, H, tp) as buf:
        Z = sentinel((T + 8, F))
        buf.ag_gemm_swiglu([s.to(dev()) for s in shards], Wt.to(dev()), Z)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    G = np.concatenate([_u16(s) for s in shards])
    rows = np.arange(T) if T * F * H <= (1 << 28) else np.unique(
        np.concatenate([[0, c - 1, c, T - 1], np.random.default_rng(1).integers(0, T, 12)]))
    ref = oracle.swiglu(oracle.gemm_rows(G, _u16(Wt), rows))
    assert_close(Z[torch.as_tensor(rows, device=dev())], ref, "skinny SwiGLU T=%d F=%d" % (T, F))
    assert is_sentinel(Z[T:]), "Z rows >= T touched"


@pytest.mark.parametrize("tp,c,H,N", [(4, 1, 256, 384), (4, 33, 512, 200), (2, 128, 256, 136)])
def test_skinny_ag_kn_matches_oracle(tp, c, H, N):
    T = c * tp
    g = synth.generator(seed=105)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    W = synth.normal_bf16((H, N), 1.0 / math.sqrt(H), g)
    with _make_buf(T, H, tp) as buf:
        Y = sentinel((T + 3, N))
        buf.ag_gemm_kn([s.to(dev()) for s in shards], W.to(dev()), Y)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    G = np.concatenate([_u16(s) for s in shards])
    assert_close(Y[:T], oracle.gemm_xw_rows(G, _u16(W), np.arange(T)), "skinny AG kn T=%d" % T)
    assert is_sentinel(Y[T:])


@pytest.mark.parametrize("tp,T,H,K", [(4, 4, 256, 200), (4, 128, 384, 512), (2, 250, 256, 136)])
def test_skinny_rs_kn_matches_oracle(tp, T, H, K):
    g = synth.generator(seed=106)
    A = [synth.normal_bf16((T, K), 1.0, g) for _ in range(tp)]
    B = [synth.normal_bf16((K, H), 1.0 / math.sqrt(K), g) for _ in range(tp)]
    c = T // tp
    with _make_buf(T, H, tp) as buf:
        pad = 2
        big = sentinel((tp * (c + pad), H))
        Ys = [big[r * (c + pad): r * (c + pad) + c] for r in range(tp)]
        buf.gemm_rs_kn([a.to(dev()) for a in A], [b.to(dev()) for b in B], Ys)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
        for r in range(tp):
            assert is_sentinel(big[r * (c + pad) + c:(r + 1) * (c + pad)])
    _, Yref = oracle.gemm_rs([_u16(a) for a in A], [np.ascontiguousarray(_u16(b).T) for b in B])
    for r in range(tp):
        assert_close(Ys[r], Yref[r], "skinny RS kn T=%d block %d" % (T, r))


def test_skinny_is_deterministic_and_agrees_with_the_tile_kernels():
    """Two calls give the same bits; the CTA-pair and single-CTA kernels give results
    within the tolerance of the same oracle (their sums run in another order)."""
    tp, c, H, N, K = 4, 50, 2048, 1536, 1024
    T = c * tp
    g = synth.generator(dev(), seed=107)
    shards = [synth.normal_bf16((c, H), 1.0, g, dev()) for _ in range(tp)]
    Wt = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g, dev())
    A = [synth.normal_bf16((T, K), 1.0, g, dev()) for _ in range(tp)]
    Bt = [synth.normal_bf16((H, K), 1.0 / math.sqrt(K), g, dev()) for _ in range(tp)]
    outs = {}
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_active_shape([T, H])
        for name, sk, pair in (("skinny", 1, -1), ("skinny2", 1, -1), ("pair", 0, 1), ("single", 0, 0)):
            buf.set_option("skinny", sk)
            buf.set_option("cta_pair", pair)
            Y = buf.ag_gemm(shards, Wt)
            Ys = buf.gemm_rs(A, Bt)
            torch.cuda.synchronize()
            assert buf.query_status() == ub.UB_OK, name
            outs[name] = (Y.clone(), torch.cat(Ys).clone())
    assert torch.equal(outs["skinny"][0].view(torch.int16), outs["skinny2"][0].view(torch.int16))
    assert torch.equal(outs["skinny"][1].view(torch.int16), outs["skinny2"][1].view(torch.int16))
    rows = np.array([0, 1, c - 1, c, 2 * c + 7, T - 1])
    ridx = torch.as_tensor(rows, device=dev())
    G = np.concatenate([_u16(s) for s in shards])
    ref_ag = oracle.gemm_rows(G, _u16(Wt), rows)
    ref_rs = sum(oracle.gemm_rows(_u16(A[j]), _u16(Bt[j]), rows) for j in range(tp))
    for name, (Y, Yrs) in outs.items():
        assert_close(Y[ridx], ref_ag, "AG " + name)
        assert_close(Yrs[ridx], ref_rs, "RS " + name)


@pytest.mark.parametrize("gather", [-1, 2])
def test_skinny_dropped_flag_times_out_and_the_handle_recovers(gather):
    """A chunk flag that is never written: the weight stream has started, the flag wait
    runs out, the call reports UB_ERR_TIMEOUT; the next call on the handle is clean."""
    tp, c, H, N = 4, 8, 1024, 2048
    T = c * tp
    g = synth.generator(seed=108)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    Wt = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g)
    with _make_buf(T, H, tp) as buf:
        buf.set_option("gather_kernel", gather)
        buf.set_option("timeout_ns", 20_000_000)
        buf.set_option("drop_flag", 2)
        Y = run_ag(buf, shards, Wt)
        assert buf.query_status() == ub.CODES["UB_ERR_TIMEOUT"]
        buf.clear_status()
        Y = run_ag(buf, shards, Wt)
        assert buf.query_status() == ub.UB_OK
    _, Yref = oracle_ag(shards, Wt)
    assert_close(Y, Yref, "skinny AG after a timed-out call")


def test_skinny_covers_every_T_up_to_its_limit_on_one_buffer():
    """Back-to-back calls with T from tp to 256 on one registered buffer (the
    active-shape stress pattern at small T): every result against the oracle, rows."""
    tp, H, N, K = 4, 512, 384, 256
    g = synth.generator(seed=109)
    Wt = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g)
    Bt = [synth.normal_bf16((H, K), 1.0 / math.sqrt(K), g) for _ in range(tp)]
    with ub.UserBuffer([1024, H], tp) as buf:
        for T in (4, 8, 60, 64, 68, 124, 128, 200, 252, 256):
            c = T // tp
            buf.set_active_shape([T, H])
            shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
            A = [synth.normal_bf16((T, K), 1.0, g) for _ in range(tp)]
            Y = run_ag(buf, shards, Wt)
            Ys, _ = run_rs(buf, A, Bt)
            assert buf.query_status() == ub.UB_OK
            _, Yref = oracle_ag(shards, Wt)
            assert_close(Y, Yref, "AG T=%d" % T)
            _, Rref = oracle.gemm_rs([_u16(a) for a in A], [_u16(b) for b in Bt])
            for r in range(tp):
                assert_close(Ys[r], Rref[r], "RS T=%d block %d" % (T, r))


@pytest.mark.parametrize("T", [64, 512])
def test_chained_gather_with_per_launch_events(T):
    """UB_OPT_PROFILE records a CUDA event before and after each GEMM launch; with the
    gather kernel chained on the call's stream (the default) an event then stands between
    the gather and its GEMM, so the GEMM runs after the gather instead of beside it. The
    results must still match the oracle, the status stay clean, and every launch be
    timed."""
    tp, H, N = 4, 1024, 384
    c = T // tp
    g = synth.generator(seed=111)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    Wt = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g)
    with _make_buf(T, H, tp) as buf:
        assert buf.get_option("gather_chain") == 1
        buf.set_option("profile", 1)
        for _ in range(3):
            Y = run_ag(buf, shards, Wt, y_rows=T + 2)
        assert ub.GATHERS[buf.counters()["last_gather"]] == "gather_kernel"
        ms, n = buf.kernel_time("ag")
        assert n == 3 and ms > 0
        assert buf.query_status() == ub.UB_OK
        G = buf.buffer()[:T].cpu()
    Gref, Yref = oracle_ag(shards, Wt)
    np.testing.assert_array_equal(_u16(G), Gref)
    assert_close(Y[:T], Yref, "chained gather with events T=%d" % T)
    assert is_sentinel(Y[T:])

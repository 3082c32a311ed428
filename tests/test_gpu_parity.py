"""GPU parity: the C-ABI path against the CPU oracle, element by element.

Floating point: |gpu - oracle| <= 2e-2 * max(1, |oracle|) with bf16 inputs and fp32
accumulation. Indexing (the gathered buffer, chunk offsets, row ownership, untouched
tails and guards): bit-exact. Integer-valued inputs make the products exact, so there
the GPU output must equal the oracle's result rounded to bf16, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_overlap_gemms_gb300 import synth, ub
from gpu_helpers import (assert_close, dev, is_sentinel, oracle_ag, oracle_rs, run_ag, run_rs,
                         sentinel)

pytestmark = pytest.mark.gpu


def _round_bf16(a: np.ndarray) -> np.ndarray:
    return np.array([oracle.round_bf16(v) for v in a.ravel()], dtype=np.uint16).reshape(a.shape)


# ------------------------------------------------------------------ tiny workload

def test_tiny_workload_ag_and_rs():
    w = synth.WORKLOADS["tiny"]
    T = synth.token_counts("tiny")[0]
    g = synth.generator()
    shards, Wt = synth.ag_inputs(T, w.hidden, w.ag_n[0], w.tp, g)
    A, Bt = synth.rs_inputs(T, w.rs_k[0], w.hidden, w.tp, g)
    with ub.UserBuffer([w.max_tokens, w.hidden], w.tp) as buf:
        buf.buffer().view(torch.int16).fill_(-1)
        buf.set_active_shape([T, w.hidden])
        Y = run_ag(buf, shards, Wt, y_rows=w.max_tokens)
        Ys, _ = run_rs(buf, A, Bt)
        assert buf.query_status() == ub.UB_OK
        G = buf.buffer().cpu()
    Gref, Yref = oracle_ag(shards, Wt)
    np.testing.assert_array_equal(synth.to_u16(G[:T]), Gref)
    assert is_sentinel(G[T:]), "user buffer rows >= T were touched"
    assert_close(Y[:T], Yref, "AG-GEMM")
    assert is_sentinel(Y[T:]), "Y rows >= T were touched"
    _, Yb = oracle_rs(A, Bt)
    for r in range(w.tp):
        assert_close(Ys[r], Yb[r], "GEMM-RS block %d" % r)


# ------------------------------------------------------------------ active-T sweeps

SWEEP_C = [1, 2, 127, 128, 129, 255, 300]

# The gather forms (UB_OPT_GATHER_KERNEL, UB_OPT_GATHER_CHAIN): 0 driver copies, 1 the
# gather kernel chained on the call's stream (the GEMM its programmatic dependent), 2
# inside the GEMM, 3 the gather kernel on the handle's side stream.
GATHER_FORMS = [0, 1, 2, 3]


def set_gather(buf, form):
    buf.set_option("gather_kernel", 1 if form == 3 else form)
    buf.set_option("gather_chain", 0 if form == 3 else 1)


@pytest.mark.parametrize("gather", GATHER_FORMS)
@pytest.mark.parametrize("pair", [1, 0])
@pytest.mark.parametrize("tp", [1, 2, 4])
def test_ag_active_T_sweep(tp, pair, gather):
    H, N = 256, 384            # two N tiles, the second one partial
    cap = tp * 320
    g = synth.generator(seed=11)
    Wt = synth.normal_bf16((N, H), H ** -0.5, g)
    with ub.UserBuffer([cap, H], tp) as buf:
        buf.set_option("cta_pair", pair)
        set_gather(buf, gather)
        for c in SWEEP_C + [cap // tp]:
            T = c * tp
            buf.buffer().view(torch.int16).fill_(-1)
            buf.set_active_shape([T, H])
            shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
            Y = run_ag(buf, shards, Wt, y_rows=cap)
            G = buf.buffer().cpu()
            Gref, Yref = oracle_ag(shards, Wt)
            np.testing.assert_array_equal(synth.to_u16(G[:T]), Gref, err_msg="gather T=%d" % T)
            assert is_sentinel(G[T:]), "buffer tail touched at T=%d" % T
            assert_close(Y[:T], Yref, "AG T=%d tp=%d" % (T, tp))
            assert is_sentinel(Y[T:]), "Y tail touched at T=%d" % T
        assert buf.query_status() == ub.UB_OK
        assert buf.counters()["device_allocations"] == 3


@pytest.mark.parametrize("pair", [1, 0])
@pytest.mark.parametrize("tp,K", [(1, 512), (2, 512), (4, 200)])
def test_rs_active_T_sweep(tp, K, pair):
    H = 256 + 64                # one full and one partial N tile
    cap = tp * 320
    g = synth.generator(seed=12)
    Bt = [synth.normal_bf16((H, K), K ** -0.5, g) for _ in range(tp)]
    with ub.UserBuffer([cap, H], tp) as buf:
        buf.set_option("cta_pair", pair)
        for c in SWEEP_C + [cap // tp]:
            T = c * tp
            buf.set_active_shape([T, H])
            A = [synth.normal_bf16((T, K), 1.0, g) for _ in range(tp)]
            Ys, _ = run_rs(buf, A, Bt)
            _, Yb = oracle_rs(A, Bt)
            for r in range(tp):
                assert_close(Ys[r], Yb[r], "RS T=%d tp=%d block %d" % (T, tp, r))
        assert buf.query_status() == ub.UB_OK


@pytest.mark.parametrize("pair", [1, 0])
def test_integer_inputs_are_bit_exact(pair):
    tp, H, N, K = 4, 256, 264, 136
    T = tp * 133
    g = synth.generator(seed=13)
    shards = [synth.small_int_bf16((T // tp, H), -3, 3, g) for _ in range(tp)]
    Wt = synth.small_int_bf16((N, H), -3, 3, g)
    A = [synth.small_int_bf16((T, K), -3, 3, g) for _ in range(tp)]
    Bt = [synth.small_int_bf16((H, K), -3, 3, g) for _ in range(tp)]
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_option("cta_pair", pair)
        Y = run_ag(buf, shards, Wt)
        Ys, _ = run_rs(buf, A, Bt)
    _, Yref = oracle_ag(shards, Wt)
    np.testing.assert_array_equal(synth.to_u16(Y), _round_bf16(Yref))
    _, Yb = oracle_rs(A, Bt)
    for r in range(tp):
        np.testing.assert_array_equal(synth.to_u16(Ys[r]), _round_bf16(Yb[r]))


# ------------------------------------------------------------------ invariants of the method

def test_active_shape_equals_exact_allocation_bitwise():
    tp, H, N, K = 4, 512, 256, 384
    T = 4 * 150
    g = synth.generator(seed=14)
    shards, Wt = synth.ag_inputs(T, H, N, tp, g)
    A, Bt = synth.rs_inputs(T, K, H, tp, g)
    with ub.UserBuffer([8192, H], tp) as big:
        big.set_active_shape([T, H])
        Y1 = run_ag(big, shards, Wt)
        R1, _ = run_rs(big, A, Bt)
    with ub.UserBuffer([T, H], tp) as exact:
        Y2 = run_ag(exact, shards, Wt)
        R2, _ = run_rs(exact, A, Bt)
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    for a, b in zip(R1, R2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_deterministic_and_consistent_across_launch_shapes():
    """Bitwise run-to-run determinism for a fixed launch shape; the same values (within
    tolerance of the oracle) for every ring start, SM margin and tile shape. The k-pieces
    of a split last wave depend on the number of CTA pairs, so different launch shapes
    may round differently."""
    tp, H, N, K = 4, 256, 512, 256
    T = 4 * 260
    g = synth.generator(seed=15)
    shards, Wt = synth.ag_inputs(T, H, N, tp, g)
    A, Bt = synth.rs_inputs(T, K, H, tp, g)
    configs = [(0, 0, 1, 1, 1), (0, 0, 1, 1, 3), (2, 0, 1, 1, 1), (3, 100, 1, 1, 2),
               (1, 0, 0, 1, 1), (0, 7, 0, 1, 4), (1, 0, 0, 1, 2), (0, 0, 1, 0, 1), (2, 90, 1, 0, 4),
               (0, 0, -1, -1, 1)]
    outs = []
    with ub.UserBuffer([T, H], tp) as buf:
        # the gather by driver copies, then inside the GEMM: it moves bytes only, so the
        # same launch shape must give the same bits either way
        for gather in (0, 2):
            buf.set_option("gather_kernel", gather)
            for self_rank, margin, pair, streamk, copy_streams in configs:
                buf.set_option("self_rank", self_rank)
                buf.set_option("sm_margin", margin)
                buf.set_option("cta_pair", pair)
                buf.set_option("streamk", streamk)
                buf.set_option("copy_streams", copy_streams)
                Y = run_ag(buf, shards, Wt)
                R, _ = run_rs(buf, A, Bt)
                outs.append((Y.view(torch.int16).clone(), [r.view(torch.int16).clone() for r in R]))
        assert buf.query_status() == ub.UB_OK
    n = len(configs)
    for i, j in [(0, 1), (4, 6)] + [(k, k + n) for k in range(n)]:
        assert torch.equal(outs[i][0], outs[j][0])
        for a, b in zip(outs[i][1], outs[j][1]):
            assert torch.equal(a, b)
    configs = configs + configs
    _, Yref = oracle_ag(shards, Wt)
    _, Yb = oracle_rs(A, Bt)
    for k, (Y, R) in enumerate(outs):
        assert_close(Y.view(torch.bfloat16), Yref, "AG config %s" % (configs[k],))
        for r in range(tp):
            assert_close(R[r].view(torch.bfloat16), Yb[r], "RS config %s block %d" % (configs[k], r))


def test_reshape_is_host_only_and_allocates_nothing():
    with ub.UserBuffer([1024, 256], 4) as buf:
        ptr = buf.buffer_ptr()
        before = torch.cuda.memory_allocated()
        for T in list(range(4, 1025, 60)) + [1024, 4]:
            buf.set_active_shape([T, 256])
            assert buf.active_shape == (T, 256)
        assert buf.buffer_ptr() == ptr
        assert buf.counters()["device_allocations"] == 3
        assert torch.cuda.memory_allocated() == before
        for bad, name in [([1028, 256], "UB_ERR_CAPACITY"), ([6, 256], "UB_ERR_DIVISIBLE"),
                          ([8, 128], "UB_ERR_HIDDEN"), ([0, 256], "UB_ERR_ZERO"),
                          ([8], "UB_ERR_RANK")]:
            with pytest.raises(ub.UbError) as ei:
                buf.set_active_shape(bad)
            assert ei.value.name == name
            assert buf.active_shape == (4, 256)   # unchanged after a rejected shape
        assert buf.capacity_shape == (1024, 256)


def test_module_level_api():
    m = ub.initialize_ub([512, 256], 2)
    try:
        ub.set_ub_active_shape([128, 256])
        assert ub.get_ub().active_shape == (128, 256)
        g = synth.generator(seed=16)
        shards, Wt = synth.ag_inputs(128, 256, 64, 2, g)
        Y = run_ag(m, shards, Wt)
        _, Yref = oracle_ag(shards, Wt)
        assert_close(Y, Yref, "module-level AG")
    finally:
        ub.destroy_ub()


def test_rejects_misaligned_and_wrong_shapes():
    tp, H = 2, 256
    with ub.UserBuffer([256, H], tp) as buf:
        buf.set_active_shape([128, H])
        shards = [torch.zeros((64, H), dtype=torch.bfloat16, device=dev()) for _ in range(tp)]
        Wt = torch.zeros((64, H), dtype=torch.bfloat16, device=dev())
        raw = torch.zeros(64 * H + 1, dtype=torch.bfloat16, device=dev())
        bad = raw[1:].view(64, H)                  # 2-byte offset: not 16-byte aligned
        with pytest.raises(ub.UbError) as ei:
            buf.ag_gemm([bad, shards[1]], Wt)
        assert ei.value.name == "UB_ERR_ALIGN"
        with pytest.raises(ValueError):
            buf.ag_gemm([shards[0][:32], shards[1]], Wt)
        with pytest.raises(ub.UbError) as ei:
            buf.ag_gemm(shards, torch.zeros((60, H), dtype=torch.bfloat16, device=dev()))
        assert ei.value.name == "UB_ERR_ALIGN"      # N % 8 != 0
        assert buf.counters()["ag_calls"] == 0


# ------------------------------------------------------------------ bounded waits

@pytest.mark.parametrize("gather", GATHER_FORMS)
@pytest.mark.parametrize("pair", [1, 0])
def test_dropped_flag_times_out_and_the_handle_recovers(pair, gather):
    """Fault injected on the host: the readiness flag of chunk 1 is never written. The
    kernel's bounded wait must expire, report UB_ERR_TIMEOUT, and leave the context and
    handle usable for the next call."""
    tp, H, N = 4, 256, 256
    T = 4 * 64
    g = synth.generator(seed=17)
    shards, Wt = synth.ag_inputs(T, H, N, tp, g)
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_option("cta_pair", pair)
        set_gather(buf, gather)
        buf.set_option("timeout_ns", 20_000_000)
        buf.set_option("drop_flag", 1)
        run_ag(buf, shards, Wt)
        assert buf.query_status() == ub.CODES["UB_ERR_TIMEOUT"]
        assert buf.get_option("drop_flag") == -1        # one-shot
        buf.clear_status()
        assert buf.query_status() == ub.UB_OK
        Y = run_ag(buf, shards, Wt)
        assert buf.query_status() == ub.UB_OK
    _, Yref = oracle_ag(shards, Wt)
    assert_close(Y, Yref, "AG after recovery")


@pytest.mark.parametrize("gather", GATHER_FORMS)
@pytest.mark.parametrize("op", ["ag", "rs", "ag_swiglu"])
def test_back_to_back_calls_at_full_hidden(op, gather):
    """Ten calls in a row on one handle at hidden 4096 without synchronising in
    between: every call's chunk copies must be able to run next to the GEMM kernels."""
    tp, H, N, K, T = 4, 4096, 1024, 1024, 2048
    g = synth.generator(dev(), seed=51)
    X = synth.normal_bf16((T, H), 1.0, g, dev())
    Wt = synth.normal_bf16((2 * N if op == "ag_swiglu" else N, H), H ** -0.5, g, dev())
    A = [synth.normal_bf16((T, K), 1.0, g, dev()) for _ in range(tp)]
    Bt = [synth.normal_bf16((H, K), K ** -0.5, g, dev()) for _ in range(tp)]
    c = T // tp
    shards = [X[r * c:(r + 1) * c] for r in range(tp)]
    with ub.UserBuffer([T, H], tp) as buf:
        set_gather(buf, gather)
        outs = []
        for _ in range(10):
            if op == "ag":
                outs.append(buf.ag_gemm(shards, Wt))
            elif op == "ag_swiglu":
                outs.append(buf.ag_gemm_swiglu(shards, Wt))
            else:
                outs.append(torch.cat(buf.gemm_rs(A, Bt)))
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))

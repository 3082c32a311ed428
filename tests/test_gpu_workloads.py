"""GPU parity at the full workload sizes, in the launch configuration the benchmark
times: every row of the gathered buffer and every capacity tail is checked exactly;
the GEMM outputs are checked on sampled rows against the oracle computed row by row.
The rows: every chunk's first, last and tile-edge rows, one seeded random row in every
64-row window of the active prefix (so every output tile of every call is hit, whatever
tiling the call chose: 256-row pair tiles by region, 128-row chunk-aligned tiles, the
split last wave, the partial tiles at region and chunk ends), plus seeded random rows.
A sampled row is compared across all of its columns."""
import math

import numpy as np
import pytest
import torch

import oracle
from gemm_overlap_gemms_gb300 import synth, ub
from gpu_helpers import assert_close, dev, is_sentinel, sentinel

pytestmark = pytest.mark.gpu


WINDOW = 64  # one sampled row per this many active rows


def sample_rows(T: int, tp: int, n_random: int, rng: np.random.Generator, window: int | None = WINDOW) -> np.ndarray:
    c = T // tp
    rows = set()
    for r in range(tp):
        for i in (0, 1, 127, 128, 255, 256, c - 1):
            if 0 <= i < c:
                rows.add(r * c + i)
    if window:
        for lo in range(0, T, window):
            rows.add(int(rng.integers(lo, min(lo + window, T))))
    rows.update(int(x) for x in rng.integers(0, T, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)


def check_ag(buf, T, N, g, rng, Wt=None, n_random=24, window=WINDOW):
    """One AG-GEMM at active T with fresh shards; returns Wt for reuse."""
    tp, H, cap = buf.tp, buf.hidden, buf.max_tokens
    c = T // tp
    buf.set_active_shape([T, H])
    X = synth.normal_bf16((T, H), 1.0, g, dev())
    shards = [X[r * c:(r + 1) * c] for r in range(tp)]
    if Wt is None:
        Wt = synth.normal_bf16((N, H), 1.0 / math.sqrt(H), g, dev())
    whole = buf.buffer()
    whole[T:].view(torch.int16).fill_(-1)
    Y = sentinel((cap, N))
    buf.ag_gemm(shards, Wt, Y)
    torch.cuda.synchronize()
    assert buf.query_status() == ub.UB_OK
    # the gathered buffer, bit for bit, against the oracle's own concatenation
    G = np.full((T, H), 0xFFFF, dtype=np.uint16)
    oracle.allgather([synth.to_u16(s) for s in shards], G, T)
    np.testing.assert_array_equal(synth.to_u16(whole[:T]), G, err_msg="gather T=%d" % T)
    assert is_sentinel(whole[T:]), "buffer rows >= %d touched" % T
    assert is_sentinel(Y[T:]), "Y rows >= %d touched" % T
    rows = sample_rows(T, tp, n_random, rng, window)
    ref = oracle.gemm_rows(G, synth.to_u16(Wt), rows)
    assert_close(Y[torch.as_tensor(rows, device=dev())], ref, "AG T=%d N=%d" % (T, N))
    return Wt


def check_rs(buf, T, K, g, rng, Bt=None, n_random=16, window=WINDOW):
    tp, H = buf.tp, buf.hidden
    c = T // tp
    buf.set_active_shape([T, H])
    A = [synth.normal_bf16((T, K), 1.0, g, dev()) for _ in range(tp)]
    if Bt is None:
        Bt = [synth.normal_bf16((H, K), 1.0 / math.sqrt(K), g, dev()) for _ in range(tp)]
    pad = 2
    big = sentinel((tp * (c + pad), H))
    Ys = [big[r * (c + pad): r * (c + pad) + c] for r in range(tp)]
    buf.gemm_rs(A, Bt, Ys)
    torch.cuda.synchronize()
    assert buf.query_status() == ub.UB_OK
    for r in range(tp):
        assert is_sentinel(big[r * (c + pad) + c:(r + 1) * (c + pad)]), "guard after block %d" % r
    rows = sample_rows(T, tp, n_random, rng, window)
    ridx = torch.as_tensor(rows, device=dev())
    ref, owner, local = oracle.gemm_rs_rows([synth.to_u16(a[ridx]) for a in A],
                                            [synth.to_u16(b) for b in Bt], rows, T)
    got = torch.stack([Ys[int(o)][int(i)] for o, i in zip(owner, local)])
    assert_close(got, ref, "RS T=%d K=%d" % (T, K))
    return Bt


def test_qkv_workload():
    w = synth.WORKLOADS["qkv"]
    g = synth.generator(dev())
    rng = np.random.default_rng(0)
    Ts = synth.token_counts("qkv")
    with ub.UserBuffer([w.max_tokens, w.hidden], w.tp) as buf:
        Wt = None
        for T in Ts[:4] + [w.max_tokens]:
            Wt = check_ag(buf, T, w.ag_n[0], g, rng, Wt)
        assert buf.counters()["device_allocations"] == 3


def test_swiglu_workload():
    w = synth.WORKLOADS["swiglu"]
    g = synth.generator(dev())
    rng = np.random.default_rng(1)
    Ts = synth.token_counts("swiglu")
    with ub.UserBuffer([w.max_tokens, w.hidden], w.tp) as buf:
        Wt = Bt = None
        for T in Ts[:3] + [w.max_tokens]:
            Wt = check_ag(buf, T, w.ag_n[0], g, rng, Wt)
            Bt = check_rs(buf, T, w.rs_k[0], g, rng, Bt)


def test_large_workload():
    w = synth.WORKLOADS["large"]
    g = synth.generator(dev())
    rng = np.random.default_rng(2)
    Ts = synth.token_counts("large")
    with ub.UserBuffer([w.max_tokens, w.hidden], w.tp) as buf:
        B = {K: None for K in w.rs_k}
        for T in Ts[:2] + [w.max_tokens]:
            for K in w.rs_k:
                B[K] = check_rs(buf, T, K, g, rng, B[K], n_random=8, window=128)


def test_active_shape_stress_64_microbatches():
    w = synth.WORKLOADS["stress"]
    g = synth.generator(dev())
    rng = np.random.default_rng(3)
    Ts = synth.token_counts("stress")
    assert len(Ts) == 64
    with ub.UserBuffer([w.max_tokens, w.hidden], w.tp) as buf:
        ptr = buf.buffer_ptr()
        Wt = Bt = None
        for T in Ts:
            # 16 seeded random rows per call on top of every chunk's edge rows
            Wt = check_ag(buf, T, w.ag_n[0], g, rng, Wt, n_random=16, window=None)
            Bt = check_rs(buf, T, w.rs_k[0], g, rng, Bt, n_random=16, window=None)
        c = buf.counters()
        assert c["device_allocations"] == 3
        assert c["ag_calls"] == 64 and c["rs_calls"] == 64
        assert buf.buffer_ptr() == ptr

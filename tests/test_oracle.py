"""Pins for the CPU oracle: it is checked against things other than itself.

* hand-worked examples and chunk offsets written out from the pages' rules
  (tests/golden/, each with its citation);
* brute force in exact integer arithmetic (numpy int64) on tiny inputs;
* the tp = 1 special case, which is a textbook GEMM (numpy float64 matmul);
* the shard-concatenation identity of the reduce-scatter sum;
* "active shape == buffer allocated at exactly T" and the untouched capacity tail;
* the five active-shape constraints, each violated on its own.

Every check is also run once against a planted mistake (a shard dropped, an operand
transposed, offsets taken from the capacity...) to show that it can fail.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
from gemm_overlap_gemms_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SENTINEL = 0xFFFF


def bf16_bits(a) -> np.ndarray:
    """Exact small values (or float arrays) -> bf16 bit patterns."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return synth.to_u16(t)


def bits_to_f64(a: np.ndarray) -> np.ndarray:
    return synth.from_u16(a).to(torch.float64).numpy()


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_special_values():
    one = 0x3F80
    assert oracle.round_bf16(1.0) == one
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == one          # tie -> even (down)
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == one + 2  # tie -> even (up)
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == one + 1  # above the tie
    assert oracle.round_bf16(-2.0) == 0xC000
    assert oracle.round_bf16(0.0) == 0x0000
    assert oracle.round_bf16(3.5e38) == 0x7F80                # past max finite -> inf
    assert oracle.round_bf16(float("nan")) == 0x7FC0


def test_round_bf16_matches_library_on_fp32_values():
    # For values that are exact in fp32, one-step rounding from double must agree
    # with the library's fp32 -> bf16 conversion (round to nearest even).
    g = torch.Generator().manual_seed(1)
    x = torch.randn(4000, generator=g, dtype=torch.float32) * 10.0
    x = torch.cat([x, torch.tensor([1e-39, -3e-40, 6e-39], dtype=torch.float32)])
    want = synth.to_u16(x.to(torch.bfloat16))
    got = np.array([oracle.round_bf16(float(v)) for v in x.tolist()], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)


# ---------------------------------------------------------------- chunk layout

def test_chunk_offsets_golden():
    cases = json.load(open(os.path.join(GOLDEN, "chunk_offsets.json")))["cases"]
    for case in cases:
        T, tp, H = case["T"], case["tp"], case["hidden"]
        assert oracle.chunk_rows(T, tp) == case["rows_per_chunk"]
        offs = [oracle.chunk_offset(T, tp, r) for r in range(tp)]
        assert offs == case["row_offsets"]
        assert [o * H * 2 for o in offs] == case["byte_offsets"]
        if case["T"] != case["capacity"]:
            assert offs != case["capacity_reading"]


def check_gather(G, shards, T):
    """Pin: rows [r*c, (r+1)*c) of G hold shard r; rows >= T hold the sentinel."""
    tp = len(shards)
    c = T // tp
    for r, s in enumerate(shards):
        if not np.array_equal(G[r * c:(r + 1) * c], s):
            return False
    return bool(np.all(G[T:] == SENTINEL))


@pytest.mark.parametrize("T,tp,cap", [(6, 3, 12), (8, 2, 8), (4, 4, 16), (12, 4, 20)])
def test_allgather_prefix_and_tail(T, tp, cap):
    H = 5
    g = synth.generator()
    shards = [synth.to_u16(synth.small_int_bf16((T // tp, H), -9, 9, g)) for _ in range(tp)]
    G = np.full((cap, H), SENTINEL, dtype=np.uint16)
    oracle.allgather(shards, G, T)
    assert check_gather(G, shards, T)
    # planted mistake: offsets from the capacity instead of T
    if cap != T:
        bad = np.full((cap, H), SENTINEL, dtype=np.uint16)
        cc = cap // tp
        for r, s in enumerate(shards):
            bad[r * cc:r * cc + T // tp] = s
        assert not check_gather(bad, shards, T)


# ---------------------------------------------------------------- worked examples

def test_worked_example_ag():
    ex = json.load(open(os.path.join(GOLDEN, "worked_examples.json")))["ag_gemm"]
    assert np.array_equal(np.array(ex["Wt_stored_NxH"]), np.array(ex["W_math_HxN"]).T)
    shards = [bf16_bits(s) for s in ex["shards"]]
    Wt = bf16_bits(ex["Wt_stored_NxH"])
    G = np.full((ex["capacity"], ex["H"]), SENTINEL, dtype=np.uint16)
    G, Y = oracle.ag_gemm(shards, Wt, G=G, T=ex["T"])
    np.testing.assert_array_equal(bits_to_f64(G[:ex["T"]]), np.array(ex["G_active_rows"]))
    assert np.all(G[ex["T"]:] == SENTINEL)
    np.testing.assert_array_equal(Y, np.array(ex["Y"], dtype=np.float64))


def test_worked_example_rs():
    ex = json.load(open(os.path.join(GOLDEN, "worked_examples.json")))["gemm_rs"]
    for bm, bt in zip(ex["B_math_KxH"], ex["Bt_stored_HxK"]):
        assert np.array_equal(np.array(bt), np.array(bm).T)
    A = [bf16_bits(a) for a in ex["A"]]
    Bt = [bf16_bits(b) for b in ex["Bt_stored_HxK"]]
    S, Y = oracle.gemm_rs(A, Bt)
    np.testing.assert_array_equal(S, np.array(ex["S"], dtype=np.float64))
    for r in range(ex["tp"]):
        np.testing.assert_array_equal(Y[r], np.array(ex["Y_blocks"][r], dtype=np.float64))


# ---------------------------------------------------------------- brute force (exact ints)

def ag_exact_int(shards, Wt):
    """Independent statement in exact integers: concatenate, then matmul in int64."""
    X = np.concatenate([bits_to_f64(s) for s in shards]).astype(np.int64)
    return X @ bits_to_f64(Wt).astype(np.int64).T


def rs_exact_int(A, Bt):
    S = np.zeros((A[0].shape[0], Bt[0].shape[0]), dtype=np.int64)
    for a, b in zip(A, Bt):
        S += bits_to_f64(a).astype(np.int64) @ bits_to_f64(b).astype(np.int64).T
    return S


def _int_cases():
    for tp in (1, 2, 3, 4):
        for T in range(tp, 17, tp):
            for H in (1, 3, 8, 16):
                yield T, H, tp


def test_ag_bruteforce_integer():
    g = synth.generator(seed=7)
    n = 0
    for T, H, tp in _int_cases():
        N = 1 + (T + H) % 5
        shards = [synth.to_u16(synth.small_int_bf16((T // tp, H), -8, 8, g)) for _ in range(tp)]
        Wt = synth.to_u16(synth.small_int_bf16((N, H), -8, 8, g))
        G = np.full((T + 3, H), SENTINEL, dtype=np.uint16)
        G, Y = oracle.ag_gemm(shards, Wt, G=G, T=T)
        np.testing.assert_array_equal(Y, ag_exact_int(shards, Wt).astype(np.float64))
        assert check_gather(G, shards, T)
        n += 1
    assert n > 100


def test_rs_bruteforce_integer():
    g = synth.generator(seed=8)
    for T, H, tp in _int_cases():
        K = 1 + (3 * T + H) % 7
        A = [synth.to_u16(synth.small_int_bf16((T, K), -8, 8, g)) for _ in range(tp)]
        Bt = [synth.to_u16(synth.small_int_bf16((H, K), -8, 8, g)) for _ in range(tp)]
        S, Y = oracle.gemm_rs(A, Bt)
        want = rs_exact_int(A, Bt).astype(np.float64)
        np.testing.assert_array_equal(S, want)
        c = T // tp
        for r in range(tp):
            np.testing.assert_array_equal(Y[r], want[r * c:(r + 1) * c])


def test_bruteforce_detects_planted_mistakes():
    g = synth.generator(seed=9)
    T, H, tp, N, K = 8, 6, 2, 5, 4
    shards = [synth.to_u16(synth.small_int_bf16((T // tp, H), -8, 8, g)) for _ in range(tp)]
    Wt = synth.to_u16(synth.small_int_bf16((N, H), -8, 8, g))
    want = ag_exact_int(shards, Wt)
    # shards in the wrong order
    _, Y = oracle.ag_gemm(shards[::-1], Wt)
    assert not np.array_equal(Y, want)
    # a square weight passed transposed
    Wsq = synth.to_u16(synth.small_int_bf16((H, H), -8, 8, g))
    _, Y = oracle.ag_gemm(shards, np.ascontiguousarray(Wsq.T))
    assert not np.array_equal(Y, ag_exact_int(shards, Wsq))
    # a dropped shard term in the reduce-scatter sum
    A = [synth.to_u16(synth.small_int_bf16((T, K), 1, 8, g)) for _ in range(tp)]
    Bt = [synth.to_u16(synth.small_int_bf16((H, K), 1, 8, g)) for _ in range(tp)]
    S1, _ = oracle.gemm_rs(A[:1], Bt[:1])
    assert not np.array_equal(S1, rs_exact_int(A, Bt))
    # a flipped sign
    neg = synth.to_u16(-synth.from_u16(A[1]))
    S2, _ = oracle.gemm_rs([A[0], neg], Bt)
    assert not np.array_equal(S2, rs_exact_int(A, Bt))


# ---------------------------------------------------------------- closed forms

def test_rs_all_ones_closed_form():
    tp, T, K, H = 4, 8, 7, 3
    A = [bf16_bits(np.ones((T, K))) for _ in range(tp)]
    Bt = [bf16_bits(np.ones((H, K))) for _ in range(tp)]
    S, Y = oracle.gemm_rs(A, Bt)
    assert np.all(S == tp * K)


def test_rs_row_ownership_encoded():
    # A_j[t][0] = t, everything else 0; Bt_j[n][0] = 1 for j == 0 only.
    # Then S[t][n] = t, so block r row i must hold r*c + i.
    tp, T, K, H = 4, 12, 2, 3
    A = [bf16_bits(np.stack([np.arange(T), np.zeros(T)], 1)) for _ in range(tp)]
    Bt = [bf16_bits(np.stack([np.full(H, 1.0 if j == 0 else 0.0), np.zeros(H)], 1))
          for j in range(tp)]
    S, Y = oracle.gemm_rs(A, Bt)
    c = T // tp
    for r in range(tp):
        assert np.all(Y[r] == (r * c + np.arange(c))[:, None])


def test_ag_one_hot_selects_weight_columns():
    # X row t is the unit vector e_{t mod H}; then Y[t] = W[t mod H, :] = Wt[:, t mod H].
    tp, T, H, N = 2, 8, 4, 3
    X = np.zeros((T, H))
    X[np.arange(T), np.arange(T) % H] = 1.0
    shards = [bf16_bits(X[r * (T // tp):(r + 1) * (T // tp)]) for r in range(tp)]
    Wt = bf16_bits(np.arange(N * H).reshape(N, H) - 5.0)
    _, Y = oracle.ag_gemm(shards, Wt)
    Wf = bits_to_f64(Wt)
    for t in range(T):
        np.testing.assert_array_equal(Y[t], Wf[:, t % H])


# ---------------------------------------------------------------- library special cases

def test_tp1_is_a_textbook_gemm():
    g = synth.generator(seed=3)
    for T, H, N in [(37, 64, 29), (128, 256, 96)]:
        shards, W = synth.ag_inputs(T, H, N, 1, g)
        s = synth.to_u16(shards[0])
        Wt = synth.to_u16(W)
        _, Y = oracle.ag_gemm([s], Wt)
        ref = bits_to_f64(s) @ bits_to_f64(Wt).T
        # both are double sums of exact products; only the summation order differs
        bound = H * 2.0 ** -52 * (np.abs(bits_to_f64(s)) @ np.abs(bits_to_f64(Wt)).T)
        assert np.all(np.abs(Y - ref) <= bound)
        S, Yb = oracle.gemm_rs([s], [Wt])
        assert np.all(np.abs(S - ref) <= bound)
        np.testing.assert_array_equal(Yb[0], S)


def test_rs_equals_gemm_on_concatenated_shards():
    g = synth.generator(seed=4)
    tp, T, K, H = 4, 24, 40, 48
    A, Bt = synth.rs_inputs(T, K, H, tp, g)
    A = [synth.to_u16(a) for a in A]
    Bt = [synth.to_u16(b) for b in Bt]
    S, Y = oracle.gemm_rs(A, Bt)
    Acat = np.concatenate(A, axis=1)           # [T, tp*K]
    Btcat = np.concatenate(Bt, axis=1)         # [H, tp*K]
    S1, _ = oracle.gemm_rs([Acat], [Btcat])
    ref = bits_to_f64(Acat) @ bits_to_f64(Btcat).T
    bound = tp * K * 2.0 ** -52 * (np.abs(bits_to_f64(Acat)) @ np.abs(bits_to_f64(Btcat)).T)
    assert np.all(np.abs(S - S1) <= 2 * bound)
    assert np.all(np.abs(S - ref) <= 2 * bound)
    np.testing.assert_array_equal(np.concatenate(Y), S)


# ---------------------------------------------------------------- active shape

def test_active_shape_equals_exact_allocation():
    g = synth.generator(seed=5)
    tp, H, N, cap = 4, 32, 24, 64
    for T in (4, 20, 36, 64):
        shards, W = synth.ag_inputs(T, H, N, tp, g)
        shards = [synth.to_u16(s) for s in shards]
        Wt = synth.to_u16(W)
        Gcap = np.full((cap, H), SENTINEL, dtype=np.uint16)
        Gcap, Ycap = oracle.ag_gemm(shards, Wt, G=Gcap, T=T)
        Gex = np.full((T, H), SENTINEL, dtype=np.uint16)
        Gex, Yex = oracle.ag_gemm(shards, Wt, G=Gex, T=T)
        np.testing.assert_array_equal(Gcap[:T], Gex)
        np.testing.assert_array_equal(Ycap.view(np.uint64), Yex.view(np.uint64))
        assert np.all(Gcap[T:] == SENTINEL)


def test_rows_helpers_agree_with_full_products():
    g = synth.generator(seed=6)
    tp, T, H, N, K = 2, 10, 16, 12, 8
    shards, W = synth.ag_inputs(T, H, N, tp, g)
    shards = [synth.to_u16(s) for s in shards]
    Wt = synth.to_u16(W)
    G, Y = oracle.ag_gemm(shards, Wt)
    rows = np.array([0, 4, 5, 9])
    np.testing.assert_array_equal(oracle.gemm_rows(G, Wt, rows), Y[rows])
    A, Bt = synth.rs_inputs(T, K, H, tp, g)
    A = [synth.to_u16(a) for a in A]
    Bt = [synth.to_u16(b) for b in Bt]
    S, Yb = oracle.gemm_rs(A, Bt)
    out, owner, local = oracle.gemm_rs_rows([a[rows] for a in A], Bt, rows, T)
    np.testing.assert_array_equal(out, S[rows])
    np.testing.assert_array_equal(owner, rows // (T // tp))
    np.testing.assert_array_equal(local, rows % (T // tp))


@pytest.mark.parametrize("shape,expect", [
    ([8, 16], 0),
    ([8], 1), ([8, 16, 1], 1),          # not two-dimensional
    ([0, 16], 2), ([8, 0], 2),          # zero
    ([40, 16], 3),                      # beyond capacity
    ([8, 32], 4),                       # hidden changed
    ([6, 16], 5),                       # not divisible by tp
    ([32, 16], 0), ([4, 16], 0),
])
def test_active_shape_constraints(shape, expect):
    assert oracle.check_active_shape(shape, cap_tokens=32, cap_hidden=16, tp=4) == expect


# ---------------------------------------------------------------- SwiGLU

def test_silu_textbook_values_and_identity():
    # silu(x) = x * sigmoid(x); sigmoid(1) = 0.7310585786300049 (textbook value)
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - 0.7310585786300049) < 1e-15
    assert abs(oracle.silu(-1.0) + 0.2689414213699951) < 1e-15
    for x in (-30.0, -2.5, -0.1, 0.3, 4.0, 25.0):
        # silu(x) - silu(-x) = x * (sigmoid(x) + sigmoid(-x)) = x
        assert abs(oracle.silu(x) - oracle.silu(-x) - x) < 1e-12 * max(1.0, abs(x))
    assert oracle.silu(-800.0) == 0.0 or abs(oracle.silu(-800.0)) < 1e-300
    assert oracle.silu(800.0) == 800.0


def test_silu_matches_library_routine():
    x = torch.linspace(-20, 20, 2001, dtype=torch.float64)
    want = torch.nn.functional.silu(x).numpy()
    got = np.array([oracle.silu(v) for v in x.tolist()])
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-300)


def test_swiglu_takes_gate_first_then_up():
    F = 3
    Y = np.array([[1.0, 0.0, -1.0, 2.0, 5.0, 7.0]])     # gate = (1, 0, -1), up = (2, 5, 7)
    Z = oracle.swiglu(Y)
    np.testing.assert_allclose(Z[0], [2 * 0.7310585786300049, 0.0, 7 * -0.2689414213699951], rtol=1e-15)
    # planted mistake: halves swapped
    Zs = oracle.swiglu(np.concatenate([Y[:, F:], Y[:, :F]], axis=1))
    assert not np.allclose(Zs, Z)


# ---------------------------------------------------------------- backward-pass products

def test_gemm_xw_brute_force_and_transpose_identity():
    g = synth.generator(seed=61)
    for T, K, N in [(5, 3, 4), (16, 16, 8), (9, 7, 13)]:
        X = synth.to_u16(synth.small_int_bf16((T, K), -8, 8, g))
        W = synth.to_u16(synth.small_int_bf16((K, N), -8, 8, g))
        rows = np.arange(T)
        Y = oracle.gemm_xw_rows(X, W, rows)
        want = bits_to_f64(X).astype(np.int64) @ bits_to_f64(W).astype(np.int64)
        np.testing.assert_array_equal(Y, want.astype(np.float64))
        # the same product through the pinned out-x-in path with the weight transposed
        np.testing.assert_array_equal(Y, oracle.gemm_rows(X, np.ascontiguousarray(W.T), rows))
        if K != N:  # planted mistake: W read as if it were stored N x K
            with pytest.raises(AssertionError):
                oracle.gemm_xw_rows(X, np.ascontiguousarray(W.T), rows)


def test_gemm_tn_brute_force_and_library():
    g = synth.generator(seed=62)
    for T, M, N in [(6, 4, 5), (33, 16, 24)]:
        D = synth.to_u16(synth.small_int_bf16((T, M), -8, 8, g))
        G = synth.to_u16(synth.small_int_bf16((T, N), -8, 8, g))
        out = oracle.gemm_tn(D, G)
        want = bits_to_f64(D).astype(np.int64).T @ bits_to_f64(G).astype(np.int64)
        np.testing.assert_array_equal(out, want.astype(np.float64))
        # gemm_tn(D, G) == gemm_tn(G, D).T (the sum over t is symmetric in its operands)
        np.testing.assert_array_equal(out, oracle.gemm_tn(G, D).T)
    D, G = [synth.to_u16(synth.normal_bf16((40, 12), 1.0, g)) for _ in range(2)]
    ref = bits_to_f64(D).T @ bits_to_f64(G)
    bound = 40 * 2.0 ** -52 * (np.abs(bits_to_f64(D)).T @ np.abs(bits_to_f64(G)))
    assert np.all(np.abs(oracle.gemm_tn(D, G) - ref) <= bound)


def test_backward_products_match_forward_identities():
    """Chain rule on a tiny layer, by finite algebra: for Y = X Wt^T the input gradient
    dY Wt and the weight gradient dY^T X are the unique linear maps with
    <dY, X' Wt^T> = <dY Wt, X'> and <dY, X Wt'^T> = <dY^T X, Wt'> for every X', Wt'."""
    g = synth.generator(seed=63)
    T, H, N = 7, 5, 6
    X = synth.to_u16(synth.small_int_bf16((T, H), -4, 4, g))
    Wt = synth.to_u16(synth.small_int_bf16((N, H), -4, 4, g))
    dY = synth.to_u16(synth.small_int_bf16((T, N), -4, 4, g))
    dX = oracle.gemm_xw_rows(dY, Wt, np.arange(T))      # dY @ Wt  ([T, N] x [N, H])
    dWt = oracle.gemm_tn(dY, X)                          # dY^T @ X ([N, H])
    for trial in range(3):
        Xp = synth.to_u16(synth.small_int_bf16((T, H), -3, 3, g))
        Wp = synth.to_u16(synth.small_int_bf16((N, H), -3, 3, g))
        lhs_x = np.sum(bits_to_f64(dY) * oracle.gemm_rows(Xp, Wt, np.arange(T)))
        assert lhs_x == np.sum(dX * bits_to_f64(Xp))
        lhs_w = np.sum(bits_to_f64(dY) * oracle.gemm_rows(X, Wp, np.arange(T)))
        assert lhs_w == np.sum(dWt * bits_to_f64(Wp))


# ---------------------------------------------------------------- bulk reduce-scatter

def test_reduce_scatter_integer_and_ownership():
    g = synth.generator(seed=81)
    for tp, T, H in [(1, 5, 3), (2, 8, 4), (4, 12, 7), (3, 9, 16)]:
        P = [synth.to_u16(synth.small_int_bf16((T, H), -8, 8, g)) for _ in range(tp)]
        Y = oracle.reduce_scatter(P)
        S = sum(bits_to_f64(p).astype(np.int64) for p in P)
        c = T // tp
        for r in range(tp):
            np.testing.assert_array_equal(Y[r], S[r * c:(r + 1) * c].astype(np.float64))
        # planted mistake: a shard left out of the sum
        if tp > 1:
            Yd = oracle.reduce_scatter(P[:-1] + [np.zeros_like(P[0])])
            assert not all(np.array_equal(a, b) for a, b in zip(Yd, Y)) or not np.any(bits_to_f64(P[-1]))


def test_reduce_scatter_of_shard_products_is_gemm_rs():
    """RS of the per-shard products equals the pinned GEMM-RS (exact on integers)."""
    g = synth.generator(seed=82)
    tp, T, K, H = 4, 8, 5, 6
    A = [synth.to_u16(synth.small_int_bf16((T, K), -3, 3, g)) for _ in range(tp)]
    Bt = [synth.to_u16(synth.small_int_bf16((H, K), -3, 3, g)) for _ in range(tp)]
    # each product is small enough to be exact in bf16, so P_j can be stored as bf16
    P = [bf16_bits(oracle.gemm_rows(a, b, np.arange(T))) for a, b in zip(A, Bt)]
    _, Yrs = oracle.gemm_rs(A, Bt)
    for a, b in zip(oracle.reduce_scatter(P), Yrs):
        np.testing.assert_array_equal(a, b)

"""The split last wave of the CTA-pair kernel (UB_OPT_STREAMK): the tiles left over after
the whole waves are cut into s equal k-pieces on s consecutive pairs; the pair holding
piece 0 adds the other pieces' fp32 partials in piece order.

Shapes are chosen so that pieces hold different numbers of k-blocks, a ragged last
k-block (K not a multiple of 64) sits in the last piece, a tile has up to seven
contributing pieces, and SM margins change the number of pairs (and so s and the
whole-wave count). Integer-valued inputs make every sum exact, so there the result must
equal the oracle's rounded to bf16 bit for bit, however the pieces are cut.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_overlap_gemms_gb300 import synth, ub
from gpu_helpers import assert_close, oracle_ag, oracle_rs, run_ag, run_rs

pytestmark = pytest.mark.gpu


def _round_bf16(a: np.ndarray) -> np.ndarray:
    return np.array([oracle.round_bf16(v) for v in a.ravel()], dtype=np.uint16).reshape(a.shape)


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int16).clone()


# (SM margin, K), 8 pair tiles: margin 0 -> 76 pairs, each tile cut into 8 pieces (seven
# contributors); margin 140 -> 6 pairs, one whole wave, then 2 tiles in 3 pieces; margin
# 97 -> 27 pairs, 8 tiles in 3 pieces. K = 2600: 41 k-blocks per shard, the last ragged,
# 164 in all, so the pieces differ in length; K = 4096: 64 per shard.
@pytest.mark.parametrize("margin,K", [(0, 2600), (0, 4096), (140, 2600), (97, 4096)])
def test_rs_split_tail_integer_inputs_bit_exact(margin, K):
    tp, H = 4, 512
    T = tp * 256
    g = synth.generator(seed=301)
    A = [synth.small_int_bf16((T, K), -3, 3, g) for _ in range(tp)]
    Bt = [synth.small_int_bf16((H, K), -3, 3, g) for _ in range(tp)]
    _, Yb = oracle_rs(A, Bt)
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_option("cta_pair", 1)
        buf.set_option("sm_margin", margin)
        res = {}
        for streamk in (1, 0):
            buf.set_option("streamk", streamk)
            Ys, _ = run_rs(buf, A, Bt)
            res[streamk] = [_bits(y) for y in Ys]
            for r in range(tp):
                np.testing.assert_array_equal(synth.to_u16(Ys[r]), _round_bf16(Yb[r]),
                                              err_msg="streamk=%d margin=%d K=%d block %d" % (streamk, margin, K, r))
        for a, b in zip(res[1], res[0]):   # exact sums: split or not, the same bits
            assert torch.equal(a, b)
        assert buf.query_status() == ub.UB_OK


@pytest.mark.parametrize("margin", [0, 13, 140])
def test_rs_split_tail_normal_inputs(margin):
    tp, H, K = 4, 768, 3000
    T = tp * 320                  # 5 x 3 pair tiles, 4 x 47 k-blocks
    g = synth.generator(seed=302)
    A, Bt = synth.rs_inputs(T, K, H, tp, g)
    _, Yb = oracle_rs(A, Bt)
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_option("cta_pair", 1)
        buf.set_option("streamk", 1)
        buf.set_option("sm_margin", margin)
        Ys, _ = run_rs(buf, A, Bt)
        first = [_bits(y) for y in Ys]
        for r in range(tp):
            assert_close(Ys[r], Yb[r], "RS split margin=%d block %d" % (margin, r))
        Ys2, _ = run_rs(buf, A, Bt)   # same launch shape: same bits
        for a, b in zip(first, Ys2):
            assert torch.equal(a, _bits(b))
        assert buf.query_status() == ub.UB_OK


@pytest.mark.parametrize("gather", [0, 1, 2])
@pytest.mark.parametrize("margin", [0, 130])
def test_ag_split_tail(margin, gather):
    """AG with each gather: the last wave's tiles, a partial N tile among them
    (N = 3 x 256 + 128), cut into k-pieces while the chunks land."""
    tp, H, N = 4, 4096, 896
    T = tp * 256
    g = synth.generator(seed=303)
    shards, Wt = synth.ag_inputs(T, H, N, tp, g)
    Gref, Yref = oracle_ag(shards, Wt)
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_option("cta_pair", 1)
        buf.set_option("streamk", 1)
        buf.set_option("sm_margin", margin)
        buf.set_option("gather_kernel", gather)
        Y = run_ag(buf, shards, Wt)
        np.testing.assert_array_equal(synth.to_u16(buf.buffer()[:T]), Gref)
        assert_close(Y, Yref, "AG split margin=%d gather=%d" % (margin, gather))
        assert buf.query_status() == ub.UB_OK


def test_swiglu_split_tail():
    tp, H, F = 4, 3072, 384           # 2F = 768: 3 pair tiles across, 48 k-blocks
    T = tp * 192
    g = synth.generator(seed=304)
    shards = [synth.normal_bf16((T // tp, H), 1.0, g) for _ in range(tp)]
    W1 = synth.normal_bf16((2 * F, H), H ** -0.5, g)
    d = torch.device("cuda", torch.cuda.current_device())
    Xu = np.concatenate([synth.to_u16(s) for s in shards])
    ref = oracle.swiglu(oracle.gemm_rows(Xu, synth.to_u16(W1), np.arange(T)))
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_option("cta_pair", 1)
        buf.set_option("streamk", 1)
        Z = torch.empty((T, F), dtype=torch.bfloat16, device=d)
        buf.ag_gemm_swiglu([s.to(d) for s in shards], W1.to(d), Z)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    assert_close(Z, ref, "SwiGLU split")


@pytest.mark.parametrize("T", [256, 512])
def test_ag_with_fewer_tiles_than_pairs_splits_by_default_and_matches(T):
    """The QKV projection at T = 256 / 512 (12 / 24 pair tiles on 76 pairs, no whole wave):
    by default every tile is cut into k-pieces over the idle pairs, behind the gather
    kernel's chunk flags; integer inputs make the sums exact, so the result equals the
    oracle's rounded to bf16 bit for bit, and the gathered buffer equals its
    concatenation."""
    tp, H, N = 4, 4096, 3072
    c = T // tp
    g = synth.generator(seed=307)
    shards = [synth.small_int_bf16((c, H), -2, 2, g) for _ in range(tp)]
    Wt = synth.small_int_bf16((N, H), -2, 2, g)
    with ub.UserBuffer([8192, H], tp) as buf:
        buf.set_active_shape([T, H])
        Y = run_ag(buf, shards, Wt)
        cnt = buf.counters()
        assert ub.KERNELS[cnt["last_kernel"]] == "pair" and cnt["last_pieces"] > 1, cnt
        assert ub.GATHERS[cnt["last_gather"]] == "gather_kernel", cnt
        assert buf.query_status() == ub.UB_OK
        G = buf.buffer()[:T].cpu()
    Gref, Yref = oracle_ag(shards, Wt)
    np.testing.assert_array_equal(synth.to_u16(G), Gref)
    assert np.abs(Yref).max() < 2 ** 24
    np.testing.assert_array_equal(synth.to_u16(Y), _round_bf16(Yref))


def test_rs_grouped_tile_order_integer_inputs_exact():
    """Weights above 256 MB (tp 8 x [4096, 4096]): the pair kernel walks tile rows in
    groups of eight, rows fastest, with the split last wave; integer inputs make the sums
    exact, so every sampled row -- two in each 256-row tile row, all 4096 columns --
    equals the oracle's rounded to bf16 bit for bit."""
    tp, H, K, T = 8, 4096, 4096, 2048
    g = synth.generator(seed=309)
    A = [synth.small_int_bf16((T, K), -1, 1, g) for _ in range(tp)]
    Bt = [synth.small_int_bf16((H, K), -1, 1, g) for _ in range(tp)]
    c = T // tp
    with ub.UserBuffer([T, H], tp) as buf:
        buf.set_active_shape([T, H])
        Ys, _ = run_rs(buf, [a.cpu() for a in A], [b.cpu() for b in Bt])
        cnt = buf.counters()
        assert ub.KERNELS[cnt["last_kernel"]] == "pair", cnt
        assert buf.query_status() == ub.UB_OK
    rows = np.unique(np.concatenate([np.arange(0, T, 256), np.arange(255, T, 256), [1, T - 2]]))
    ridx = torch.as_tensor(rows)
    ref, owner, local = oracle.gemm_rs_rows([synth.to_u16(a.cpu()[ridx]) for a in A],
                                            [synth.to_u16(b.cpu()) for b in Bt], rows, T)
    assert np.abs(ref).max() < 2 ** 24
    got = torch.stack([Ys[int(o)][int(i)] for o, i in zip(owner, local)])
    np.testing.assert_array_equal(synth.to_u16(got), _round_bf16(ref))

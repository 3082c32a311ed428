"""The CTA-pair AG kernel's tile order: tile rows walked in groups (rows fastest inside a
group) -- groups of eight when the first wave reads only the self chunk's in-place rows,
else groups of one chunk's tile rows -- across the in-place region and the gathered
regions, with partial groups and a partial last tile row. Integer-valued inputs make
every sum exact, so the sampled rows -- the first and last row of every 256-row tile
row, and the rows around every chunk boundary -- must equal the oracle's rounded to
bf16 bit for bit, and the gathered buffer its concatenation.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_overlap_gemms_gb300 import synth, ub
from gpu_helpers import assert_close, dev, is_sentinel, sentinel

pytestmark = pytest.mark.gpu


def _round_bf16(a: np.ndarray) -> np.ndarray:
    return np.array([oracle.round_bf16(v) for v in a.ravel()], dtype=np.uint16).reshape(a.shape)


def _rows(T: int, c: int) -> np.ndarray:
    tiles = np.arange(0, T, 256)
    bounds = np.arange(c, T, c)
    return np.unique(np.clip(np.concatenate([tiles, np.minimum(tiles + 255, T - 1), bounds - 1, bounds, [T - 1]]),
                             0, T - 1))


# (T, N, self rank): N = 7168 (28 tile columns): the self chunk's 5 tile rows are 140 pair
# tiles, more than a wave, so groups of eight; N = 3584 (14 columns): 70 tiles, less than
# a wave, so groups of one chunk's 4 tile rows. Self rank 2 puts the chunks before it in a
# third region, walked last.
@pytest.mark.parametrize("T,N,self_rank", [(4640, 7168, 0), (4640, 3584, 0), (4640, 7168, 2), (8192, 3584, 1)])
def test_ag_grouped_order_integer_inputs_exact(T, N, self_rank):
    tp, H = 4, 4096
    c = T // tp
    g = synth.generator(seed=401)
    shards = [synth.small_int_bf16((c, H), -2, 2, g) for _ in range(tp)]
    Wt = synth.small_int_bf16((N, H), -2, 2, g)
    with ub.UserBuffer([8192, H], tp) as buf:
        buf.set_active_shape([T, H])
        buf.set_option("self_rank", self_rank)
        Y = sentinel((T + 3, N))
        buf.ag_gemm([s.to(dev()) for s in shards], Wt.to(dev()), Y[:T])
        torch.cuda.synchronize()
        cnt = buf.counters()
        assert ub.KERNELS[cnt["last_kernel"]] == "pair", cnt
        assert buf.query_status() == ub.UB_OK
        G = buf.buffer()[:T].cpu()
    Xu = np.concatenate([synth.to_u16(s) for s in shards])
    np.testing.assert_array_equal(synth.to_u16(G), Xu)
    rows = _rows(T, c)
    ref = oracle.gemm_rows(Xu, synth.to_u16(Wt), rows)
    assert np.abs(ref).max() < 2 ** 24
    got = Y[torch.as_tensor(rows, device=dev())]
    np.testing.assert_array_equal(synth.to_u16(got), _round_bf16(ref))
    assert is_sentinel(Y[T:])


def test_ag_swiglu_grouped_order_matches_oracle():
    """AG + SwiGLU at the benchmark's T = 4640 (groups of eight), sampled rows of every
    tile row against the oracle's SwiGLU of its exact products."""
    tp, H, F = 4, 4096, 3584
    T = 4640
    c = T // tp
    g = synth.generator(seed=402)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    W1 = synth.normal_bf16((2 * F, H), H ** -0.5, g)
    with ub.UserBuffer([8192, H], tp) as buf:
        buf.set_active_shape([T, H])
        Z = sentinel((T + 2, F))
        buf.ag_gemm_swiglu([s.to(dev()) for s in shards], W1.to(dev()), Z[:T])
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    Xu = np.concatenate([synth.to_u16(s) for s in shards])
    rows = _rows(T, c)
    ref = oracle.swiglu(oracle.gemm_rows(Xu, synth.to_u16(W1), rows))
    assert_close(Z[torch.as_tensor(rows, device=dev())], ref, "SwiGLU grouped order")
    assert is_sentinel(Z[T:])


def test_ag_kn_and_from_buffer_grouped_order_integer_inputs_exact():
    """The K x N-weight AG (the dgrad of the row-parallel layer) and the AG from a buffer
    gathered ahead (groups of eight at any T: no chunk to wait for), T = 4640."""
    tp, H, N = 4, 4096, 3584
    T = 4640
    c = T // tp
    g = synth.generator(seed=403)
    shards = [synth.small_int_bf16((c, H), -2, 2, g) for _ in range(tp)]
    W = synth.small_int_bf16((H, N), -2, 2, g)          # K x N
    Wt = W.t().contiguous()                              # N x K, the same weights
    with ub.UserBuffer([8192, H], tp) as buf:
        buf.set_active_shape([T, H])
        sh = [s.to(dev()) for s in shards]
        Ykn = sentinel((T + 2, N))
        buf.ag_gemm_kn(sh, W.to(dev()), Ykn[:T])
        Yfb = sentinel((T + 2, N))
        buf.ag_gemm_from_buffer(Wt.to(dev()), Yfb[:T])   # the buffer holds the gather above
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    Xu = np.concatenate([synth.to_u16(s) for s in shards])
    rows = _rows(T, c)
    ref = _round_bf16(oracle.gemm_rows(Xu, synth.to_u16(Wt), rows))
    ridx = torch.as_tensor(rows, device=dev())
    np.testing.assert_array_equal(synth.to_u16(Ykn[ridx]), ref)
    np.testing.assert_array_equal(synth.to_u16(Yfb[ridx]), ref)
    assert is_sentinel(Ykn[T:]) and is_sentinel(Yfb[T:])

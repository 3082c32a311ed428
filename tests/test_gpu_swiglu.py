"""AG-GEMM with the fused SwiGLU epilogue (fc1 + activation of the MLP diagram) against
the oracle: gather, fp64 product, then silu(gate) * up."""
import math

import numpy as np
import pytest
import torch

import oracle
from gemm_overlap_gemms_gb300 import synth, ub
from gpu_helpers import assert_close, dev, is_sentinel, sentinel

pytestmark = pytest.mark.gpu


def oracle_swiglu_rows(shards, Wt, rows=None):
    G = np.concatenate([synth.to_u16(s) for s in shards])
    if rows is None:
        rows = np.arange(G.shape[0])
    return oracle.swiglu(oracle.gemm_rows(G, synth.to_u16(Wt), rows))


@pytest.mark.parametrize("tp,c,F,H,split", [(2, 192, 192, 256, -1), (4, 1, 128, 256, -1),
                                              (4, 129, 328, 256, -1), (4, 300, 256, 256, 1),
                                              (1, 77, 136, 256, 0), (4, 64, 1024, 256, -1),
                                              (4, 256, 512, 2048, 1), (2, 200, 200, 2048, 1)])
def test_swiglu_epilogue_matches_oracle(tp, c, F, H, split):
    """Whole tiles and split tail tiles (H = 2048 gives 32 k-blocks: two pieces)."""
    T = c * tp
    g = synth.generator(seed=41)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    Wt = synth.normal_bf16((2 * F, H), 1.0 / math.sqrt(H), g)
    with ub.UserBuffer([T + 4 * tp, H], tp) as buf:
        buf.set_option("streamk", split)
        buf.set_active_shape([T, H])
        Z = sentinel((T + 8, F))
        buf.ag_gemm_swiglu([s.to(dev()) for s in shards], Wt.to(dev()), Z)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
        G = buf.buffer()[:T].cpu()
    np.testing.assert_array_equal(synth.to_u16(G), np.concatenate([synth.to_u16(s) for s in shards]))
    assert_close(Z[:T], oracle_swiglu_rows(shards, Wt), "SwiGLU tp=%d c=%d F=%d" % (tp, c, F))
    assert is_sentinel(Z[T:]), "Z rows >= T touched"


@pytest.mark.parametrize("tp,c,F,H", [(4, 1, 128, 256), (4, 129, 328, 256), (2, 200, 200, 512),
                                      (1, 77, 136, 256), (4, 128, 3584, 1024)])
def test_swiglu_on_single_ctas_matches_oracle(tp, c, F, H):
    """The single-CTA kernel's SwiGLU epilogue (128 gate + 128 up rows per 256-column
    tile, chunk-aligned 128-row tiles), forced on."""
    T = c * tp
    g = synth.generator(seed=42)
    shards = [synth.normal_bf16((c, H), 1.0, g) for _ in range(tp)]
    Wt = synth.normal_bf16((2 * F, H), 1.0 / math.sqrt(H), g)
    with ub.UserBuffer([T + 4 * tp, H], tp) as buf:
        buf.set_option("cta_pair", 0)
        buf.set_option("skinny", 0)
        buf.set_active_shape([T, H])
        Z = sentinel((T + 8, F))
        buf.ag_gemm_swiglu([s.to(dev()) for s in shards], Wt.to(dev()), Z)
        torch.cuda.synchronize()
        assert buf.query_status() == ub.UB_OK
    rows = np.arange(T) if T * F <= 600000 else np.unique(
        np.concatenate([[0, c - 1, c, T - 1], np.random.default_rng(2).integers(0, T, 16)]))
    assert_close(Z[torch.as_tensor(rows, device=dev())], oracle_swiglu_rows(shards, Wt, rows),
                 "single-CTA SwiGLU tp=%d c=%d F=%d" % (tp, c, F))
    assert is_sentinel(Z[T:]), "Z rows >= T touched"


def test_swiglu_full_size_repeated_calls():
    """SwiGLU fc1 of the MLP workload (hidden 4096, F = 3584 per rank), three calls in a
    row on one handle with fresh inputs each time: later calls overlap their chunk copies
    with the GEMM (the first call of a process may not), so they are the ones that show
    whether the copies can run next to the GEMM."""
    w = synth.WORKLOADS["swiglu"]
    H, F, tp = w.hidden, w.ag_n[0] // 2, w.tp
    g = synth.generator(dev())
    Wt = synth.normal_bf16((2 * F, H), 1.0 / math.sqrt(H), g, dev())
    rng = np.random.default_rng(5)
    with ub.UserBuffer([w.max_tokens, H], tp) as buf:
        for T in (4640, 1024, 8192):
            X = synth.normal_bf16((T, H), 1.0, g, dev())
            c = T // tp
            shards = [X[r * c:(r + 1) * c] for r in range(tp)]
            buf.set_active_shape([T, H])
            Z = buf.ag_gemm_swiglu(shards, Wt)
            torch.cuda.synchronize()
            assert buf.query_status() == ub.UB_OK, "T=%d" % T
            rows = np.unique(np.concatenate([[0, c - 1, c, 2 * c + 5, T - 1], rng.integers(0, T, 24)]))
            ref = oracle.swiglu(oracle.gemm_rows(synth.to_u16(X), synth.to_u16(Wt), rows))
            assert_close(Z[torch.as_tensor(rows, device=dev())], ref, "SwiGLU T=%d" % T)

"""Seeded synthetic workloads: packed-sequence token counts and bf16 operands.

This module holds no arithmetic of the method: it only draws random inputs. The
tests, the benchmark and the oracle checks all take their inputs from here, so the
GPU path and the CPU oracle see identical bytes.

Workloads (packed THD microbatches; T is the total token count of one microbatch,
"Support dynamic token counts in TP communication/GEMM overlap", section "Problem"):

* ``tiny``   -- tp=2, hidden=256, capacity 512, T=384; AG: W ~ N(0, 1/256), N=384;
  RS: K=512 per shard, B ~ N(0, 1/512).
* ``qkv``    -- tp=4, hidden=4096, capacity 8192, N=3072 (= 3*hidden/tp, the QKV
  projection of the column-parallel diagram); 16 microbatches, each the sum of
  sequence lengths ~ U[128, 4096] drawn until the next would pass 8192, rounded
  down to a multiple of 4.
* ``swiglu`` -- tp=4, hidden=4096, ffn=14336; fc1 AG with N=7168 (= 2*ffn/tp),
  fc2 RS with K=3584 (= ffn/tp) per shard; T ~ U{1024..8192 step 4}; capacity 8192.
* ``large``  -- tp=8, hidden=8192, capacity 16384; RS with K=1024 (attention out)
  and K=3584 (fc2); lengths round(lognormal(ln 1024, 1.0)) clipped to [1, 8192]
  summed until the next would pass 16384, T rounded down to a multiple of 8.
* ``stress`` -- tp=4, hidden=4096, capacity 16384, 64 microbatches on one buffer;
  T from {4, 64, 512, 4092, 8192, 16384} with probability 1/2, else a uniform
  multiple of 4 in [4, 16384]; AG N=3072 and RS K=3584 each step.

Activations are ~ N(0, 1); weights ~ N(0, 1/fan_in). Values come from a seeded
``torch.Generator`` on the requested device (CPU for tests that feed the oracle,
CUDA for large benchmark tensors); token counts from ``numpy.random.default_rng``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

SEED = 0


@dataclass(frozen=True)
class Workload:
    name: str
    tp: int
    hidden: int
    max_tokens: int
    ag_n: tuple = ()          # AG-GEMM output widths (one per column-parallel layer)
    rs_k: tuple = ()          # GEMM-RS per-shard inner sizes (one per row-parallel layer)
    microbatches: int = 1
    notes: str = ""
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny": Workload("tiny", tp=2, hidden=256, max_tokens=512, ag_n=(384,), rs_k=(512,),
                     microbatches=1),
    "qkv": Workload("qkv", tp=4, hidden=4096, max_tokens=8192, ag_n=(3072,), rs_k=(),
                    microbatches=16),
    "swiglu": Workload("swiglu", tp=4, hidden=4096, max_tokens=8192, ag_n=(7168,),
                       rs_k=(3584,), microbatches=16, extra={"ffn": 14336}),
    "large": Workload("large", tp=8, hidden=8192, max_tokens=16384, ag_n=(),
                      rs_k=(1024, 3584), microbatches=16),
    "stress": Workload("stress", tp=4, hidden=4096, max_tokens=16384, ag_n=(3072,),
                       rs_k=(3584,), microbatches=64),
}


def _packed_total(rng: np.random.Generator, draw, cap: int) -> int:
    """Sum sequence lengths from ``draw`` until adding the next would pass ``cap``."""
    total = 0
    while True:
        n = int(draw(rng))
        if total + n > cap:
            return total
        total += n


def token_counts(name: str, seed: int = SEED) -> list[int]:
    """Active token count T of every microbatch of workload ``name``."""
    w = WORKLOADS[name]
    rng = np.random.default_rng(seed)
    out = []
    if name == "tiny":
        return [384]
    for _ in range(w.microbatches):
        if name == "qkv":
            t = _packed_total(rng, lambda g: g.integers(128, 4096, endpoint=True), 8192)
            t -= t % 4
        elif name == "swiglu":
            t = int(rng.integers(1024 // 4, 8192 // 4, endpoint=True)) * 4
        elif name == "large":
            def draw(g):
                v = int(round(float(g.lognormal(mean=math.log(1024.0), sigma=1.0))))
                return min(max(v, 1), 8192)
            t = _packed_total(rng, draw, 16384)
            t -= t % 8
        elif name == "stress":
            if rng.random() < 0.5:
                t = int(rng.choice([4, 64, 512, 4092, 8192, 16384]))
            else:
                t = int(rng.integers(1, 16384 // 4, endpoint=True)) * 4
        else:
            raise KeyError(name)
        out.append(max(t, w.tp))
    return out


def generator(device="cpu", seed: int = SEED) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """bf16 tensor with entries ~ N(0, std^2) (drawn in fp32, rounded to bf16)."""
    t = torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def small_int_bf16(shape, lo: int, hi: int, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """bf16 tensor of integers uniform in [lo, hi] (exact in bf16 for |v| <= 256)."""
    t = torch.randint(lo, hi + 1, tuple(shape), generator=gen, device=device,
                      dtype=torch.int32)
    return t.to(torch.bfloat16)


def ag_inputs(T: int, hidden: int, N: int, tp: int, gen: torch.Generator, device="cpu",
              W: torch.Tensor | None = None):
    """tp token shards X_r [T/tp, hidden] ~ N(0,1) and the column-parallel weight,
    stored out x in as Wt [N, hidden] ~ N(0, 1/hidden)."""
    assert T % tp == 0
    c = T // tp
    shards = [normal_bf16((c, hidden), 1.0, gen, device) for _ in range(tp)]
    if W is None:
        W = normal_bf16((N, hidden), 1.0 / math.sqrt(hidden), gen, device)
    return shards, W


def rs_inputs(T: int, K: int, hidden: int, tp: int, gen: torch.Generator, device="cpu",
              B: list | None = None):
    """tp partial-product operands A_j [T, K] ~ N(0,1) and the row-parallel shard
    weights, stored out x in as Bt_j [hidden, K] ~ N(0, 1/K)."""
    A = [normal_bf16((T, K), 1.0, gen, device) for _ in range(tp)]
    if B is None:
        B = [normal_bf16((hidden, K), 1.0 / math.sqrt(K), gen, device) for _ in range(tp)]
    return A, B


def to_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_u16(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

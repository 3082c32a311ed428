"""The seeded workload generators produce the token counts their recipes state."""
import torch

from gemm_overlap_gemms_gb300 import synth


def test_token_counts_follow_recipes():
    w = synth.WORKLOADS
    assert synth.token_counts("tiny") == [384]
    for name in ("qkv", "swiglu", "large", "stress"):
        ts = synth.token_counts(name)
        assert len(ts) == w[name].microbatches
        assert all(w[name].tp <= t <= w[name].max_tokens for t in ts)
        assert all(t % w[name].tp == 0 for t in ts)
        assert ts == synth.token_counts(name)          # seeded: reproducible
    assert all(t % 4 == 0 and t >= 8192 - 4096 - 3 for t in synth.token_counts("qkv"))
    assert all(1024 <= t <= 8192 for t in synth.token_counts("swiglu"))
    assert all(t % 8 == 0 for t in synth.token_counts("large"))
    st = synth.token_counts("stress")
    assert {4, 64, 512, 4092, 8192, 16384} & set(st)


def test_value_generators_are_seeded():
    a = synth.normal_bf16((64, 32), 0.5, synth.generator(seed=1))
    b = synth.normal_bf16((64, 32), 0.5, synth.generator(seed=1))
    assert a.dtype == torch.bfloat16 and torch.equal(a, b)
    assert 0.4 < a.float().std().item() < 0.6
    x = synth.small_int_bf16((1000,), -3, 3, synth.generator(seed=2))
    assert set(x.float().unique().tolist()) <= set(range(-3, 4))
    u = synth.to_u16(a)
    assert torch.equal(synth.from_u16(u), a)

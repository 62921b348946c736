"""The seeded input generators: shapes, dtypes, layouts and length mixes of
the workloads the tests and the benchmark use (no arithmetic of the method
lives here)."""
import torch

from ragged_gqa_attention_varlen_gb300 import workloads as W


def _lengths(p):
    lq, lk = p.lengths()
    return lq, lk


def test_named_workloads_follow_their_recipes():
    cases = {
        # name: (B, Hq, dtype, token step, feature pad)
        "q_short_k_long": (18, 48, torch.bfloat16, 2, 192),
        "k_short_q_long": (52, 96, torch.float16, 3, 176),
        "mixed_h64": (32, 64, torch.bfloat16, 2, 160),
        "mixed_h80": (32, 80, torch.bfloat16, 2, 160),
        "long_balanced": (24, 96, torch.bfloat16, 2, 160),
    }
    for name, (B, Hq, dtype, step, pad) in cases.items():
        p = W.WORKLOADS[name](length_scale=1 / 256)
        assert (p.B, p.Hq, p.q.dtype) == (B, Hq, dtype), name
        assert p.q.shape[1:] == (Hq, 160) and p.k.shape[1:] == (1, 160), name
        assert p.q.stride(0) == step * Hq * pad and p.q.stride(1) == pad, name
        assert p.alibi_slopes.shape == (B, Hq) and p.alibi_slopes.dtype == torch.float32
        assert int(p.cu_q[-1]) == p.q.shape[0] and int(p.cu_k[-1]) == p.k.shape[0]


def test_length_ranges():
    """Lengths drawn from each recipe's ranges (checked on 1/16-length
    replicas, whose lengths are the full draws scaled and rounded)."""
    s = 1 / 16
    rng = lambda xs, lo, hi: all(max(1, round(lo * s)) <= x <= round(hi * s) for x in xs)
    lq, lk = _lengths(W.q_short(length_scale=s))
    assert rng(lq, 16, 256) and rng(lk, 1024, 4096)
    lq, lk = _lengths(W.k_short(length_scale=s))
    assert rng(lq, 1024, 4096) and rng(lk, 32, 384)
    lq, lk = _lengths(W.long_balanced(length_scale=s))
    assert lq == lk and rng(lq, 6144, 12288)
    lq, lk = _lengths(W.mixed(length_scale=s))
    assert rng(lq + lk, 1, 8192)
    assert all(lq[b] == 1 for b in W.MIXED_LQ1) and all(lk[b] == 1 for b in W.MIXED_LK1)


def test_generators_are_seeded_and_padding_is_poisoned():
    a, b = W.tiny(seed=3), W.tiny(seed=3)
    for n in ("q", "k", "v", "dout"):
        assert torch.equal(getattr(a, n), getattr(b, n))
    assert not torch.equal(W.tiny(seed=4).q, a.q)
    p = W.custom([5, 3], [4, 6], 8, step=2, pad=192)
    raw = torch.empty(0, dtype=p.q.dtype).set_(p.q.untyped_storage())
    assert int(torch.isnan(raw).sum()) == raw.numel() - p.q.numel()
    assert not torch.isnan(p.q).any()


def test_options_shape_the_views():
    p = W.custom([7, 2], [9, 4], 12, Hkv=4, d=128)
    assert p.k.shape == (13, 4, 128) and p.q.shape == (9, 12, 128)
    p = W.long_balanced(length_scale=1 / 256, Hkv=8, d=64)
    assert p.k.shape[1:] == (8, 64) and p.q.shape[1:] == (96, 64)


def test_gated_family_follows_its_page():
    p = W.gated(length_scale=1 / 256, d=64, R=32, Hq=16, Hkv=4)
    assert p.q.shape[1:] == (16, 64) and p.k.shape[1:] == (4, 64)
    assert p.q_gate.shape == (p.q.shape[0], 16, 32) and p.k_gate.shape == (p.k.shape[0], 4, 32)
    assert p.causal and p.softcap == 0.0 and float(p.alibi_slopes.abs().max()) == 0.0
    lq, lk = p.lengths()
    assert lq == lk and all(4 <= x <= 64 for x in lq)

"""Pins for the fp64 CPU oracle: each test ties the oracle to something other
than its own formula -- a library routine, a closed form of a special case,
finite differences of its own forward, or an invariant of the mathematics.

The method follows "Noncausal Global Extreme-GQA Ragged Attention Full VJP"
(sections "Hard Constraints" and "What You Have") and, for empty rows and
recompute, "ragged flash attention gradient recompute" ("Root causes
addressed", "Verification").
"""
import math

import numpy as np
import pytest
import torch

from ragged_gqa_attention_varlen_gb300 import workloads as W

D = 160


def sigma(sm=0.75):
    return sm / math.sqrt(D)


def f32(x):
    """x rounded to fp32, the slopes' storage type."""
    return float(torch.tensor(x, dtype=torch.float32))


def f64_problem(lq, lk, Hq, seed=0, qk_std=1.0, slope_max=0.25, **mask):
    """Problem whose inputs are fp64 (used for exact special cases and FD)."""
    return W.custom(lq, lk, Hq, dtype=torch.float64, seed=seed, qk_std=qk_std,
                    slope_max=slope_max, **mask)


# ---------------------------------------------------------------- decoding

def test_decode_every_16bit_pattern(oracle_mod):
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    for dt in (torch.float16, torch.bfloat16):
        ref = bits.view(dt).double()
        got = torch.tensor([oracle_mod.decode(dt, int(b) & 0xFFFF) for b in range(65536)],
                           dtype=torch.float64)
        nan = torch.isnan(ref)
        assert torch.equal(torch.isnan(got), nan)
        assert torch.equal(got[~nan], ref[~nan])


# ------------------------------------------- library special case: plain SDPA

def _sdpa_reference(p, scale):
    """Per sequence: torch SDPA in fp64 with its own grouped-query head
    mapping (``enable_gqa``: Hq query heads over Hkv K/V heads), and autograd
    for the VJP (dk/dv sum over the heads of each group)."""
    outs, dqs, dks, dvs, lses = [], [], [], [], []
    Hkv = p.k.shape[1]
    for b in range(p.B):
        q0, q1 = int(p.cu_q[b]), int(p.cu_q[b + 1])
        k0, k1 = int(p.cu_k[b]), int(p.cu_k[b + 1])
        q = p.q[q0:q1].double().permute(1, 0, 2).clone().requires_grad_(True)  # [H, Lq, d]
        k = p.k[k0:k1].double().permute(1, 0, 2).clone().requires_grad_(True)  # [Hkv, Lk, d]
        v = p.v[k0:k1].double().permute(1, 0, 2).clone().requires_grad_(True)
        do = p.dout[q0:q1].double().permute(1, 0, 2)
        o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None],
                                                             scale=scale, enable_gqa=Hkv > 1)[0]
        gq, gk, gv = torch.autograd.grad(o, (q, k, v), do)
        # lse: the logits of each query head against the keys of its group
        kk = k.detach().repeat_interleave(p.Hq // Hkv, dim=0)
        lse = torch.logsumexp(scale * q.detach() @ kk.transpose(-1, -2), dim=-1)
        outs.append(o.detach().permute(1, 0, 2))
        dqs.append(gq.permute(1, 0, 2))
        dks.append(gk.permute(1, 0, 2))
        dvs.append(gv.permute(1, 0, 2))
        lses.append(lse.permute(1, 0))
    return (torch.cat(outs), torch.cat(lses), torch.cat(dqs), torch.cat(dks), torch.cat(dvs))


@pytest.mark.parametrize("softcap,Hkv,d", [(0.0, 1, 160), (1e7, 1, 160), (0.0, 2, 160),
                                           (0.0, 4, 160), (0.0, 1, 128), (0.0, 2, 64)])
def test_reduces_to_sdpa_without_cap_and_alibi(oracle_mod, softcap, Hkv, d):
    p = f64_problem([3, 7, 1, 12], [5, 2, 9, 12], Hq=4, seed=3, Hkv=Hkv, d=d)
    p.alibi_slopes.zero_()
    p.softcap = softcap
    r = oracle_mod.fvjp(p)
    out, lse, dq, dk, dv = _sdpa_reference(p, 0.75 / math.sqrt(d))
    tol = dict(rtol=1e-9, atol=1e-11)
    torch.testing.assert_close(r["out"], out, **tol)
    torch.testing.assert_close(r["lse"], lse, **tol)
    torch.testing.assert_close(r["dq"], dq, **tol)
    torch.testing.assert_close(r["dk"], dk, **tol)
    torch.testing.assert_close(r["dv"], dv, **tol)


def test_fp16_inputs_decode_like_torch_in_sdpa_case(oracle_mod):
    p = W.custom([6, 4], [3, 8], Hq=2, dtype=torch.float16, seed=5)
    p.alibi_slopes.zero_()
    p.softcap = 0.0
    r = oracle_mod.fvjp(p)
    out, lse, dq, dk, dv = _sdpa_reference(p, sigma())
    torch.testing.assert_close(r["out"], out, rtol=1e-10, atol=1e-12)
    torch.testing.assert_close(r["dk"], dk, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------- closed forms

def test_two_keys_softcap_then_alibi_closed_form(oracle_mod):
    """One query, two keys, q = a e0, k0 = e0, k1 = 0: s0 = sigma a, s1 = 0.
    The ALiBi distances are |0 + 2 - 1 - j| = (1, 0), so with the cap applied
    first, z0 = 3 tanh(sigma a / 3) - slope and z1 = 0, and the softmax over two
    keys is the logistic function of z0."""
    p = f64_problem([1], [2], Hq=1)
    a, slope = 60.0, 0.3
    p.q.zero_()
    p.q[0, 0, 0] = a
    p.k.zero_()
    p.k[0, 0, 0] = 1.0
    p.alibi_slopes.fill_(slope)
    r = oracle_mod.fvjp(p)
    z0 = 3.0 * math.tanh(sigma() * a / 3.0) - f32(slope)
    w0 = 1.0 / (1.0 + math.exp(-z0))
    expect = w0 * p.v[0, 0] + (1.0 - w0) * p.v[1, 0]
    torch.testing.assert_close(r["out"][0, 0], expect, rtol=1e-13, atol=1e-14)
    assert abs(float(r["lse"][0, 0]) - math.log(math.exp(z0) + 1.0)) < 1e-13
    # the cap is active: without it the weight would differ markedly
    z0_nocap = sigma() * a - f32(slope)
    assert abs(1.0 / (1.0 + math.exp(-z0_nocap)) - w0) > 0.05


# Distances |i + Lk - Lq - j| written out by hand for small shapes.
ALIBI_TABLES = {
    (2, 4): [[2, 1, 0, 1], [3, 2, 1, 0]],
    (4, 2): [[2, 3], [1, 2], [0, 1], [1, 0]],
    (3, 3): [[0, 1, 2], [1, 0, 1], [2, 1, 0]],
}


@pytest.mark.parametrize("shape", sorted(ALIBI_TABLES))
def test_alibi_distance_tables(oracle_mod, shape):
    """With q = 0 every logit is 0 (softcap of 0 is 0), so the weights are a
    softmax of -slope * distance alone."""
    Lq, Lk = shape
    p = f64_problem([Lq], [Lk], Hq=2, seed=1)
    p.q.zero_()
    p.alibi_slopes.copy_(torch.tensor([[0.7, 0.2]]))
    r = oracle_mod.fvjp(p)
    dist = np.array(ALIBI_TABLES[shape], dtype=np.float64)
    for h, slope in enumerate((0.7, 0.2)):
        w = np.exp(-f32(slope) * dist)
        lse = np.log(w.sum(1))
        w = w / w.sum(1, keepdims=True)
        expect = torch.from_numpy(w) @ p.v[:, 0]
        torch.testing.assert_close(r["out"][:, h], expect, rtol=1e-13, atol=1e-14)
        torch.testing.assert_close(r["lse"][:, h], torch.from_numpy(lse), rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("shape", sorted(ALIBI_TABLES))
def test_alibi_negative_slope_favours_far_keys(oracle_mod, shape):
    """A negative slope enters with its sign: with q = 0 the weights are
    exp(|slope| * distance) normalised, largest at the farthest key."""
    Lq, Lk = shape
    p = f64_problem([Lq], [Lk], Hq=2, seed=3)
    p.q.zero_()
    p.alibi_slopes.copy_(torch.tensor([[-0.7, -0.05]]))
    r = oracle_mod.fvjp(p)
    dist = np.array(ALIBI_TABLES[shape], dtype=np.float64)
    for h, slope in enumerate((-0.7, -0.05)):
        w = np.exp(-f32(slope) * dist)
        lse = np.log(w.sum(1))
        w = w / w.sum(1, keepdims=True)
        assert (w.argmax(1) == dist.argmax(1)).all()
        expect = torch.from_numpy(w) @ p.v[:, 0]
        torch.testing.assert_close(r["out"][:, h], expect, rtol=1e-13, atol=1e-14)
        torch.testing.assert_close(r["lse"][:, h], torch.from_numpy(lse), rtol=1e-13, atol=1e-14)


def test_alibi_equal_lengths_is_abs_i_minus_j(oracle_mod):
    """Equal lengths: Lq = Lk makes the distance |i - j|."""
    L = 7
    p = f64_problem([L], [L], Hq=1, seed=2)
    p.q.zero_()
    p.alibi_slopes.fill_(0.4)
    r = oracle_mod.fvjp(p)
    dist = np.abs(np.subtract.outer(np.arange(L), np.arange(L))).astype(np.float64)
    w = np.exp(-f32(0.4) * dist)
    w /= w.sum(1, keepdims=True)
    torch.testing.assert_close(r["out"][:, 0], torch.from_numpy(w) @ p.v[:, 0], rtol=1e-13,
                               atol=1e-14)


# Admissible key sets written out by hand (k0 = i + Lk - Lq).
MASK_CASES = [
    # (Lq, Lk, causal, wl, wr, sets per row)
    (3, 5, True, -1, -1, [{0, 1, 2}, {0, 1, 2, 3}, {0, 1, 2, 3, 4}]),
    (3, 5, False, 1, 1, [{1, 2, 3}, {2, 3, 4}, {3, 4}]),
    (3, 5, True, 1, -1, [{1, 2}, {2, 3}, {3, 4}]),
    (3, 5, True, 1, 4, [{1, 2}, {2, 3}, {3, 4}]),  # causal overrides the right window
    (5, 2, True, -1, -1, [set(), set(), set(), {0}, {0, 1}]),
    (4, 6, False, 0, -1, [{2, 3, 4, 5}, {3, 4, 5}, {4, 5}, {5}]),
]


@pytest.mark.parametrize("case", MASK_CASES)
def test_mask_admissible_sets(oracle_mod, case):
    """q = 0 and zero slopes give uniform weights over the admissible keys."""
    Lq, Lk, causal, wl, wr, sets = case
    p = f64_problem([Lq], [Lk], Hq=2, seed=4, causal=causal, window_left=wl, window_right=wr)
    p.q.zero_()
    p.alibi_slopes.zero_()
    r = oracle_mod.fvjp(p)
    for i, s in enumerate(sets):
        for h in range(2):
            if not s:
                assert float(r["lse"][i, h]) == -math.inf
                assert torch.equal(r["out"][i, h], torch.zeros(D, dtype=torch.float64))
                assert torch.equal(r["dq"][i, h], torch.zeros(D, dtype=torch.float64))
            else:
                expect = p.v[sorted(s), 0].mean(0)
                torch.testing.assert_close(r["out"][i, h], expect, rtol=1e-13, atol=1e-14)
                assert abs(float(r["lse"][i, h]) - math.log(len(s))) < 1e-13


def test_single_key(oracle_mod):
    """Lk = 1: out = v0, dq = dk = 0, dv0 = sum over heads and rows of dO."""
    p = f64_problem([4, 3], [1, 1], Hq=3, seed=6, qk_std=2.0)
    r = oracle_mod.fvjp(p)
    for b in range(2):
        q0, q1 = int(p.cu_q[b]), int(p.cu_q[b + 1])
        assert torch.equal(r["out"][q0:q1], p.v[b, 0].expand(q1 - q0, 3, D))
        torch.testing.assert_close(r["dv"][b, 0], p.dout[q0:q1].sum((0, 1)), rtol=1e-13,
                                   atol=1e-13)
    assert torch.all(r["dq"] == 0) and torch.all(r["dk"] == 0)


# -------------------------------------------------- finite differences (VJP)

def _loss(oracle_mod, p):
    r = oracle_mod.fvjp(p, nthreads=1)
    return float((r["out"] * p.dout.double()).sum())


@pytest.mark.parametrize("mask", [dict(), dict(causal=True), dict(window_left=1, window_right=2)])
def test_vjp_matches_central_differences(oracle_mod, mask):
    """d<dout, out>/dx by central differences of the oracle's own forward, with
    softcap and ALiBi active, against the analytic dq/dk/dv."""
    p = f64_problem([3, 5], [4, 2], Hq=3, seed=7, qk_std=3.0, slope_max=0.5, **mask)
    r = oracle_mod.fvjp(p)
    gen = torch.Generator().manual_seed(11)
    h = 1e-6
    for name, grad in (("q", r["dq"]), ("k", r["dk"]), ("v", r["dv"])):
        x = getattr(p, name)
        for _ in range(12):
            idx = tuple(int(torch.randint(0, n, (1,), generator=gen)) for n in x.shape)
            old = float(x[idx])
            x[idx] = old + h
            lp = _loss(oracle_mod, p)
            x[idx] = old - h
            lm = _loss(oracle_mod, p)
            x[idx] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - float(grad[idx])) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd,
                                                                          float(grad[idx]))


# ------------------------------------------------------------ invariants

def test_row_invariants_on_tiny(oracle_mod):
    p = W.tiny()
    r = oracle_mod.fvjp(p, diagnostics=True)
    torch.testing.assert_close(r["p_rowsum"], torch.ones_like(r["p_rowsum"]), rtol=0,
                               atol=1e-13)
    # the gradient at the softmax input sums to zero over each row
    assert float(r["dz_rowsum"].abs().max()) < 1e-12
    # D is the row dot product of dO with out
    torch.testing.assert_close(r["D"], (p.dout.double() * r["out"]).sum(-1), rtol=1e-12,
                               atol=1e-12)
    # dv summed over a sequence's keys equals dO summed over its rows and heads
    for b in range(p.B):
        q0, q1 = int(p.cu_q[b]), int(p.cu_q[b + 1])
        k0, k1 = int(p.cu_k[b]), int(p.cu_k[b + 1])
        torch.testing.assert_close(r["dv"][k0:k1].sum((0, 1)),
                                   p.dout[q0:q1].double().sum((0, 1)), rtol=1e-11, atol=1e-10)


def test_identical_heads_scale_dk(oracle_mod):
    """All query heads equal (and equal slopes): out per head equals the
    single-head out, and dk/dv are Hq times the single-head values."""
    one = f64_problem([6, 3], [5, 7], Hq=1, seed=9, qk_std=2.0)
    Hq = 5
    many = W.custom([6, 3], [5, 7], Hq=Hq, dtype=torch.float64, seed=9)
    many.q.copy_(one.q.expand(-1, Hq, -1))
    many.dout.copy_(one.dout.expand(-1, Hq, -1))
    many.k.copy_(one.k)
    many.v.copy_(one.v)
    many.alibi_slopes.copy_(one.alibi_slopes.expand(-1, Hq))
    r1, rm = oracle_mod.fvjp(one), oracle_mod.fvjp(many)
    for h in range(Hq):
        torch.testing.assert_close(rm["out"][:, h], r1["out"][:, 0], rtol=1e-14, atol=1e-15)
        torch.testing.assert_close(rm["dq"][:, h], r1["dq"][:, 0], rtol=1e-14, atol=1e-15)
    torch.testing.assert_close(rm["dk"], Hq * r1["dk"], rtol=1e-12, atol=1e-13)
    torch.testing.assert_close(rm["dv"], Hq * r1["dv"], rtol=1e-12, atol=1e-13)


def test_empty_rows_contribute_nothing(oracle_mod):
    """Causal with Lq > Lk leaves rows 0..2 empty: their lse is -inf, their
    out and dq are exactly 0, and removing their dO changes no gradient."""
    p = f64_problem([5], [2], Hq=2, seed=12, causal=True)
    r = oracle_mod.fvjp(p)
    assert torch.all(r["lse"][:3] == -math.inf)
    assert torch.all(r["out"][:3] == 0) and torch.all(r["dq"][:3] == 0)
    p2 = f64_problem([5], [2], Hq=2, seed=12, causal=True)
    p2.dout[:3] = 1e3
    r2 = oracle_mod.fvjp(p2)
    for name in ("dk", "dv"):
        assert torch.equal(r[name], r2[name])
    assert torch.equal(r["dq"][3:], r2["dq"][3:])


# ------------------------------------------------------------- structure

@pytest.mark.parametrize("Hq,Hkv", [(6, 3), (4, 4), (8, 2)])
def test_kv_head_groups_are_independent_problems(oracle_mod, Hq, Hkv):
    """With Hkv K/V heads, group g (query heads g*R .. g*R+R-1, R = Hq/Hkv,
    with K/V head g) gives bitwise the results of the one-K/V-head problem
    made of those heads alone: the head mapping, the per-group dk/dv sums
    and their order all match the pinned Hkv = 1 case."""
    R = Hq // Hkv
    lq, lk = [4, 9, 2], [7, 3, 11]
    p = W.custom(lq, lk, Hq, seed=21, Hkv=Hkv, causal=True, window_left=5)
    r = oracle_mod.fvjp(p)
    for g in range(Hkv):
        pg = W.custom(lq, lk, R, seed=21, causal=True, window_left=5)
        pg.q.copy_(p.q[:, g * R:(g + 1) * R])
        pg.dout.copy_(p.dout[:, g * R:(g + 1) * R])
        pg.k.copy_(p.k[:, g:g + 1])
        pg.v.copy_(p.v[:, g:g + 1])
        pg.alibi_slopes.copy_(p.alibi_slopes[:, g * R:(g + 1) * R])
        rg = oracle_mod.fvjp(pg)
        for name in ("out", "dq", "lse", "D"):
            assert torch.equal(r[name][:, g * R:(g + 1) * R], rg[name]), (name, g)
        for name in ("dk", "dv"):
            assert torch.equal(r[name][:, g:g + 1], rg[name]), (name, g)
    # the row-sampled path maps heads the same way
    tok, head = [0, 5, 13, 14], [Hq - 1, 0, R, Hq // 2]
    s = oracle_mod.rows(p, tok, head)
    for n, (t, h) in enumerate(zip(tok, head)):
        assert torch.equal(s["out"][n], r["out"][t, h])
        assert torch.equal(s["dq"][n], r["dq"][t, h])
        assert float(s["lse"][n]) == float(r["lse"][t, h])


def test_sequences_are_independent_and_permutable(oracle_mod):
    p = W.custom([4, 9, 2], [7, 3, 11], Hq=4, seed=13)
    r = oracle_mod.fvjp(p)
    # perturb sequence 1 only: other sequences stay bitwise identical
    p2 = W.custom([4, 9, 2], [7, 3, 11], Hq=4, seed=13)
    p2.q[4:13] = -p2.q[4:13]
    p2.k[7:10] = 2 * p2.k[7:10]
    r2 = oracle_mod.fvjp(p2)
    for name, sl in (("out", [slice(0, 4), slice(13, 15)]), ("dq", [slice(0, 4), slice(13, 15)]),
                     ("dk", [slice(0, 7), slice(10, 21)]), ("dv", [slice(0, 7), slice(10, 21)])):
        for s in sl:
            assert torch.equal(r[name][s], r2[name][s]), name
    # reversing the sequence order (slopes rows too) reverses the outputs
    order = [2, 1, 0]
    lq, lk = p.lengths()
    pr = W.custom([lq[b] for b in order], [lk[b] for b in order], Hq=4, seed=13)
    qs = [p.q[int(p.cu_q[b]):int(p.cu_q[b + 1])] for b in order]
    ks = [p.k[int(p.cu_k[b]):int(p.cu_k[b + 1])] for b in order]
    vs = [p.v[int(p.cu_k[b]):int(p.cu_k[b + 1])] for b in order]
    ds = [p.dout[int(p.cu_q[b]):int(p.cu_q[b + 1])] for b in order]
    pr.q.copy_(torch.cat(qs))
    pr.k.copy_(torch.cat(ks))
    pr.v.copy_(torch.cat(vs))
    pr.dout.copy_(torch.cat(ds))
    pr.alibi_slopes.copy_(p.alibi_slopes[order])
    rr = oracle_mod.fvjp(pr)
    for name, cu, cur in (("out", p.cu_q, pr.cu_q), ("dq", p.cu_q, pr.cu_q),
                          ("lse", p.cu_q, pr.cu_q), ("dk", p.cu_k, pr.cu_k),
                          ("dv", p.cu_k, pr.cu_k)):
        for nb, b in enumerate(order):
            a = r[name][int(cu[b]):int(cu[b + 1])]
            c = rr[name][int(cur[nb]):int(cur[nb + 1])]
            assert torch.equal(a, c), name


def test_thread_count_does_not_change_bits(oracle_mod):
    p = W.tiny()
    r1 = oracle_mod.fvjp(p, nthreads=1)
    r5 = oracle_mod.fvjp(p, nthreads=5)
    for name in ("out", "lse", "dq", "dk", "dv"):
        assert torch.equal(r1[name], r5[name])


def test_row_sampler_matches_full_pass(oracle_mod):
    p = W.custom([5, 17, 33], [40, 9, 64], Hq=8, dtype=torch.bfloat16, step=2, pad=192, seed=14)
    r = oracle_mod.fvjp(p)
    tok = torch.tensor([0, 4, 5, 21, 54, 30])
    head = torch.tensor([0, 7, 3, 1, 6, 2], dtype=torch.int32)
    s = oracle_mod.rows(p, tok, head)
    for n in range(len(tok)):
        t, h = int(tok[n]), int(head[n])
        assert torch.equal(s["out"][n], r["out"][t, h])
        assert torch.equal(s["dq"][n], r["dq"][t, h])
        assert float(s["lse"][n]) == float(r["lse"][t, h])


@pytest.mark.parametrize("mask", [dict(), dict(causal=True), dict(window_left=3, window_right=1)])
def test_key_sampler_matches_full_pass(oracle_mod, mask):
    """The key sampler's dk/dv rows are the full pass's, bit for bit (it runs
    the same row arithmetic without dq, then the same key pass), with several
    K/V heads and empty sequences among the sampled ones."""
    p = W.custom([5, 0, 9, 4], [7, 3, 12, 1], 8, seed=5, Hkv=2, **mask)
    ref = oracle_mod.fvjp(p)
    tok = torch.tensor([0, 6, 7, 9, 11, 21, 10, 22])
    head = torch.tensor([0, 1, 1, 0, 1, 0, 0, 1], dtype=torch.int32)
    r = oracle_mod.keys(p, tok, head)
    for n in ("dk", "dv"):
        assert torch.equal(r[n], ref[n][tok, head.long()]), n


def test_strided_poisoned_views_match_dense(oracle_mod):
    """Padding and skipped token rows hold NaN; the oracle never reads them."""
    p = W.custom([5, 3], [6, 4], Hq=3, dtype=torch.float16, step=3, pad=176, seed=15)
    r = oracle_mod.fvjp(p)
    dense = W.custom([5, 3], [6, 4], Hq=3, dtype=torch.float16, step=1, pad=160, seed=15)
    for name in ("q", "k", "v", "dout"):
        getattr(dense, name).copy_(getattr(p, name))
    rd = oracle_mod.fvjp(dense)
    for name in ("out", "lse", "dq", "dk", "dv"):
        assert torch.equal(r[name], rd[name])
    assert all(torch.isfinite(r[n]).all() for n in ("out", "dq", "dk", "dv"))


@pytest.mark.parametrize("softcap,std", [(3.0, 1e3), (0.0, 60.0)])
def test_extreme_logits_stay_finite(oracle_mod, softcap, std):
    p = f64_problem([6, 4], [5, 9], Hq=2, seed=16, qk_std=std)
    p.softcap = softcap
    r = oracle_mod.fvjp(p, diagnostics=True)
    for n in ("out", "lse", "dq", "dk", "dv"):
        assert torch.isfinite(r[n]).all(), n
    torch.testing.assert_close(r["p_rowsum"], torch.ones_like(r["p_rowsum"]), rtol=0, atol=1e-12)


# ------------------------------------------------------------------ dropout

def test_splitmix64_matches_the_generators_first_outputs(oracle_mod):
    """SplitMix64 started from state 0 produces 0xE220A8397B1DCDAF,
    0x6E789E6AA1B965F4, 0x06C45D188009454F: its output function of the state
    after one, two and three Weyl increments (the function adds the
    increment itself, so it is applied to 0, phi and 2 phi)."""
    phi = 0x9E3779B97F4A7C15
    got = [oracle_mod.splitmix64((n * phi) & 0xFFFFFFFFFFFFFFFF) for n in range(3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_dropout_factors_are_zero_or_the_scale_at_the_rate(oracle_mod):
    rate = 0.3
    f = torch.tensor([oracle_mod.drop_factor(1234, rate, b, h, i, j)
                      for b in range(2) for h in range(3) for i in range(40) for j in range(50)],
                     dtype=torch.float64)
    scale = 1.0 / (1.0 - float(torch.tensor(rate, dtype=torch.float32)))
    assert torch.all((f == 0) | (f == scale))
    n, kept = f.numel(), int((f > 0).sum())
    p_keep = 1.0 - int(rate * 2 ** 16) / 2 ** 16
    assert abs(kept - n * p_keep) < 5 * math.sqrt(n * p_keep * (1 - p_keep))
    # rate 0 keeps everything at scale 1; rate 1 drops everything
    assert oracle_mod.drop_factor(7, 0.0, 0, 0, 3, 4) == 1.0
    assert oracle_mod.drop_factor(7, 1.0, 0, 0, 3, 4) == 0.0
    # the factor depends on (seed, b, h, i, j) alone
    assert oracle_mod.drop_factor(5, rate, 1, 2, 3, 4) == oracle_mod.drop_factor(5, rate, 1, 2, 3, 4)
    assert len({oracle_mod.drop_factor(s, 0.5, 0, 0, 0, 0) for s in range(64)}) == 2


def test_dropout_keys_sharing_a_hash_are_independent_draws(oracle_mod):
    """The four keys of one hash (j = 4m .. 4m + 3) take separate 16-bit
    fields: each position keeps at the rate, and two keys of one hash are kept
    together at the product rate (a field used twice would make them equal)."""
    rate = 0.5
    keep = torch.tensor([[oracle_mod.drop_factor(99, rate, 0, h, i, j) > 0 for j in range(64)]
                         for h in range(4) for i in range(64)], dtype=torch.float64)
    n = keep.shape[0] * 16
    for pos in range(4):
        k = int(keep[:, pos::4].sum())
        assert abs(k - n * 0.5) < 5 * math.sqrt(n * 0.25), pos
    for a, b in ((0, 1), (0, 3), (1, 2), (2, 3)):  # inside one hash
        both = int((keep[:, a::4] * keep[:, b::4]).sum())
        assert abs(both - n * 0.25) < 5 * math.sqrt(n * 0.25 * 0.75), (a, b)
    both = int((keep[:, 3::4][:, :-1] * keep[:, 4::4]).sum())  # across two hashes
    m = keep.shape[0] * 15
    assert abs(both - m * 0.25) < 5 * math.sqrt(m * 0.25 * 0.75)


def test_dropout_rate_zero_is_no_dropout(oracle_mod):
    p = f64_problem([7, 3], [5, 9], Hq=4, seed=2, causal=True)
    r0 = oracle_mod.fvjp(p)
    p.dropout_seed, p.dropout_rate = 99, 0.0
    r1 = oracle_mod.fvjp(p)
    for n in ("out", "lse", "dq", "dk", "dv"):
        assert torch.equal(r0[n], r1[n]), n


def _dropout_reference(oracle_mod, p):
    """torch fp64 autograd of the definition with an explicit keep mask built
    from the oracle's per-element factors: z = softcap(sigma q.k) - ALiBi,
    P = softmax(z), out = (P * M) v, grads of <dout, out>."""
    outs, dqs, dks, dvs = [], [], [], []
    sm = p.scale_multiplier / math.sqrt(p.q.shape[-1])
    for b in range(p.B):
        q0, q1 = int(p.cu_q[b]), int(p.cu_q[b + 1])
        k0, k1 = int(p.cu_k[b]), int(p.cu_k[b + 1])
        Lq, Lk = q1 - q0, k1 - k0
        q = p.q[q0:q1].double().permute(1, 0, 2).clone().requires_grad_(True)
        k = p.k[k0:k1, 0].double().clone().requires_grad_(True)
        v = p.v[k0:k1, 0].double().clone().requires_grad_(True)
        do = p.dout[q0:q1].double().permute(1, 0, 2)
        s = sm * q @ k.T
        t = p.softcap * torch.tanh(s / p.softcap)
        i = torch.arange(Lq, dtype=torch.float64)[:, None]
        j = torch.arange(Lk, dtype=torch.float64)[None, :]
        dist = (i + Lk - Lq - j).abs()
        z = t - p.alibi_slopes[b].double()[:, None, None] * dist
        P = torch.softmax(z, dim=-1)
        M = torch.tensor([[[oracle_mod.drop_factor(p.dropout_seed, p.dropout_rate, b, h, ii, jj)
                            for jj in range(Lk)] for ii in range(Lq)] for h in range(p.Hq)],
                         dtype=torch.float64)
        o = (P * M) @ v
        gq, gk, gv = torch.autograd.grad(o, (q, k, v), do)
        outs.append(o.detach().permute(1, 0, 2))
        dqs.append(gq.permute(1, 0, 2))
        dks.append(gk[:, None])
        dvs.append(gv[:, None])
    return torch.cat(outs), torch.cat(dqs), torch.cat(dks), torch.cat(dvs)


def test_dropout_forward_and_vjp_match_autograd_of_the_definition(oracle_mod):
    p = f64_problem([6, 9], [8, 5], Hq=3, seed=4, qk_std=2.0)
    p.dropout_seed, p.dropout_rate = 2024, 0.25
    r = oracle_mod.fvjp(p, diagnostics=True)
    out, dq, dk, dv = _dropout_reference(oracle_mod, p)
    tol = dict(rtol=1e-10, atol=1e-12)
    torch.testing.assert_close(r["out"], out, **tol)
    torch.testing.assert_close(r["dq"], dq, **tol)
    torch.testing.assert_close(r["dk"], dk, **tol)
    torch.testing.assert_close(r["dv"], dv, **tol)
    # lse stays the undropped one, and the softmax-input gradient still sums to 0
    p.dropout_seed = None
    r0 = oracle_mod.fvjp(p)
    assert torch.equal(r["lse"], r0["lse"])
    assert float(r["dz_rowsum"].abs().max()) < 1e-12


def test_dropout_per_token_rates(oracle_mod):
    """A per-token rate of 0 leaves that token's rows exactly as without
    dropout; the others follow their own rate."""
    p = f64_problem([6, 5], [7, 4], Hq=2, seed=8)
    base = oracle_mod.fvjp(p)
    rates = torch.zeros(11, dtype=torch.float32)
    rates[[1, 4, 7]] = 0.5
    p.dropout_seed, p.dropout_rates = 77, rates
    r = oracle_mod.fvjp(p)
    for t in range(11):
        same = torch.equal(r["out"][t], base["out"][t]) and torch.equal(r["dq"][t], base["dq"][t])
        assert same == (float(rates[t]) == 0.0) or float(rates[t]) > 0, t
    assert not torch.equal(r["dk"], base["dk"])
    # equal to a scalar rate where every token has that rate
    p2 = f64_problem([6, 5], [7, 4], Hq=2, seed=8)
    p2.dropout_seed, p2.dropout_rate = 77, 0.5
    p.dropout_rates = torch.full((11,), 0.5, dtype=torch.float32)
    ra, rb = oracle_mod.fvjp(p), oracle_mod.fvjp(p2)
    for n in ("out", "dq", "dk", "dv"):
        assert torch.equal(ra[n], rb[n]), n


# ------------------------------------------------------- gated variant (f4)

import oracle as _oracle  # noqa: E402  (the helper below needs its keep factors)


def _gated_problem(lq, lk, Hq, Hkv, R, seed, **mask):
    p = f64_problem(lq, lk, Hq=Hq, seed=seed, qk_std=1.5, Hkv=Hkv, **mask)
    g = torch.Generator().manual_seed(seed + 100)
    p.q_gate = torch.randn((sum(lq), Hq, R), generator=g, dtype=torch.float64)
    p.k_gate = torch.randn((sum(lk), Hkv, R), generator=g, dtype=torch.float64)
    return p


def _gated_reference(p):
    """torch fp64 autograd of the gated definition: out = (softmax(z) * G) v
    with z = softcap(sigma q.k) - ALiBi (masked), G = sigmoid(qg.kg / sqrt(R)),
    K/V and gate-key heads shared by consecutive query heads."""
    Hkv, R = p.k.shape[1], p.q_gate.shape[-1]
    rep = p.Hq // Hkv
    sm = p.scale_multiplier / math.sqrt(p.q.shape[-1])
    res = {n: [] for n in ("out", "dq", "dk", "dv", "dq_gate", "dk_gate")}
    for b in range(p.B):
        q0, q1 = int(p.cu_q[b]), int(p.cu_q[b + 1])
        k0, k1 = int(p.cu_k[b]), int(p.cu_k[b + 1])
        Lq, Lk = q1 - q0, k1 - k0
        q = p.q[q0:q1].permute(1, 0, 2).clone().requires_grad_(True)
        k = p.k[k0:k1].permute(1, 0, 2).clone().requires_grad_(True)
        v = p.v[k0:k1].permute(1, 0, 2).clone().requires_grad_(True)
        qg = p.q_gate[q0:q1].permute(1, 0, 2).clone().requires_grad_(True)
        kg = p.k_gate[k0:k1].permute(1, 0, 2).clone().requires_grad_(True)
        do = p.dout[q0:q1].permute(1, 0, 2)
        kk, vv, kkg = (x.repeat_interleave(rep, dim=0) for x in (k, v, kg))
        t = p.softcap * torch.tanh(sm * q @ kk.transpose(1, 2) / p.softcap)
        i = torch.arange(Lq, dtype=torch.float64)[:, None]
        j = torch.arange(Lk, dtype=torch.float64)[None, :]
        z = t - p.alibi_slopes[b][:, None, None] * (i + Lk - Lq - j).abs()
        k0_ = i + Lk - Lq
        ok = torch.ones(Lq, Lk, dtype=torch.bool)
        wr = 0 if p.causal else p.window_right
        if p.window_left >= 0:
            ok &= j >= k0_ - p.window_left
        if wr >= 0:
            ok &= j <= k0_ + wr
        z = z.masked_fill(~ok, -math.inf)
        P = torch.softmax(z, dim=-1).nan_to_num(0.0)
        G = torch.sigmoid(qg @ kkg.transpose(1, 2) / math.sqrt(R))
        if p.dropout_seed is not None:  # the oracle's own keep factors, as an explicit mask
            G = G * torch.tensor(
                [[[_oracle.drop_factor(p.dropout_seed, p.dropout_rate, b, h, ii, jj)
                   for jj in range(Lk)] for ii in range(Lq)] for h in range(p.Hq)],
                dtype=torch.float64)
        o = (P * G) @ vv
        grads = torch.autograd.grad(o, (q, k, v, qg, kg), do)
        res["out"].append(o.detach().permute(1, 0, 2))
        for n, gr in zip(("dq", "dk", "dv", "dq_gate", "dk_gate"), grads):
            res[n].append(gr.permute(1, 0, 2))
    return {n: torch.cat(x) for n, x in res.items()}


@pytest.mark.parametrize("Hq,Hkv,R,mask", [(4, 1, 8, dict()), (6, 2, 4, dict(causal=True)),
                                           (4, 4, 16, dict(window_left=2, window_right=1))])
def test_gated_forward_and_five_gradients_match_autograd(oracle_mod, Hq, Hkv, R, mask):
    p = _gated_problem([5, 8, 1], [6, 3, 4], Hq, Hkv, R, seed=31, **mask)
    r = oracle_mod.fvjp(p, diagnostics=True)
    ref = _gated_reference(p)
    tol = dict(rtol=1e-10, atol=1e-12)
    for n in ("out", "dq", "dk", "dv", "dq_gate", "dk_gate"):
        torch.testing.assert_close(r[n], ref[n], **tol, msg=n)
    # the softmax-input gradient still sums to zero over each row
    assert float(r["dz_rowsum"].abs().max()) < 1e-12


def test_gate_with_dropout_matches_autograd(oracle_mod):
    """Gate and dropout compose: out = (P * G * keep * scale) v."""
    p = _gated_problem([6, 4], [5, 7], 4, 2, 8, seed=17, causal=True)
    p.dropout_seed, p.dropout_rate = 99, 0.3
    r = oracle_mod.fvjp(p)
    ref = _gated_reference(p)
    for n in ("out", "dq", "dk", "dv", "dq_gate", "dk_gate"):
        torch.testing.assert_close(r[n], ref[n], rtol=1e-10, atol=1e-12, msg=n)


def test_constant_gate_halves_the_ungated_results(oracle_mod):
    """qg = 0 makes every gate sigmoid(0) = 1/2: out and dq, dk, dv are half
    the ungated ones, and nothing reaches the gate keys."""
    p = _gated_problem([4, 6], [5, 3], 4, 2, 8, seed=5)
    p.q_gate.zero_()
    r = oracle_mod.fvjp(p)
    p0 = _gated_problem([4, 6], [5, 3], 4, 2, 8, seed=5)
    p0.q_gate = p0.k_gate = None
    r0 = oracle_mod.fvjp(p0)
    for n in ("out", "dq", "dk", "dv"):
        torch.testing.assert_close(r[n], 0.5 * r0[n], rtol=1e-13, atol=1e-15, msg=n)
    assert torch.equal(r["dk_gate"], torch.zeros_like(r["dk_gate"]))
    assert torch.equal(r["lse"], r0["lse"])


def test_gated_bf16_inputs_decode_like_torch(oracle_mod):
    """16-bit gate projections are decoded exactly: the oracle on a bf16 gated
    problem equals the oracle on its fp64 copy."""
    p = W.gated(length_scale=1 / 1024, d=64, R=32, Hq=4, Hkv=2)
    r = oracle_mod.fvjp(p)
    p64 = W.gated(length_scale=1 / 1024, d=64, R=32, Hq=4, Hkv=2)
    for n in ("q", "k", "v", "dout", "q_gate", "k_gate"):
        setattr(p64, n, getattr(p, n).double())
    r64 = oracle_mod.fvjp(p64)
    for n in ("out", "lse", "dq", "dk", "dv", "dq_gate", "dk_gate"):
        assert torch.equal(r[n], r64[n]), n
        assert torch.isfinite(r[n]).all(), n

"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerances: relative Frobenius <= 1e-2 (fp16) / 2e-2 (bf16) and max-abs <=
5e-2 max|ref| on out/dq/dk/dv; lse within 1e-3 absolute, -inf rows exact.
Repeated calls must be bitwise identical; inputs must not change.
"""
import math

import pytest
import torch

from helpers import check_all, check_lse, check_tensor, nan_like_strided, row_mask, view_bytes_hash
from ragged_gqa_attention_varlen_gb300 import binding as BND
from ragged_gqa_attention_varlen_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from ragged_gqa_attention_varlen_gb300 import _build

    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return BND.load()


def run(p, **kw):
    r = BND.attention_varlen_fvjp(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout,
                                  p.causal, p.window_left, p.window_right, p.softcap,
                                  p.scale_multiplier, **kw)
    torch.cuda.synchronize()
    st = BND.device_status(r["workspace"])
    assert st == 0, f"device status {st:#x}"
    return r


def bits_equal(a, b):
    it = torch.int16 if a.element_size() == 2 else torch.int32
    return bool((a.contiguous().view(it) == b.contiguous().view(it)).all())


def parity(p_cpu, oracle_mod, seq_sel=None):
    p = p_cpu.to("cuda")
    res = run(p)
    ref = oracle_mod.fvjp(p_cpu, seq_sel=seq_sel)
    if seq_sel is None:
        return check_all(res, ref, p_cpu.dtype), res
    mq, mk = row_mask(p_cpu, seq_sel)
    return check_all(res, ref, p_cpu.dtype, rows=mq, keys=mk), res


# ---------------------------------------------------------------- tiny config

TINY_MASKS = [dict(), dict(causal=True), dict(window_left=16, window_right=16),
              dict(causal=True, window_left=16, window_right=16)]


@pytest.mark.parametrize("mask", TINY_MASKS, ids=["global", "causal", "win16", "causal_win16"])
def test_tiny_parity(oracle_mod, mask):
    parity(W.tiny(**mask), oracle_mod)


def test_tiny_bitwise_repeat_and_inputs_unchanged():
    p = W.tiny().to("cuda")
    hashes = [view_bytes_hash(getattr(p, n)) for n in ("q", "k", "v", "dout")]
    r1 = run(p)
    snap = {n: r1[n].clone() for n in ("out", "dq", "dk", "dv", "lse")}
    r2 = run(p)
    for n, x in snap.items():
        assert bits_equal(x, r2[n]), n
    assert hashes == [view_bytes_hash(getattr(p, n)) for n in ("q", "k", "v", "dout")]


@pytest.mark.slow
def test_repeated_calls_bitwise_identical():
    """Eight back-to-back calls on the long balanced workload at half length
    give identical bits in every output.  A missed dependency between the
    tile loads, the two MMA-issuing threads and the elementwise warps shows
    up here as an occasional difference in a few rows of one tile."""
    p = W.long_balanced(device="cuda", length_scale=0.5, poison=False)
    r1 = run(p)
    snap = {n: r1[n].clone() for n in ("out", "dq", "dk", "dv", "lse")}
    del r1
    for _ in range(7):
        r = run(p)
        for n, x in snap.items():
            assert bits_equal(x, r[n]), n
        del r


def test_strided_outputs_written_exactly_and_match_dense():
    """Outputs given as NaN-filled padded views: every valid element is written,
    padding stays NaN, values equal the dense-output call bit for bit."""
    p = W.q_short(length_scale=0.125).to("cuda")
    dense = run(p)
    outs = dict(out=nan_like_strided(p.q), dq=nan_like_strided(p.dout), dk=nan_like_strided(p.k),
                dv=nan_like_strided(p.v))
    strided = run(p, **outs)
    for n in ("out", "dq", "dk", "dv"):
        assert torch.equal(strided[n].contiguous(), dense[n]), n
        base = strided[n].untyped_storage()
        raw = torch.empty(0, dtype=strided[n].dtype, device="cuda").set_(base)
        n_nan = int(torch.isnan(raw).sum())
        assert n_nan == raw.numel() - strided[n].numel(), n


# ------------------------------------------------- scaled replicas (full oracle)

REPLICAS = [
    ("q_short_k_long", dict(length_scale=0.25), None),
    ("k_short_q_long", dict(length_scale=0.125), None),
    ("mixed_h64", dict(length_scale=1 / 16), None),
    ("mixed_h80", dict(length_scale=1 / 16), None),
    ("long_balanced", dict(length_scale=1 / 32), [0, 7, 13, 23]),
]


@pytest.mark.parametrize("name,kw,sel", REPLICAS, ids=[r[0] for r in REPLICAS])
def test_replica_parity(oracle_mod, name, kw, sel):
    p = W.WORKLOADS[name](**kw)
    parity(p, oracle_mod, seq_sel=sel)


# ----------------------------------------------------------------- edge cases

EDGE = [
    dict(lq=[0, 5, 3, 0, 9], lk=[4, 0, 6, 0, 130], Hq=16),          # empty sequences
    dict(lq=[1], lk=[1], Hq=48),                                     # single token each
    dict(lq=[1000], lk=[1000], Hq=16, dtype=torch.bfloat16),         # many tiles, ragged tail
    dict(lq=[16, 8], lk=[128, 256], Hq=16),                          # exact tile multiples
    dict(lq=[7, 33, 2], lk=[300, 5, 129], Hq=1),                     # one head (G = 1)
    dict(lq=[7, 33, 2], lk=[300, 5, 129], Hq=3),                     # odd head count
    dict(lq=[17, 9], lk=[150, 70], Hq=80, dtype=torch.bfloat16, step=2, pad=192),
    dict(lq=[40, 3], lk=[20, 200], Hq=16, causal=True),              # empty rows (Lq > Lk)
    dict(lq=[40, 300], lk=[200, 140], Hq=16, window_left=5, window_right=60),
    dict(lq=[40, 300], lk=[200, 140], Hq=16, causal=True, window_left=70),
    dict(lq=[30, 12], lk=[200, 40], Hq=16, qk_std=100.0),           # saturated softcap
    dict(lq=[0, 5], lk=[7, 0], Hq=16),            # no dk/dv tile at all, keys still zeroed
    dict(lq=[0, 5, 0], lk=[7, 0, 300], Hq=16, Hkv=4, d=128),
]


@pytest.mark.parametrize("case", EDGE, ids=[f"edge{i}" for i in range(len(EDGE))])
def test_edge_parity(oracle_mod, case):
    case = dict(case)
    lq, lk, Hq = case.pop("lq"), case.pop("lk"), case.pop("Hq")
    p = W.custom(lq, lk, Hq, **case)
    parity(p, oracle_mod)


# ------------------------------------------------ masks over many tiles
# Tiles that no admissible (query, key) pair reaches are skipped; the cases
# below span many 128-key tiles and query blocks so that skipped, partly cut
# and fully admissible tiles all occur, in every mask shape.

MASKED = [
    dict(lq=[1000, 260, 700], lk=[1000, 900, 300], Hq=16, causal=True),
    dict(lq=[900, 500], lk=[1100, 500], Hq=16, window_left=150, window_right=40,
         dtype=torch.bfloat16),
    dict(lq=[800, 90], lk=[800, 600], Hq=16, window_left=200),    # left bound only
    dict(lq=[600, 64], lk=[900, 700], Hq=16, window_right=100),   # right bound only
    dict(lq=[700], lk=[700], Hq=32, causal=True, window_left=256, dtype=torch.bfloat16, step=2),
    dict(lq=[513, 40], lk=[129, 300], Hq=16, window_left=0, window_right=0),  # one diagonal
    dict(lq=[400, 150], lk=[350, 600], Hq=16, causal=True, softcap=0.0),      # running max
    dict(lq=[300], lk=[300], Hq=8, causal=True, softcap=30.0),                # wide softcap
]


# Key tiles that no query may attend to are left out of the dk/dv schedule
# (their rows are zeroed up front): runs of such tiles, drawn back to back by
# one CTA, once stalled the lookahead of the column-scalar warp.
MASKED += [
    dict(lq=[90, 40], lk=[2000, 1500], Hq=16, window_left=200),          # 13 + 11 empty tiles
    dict(lq=[0, 300, 0, 64], lk=[900, 400, 700, 1300], Hq=16, causal=True),
    dict(lq=[0, 0, 37], lk=[1000, 600, 40], Hq=16),                      # empty query sets
]


@pytest.mark.parametrize("case", MASKED, ids=[f"masked{i}" for i in range(len(MASKED))])
def test_masked_parity(oracle_mod, case):
    case = dict(case)
    lq, lk, Hq = case.pop("lq"), case.pop("lk"), case.pop("Hq")
    softcap = case.pop("softcap", None)
    p = W.custom(lq, lk, Hq, **case)
    if softcap is not None:
        p.softcap = softcap
    parity(p, oracle_mod)


# ------------------------------------------------ negative ALiBi slopes
# A negative slope makes the ALiBi term grow with the distance: the forward's
# fixed softmax reference then sits at the row's farthest admissible key, and
# dk/dv's per-key bias of a tile that straddles a column's aligned key takes
# the slope's sign from the staged scalars.  Slopes here are drawn in
# U(-0.25, 0.25) per (sequence, head), both signs in every sequence.

NEG_SLOPES = [
    dict(lq=[300, 129, 40], lk=[257, 400, 170], Hq=8),
    dict(lq=[260, 90], lk=[300, 600], Hq=16, dtype=torch.bfloat16, causal=True),
    dict(lq=[200, 300], lk=[350, 300], Hq=16, window_left=100, window_right=30),
    dict(lq=[150, 64], lk=[400, 200], Hq=16, softcap=0.0),             # running max path
    dict(lq=[130, 70], lk=[260, 500], Hq=16, Hkv=2, d=128, dtype=torch.bfloat16),
]


@pytest.mark.parametrize("case", NEG_SLOPES, ids=[f"neg{i}" for i in range(len(NEG_SLOPES))])
def test_negative_slope_parity(oracle_mod, case):
    case = dict(case)
    lq, lk, Hq = case.pop("lq"), case.pop("lk"), case.pop("Hq")
    softcap = case.pop("softcap", None)
    p = W.custom(lq, lk, Hq, slope_max=0.5, **case)
    p.alibi_slopes = p.alibi_slopes - 0.25
    assert (p.alibi_slopes < 0).any() and (p.alibi_slopes > 0).any()
    if softcap is not None:
        p.softcap = softcap
    parity(p, oracle_mod)


# ------------------------------------------------ dk/dv's diagonal band
# A dk/dv key tile walks the query steps whose columns' aligned keys fall
# inside the tile (the band) after all others, and without a mask the steps
# outside the band take the one-sided bias form only.  Steep slopes make a
# wrong bias form visible; the lengths put the band at the tile's start, end
# and middle, with Lq != Lk (the aligned key shifted) and token blocks of 8,
# 16, 32, 64 and 128 tokens (query heads per K/V head 16, 8, 4, 2 and 3).

BAND = [
    dict(lq=[300, 129, 40], lk=[300, 129, 40], Hq=16),
    dict(lq=[250, 70], lk=[400, 64], Hq=8, dtype=torch.bfloat16),
    dict(lq=[500, 33], lk=[260, 300], Hq=8, Hkv=2),
    dict(lq=[190, 257], lk=[450, 127], Hq=4, Hkv=2, d=128),
    dict(lq=[333, 128], lk=[333, 200], Hq=6, Hkv=2, dtype=torch.bfloat16, d=64),
]


@pytest.mark.parametrize("case", BAND, ids=[f"band{i}" for i in range(len(BAND))])
def test_dkdv_band_parity(oracle_mod, case):
    case = dict(case)
    lq, lk, Hq = case.pop("lq"), case.pop("lk"), case.pop("Hq")
    p = W.custom(lq, lk, Hq, slope_max=0.8, **case)
    parity(p, oracle_mod)


def test_window_wider_than_every_sequence_is_bitwise_unmasked():
    """A two-sided window that admits every pair takes the unmasked code path
    on every tile, so the result is bitwise the unmasked call's."""
    p = W.custom([300, 5, 129], [260, 400, 1], 16, dtype=torch.bfloat16).to("cuda")
    ref = run(p)
    ref = {n: ref[n].clone() for n in ("out", "lse", "dq", "dk", "dv")}
    p.window_left = p.window_right = 10 ** 9
    wide = run(p)
    for n, x in ref.items():
        assert bits_equal(x, wide[n]), n


# ------------------------------------------------ several K/V heads
# Query heads g*R .. g*R+R-1 (R = Hq/Hkv) read K/V head g; each group runs
# as its own one-K/V-head problem.

GQA = [
    dict(lq=[300, 37, 1, 129], lk=[260, 400, 9, 0], Hq=16, Hkv=2),
    dict(lq=[200, 64], lk=[333, 90], Hq=48, Hkv=8, dtype=torch.bfloat16, step=2),  # R 6, G 2
    dict(lq=[150, 20], lk=[140, 300], Hq=12, Hkv=4, causal=True, window_left=40),  # R 3, G 1
    dict(lq=[90], lk=[130], Hq=8, Hkv=8, pad=192, dtype=torch.bfloat16),            # one head each
]


@pytest.mark.parametrize("case", GQA, ids=[f"gqa{i}" for i in range(len(GQA))])
def test_gqa_parity(oracle_mod, case):
    case = dict(case)
    lq, lk, Hq = case.pop("lq"), case.pop("lk"), case.pop("Hq")
    p = W.custom(lq, lk, Hq, **case)
    _, res = parity(p, oracle_mod)
    # the split calls run the same kernels
    split = _split(p.to("cuda"))
    for n in ("out", "lse", "dq", "dk", "dv"):
        assert bits_equal(res[n], split[n]), n


def test_gqa_call_is_bitwise_its_head_groups_alone():
    """A call with Hkv = 2 gives bitwise what two one-K/V-head calls give on
    its two head groups (strided head slices of the same tensors)."""
    Hq, Hkv = 16, 2
    R = Hq // Hkv
    p = W.custom([300, 37, 129], [260, 400, 9], Hq, Hkv=Hkv, dtype=torch.bfloat16).to("cuda")
    full = run(p)
    full = {n: full[n].clone() for n in ("out", "lse", "dq", "dk", "dv")}
    for g in range(Hkv):
        hs = slice(g * R, (g + 1) * R)
        r = BND.attention_varlen_fvjp(p.q[:, hs], p.k[:, g:g + 1], p.v[:, g:g + 1], p.cu_q,
                                      p.cu_k, p.alibi_slopes[:, hs], p.dout[:, hs])
        torch.cuda.synchronize()
        assert BND.device_status(r["workspace"]) == 0
        for n in ("out", "lse", "dq"):
            assert bits_equal(full[n][:, hs], r[n]), (n, g)
        for n in ("dk", "dv"):
            assert bits_equal(full[n][:, g:g + 1], r[n]), (n, g)


def test_gqa_rejects_uneven_head_split():
    p = W.custom([5], [7], 12, Hkv=1).to("cuda")
    k = torch.zeros((7, 5, 160), dtype=p.k.dtype, device="cuda")
    with pytest.raises(ValueError):
        BND.attention_varlen_fvjp(p.q, k, k, p.cu_q, p.cu_k, p.alibi_slopes, p.dout)


# ------------------------------------------------ head dimensions 128 and 64
# The tiles span 160 features; the TMA maps fill features past d with zeros
# and every other load and store stops at d.

HEAD_DIMS = [
    dict(lq=[300, 37, 1, 129], lk=[260, 400, 9, 0], Hq=16, d=128),
    dict(lq=[200, 64], lk=[333, 90], Hq=48, d=64, dtype=torch.bfloat16, step=2),
    dict(lq=[150, 20], lk=[140, 300], Hq=12, Hkv=4, d=128, causal=True, window_left=40,
         dtype=torch.bfloat16),
    dict(lq=[90, 500], lk=[130, 450], Hq=8, d=64, pad=192),  # NaN past feature 64
    dict(lq=[1000], lk=[1000], Hq=16, d=128, dtype=torch.bfloat16, step=3, pad=136),
]


@pytest.mark.parametrize("case", HEAD_DIMS, ids=[f"d{c['d']}_{i}" for i, c in enumerate(HEAD_DIMS)])
def test_head_dim_parity(oracle_mod, case):
    case = dict(case)
    lq, lk, Hq = case.pop("lq"), case.pop("lk"), case.pop("Hq")
    parity(W.custom(lq, lk, Hq, **case), oracle_mod)


@pytest.mark.parametrize("d", [64, 128])
def test_head_dim_outputs_written_exactly(d):
    """Padded NaN-filled output views with d features: exactly the d
    features of every row are written (the padding past d stays NaN), and
    the values equal those of dense outputs bit for bit."""
    p = W.custom([70, 5, 300], [40, 260, 0], 16, d=d, dtype=torch.bfloat16, step=2,
                 pad=192).to("cuda")
    dense = run(p)
    outs = dict(out=nan_like_strided(p.q), dq=nan_like_strided(p.dout), dk=nan_like_strided(p.k),
                dv=nan_like_strided(p.v))
    strided = run(p, **outs)
    for n in ("out", "dq", "dk", "dv"):
        assert torch.equal(strided[n].contiguous(), dense[n]), n
        raw = torch.empty(0, dtype=strided[n].dtype, device="cuda").set_(
            strided[n].untyped_storage())
        assert int(torch.isnan(raw).sum()) == raw.numel() - strided[n].numel(), n


# --------------------------------------------- host-resident inputs/outputs

def _host_cases():
    return [("tiny", lambda: W.tiny()),
            ("ragged_bf16_padded", lambda: W.custom([0, 37, 300, 1, 80], [9, 0, 260, 130, 75],
                                                    16, dtype=torch.bfloat16, step=2, pad=192)),
            ("gqa_d128_causal", lambda: W.custom([150, 20, 64], [140, 300, 64], 12, Hkv=4,
                                                 d=128, causal=True))]


@pytest.mark.parametrize("chunks", [1, 2, 3, 9])
@pytest.mark.parametrize("idx", range(3), ids=[c[0] for c in _host_cases()])
def test_host_buffers_bitwise_equal_device_call(idx, chunks):
    """The host-buffer entry point (chunked copies overlapped with the
    kernels) gives bitwise the device call's results for every chunking,
    including host layouts with padded heads (copied one head at a time)."""
    p_cpu = _host_cases()[idx][1]()
    dev = run(p_cpu.to("cuda"))
    r = BND.attention_varlen_fvjp_host(p_cpu.q, p_cpu.k, p_cpu.v, p_cpu.cu_q, p_cpu.cu_k,
                                       p_cpu.alibi_slopes, p_cpu.dout, p_cpu.causal,
                                       p_cpu.window_left, p_cpu.window_right, p_cpu.softcap,
                                       p_cpu.scale_multiplier, chunks=chunks)
    torch.cuda.synchronize()
    assert torch.all(r["status"] == 0), r["status"]
    for n in ("out", "lse", "dq", "dk", "dv"):
        assert bits_equal(dev[n].cpu(), r[n]), n


def test_host_buffers_leave_output_padding_alone():
    p_cpu = W.custom([40, 3], [20, 70], 16, dtype=torch.bfloat16, step=2, pad=192)
    outs = dict(out=nan_like_strided(p_cpu.q), dq=nan_like_strided(p_cpu.dout),
                dk=nan_like_strided(p_cpu.k), dv=nan_like_strided(p_cpu.v))
    r = BND.attention_varlen_fvjp_host(p_cpu.q, p_cpu.k, p_cpu.v, p_cpu.cu_q, p_cpu.cu_k,
                                       p_cpu.alibi_slopes, p_cpu.dout, chunks=2, **outs)
    torch.cuda.synchronize()
    for n in ("out", "dq", "dk", "dv"):
        raw = torch.empty(0, dtype=r[n].dtype).set_(r[n].untyped_storage())
        assert int(torch.isnan(raw).sum()) == raw.numel() - r[n].numel(), n


# ------------------------------------------------------------------ dropout
# Counter-based dropout: the keep decisions are integer hashes of (seed,
# sequence, head, row, column) on both sides, so the GPU and the oracle drop
# the same elements.

DROPOUT = [
    dict(lq=[70, 300, 1], lk=[90, 260, 40], Hq=16, rate=0.2),
    dict(lq=[200, 64], lk=[333, 90], Hq=48, dtype=torch.bfloat16, step=2, rate=0.5, causal=True),
    dict(lq=[150, 20], lk=[140, 300], Hq=12, Hkv=4, rate=None),   # per-token rates
    dict(lq=[40, 7], lk=[50, 30], Hq=16, rate=0.0),               # keeps everything
    dict(lq=[260, 33], lk=[300, 140], Hq=16, d=128, rate=0.3),    # head dimensions 128, 64
    dict(lq=[190, 70], lk=[150, 270], Hq=8, Hkv=2, d=64, dtype=torch.bfloat16, rate=0.1,
         causal=True),
    dict(lq=[120, 9], lk=[200, 45], Hq=16, d=128, rate=None),     # per-token rates, d = 128
]


def _with_dropout(case, seed=4321):
    case = dict(case)
    lq, lk, Hq, rate = case.pop("lq"), case.pop("lk"), case.pop("Hq"), case.pop("rate")
    p = W.custom(lq, lk, Hq, **case)
    p.dropout_seed = seed
    if rate is None:
        g = torch.Generator().manual_seed(3)
        p.dropout_rates = torch.rand(sum(lq), generator=g) * 0.6
    else:
        p.dropout_rate = rate
    return p


def _run_dropout(p, **kw):
    r = BND.attention_varlen_fvjp(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout,
                                  p.causal, p.window_left, p.window_right, p.softcap,
                                  p.scale_multiplier, dropout_seed=p.dropout_seed,
                                  dropout_rate=p.dropout_rate, dropout_rates=p.dropout_rates, **kw)
    torch.cuda.synchronize()
    assert BND.device_status(r["workspace"]) == 0
    return r


@pytest.mark.parametrize("idx", range(len(DROPOUT)), ids=[f"drop{i}" for i in range(len(DROPOUT))])
def test_dropout_parity(oracle_mod, idx):
    p_cpu = _with_dropout(DROPOUT[idx])
    p = p_cpu.to("cuda")
    res = _run_dropout(p)
    check_all(res, oracle_mod.fvjp(p_cpu), p_cpu.dtype)
    # repeatable, and the split calls regenerate the same keep bits
    again = _run_dropout(p)
    mask = (p.causal, p.window_left, p.window_right, p.softcap, p.scale_multiplier)
    drop = dict(dropout_seed=p.dropout_seed, dropout_rate=p.dropout_rate,
                dropout_rates=p.dropout_rates)
    out, lse = BND.attention_varlen_fwd(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, *mask,
                                        **drop)
    dq, dk, dv = BND.attention_varlen_bwd(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout,
                                          out, lse, *mask, **drop)
    torch.cuda.synchronize()
    for n, x in (("out", out), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert bits_equal(res[n], again[n]), n
        assert bits_equal(res[n], x), n
    # the keep bits stored by the forward and read by the backward: bitwise
    # the regenerated ones, fused and split (the mask buffer starts dirty)
    Hkv = p.k.shape[1]
    nbytes = BND.dropout_mask_bytes(p.cu_q, p.cu_k, p.Hq, Hkv)
    km = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    stored = _run_dropout(p, keep_mask=km)
    km2 = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device="cuda")
    out2, lse2 = BND.attention_varlen_fwd(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, *mask,
                                          keep_mask=km2, **drop)
    dq2, dk2, dv2 = BND.attention_varlen_bwd(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes,
                                             p.dout, out2, lse2, *mask, keep_mask=km2, **drop)
    torch.cuda.synchronize()
    for n, x in (("out", out2), ("lse", lse2), ("dq", dq2), ("dk", dk2), ("dv", dv2)):
        assert bits_equal(res[n], stored[n]), n
        assert bits_equal(res[n], x), n


def test_dropout_mask_too_small_sets_status():
    """A keep-mask buffer below what the lengths need is caught on the device:
    the status word carries the mask-space bit and the kernels do nothing."""
    p = _with_dropout(DROPOUT[0]).to("cuda")
    nbytes = BND.dropout_mask_bytes(p.cu_q, p.cu_k, p.Hq, p.k.shape[1])
    km = torch.zeros(nbytes - 2048, dtype=torch.uint8, device="cuda")
    out = torch.full(p.q.shape, float("nan"), dtype=p.q.dtype, device="cuda")
    r = BND.attention_varlen_fvjp(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout,
                                  p.causal, p.window_left, p.window_right, p.softcap,
                                  p.scale_multiplier, dropout_seed=p.dropout_seed,
                                  dropout_rate=p.dropout_rate, keep_mask=km, out=out)
    torch.cuda.synchronize()
    assert BND.device_status(r["workspace"]) & BND.DEV_MASK_SPACE
    assert bool(torch.isnan(out).all())


def test_dropout_seed_changes_the_result():
    p = _with_dropout(DROPOUT[0]).to("cuda")
    a = {n: x.clone() for n, x in _run_dropout(p).items() if n != "workspace"}
    p.dropout_seed = 4322
    b = _run_dropout(p)
    assert not bits_equal(a["out"], b["out"]) and bits_equal(a["lse"], b["lse"])


# ------------------------------------------- split forward / backward calls

def _split_cases():
    return [("tiny", lambda: W.tiny()),
            ("tiny_causal_win16", lambda: W.tiny(causal=True, window_left=16, window_right=16)),
            ("ragged_bf16_strided", lambda: W.custom([0, 37, 300, 1], [9, 0, 260, 130], 16,
                                                     dtype=torch.bfloat16, step=2))]


def _split(p, out=None, lse=None):
    mask = (p.causal, p.window_left, p.window_right, p.softcap, p.scale_multiplier)
    if out is None:
        out, lse = BND.attention_varlen_fwd(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, *mask)
    dq, dk, dv = BND.attention_varlen_bwd(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout,
                                          out, lse, *mask)
    torch.cuda.synchronize()
    return dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv)


@pytest.mark.parametrize("idx", range(3), ids=[c[0] for c in _split_cases()])
def test_split_calls_bitwise_equal_fused_and_match_oracle(oracle_mod, idx):
    """Forward then backward as two calls gives bitwise the fused call's five
    tensors (the same kernels run), and agrees with the oracle."""
    p_cpu = _split_cases()[idx][1]()
    p = p_cpu.to("cuda")
    fused = run(p)
    split = _split(p)
    for n in ("out", "lse", "dq", "dk", "dv"):
        assert bits_equal(fused[n], split[n]), n
    check_all(split, oracle_mod.fvjp(p_cpu), p_cpu.dtype)


def test_split_backward_reads_out_and_lse_without_writing_them():
    p = W.tiny().to("cuda")
    out, lse = BND.attention_varlen_fwd(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes)
    torch.cuda.synchronize()
    h = [view_bytes_hash(out), view_bytes_hash(lse)]
    r1 = _split(p, out, lse)
    r2 = _split(p, out, lse)
    assert h == [view_bytes_hash(out), view_bytes_hash(lse)]
    for n in ("dq", "dk", "dv"):
        assert bits_equal(r1[n], r2[n]), n


def test_split_degenerate_sizes():
    p = W.custom([5, 3], [0, 0], 16).to("cuda")
    r = _split(p)
    assert torch.all(r["out"] == 0) and torch.all(r["dq"] == 0)
    assert torch.all(r["lse"] == -math.inf)
    p = W.custom([0, 0], [7, 3], 16).to("cuda")
    r = _split(p)
    assert torch.all(r["dk"] == 0) and torch.all(r["dv"] == 0)


def test_no_cap_large_logits(oracle_mod):
    p = W.custom([50, 20], [300, 90], 16, qk_std=6.0)
    p.softcap = 0.0
    parity(p, oracle_mod)


def test_no_keys_at_all():
    p = W.custom([5, 3], [0, 0], 16).to("cuda")
    r = run(p)
    assert torch.all(r["out"] == 0) and torch.all(r["dq"] == 0)
    assert torch.all(r["lse"] == -math.inf)


def test_no_queries_at_all():
    p = W.custom([0, 0], [7, 3], 16).to("cuda")
    r = run(p)
    assert torch.all(r["dk"] == 0) and torch.all(r["dv"] == 0)


def test_bad_cu_sets_device_status():
    """A non-monotone cu_q is caught on the device: the status word gets the
    bad-cu bit and no kernel computes anything."""
    p = W.custom([5, 6], [7, 8], 16).to("cuda")
    p.cu_q = torch.tensor([0, 9, 11], dtype=torch.int32, device="cuda")  # total 11, ok
    p.cu_q[1] = 12  # now cu_q[1] > cu_q[2]
    r = BND.attention_varlen_fvjp(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout)
    torch.cuda.synchronize()
    assert BND.device_status(r["workspace"]) == BND.DEV_BAD_CU


def test_host_rejects_misaligned_stride():
    p = W.custom([5], [7], 16).to("cuda")
    base = torch.zeros((5, 16, 164), dtype=p.q.dtype, device="cuda")
    q = base[:, :, :160]
    q.copy_(p.q)
    with pytest.raises(BND.AttnError) as e:
        BND.attention_varlen_fvjp(q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout)
    assert e.value.code == -3


# ------------------------------------------- full-size configs, sampled checks

FULL = ["q_short_k_long", "k_short_q_long", "mixed_h64", "mixed_h80", "long_balanced"]


def _sample_rows(p, gen, n=48):
    """Packed (token, head) rows: first and last token of random sequences and
    random interior tokens, random heads."""
    toks, heads = [], []
    lq, _ = p.lengths()
    nonempty = [b for b in range(p.B) if lq[b] > 0]
    for s in range(n):
        b = nonempty[int(torch.randint(0, len(nonempty), (1,), generator=gen))]
        q0 = int(p.cu_q[b])
        off = [0, lq[b] - 1, int(torch.randint(0, lq[b], (1,), generator=gen))][s % 3]
        toks.append(q0 + off)
        heads.append(int(torch.randint(0, p.Hq, (1,), generator=gen)))
    return torch.tensor(toks), torch.tensor(heads, dtype=torch.int32)


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(oracle_mod, name):
    p = W.WORKLOADS[name](device="cuda")
    r1 = run(p)
    snap = {n: r1[n].clone() for n in ("out", "dq", "dk", "dv", "lse")}
    r2 = run(p)
    for n, x in snap.items():  # bitwise repeat at full size
        assert bits_equal(x, r2[n]), n
    gen = torch.Generator().manual_seed(99)
    tok, head = _sample_rows(p, gen)
    # per-sequence CPU copies keep the oracle's input small
    lq, lk = p.lengths()
    got_out, got_dq, got_lse, ref_out, ref_dq, ref_lse = [], [], [], [], [], []
    for b in sorted(set(int(torch.searchsorted(p.cu_q.cpu(), t, right=True)) - 1 for t in tok)):
        sel = [n for n in range(len(tok)) if int(p.cu_q[b]) <= int(tok[n]) < int(p.cu_q[b + 1])]
        if not sel:
            continue
        sp = p.sequence(b)
        q0 = int(p.cu_q[b])
        rr = oracle_mod.rows(sp, tok[sel] - q0, head[sel])
        for m, n in enumerate(sel):
            t, h = int(tok[n]), int(head[n])
            got_out.append(r1["out"][t, h].float().cpu())
            got_dq.append(r1["dq"][t, h].float().cpu())
            got_lse.append(r1["lse"][t, h].cpu())
            ref_out.append(rr["out"][m])
            ref_dq.append(rr["dq"][m])
            ref_lse.append(rr["lse"][m])
    check_tensor("out(sampled)", torch.stack(got_out), torch.stack(ref_out), p.dtype)
    check_tensor("dq(sampled)", torch.stack(got_dq), torch.stack(ref_dq), p.dtype)
    check_lse(torch.stack(got_lse), torch.stack(ref_lse))
    # dk/dv: in full on the two cheapest sequences (by Lq*Lk); in the balanced
    # long case, where every sequence is long, on 64 sampled keys of the
    # cheapest one (their lse and D come from the oracle's own row pass over
    # every head of that sequence)
    if name == "long_balanced":
        b = min(range(p.B), key=lambda i: lq[i] * lk[i])
        L = lk[b]
        kg = torch.Generator().manual_seed(7)
        keys = sorted(set([0, 1, 127, 128, 129, L // 2, L - 129, L - 128, L - 2, L - 1] +
                          torch.randint(0, L, (54,), generator=kg).tolist()))
        sp = p.sequence(b)
        ref = oracle_mod.keys(sp, keys, [0] * len(keys))
        k0 = int(p.cu_k[b])
        rows = torch.tensor(keys) + k0
        check_tensor(f"dk(seq {b}, sampled keys)", r1["dk"][rows.cuda(), 0].cpu(), ref["dk"], p.dtype)
        check_tensor(f"dv(seq {b}, sampled keys)", r1["dv"][rows.cuda(), 0].cpu(), ref["dv"], p.dtype)
    else:
        work = sorted(range(p.B), key=lambda b: lq[b] * lk[b])
        for b in [w for w in work if lq[w] > 0 and lk[w] > 0][:2]:
            sp = p.sequence(b)
            ref = oracle_mod.fvjp(sp)
            k0, k1 = int(p.cu_k[b]), int(p.cu_k[b + 1])
            check_tensor(f"dk(seq {b})", r1["dk"][k0:k1].cpu(), ref["dk"], p.dtype)
            check_tensor(f"dv(seq {b})", r1["dv"][k0:k1].cpu(), ref["dv"], p.dtype)
    # a property at any size: per sequence, sum_j dv_j = sum_{h,i} dO_i
    for b in range(p.B):
        if lq[b] == 0 or lk[b] == 0:
            continue
        q0, q1 = int(p.cu_q[b]), int(p.cu_q[b + 1])
        k0, k1 = int(p.cu_k[b]), int(p.cu_k[b + 1])
        lhs = r1["dv"][k0:k1].double().sum((0, 1)).cpu()
        rhs = p.dout[q0:q1].double().sum((0, 1)).cpu()
        err = float((lhs - rhs).norm() / max(float(rhs.norm()), 1e-30))
        assert err < 2e-2, (b, err)

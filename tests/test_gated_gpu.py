"""The sigmoid-gated variant on the GPU ("Pairwise-Gated Attention Engine",
"Why it is hard"): out = (softmax(z) o sigmoid(q_g k_g^T / sqrt(R))) v and
its five gradients through the C ABI, against the fp64 oracle's gated
definition (itself pinned against torch autograd), at the tolerances of the
rest of the suite; bitwise repeats; the forward-only call equals the fused
one."""
import pytest
import torch

from helpers import check_lse, check_tensor
from ragged_gqa_attention_varlen_gb300 import binding as BND
from ragged_gqa_attention_varlen_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from ragged_gqa_attention_varlen_gb300 import _build

    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return BND.load()


def run(p):
    r = BND.attention_varlen_gated(p.q, p.k, p.v, p.q_gate, p.k_gate, p.cu_q, p.cu_k,
                                   p.alibi_slopes, p.dout, p.causal, p.window_left,
                                   p.window_right, p.scale_multiplier)
    torch.cuda.synchronize()
    st = BND.device_status(r["workspace"])
    assert st == 0, f"device status {st:#x}"
    return r


GRAD = ("out", "dq", "dk", "dv", "dq_gate", "dk_gate")


def parity(p_cpu, oracle_mod):
    p = p_cpu.to("cuda")
    res = run(p)
    ref = oracle_mod.fvjp(p_cpu)
    for n in GRAD:
        check_tensor(n, res[n], ref[n], p_cpu.dtype)
    check_lse(res["lse"], ref["lse"])
    return p, res


def gated_custom(lq, lk, Hq, Hkv=1, R=64, d=128, seed=0, slopes=False, **kw):
    p = W.custom(lq, lk, Hq, dtype=kw.pop("dtype", torch.bfloat16), seed=seed, Hkv=Hkv, d=d,
                 pad=d, **kw)
    p.softcap = 0.0
    p.scale_multiplier = 1.0
    if not slopes:
        p.alibi_slopes = torch.zeros_like(p.alibi_slopes)
    g = torch.Generator().manual_seed(seed + 500)
    p.q_gate = torch.randn((sum(lq), Hq, R), generator=g).to(p.dtype)
    p.k_gate = torch.randn((sum(lk), Hkv, R), generator=g).to(p.dtype)
    return p


# the page's training shapes at reduced length: 8 causal sequences, Hq 32
# over 8 K/V heads, head sizes 64/128, gate widths 32/64
@pytest.mark.parametrize("d,R", [(128, 64), (128, 32), (64, 64), (64, 32)])
def test_gated_workload_replica_parity_and_repeat(oracle_mod, d, R):
    p_cpu = W.gated(length_scale=1 / 32, d=d, R=R)
    p, res = parity(p_cpu, oracle_mod)
    again = run(p)
    for n in GRAD + ("lse",):
        assert torch.equal(res[n], again[n]), n


CASES = [
    dict(lq=[300, 129, 40], lk=[257, 400, 170], Hq=16),                       # global
    dict(lq=[200, 300], lk=[350, 300], Hq=8, Hkv=2, window_left=100, window_right=30),
    dict(lq=[150, 64, 0], lk=[400, 200, 70], Hq=16, slopes=True, causal=True),  # ALiBi
    dict(lq=[0, 5, 90], lk=[7, 0, 300], Hq=4, Hkv=4, R=48, d=64),             # empty sequences
    dict(lq=[180, 33], lk=[90, 260], Hq=12, Hkv=3, dtype=torch.float16, R=16),
    dict(lq=[1, 7], lk=[3, 2], Hq=8),                                         # few keys
]


@pytest.mark.parametrize("case", CASES, ids=[f"gate{i}" for i in range(len(CASES))])
def test_gated_edge_parity(oracle_mod, case):
    case = dict(case)
    lq, lk, Hq = case.pop("lq"), case.pop("lk"), case.pop("Hq")
    parity(gated_custom(lq, lk, Hq, seed=len(lq) + Hq, **case), oracle_mod)


def test_gated_single_key(oracle_mod):
    """One key per sequence: P = 1, so out = G v and dS = G dP - D vanishes in
    exact arithmetic (dq = dk = 0; the fp64 oracle leaves only rounding
    there).  out, lse, dv and both gate gradients are checked at the usual
    tolerances; dq and dk against the rounding of the 16-bit out that D is
    formed from: |dS| <= 2^-7 |dP|, so |dq| <= 2^-7 sigma max|dO . v| max|k|
    (and the same with max|q| for dk)."""
    p_cpu = gated_custom([1, 1], [1, 1], 8, seed=9)
    p = p_cpu.to("cuda")
    res = run(p)
    ref = oracle_mod.fvjp(p_cpu)
    for n in ("out", "dv", "dq_gate", "dk_gate"):
        check_tensor(n, res[n], ref[n], p_cpu.dtype)
    check_lse(res["lse"], ref["lse"])
    sigma = p_cpu.scale_multiplier / p_cpu.q.shape[-1] ** 0.5
    dp = (p_cpu.dout.double() * p_cpu.v.double().expand_as(p_cpu.dout)).sum(-1).abs().max()
    for n, x in (("dq", p_cpu.k), ("dk", p_cpu.q)):
        bound = 2.0 ** -7 * sigma * float(dp) * float(x.double().abs().max()) * (
            p_cpu.Hq if n == "dk" else 1)
        assert float(res[n].double().abs().max()) <= bound, n


def test_gated_forward_only_equals_fused():
    p = gated_custom([260, 70], [300, 129], 16, Hkv=4, causal=True, seed=3).to("cuda")
    fused = run(p)
    f = BND.attention_varlen_gated(p.q, p.k, p.v, p.q_gate, p.k_gate, p.cu_q, p.cu_k,
                                   p.alibi_slopes, None, p.causal, p.window_left,
                                   p.window_right, p.scale_multiplier)
    torch.cuda.synchronize()
    assert BND.device_status(f["workspace"]) == 0
    assert torch.equal(f["out"], fused["out"]) and torch.equal(f["lse"], fused["lse"])


def test_gated_rejects_unsupported_shapes():
    p = gated_custom([10], [10], 4, R=64).to("cuda")
    with pytest.raises(BND.AttnError):  # gate width above 64
        BND.attention_varlen_gated(p.q, p.k, p.v, torch.zeros((10, 4, 72), dtype=p.dtype,
                                                              device="cuda"),
                                   torch.zeros((10, 1, 72), dtype=p.dtype, device="cuda"),
                                   p.cu_q, p.cu_k, None, p.dout)

"""The sharded path's GPU pieces on one device: every rank's share of a
two-rank plan run one after the other through the C ABI (head-sliced calls
for the parts of a cut sequence), the partial dk/dv added by the library's
fixed-order sum, and the assembled batch checked against the fp64 oracle.
(Ranks that wait on one another never run as separate launches on one GPU:
here nothing waits, the partials are handed over between launches.)"""
import pytest
import torch

from helpers import check_all
from ragged_gqa_attention_varlen_gb300 import binding as BND
from ragged_gqa_attention_varlen_gb300 import shard
from ragged_gqa_attention_varlen_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from ragged_gqa_attention_varlen_gb300 import _build

    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return BND.load()


def _compute(sub):
    r = BND.attention_varlen_fvjp(sub.q, sub.k, sub.v, sub.cu_q, sub.cu_k, sub.alibi_slopes,
                                  sub.dout, sub.causal, sub.window_left, sub.window_right,
                                  sub.softcap, sub.scale_multiplier)
    torch.cuda.synchronize()
    assert BND.device_status(r["workspace"]) == 0
    return r


def _reduce(parts):
    out = torch.empty_like(parts[0])
    BND.sum_partials(parts, out)
    return out


CASES = [
    dict(lq=[600, 40, 90, 30], lk=[700, 50, 60, 20], Hq=16),
    dict(lq=[600, 40, 90], lk=[600, 50, 200], Hq=16, causal=True, dtype=torch.bfloat16, step=2),
    dict(lq=[700, 60, 20], lk=[650, 40, 300], Hq=16, Hkv=4, d=128),
]


@pytest.mark.parametrize("case", CASES, ids=["cut", "cut_causal_bf16", "gqa_d128"])
def test_two_rank_plan_on_one_gpu_matches_oracle_and_repeats(oracle_mod, case):
    case = dict(case)
    lq, lk, Hq = case.pop("lq"), case.pop("lk"), case.pop("Hq")
    p_cpu = W.custom(lq, lk, Hq, seed=21, **case)
    p = p_cpu.to("cuda")
    plan, pieces = shard.run_ranks_in_one_process(p, 2, _compute, _reduce)
    assert len(plan.parts(0)) == 2  # the dominant sequence was cut
    got = shard.assemble(p, pieces)
    ref = oracle_mod.fvjp(p_cpu)
    check_all(got, ref, p_cpu.dtype)
    _, again = shard.run_ranks_in_one_process(p, 2, _compute, _reduce)
    got2 = shard.assemble(p, again)
    for n in ("out", "dq", "dk", "dv", "lse"):
        assert torch.equal(got[n], got2[n]), n


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_sum_partials_is_the_fp32_sum_in_part_order(dtype):
    g = torch.Generator(device="cuda").manual_seed(3)
    base = torch.randn((3, 513, 1, 192), generator=g, device="cuda").to(dtype)
    parts = [base[i, :, :, :160] for i in range(3)]  # row stride 192
    out_base = torch.full((513, 1, 176), float("nan"), dtype=dtype, device="cuda")
    out = out_base[:, :, :160]
    BND.sum_partials(parts, out)
    torch.cuda.synchronize()
    expect = ((parts[0].float() + parts[1].float()) + parts[2].float()).to(dtype)
    assert torch.equal(out, expect)
    assert torch.isnan(out_base[:, :, 160:]).all()  # padding untouched

"""The no-allocation entry point, checked on the GPU against the ordinary one.

Some callers may not allocate device memory (a plugin inside a framework that
owns every device allocation, a service that forbids allocator calls while it
serves).  For them the library has attn_varlen_fvjp_fwd_bwd_noalloc, which
takes inputs and outputs only and keeps its scratch in a fixed device array
inside the library.  This file is collected last so that a failure here
never hides the rest of the suite.
"""
import pytest
import torch

from ragged_gqa_attention_varlen_gb300 import binding as BND
from ragged_gqa_attention_varlen_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from ragged_gqa_attention_varlen_gb300 import _build

    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return BND.load()


def _bits(x):
    return x.contiguous().view(torch.int16 if x.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("order", ["large_then_small", "small_then_large"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(order):
    """Two calls in a row through the no-allocation entry point (different
    problem sizes, so the second inherits the first's scratch contents), each
    bitwise equal to the ordinary entry point on the same inputs: both run the
    same kernels on the same schedule, so any difference (a counter or status
    word left over from the previous call) shows."""
    probs = [W.q_short(length_scale=0.25).to("cuda"), W.tiny().to("cuda")]
    if order == "small_then_large":
        probs.reverse()
    for p in probs:
        ref = BND.attention_varlen_fvjp(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout,
                                        p.causal, p.window_left, p.window_right, p.softcap,
                                        p.scale_multiplier)
        torch.cuda.synchronize()
        assert BND.device_status(ref["workspace"]) == 0
        out, dq = torch.empty_like(ref["out"]), torch.empty_like(ref["dq"])
        dk, dv = torch.empty_like(ref["dk"]), torch.empty_like(ref["dv"])
        lse = torch.empty_like(ref["lse"])
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        BND.attention_varlen_fvjp_noalloc(p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout,
                                          out, dq, dk, dv, lse, status, p.causal,
                                          p.window_left, p.window_right, p.softcap,
                                          p.scale_multiplier)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for name, x in (("out", out), ("dq", dq), ("dk", dk), ("dv", dv), ("lse", lse)):
            assert torch.equal(_bits(x), _bits(ref[name])), name

"""The flop count bench.py reports: admissible (query, key) pairs under each
mask shape, checked against a direct count over every pair."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from ragged_gqa_attention_varlen_gb300 import workloads as W  # noqa: E402


def _direct(lq, lk, causal, wl, wr):
    n = 0
    for a, b in zip(lq, lk):
        for i in range(a):
            k0 = i + b - a
            for j in range(b):
                if wl >= 0 and j < k0 - wl:
                    continue
                if (0 if causal else wr) >= 0 and j > k0 + (0 if causal else wr):
                    continue
                n += 1
    return n


@pytest.mark.parametrize("mask", [(False, -1, -1), (True, -1, -1), (False, 7, 3), (False, 5, -1),
                                  (False, -1, 0), (True, 4, 9), (False, 0, 0)])
def test_scored_pairs_match_direct_count(mask):
    lq, lk = [0, 5, 40, 13, 1], [9, 0, 17, 60, 1]
    p = W.custom(lq, lk, 2)
    p.causal, p.window_left, p.window_right = mask
    assert bench.scored_pairs(p) == _direct(lq, lk, *mask)
    if mask == (False, -1, -1):
        assert bench.scored_pairs(p) == p.sum_lq_lk()
    assert bench.counted_flops(p) == 14.0 * 160 * 2 * bench.scored_pairs(p)


def test_mufu_bound_counts_two_transcendentals_per_unit_and_kernel():
    """tanh at 16 and exp2 at 32 per clock per SM: 3/32 SM clocks per unit and
    kernel with the softcap, 1/32 without."""
    import bench
    from ragged_gqa_attention_varlen_gb300 import workloads as W

    p = W.tiny()
    units = p.Hq * p.sum_lq_lk()
    m = bench.mufu_bound(p, call_ms=1.0, kernel_ms=None, sm_mhz=1000.0, sms=2)
    one = units * (1 / 16 + 1 / 32) / 2 / 1e9 * 1e3
    assert m["units"] == units
    assert abs(m["bound_ms"] - 3 * one) < 1e-15
    p.softcap = 0.0
    m0 = bench.mufu_bound(p, call_ms=1.0, kernel_ms={"forward": 1.0, "dkdv": 2.0, "dq": 1.0},
                          sm_mhz=1000.0, sms=2)
    assert abs(m0["bound_ms"] - 3 * units / 32 / 2 / 1e9 * 1e3) < 1e-15
    assert abs(m0["per_kernel"]["dkdv"]["frac"] - m0["per_kernel"]["forward"]["frac"] / 2) < 1e-15

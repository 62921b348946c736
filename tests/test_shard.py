"""The sharded path on CPU: the library's shard plan, and two gloo ranks that
each run the oracle on their share and exchange partial key gradients.

Sequences are independent, so whole sequences on different ranks give
bitwise the rows of one run over the batch; a sequence cut by query head
gives partial dk/dv per part, added in part order on the rank holding part
0 (checked bitwise against that sum, and against the one-rank result up to
fp64 rounding)."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from ragged_gqa_attention_varlen_gb300 import _build, binding

    _build.build()
    return binding.load()


def _plan(cu_q, cu_k, Hq, Hkv, n, **mask):
    from ragged_gqa_attention_varlen_gb300 import binding

    return binding.shard_plan(torch.tensor(cu_q, dtype=torch.int32),
                              torch.tensor(cu_k, dtype=torch.int32), Hq, Hkv, n, **mask)


def _cu(ls):
    out = [0]
    for x in ls:
        out.append(out[-1] + x)
    return out


def _pairs(lq, lk, causal=False, window_left=-1, window_right=-1):
    wr = 0 if causal else window_right
    n = 0
    for i in range(lq):
        k0 = i + lk - lq
        lo = max(0, k0 - window_left) if window_left >= 0 else 0
        hi = min(lk - 1, k0 + wr) if wr >= 0 else lk - 1
        n += max(0, hi - lo + 1)
    return n


@pytest.mark.parametrize("n", [1, 2, 3, 8])
@pytest.mark.parametrize("mask", [dict(), dict(causal=True), dict(window_left=50, window_right=7)])
def test_plan_covers_every_head_once_and_balances(lib, n, mask):
    g = torch.Generator().manual_seed(n)
    lq = torch.randint(1, 400, (30,), generator=g).tolist()
    lk = torch.randint(1, 400, (30,), generator=g).tolist()
    lq[3], lk[3] = 3000, 2500  # one dominant sequence
    Hq = 16
    units, work = _plan(_cu(lq), _cu(lk), Hq, 1, n, **mask)
    w = [Hq * _pairs(a, b, **mask) for a, b in zip(lq, lk)]
    total = sum(w)
    # every (sequence, head) exactly once; units in (sequence, head) order
    cover = {}
    for b, h0, h1, r in units:
        assert 0 <= r < n and 0 <= h0 < h1 <= Hq
        for h in range(h0, h1):
            assert (b, h) not in cover
            cover[(b, h)] = r
    assert len(cover) == 30 * Hq
    assert units == sorted(units)
    # the ranks' work adds up; parts of one sequence sit on different ranks
    assert sum(work) == pytest.approx(total)
    for b in range(30):
        ranks = [r for bb, _, _, r in units if bb == b]
        assert len(ranks) == len(set(ranks))
    # list scheduling bound: no rank exceeds the mean by more than one unit
    biggest = max(w[b] * (h1 - h0) / Hq for b, h0, h1, _ in units)
    assert max(work) <= total / n + biggest + 1e-6
    for b in range(30):  # exactly the sequences above the mean share are cut
        assert (sum(1 for u in units if u[0] == b) > 1) == (n > 1 and w[b] > total / n)
    if n == 1:
        assert all((h0, h1) == (0, Hq) for _, h0, h1, _ in units)
    # deterministic
    assert _plan(_cu(lq), _cu(lk), Hq, 1, n, **mask) == (units, work)


def test_plan_cuts_kv_groups_whole(lib):
    units, _ = _plan(_cu([2000, 10, 10]), _cu([2000, 10, 10]), 16, 4, 8)
    parts = [(h0, h1) for b, h0, h1, _ in units if b == 0]
    assert parts == [(0, 4), (4, 8), (8, 12), (12, 16)]  # at most Hkv parts, R = 4 heads each


def test_plan_rejects_bad_arguments(lib):
    from ragged_gqa_attention_varlen_gb300 import binding

    with pytest.raises(ValueError):
        _plan(_cu([3]), _cu([4]), 6, 4, 2)  # 6 heads over 4 K/V heads
    with pytest.raises(ValueError):
        _plan(_cu([3]), _cu([4]), 8, 1, 17)  # more than 16 ranks
    with pytest.raises(ValueError):
        binding.shard_plan(torch.tensor([0, 5, 3], dtype=torch.int32),
                           torch.tensor([0, 1, 2], dtype=torch.int32), 8, 1, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CASES = {
    "cut": dict(lq=[40, 5, 9, 3], lk=[50, 7, 4, 6], Hq=4),
    "cut_causal": dict(lq=[40, 5, 9, 3], lk=[50, 7, 4, 6], Hq=4, causal=True),
    "gqa": dict(lq=[40, 5, 9, 3], lk=[50, 7, 4, 6], Hq=8, Hkv=2),
    "balanced": dict(lq=[12, 15, 9, 11, 0], lk=[10, 14, 13, 8, 5], Hq=3),
}


def _problem(case):
    sys.path.insert(0, ROOT)
    from ragged_gqa_attention_varlen_gb300 import workloads as W

    c = dict(CASES[case])
    lq, lk, Hq = c.pop("lq"), c.pop("lk"), c.pop("Hq")
    return W.custom(lq, lk, Hq, seed=11, **c)


def _sum_in_order(parts):
    acc = parts[0].clone()
    for t in parts[1:]:
        acc = acc + t
    return acc


def _worker(rank, world, port, case, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from ragged_gqa_attention_varlen_gb300 import shard

    dist.init_process_group("gloo", rank=rank, world_size=world)
    p = _problem(case)
    plan, pieces = shard.run_rank(p, world, rank, oracle.fvjp, _sum_in_order, dist)
    gathered = [None] * world
    dist.all_gather_object(gathered, pieces)
    if rank == 0:
        out["pieces"] = [x for g in gathered for x in g]
        out["units"] = [(u.seq, u.h0, u.h1, u.rank) for u in plan.units]
    dist.destroy_process_group()


@pytest.mark.parametrize("case", sorted(CASES))
def test_two_gloo_ranks_reproduce_the_one_rank_oracle(lib, oracle_mod, case):
    from ragged_gqa_attention_varlen_gb300 import shard

    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, case, out)) for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=300)
        assert pr.exitcode == 0
    p = _problem(case)
    got = shard.assemble(p, list(out["pieces"]))
    ref = oracle_mod.fvjp(p)
    units = list(out["units"])
    assert len({r for *_, r in units}) == 2  # both ranks had work
    plan = shard.Plan([shard.Unit(*u) for u in units], [], world, p.Hq, p.k.shape[1])
    cut = plan.partial_sequences()
    if case.startswith("cut"):
        assert cut == [0]
    else:
        assert cut == []
    for n in ("out", "dq", "lse"):  # query rows: bitwise, whoever computed them
        assert torch.equal(got[n], ref[n]), n
    mk = torch.ones(p.total_k, dtype=torch.bool)
    for b in cut:
        mk[int(p.cu_k[b]):int(p.cu_k[b + 1])] = False
    for n in ("dk", "dv"):  # keys of whole sequences (and K/V groups): bitwise
        assert torch.equal(got[n][mk], ref[n][mk]), n
    for b in cut:  # cut sequences: the part-order sum, and the one-rank value
        k0, k1 = int(p.cu_k[b]), int(p.cu_k[b + 1])
        part_res = [oracle_mod.fvjp(s.problem) for r in range(world)
                    for s in shard.shares(p, plan, r) if s.partial and s.seqs == [b]]
        order = sorted(range(len(part_res)),
                       key=lambda i: [s.h0 for r in range(world) for s in shard.shares(p, plan, r)
                                      if s.partial and s.seqs == [b]][i])
        for n in ("dk", "dv"):
            expect = _sum_in_order([part_res[i][n] for i in order])
            assert torch.equal(got[n][k0:k1], expect), n
            torch.testing.assert_close(got[n][k0:k1], ref[n][k0:k1], rtol=1e-12, atol=1e-13)

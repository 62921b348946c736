"""One batch over several processes (one GPU each): the plan, each rank's
share of the work, and the one exchange step.

The plan comes from the library (``attn_varlen_shard_plan``): whole
sequences, longest processing time first, and for a sequence holding more
than 1/N of the batch's work, parts by query head (one K/V head) or by K/V
head group.  Sequences attend only within themselves ("Noncausal Global
Extreme-GQA Ragged Attention Full VJP", "Hard Constraints"), so whole
sequences need no exchange; the parts of a one-K/V-head sequence each give a
partial dk/dv of its keys, which the rank holding part 0 receives and adds in
part order.

This module only moves tensors and calls a compute function on each rank's
share; the arithmetic runs in that function (the library's kernels on a GPU,
or the oracle in the CPU tests) and in the library's fixed-order sum.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Callable, Dict, List, Optional, Tuple

import torch

from . import binding
from .workloads import Problem


@dataclass(frozen=True)
class Unit:
    seq: int
    h0: int
    h1: int
    rank: int


class Plan:
    """The library's shard plan of one problem over ``nranks`` ranks."""

    def __init__(self, units: List[Unit], work: List[float], nranks: int, Hq: int, Hkv: int):
        self.units, self.work, self.nranks, self.Hq, self.Hkv = units, work, nranks, Hq, Hkv

    def of_rank(self, r: int) -> List[Unit]:
        return [u for u in self.units if u.rank == r]

    def parts(self, b: int) -> List[Unit]:
        return sorted((u for u in self.units if u.seq == b), key=lambda u: u.h0)

    def partial_sequences(self) -> List[int]:
        """Sequences whose dk/dv are sums of partials (one K/V head, cut)."""
        if self.Hkv != 1:
            return []
        seqs = sorted({u.seq for u in self.units})
        return [b for b in seqs if len(self.parts(b)) > 1]

    def owner(self, b: int) -> int:
        return self.parts(b)[0].rank


def make_plan(p: Problem, nranks: int) -> Plan:
    Hkv = p.k.shape[1]
    units, work = binding.shard_plan(p.cu_q, p.cu_k, p.Hq, Hkv, nranks, p.causal,
                                     p.window_left, p.window_right)
    return Plan([Unit(*u) for u in units], work, nranks, p.Hq, Hkv)


@dataclass
class Share:
    """A piece of one rank's work: a problem and where its rows belong."""

    problem: Problem
    seqs: List[int]      # sequences of the batch, in the problem's order
    h0: int              # query heads [h0, h1) of the batch
    h1: int
    partial: bool        # dk/dv of its (single) sequence are a partial sum


def _gather(x: torch.Tensor, ranges: List[Tuple[int, int]]) -> torch.Tensor:
    return torch.cat([x[a:b] for a, b in ranges]) if ranges else x[:0].clone()


def shares(p: Problem, plan: Plan, rank: int) -> List[Share]:
    """The problems rank ``rank`` computes: its whole sequences gathered into
    one packed problem (dense copies), and one problem per part of a cut
    sequence (head-sliced views of the batch's tensors)."""
    cu_q = p.cu_q.cpu().tolist()
    cu_k = p.cu_k.cpu().tolist()
    mine = plan.of_rank(rank)
    out = []
    whole = [u.seq for u in mine if (u.h0, u.h1) == (0, p.Hq)]
    if whole:
        rq = [(cu_q[b], cu_q[b + 1]) for b in whole]
        rk = [(cu_k[b], cu_k[b + 1]) for b in whole]
        lq = [b - a for a, b in rq]
        lk = [b - a for a, b in rk]
        dev = p.cu_q.device
        cq = torch.tensor([0] + list(torch.tensor(lq).cumsum(0).tolist()), dtype=torch.int32)
        ck = torch.tensor([0] + list(torch.tensor(lk).cumsum(0).tolist()), dtype=torch.int32)
        sub = replace(p, name=f"{p.name}[rank {rank} whole]", B=len(whole),
                      cu_q=cq.to(dev), cu_k=ck.to(dev),
                      q=_gather(p.q, rq), k=_gather(p.k, rk), v=_gather(p.v, rk),
                      dout=_gather(p.dout, rq),
                      alibi_slopes=p.alibi_slopes[torch.tensor(whole, device=p.alibi_slopes.device)]
                      .contiguous(), meta=dict(p.meta))
        out.append(Share(sub, whole, 0, p.Hq, False))
    R = p.Hq // p.k.shape[1]
    for u in mine:
        if (u.h0, u.h1) == (0, p.Hq):
            continue
        b = u.seq
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        g0, g1 = (u.h0 // R, u.h1 // R) if plan.Hkv > 1 else (0, 1)
        dev = p.cu_q.device
        sub = replace(p, name=f"{p.name}[seq {b} heads {u.h0}:{u.h1}]", B=1, Hq=u.h1 - u.h0,
                      cu_q=torch.tensor([0, q1 - q0], dtype=torch.int32, device=dev),
                      cu_k=torch.tensor([0, k1 - k0], dtype=torch.int32, device=dev),
                      q=p.q[q0:q1, u.h0:u.h1], k=p.k[k0:k1, g0:g1], v=p.v[k0:k1, g0:g1],
                      dout=p.dout[q0:q1, u.h0:u.h1],
                      alibi_slopes=p.alibi_slopes[b:b + 1, u.h0:u.h1], meta=dict(p.meta))
        out.append(Share(sub, [b], u.h0, u.h1, plan.Hkv == 1))
    return out


Result = Dict[str, torch.Tensor]  # out, lse, dq, dk, dv of one share


def exchange(p: Problem, plan: Plan, rank: int, mine: List[Share], results: List[Result],
             reduce: Callable[[List[torch.Tensor]], torch.Tensor], dist=None) -> Dict[int, Result]:
    """The exchange step: for every sequence cut by query head (in sequence
    order), each rank holding a later part sends its partial dk/dv to the
    rank holding part 0, which adds them in part order with ``reduce``.
    Returns {sequence: {"dk", "dv"}} of the sums this rank owns."""
    cu_k = p.cu_k.cpu().tolist()
    have = {}
    for s, r in zip(mine, results):
        if s.partial:
            have[(s.seqs[0], s.h0)] = r
    sums = {}
    for b in plan.partial_sequences():
        parts = plan.parts(b)
        owner = parts[0].rank
        if rank != owner and all(u.rank != rank for u in parts):
            continue
        got = {"dk": [], "dv": []}
        for u in parts:
            for name in ("dk", "dv"):
                if u.rank == rank and rank == owner:
                    got[name].append(have[(b, u.h0)][name])
                elif u.rank == rank:
                    dist.send(have[(b, u.h0)][name].contiguous(), dst=owner)
                elif rank == owner:
                    Lk = cu_k[b + 1] - cu_k[b]
                    ref = have[(b, parts[0].h0)][name]
                    buf = torch.empty((Lk,) + tuple(ref.shape[1:]), dtype=ref.dtype,
                                      device=ref.device)
                    dist.recv(buf, src=u.rank)
                    got[name].append(buf)
        if rank == owner:
            sums[b] = {n: reduce(got[n]) for n in ("dk", "dv")}
    return sums


def owned_pieces(p: Problem, plan: Plan, mine: List[Share], results: List[Result],
                 sums: Dict[int, Result]) -> list:
    """What this rank holds of the batch's results, as (kind, sequence, h0,
    h1, tensors) tuples on the CPU: query rows ("q": out, dq, lse) of every
    share, and key rows ("k": dk, dv) of whole sequences and of the sums it
    owns."""
    cu_q = p.cu_q.cpu().tolist()
    cu_k = p.cu_k.cpu().tolist()
    pieces = []
    for s, r in zip(mine, results):
        oq = ok = 0
        for b in s.seqs:
            lq, lk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
            pieces.append(("q", b, s.h0, s.h1, {n: r[n][oq:oq + lq].cpu()
                                                  for n in ("out", "dq", "lse")}))
            if not s.partial:
                pieces.append(("k", b, s.h0, s.h1, {n: r[n][ok:ok + lk].cpu()
                                                      for n in ("dk", "dv")}))
            oq += lq
            ok += lk
    for b, r in sums.items():
        pieces.append(("k", b, 0, p.Hq, {n: r[n].cpu() for n in ("dk", "dv")}))
    return pieces


def assemble(p: Problem, all_pieces: list, dtype=torch.float64) -> Result:
    """The batch's results from every rank's pieces (for checks)."""
    Tq, Tk, d = p.total_q, p.total_k, p.q.shape[-1]
    Hkv = p.k.shape[1]
    R = p.Hq // Hkv
    res = dict(out=torch.full((Tq, p.Hq, d), float("nan"), dtype=dtype),
               dq=torch.full((Tq, p.Hq, d), float("nan"), dtype=dtype),
               lse=torch.full((Tq, p.Hq), float("nan"), dtype=dtype),
               dk=torch.full((Tk, Hkv, d), float("nan"), dtype=dtype),
               dv=torch.full((Tk, Hkv, d), float("nan"), dtype=dtype))
    cu_q = p.cu_q.cpu().tolist()
    cu_k = p.cu_k.cpu().tolist()
    for kind, b, h0, h1, t in all_pieces:
        if kind == "q":
            for n in ("out", "dq", "lse"):
                res[n][cu_q[b]:cu_q[b + 1], h0:h1] = t[n].to(dtype)
        else:
            g0, g1 = (h0 // R, h1 // R) if Hkv > 1 else (0, 1)
            for n in ("dk", "dv"):
                res[n][cu_k[b]:cu_k[b + 1], g0:g1] = t[n].to(dtype)
    return res


def run_rank(p: Problem, nranks: int, rank: int, compute: Callable[[Problem], Result],
             reduce: Callable[[List[torch.Tensor]], torch.Tensor], dist=None,
             plan: Optional[Plan] = None):
    """This rank's share of the batch: plan, compute, exchange.  Returns
    (plan, pieces this rank owns)."""
    plan = plan or make_plan(p, nranks)
    mine = shares(p, plan, rank)
    results = [compute(s.problem) for s in mine]
    sums = exchange(p, plan, rank, mine, results, reduce, dist)
    return plan, owned_pieces(p, plan, mine, results, sums)


def run_ranks_in_one_process(p: Problem, nranks: int, compute: Callable[[Problem], Result],
                             reduce: Callable[[List[torch.Tensor]], torch.Tensor]):
    """Every rank's share computed one after the other in this process, the
    partials handed over directly (for checks on one device).  Returns
    (plan, pieces of all ranks)."""
    plan = make_plan(p, nranks)
    per_rank = []
    for r in range(nranks):
        mine = shares(p, plan, r)
        per_rank.append((mine, [compute(s.problem) for s in mine]))
    partials = {}
    for mine, results in per_rank:
        for s, res in zip(mine, results):
            if s.partial:
                partials[(s.seqs[0], s.h0)] = res
    pieces = []
    for r, (mine, results) in enumerate(per_rank):
        sums = {}
        for b in plan.partial_sequences():
            if plan.owner(b) == r:
                sums[b] = {n: reduce([partials[(b, u.h0)][n] for u in plan.parts(b)])
                           for n in ("dk", "dv")}
        pieces += owned_pieces(p, plan, mine, results, sums)
    return plan, pieces

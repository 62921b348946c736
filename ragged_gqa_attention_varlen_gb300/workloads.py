"""Seeded synthetic inputs for packed ragged GQA attention.

This module only draws inputs (lengths, values, ALiBi slopes) and lays them out
as the strided packed views the attention op consumes.  It holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it.

The input family follows "Noncausal Global Extreme-GQA Ragged Attention Full
VJP", section "What You Have": 18-52 independent ragged sequences, 48-96 query
heads sharing one K/V head, head dimension 160, fp16/bf16 activations, q/k/v
and dout given as views with feature padding and token steps of two or three,
fp32 ALiBi slopes of shape [batch, q_heads], softcap 3 and scale multiplier
0.75.  The concrete length and value distributions of each named workload are
listed in ``WORKLOADS``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

HEAD_DIM = 160


@dataclass
class Problem:
    """One call's inputs.  q/dout: [T_q, Hq, 160]; k/v: [T_k, 1, 160] views."""

    name: str
    dtype: torch.dtype
    B: int
    Hq: int
    cu_q: torch.Tensor  # int32 [B+1]
    cu_k: torch.Tensor  # int32 [B+1]
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dout: torch.Tensor
    alibi_slopes: torch.Tensor  # fp32 [B, Hq]
    causal: bool = False
    window_left: int = -1
    window_right: int = -1
    softcap: float = 3.0
    scale_multiplier: float = 0.75
    # counter-based dropout: off when dropout_seed is None; one rate, or one
    # per query token (fp32 [total_q]) when dropout_rates is given
    dropout_seed: Optional[int] = None
    dropout_rate: float = 0.0
    dropout_rates: Optional[torch.Tensor] = None
    # sigmoid gate projections (the gated variant): [T_q, Hq, R], [T_k, Hkv, R]
    q_gate: Optional[torch.Tensor] = None
    k_gate: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)

    @property
    def total_q(self) -> int:
        return int(self.cu_q[-1])

    @property
    def total_k(self) -> int:
        return int(self.cu_k[-1])

    def lengths(self):
        lq = (self.cu_q[1:] - self.cu_q[:-1]).tolist()
        lk = (self.cu_k[1:] - self.cu_k[:-1]).tolist()
        return lq, lk

    def sum_lq_lk(self) -> int:
        lq, lk = self.lengths()
        return sum(a * b for a, b in zip(lq, lk))

    def to(self, device) -> "Problem":
        """Copy every tensor to ``device`` keeping the strided view layout."""
        out = Problem(**{**self.__dict__})
        for name in ("q", "k", "v", "dout"):
            out.__dict__[name] = _copy_view(getattr(self, name), device)
        for name in ("q_gate", "k_gate"):
            if getattr(self, name) is not None:
                out.__dict__[name] = _copy_view(getattr(self, name), device)
        out.cu_q = self.cu_q.to(device)
        out.cu_k = self.cu_k.to(device)
        out.alibi_slopes = self.alibi_slopes.to(device)
        if self.dropout_rates is not None:
            out.dropout_rates = self.dropout_rates.to(device)
        return out

    def sequence(self, b: int) -> "Problem":
        """Sequence b alone, as a B=1 problem with dense CPU copies (without
        dropout: its hash depends on the sequence index)."""
        assert self.dropout_seed is None, "a dropout problem cannot be cut into sequences"
        q0, q1 = int(self.cu_q[b]), int(self.cu_q[b + 1])
        k0, k1 = int(self.cu_k[b]), int(self.cu_k[b + 1])
        return Problem(
            name=f"{self.name}[seq {b}]", dtype=self.dtype, B=1, Hq=self.Hq,
            cu_q=torch.tensor([0, q1 - q0], dtype=torch.int32),
            cu_k=torch.tensor([0, k1 - k0], dtype=torch.int32),
            q=self.q[q0:q1].cpu().contiguous(), k=self.k[k0:k1].cpu().contiguous(),
            v=self.v[k0:k1].cpu().contiguous(), dout=self.dout[q0:q1].cpu().contiguous(),
            alibi_slopes=self.alibi_slopes[b:b + 1].cpu().contiguous(),
            causal=self.causal, window_left=self.window_left, window_right=self.window_right,
            softcap=self.softcap, scale_multiplier=self.scale_multiplier)


def _copy_view(x: torch.Tensor, device) -> torch.Tensor:
    """Copy a strided view to ``device`` with the same strides (same padding)."""
    if x.is_contiguous():
        return x.to(device)
    base = torch.full((x.untyped_storage().nbytes() // x.element_size(),), float("nan"),
                      dtype=x.dtype, device=device)
    y = base.as_strided(x.shape, x.stride(), x.storage_offset())
    y.copy_(x)
    return y


def strided_view(T: int, H: int, step: int, pad: int, dtype, device, poison: bool = True,
                 d: int = HEAD_DIM):
    """An uninitialised [T, H, d] view into a [step*T, H, pad] buffer.

    The gaps (token rows skipped by the step, features d..pad-1) hold NaN
    when ``poison`` is set, so a kernel that reads them shows it."""
    base = torch.empty((max(step * T, 1), H, pad), dtype=dtype, device=device)
    if poison and (step > 1 or pad > d):
        base.fill_(float("nan"))
    return base[: step * T: step, :, :d] if T > 0 else base[:0, :, :d]


def _fill_normal(view: torch.Tensor, std: float, gen: torch.Generator, chunk_tokens: int = 4096):
    """Fill a view with std * N(0, 1) drawn token-chunk by token-chunk in fp32."""
    T = view.shape[0]
    for t0 in range(0, T, chunk_tokens):
        t1 = min(T, t0 + chunk_tokens)
        x = torch.randn((t1 - t0,) + tuple(view.shape[1:]), generator=gen,
                        dtype=torch.float32, device=view.device)
        if std != 1.0:
            x.mul_(std)
        view[t0:t1].copy_(x)


def _cu(lengths):
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def _uniform_int(gen, lo, hi, n):
    """n integers uniform on [lo, hi], both ends included."""
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


def _log_uniform_int(gen, lo, hi, n):
    """floor(exp(U(log lo, log hi))), at least 1."""
    u = torch.rand((n,), generator=gen, dtype=torch.float64)
    x = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return [max(1, int(math.floor(float(a)))) for a in x]


def _alibi_geometric(Hq):
    """Standard ALiBi slopes 2^(-8h/H) for h = 1..H."""
    return torch.tensor([2.0 ** (-8.0 * h / Hq) for h in range(1, Hq + 1)], dtype=torch.float32)


def build(name, lq, lk, Hq, dtype, step, pad, slopes, qk_std=1.0, v_std=1.0, do_std=1.0,
          seed=0, device="cpu", poison=True, Hkv=1, d=HEAD_DIM, **mask) -> Problem:
    """Draw the values of a problem whose lengths and slopes are already fixed
    (k and v get Hkv heads; every row has d features)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1000003 + 17)
    cu_q, cu_k = _cu(lq), _cu(lk)
    Tq, Tk = int(cu_q[-1]), int(cu_k[-1])
    pad = max(pad, d)
    q = strided_view(Tq, Hq, step, pad, dtype, device, poison, d)
    k = strided_view(Tk, Hkv, step, pad, dtype, device, poison, d)
    v = strided_view(Tk, Hkv, step, pad, dtype, device, poison, d)
    dout = strided_view(Tq, Hq, step, pad, dtype, device, poison, d)
    _fill_normal(q, qk_std, gen)
    _fill_normal(k, qk_std, gen)
    _fill_normal(v, v_std, gen)
    _fill_normal(dout, do_std, gen)
    return Problem(name=name, dtype=dtype, B=len(lq), Hq=Hq, cu_q=cu_q.to(device),
                   cu_k=cu_k.to(device), q=q, k=k, v=v, dout=dout,
                   alibi_slopes=slopes.contiguous().to(device),
                   meta=dict(step=step, pad=pad, seed=seed), **mask)


# ---- the named workloads ----------------------------------------------------

def tiny(seed=0, device="cpu", causal=False, window_left=-1, window_right=-1):
    """3 sequences, Lq=[5,17,33], Lk=[40,9,64], Hq=8, fp16, contiguous,
    N(0,1) values, slopes U(0, 0.25)."""
    g = torch.Generator().manual_seed(seed)
    slopes = torch.rand((3, 8), generator=g, dtype=torch.float32) * 0.25
    return build("tiny", [5, 17, 33], [40, 9, 64], 8, torch.float16, 1, HEAD_DIM, slopes,
                 seed=seed, device=device, causal=causal, window_left=window_left,
                 window_right=window_right)


def q_short(seed=1, device="cpu", length_scale=1.0):
    """18 sequences, Lq U[16,256], Lk U[1024,4096], Hq=48, bf16, features padded
    to 192, token step 2, N(0,1) values, slopes 2^(-8h/48) x U(0.5,1.5) per
    sequence."""
    g = torch.Generator().manual_seed(seed)
    B, Hq = 18, 48
    lq = _uniform_int(g, 16, 256, B)
    lk = _uniform_int(g, 1024, 4096, B)
    lq, lk = _scale(lq, length_scale), _scale(lk, length_scale)
    factor = 0.5 + torch.rand((B, 1), generator=g, dtype=torch.float32)
    slopes = _alibi_geometric(Hq)[None, :] * factor
    return build("q_short_k_long", lq, lk, Hq, torch.bfloat16, 2, 192, slopes, seed=seed,
                 device=device)


def k_short(seed=2, device="cpu", length_scale=1.0):
    """52 sequences, Lq U[1024,4096], Lk U[32,384], Hq=96, fp16, features padded
    to 176, token step 3, q/k/v N(0,1), dout N(0,0.5), slopes U(0, 0.2)."""
    g = torch.Generator().manual_seed(seed)
    B, Hq = 52, 96
    lq = _uniform_int(g, 1024, 4096, B)
    lk = _uniform_int(g, 32, 384, B)
    lq, lk = _scale(lq, length_scale), _scale(lk, length_scale)
    slopes = torch.rand((B, Hq), generator=g, dtype=torch.float32) * 0.2
    return build("k_short_q_long", lq, lk, Hq, torch.float16, 3, 176, slopes, do_std=0.5,
                 seed=seed, device=device)


# Sequences forced to length 1 in the mixed workload (query side, key side).
MIXED_LQ1 = (5, 17)
MIXED_LK1 = (11, 23)


def mixed(seed=3, Hq=64, device="cpu", length_scale=1.0):
    """32 sequences, Lq and Lk independently log-uniform on [8, 8192] with
    Lq = 1 forced at two sequences and Lk = 1 at two others, bf16, token step
    2, dense features, q/k 4 x N(0,1) (the softcap saturates), v/dout N(0,1),
    slopes U(0, 0.5)."""
    g = torch.Generator().manual_seed(seed)
    B = 32
    lq = _log_uniform_int(g, 8, 8192, B)
    lk = _log_uniform_int(g, 8, 8192, B)
    lq, lk = _scale(lq, length_scale), _scale(lk, length_scale)
    for b in MIXED_LQ1:
        lq[b] = 1
    for b in MIXED_LK1:
        lk[b] = 1
    slopes = torch.rand((B, Hq), generator=g, dtype=torch.float32) * 0.5
    return build(f"mixed_h{Hq}", lq, lk, Hq, torch.bfloat16, 2, HEAD_DIM, slopes, qk_std=4.0,
                 seed=seed, device=device)


def long_balanced(seed=5, device="cpu", length_scale=1.0, poison=True, Hkv=1, d=HEAD_DIM):
    """24 sequences with Lq = Lk ~ U[6144, 12288], Hq=96, bf16, dense features,
    token step 2, N(0,1) values, slopes 2^(-8h/96); Hkv K/V heads (1 unless
    asked)."""
    g = torch.Generator().manual_seed(seed)
    B, Hq = 24, 96
    L = _scale(_uniform_int(g, 6144, 12288, B), length_scale)
    slopes = _alibi_geometric(Hq)[None, :].expand(B, Hq).contiguous()
    return build("long_balanced", L, list(L), Hq, torch.bfloat16, 2, d, slopes,
                 seed=seed, device=device, poison=poison, Hkv=Hkv, d=d)


def gated(seed=6, device="cpu", length_scale=1.0, d=128, R=64, Hq=32, Hkv=8, poison=True):
    """The gated variant's training shape family ("Pairwise-Gated Attention
    Engine", "The task": head sizes 64 and 128, gate sizes 32 and 64,
    grouped K/V heads, sequences up to 16,384 tokens): 8 causal sequences with
    Lq = Lk ~ U[1024, 16384], bf16, dense layouts, no softcap and no ALiBi
    (the page's plain softmax with logits q.k / sqrt(d): scale multiplier 1),
    q/k/v/dout and the gate projections N(0,1)."""
    g = torch.Generator().manual_seed(seed)
    B = 8
    L = _scale(_uniform_int(g, 1024, 16384, B), length_scale)
    p = build("gated", L, list(L), Hq, torch.bfloat16, 1, d, torch.zeros(B, Hq), seed=seed,
              device=device, poison=poison, Hkv=Hkv, d=d, causal=True)
    p.softcap = 0.0
    p.scale_multiplier = 1.0
    gg = torch.Generator(device=device).manual_seed(seed * 7 + 1)
    p.q_gate = torch.randn((sum(L), Hq, R), generator=gg, dtype=torch.float32,
                           device=device).to(torch.bfloat16)
    p.k_gate = torch.randn((sum(L), Hkv, R), generator=gg, dtype=torch.float32,
                           device=device).to(torch.bfloat16)
    return p


def _scale(lengths, s):
    if s == 1.0:
        return list(lengths)
    return [max(1, int(round(L * s))) for L in lengths]


WORKLOADS = {
    "tiny": tiny,
    "q_short_k_long": q_short,
    "k_short_q_long": k_short,
    "mixed_h64": lambda **kw: mixed(seed=kw.pop("seed", 3), Hq=64, **kw),
    "mixed_h80": lambda **kw: mixed(seed=kw.pop("seed", 4), Hq=80, **kw),
    "long_balanced": long_balanced,
}


def custom(lq, lk, Hq, dtype=torch.float16, step=1, pad=HEAD_DIM, seed=0, device="cpu",
           slope_max=0.25, qk_std=1.0, poison=True, Hkv=1, d=HEAD_DIM, **mask) -> Problem:
    """A small problem with given lengths, for edge cases."""
    g = torch.Generator().manual_seed(seed)
    slopes = torch.rand((len(lq), Hq), generator=g, dtype=torch.float32) * slope_max
    return build("custom", list(lq), list(lk), Hq, dtype, step, pad, slopes, qk_std=qk_std,
                 seed=seed, device=device, poison=poison, Hkv=Hkv, d=d, **mask)

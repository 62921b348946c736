"""fp64 CPU oracle for ragged GQA attention and its full VJP -- test
infrastructure only.

Only the test-suite, the package smoke check and the benchmark's CPU-baseline
leg import this module.  It loads ``liboracle.so`` built from
``attn_oracle.c`` (plain C, fp64, POSIX threads), which shares no code with the
CUDA path.  See that file's header for the definition it follows and the page
sections it cites.

Parity unpinned: none.  Every output of ``fvjp`` and ``rows`` is pinned by the
CPU tests in ``tests/test_oracle.py`` (library special cases, closed forms,
finite differences, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "attn_oracle.c")
_LIB = os.path.join(_DIR, "liboracle.so")
_lib = None

DTYPE_CODE = {torch.float16: 0, torch.bfloat16: 1, torch.float64: 2}


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc, no GPU needed)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-fPIC",
                               "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        U64, F32 = ctypes.c_uint64, ctypes.c_float
        common = ([I, I, I, I, I, P, L, L, P, L, L, P, L, L, P, L, L, P, P, P, L, I, I, I, D, D] +
                  [I, U64, F32, P] + [I, P, L, L, P, L, L])
        lib.oracle_fvjp.argtypes = common + [P] + [P] * 10 + [I]
        lib.oracle_fvjp.restype = I
        lib.oracle_rows.argtypes = common + [I, P, P, P, P, P, P, I]
        lib.oracle_rows.restype = I
        lib.oracle_keys.argtypes = common + [I, P, P, P, P, I]
        lib.oracle_keys.restype = I
        lib.oracle_decode.argtypes = [I, ctypes.c_uint16]
        lib.oracle_decode.restype = D
        lib.oracle_splitmix64.argtypes = [U64]
        lib.oracle_splitmix64.restype = U64
        lib.oracle_drop_factor.argtypes = [U64, F32, I, I, I, I]
        lib.oracle_drop_factor.restype = D
        _lib = lib
    return _lib


def _raw(x: torch.Tensor) -> torch.Tensor:
    """The tensor's bits as a same-strided CPU view (16-bit types as int16)."""
    assert x.device.type == "cpu"
    if x.dtype in (torch.float16, torch.bfloat16):
        return x.view(torch.int16)
    assert x.dtype == torch.float64
    return x


def _args(p):
    q, k, v, do = _raw(p.q), _raw(p.k), _raw(p.v), _raw(p.dout)
    for t in (q, k, v, do):
        assert t.stride(-1) == 1, "feature axis must be contiguous"
    cu_q = p.cu_q.to(torch.int32).cpu().contiguous()
    cu_k = p.cu_k.to(torch.int32).cpu().contiguous()
    slopes = None if p.alibi_slopes is None else p.alibi_slopes.float().cpu()
    if slopes is not None:
        assert slopes.stride(1) == 1
    seed = getattr(p, "dropout_seed", None)
    rates = getattr(p, "dropout_rates", None)
    if rates is not None:
        rates = rates.float().cpu().contiguous()
        assert rates.shape == (p.q.shape[0],)
    qg, kg = getattr(p, "q_gate", None), getattr(p, "k_gate", None)
    R = 0
    if qg is not None:
        qg, kg = _raw(qg), _raw(kg)
        R = qg.shape[-1]
        assert kg.shape[-1] == R and qg.stride(-1) == 1 and kg.stride(-1) == 1
    keep = (q, k, v, do, cu_q, cu_k, slopes, rates, qg, kg)
    Hkv = p.k.shape[1]
    assert v.shape[1] == Hkv and p.Hq % Hkv == 0
    args = [DTYPE_CODE[p.q.dtype], p.B, p.Hq, Hkv, p.q.shape[-1],
            q.data_ptr(), q.stride(0), q.stride(1),
            k.data_ptr(), k.stride(0), k.stride(1), v.data_ptr(), v.stride(0), v.stride(1),
            do.data_ptr(), do.stride(0), do.stride(1),
            cu_q.data_ptr(), cu_k.data_ptr(),
            slopes.data_ptr() if slopes is not None else None,
            slopes.stride(0) if slopes is not None else 0,
            int(bool(p.causal)), int(p.window_left), int(p.window_right),
            float(p.softcap), float(p.scale_multiplier),
            int(seed is not None), int(seed or 0) & 0xFFFFFFFFFFFFFFFF,
            float(getattr(p, "dropout_rate", 0.0)), rates.data_ptr() if rates is not None else None,
            R, qg.data_ptr() if R else None, qg.stride(0) if R else 0, qg.stride(1) if R else 0,
            kg.data_ptr() if R else None, kg.stride(0) if R else 0, kg.stride(1) if R else 0]
    return args, keep


def fvjp(p, seq_sel=None, nthreads: int = 0, diagnostics: bool = False) -> dict:
    """Forward and full VJP of problem ``p`` (CPU tensors) in fp64.

    Returns float64 tensors out/dq [T_q,Hq,d], lse/D [T_q,Hq], dk/dv [T_k,Hkv,d]
    (plus dz_rowsum, p_rowsum when ``diagnostics``), and the thread count.
    With ``seq_sel`` (iterable of sequence indices) only those sequences are
    computed; other rows hold NaN."""
    lib = _load()
    args, keep = _args(p)
    Tq, Tk, H, d = p.q.shape[0], p.k.shape[0], p.Hq, p.q.shape[-1]
    Hkv = p.k.shape[1]
    f64 = dict(dtype=torch.float64)
    res = dict(out=torch.full((Tq, H, d), float("nan"), **f64),
               lse=torch.full((Tq, H), float("nan"), **f64),
               dq=torch.full((Tq, H, d), float("nan"), **f64),
               dk=torch.full((Tk, Hkv, d), float("nan"), **f64),
               dv=torch.full((Tk, Hkv, d), float("nan"), **f64),
               D=torch.full((Tq, H), float("nan"), **f64))
    if diagnostics:
        res["dz_rowsum"] = torch.full((Tq, H), float("nan"), **f64)
        res["p_rowsum"] = torch.full((Tq, H), float("nan"), **f64)
    if getattr(p, "q_gate", None) is not None:
        R = p.q_gate.shape[-1]
        res["dq_gate"] = torch.full((Tq, H, R), float("nan"), **f64)
        res["dk_gate"] = torch.full((Tk, Hkv, R), float("nan"), **f64)
    sel = None
    if seq_sel is not None:
        mask = np.zeros(p.B, dtype=np.uint8)
        mask[list(seq_sel)] = 1
        sel = torch.from_numpy(mask)
    ptr = lambda name: res[name].data_ptr() if name in res else None
    nt = lib.oracle_fvjp(*args, sel.data_ptr() if sel is not None else None,
                         ptr("out"), ptr("lse"), ptr("dq"), ptr("dk"), ptr("dv"), ptr("D"),
                         ptr("dz_rowsum"), ptr("p_rowsum"), ptr("dq_gate"), ptr("dk_gate"),
                         int(nthreads))
    del keep
    res["threads"] = nt
    return res


def rows(p, tok, head, nthreads: int = 0) -> dict:
    """out, lse, D and dq of the sampled packed rows (tok[r], head[r])
    (ungated problems)."""
    if getattr(p, "q_gate", None) is not None:
        raise NotImplementedError("the row sampler serves ungated problems")
    lib = _load()
    args, keep = _args(p)
    tok = torch.as_tensor(tok, dtype=torch.int64).contiguous()
    head = torch.as_tensor(head, dtype=torch.int32).contiguous()
    n, d = tok.numel(), p.q.shape[-1]
    f64 = dict(dtype=torch.float64)
    res = dict(out=torch.empty((n, d), **f64), lse=torch.empty((n,), **f64),
               dq=torch.empty((n, d), **f64), D=torch.empty((n,), **f64))
    nt = lib.oracle_rows(*args, n, tok.data_ptr(), head.data_ptr(), res["out"].data_ptr(),
                         res["lse"].data_ptr(), res["dq"].data_ptr(), res["D"].data_ptr(),
                         int(nthreads))
    del keep
    res["threads"] = nt
    return res


def keys(p, tok, head, nthreads: int = 0) -> dict:
    """dk and dv of the sampled packed keys (tok[r], K/V head head[r])
    (ungated problems), equal bit for bit to ``fvjp``'s rows: every sequence
    holding a sampled key takes the row pass without its dq part, then each
    sampled key the key pass."""
    if getattr(p, "q_gate", None) is not None:
        raise NotImplementedError("the key sampler serves ungated problems")
    lib = _load()
    args, keep = _args(p)
    tok = torch.as_tensor(tok, dtype=torch.int64).contiguous()
    head = torch.as_tensor(head, dtype=torch.int32).contiguous()
    n, d = tok.numel(), p.q.shape[-1]
    f64 = dict(dtype=torch.float64)
    res = dict(dk=torch.empty((n, d), **f64), dv=torch.empty((n, d), **f64))
    nt = lib.oracle_keys(*args, n, tok.data_ptr(), head.data_ptr(), res["dk"].data_ptr(),
                         res["dv"].data_ptr(), int(nthreads))
    del keep
    if nt == 0:
        raise ValueError("oracle_keys rejected its arguments")
    res["threads"] = nt
    return res


def decode(dtype: torch.dtype, bits: int) -> float:
    """The oracle's own decoding of one 16-bit pattern."""
    return _load().oracle_decode(DTYPE_CODE[dtype], bits & 0xFFFF)


def splitmix64(x: int) -> int:
    """The oracle's SplitMix64 output function of one 64-bit value."""
    return int(_load().oracle_splitmix64(x & 0xFFFFFFFFFFFFFFFF))


def drop_factor(seed: int, rate: float, b: int, h: int, i: int, j: int) -> float:
    """The oracle's dropout factor (keep * 1/(1-rate), or 0) of one element."""
    return float(_load().oracle_drop_factor(seed & 0xFFFFFFFFFFFFFFFF, rate, b, h, i, j))


def cores() -> int:
    return os.cpu_count() or 1

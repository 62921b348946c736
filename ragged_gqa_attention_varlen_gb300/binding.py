"""ctypes binding of libattn_varlen.so (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; PyTorch only
provides device memory and the current stream.  There is no fallback: if the
library is missing or no CUDA device is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn_varlen.so")
HEAD_DIM = 160            # the pages' head dimension
HEAD_DIMS = (64, 128, 160)  # head dimensions the library accepts
_lib = None

ATTN_F16, ATTN_BF16 = 0, 1
DEV_BAD_CU, DEV_TIMEOUT_FWD, DEV_TIMEOUT_DKDV, DEV_TIMEOUT_DQ = 0x1, 0x2, 0x4, 0x8
DEV_MASK_SPACE = 0x20

EXPORTS = ("attn_varlen_fvjp_fwd_bwd", "attn_varlen_fvjp_workspace_size", "attn_status_string",
           "attn_varlen_fvjp_launch_count", "attn_varlen_fvjp_record_events",
           "attn_varlen_fvjp_fwd_bwd_noalloc", "attn_varlen_fwd", "attn_varlen_bwd",
           "attn_varlen_launch_count", "attn_varlen_fvjp_fwd_bwd_host",
           "attn_varlen_fvjp_host_buffer_size", "attn_varlen_fvjp_host_buffer_size_for",
           "attn_varlen_fvjp_fwd_bwd_dropout",
           "attn_varlen_fwd_dropout", "attn_varlen_bwd_dropout", "attn_varlen_host_chunks",
           "attn_varlen_shard_plan", "attn_varlen_sum_partials",
           "attn_varlen_gated_fvjp_fwd_bwd", "attn_varlen_gated_fwd",
           "attn_varlen_fvjp_fwd_bwd_dropout_mask", "attn_varlen_fwd_dropout_mask",
           "attn_varlen_bwd_dropout_mask", "attn_varlen_dropout_mask_bytes")
NOALLOC_SCRATCH_BYTES = 64 << 20
KERNELS = ("schedule", "forward", "preprocess", "dkdv", "dq")


class AttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"attn_varlen error {code}: {msg}")
        self.code = code


def load(path: str = LIB_PATH):
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing "
                           "(run __graft_entry__.build() or ragged_gqa_attention_varlen_gb300/_build.py)")
    lib = ctypes.CDLL(path)
    P, I, L, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.attn_varlen_fvjp_workspace_size.argtypes = [I, I, L, L]
    lib.attn_varlen_fvjp_workspace_size.restype = ctypes.c_size_t
    lib.attn_varlen_fvjp_launch_count.argtypes = [I, I, L, L]
    lib.attn_varlen_fvjp_launch_count.restype = I
    lib.attn_varlen_launch_count.argtypes = [I, I, I, I, L, L]
    lib.attn_varlen_launch_count.restype = I
    lib.attn_status_string.argtypes = [I]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_varlen_fvjp_fwd_bwd.argtypes = (
        [I, I, I, I, I, L, L] + [P, L, L] * 4 + [P, P, P, L, I, I, I, F, F] + [P, L, L] * 4 +
        [P, P, ctypes.c_size_t, P, P])
    lib.attn_varlen_fvjp_fwd_bwd.restype = I
    lib.attn_varlen_fvjp_fwd_bwd_noalloc.argtypes = (
        [I, I, I, I, I, L, L] + [P, L, L] * 4 + [P, P, P, L, I, I, I, F, F] + [P, L, L] * 4 +
        [P, P, P])
    lib.attn_varlen_fvjp_fwd_bwd_noalloc.restype = I
    lib.attn_varlen_fwd.argtypes = (
        [I, I, I, I, I, L, L] + [P, L, L] * 3 + [P, P, P, L, I, I, I, F, F] + [P, L, L] +
        [P, P, ctypes.c_size_t, P, P])
    lib.attn_varlen_fwd.restype = I
    lib.attn_varlen_bwd.argtypes = (
        [I, I, I, I, I, L, L] + [P, L, L] * 4 + [P, P, P, L, I, I, I, F, F] + [P, L, L, P] +
        [P, L, L] * 3 + [P, ctypes.c_size_t, P, P])
    lib.attn_varlen_bwd.restype = I
    lib.attn_varlen_fvjp_fwd_bwd_host.argtypes = (
        [I, I, I, I, I, L, L] + [P, L, L] * 4 + [P, P, P, L, I, I, I, F, F] + [P, L, L] * 4 +
        [P, P, ctypes.c_size_t, I, P, P])
    lib.attn_varlen_fvjp_fwd_bwd_host.restype = I
    lib.attn_varlen_fvjp_host_buffer_size.argtypes = [I, I, I, I, L, L, I]
    lib.attn_varlen_fvjp_host_buffer_size.restype = ctypes.c_size_t
    lib.attn_varlen_fvjp_host_buffer_size_for.argtypes = [I, P, P, I, I, I, I]
    lib.attn_varlen_fvjp_host_buffer_size_for.restype = ctypes.c_size_t
    lib.attn_varlen_host_chunks.argtypes = [I, P, P, I, P]
    lib.attn_varlen_host_chunks.restype = I
    DR = [ctypes.c_uint64, F, P]  # dropout seed, rate, per-token rates
    lib.attn_varlen_fvjp_fwd_bwd_dropout.argtypes = (
        [I, I, I, I, I, L, L] + [P, L, L] * 4 + [P, P, P, L, I, I, I, F, F] + DR +
        [P, L, L] * 4 + [P, P, ctypes.c_size_t, P, P])
    lib.attn_varlen_fvjp_fwd_bwd_dropout.restype = I
    lib.attn_varlen_fwd_dropout.argtypes = (
        [I, I, I, I, I, L, L] + [P, L, L] * 3 + [P, P, P, L, I, I, I, F, F] + DR + [P, L, L] +
        [P, P, ctypes.c_size_t, P, P])
    lib.attn_varlen_fwd_dropout.restype = I
    lib.attn_varlen_bwd_dropout.argtypes = (
        [I, I, I, I, I, L, L] + [P, L, L] * 4 + [P, P, P, L, I, I, I, F, F] + DR +
        [P, L, L, P] + [P, L, L] * 3 + [P, ctypes.c_size_t, P, P])
    lib.attn_varlen_bwd_dropout.restype = I
    DRM = DR + [P, ctypes.c_size_t]  # ... plus the keep mask and its size
    lib.attn_varlen_fvjp_fwd_bwd_dropout_mask.argtypes = (
        [I, I, I, I, I, L, L] + [P, L, L] * 4 + [P, P, P, L, I, I, I, F, F] + DRM +
        [P, L, L] * 4 + [P, P, ctypes.c_size_t, P, P])
    lib.attn_varlen_fvjp_fwd_bwd_dropout_mask.restype = I
    lib.attn_varlen_fwd_dropout_mask.argtypes = (
        [I, I, I, I, I, L, L] + [P, L, L] * 3 + [P, P, P, L, I, I, I, F, F] + DRM + [P, L, L] +
        [P, P, ctypes.c_size_t, P, P])
    lib.attn_varlen_fwd_dropout_mask.restype = I
    lib.attn_varlen_bwd_dropout_mask.argtypes = (
        [I, I, I, I, I, L, L] + [P, L, L] * 4 + [P, P, P, L, I, I, I, F, F] + DRM +
        [P, L, L, P] + [P, L, L] * 3 + [P, ctypes.c_size_t, P, P])
    lib.attn_varlen_bwd_dropout_mask.restype = I
    lib.attn_varlen_dropout_mask_bytes.argtypes = [I, P, P, I, I]
    lib.attn_varlen_dropout_mask_bytes.restype = ctypes.c_size_t
    lib.attn_varlen_gated_fvjp_fwd_bwd.argtypes = (
        [I, I, I, I, I, I, L, L] + [P, L, L] * 6 + [P, P, P, L, I, I, I, F] + [P, L, L] * 6 +
        [P, P, ctypes.c_size_t, P, P])
    lib.attn_varlen_gated_fvjp_fwd_bwd.restype = I
    lib.attn_varlen_gated_fwd.argtypes = (
        [I, I, I, I, I, I, L, L] + [P, L, L] * 5 + [P, P, P, L, I, I, I, F] + [P, L, L] +
        [P, P, ctypes.c_size_t, P, P])
    lib.attn_varlen_gated_fwd.restype = I
    lib.attn_varlen_shard_plan.argtypes = [I, P, P, I, I, I, I, I, I, I, P, P, P, P, P]
    lib.attn_varlen_shard_plan.restype = I
    lib.attn_varlen_sum_partials.argtypes = [I, I, P, L, I, L, P, L, P]
    lib.attn_varlen_sum_partials.restype = I
    lib.attn_varlen_fvjp_record_events.argtypes = [P, I]
    lib.attn_varlen_fvjp_record_events.restype = I
    _lib = lib
    return lib


def workspace_size(B: int, Hq: int, total_q: int, total_k: int) -> int:
    return int(load().attn_varlen_fvjp_workspace_size(B, Hq, total_q, total_k))


def launch_count(B: int, Hq: int, total_q: int, total_k: int, Hkv: int = 1, mode: int = 3) -> int:
    """Kernel launches of one call (mode 1 forward, 2 backward, 3 fused)."""
    return int(load().attn_varlen_launch_count(mode, B, Hq, Hkv, total_q, total_k))


def record_events_next_call(events):
    """Arm the library's one-shot timing hook for the next call on this host
    thread: ``events`` is a list of 6 torch.cuda.Event (created with timing)."""
    lib = load()
    if len(events) != 6 or any(e.cuda_event == 0 for e in events):
        raise ValueError("need 6 created events (torch creates an event at its first record())")
    arr = (ctypes.c_void_p * 6)(*[e.cuda_event for e in events])
    code = lib.attn_varlen_fvjp_record_events(arr, 6)
    if code != 0:
        raise AttnError(code, lib.attn_status_string(code).decode())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dropout_args(dropout_seed, dropout_rate, dropout_rates, Tq):
    """(seed, rate, rates pointer) for the dropout entry points; rates is an
    fp32 CUDA vector of one rate per query token, or None."""
    if dropout_rates is not None:
        if (not dropout_rates.is_cuda or dropout_rates.dtype != torch.float32 or
                dropout_rates.shape != (Tq,) or not dropout_rates.is_contiguous()):
            raise ValueError("dropout_rates must be a contiguous fp32 CUDA vector [T_q]")
    return [int(dropout_seed) & 0xFFFFFFFFFFFFFFFF, float(dropout_rate), _ptr(dropout_rates)]


def _kv_heads(q, k):
    """Hkv of a call: k's head count, which must divide q's (and k's head
    dimension must be q's)."""
    Hkv = k.shape[1] if k.dim() == 3 else 1
    if Hkv < 1 or q.shape[1] % Hkv:
        raise ValueError(f"q's {q.shape[1]} heads are not a multiple of k's {Hkv}")
    if k.shape[-1] != q.shape[-1]:
        raise ValueError("q and k must have the same head dimension")
    return Hkv


def _check_qlike(name, t, dtype, Hq=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if t.dim() != 3 or t.shape[-1] not in HEAD_DIMS or t.stride(-1) != 1:
        raise ValueError(f"{name} must be [tokens, heads, d] (d in {HEAD_DIMS}) with a "
                         "contiguous feature axis")
    if Hq is not None and t.shape[1] != Hq:
        raise ValueError(f"{name} must have {Hq} heads")


def _like(x: torch.Tensor) -> torch.Tensor:
    """A dense tensor of x's shape and dtype on x's device."""
    return torch.empty(x.shape, dtype=x.dtype, device=x.device)


def attention_varlen_fvjp(q, k, v, cu_q, cu_k, alibi_slopes, dout, causal=False,
                          window_left=-1, window_right=-1, softcap=3.0, scale_multiplier=0.75,
                          out=None, dq=None, dk=None, dv=None, lse=None, workspace=None,
                          stream=None, dropout_seed=None, dropout_rate=0.0, dropout_rates=None,
                          keep_mask=None):
    """Forward + full VJP in one library call.

    q, dout: [T_q, Hq, d]; k, v: [T_k, Hkv, d] CUDA views (fp16 or bf16,
    d in 64/128/160 -- 160 is the pages' case, as is Hkv = 1 -- Hq a multiple
    of Hkv, any token/head strides that are multiples of 8 elements).  cu_q, cu_k: int32
    [B+1] on the device.  alibi_slopes: fp32 [B, Hq] or None.  Outputs may be
    passed in (any strides of the same rules); otherwise dense ones are
    allocated.  Returns dict(out, dq, dk, dv, lse, workspace).  The call is
    asynchronous on ``stream`` (default: the current stream).  With a
    ``dropout_seed`` the attention weights get counter-based dropout at
    ``dropout_rate`` (or per query token from ``dropout_rates``); with a
    ``keep_mask`` (uint8 CUDA buffer of dropout_mask_bytes) the forward stores
    the keep bits there and the backward reads them instead of hashing again
    (bitwise the same results)."""
    lib = load()
    dtype = q.dtype
    if dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("q must be fp16 or bf16")
    Hq = q.shape[1]
    Hkv = _kv_heads(q, k)
    _check_qlike("q", q, dtype)
    _check_qlike("dout", dout, dtype, Hq)
    _check_qlike("k", k, dtype, Hkv)
    _check_qlike("v", v, dtype, Hkv)
    if dout.shape[0] != q.shape[0] or v.shape[0] != k.shape[0]:
        raise ValueError("dout must match q and v must match k in length")
    for name, c in (("cu_q", cu_q), ("cu_k", cu_k)):
        if not c.is_cuda or c.dtype != torch.int32 or c.dim() != 1 or not c.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA vector")
    B = cu_q.numel() - 1
    if cu_k.numel() != B + 1:
        raise ValueError("cu_q and cu_k must have the same length")
    if alibi_slopes is not None:
        if (not alibi_slopes.is_cuda or alibi_slopes.dtype != torch.float32 or
                alibi_slopes.shape != (B, Hq) or alibi_slopes.stride(1) != 1):
            raise ValueError("alibi_slopes must be fp32 [B, Hq] on the device, head stride 1")
    Tq, Tk = q.shape[0], k.shape[0]
    out = _like(q) if out is None else out
    dq = _like(q) if dq is None else dq
    dk = _like(k) if dk is None else dk
    dv = _like(v) if dv is None else dv
    for name, t, H in (("out", out, Hq), ("dq", dq, Hq), ("dk", dk, Hkv), ("dv", dv, Hkv)):
        _check_qlike(name, t, dtype, H)
    if lse is None:
        lse = torch.empty((Tq, Hq), dtype=torch.float32, device=q.device)
    ws_bytes = workspace_size(B, Hq, Tq, Tk)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    drop = ([] if dropout_seed is None else
            _dropout_args(dropout_seed, dropout_rate, dropout_rates, Tq))
    fn, drop = _drop_fn(lib, "attn_varlen_fvjp_fwd_bwd", drop, keep_mask)
    code = fn(
        ATTN_BF16 if dtype == torch.bfloat16 else ATTN_F16, B, Hq, Hkv, q.shape[-1], Tq, Tk,
        _ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), k.stride(1),
        _ptr(v), v.stride(0), v.stride(1), _ptr(dout), dout.stride(0), dout.stride(1),
        _ptr(cu_q), _ptr(cu_k), _ptr(alibi_slopes),
        alibi_slopes.stride(0) if alibi_slopes is not None else 0,
        int(bool(causal)), int(window_left), int(window_right), float(softcap),
        float(scale_multiplier), *drop,
        _ptr(out), out.stride(0), out.stride(1), _ptr(dq), dq.stride(0), dq.stride(1),
        _ptr(dk), dk.stride(0), dk.stride(1), _ptr(dv), dv.stride(0), dv.stride(1),
        _ptr(lse), _ptr(workspace), workspace.numel(), None, stream.cuda_stream)
    if code != 0:
        raise AttnError(code, lib.attn_status_string(code).decode())
    return dict(out=out, dq=dq, dk=dk, dv=dv, lse=lse, workspace=workspace)


def _check_common(q, k, v, cu_q, cu_k, alibi_slopes, dout=None):
    """Validate the inputs shared by every entry point; returns (dtype, B, Hq)."""
    dtype = q.dtype
    if dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("q must be fp16 or bf16")
    Hq = q.shape[1]
    Hkv = _kv_heads(q, k)
    _check_qlike("q", q, dtype)
    _check_qlike("k", k, dtype, Hkv)
    _check_qlike("v", v, dtype, Hkv)
    if v.shape[0] != k.shape[0]:
        raise ValueError("v must match k in length")
    if dout is not None:
        _check_qlike("dout", dout, dtype, Hq)
        if dout.shape[0] != q.shape[0]:
            raise ValueError("dout must match q in length")
    for name, c in (("cu_q", cu_q), ("cu_k", cu_k)):
        if not c.is_cuda or c.dtype != torch.int32 or c.dim() != 1 or not c.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA vector")
    B = cu_q.numel() - 1
    if cu_k.numel() != B + 1:
        raise ValueError("cu_q and cu_k must have the same length")
    if alibi_slopes is not None:
        if (not alibi_slopes.is_cuda or alibi_slopes.dtype != torch.float32 or
                alibi_slopes.shape != (B, Hq) or alibi_slopes.stride(1) != 1):
            raise ValueError("alibi_slopes must be fp32 [B, Hq] on the device, head stride 1")
    return dtype, B, Hq, Hkv


def _workspace(workspace, B, Hq, Tq, Tk, device):
    ws_bytes = workspace_size(B, Hq, Tq, Tk)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
    return workspace


def attention_varlen_fwd(q, k, v, cu_q, cu_k, alibi_slopes, causal=False, window_left=-1,
                         window_right=-1, softcap=3.0, scale_multiplier=0.75, out=None, lse=None,
                         workspace=None, stream=None, dropout_seed=None, dropout_rate=0.0,
                         dropout_rates=None, keep_mask=None):
    """Forward only: returns (out, lse).  Same argument rules as
    attention_varlen_fvjp; lse is fp32 [T_q, Hq] (natural log), the value the
    backward call reads back.  Asynchronous on ``stream``."""
    lib = load()
    dtype, B, Hq, Hkv = _check_common(q, k, v, cu_q, cu_k, alibi_slopes)
    Tq, Tk = q.shape[0], k.shape[0]
    out = _like(q) if out is None else out
    _check_qlike("out", out, dtype, Hq)
    if lse is None:
        lse = torch.empty((Tq, Hq), dtype=torch.float32, device=q.device)
    _check_lse(lse, Tq, Hq)
    workspace = _workspace(workspace, B, Hq, Tq, Tk, q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    drop = ([] if dropout_seed is None else
            _dropout_args(dropout_seed, dropout_rate, dropout_rates, Tq))
    fn, drop = _drop_fn(lib, "attn_varlen_fwd", drop, keep_mask)
    code = fn(
        ATTN_BF16 if dtype == torch.bfloat16 else ATTN_F16, B, Hq, Hkv, q.shape[-1], Tq, Tk,
        _ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), k.stride(1),
        _ptr(v), v.stride(0), v.stride(1),
        _ptr(cu_q), _ptr(cu_k), _ptr(alibi_slopes),
        alibi_slopes.stride(0) if alibi_slopes is not None else 0,
        int(bool(causal)), int(window_left), int(window_right), float(softcap),
        float(scale_multiplier), *drop, _ptr(out), out.stride(0), out.stride(1),
        _ptr(lse), _ptr(workspace), workspace.numel(), None, stream.cuda_stream)
    if code != 0:
        raise AttnError(code, lib.attn_status_string(code).decode())
    return out, lse


def attention_varlen_bwd(q, k, v, cu_q, cu_k, alibi_slopes, dout, out, lse, causal=False,
                         window_left=-1, window_right=-1, softcap=3.0, scale_multiplier=0.75,
                         dq=None, dk=None, dv=None, workspace=None, stream=None,
                         dropout_seed=None, dropout_rate=0.0, dropout_rates=None,
                         keep_mask=None):
    """Backward only: given the forward's out and lse for the same inputs and
    options, returns (dq, dk, dv).  out and lse are read, not modified.  For
    the same inputs the result is bitwise the one attention_varlen_fvjp gives.
    Asynchronous on ``stream``."""
    lib = load()
    dtype, B, Hq, Hkv = _check_common(q, k, v, cu_q, cu_k, alibi_slopes, dout)
    Tq, Tk = q.shape[0], k.shape[0]
    _check_qlike("out", out, dtype, Hq)
    if out.shape[0] != Tq:
        raise ValueError("out must match q in length")
    _check_lse(lse, Tq, Hq)
    dq = _like(q) if dq is None else dq
    dk = _like(k) if dk is None else dk
    dv = _like(v) if dv is None else dv
    for name, t, H in (("dq", dq, Hq), ("dk", dk, Hkv), ("dv", dv, Hkv)):
        _check_qlike(name, t, dtype, H)
    workspace = _workspace(workspace, B, Hq, Tq, Tk, q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    drop = ([] if dropout_seed is None else
            _dropout_args(dropout_seed, dropout_rate, dropout_rates, Tq))
    fn, drop = _drop_fn(lib, "attn_varlen_bwd", drop, keep_mask)
    code = fn(
        ATTN_BF16 if dtype == torch.bfloat16 else ATTN_F16, B, Hq, Hkv, q.shape[-1], Tq, Tk,
        _ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), k.stride(1),
        _ptr(v), v.stride(0), v.stride(1), _ptr(dout), dout.stride(0), dout.stride(1),
        _ptr(cu_q), _ptr(cu_k), _ptr(alibi_slopes),
        alibi_slopes.stride(0) if alibi_slopes is not None else 0,
        int(bool(causal)), int(window_left), int(window_right), float(softcap),
        float(scale_multiplier), *drop, _ptr(out), out.stride(0), out.stride(1), _ptr(lse),
        _ptr(dq), dq.stride(0), dq.stride(1), _ptr(dk), dk.stride(0), dk.stride(1),
        _ptr(dv), dv.stride(0), dv.stride(1),
        _ptr(workspace), workspace.numel(), None, stream.cuda_stream)
    if code != 0:
        raise AttnError(code, lib.attn_status_string(code).decode())
    return dq, dk, dv


def dropout_mask_bytes(cu_q, cu_k, Hq: int, Hkv: int = 1) -> int:
    """Bytes of keep mask the stored-mask dropout calls need for these lengths
    (cu_q, cu_k: int32 [B+1], host or device)."""
    cq = cu_q.detach().to("cpu", torch.int32).contiguous()
    ck = cu_k.detach().to("cpu", torch.int32).contiguous()
    n = int(load().attn_varlen_dropout_mask_bytes(cq.numel() - 1, _ptr(cq), _ptr(ck), Hq, Hkv))
    if n == 0:
        raise ValueError("invalid lengths or heads for the keep mask")
    return n


def _mask_args(keep_mask):
    """(pointer, bytes) of a keep-mask buffer: a CUDA uint8 tensor."""
    if not keep_mask.is_cuda or keep_mask.dtype != torch.uint8 or not keep_mask.is_contiguous():
        raise ValueError("keep_mask must be a contiguous uint8 CUDA tensor")
    return [_ptr(keep_mask), keep_mask.numel()]


def _drop_fn(lib, name, drop, keep_mask):
    """The entry point and its dropout arguments: plain, dropout, or dropout
    with the stored keep mask."""
    if not drop:
        if keep_mask is not None:
            raise ValueError("keep_mask needs a dropout_seed")
        return getattr(lib, name), []
    if keep_mask is None:
        return getattr(lib, name + "_dropout"), drop
    return getattr(lib, name + "_dropout_mask"), drop + _mask_args(keep_mask)


def _check_lse(lse, Tq, Hq):
    if (not lse.is_cuda or lse.dtype != torch.float32 or lse.shape != (Tq, Hq) or
            not lse.is_contiguous()):
        raise ValueError(f"lse must be a contiguous fp32 [{Tq}, {Hq}] CUDA tensor")


def host_buffer_size_for(cu_q, cu_k, Hq: int, Hkv: int, d: int, chunks: int) -> int:
    """Device buffer bytes of the host-buffer call for these lengths (host
    int32 cu arrays)."""
    cq = cu_q.detach().to("cpu", torch.int32).contiguous()
    ck = cu_k.detach().to("cpu", torch.int32).contiguous()
    return int(load().attn_varlen_fvjp_host_buffer_size_for(cq.numel() - 1, _ptr(cq), _ptr(ck),
                                                            Hq, Hkv, d, chunks))


def host_buffer_size(B: int, Hq: int, Hkv: int, d: int, total_q: int, total_k: int,
                     chunks: int) -> int:
    return int(load().attn_varlen_fvjp_host_buffer_size(B, Hq, Hkv, d, total_q, total_k, chunks))


def host_chunks(cu_q, cu_k, chunks: int):
    """Sequence boundaries of the host-buffer entry point's chunks (host int32
    cu tensors)."""
    B = cu_q.numel() - 1
    cuts = torch.zeros(chunks + 1, dtype=torch.int32)
    n = load().attn_varlen_host_chunks(B, _ptr(cu_q), _ptr(cu_k), chunks, _ptr(cuts))
    return cuts[:n + 1].tolist()


def _check_host(name, t, dtype, H):
    if t.is_cuda or t.dtype != dtype or t.dim() != 3 or t.shape[1] != H or t.stride(-1) != 1:
        raise ValueError(f"{name} must be a host [tokens, {H}, d] {dtype} tensor with a "
                         "contiguous feature axis")


def attention_varlen_fvjp_host(q, k, v, cu_q, cu_k, alibi_slopes, dout, causal=False,
                               window_left=-1, window_right=-1, softcap=3.0,
                               scale_multiplier=0.75, chunks=4, out=None, dq=None, dk=None,
                               dv=None, lse=None, device_buffer=None, host_status=None,
                               device=None, stream=None):
    """The fused call on HOST tensors (pinned for asynchronous copies): the
    library copies ``chunks`` runs of whole sequences to the device, computes
    and copies the results back, overlapping the copies with the kernels.
    cu_q, cu_k (int32) and alibi_slopes (fp32 [B, Hq] or None) are host
    tensors too.  Outputs (host) may be passed in; otherwise pinned ones are
    allocated.  Returns dict(out, dq, dk, dv, lse, status, device_buffer); the
    results are complete once ``stream`` has passed the call (synchronise
    before reading them), and ``status`` then holds one device status word per
    chunk."""
    lib = load()
    dtype = q.dtype
    if dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("q must be fp16 or bf16")
    Hq, Hkv, d = q.shape[1], k.shape[1], q.shape[-1]
    if d not in HEAD_DIMS or Hq % Hkv or k.shape[-1] != d:
        raise ValueError("bad head dimension or head split")
    for name, t, H in (("q", q, Hq), ("dout", dout, Hq), ("k", k, Hkv), ("v", v, Hkv)):
        _check_host(name, t, dtype, H)
    for name, c in (("cu_q", cu_q), ("cu_k", cu_k)):
        if c.is_cuda or c.dtype != torch.int32 or c.dim() != 1 or not c.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 host vector")
    B = cu_q.numel() - 1
    Tq, Tk = q.shape[0], k.shape[0]
    if alibi_slopes is not None and (alibi_slopes.is_cuda or alibi_slopes.dtype != torch.float32
                                     or alibi_slopes.shape != (B, Hq)
                                     or alibi_slopes.stride(1) != 1):
        raise ValueError("alibi_slopes must be a host fp32 [B, Hq] tensor, head stride 1")
    pin = dict(dtype=dtype, pin_memory=True)
    out = torch.empty(q.shape, **pin) if out is None else out
    dq = torch.empty(q.shape, **pin) if dq is None else dq
    dk = torch.empty(k.shape, **pin) if dk is None else dk
    dv = torch.empty(v.shape, **pin) if dv is None else dv
    for name, t, H in (("out", out, Hq), ("dq", dq, Hq), ("dk", dk, Hkv), ("dv", dv, Hkv)):
        _check_host(name, t, dtype, H)
    if lse is None:
        lse = torch.empty((Tq, Hq), dtype=torch.float32, pin_memory=True)
    if lse.is_cuda or lse.dtype != torch.float32 or lse.shape != (Tq, Hq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous host fp32 [T_q, Hq] tensor")
    if host_status is None:
        host_status = torch.zeros(chunks, dtype=torch.int32, pin_memory=True)
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    nbytes = host_buffer_size_for(cu_q, cu_k, Hq, Hkv, d, chunks)
    if device_buffer is None:
        device_buffer = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if stream is None:
        stream = torch.cuda.current_stream(device)
    code = lib.attn_varlen_fvjp_fwd_bwd_host(
        ATTN_BF16 if dtype == torch.bfloat16 else ATTN_F16, B, Hq, Hkv, d, Tq, Tk,
        _ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), k.stride(1),
        _ptr(v), v.stride(0), v.stride(1), _ptr(dout), dout.stride(0), dout.stride(1),
        _ptr(cu_q), _ptr(cu_k), _ptr(alibi_slopes),
        alibi_slopes.stride(0) if alibi_slopes is not None else 0,
        int(bool(causal)), int(window_left), int(window_right), float(softcap),
        float(scale_multiplier),
        _ptr(out), out.stride(0), out.stride(1), _ptr(dq), dq.stride(0), dq.stride(1),
        _ptr(dk), dk.stride(0), dk.stride(1), _ptr(dv), dv.stride(0), dv.stride(1),
        _ptr(lse), _ptr(device_buffer), device_buffer.numel(), int(chunks), _ptr(host_status),
        stream.cuda_stream)
    if code != 0:
        raise AttnError(code, lib.attn_status_string(code).decode())
    return dict(out=out, dq=dq, dk=dk, dv=dv, lse=lse, status=host_status,
                device_buffer=device_buffer)


def attention_varlen_fvjp_noalloc(q, k, v, cu_q, cu_k, alibi_slopes, dout, out, dq, dk, dv, lse,
                                  device_status, causal=False, window_left=-1, window_right=-1,
                                  softcap=3.0, scale_multiplier=0.75, stream=None):
    """The library's no-allocation entry point: the caller passes every input
    and output (plus an int32 device status word); the library uses its own
    fixed scratch array instead of a workspace, for callers that may not
    allocate device memory.  Asynchronous on ``stream``."""
    lib = load()
    dtype = q.dtype
    Hq = q.shape[1]
    Hkv = _kv_heads(q, k)
    for name, t, H in (("q", q, Hq), ("dout", dout, Hq), ("k", k, Hkv), ("v", v, Hkv),
                       ("out", out, Hq), ("dq", dq, Hq), ("dk", dk, Hkv), ("dv", dv, Hkv)):
        _check_qlike(name, t, dtype, H)
    B = cu_q.numel() - 1
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    # the library uses the scratch array of the current device
    with torch.cuda.device(q.device):
        code = _noalloc_call(lib, q, k, v, cu_q, cu_k, alibi_slopes, dout, out, dq, dk, dv, lse,
                             device_status, causal, window_left, window_right, softcap,
                             scale_multiplier, stream, dtype, B, Hq, Hkv)
    if code != 0:
        raise AttnError(code, lib.attn_status_string(code).decode())


def _noalloc_call(lib, q, k, v, cu_q, cu_k, alibi_slopes, dout, out, dq, dk, dv, lse,
                  device_status, causal, window_left, window_right, softcap, scale_multiplier,
                  stream, dtype, B, Hq, Hkv):
    return lib.attn_varlen_fvjp_fwd_bwd_noalloc(
        ATTN_BF16 if dtype == torch.bfloat16 else ATTN_F16, B, Hq, Hkv, q.shape[-1], q.shape[0],
        k.shape[0], _ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), k.stride(1),
        _ptr(v), v.stride(0), v.stride(1), _ptr(dout), dout.stride(0), dout.stride(1),
        _ptr(cu_q), _ptr(cu_k), _ptr(alibi_slopes),
        alibi_slopes.stride(0) if alibi_slopes is not None else 0,
        int(bool(causal)), int(window_left), int(window_right), float(softcap),
        float(scale_multiplier),
        _ptr(out), out.stride(0), out.stride(1), _ptr(dq), dq.stride(0), dq.stride(1),
        _ptr(dk), dk.stride(0), dk.stride(1), _ptr(dv), dv.stride(0), dv.stride(1),
        _ptr(lse), _ptr(device_status), stream.cuda_stream)


def attention_varlen_gated(q, k, v, q_gate, k_gate, cu_q, cu_k, alibi_slopes, dout=None,
                           causal=False, window_left=-1, window_right=-1, scale_multiplier=1.0,
                           out=None, dq=None, dk=None, dv=None, dq_gate=None, dk_gate=None,
                           lse=None, workspace=None, stream=None):
    """The sigmoid-gated call: with ``dout`` the fused forward and backward
    (returns out, lse, dq, dk, dv, dq_gate, dk_gate, workspace), without it
    the forward only (out, lse, workspace).  Head dimension 64 or 128, gate
    width a multiple of 8 up to 64; no softcap (the gated page's plain
    softmax)."""
    lib = load()
    dtype = q.dtype
    Hq, R = q.shape[1], q_gate.shape[-1]
    Hkv = _kv_heads(q, k)
    for name, t, H in (("q", q, Hq), ("k", k, Hkv), ("v", v, Hkv)):
        _check_qlike(name, t, dtype, H)
    for name, t, H in (("q_gate", q_gate, Hq), ("k_gate", k_gate, Hkv)):
        if not t.is_cuda or t.dtype != dtype or t.dim() != 3 or t.shape[1] != H or \
                t.stride(-1) != 1 or t.shape[-1] != R:
            raise ValueError(f"{name} must be a CUDA [tokens, {H}, R] tensor of {dtype} with a "
                             "contiguous last axis")
    B = cu_q.numel() - 1
    Tq, Tk, d = q.shape[0], k.shape[0], q.shape[-1]
    out = _like(q) if out is None else out
    lse = torch.empty((Tq, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    if workspace is None:
        workspace = torch.empty(max(workspace_size(B, Hq, Tq, Tk), 256), dtype=torch.uint8,
                                device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    code_dt = ATTN_BF16 if dtype == torch.bfloat16 else ATTN_F16
    head = [code_dt, B, Hq, Hkv, d, R, Tq, Tk, _ptr(q), q.stride(0), q.stride(1), _ptr(k),
            k.stride(0), k.stride(1), _ptr(v), v.stride(0), v.stride(1)]
    gates = [_ptr(q_gate), q_gate.stride(0), q_gate.stride(1), _ptr(k_gate), k_gate.stride(0),
             k_gate.stride(1)]
    mid = [_ptr(cu_q), _ptr(cu_k), _ptr(alibi_slopes),
           alibi_slopes.stride(0) if alibi_slopes is not None else 0, int(bool(causal)),
           int(window_left), int(window_right), float(scale_multiplier)]
    tail = [_ptr(lse), _ptr(workspace), workspace.numel(), None, stream.cuda_stream]
    if dout is None:
        code = lib.attn_varlen_gated_fwd(*head, *gates, *mid, _ptr(out), out.stride(0),
                                         out.stride(1), *tail)
        if code != 0:
            raise AttnError(code, lib.attn_status_string(code).decode())
        return dict(out=out, lse=lse, workspace=workspace)
    _check_qlike("dout", dout, dtype, Hq)
    dq = _like(q) if dq is None else dq
    dk = _like(k) if dk is None else dk
    dv = _like(v) if dv is None else dv
    dq_gate = _like(q_gate) if dq_gate is None else dq_gate
    dk_gate = _like(k_gate) if dk_gate is None else dk_gate
    code = lib.attn_varlen_gated_fvjp_fwd_bwd(
        *head, _ptr(dout), dout.stride(0), dout.stride(1), *gates, *mid,
        _ptr(out), out.stride(0), out.stride(1), _ptr(dq), dq.stride(0), dq.stride(1),
        _ptr(dk), dk.stride(0), dk.stride(1), _ptr(dv), dv.stride(0), dv.stride(1),
        _ptr(dq_gate), dq_gate.stride(0), dq_gate.stride(1),
        _ptr(dk_gate), dk_gate.stride(0), dk_gate.stride(1), *tail)
    if code != 0:
        raise AttnError(code, lib.attn_status_string(code).decode())
    return dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv, dq_gate=dq_gate, dk_gate=dk_gate,
                workspace=workspace)


def shard_plan(cu_q, cu_k, Hq: int, Hkv: int, nranks: int, causal=False, window_left=-1,
               window_right=-1):
    """The library's shard plan of one batch over ``nranks`` processes: a list
    of units (sequence, first head, end head, rank) in (sequence, head) order
    and the work of each rank.  cu arrays may live on any device (read on the
    host)."""
    lib = load()
    cq = cu_q.detach().to("cpu", torch.int32).contiguous()
    ck = cu_k.detach().to("cpu", torch.int32).contiguous()
    B = cq.numel() - 1
    cap = B + (nranks - 1) ** 2 + 1
    bufs = [torch.empty(cap, dtype=torch.int32) for _ in range(4)]
    work = torch.empty(max(nranks, 1), dtype=torch.float64)
    n = lib.attn_varlen_shard_plan(B, _ptr(cq), _ptr(ck), Hq, Hkv, int(bool(causal)),
                                   int(window_left), int(window_right), nranks, cap,
                                   *[_ptr(b) for b in bufs], _ptr(work))
    if n < 0:
        raise ValueError("attn_varlen_shard_plan rejected its arguments")
    units = [tuple(int(b[u]) for b in bufs) for u in range(n)]
    return units, work.tolist()


def sum_partials(parts, out, stream=None):
    """out = parts[0] + parts[1] + ... (in this order, fp32 accumulation, one
    rounding): 16-bit [rows, (1,) d] tensors with a contiguous feature axis."""
    lib = load()
    d = out.shape[-1]
    rows = out.shape[0]
    assert out.dim() == 2 or (out.dim() == 3 and out.shape[1] == 1), "one K/V head"
    for t in parts:
        assert t.dtype == out.dtype and t.shape == out.shape and t.device == out.device
        assert t.stride(-1) == 1
    assert out.stride(-1) == 1
    if stream is None:
        stream = torch.cuda.current_stream(out.device)
    arr = (ctypes.c_void_p * len(parts))(*[t.data_ptr() for t in parts])
    code = lib.attn_varlen_sum_partials(
        ATTN_BF16 if out.dtype == torch.bfloat16 else ATTN_F16, len(parts), arr, rows, d,
        parts[0].stride(0), _ptr(out), out.stride(0), stream.cuda_stream)
    if code != 0:
        raise AttnError(code, lib.attn_status_string(code).decode())


def device_status(workspace: torch.Tensor) -> int:
    """Synchronise and read the call's device status word (0 = clean)."""
    return int(workspace[:4].view(torch.int32).item())


def attention_varlen_feature_full_vjp(q, k, v, cu_q, cu_k, alibi_slopes, dout, causal=False,
                                      window_left=-1, window_right=-1, softcap=3.0,
                                      scale_multiplier=0.75):
    """The pages' entry point: returns (out, dq, dk, dv) with the inputs' shapes
    and dtypes ("Noncausal Global Extreme-GQA Ragged Attention Full VJP",
    "Hard Constraints").  cu arrays of another integer type are converted to
    int32; inputs are never modified."""
    if cu_q.dtype != torch.int32:
        cu_q = cu_q.to(torch.int32)
    if cu_k.dtype != torch.int32:
        cu_k = cu_k.to(torch.int32)
    if k.dim() == 2:
        k = k.unsqueeze(1)
    if v.dim() == 2:
        v = v.unsqueeze(1)
    r = attention_varlen_fvjp(q, k, v, cu_q.contiguous(), cu_k.contiguous(), alibi_slopes, dout,
                              causal, window_left, window_right, softcap, scale_multiplier)
    return r["out"], r["dq"], r["dk"], r["dv"]

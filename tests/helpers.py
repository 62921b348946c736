"""Shared test helpers: tolerance checks against the fp64 oracle."""
import math

import torch

# Tolerances stated for the hot path: relative Frobenius error <= 1e-2 (fp16)
# or <= 2e-2 (bf16), max-abs error <= 5e-2 * max|ref| on out/dq/dk/dv, and the
# log-sum-exp within 1e-3 (absolute) on finite rows; -inf rows match exactly.
REL_FRO = {torch.float16: 1e-2, torch.bfloat16: 2e-2}
MAX_ABS_FRAC = 5e-2
LSE_ATOL = 1e-3
# A reference that is identically zero (e.g. dq and dk when a sequence has a
# single key: dZ = P (dP - D) vanishes exactly in exact arithmetic) has no
# scale for a relative bound; the GPU's fp32 accumulations leave rounding
# noise there, held to this absolute bound.
ZERO_ATOL = 1e-4


def rel_fro(x: torch.Tensor, ref: torch.Tensor) -> float:
    x = x.double()
    ref = ref.double()
    den = float(torch.linalg.vector_norm(ref))
    num = float(torch.linalg.vector_norm(x - ref))
    return num / den if den > 0 else num


def check_tensor(name, x, ref, dtype):
    """x: GPU result (any float type, moved to CPU); ref: oracle fp64."""
    x = x.detach().cpu().double()
    ref = ref.detach().cpu().double()
    assert x.shape == ref.shape, (name, x.shape, ref.shape)
    assert torch.isfinite(x).all(), f"{name}: non-finite values"
    rf = rel_fro(x, ref)
    amax = float(ref.abs().max()) if ref.numel() else 0.0
    mad = float((x - ref).abs().max()) if ref.numel() else 0.0
    if amax == 0:
        assert mad <= ZERO_ATOL, f"{name}: zero reference, max-abs {mad:.3e} > {ZERO_ATOL}"
        return rf, mad
    assert rf <= REL_FRO[dtype], f"{name}: rel-Frobenius {rf:.3e} > {REL_FRO[dtype]}"
    assert mad <= MAX_ABS_FRAC * amax, f"{name}: max-abs {mad:.3e} > {MAX_ABS_FRAC} * {amax:.3e}"
    return rf, mad


def check_lse(lse, ref):
    lse = lse.detach().cpu().double()
    ref = ref.detach().cpu().double()
    inf_ref = torch.isinf(ref)
    assert torch.equal(torch.isinf(lse), inf_ref), "lse: -inf rows differ"
    if inf_ref.any():
        assert torch.all(lse[inf_ref] == ref[inf_ref])
    fin = ~inf_ref
    if fin.any():
        err = float((lse[fin] - ref[fin]).abs().max())
        assert err <= LSE_ATOL, f"lse: max abs error {err:.3e} > {LSE_ATOL}"
        return err
    return 0.0


def check_all(res, ref, dtype, rows=None, keys=None):
    """Compare a GPU result dict with an oracle dict, optionally restricted to
    packed query rows / key rows (index tensors)."""
    report = {}
    sel_q = (lambda t: t) if rows is None else (lambda t: t[rows])
    sel_k = (lambda t: t) if keys is None else (lambda t: t[keys])
    report["out"] = check_tensor("out", sel_q(res["out"].cpu()), sel_q(ref["out"]), dtype)
    report["dq"] = check_tensor("dq", sel_q(res["dq"].cpu()), sel_q(ref["dq"]), dtype)
    report["dk"] = check_tensor("dk", sel_k(res["dk"].cpu()), sel_k(ref["dk"]), dtype)
    report["dv"] = check_tensor("dv", sel_k(res["dv"].cpu()), sel_k(ref["dv"]), dtype)
    report["lse"] = check_lse(sel_q(res["lse"].cpu()), sel_q(ref["lse"]))
    return report


def view_bytes_hash(t: torch.Tensor) -> int:
    """Hash of a tensor's whole underlying storage (catches writes to padding)."""
    st = t.untyped_storage()
    raw = torch.empty(0, dtype=torch.uint8, device=t.device).set_(st).cpu()
    return hash(raw.numpy().tobytes())


def row_mask(p, seqs):
    """Boolean masks of the packed query rows / key rows of sequences `seqs`."""
    mq = torch.zeros(p.total_q, dtype=torch.bool)
    mk = torch.zeros(p.total_k, dtype=torch.bool)
    for b in seqs:
        mq[int(p.cu_q[b]):int(p.cu_q[b + 1])] = True
        mk[int(p.cu_k[b]):int(p.cu_k[b + 1])] = True
    return mq, mk


def nan_like_strided(x: torch.Tensor) -> torch.Tensor:
    """A tensor with x's shape, dtype, device and strides, NaN everywhere
    (including padding), for checking that outputs are fully written."""
    base = torch.full((x.untyped_storage().nbytes() // x.element_size(),), math.nan,
                      dtype=x.dtype, device=x.device)
    return base.as_strided(x.shape, x.stride(), x.storage_offset())

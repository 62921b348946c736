"""CPU-only checks of the C ABI: the library loads, exports every function
declared in include/attn_varlen.h, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from ragged_gqa_attention_varlen_gb300 import _build, binding

    _build.build()
    return binding.load()


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "attn_varlen_fvjp_fwd_bwd" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(0, -8, -1):
        assert lib.attn_status_string(code)
    assert lib.attn_status_string(-3).decode().startswith("pointer or stride")


def test_workspace_size_grows_with_rows(lib):
    a = lib.attn_varlen_fvjp_workspace_size(4, 16, 100, 50)
    b = lib.attn_varlen_fvjp_workspace_size(4, 16, 1000, 50)
    assert b - a >= 900 * 16 * 4
    assert a % 256 == 0 and b % 256 == 0


def _call(lib, **over):
    """A call whose arguments pass or fail host validation; the fake device
    pointers are never dereferenced because every case fails validation."""
    fake = 0x10000  # 16-byte aligned, never touched
    a = dict(dtype=0, B=2, Hq=16, Hkv=1, hd=160, tq=10, tk=12,
             q=fake, qts=16 * 160, qhs=160, k=fake, kts=160, khs=160, v=fake, vts=160, vhs=160,
             do=fake, dts=16 * 160, dhs=160, cuq=fake, cuk=fake, sl=fake, slb=16,
             causal=0, wl=-1, wr=-1, cap=3.0, sm=0.75,
             out=fake, ots=16 * 160, ohs=160, dq=fake, dqts=16 * 160, dqhs=160,
             dk=fake, dkts=160, dkhs=160, dv=fake, dvts=160, dvhs=160,
             lse=fake, ws=fake, wsb=0, st=None, stream=None)
    a.update(over)
    return lib.attn_varlen_fvjp_fwd_bwd(*a.values())


def test_host_validation_codes(lib):
    assert _call(lib, dtype=7) == -1
    assert _call(lib, hd=96) == -2              # head dims: 64, 128 and 160
    assert _call(lib, hd=128) == -4 and _call(lib, hd=64) == -4
    assert _call(lib, Hkv=3) == -1             # 16 query heads do not split over 3
    assert _call(lib, Hkv=0) == -1
    assert _call(lib, Hkv=2, khs=164) == -3     # head strides count once Hkv > 1
    assert _call(lib, Hkv=1, khs=164) == -4     # ... and are ignored for one K/V head
    assert _call(lib, Hkv=2) == -4              # a valid split reaches the workspace check
    assert _call(lib, B=20000) == -2
    assert _call(lib, q=0x10008) == -3          # base not 16-byte aligned
    assert _call(lib, qhs=164) == -3            # stride not a multiple of 8 elements
    assert _call(lib, ws=0) == -4               # no workspace
    assert _call(lib, wsb=16) == -4             # workspace too small
    assert _call(lib, B=0) == -1                # B = 0 with tokens
    assert _call(lib, q=None) == -1


def test_launch_counts(lib):
    f = lib.attn_varlen_launch_count
    assert f(3, 2, 16, 1, 10, 12) == 5 == lib.attn_varlen_fvjp_launch_count(2, 16, 10, 12)
    assert f(1, 2, 16, 1, 10, 12) == 2 and f(2, 2, 16, 1, 10, 12) == 4
    assert f(3, 2, 16, 4, 10, 12) == 1 + 4 + 1 + 2 * 4
    assert f(3, 2, 16, 4, 0, 12) == 2 and f(1, 2, 16, 4, 0, 12) == 0
    assert f(3, 2, 16, 1, 10, 0) == 3 and f(0, 2, 16, 1, 10, 12) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    """The no-allocation entry point refuses, before touching the device, a
    problem whose workspace would exceed its fixed scratch array."""
    fake = 0x10000
    big_q = (64 << 20) // (4 * 96) + 1  # D alone needs more than the scratch
    args = [0, 2, 96, 1, 160, big_q, 12,
            fake, 96 * 160, 160, fake, 160, 160, fake, 160, 160, fake, 96 * 160, 160,
            fake, fake, fake, 96, 0, -1, -1, 3.0, 0.75,
            fake, 96 * 160, 160, fake, 96 * 160, 160, fake, 160, 160, fake, 160, 160,
            fake, None, None]
    assert lib.attn_varlen_fvjp_fwd_bwd_noalloc(*args) == -8
    assert b"scratch" in lib.attn_status_string(-8)


def test_noalloc_scratch_limit_is_the_documented_formula(lib):
    """The header's size formula for the no-allocation call (status and
    counters, schedule, fp32 D; no dropout rate table) decides acceptance:
    the largest total_q that fits passes the size check, one more token is
    refused.  A misaligned q makes the accepted call stop at the host checks,
    so nothing is launched on any machine."""
    A = lambda x: (x + 255) // 256 * 256
    B, Hq, cap = 2, 96, 64 << 20

    def need(tq):
        return A(16 + 12 * max(Hq, 2)) + A(4 * (5 * B + 2)) + A(4 * tq * Hq)

    tq = (cap - need(0)) // (4 * Hq)
    while need(tq + 1) <= cap:
        tq += 1
    assert need(tq) <= cap < need(tq + 1)
    fake, bad = 0x10000, 0x10008

    def call(total_q):
        args = [0, 2, Hq, 1, 160, total_q, 12,
                bad, 96 * 160, 160, fake, 160, 160, fake, 160, 160, fake, 96 * 160, 160,
                fake, fake, fake, 96, 0, -1, -1, 3.0, 0.75,
                fake, 96 * 160, 160, fake, 96 * 160, 160, fake, 160, 160, fake, 160, 160,
                fake, None, None]
        return lib.attn_varlen_fvjp_fwd_bwd_noalloc(*args)

    assert call(tq + 1) == -8
    # past the size check: ALIGNMENT (-3) where a device exists, CUDA (-5) here
    assert call(tq) in (-3, -5)


def test_host_entry_point_validates_before_touching_the_device(lib):
    """The host-buffer entry point checks its arguments (and reads the host cu
    arrays) before any CUDA call: these all fail on a machine without a GPU
    with the documented codes."""
    import ctypes

    import numpy as np

    cu_q = np.array([0, 5, 9], dtype=np.int32)
    cu_k = np.array([0, 7, 12], dtype=np.int32)
    fake = 0x10000  # host pointers that the failing calls never dereference
    status = np.zeros(4, dtype=np.int32)

    def call(**over):
        a = dict(dtype=0, B=2, Hq=16, Hkv=1, hd=160, tq=9, tk=12,
                 q=fake, qts=16 * 160, qhs=160, k=fake, kts=160, khs=160, v=fake, vts=160,
                 vhs=160, do=fake, dts=16 * 160, dhs=160, cuq=cu_q.ctypes.data,
                 cuk=cu_k.ctypes.data, sl=None, slb=16, causal=0, wl=-1, wr=-1, cap=3.0,
                 sm=0.75, out=fake, ots=16 * 160, ohs=160, dq=fake, dqts=16 * 160, dqhs=160,
                 dk=fake, dkts=160, dkhs=160, dv=fake, dvts=160, dvhs=160, lse=fake,
                 buf=None, bufb=0, chunks=2, st=status.ctypes.data, stream=None)
        a.update(over)
        return lib.attn_varlen_fvjp_fwd_bwd_host(*a.values())

    assert call(chunks=0) == -1
    assert call(Hkv=3) == -1
    assert call(hd=96) == -2
    assert call(qts=100) == -3                 # a token pitch shorter than its heads
    bad = np.array([0, 6, 9], dtype=np.int32)
    assert call(cuk=bad.ctypes.data) == -1     # cu_k[B] != total_k
    assert call() == -4                        # no device buffer
    need = lib.attn_varlen_fvjp_host_buffer_size_for(2, cu_q.ctypes.data, cu_k.ctypes.data, 16,
                                                     1, 160, 2)
    assert need > lib.attn_varlen_fvjp_workspace_size(2, 16, 9, 12)
    assert need <= lib.attn_varlen_fvjp_host_buffer_size(2, 16, 1, 160, 9, 12, 2)
    assert call(buf=0x100000, bufb=need - 1) == -4
    # past every host check the call needs the device: on a machine without
    # one that is CUDA (-5), and host_status is left as it was (where a GPU
    # exists the fake pointers would be used, so the check stops here)
    import torch

    if not torch.cuda.is_available():
        status[:] = 7
        assert call(buf=0x100000, bufb=need) == -5
        assert (status == 7).all()


def test_host_buffer_is_slots_of_the_largest_chunk(lib):
    """The host-buffer call's device buffer holds min(4, chunks) slots sized
    for the largest chunk (the chunking's own cuts): within a few per cent
    of that many buffers of one chunk-sized sequence, far below the
    whole-batch bound, and never below a dominant sequence's own slot."""
    import numpy as np

    from ragged_gqa_attention_varlen_gb300 import binding
    import torch

    def size_for(lengths, chunks):
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        return lib.attn_varlen_fvjp_host_buffer_size_for(len(lengths), cu.ctypes.data,
                                                         cu.ctypes.data, 16, 1, 128, chunks)

    lengths = [1000] * 8
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    for chunks in (1, 2, 4, 8):
        cuts = binding.host_chunks(cu, cu, chunks)
        n = len(cuts) - 1
        largest = max(sum(lengths[a:b]) for a, b in zip(cuts, cuts[1:]))
        model = min(4, n) * size_for([largest], 1)
        assert abs(size_for(lengths, chunks) - model) <= 0.05 * model, chunks
    bound = lib.attn_varlen_fvjp_host_buffer_size(8, 16, 1, 128, 8000, 8000, 8)
    assert size_for(lengths, 8) < bound / 3
    assert size_for([7000] + [143] * 7, 8) >= size_for([7000], 1)

def test_host_chunks_cut_whole_sequences_of_balanced_work(lib):
    """The host-buffer entry point's chunking: strictly increasing sequence
    boundaries from 0 to B, at most `chunks` runs, and every run's weight
    (sum of Lq*Lk + 1) within one sequence's weight of its share: equal
    shares, except that with three chunks or more the first and the last
    take a quarter of the others'."""
    import torch

    from ragged_gqa_attention_varlen_gb300 import binding

    g = torch.Generator().manual_seed(1)
    for trial in range(200):
        B = int(torch.randint(0, 40, (1,), generator=g))
        lq = torch.randint(0, 500, (B,), generator=g)
        lk = torch.randint(0, 500, (B,), generator=g)
        cu_q = torch.cat([torch.zeros(1, dtype=torch.int64), lq.cumsum(0)]).to(torch.int32)
        cu_k = torch.cat([torch.zeros(1, dtype=torch.int64), lk.cumsum(0)]).to(torch.int32)
        chunks = int(torch.randint(1, 9, (1,), generator=g))
        cuts = binding.host_chunks(cu_q, cu_k, chunks)
        assert cuts[0] == 0 and cuts[-1] == B
        assert 1 <= len(cuts) - 1 <= max(1, min(chunks, B))
        assert all(a < b for a, b in zip(cuts, cuts[1:])) or B == 0
        w = (lq * lk + 1).double()
        shares = [0.25 if chunks >= 3 and c in (0, chunks - 1) else 1.0 for c in range(chunks)]
        unit, wmax = float(w.sum()) / sum(shares), float(w.max()) if B else 0.0
        for c, (a, b) in enumerate(zip(cuts, cuts[1:])):
            if b < B:  # the last run takes whatever is left
                assert float(w[a:b].sum()) <= shares[c] * unit + wmax + 1e-6


def test_python_entry_points_refuse_host_tensors(lib):
    """There is no CPU fallback: the device entry points reject host tensors
    before calling the library (and the library needs a GPU to compute)."""
    import torch

    from ragged_gqa_attention_varlen_gb300 import binding, workloads

    p = workloads.tiny()
    for fn, args in (
            (binding.attention_varlen_fvjp, (p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout)),
            (binding.attention_varlen_fwd, (p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes)),
            (binding.attention_varlen_bwd, (p.q, p.k, p.v, p.cu_q, p.cu_k, p.alibi_slopes, p.dout,
                                            p.q, torch.zeros(p.q.shape[:2])))):
        try:
            fn(*args)
        except ValueError as e:
            assert "CUDA" in str(e)
        else:
            raise AssertionError(f"{fn.__name__} accepted host tensors")


def test_python_host_entry_point_rejects_device_layout_errors(lib):
    """The host-buffer wrapper checks its tensors on the host side too."""
    import pytest
    import torch

    from ragged_gqa_attention_varlen_gb300 import binding, workloads

    p = workloads.tiny()
    with pytest.raises(ValueError):  # cu arrays must be int32
        binding.attention_varlen_fvjp_host(p.q, p.k, p.v, p.cu_q.long(), p.cu_k, p.alibi_slopes,
                                           p.dout)
    with pytest.raises(ValueError):  # 7 query heads over 2 K/V heads
        q = torch.zeros((p.q.shape[0], 7, 160), dtype=p.q.dtype)
        k = torch.zeros((p.k.shape[0], 2, 160), dtype=p.q.dtype)
        binding.attention_varlen_fvjp_host(q, k, k, p.cu_q, p.cu_k, None, q)


def _gated_call(lib, **over):
    """A gated call whose arguments fail host validation (fake pointers are
    never dereferenced)."""
    fake = 0x10000
    a = dict(dtype=1, B=2, Hq=8, Hkv=2, hd=128, R=64, tq=10, tk=12,
             q=fake, qts=8 * 128, qhs=128, k=fake, kts=2 * 128, khs=128, v=fake, vts=2 * 128,
             vhs=128, do=fake, dts=8 * 128, dhs=128, qg=fake, qgts=8 * 64, qghs=64, kg=fake,
             kgts=2 * 64, kghs=64, cuq=fake, cuk=fake, sl=None, slb=0, causal=1, wl=-1, wr=-1,
             sm=1.0, out=fake, ots=8 * 128, ohs=128, dq=fake, dqts=8 * 128, dqhs=128,
             dk=fake, dkts=2 * 128, dkhs=128, dv=fake, dvts=2 * 128, dvhs=128,
             dqg=fake, dqgts=8 * 64, dqghs=64, dkg=fake, dkgts=2 * 64, dkghs=64,
             lse=fake, ws=fake, wsb=0, st=None, stream=None)
    a.update(over)
    return lib.attn_varlen_gated_fvjp_fwd_bwd(*a.values())


def test_gated_host_validation_codes(lib):
    assert _gated_call(lib) == -4                 # valid up to the missing workspace
    assert _gated_call(lib, hd=160) == -2         # head dimensions 64 and 128 only
    assert _gated_call(lib, R=72) == -2           # gate width up to 64
    assert _gated_call(lib, R=20) == -2           # ... in multiples of 8
    assert _gated_call(lib, hd=64, R=32) == -4
    assert _gated_call(lib, qg=0x10008) == -3     # gate base not 16-byte aligned
    assert _gated_call(lib, kgts=2 * 64 + 4) == -3
    assert _gated_call(lib, dkg=None) == -1       # the backward needs both gate gradients
    assert _gated_call(lib, Hkv=3) == -1


def test_dropout_mask_bytes_is_the_documented_layout(lib):
    """attn_varlen_dropout_mask_bytes: a 256-byte-rounded header of B + 1
    int32, then Hkv groups of 2 KB blocks, one per (query tile, key tile) of
    every sequence; query tiles are 128/G tokens x G heads with G the largest
    power of two up to 16 dividing the heads per K/V head."""
    import numpy as np

    def expect(lq, lk, Hq, Hkv):
        R = Hq // Hkv
        G = 16
        while R % G:
            G //= 2
        rows_tok, ngroups = 128 // G, R // G
        blocks = sum(-(-a // rows_tok) * ngroups * -(-b // 128) for a, b in zip(lq, lk))
        header = -(-4 * (len(lq) + 1) // 256) * 256
        return header + Hkv * blocks * 2048

    for lq, lk, Hq, Hkv in (([70, 300, 1], [90, 260, 40], 16, 1), ([0, 5], [7, 0], 12, 4),
                            ([8000, 129], [128, 12000], 96, 1), ([190, 70], [150, 270], 8, 2),
                            ([], [], 16, 1)):
        cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
        cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
        got = lib.attn_varlen_dropout_mask_bytes(len(lq), cu_q.ctypes.data, cu_k.ctypes.data,
                                                 Hq, Hkv)
        assert got == expect(lq, lk, Hq, Hkv), (lq, lk, Hq, Hkv)
    cu = np.array([0, 5], dtype=np.int32)
    assert lib.attn_varlen_dropout_mask_bytes(1, cu.ctypes.data, cu.ctypes.data, 12, 5) == 0
    bad = np.array([0, 5, 3], dtype=np.int32)  # decreasing
    assert lib.attn_varlen_dropout_mask_bytes(2, bad.ctypes.data, bad.ctypes.data, 16, 1) == 0


def test_dropout_mask_calls_validate_the_buffer(lib):
    """The stored-mask calls refuse a missing, short or misaligned keep mask
    before anything is enqueued."""
    fake = 0x10000
    head = [0, 2, 16, 1, 160, 10, 12,
            fake, 16 * 160, 160, fake, 160, 160, fake, 160, 160, fake, 16 * 160, 160,
            fake, fake, fake, 16, 0, -1, -1, 3.0, 0.75, 7, 0.1, None]
    tail = [fake, 16 * 160, 160, fake, 16 * 160, 160, fake, 160, 160, fake, 160, 160,
            fake, fake, 0, None, None]
    f = lib.attn_varlen_fvjp_fwd_bwd_dropout_mask
    assert f(*head, None, 1 << 20, *tail) == -1        # no mask
    assert f(*head, fake, 16, *tail) == -1             # smaller than the header
    assert f(*head, fake + 16, 1 << 20, *tail) == -3   # not 256-byte aligned
    assert f(*head, fake, 1 << 20, *tail) == -4        # valid up to the missing workspace

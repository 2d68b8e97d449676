"""C-ABI tests that need no GPU: the library builds, loads and exports every function declared in
include/fa.h, and host-side validation rejects bad arguments before any CUDA call."""

import ctypes
import math
import os
import re

import pytest

import exact_io_aware_38_gb300 as fa
from exact_io_aware_38_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return fa.lib()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_status_string"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for rc in (0, -1, -2, -3, -4, -5, -6, 7):
        s = fa.fa_status_string(rc)
        assert isinstance(s, str) and s


def test_workspace_bytes(L):
    B, H, N, d = 2, 3, 130, 64
    rows = B * H * N
    r256 = lambda x: (x + 255) // 256 * 256
    assert fa.fa_bwd_workspace_bytes(B, H, N, d) == r256(rows * 4) + r256(rows * d * 4) + 256
    assert fa.fa_bwd_workspace_bytes(1, 1, 1, 96) == 0
    assert fa.fa_bwd_workspace_bytes(0, 1, 1, 64) == 0


# Fake, never-dereferenced device addresses: validation must fail before any launch.
A = 0x10000


def fwd_rc(**kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=128, d=64, causal=0, block_mask=None, seqlens_k=None, scale=0.125,
                tile_visits=None, dev_status=None, stream=None)
    args.update(kw)
    return fa.fa_fwd(**args)


def bwd_rc(**kw):
    args = dict(q=A, k=A, v=A, o=A, dout=A, lse=A, dq=A, dk=A, dv=A, B=1, H=1, N=128, d=64, causal=0, block_mask=None,
                seqlens_k=None, scale=0.125, workspace=A, workspace_bytes=1 << 30, dev_status=None, stream=None)
    args.update(kw)
    return fa.fa_bwd(**args)


@pytest.mark.parametrize("kw,rc", [
    (dict(q=None), -1), (dict(lse=None), -1), (dict(B=0), -1), (dict(N=0), -1), (dict(H=-1), -1),
    (dict(causal=2), -1), (dict(scale=0.0), -1), (dict(scale=-1.0), -1), (dict(scale=float("nan")), -1),
    (dict(scale=float("inf")), -1), (dict(d=96), -2), (dict(d=256), -2), (dict(B=1 << 14, H=1 << 10, N=1 << 10), -2),
    (dict(q=A + 8), -3), (dict(o=A + 2), -3), (dict(lse=A + 2), -3), (dict(seqlens_k=A + 1), -3),
])
def test_fwd_validation(L, kw, rc):
    assert fwd_rc(**kw) == rc


@pytest.mark.parametrize("kw,rc", [
    (dict(dout=None), -1), (dict(workspace=None), -1), (dict(workspace_bytes=16), -1), (dict(d=32), -2),
    (dict(dq=A + 8), -3), (dict(workspace=A + 16), -3), (dict(scale=float("nan")), -1),
])
def test_bwd_validation(L, kw, rc):
    assert bwd_rc(**kw) == rc


def gqa_fwd_rc(**kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=4, Hkv=2, N=128, d=64, causal=0, block_mask=None, seqlens_k=None,
                scale=0.125, tile_visits=None, dev_status=None, stream=None)
    args.update(kw)
    return fa.fa_fwd_gqa(**args)


def gqa_bwd_rc(**kw):
    args = dict(q=A, k=A, v=A, o=A, dout=A, lse=A, dq=A, dk=A, dv=A, B=1, H=4, Hkv=2, N=128, d=64, causal=0,
                block_mask=None, seqlens_k=None, scale=0.125, workspace=A, workspace_bytes=1 << 30, dev_status=None,
                stream=None)
    args.update(kw)
    return fa.fa_bwd_gqa(**args)


@pytest.mark.parametrize("kw,rc", [
    (dict(Hkv=0), -1), (dict(Hkv=-2), -1), (dict(Hkv=3), -1), (dict(Hkv=8), -1), (dict(H=6, Hkv=4), -1),
    (dict(k=None), -1), (dict(d=96), -2), (dict(v=A + 8), -3),
])
def test_gqa_validation(L, kw, rc):
    assert gqa_fwd_rc(**kw) == rc
    assert gqa_bwd_rc(**kw) == rc


def test_binding_refuses_cpu_tensors(L):
    import torch

    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd(q, q, q)


def test_binding_checks_optional_buffers(L):
    """lse, status, tile visits, workspace and partials handed to the kernels: dtype, size,
    contiguity and device are checked before any call (sizes are minimums)."""
    import torch

    dev = torch.device("cpu")
    fa._check_aux("lse", None, torch.float32, 6, dev)
    fa._check_aux("lse", torch.zeros(6), torch.float32, 6, dev)
    fa._check_aux("lse", torch.zeros(8), torch.float32, 6, dev)
    for bad in (torch.zeros(5), torch.zeros(6, dtype=torch.bfloat16), torch.zeros(12)[::2],
                torch.zeros(6, device="meta")):
        with pytest.raises(ValueError):
            fa._check_aux("lse", bad, torch.float32, 6, dev)
    fa._check_aux("workspace", torch.zeros(64, dtype=torch.uint8), None, 64, dev)
    fa._check_aux("workspace", torch.zeros(16), None, 64, dev)  # sized in bytes
    with pytest.raises(ValueError):
        fa._check_aux("workspace", torch.zeros(64, dtype=torch.uint8), None, 65, dev)
    fa._same_device(torch.zeros(1), torch.zeros(2), None)
    with pytest.raises(ValueError):
        fa._same_device(torch.zeros(1), torch.zeros(1, device="meta"))


def varlen_rc(bwd=False, problem=None, **kw):
    p = fa.VarlenProblem(2, 4, 2, 64, 100, 120, None, None, 0, 0, 1, 0.125) if problem is None else problem
    for name, val in kw.items():
        setattr(p, name, val)
    st = fa.Strides(4 * 64, 64, 100 * 4 * 64)
    sk = fa.Strides(2 * 64, 64, 120 * 2 * 64)
    if not bwd:
        return fa.fa_fwd_varlen(p, A, st, A, sk, A, sk, A, st, A, None, None)
    return fa.fa_bwd_varlen(p, A, st, A, sk, A, sk, A, st, A, st, A, A, st, A, sk, A, sk, A, 1 << 30, None, None)


@pytest.mark.parametrize("kw,rc", [
    (dict(Hkv=3), -1), (dict(B=0), -1), (dict(seqlen_q=0), -1), (dict(causal=5), -1), (dict(scale=0.0), -1),
    (dict(d=32), -2), (dict(cu_seqlens_q=A), -1), (dict(cu_seqlens_k=A), -1),
    (dict(cu_seqlens_q=A, cu_seqlens_k=A, rows_q=0, rows_k=10), -1),
    (dict(cu_seqlens_q=A + 2, cu_seqlens_k=A, rows_q=10, rows_k=10), -3),
])
def test_varlen_validation(L, kw, rc):
    assert varlen_rc(False, **kw) == rc
    assert varlen_rc(True, **kw) == rc


def test_varlen_bad_strides(L):
    p = fa.VarlenProblem(2, 4, 4, 64, 100, 100, None, None, 0, 0, 0, 0.125)
    good = fa.Strides(4 * 64, 64, 100 * 4 * 64)
    for bad in (fa.Strides(0, 64, 25600), fa.Strides(4 * 64, 60, 25600), fa.Strides(4 * 64, 64, 0),
                fa.Strides(-256, 64, 25600)):
        assert fa.fa_fwd_varlen(p, A, bad, A, good, A, good, A, good, A, None, None) == -1
        assert fa.fa_fwd_varlen(p, A, good, A, good, A, good, A, bad, A, None, None) == -1
    assert fa.fa_fwd_varlen(p, A + 16, good, A, good, A, good, A, good, A + 2, None, None) == -3


def test_varlen_workspace_bytes(L):
    r256 = lambda x: (x + 255) // 256 * 256
    p = fa.VarlenProblem(3, 4, 2, 128, 100, 70, None, None, 0, 0, 1, 0.1)
    rows = 3 * 4 * 100
    assert fa.fa_bwd_varlen_workspace_bytes(p) == r256(rows * 4) + r256(rows * 128 * 4) + 256
    p = fa.VarlenProblem(3, 4, 2, 64, 100, 70, A, A, 257, 180, 1, 0.1)
    rows = 4 * 257
    assert fa.fa_bwd_varlen_workspace_bytes(p) == r256(rows * 4) + r256(rows * 64 * 4) + 256
    p.Hkv = 3
    assert fa.fa_bwd_varlen_workspace_bytes(p) == 0


def test_splitkv_host_rules(L):
    r256 = lambda x: (x + 255) // 256 * 256
    p = fa.VarlenProblem(1, 8, 2, 128, 1, 8192, None, None, 0, 0, 1, 0.1)
    # Estimated cost in key-tile units: waves x (6 fixed + key tiles per split), + 3 for a merge.
    # One query row with grouped heads runs as G rows of each K/V head (one CTA per K/V head); a
    # split with one query tile per (batch, head) runs two CTAs per SM.
    assert fa.fa_fwd_splitkv_splits(p, 152) == 16        # 2 CTAs: 16 splits (cap 64/4), one wave
    p2 = fa.VarlenProblem(4, 32, 32, 128, 4096, 4096, None, None, 0, 0, 1, 0.1)
    assert fa.fa_fwd_splitkv_splits(p2, 152) == 1        # 2048 CTAs: a split only adds waves
    p3 = fa.VarlenProblem(1, 1, 1, 64, 1, 300, None, None, 0, 0, 0, 0.1)
    assert fa.fa_fwd_splitkv_splits(p3, 152) == 1        # 3 key tiles: fewer than four per split
    p4 = fa.VarlenProblem(8, 32, 8, 128, 1, 8192, None, None, 0, 0, 1, 0.1)
    assert fa.fa_fwd_splitkv_splits(p4, 152) == 4        # decode at batch 8: 64 CTAs; 4 splits, one wave of 2/SM
    p5 = fa.VarlenProblem(1, 32, 8, 128, 1, 8192, None, None, 0, 0, 1, 0.1)
    assert fa.fa_fwd_splitkv_splits(p5, 152) == 16       # 8 CTAs: 16 splits, one wave
    p6 = fa.VarlenProblem(1, 32, 32, 128, 1, 8192, None, None, 0, 0, 1, 0.1)
    assert fa.fa_fwd_splitkv_splits(p6, 152) == 8        # 32 CTAs (no grouping): 8 splits, one wave of 2/SM
    rows = 8 * 1
    assert fa.fa_fwd_splitkv_workspace_bytes(p, 5) == r256(5 * rows * 4) + r256(5 * rows * 128 * 4)
    assert fa.fa_fwd_splitkv_workspace_bytes(p, 0) == 0 and fa.fa_fwd_splitkv_workspace_bytes(p, 257) == 0
    st = fa.Strides(8 * 128, 128, 8 * 128)
    sk = fa.Strides(2 * 128, 128, 8192 * 2 * 128)
    for ns, ws, nbytes, rc in ((0, A, 1 << 30, -1), (257, A, 1 << 30, -1), (4, None, 1 << 30, -1), (4, A, 16, -1),
                               (4, A + 16, 1 << 30, -3)):
        assert fa.fa_fwd_splitkv(p, ns, A, st, A, sk, A, sk, A, st, A, ws, nbytes, None, None) == rc


def test_bwd_ex_validation(L):
    """fa_bwd_ex checks its extras on the host too: a misaligned step-visit array is rejected
    before any launch, and every fa_bwd check still applies."""
    base = dict(q=A, k=A, v=A, o=A, dout=A, lse=A, dq=A, dk=A, dv=A, B=1, H=2, Hkv=1, N=128, d=64, causal=0,
                block_mask=None, seqlens_k=None, scale=0.125, workspace=A, workspace_bytes=1 << 30, dev_status=None,
                stream=None)
    bad = fa.BwdExtras(A + 2, None, None)
    assert fa.fa_bwd_ex(**base, extras=bad) == -3
    assert fa.fa_bwd_ex(**dict(base, q=None), extras=fa.BwdExtras(A, None, None)) == -1
    assert fa.fa_bwd_ex(**dict(base, Hkv=3), extras=None) == -1
    assert fa.fa_bwd_ex(**dict(base, d=96), extras=None) == -2


def test_fwd_fp8_validation(L):
    """fa_fwd_fp8 checks its arguments on the host: d must be 128 and N a multiple of 16 (the V^T rows
    start on 16-byte boundaries), every descale array is required and 4-byte aligned."""
    base = dict(q=A, k=A, vt=A, o=A, lse=A, B=1, H=2, Hkv=1, N=256, d=128, causal=1, block_mask=None,
                seqlens_k=None, q_descale=A, k_descale=A, v_descale=A, scale=0.088, tile_visits=None,
                dev_status=None, stream=None)
    assert fa.fa_fwd_fp8(**dict(base, d=64)) == -2
    assert fa.fa_fwd_fp8(**dict(base, N=100)) == -2
    assert fa.fa_fwd_fp8(**dict(base, q_descale=None)) == -1
    assert fa.fa_fwd_fp8(**dict(base, vt=None)) == -1
    assert fa.fa_fwd_fp8(**dict(base, Hkv=3)) == -1
    assert fa.fa_fwd_fp8(**dict(base, vt=A + 8)) == -3
    assert fa.fa_fwd_fp8(**dict(base, k_descale=A + 2)) == -3
    assert fa.fa_fwd_fp8(**dict(base, scale=0.0)) == -1

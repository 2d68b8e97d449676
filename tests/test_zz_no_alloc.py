"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory (for example
a plugin inside another framework, which gets only its input and output buffers while that
framework owns the device memory pool). It must give the same gradients as fa_bwd with a
caller-supplied workspace, call after call, although its fixed scratch array keeps the previous
call's contents. This file is collected last on purpose."""

import os
import re

import numpy as np
import pytest
import torch

import exact_io_aware_38_gb300 as fa
import oracle
from exact_io_aware_38_gb300 import build, workloads

REL_FRO = 2e-2  # the gradient tolerance of the parity tests


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm())


def _case(seed, causal, padded):
    B, H, N, d = 2, 4, 1000, 128
    inp = workloads.random_inputs(B, H, N, d, seed)
    dev = "cuda"
    t = {n: inp[n].to(dev) for n in ("q", "k", "v", "do")}
    sl = torch.tensor([1000, 613], dtype=torch.int32, device=dev) if padded else None
    return t, dict(causal=causal, seqlens_k=sl, scale=1.0 / np.sqrt(d)), (B, H, N, d)


def _noalloc(t, kw, shape, o, lse, status):
    B, H, N, d = shape
    dq, dk, dv = (torch.empty_like(t["q"]) for _ in range(3))
    rc = fa.fa_bwd_noalloc(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), o.data_ptr(), t["do"].data_ptr(),
                           lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, int(kw["causal"]),
                           None, None if kw["seqlens_k"] is None else kw["seqlens_k"].data_ptr(), kw["scale"],
                           status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, fa.fa_status_string(rc)
    return dq, dk, dv


@pytest.mark.gpu
def test_noalloc_matches_fa_bwd_on_consecutive_calls():
    """Two calls in a row, with different problems, each against fa_bwd with a workspace (the scratch
    keeps the previous call's contents) and the first also against the fp64 oracle."""
    build.build()
    fa.lib()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for seed, causal, padded in ((21, True, False), (22, False, True)):
        t, kw, shape = _case(seed, causal, padded)
        o, lse = fa.fwd(t["q"], t["k"], t["v"], status=status, **kw)
        ref = fa.bwd(t["q"], t["k"], t["v"], o, lse, t["do"], status=status, **kw)
        got = _noalloc(t, kw, shape, o, lse, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, fa.fa_status_string(int(status.item()))
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(a.float()).all(), name
            assert _rel(a, b) <= REL_FRO, (seed, name, _rel(a, b))
        if seed == 21:
            f = lambda x: x.double().cpu().numpy()
            want = oracle.attention_backward(f(t["q"]), f(t["k"]), f(t["v"]), f(t["do"]), kw["scale"], causal=causal)
            for name, a, w in zip(("dq", "dk", "dv"), got, want):
                r = float(np.linalg.norm(f(a) - w) / np.linalg.norm(w))
                assert r <= REL_FRO, (name, r)


def test_noalloc_scratch_size_matches_the_header():
    """The binding's constant is the header's FA_NOALLOC_SCRATCH_BYTES."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = open(os.path.join(root, "include", "fa.h")).read()
    m = re.search(r"#define\s+FA_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "FA_NOALLOC_SCRATCH_BYTES not found"
    assert fa.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_noalloc_rejects_problems_beyond_its_scratch():
    build.build()
    A = 0x10000
    B, H, N, d = 1, 32, 8192, 128  # needs ~135 MB of scratch
    assert fa.fa_bwd_workspace_bytes(B, H, N, d) > fa.NOALLOC_SCRATCH_BYTES
    rc = fa.fa_bwd_noalloc(A, A, A, A, A, A, A, A, A, B, H, N, d, 1, None, None, 0.088, None, None)
    assert rc == -7 and "SCRATCH" in fa.fa_status_string(rc)

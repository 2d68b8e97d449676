"""Failure detection without a GPU fault: every wait inside the kernels is bounded. A test-only
build of the library whose forward and backward producers never load K/V (the flag nothing sets)
must make the consumers' waits run out; the kernel must record FA_ERR_DEVICE_TIMEOUT in the status
word, stop issuing copies, MMAs and barrier arrivals, let the copies it already issued land, release
its tensor memory and return, and the GPU must stay usable for a normal call.

Each case runs in a child process of its own, so whatever happens there cannot reach the CUDA
context of the test session; the child also checks a normal call against the oracle afterwards.
Both head dimensions run, so each kernel layout is covered: the forward's pair mode (d = 128) and
single mode (d = 64), the backward's two-buffer layout (d = 128) and single mode (d = 64).
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r'''
import ctypes, sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
import exact_io_aware_38_gb300 as fa
import oracle
from exact_io_aware_38_gb300 import build, workloads

build.build()
L = ctypes.CDLL(build.build_withhold_kv_test_lib())
P, I = ctypes.c_void_p, ctypes.c_int
status = torch.zeros(1, dtype=torch.int32, device="cuda")
f = lambda t: t.double().numpy()
if CASE == "fwd":
    L.fa_fwd.restype = I
    L.fa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P, ctypes.c_float, P, P, P]
    B, H, N, d = 1, 2, 256, D
    inp = workloads.random_inputs(B, H, N, d, seed=3)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    rc = L.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, 1, None,
                  None, 0.088, None, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert int(status.item()) == -5, int(status.item())  # FA_ERR_DEVICE_TIMEOUT
    # The context and the GPU are still healthy: the real library computes correct results.
    status.zero_()
    o2, lse2 = fa.fwd(q, k, v, causal=True, scale=0.088, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rl = oracle.attention_forward(f(inp["q"]), f(inp["k"]), f(inp["v"]), 0.088, causal=True)
    assert np.abs(f(o2.cpu()) - ro).max() <= 2e-2
    assert np.abs(lse2.cpu().double().numpy() - rl).max() <= 1e-3
else:
    L.fa_bwd.restype = I
    L.fa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, ctypes.c_float, P, ctypes.c_size_t, P, P]
    L.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
    L.fa_bwd_workspace_bytes.argtypes = [I, I, I, I]
    # 512 key tiles on the persistent grid: after its abort each CTA still takes tiles through the
    # queue, the per-tile done / accumulator waits and the step barriers.
    B, H, N, d, scale = 1, 64, 1024, D, 0.125
    g = torch.Generator("cuda").manual_seed(11)
    q, k, v, o, do = (torch.randn((B, H, N, d), generator=g, device="cuda").to(torch.bfloat16) for _ in range(5))
    lse = torch.randn((B, H, N), generator=g, device="cuda")
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    nbytes = int(L.fa_bwd_workspace_bytes(B, H, N, d))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    rc = L.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                  dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, 1, None, None, scale, ws.data_ptr(),
                  nbytes, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert int(status.item()) == -5, int(status.item())  # FA_ERR_DEVICE_TIMEOUT
    # The context and the GPU are still healthy: the real library's backward matches the oracle.
    B, H, N = 1, 2, 384
    inp = workloads.random_inputs(B, H, N, d, seed=5)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    status.zero_()
    o, lse = fa.fwd(q, k, v, causal=True, scale=scale, status=status)
    dq2, dk2, dv2 = fa.bwd(q, k, v, o, lse, do, causal=True, scale=scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.attention_backward(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["do"]), scale, causal=True)
    for got, want in zip((dq2, dk2, dv2), ref):
        assert np.linalg.norm(f(got.cpu()) - want) <= 2e-2 * np.linalg.norm(want)
print("CHILD_OK")
'''


def _run_child(case, d):
    code = f"ROOT = {ROOT!r}\nCASE = {case!r}\nD = {d}\n" + _CHILD
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0 and "CHILD_OK" in r.stdout, (r.returncode, r.stdout[-2000:], r.stderr[-4000:])


@pytest.mark.parametrize("d", [64, 128])
def test_forward_bounded_wait_reports_timeout_and_gpu_stays_usable(d):
    _run_child("fwd", d)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_bounded_wait_reports_timeout_and_gpu_stays_usable(d):
    """The persistent backward under the same test build: its key-tile queue, the per-tile done and
    accumulator-release waits and the step barriers all give up, every role leaves its tile loop,
    and the next normal call on the context is correct."""
    _run_child("bwd", d)

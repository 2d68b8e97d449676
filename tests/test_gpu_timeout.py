"""Failure detection without a GPU fault: every wait inside the kernels is bounded. A test-only
build of the library whose forward producer never loads K/V (the flag nothing sets) must make
the consumers' waits run out; the kernel must record FA_ERR_DEVICE_TIMEOUT in the status word,
release its tensor memory and return, and the GPU must stay usable for a normal call."""

import ctypes

import numpy as np
import pytest
import torch

import exact_io_aware_38_gb300 as fa
import oracle
from exact_io_aware_38_gb300 import build, workloads

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_gpu_stays_usable():
    build.build()
    path = build.build_withhold_kv_test_lib()
    L = ctypes.CDLL(path)
    P, I = ctypes.c_void_p, ctypes.c_int
    L.fa_fwd.restype = I
    L.fa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P, ctypes.c_float, P, P, P]
    B, H, N, d = 1, 2, 256, 128
    inp = workloads.random_inputs(B, H, N, d, seed=3)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, 1, None, None,
                  0.088, None, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == -5  # FA_ERR_DEVICE_TIMEOUT

    # The context and the GPU are still healthy: the real library computes correct results.
    status.zero_()
    o2, lse2 = fa.fwd(q, k, v, causal=True, scale=0.088, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    f = lambda t: t.double().numpy()
    ro, rl = oracle.attention_forward(f(inp["q"]), f(inp["k"]), f(inp["v"]), 0.088, causal=True)
    assert np.abs(f(o2.cpu()) - ro).max() <= 2e-2
    assert np.abs(lse2.cpu().double().numpy() - rl).max() <= 1e-3

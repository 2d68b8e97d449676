"""Fused exact attention for GB300 (sm_103a): thin Python binding of ``libfa.so``.

The binding only marshals arguments: every step of the forward and backward pass runs in the
library's CUDA kernels. PyTorch provides device memory and the current stream. There is no CPU
fallback: if the library is missing, every call raises.

Raw C-ABI names (same signatures as ``include/fa.h``, pointers as ints):
    fa_fwd, fa_bwd, fa_fwd_gqa, fa_bwd_gqa, fa_bwd_ex (with the BwdExtras struct), fa_bwd_workspace_bytes,
    fa_status_string, fa_bwd_noalloc,
    fa_fwd_varlen, fa_bwd_varlen, fa_bwd_varlen_accumulate, fa_bwd_varlen_workspace_bytes (with the Strides /
    VarlenProblem structs)
Tensor helpers (grouped-query attention when k, v have fewer heads than q):
    fwd(q, k, v, ...) -> (o, lse);  bwd(q, k, v, o, lse, do, ...) -> (dq, dk, dv)
    fwd_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, ...) -> (o, lse): e4m3 inputs (fa_fwd_fp8)
    fwd_varlen(q, k, v, ...), bwd_varlen(...): [B, N, H, d] views with any strides, or packed
    [rows, H, d] sequences located by cu_seqlens; query and key lengths may differ.
    fwd_splitkv(q, k, v, ..., num_splits=None): the forward split over keys (decode shapes).
    fwd_partial / merge_partials / finalize_partials: per-key-block partials and their
    log-sum-exp merge (ring.py builds sequence-sharded ring attention on them).
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int


class Strides(ctypes.Structure):
    """fa_strides: element strides of a [batch][row][head][d] view."""
    _fields_ = [("row", ctypes.c_int64), ("head", ctypes.c_int64), ("batch", ctypes.c_int64)]


class VarlenProblem(ctypes.Structure):
    """fa_varlen_problem (include/fa.h)."""
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("Hkv", ctypes.c_int), ("d", ctypes.c_int),
                ("seqlen_q", ctypes.c_int), ("seqlen_k", ctypes.c_int),
                ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
                ("rows_q", ctypes.c_int), ("rows_k", ctypes.c_int), ("causal", ctypes.c_int),
                ("scale", ctypes.c_float)]


class BwdExtras(ctypes.Structure):
    """fa_bwd_extras (include/fa.h): optional step-visit counts and events around the main pass."""
    _fields_ = [("step_visits", ctypes.c_void_p), ("main_begin_event", ctypes.c_void_p),
                ("main_end_event", ctypes.c_void_p)]


_VP = ctypes.POINTER(VarlenProblem)
_SIGS = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, ctypes.c_float, _P, _P, _P]),
    "fa_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "fa_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, ctypes.c_float, _P,
                    ctypes.c_size_t, _P, _P]),
    "fa_fwd_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, ctypes.c_float, _P, _P, _P]),
    "fa_bwd_gqa": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, ctypes.c_float, _P,
                        ctypes.c_size_t, _P, _P]),
    "fa_bwd_ex": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, ctypes.c_float, _P,
                       ctypes.c_size_t, ctypes.POINTER(BwdExtras), _P, _P]),
    "fa_fwd_varlen": (_I, [_VP, _P, Strides, _P, Strides, _P, Strides, _P, Strides, _P, _P, _P]),
    "fa_bwd_varlen_workspace_bytes": (ctypes.c_size_t, [_VP]),
    "fa_bwd_varlen": (_I, [_VP, _P, Strides, _P, Strides, _P, Strides, _P, Strides, _P, Strides, _P, _P, Strides,
                           _P, Strides, _P, Strides, _P, ctypes.c_size_t, _P, _P]),
    "fa_bwd_varlen_accumulate": (_I, [_VP, _P, Strides, _P, Strides, _P, Strides, _P, Strides, _P, Strides, _P, _P,
                                      Strides, _P, Strides, _P, Strides, _P, ctypes.c_size_t, _P, _P]),
    "fa_fwd_splitkv_splits": (_I, [_VP, _I]),
    "fa_fwd_splitkv_workspace_bytes": (ctypes.c_size_t, [_VP, _I]),
    "fa_fwd_splitkv": (_I, [_VP, _I, _P, Strides, _P, Strides, _P, Strides, _P, Strides, _P, _P, ctypes.c_size_t, _P,
                            _P]),
    "fa_partial_rows": (ctypes.c_size_t, [_VP]),
    "fa_fwd_partial": (_I, [_VP, _P, Strides, _P, Strides, _P, Strides, _P, _P, _P, _P]),
    "fa_merge_partials": (_I, [_VP, _P, _P, _P, _P, _P]),
    "fa_finalize_partials": (_I, [_VP, _P, _P, _P, Strides, _P, _P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, ctypes.c_float, _P, _P]),
}

# Size of the fixed device scratch fa_bwd_noalloc uses instead of a workspace (FA_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 32 << 20


class FaError(RuntimeError):
    def __init__(self, rc: int):
        super().__init__(fa_status_string(rc))
        self.rc = rc


def lib() -> ctypes.CDLL:
    """Load libfa.so (built by ``exact_io_aware_38_gb300.build``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run exact_io_aware_38_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ----------------------------------------------------------------------------- raw ABI


def fa_status_string(rc: int) -> str:
    return lib().fa_status_string(int(rc)).decode()


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, H, N, d))


def fa_fwd(q, k, v, o, lse, B, H, N, d, causal, block_mask, seqlens_k, scale, tile_visits, dev_status, stream) -> int:
    return int(lib().fa_fwd(q, k, v, o, lse, B, H, N, d, causal, block_mask, seqlens_k, scale, tile_visits, dev_status,
                            stream))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, block_mask, seqlens_k, scale, workspace,
           workspace_bytes, dev_status, stream) -> int:
    return int(lib().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, block_mask, seqlens_k, scale,
                            workspace, workspace_bytes, dev_status, stream))


def fa_fwd_gqa(q, k, v, o, lse, B, H, Hkv, N, d, causal, block_mask, seqlens_k, scale, tile_visits, dev_status,
               stream) -> int:
    return int(lib().fa_fwd_gqa(q, k, v, o, lse, B, H, Hkv, N, d, causal, block_mask, seqlens_k, scale, tile_visits,
                                dev_status, stream))


def fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, d, causal, block_mask, seqlens_k, scale, workspace,
               workspace_bytes, dev_status, stream) -> int:
    return int(lib().fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, d, causal, block_mask, seqlens_k,
                                scale, workspace, workspace_bytes, dev_status, stream))


def fa_fwd_fp8(q, k, vt, o, lse, B, H, Hkv, N, d, causal, block_mask, seqlens_k, q_descale, k_descale, v_descale,
               scale, tile_visits, dev_status, stream) -> int:
    return int(lib().fa_fwd_fp8(q, k, vt, o, lse, B, H, Hkv, N, d, causal, block_mask, seqlens_k, q_descale, k_descale,
                                v_descale, scale, tile_visits, dev_status, stream))


def fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, d, causal, block_mask, seqlens_k, scale, workspace,
              workspace_bytes, extras, dev_status, stream) -> int:
    """extras: a BwdExtras or None."""
    x = None if extras is None else ctypes.byref(extras)
    return int(lib().fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, d, causal, block_mask, seqlens_k,
                               scale, workspace, workspace_bytes, x, dev_status, stream))


def fa_fwd_varlen(p, q, sq, k, sk, v, sv, o, so, lse, dev_status, stream) -> int:
    return int(lib().fa_fwd_varlen(ctypes.byref(p), q, sq, k, sk, v, sv, o, so, lse, dev_status, stream))


def fa_bwd_varlen_workspace_bytes(p) -> int:
    return int(lib().fa_bwd_varlen_workspace_bytes(ctypes.byref(p)))


def fa_bwd_varlen(p, q, sq, k, sk, v, sv, o, so, dout, sdo, lse, dq, sdq, dk, sdk, dv, sdv, workspace,
                  workspace_bytes, dev_status, stream) -> int:
    return int(lib().fa_bwd_varlen(ctypes.byref(p), q, sq, k, sk, v, sv, o, so, dout, sdo, lse, dq, sdq, dk, sdk, dv,
                                   sdv, workspace, workspace_bytes, dev_status, stream))


def fa_fwd_splitkv_splits(p, num_sms) -> int:
    return int(lib().fa_fwd_splitkv_splits(ctypes.byref(p), num_sms))


def fa_fwd_splitkv_workspace_bytes(p, num_splits) -> int:
    return int(lib().fa_fwd_splitkv_workspace_bytes(ctypes.byref(p), num_splits))


def fa_fwd_splitkv(p, num_splits, q, sq, k, sk, v, sv, o, so, lse, workspace, workspace_bytes, dev_status,
                   stream) -> int:
    return int(lib().fa_fwd_splitkv(ctypes.byref(p), num_splits, q, sq, k, sk, v, sv, o, so, lse, workspace,
                                    workspace_bytes, dev_status, stream))


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, block_mask, seqlens_k, scale, dev_status,
                   stream) -> int:
    """fa_bwd without a workspace: for callers that cannot allocate device memory (see fa.h)."""
    return int(lib().fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, block_mask, seqlens_k,
                                    scale, dev_status, stream))


# ----------------------------------------------------------------------------- tensor helpers


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_qkv(*ts):
    ref = ts[0]
    for t in ts:
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.shape == ref.shape
                and t.device == ref.device):
            raise ValueError("q, k, v, o, dO must be contiguous bf16 CUDA tensors of one shape [B, H, N, d], "
                             "on one device")
    if ref.dim() != 4:
        raise ValueError("expected [B, H, N, d]")


def _check_aux(name, t, dtype, numel, dev):
    """An optional buffer the kernels read or write: None, or a contiguous tensor of `dtype` with at
    least `numel` elements on `dev` (dtype None: any, sized in bytes)."""
    if t is None:
        return
    n = t.numel() * t.element_size() if dtype is None else t.numel()
    if not ((dtype is None or t.dtype == dtype) and t.is_contiguous() and t.device == dev and n >= numel):
        kind = "" if dtype is None else f" {dtype}"
        unit = "bytes" if dtype is None else "elements"
        raise ValueError(f"{name} must be a contiguous{kind} tensor with at least {numel} {unit} on {dev}")


def _check_kv(q, k, v):
    """k, v: [B, Hkv, N, d] with Hkv dividing q's head count H; returns Hkv."""
    _check_qkv(k, v)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if (k.shape[0], k.shape[2], k.shape[3]) != (B, N, d) or H % Hkv != 0:
        raise ValueError("k, v must be [B, Hkv, N, d] with Hkv dividing the query head count")
    return Hkv


def _masks(block_mask, seqlens_k, N, B, dev):
    nb = (N + 127) // 128
    if block_mask is not None:
        if not (block_mask.dtype == torch.uint8 and block_mask.is_contiguous() and block_mask.numel() == nb * nb
                and block_mask.device == dev):
            raise ValueError(f"block_mask must be a contiguous uint8 [{nb}, {nb}] tensor on {dev}")
    if seqlens_k is not None:
        if not (seqlens_k.dtype == torch.int32 and seqlens_k.is_contiguous() and seqlens_k.numel() == B
                and seqlens_k.device == dev):
            raise ValueError(f"seqlens_k must be a contiguous int32 [{B}] tensor on {dev}")


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def fwd(q, k, v, *, causal=False, block_mask=None, seqlens_k=None, scale=None, out=None, lse=None,
        tile_visits=None, status=None, stream=None):
    """O, LSE = attention(q, k, v) on the current CUDA stream. Outputs are allocated unless given.
    k and v may have fewer heads than q (grouped-query attention, fa_fwd_gqa)."""
    _check_qkv(q)
    Hkv = _check_kv(q, k, v)
    B, H, N, d = q.shape
    _masks(block_mask, seqlens_k, N, B, q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    _check_qkv(q, o)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_aux("lse", lse, torch.float32, B * H * N, q.device)
    _check_aux("tile_visits", tile_visits, torch.int32, B * H * ((N + 127) // 128), q.device)
    _check_aux("status", status, torch.int32, 1, q.device)
    rc = fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv, N, d,
                    int(causal), _ptr(block_mask), _ptr(seqlens_k), scale, _ptr(tile_visits), _ptr(status),
                    _stream(stream))
    if rc != 0:
        raise FaError(rc)
    return o, lse


def fwd_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, *, causal=False, block_mask=None, seqlens_k=None, scale=None,
            out=None, lse=None, tile_visits=None, status=None, stream=None):
    """O (bf16), LSE of attention over e4m3 inputs (fa_fwd_fp8): q8 [B, H, N, d], k8 [B, Hkv, N, d] and
    vt8 = V^T [B, Hkv, d, N] as torch.float8_e4m3fn tensors, with fp32 per-head descales q_descale
    [B, H], k_descale and v_descale [B, Hkv] (the inputs are descale * values). d = 128."""
    f8 = torch.float8_e4m3fn
    for name, t in (("q8", q8), ("k8", k8), ("vt8", vt8)):
        if not (t.is_cuda and t.dtype == f8 and t.is_contiguous() and t.dim() == 4 and t.device == q8.device):
            raise ValueError(f"{name} must be a contiguous 4-D float8_e4m3fn CUDA tensor on {q8.device}")
    B, H, N, d = q8.shape
    Hkv = k8.shape[1]
    if k8.shape != (B, Hkv, N, d) or vt8.shape != (B, Hkv, d, N) or H % Hkv != 0:
        raise ValueError("k8 must be [B, Hkv, N, d] and vt8 [B, Hkv, d, N] with Hkv dividing H")
    _masks(block_mask, seqlens_k, N, B, q8.device)
    for name, t, n in (("q_descale", q_descale, B * H), ("k_descale", k_descale, B * Hkv),
                       ("v_descale", v_descale, B * Hkv)):
        if t is None:
            raise ValueError(f"{name} is required")
        _check_aux(name, t, torch.float32, n, q8.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    _check_qkv(o)
    if o.shape != (B, H, N, d) or o.device != q8.device:
        raise ValueError("out must be a bf16 [B, H, N, d] tensor on the inputs' device")
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    _check_aux("lse", lse, torch.float32, B * H * N, q8.device)
    _check_aux("tile_visits", tile_visits, torch.int32, B * H * ((N + 127) // 128), q8.device)
    _check_aux("status", status, torch.int32, 1, q8.device)
    rc = fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv, N, d,
                    int(causal), _ptr(block_mask), _ptr(seqlens_k), q_descale.data_ptr(), k_descale.data_ptr(),
                    v_descale.data_ptr(), scale, _ptr(tile_visits), _ptr(status), _stream(stream))
    if rc != 0:
        raise FaError(rc)
    return o, lse


def bwd(q, k, v, o, lse, do, *, causal=False, block_mask=None, seqlens_k=None, scale=None, dq=None, dk=None, dv=None,
        workspace=None, status=None, stream=None, step_visits=None, main_events=None):
    """dQ, dK, dV of attention on the current CUDA stream (outputs/workspace allocated unless given).
    k and v may have fewer heads than q (grouped-query attention, fa_bwd_gqa); dk, dv are shaped like k.
    step_visits: optional int32 [B * Hkv * nb] tensor receiving the query steps the main pass visited per
    (b, K/V head, key tile); main_events: optional (begin, end) torch.cuda.Event pair recorded around the
    main pass (fa_bwd_ex)."""
    _check_qkv(q, o, do)
    Hkv = _check_kv(q, k, v)
    B, H, N, d = q.shape
    _masks(block_mask, seqlens_k, N, B, q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    _check_qkv(q, dq)
    _check_qkv(k, dk, dv)
    nbytes = fa_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check_aux("lse", lse, torch.float32, B * H * N, q.device)
    _check_aux("workspace", workspace, None, nbytes, q.device)
    _check_aux("status", status, torch.int32, 1, q.device)
    _check_aux("step_visits", step_visits, torch.int32, B * Hkv * ((N + 127) // 128), q.device)
    extras = None
    if step_visits is not None or main_events is not None:
        if main_events is not None:
            for e in main_events:
                if not e.cuda_event:  # torch creates its event at the first record
                    e.record()
        ev = (None, None) if main_events is None else tuple(e.cuda_event for e in main_events)
        extras = BwdExtras(_ptr(step_visits), ev[0], ev[1])
    rc = fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                   dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Hkv, N, d, int(causal), _ptr(block_mask),
                   _ptr(seqlens_k), scale, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                   extras, _ptr(status), _stream(stream))
    if rc != 0:
        raise FaError(rc)
    return dq, dk, dv


# ----------------------------------------------------------------------------- varlen / strided


def _view(t, packed):
    """Strides of a [B, N, H, d] view (or a packed [rows, H, d] tensor) as fa_strides."""
    if not (t.is_cuda and t.dtype == torch.bfloat16 and t.stride(-1) == 1):
        raise ValueError("tensors must be bf16 CUDA tensors with a contiguous last (head) dimension")
    if packed:
        if t.dim() != 3:
            raise ValueError("packed tensors are [rows, heads, d]")
        return Strides(t.stride(0), t.stride(1), 0)
    if t.dim() != 4:
        raise ValueError("fixed-length tensors are [B, N, H, d] views")
    return Strides(t.stride(1), t.stride(2), t.stride(0))


def _problem(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal, scale):
    packed = cu_seqlens_q is not None
    if packed != (cu_seqlens_k is not None):
        raise ValueError("give both cu_seqlens_q and cu_seqlens_k, or neither")
    d = q.shape[-1]
    H, Hkv = q.shape[-2], k.shape[-2]
    if packed:
        for cu in (cu_seqlens_q, cu_seqlens_k):
            if not (cu.dtype == torch.int32 and cu.is_contiguous() and cu.device == q.device and cu.dim() == 1):
                raise ValueError("cu_seqlens must be contiguous int32 [B + 1] tensors on the tensors' device")
        if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
            raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B + 1 >= 2 entries")
        if max_seqlen_q is None or max_seqlen_k is None:
            raise ValueError("packed batches need max_seqlen_q and max_seqlen_k")
        B, Nq, Nk = cu_seqlens_q.numel() - 1, int(max_seqlen_q), int(max_seqlen_k)
        rows_q, rows_k = q.shape[0], k.shape[0]
    else:
        B, Nq, Nk = q.shape[0], q.shape[1], k.shape[1]
        rows_q = rows_k = 0
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    p = VarlenProblem(B, H, Hkv, d, Nq, Nk, _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), rows_q, rows_k, int(causal),
                      scale)
    return p, packed


def _lse_shape(q, p, packed):
    return (p.H, q.shape[0]) if packed else (p.B, p.H, p.seqlen_q)


def _lse_numel(q, p, packed):
    return math.prod(_lse_shape(q, p, packed))


def _same_device(q, *ts):
    for t in ts:
        if t is not None and t.device != q.device:
            raise ValueError(f"every tensor must be on {q.device}")


def fwd_varlen(q, k, v, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None, *,
               causal=False, scale=None, out=None, lse=None, status=None, stream=None):
    """O, LSE for a fixed-length batch of [B, N, H, d] views (any strides; N_q may differ from
    N_k) or a packed batch ([rows, H, d] tensors with cu_seqlens). Causal is aligned to the
    bottom-right corner. LSE is [B, H, N_q] (fixed) or [H, rows_q] (packed)."""
    p, packed = _problem(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal, scale)
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty(_lse_shape(q, p, packed), dtype=torch.float32, device=q.device) if lse is None else lse
    _same_device(q, k, v, o)
    _check_aux("lse", lse, torch.float32, _lse_numel(q, p, packed), q.device)
    _check_aux("status", status, torch.int32, 1, q.device)
    rc = fa_fwd_varlen(p, q.data_ptr(), _view(q, packed), k.data_ptr(), _view(k, packed), v.data_ptr(),
                       _view(v, packed), o.data_ptr(), _view(o, packed), lse.data_ptr(), _ptr(status), _stream(stream))
    if rc != 0:
        raise FaError(rc)
    return o, lse


def bwd_varlen(q, k, v, o, lse, do, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None, *,
               causal=False, scale=None, dq=None, dk=None, dv=None, workspace=None, status=None, stream=None):
    """dQ, dK, dV for the batch layouts of fwd_varlen (outputs shaped like q, k, v)."""
    p, packed = _problem(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal, scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nbytes = fa_bwd_varlen_workspace_bytes(p)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _same_device(q, k, v, o, do, dq, dk, dv)
    _check_aux("lse", lse, torch.float32, _lse_numel(q, p, packed), q.device)
    _check_aux("workspace", workspace, None, nbytes, q.device)
    _check_aux("status", status, torch.int32, 1, q.device)
    rc = fa_bwd_varlen(p, q.data_ptr(), _view(q, packed), k.data_ptr(), _view(k, packed), v.data_ptr(),
                       _view(v, packed), o.data_ptr(), _view(o, packed), do.data_ptr(), _view(do, packed),
                       lse.data_ptr(), dq.data_ptr(), _view(dq, packed), dk.data_ptr(), _view(dk, packed),
                       dv.data_ptr(), _view(dv, packed), workspace.data_ptr(),
                       workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream))
    if rc != 0:
        raise FaError(rc)
    return dq, dk, dv


def _view_f32(t, packed):
    """Strides of an fp32 accumulator laid out like a bf16 tensor view (d contiguous)."""
    if not (t.is_cuda and t.dtype == torch.float32 and t.stride(-1) == 1):
        raise ValueError("accumulators must be fp32 CUDA tensors with a contiguous last (head) dimension")
    if packed:
        if t.dim() != 3:
            raise ValueError("packed accumulators are [rows, heads, d]")
        return Strides(t.stride(0), t.stride(1), 0)
    if t.dim() != 4:
        raise ValueError("fixed-length accumulators are [B, N, H, d] views")
    return Strides(t.stride(1), t.stride(2), t.stride(0))


def bwd_varlen_accumulate(q, k, v, o, lse, do, dq_acc, dk_acc, dv_acc, cu_seqlens_q=None, cu_seqlens_k=None,
                          max_seqlen_q=None, max_seqlen_k=None, *, causal=False, scale=None, workspace=None,
                          status=None, stream=None):
    """bwd_varlen whose fp32 dQ, dK, dV shares are added into dq_acc, dk_acc, dv_acc (fp32 tensors
    shaped like q, k, v) in place (fa_bwd_varlen_accumulate)."""
    p, packed = _problem(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal, scale)
    for name, acc, ref in (("dq_acc", dq_acc, q), ("dk_acc", dk_acc, k), ("dv_acc", dv_acc, v)):
        if acc.shape != ref.shape:
            raise ValueError(f"{name} must have the shape of its tensor {tuple(ref.shape)}")
    nbytes = fa_bwd_varlen_workspace_bytes(p)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _same_device(q, k, v, o, do, dq_acc, dk_acc, dv_acc)
    _check_aux("lse", lse, torch.float32, _lse_numel(q, p, packed), q.device)
    _check_aux("workspace", workspace, None, nbytes, q.device)
    _check_aux("status", status, torch.int32, 1, q.device)
    rc = int(lib().fa_bwd_varlen_accumulate(
        ctypes.byref(p), q.data_ptr(), _view(q, packed), k.data_ptr(), _view(k, packed), v.data_ptr(),
        _view(v, packed), o.data_ptr(), _view(o, packed), do.data_ptr(), _view(do, packed), lse.data_ptr(),
        dq_acc.data_ptr(), _view_f32(dq_acc, packed), dk_acc.data_ptr(), _view_f32(dk_acc, packed),
        dv_acc.data_ptr(), _view_f32(dv_acc, packed), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)))
    if rc != 0:
        raise FaError(rc)
    return dq_acc, dk_acc, dv_acc


def fwd_splitkv(q, k, v, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None, *,
                num_splits=None, causal=False, scale=None, out=None, lse=None, workspace=None, status=None,
                stream=None):
    """fwd_varlen with the key tiles split into num_splits ranges whose partial results are merged
    by their log-sum-exp (for decode shapes); num_splits=None picks about one wave of CTAs."""
    p, packed = _problem(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal, scale)
    if num_splits is None:
        num_splits = fa_fwd_splitkv_splits(p, torch.cuda.get_device_properties(q.device).multi_processor_count)
        if num_splits == 1:  # no split pays: the plain forward skips the partials and the merge
            return fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal=causal,
                              scale=scale, out=out, lse=lse, status=status, stream=stream)
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty(_lse_shape(q, p, packed), dtype=torch.float32, device=q.device) if lse is None else lse
    nbytes = fa_fwd_splitkv_workspace_bytes(p, num_splits)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _same_device(q, k, v, o)
    _check_aux("lse", lse, torch.float32, _lse_numel(q, p, packed), q.device)
    _check_aux("workspace", workspace, None, nbytes, q.device)
    _check_aux("status", status, torch.int32, 1, q.device)
    rc = fa_fwd_splitkv(p, num_splits, q.data_ptr(), _view(q, packed), k.data_ptr(), _view(k, packed), v.data_ptr(),
                        _view(v, packed), o.data_ptr(), _view(o, packed), lse.data_ptr(), workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream))
    if rc != 0:
        raise FaError(rc)
    return o, lse


# ----------------------------------------------------------------------------- partials


def fwd_partial(q, k, v, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None, *,
                causal=False, scale=None, status=None, stream=None):
    """Partial of one key block: (O fp32 [rows, d], LSE fp32 [rows]) in the LSE's row order."""
    p, packed = _problem(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal, scale)
    rows = int(lib().fa_partial_rows(ctypes.byref(p)))
    _same_device(q, k, v)
    _check_aux("status", status, torch.int32, 1, q.device)
    po = torch.empty((rows, p.d), dtype=torch.float32, device=q.device)
    pl = torch.full((rows,), float("-inf"), dtype=torch.float32, device=q.device)
    rc = int(lib().fa_fwd_partial(ctypes.byref(p), q.data_ptr(), _view(q, packed), k.data_ptr(), _view(k, packed),
                                  v.data_ptr(), _view(v, packed), po.data_ptr(), pl.data_ptr(), _ptr(status),
                                  _stream(stream)))
    if rc != 0:
        raise FaError(rc)
    return po, pl


def merge_partials(q, k, acc, part, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None,
                   *, stream=None):
    """acc <- merge(acc, part) in place (both from fwd_partial for the same query rows)."""
    p, _ = _problem(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, False, None)
    rows = int(lib().fa_partial_rows(ctypes.byref(p)))
    for name, (t_o, t_l) in (("acc", acc), ("part", part)):
        _check_aux(name + " O", t_o, torch.float32, rows * p.d, q.device)
        _check_aux(name + " LSE", t_l, torch.float32, rows, q.device)
    rc = int(lib().fa_merge_partials(ctypes.byref(p), acc[0].data_ptr(), acc[1].data_ptr(), part[0].data_ptr(),
                                     part[1].data_ptr(), _stream(stream)))
    if rc != 0:
        raise FaError(rc)
    return acc


def finalize_partials(q, k, acc, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None, *,
                      out=None, lse=None, stream=None):
    """bf16 O (shaped like q) and fp32 LSE (as fwd_varlen) from a merged accumulator."""
    p, packed = _problem(q, k, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, False, None)
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty(_lse_shape(q, p, packed), dtype=torch.float32, device=q.device) if lse is None else lse
    rows = int(lib().fa_partial_rows(ctypes.byref(p)))
    _same_device(q, o)
    _check_aux("acc O", acc[0], torch.float32, rows * p.d, q.device)
    _check_aux("acc LSE", acc[1], torch.float32, rows, q.device)
    _check_aux("lse", lse, torch.float32, _lse_numel(q, p, packed), q.device)
    rc = int(lib().fa_finalize_partials(ctypes.byref(p), acc[0].data_ptr(), acc[1].data_ptr(), o.data_ptr(),
                                        _view(o, packed), lse.data_ptr(), _stream(stream)))
    if rc != 0:
        raise FaError(rc)
    return o, lse

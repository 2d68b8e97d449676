"""FP8 (e4m3) reading of the forward pass: the quantiser and the attention it defines, in fp64.

TEST INFRASTRUCTURE (like ``oracle.attention``): only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU legs of ``bench.py`` may import this module; the CUDA library never calls it.

The pages name FP8 only as the direction FlashAttention-3 took on H100 ("FlashAttention." plate,
section "Never write the scores") and fix no scheme. The reading adopted here:

  * Inputs. Q, K and V arrive as e4m3 values with one fp32 descale factor per (sequence, head):
    the attention inputs are q = qs * Q8, k = ks * K8, v = vs * V8 (V8 is supplied transposed,
    V8^T with the keys contiguous, which is how the second product wants its operand; the
    transpose does not change what is computed).
  * What is computed. Exact attention over those dequantised inputs: O = softmax(c q k^T [mask]) v
    and LSE = ln sum_j exp(c q k_j) over the valid keys, in fp64 here (``attention_forward_fp8``).
    The fused kernel reaches it up to rounding: its scores are exact fp8 products summed in fp32;
    its probabilities P are rounded to e4m3 (after scaling by 2^8, relative to a running maximum
    that lags the row's true maximum by at most 0.8 in log2 units, so that 2^8 P <= 2^8.8 < 448
    never saturates) before the P V product. That rounding is the dominant error; its per-element
    bound is ``p_rounding_bound``.

The e4m3 format (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no infinities; the code
S.1111.111 is NaN): normal values (-1)^s 2^(e-7) (1 + m/8) for e = 1..15 (largest finite
448 = 2^8 * 1.75), subnormal values (-1)^s 2^-6 (m/8) for e = 0 (smallest 2^-9). Conversion from a
wider float rounds to the nearest value, ties to the even mantissa, and saturates to +-448
("satfinite": a finite result, never NaN, for every finite or infinite input).
"""

from __future__ import annotations

import numpy as np

from .attention import attention_forward

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_MIN_SUBNORMAL = 2.0 ** -9
P_SCALE = 256.0  # probabilities are quantised as 2^8 * P (at most 2^8.8 < 448: the running max lags by <= 0.8)


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of e4m3 bit patterns (uint8); NaN for the two NaN codes."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = s * val
    return np.where((e == 15) & ((c & 7) == 7), np.nan, val)


def e4m3_quantize(x) -> np.ndarray:
    """Round float64 values to e4m3 (nearest, ties to even), saturating to +-448; NaN stays NaN.

    Magnitudes at or above the smallest normal 2^-6 use the spacing 2^(E-3) of their binade
    [2^E, 2^(E+1)); smaller ones the subnormal spacing 2^-9. Dividing by a power of two is exact in
    float64, and ``np.rint`` rounds halves to even, so the result is the correctly rounded value.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, E = np.frexp(np.where(a > 0, a, 1.0))  # a = f 2^E with f in [0.5, 1): binade exponent E - 1
    binade = E.astype(np.float64) - 1.0
    spacing = np.where(a >= E4M3_MIN_NORMAL, np.exp2(binade - 3.0), E4M3_MIN_SUBNORMAL)
    with np.errstate(invalid="ignore"):
        q = np.rint(a / spacing) * spacing
    q = np.minimum(np.where(np.isinf(a), E4M3_MAX, q), E4M3_MAX)
    out = np.copysign(q, x)
    return np.where(np.isnan(x), np.nan, out)


def attention_forward_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, scale, causal=False, block_mask=None,
                          seqlens_k=None, workers=None):
    """O, LSE of exact attention over the dequantised FP8 inputs (fp64).

    q8 [B, H, N, d], k8 [B, Hkv, N, d] and vt8 [B, Hkv, d, N] hold e4m3 values (as floats);
    q_descale [B, H], k_descale and v_descale [B, Hkv] are the per-head factors. Masks as for
    ``attention_forward``.
    """
    q = np.asarray(q8, np.float64) * np.asarray(q_descale, np.float64)[:, :, None, None]
    k = np.asarray(k8, np.float64) * np.asarray(k_descale, np.float64)[:, :, None, None]
    v = np.swapaxes(np.asarray(vt8, np.float64), -1, -2) * np.asarray(v_descale, np.float64)[:, :, None, None]
    return attention_forward(q, k, v, scale, causal=causal, block_mask=block_mask, seqlens_k=seqlens_k,
                             workers=workers)


def p_rounding_bound(p, v_abs):
    """Per-element bound on |O - O_exact| from rounding 2^8 P to e4m3 (one row block).

    p [rows, keys] are the exact probabilities (row sums 1), v_abs [keys, d] the |v| of the keys.
    The kernel's exponentials are taken relative to a running maximum m at or below the row's true
    maximum, and it divides by their unrounded row sum l >= 1 (the row's maximum contributes at
    least 1), so the error of each weight is at most half an e4m3 spacing of 2^8 P, over 2^8:
    2^-4 P for normal values (3 mantissa bits), 2^-10 / 2^8 = 2^-18 in the subnormal range.
    Hence |dO_ik| <= sum_j max(2^-4 P_ij, 2^-18) |v_jk|.
    """
    w = np.maximum(2.0 ** -4 * np.asarray(p, np.float64), 2.0 ** -18)
    return w @ np.asarray(v_abs, np.float64)


def p_rounding_rms(p, v):
    """Expected size of the same error: each weight's rounding error is at most 2^-4 P_ij (normal
    range) and, taken as uniform on that interval and independent across keys, has variance
    (2^-4 P_ij)^2 / 3, so |dO_ik| has the root-mean-square sqrt(sum_j (2^-4 P_ij)^2 v_jk^2 / 3).
    It is an upper estimate (the half-spacing is 2^-4 P only at the bottom of a binade)."""
    w2 = (2.0 ** -4 * np.asarray(p, np.float64)) ** 2 / 3.0
    return np.sqrt(w2 @ np.asarray(v, np.float64) ** 2)

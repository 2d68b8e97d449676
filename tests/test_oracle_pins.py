"""Pins for the fp64 oracle, from what the pages and the mathematics fix (CPU only).

* Every softmax row sums to 1; Q = 0 gives the mean of the valid values with LSE = ln(count);
  one-hot keys give one-hot attention (closed form for any scale); masked attention equals
  attention over only the unmasked keys; N = 1; brute-force central finite differences of
  L = sum(dO * O); exact gradient identities; shift invariance.
* A library cross-check: torch.nn.functional.scaled_dot_product_attention in float64 (and its
  autograd) for the same textbook definition.
* Planted mistakes: each plausible slip in the oracle (dropped scale, reversed causal mask, a
  transposed block mask, log2 for ln, a dropped D term, a missing gradient scale) is planted with
  monkeypatch and must make at least one pin fail.

Sources: the FlashAttention plate ("FlashAttention.", Kernels and Efficiency plate 4, 'Never write
the scores') fixes the result as softmax(QK^T/sqrt d)V up to rounding; the essay ("Flash Attention:
IO-Aware Attention Computation", paragraph 4) describes the running max and sum; paragraph 5 the
skipping of masked blocks.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import oracle.attention as OA

RNG = np.random.default_rng(1234)


def brute_valid(i, j, causal, bm, L, tile=128):
    """Brute-force mask predicate for tiny inputs (pure Python)."""
    if causal and j > i:
        return False
    if L is not None and j >= L:
        return False
    if bm is not None and bm[i // tile][j // tile] == 0:
        return False
    return True


MASKS = [
    dict(causal=False, L=None, bm=None),
    dict(causal=True, L=None, bm=None),
    dict(causal=False, L=200, bm=None),
    dict(causal=True, L=170, bm=None),
    dict(causal=False, L=None, bm=np.array([[1, 0, 1], [0, 1, 0], [1, 1, 1]], dtype=np.uint8)),
    dict(causal=True, L=281, bm=np.array([[1, 0, 0], [1, 0, 0], [0, 1, 1]], dtype=np.uint8)),
]


def _fwd1(q, k, v, c, m):
    o, lse = oracle.attention_forward(q[None, None], k[None, None], v[None, None], c, m["causal"], m["bm"],
                                      None if m["L"] is None else np.array([m["L"]]), workers=1)
    return o[0, 0], lse[0, 0]


def _bwd1(q, k, v, do, c, m):
    g = oracle.attention_backward(q[None, None], k[None, None], v[None, None], do[None, None], c, m["causal"],
                                  m["bm"], None if m["L"] is None else np.array([m["L"]]), workers=1)
    return [x[0, 0] for x in g]


# --------------------------------------------------------------------------- pins


def pin_row_sums():
    N, d = 300, 16
    q, k = RNG.standard_normal((N, d)), RNG.standard_normal((N, d))
    for m in MASKS:
        valid = OA.valid_matrix(np.arange(N), N, m["causal"], m["bm"], m["L"])
        p, _, _ = OA.row_softmax(OA.scores(q, k, 0.25), valid)
        rs = p.sum(axis=1)
        nonempty = valid.any(axis=1)
        assert np.abs(rs[nonempty] - 1.0).max() <= 1e-14
        assert (rs[~nonempty] == 0).all()
        assert (p[~valid] == 0).all()


def pin_q_zero():
    """Q = 0: P uniform over valid keys, O_i = their mean, LSE_i = ln(count_i) exactly."""
    N, d = 300, 8
    q = np.zeros((N, d))
    k, v = RNG.standard_normal((N, d)), RNG.standard_normal((N, d))
    for m in MASKS:
        o, lse = _fwd1(q, k, v, 0.3, m)
        for i in range(N):
            js = [j for j in range(N) if brute_valid(i, j, m["causal"], m["bm"], m["L"])]
            if not js:
                assert lse[i] == -np.inf and (o[i] == 0).all()
                continue
            assert abs(lse[i] - math.log(len(js))) <= 1e-13
            assert np.abs(o[i] - v[js].mean(axis=0)).max() <= 1e-13
    # closed form of the causal count: row i sees i + 1 keys
    o, lse = _fwd1(q, k, v, 0.3, dict(causal=True, L=None, bm=None))
    assert np.abs(lse - np.log(np.arange(1, N + 1))).max() <= 1e-13


def pin_one_hot():
    """q_i = k_i = a e_i (N <= d): s_ii = c a^2, s_ij = 0. Closed forms for P, LSE and O,
    non-causal and causal; at c a^2 = 60 attention is one-hot (O_i = v_i)."""
    N, d = 12, 16
    v = RNG.standard_normal((N, d))
    for a, c in ((1.3, 0.25), (2.0, 1.0 / math.sqrt(d)), (math.sqrt(60 / 0.125), 0.125)):
        q = np.zeros((N, d))
        q[np.arange(N), np.arange(N)] = a
        k = q.copy()
        e = math.exp(c * a * a)
        o, lse = _fwd1(q, k, v, c, dict(causal=False, L=None, bm=None))
        pii = e / (e + N - 1)
        for i in range(N):
            assert abs(lse[i] - math.log(e + N - 1)) <= 1e-13 * max(1.0, abs(lse[i]))
            others = (v.sum(axis=0) - v[i]) / (N - 1)
            assert np.abs(o[i] - (pii * v[i] + (1 - pii) * others)).max() <= 1e-13
        o, lse = _fwd1(q, k, v, c, dict(causal=True, L=None, bm=None))
        for i in range(N):
            assert abs(lse[i] - math.log(e + i)) <= 1e-13 * max(1.0, abs(lse[i]))
            pii = e / (e + i)
            rest = v[:i].mean(axis=0) if i else 0.0
            assert np.abs(o[i] - (pii * v[i] + (1 - pii) * rest)).max() <= 1e-13
        if c * a * a >= 60:
            assert np.abs(o - v).max() <= 1e-12


def pin_mask_equivalence():
    """Masked attention of row i == unmasked attention over the gathered valid keys of row i."""
    N, d = 300, 8
    q, k, v = (RNG.standard_normal((N, d)) for _ in range(3))
    for m in MASKS:
        o, lse = _fwd1(q, k, v, 0.4, m)
        for i in range(0, N, 7):
            js = [j for j in range(N) if brute_valid(i, j, m["causal"], m["bm"], m["L"])]
            if not js:
                assert lse[i] == -np.inf
                continue
            oi, li = oracle.head_forward(q[i : i + 1], k[js], v[js], 0.4)
            assert np.abs(o[i] - oi[0]).max() <= 1e-13
            assert abs(lse[i] - li[0]) <= 1e-13


def pin_n1():
    d = 8
    q, k, v = (RNG.standard_normal((1, d)) for _ in range(3))
    o, lse = _fwd1(q, k, v, 0.7, dict(causal=True, L=None, bm=None))
    assert np.abs(o[0] - v[0]).max() == 0
    assert abs(lse[0] - 0.7 * float(q[0] @ k[0])) <= 1e-15


def _loss(q, k, v, do, c, m):
    o, _ = _fwd1(q, k, v, c, m)
    return float((o * do).sum())


def pin_finite_differences():
    """Central differences of L = sum(dO * O), step 1e-6, relative error <= 1e-6.

    Tiny shapes; N = 136 with d = 2 spans two 128-blocks (ragged tail) so a block mask bites."""
    cases = [
        (6, 3, dict(causal=False, L=None, bm=None)),
        (7, 4, dict(causal=True, L=None, bm=None)),
        (8, 3, dict(causal=False, L=5, bm=None)),
        (8, 2, dict(causal=True, L=6, bm=None)),
        (136, 2, dict(causal=False, L=None, bm=np.array([[1, 0], [1, 1]], dtype=np.uint8))),
        (136, 2, dict(causal=True, L=133, bm=np.array([[1, 1], [0, 1]], dtype=np.uint8))),
    ]
    h = 1e-6
    for N, d, m in cases:
        q, k, v, do = (RNG.standard_normal((N, d)) for _ in range(4))
        c = 0.6
        dq, dk, dv = _bwd1(q, k, v, do, c, m)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            flat = list(np.ndindex(x.shape))
            if len(flat) > 24:
                flat = [flat[t] for t in RNG.choice(len(flat), 24, replace=False)]
            num = np.empty(len(flat))
            ana = np.empty(len(flat))
            for t, idx in enumerate(flat):
                x0 = x[idx]
                x[idx] = x0 + h
                lp = _loss(q, k, v, do, c, m)
                x[idx] = x0 - h
                lm = _loss(q, k, v, do, c, m)
                x[idx] = x0
                num[t] = (lp - lm) / (2 * h)
                ana[t] = g[idx]
            err = np.abs(num - ana).max() / max(1e-3, np.abs(ana).max())
            assert err <= 1e-6, (N, d, m, name, err)


def pin_grad_identities():
    """sum_j dK_j = 0; sum_j dV_j = sum over non-empty rows of dO_i; shift invariance of O in K."""
    N, d = 260, 8
    q, k, v, do = (RNG.standard_normal((N, d)) for _ in range(4))
    for m in MASKS:
        dq, dk, dv = _bwd1(q, k, v, do, 0.35, m)
        valid = OA.valid_matrix(np.arange(N), N, m["causal"], m["bm"], m["L"])
        nonempty = valid.any(axis=1)
        assert np.abs(dk.sum(axis=0)).max() <= 1e-12
        assert np.abs(dv.sum(axis=0) - do[nonempty].sum(axis=0)).max() <= 1e-11
        assert (dq[~nonempty] == 0).all()
        u = RNG.standard_normal(d)
        o1, _ = _fwd1(q, k, v, 0.35, m)
        o2, _ = _fwd1(q, k + u, v, 0.35, m)
        assert np.abs(o1 - o2).max() <= 1e-12


def pin_library_crosscheck():
    """torch SDPA in float64 (CPU) with its own causal flag / boolean mask, and autograd."""
    for N, d, m in ((130, 16, dict(causal=False, L=None, bm=None)), (200, 8, dict(causal=True, L=None, bm=None)),
                    (256, 8, dict(causal=False, L=190, bm=None))):
        q, k, v, do = (RNG.standard_normal((N, d)) for _ in range(4))
        c = 1 / math.sqrt(d)
        tq, tk, tv = (torch.tensor(x[None, None], requires_grad=True) for x in (q, k, v))
        mask = None
        if m["L"] is not None:
            mask = (torch.arange(N) < m["L"])[None, :].expand(N, N)[None, None]
        to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, is_causal=m["causal"], scale=c)
        to.backward(torch.tensor(do[None, None]))
        o, _ = _fwd1(q, k, v, c, m)
        dq, dk, dv = _bwd1(q, k, v, do, c, m)
        assert np.abs(o - to.detach().numpy()[0, 0]).max() <= 1e-12
        for a, b in ((dq, tq), (dk, tk), (dv, tv)):
            assert np.abs(a - b.grad.numpy()[0, 0]).max() <= 1e-11


def pin_gqa_head_mapping():
    """Grouped-query attention: with V of K/V head hk equal to the constant 10 b + hk, every valid
    row of O of query head h equals 10 b + h // G (rows of P sum to 1), for G = H / Hkv."""
    B, H, N, d = 2, 6, 9, 4
    for Hkv in (1, 2, 3, 6):
        q = RNG.standard_normal((B, H, N, d))
        k = RNG.standard_normal((B, Hkv, N, d))
        v = np.empty((B, Hkv, N, d))
        for b in range(B):
            for hk in range(Hkv):
                v[b, hk] = 10 * b + hk
        o, _ = oracle.attention_forward(q, k, v, 0.5, causal=True, workers=1)
        G = H // Hkv
        for b in range(B):
            for h in range(H):
                assert np.abs(o[b, h] - (10 * b + h // G)).max() <= 1e-12, (Hkv, b, h)


def pin_gqa_finite_differences():
    """Central differences of L = sum(dO * O) with K/V heads shared by two or four query heads:
    each entry of a shared K or V moves the outputs of every query head of its group."""
    B, H, N, d = 1, 4, 7, 3
    h_step = 1e-6
    for Hkv, causal, L in ((2, True, None), (1, False, 5)):
        q, do = RNG.standard_normal((B, H, N, d)), RNG.standard_normal((B, H, N, d))
        k, v = RNG.standard_normal((B, Hkv, N, d)), RNG.standard_normal((B, Hkv, N, d))
        sl = None if L is None else np.array([L], dtype=np.int32)
        kw = dict(causal=causal, seqlens_k=sl, workers=1)

        def loss():
            return float((oracle.attention_forward(q, k, v, 0.7, **kw)[0] * do).sum())

        dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.7, **kw)
        assert dk.shape == k.shape and dv.shape == v.shape
        for x, g in ((q, dq), (k, dk), (v, dv)):
            flat = list(np.ndindex(x.shape))
            for idx in [flat[t] for t in RNG.choice(len(flat), 16, replace=False)]:
                x0 = x[idx]
                x[idx] = x0 + h_step
                lp = loss()
                x[idx] = x0 - h_step
                lm = loss()
                x[idx] = x0
                num = (lp - lm) / (2 * h_step)
                assert abs(num - g[idx]) <= 1e-6 * max(1.0, abs(num)), (idx, num, g[idx])


def pin_gqa_library_crosscheck():
    """torch SDPA in float64 with its own grouped-query option (K/V heads expanded by
    repeat_interleave), and autograd, against the oracle for G = 4."""
    B, H, Hkv, N, d = 1, 8, 2, 140, 16
    q, do = RNG.standard_normal((B, H, N, d)), RNG.standard_normal((B, H, N, d))
    k, v = RNG.standard_normal((B, Hkv, N, d)), RNG.standard_normal((B, Hkv, N, d))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = H // Hkv
    # torch's own expansion of shared K/V heads (the enable_gqa option applies the same rule)
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk.repeat_interleave(G, dim=1),
                                                          tv.repeat_interleave(G, dim=1), is_causal=True, scale=0.25)
    to.backward(torch.tensor(do))
    o, _ = oracle.attention_forward(q, k, v, 0.25, causal=True, workers=1)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.25, causal=True, workers=1)
    assert np.abs(o - to.detach().numpy()).max() <= 1e-12
    for a, b in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.abs(a - b.grad.numpy()).max() <= 1e-11


def pin_causal_decode_row():
    """Bottom-right causal with one query: the query is the last position, so it sees every key
    and the result equals unmasked attention of that row (and its gradients too)."""
    for Lk, d in ((1, 4), (9, 3), (130, 8)):
        q, do = RNG.standard_normal((1, d)), RNG.standard_normal((1, d))
        k, v = RNG.standard_normal((Lk, d)), RNG.standard_normal((Lk, d))
        oc, lc = OA.head_forward(q, k, v, 0.4, causal=True)
        on, ln = OA.head_forward(q, k, v, 0.4, causal=False)
        assert np.abs(oc - on).max() <= 1e-13 and np.abs(lc - ln).max() <= 1e-13
        gc = OA.head_dkdv(q, k, v, do, 0.4, causal=True)
        gn = OA.head_dkdv(q, k, v, do, 0.4, causal=False)
        for x, y in zip(gc, gn):
            assert np.abs(x - y).max() <= 1e-13


def pin_causal_front_padding():
    """Bottom-right alignment as an identity: with L_q < L_k, causal attention of the L_q queries
    equals the last L_q rows of the square causal problem whose first L_k - L_q queries are
    arbitrary; with L_q > L_k the first L_q - L_k rows see no key (O = 0, LSE = -inf) and the rest
    equal the square problem on the last L_k queries."""
    d = 5
    for Lq, Lk in ((3, 11), (40, 170), (11, 3), (170, 40)):
        q, k, v = RNG.standard_normal((Lq, d)), RNG.standard_normal((Lk, d)), RNG.standard_normal((Lk, d))
        o, lse = OA.head_forward(q, k, v, 0.7, causal=True)
        if Lq <= Lk:
            qpad = np.vstack([RNG.standard_normal((Lk - Lq, d)), q])
            os_, ls_ = OA.head_forward(qpad, k, v, 0.7, causal=True)
            assert np.abs(o - os_[Lk - Lq:]).max() <= 1e-13 and np.abs(lse - ls_[Lk - Lq:]).max() <= 1e-13
        else:
            assert (o[: Lq - Lk] == 0).all() and np.isneginf(lse[: Lq - Lk]).all()
            os_, ls_ = OA.head_forward(q[Lq - Lk:], k, v, 0.7, causal=True)
            assert np.abs(o[Lq - Lk:] - os_).max() <= 1e-13 and np.abs(lse[Lq - Lk:] - ls_).max() <= 1e-13


def pin_varlen_library_crosscheck():
    """Packed batch (ragged lengths, an empty sequence, L_q != L_k, K/V heads shared by two query
    heads) against torch SDPA in float64, one sequence at a time, with the causal mask built by
    torch's own tril at diagonal L_k - L_q; forward and autograd gradients."""
    H, Hkv, d = 4, 2, 6
    lq, lk = [5, 0, 131, 17, 1], [9, 4, 131, 3, 7]
    cu_q, cu_k = np.cumsum([0] + lq), np.cumsum([0] + lk)
    for causal in (False, True):
        q, do = RNG.standard_normal((cu_q[-1] + 2, H, d)), RNG.standard_normal((cu_q[-1] + 2, H, d))
        k, v = RNG.standard_normal((cu_k[-1], Hkv, d)), RNG.standard_normal((cu_k[-1], Hkv, d))
        o, lse = oracle.attention_forward_varlen(q, k, v, cu_q, cu_k, 0.3, causal=causal)
        dq, dk, dv = oracle.attention_backward_varlen(q, k, v, do, cu_q, cu_k, 0.3, causal=causal)
        assert (o[cu_q[-1]:] == 0).all() and np.isneginf(lse[:, cu_q[-1]:]).all()
        ref_dk, ref_dv = np.zeros_like(k), np.zeros_like(v)
        for b in range(len(lq)):
            if lq[b] == 0:
                continue
            sl_q, sl_k = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
            tq = torch.tensor(q[sl_q].transpose(1, 0, 2)[None], requires_grad=True)
            tk = torch.tensor(k[sl_k].transpose(1, 0, 2)[None], requires_grad=True)
            tv = torch.tensor(v[sl_k].transpose(1, 0, 2)[None], requires_grad=True)
            mask = None
            if causal:
                mask = torch.ones(lq[b], lk[b], dtype=torch.bool).tril(diagonal=lk[b] - lq[b])
            kk, vv = tk.repeat_interleave(H // Hkv, dim=1), tv.repeat_interleave(H // Hkv, dim=1)
            to = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, attn_mask=mask, scale=0.3)
            to = torch.nan_to_num(to)  # rows with no visible key: SDPA gives NaN, the reading is 0
            to.backward(torch.tensor(do[sl_q].transpose(1, 0, 2)[None]))
            assert np.abs(o[sl_q] - to.detach().numpy()[0].transpose(1, 0, 2)).max() <= 1e-12
            assert np.abs(dq[sl_q] - torch.nan_to_num(tq.grad).numpy()[0].transpose(1, 0, 2)).max() <= 1e-11
            ref_dk[sl_k] += torch.nan_to_num(tk.grad).numpy()[0].transpose(1, 0, 2)
            ref_dv[sl_k] += torch.nan_to_num(tv.grad).numpy()[0].transpose(1, 0, 2)
        assert np.abs(dk - ref_dk).max() <= 1e-11 and np.abs(dv - ref_dv).max() <= 1e-11


def pin_block_backward_shares():
    """Sequence-sharded backward: with the rows' final O and LSE, the per-key-block shares of
    attention_backward_block add up to the whole-sequence gradients (causal: own block square,
    earlier blocks whole, later blocks absent), for query blocks against key blocks of a 3-way
    partition, grouped K/V heads included."""
    W, blk, H, Hkv, d, c = 3, 10, 4, 2, 5, 0.4
    N = W * blk
    for causal in (False, True):
        q, do = RNG.standard_normal((1, H, N, d)), RNG.standard_normal((1, H, N, d))
        k, v = RNG.standard_normal((1, Hkv, N, d)), RNG.standard_normal((1, Hkv, N, d))
        o, lse = oracle.attention_forward(q, k, v, c, causal=causal)
        dq, dk, dv = oracle.attention_backward(q, k, v, do, c, causal=causal)
        sq, sk, sv = np.zeros_like(dq), np.zeros_like(dk), np.zeros_like(dv)
        for r in range(W):
            rq = slice(r * blk, (r + 1) * blk)
            for src in range(W):
                if causal and src > r:
                    continue
                ks = slice(src * blk, (src + 1) * blk)
                gq, gk, gv = OA.attention_backward_block(q[:, :, rq], k[:, :, ks], v[:, :, ks], o[:, :, rq],
                                                         lse[:, :, rq], do[:, :, rq], c,
                                                         causal=causal and src == r)
                sq[:, :, rq] += gq
                sk[:, :, ks] += gk
                sv[:, :, ks] += gv
        assert np.abs(sq - dq).max() <= 1e-12
        assert np.abs(sk - dk).max() <= 1e-12 and np.abs(sv - dv).max() <= 1e-12


PINS = [pin_row_sums, pin_q_zero, pin_one_hot, pin_mask_equivalence, pin_n1, pin_finite_differences,
        pin_grad_identities, pin_library_crosscheck, pin_gqa_head_mapping, pin_gqa_finite_differences,
        pin_gqa_library_crosscheck, pin_causal_decode_row, pin_causal_front_padding, pin_varlen_library_crosscheck,
        pin_block_backward_shares]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_sampled_rows_and_cols_match_full():
    """The sampled-row / sampled-column entry points used at large N equal the full oracle."""
    N, d = 300, 8
    q, k, v, do = (RNG.standard_normal((N, d)) for _ in range(4))
    for m in MASKS:
        dq, dk, dv = _bwd1(q, k, v, do, 0.3, m)
        rows = np.array([0, 5, 127, 128, 299])
        cols = np.array([1, 64, 200, 256, 299])
        sq = oracle.head_dq(q, k, v, do, 0.3, m["causal"], m["bm"], m["L"], rows=rows, chunk=2)
        sk, sv = oracle.head_dkdv(q, k, v, do, 0.3, m["causal"], m["bm"], m["L"], cols=cols)
        assert np.abs(sq - dq[rows]).max() <= 1e-13
        assert np.abs(sk - dk[cols]).max() <= 1e-13
        assert np.abs(sv - dv[cols]).max() <= 1e-13


# --------------------------------------------------------------------------- planted mistakes


def _mut_scores_no_scale(q_rows, k_cols, scale):
    return q_rows @ k_cols.T


def _mut_valid_reversed_causal(rows, n_keys, causal=False, block_mask=None, key_len=None, tile=128, offset=0):
    i = np.asarray(rows)[:, None]
    j = np.arange(n_keys)[None, :]
    ok = np.ones((i.shape[0], n_keys), dtype=bool)
    if causal:
        ok &= j >= i + offset
    if key_len is not None:
        ok &= j < key_len
    if block_mask is not None:
        ok &= np.asarray(block_mask)[i // tile, j // tile] != 0
    return ok


def _mut_valid_transposed_blocks(rows, n_keys, causal=False, block_mask=None, key_len=None, tile=128, offset=0):
    i = np.asarray(rows)[:, None]
    j = np.arange(n_keys)[None, :]
    ok = np.ones((i.shape[0], n_keys), dtype=bool)
    if causal:
        ok &= j <= i + offset
    if key_len is not None:
        ok &= j < key_len
    if block_mask is not None:
        ok &= np.asarray(block_mask)[j // tile, i // tile] != 0
    return ok


def _mut_lse_log2(m, l):
    empty = ~(l > 0)
    return np.where(empty, -np.inf, m + np.log2(np.where(empty, 1.0, l)))


_real_dkdv = OA.head_dkdv


def _mut_dkdv_no_scale(q, k, v, do, scale, causal=False, block_mask=None, key_len=None, cols=None, stats=None):
    dk, dv = _real_dkdv(q, k, v, do, scale, causal, block_mask, key_len, cols, stats)
    return dk / scale, dv


def _mut_row_stats_no_D(q, k, v, do, scale, causal=False, block_mask=None, key_len=None, chunk=1024):
    n = q.shape[0]
    m_all, l_all = np.empty(n), np.empty(n)
    for a in range(0, n, chunk):
        r = np.arange(a, min(n, a + chunk))
        valid = OA.valid_matrix(r, k.shape[0], causal, block_mask, key_len)
        _, m, l = OA.row_softmax(OA.scores(q[r], k, scale), valid)
        m_all[r], l_all[r] = m, l
    return m_all, l_all, np.zeros(n)


def _mut_kv_head_interleaved(h, H, Hkv):
    return h % Hkv


def _mut_valid_top_left(rows, n_keys, causal=False, block_mask=None, key_len=None, tile=128, offset=0):
    return _real_valid(rows, n_keys, causal, block_mask, key_len, tile, 0)


_real_valid = OA.valid_matrix


def _mut_block_local_softmax(q, k, v, o, lse, do, scale, causal=False):
    # the block's own softmax (its own LSE and D) instead of the row's over all keys
    return oracle.attention_backward(q, k, v, do, scale, causal=causal)


MUTANTS = [
    ("attention_backward_block", _mut_block_local_softmax),
    ("kv_head", _mut_kv_head_interleaved),
    ("valid_matrix", _mut_valid_top_left),
    ("scores", _mut_scores_no_scale),
    ("valid_matrix", _mut_valid_reversed_causal),
    ("valid_matrix", _mut_valid_transposed_blocks),
    ("lse_from_stats", _mut_lse_log2),
    ("head_dkdv", _mut_dkdv_no_scale),
    ("head_row_stats", _mut_row_stats_no_D),
]


@pytest.mark.parametrize("attr,mutant", MUTANTS, ids=lambda x: getattr(x, "__name__", str(x)))
def test_planted_mistake_is_caught(monkeypatch, attr, mutant):
    monkeypatch.setattr(OA, attr, mutant)
    failed = []
    for pin in PINS:
        if pin is pin_finite_differences and attr in ("lse_from_stats",):
            continue
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake in {attr}"


def test_fixed_and_packed_entries_agree_for_unequal_lengths():
    """The [B, H, N, d] entry with N_q != N_k and the packed entry (equal-length sequences) must
    give the same numbers: both reduce to the per-head functions with the bottom-right offset."""
    B, H, Hkv, Nq, Nk, d = 2, 4, 2, 7, 19, 3
    q, do = RNG.standard_normal((B, H, Nq, d)), RNG.standard_normal((B, H, Nq, d))
    k, v = RNG.standard_normal((B, Hkv, Nk, d)), RNG.standard_normal((B, Hkv, Nk, d))
    cu_q, cu_k = np.arange(B + 1) * Nq, np.arange(B + 1) * Nk
    pk = lambda x: x.transpose(0, 2, 1, 3).reshape(-1, x.shape[1], d)  # [B, H, N, d] -> [B*N, H, d]
    for causal in (False, True):
        o, lse = oracle.attention_forward(q, k, v, 0.5, causal=causal, workers=1)
        o2, lse2 = oracle.attention_forward_varlen(pk(q), pk(k), pk(v), cu_q, cu_k, 0.5, causal=causal)
        assert np.abs(pk(o) - o2).max() <= 1e-14
        assert np.array_equal(lse.transpose(1, 0, 2).reshape(H, -1), lse2)
        g1 = oracle.attention_backward(q, k, v, do, 0.5, causal=causal, workers=1)
        g2 = oracle.attention_backward_varlen(pk(q), pk(k), pk(v), pk(do), cu_q, cu_k, 0.5, causal=causal)
        for a, b in zip(g1, g2):
            assert np.abs(pk(a) - b).max() <= 1e-13

"""fp64 CPU oracle for exact (masked) scaled-dot-product attention and its gradients.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline and
reference legs of ``bench.py`` may import this module. The CUDA library never calls it, and it
shares no code with the CUDA library (only the seeded input generators are common to both).

What it computes
----------------
The plain definition. The FlashAttention plate ("FlashAttention.", Vol. XVI Kernels and Efficiency,
plate 4, section "Never write the scores") says the fused, tiled kernel returns softmax(Q K^T / sqrt d) V,
the same as standard attention apart from floating-point rounding; page 1 ("FlashAttention: Fast and
Memory-Efficient Exact Attention with IO-Awareness", abstract) calls the method exact. So the oracle
is standard, materialised attention, in float64, on the bf16 inputs upcast exactly:

  1. s_ij = c * sum_k q_ik k_jk                                  (c = softmax scale, normally 1/sqrt d)
  2. s_ij = -inf where key j is not valid for query i (see ``valid_matrix``)
  3. m_i = max_j s_ij,  l_i = sum_j exp(s_ij - m_i),  P_ij = exp(s_ij - m_i) / l_i
  4. O_i = sum_j P_ij v_j,  LSE_i = m_i + ln l_i   (natural log of the scaled scores)
     A row with no valid key has O_i = 0, LSE_i = -inf and contributes no gradient.
  5. Gradients of L = sum(dO * O) (the pages print none; textbook softmax calculus):
     dV = P^T dO;  dP = dO V^T;  D_i = sum_j P_ij dP_ij;  dS = P * (dP - D);
     dQ = c dS K;  dK = c dS^T Q.

The backward pass of the method recomputes the scores from Q, K and the saved log-sum-exp rather
than storing P (plate, "Never write the scores"); the oracle has no such constraint and simply
evaluates the formulas above.

Readings where the pages are silent (all are the plainest reading):
  * causal: key j is visible to query i iff j <= i (square, top-left aligned);
  * key padding: keys j >= L_b are masked for every query row of sequence b; query rows are not
    masked;
  * block mask: a uint8 [ceil(N/128), ceil(N/128)] grid shared by all (b, h); entry (I, J) != 0
    keeps the 128 x 128 block of queries I*128.. and keys J*128..; it is ANDed with the other two.
    Block-sparse attention is exact for the masked problem (the abstract calls it approximate only
    relative to dense attention; the essay "Flash Attention: IO-Aware Attention Computation",
    paragraph 5, describes it as skipping zero or irrelevant blocks).
  * grouped-query attention (the essay, paragraph 16, names multi-query and grouped-query
    attention, K/V heads shared across query heads, and fixes nothing more): K and V may have
    Hkv heads with Hkv dividing H; consecutive groups of G = H / Hkv query heads share one K/V
    head (query head h reads K/V head h // G, see ``kv_head``). The forward pass is the definition
    above with each K/V head repeated G times; dK and dV of a K/V head are, by the chain rule, the
    sums of the per-query-head dK and dV over its group.

Memory
------
Every output row depends only on its own row of S, so forward rows and dQ rows are evaluated in
independent chunks of rows (no sum is split). dK and dV for a set of key columns J are sums over all
query rows i; they are computed from the full column block P[:, J] in one matrix product each, so
no sum is split there either. Tests at large N evaluate a sample of rows and columns this way.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py`` (row sums, Q = 0,
one-hot keys, mask equivalence, N = 1, finite differences, gradient identities, a library
cross-check and planted mistakes). No function is "parity unpinned".
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

TILE = 128  # granularity of the block mask (128 x 128 blocks)


# ----------------------------------------------------------------------------- masks


def valid_matrix(rows, n_keys, causal=False, block_mask=None, key_len=None, tile=TILE, offset=0):
    """Boolean validity of (query row, key) pairs for one (b, h).

    rows: 1-D int array of query indices; returns bool [len(rows), n_keys].
    valid(i, j) = [not causal or j <= i + offset] and [j < key_len] and [block_mask[i // tile, j // tile] != 0]
    offset = (number of keys) - (number of queries): 0 for the square case; a query block shorter
    than its keys is aligned to the bottom-right corner (its last query sees every key).
    """
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(n_keys, dtype=np.int64)[None, :]
    ok = np.ones((i.shape[0], n_keys), dtype=bool)
    if causal:
        ok &= j <= i + offset
    if key_len is not None:
        ok &= j < int(key_len)
    if block_mask is not None:
        bm = np.asarray(block_mask)
        ok &= bm[i // tile, j // tile] != 0
    return ok


def valid_cols(cols, n_rows, causal=False, block_mask=None, key_len=None, tile=TILE, offset=0):
    """Validity for all query rows against a set of key columns: bool [n_rows, len(cols)]."""
    i = np.arange(n_rows, dtype=np.int64)[:, None]
    j = np.asarray(cols, dtype=np.int64)[None, :]
    ok = np.ones((n_rows, j.shape[1]), dtype=bool)
    if causal:
        ok &= j <= i + offset
    if key_len is not None:
        ok &= j < int(key_len)
    if block_mask is not None:
        bm = np.asarray(block_mask)
        ok &= bm[i // tile, j // tile] != 0
    return ok


# ----------------------------------------------------------------------------- one head


def scores(q_rows, k_cols, scale):
    """Step 1: s = c * Q K^T (fp64)."""
    return scale * (q_rows @ k_cols.T)


def row_softmax(s, valid):
    """Steps 2-3 for whole rows: returns P (0 where invalid), row max m and row sum l.

    For a row with no valid key, P is all zero and m = -inf, l = 0.
    """
    s = np.where(valid, s, -np.inf)
    m = s.max(axis=1)
    empty = ~valid.any(axis=1)
    m_fin = np.where(empty, 0.0, m)
    e = np.where(valid, np.exp(s - m_fin[:, None]), 0.0)
    l = e.sum(axis=1)
    p = e / np.where(empty, 1.0, l)[:, None]
    return p, m, l


def lse_from_stats(m, l):
    """Step 4: LSE_i = m_i + ln l_i, and -inf for a row with no valid key."""
    empty = ~(l > 0)
    return np.where(empty, -np.inf, m + np.log(np.where(empty, 1.0, l)))


def probs_from_stats(s, valid, m, l):
    """P_ij = exp(s_ij - m_i) / l_i for an arbitrary block of (i, j), given the row statistics
    of step 3 computed over the full rows. Zero where invalid or where row i is empty."""
    empty = ~(l > 0)
    m_fin = np.where(empty, 0.0, m)
    e = np.where(valid, np.exp(np.where(valid, s, 0.0) - m_fin[:, None]), 0.0)
    return e / np.where(empty, 1.0, l)[:, None]


def _row_chunks(rows, chunk):
    rows = np.asarray(rows, dtype=np.int64)
    for a in range(0, rows.shape[0], chunk):
        yield rows[a : a + chunk]


def head_forward(q, k, v, scale, causal=False, block_mask=None, key_len=None, rows=None, chunk=1024):
    """O and LSE of one (b, h) head for the query rows ``rows`` (default all)."""
    n = q.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    o = np.empty((rows.shape[0], v.shape[1]))
    lse = np.empty(rows.shape[0])
    at = 0
    for r in _row_chunks(rows, chunk):
        valid = valid_matrix(r, k.shape[0], causal, block_mask, key_len, offset=k.shape[0] - n)
        p, m, l = row_softmax(scores(q[r], k, scale), valid)
        o[at : at + r.shape[0]] = p @ v
        lse[at : at + r.shape[0]] = lse_from_stats(m, l)
        at += r.shape[0]
    return o, lse


def head_row_stats(q, k, v, do, scale, causal=False, block_mask=None, key_len=None, chunk=1024):
    """Row statistics m, l and D_i = sum_j P_ij dP_ij for every query row of one head."""
    n = q.shape[0]
    m_all = np.empty(n)
    l_all = np.empty(n)
    d_all = np.empty(n)
    for r in _row_chunks(np.arange(n), chunk):
        valid = valid_matrix(r, k.shape[0], causal, block_mask, key_len, offset=k.shape[0] - n)
        p, m, l = row_softmax(scores(q[r], k, scale), valid)
        dp = do[r] @ v.T
        m_all[r] = m
        l_all[r] = l
        d_all[r] = (p * dp).sum(axis=1)
    return m_all, l_all, d_all


def head_dq(q, k, v, do, scale, causal=False, block_mask=None, key_len=None, rows=None, chunk=1024):
    """dQ rows of one head: dQ_i = c * sum_j P_ij (dP_ij - D_i) k_j."""
    n = q.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    dq = np.empty((rows.shape[0], q.shape[1]))
    at = 0
    for r in _row_chunks(rows, chunk):
        valid = valid_matrix(r, k.shape[0], causal, block_mask, key_len, offset=k.shape[0] - n)
        p, _, _ = row_softmax(scores(q[r], k, scale), valid)
        dp = do[r] @ v.T
        dd = (p * dp).sum(axis=1)
        ds = p * (dp - dd[:, None])
        dq[at : at + r.shape[0]] = scale * (ds @ k)
        at += r.shape[0]
    return dq


def head_dkdv(q, k, v, do, scale, causal=False, block_mask=None, key_len=None, cols=None, stats=None):
    """dK and dV for key columns ``cols`` of one head (default all):
    dV_j = sum_i P_ij dO_i,  dK_j = c * sum_i P_ij (dP_ij - D_i) q_i.

    ``stats`` = (m, l, D) over all rows from ``head_row_stats`` (computed here when None).
    """
    n = q.shape[0]
    cols = np.arange(k.shape[0]) if cols is None else np.asarray(cols)
    if stats is None:
        stats = head_row_stats(q, k, v, do, scale, causal, block_mask, key_len)
    m, l, dd = stats
    valid = valid_cols(cols, n, causal, block_mask, key_len, offset=k.shape[0] - n)
    p = probs_from_stats(scores(q, k[cols], scale), valid, m, l)  # [n, |cols|]
    dp = do @ v[cols].T
    ds = p * (dp - dd[:, None])
    dv = p.T @ do
    dk = scale * (ds.T @ q)
    return dk, dv


# ----------------------------------------------------------------------------- [B, H, N, d]


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def _key_len(seqlens_k, b):
    return None if seqlens_k is None else int(np.asarray(seqlens_k)[b])


def _map_heads(fn, B, H, workers):
    heads = [(b, h) for b in range(B) for h in range(H)]
    if workers is None:
        workers = min(len(heads), len(os.sched_getaffinity(0)))
    if workers <= 1:
        return [fn(bh) for bh in heads]
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(fn, heads))


def kv_head(h, H, Hkv):
    """K/V head that query head h reads when H query heads share Hkv K/V heads: consecutive groups
    of G = H / Hkv query heads share one (grouped-query attention; Hkv = H is ordinary multi-head
    attention, Hkv = 1 multi-query attention)."""
    if Hkv < 1 or H % Hkv != 0:
        raise ValueError(f"{Hkv} K/V heads cannot be shared evenly by {H} query heads")
    return h // (H // Hkv)


def attention_forward(q, k, v, scale, causal=False, block_mask=None, seqlens_k=None, workers=None):
    """O [B,H,N,d] and LSE [B,H,N] in float64; q is [B, H, N, d], k and v [B, Hkv, N, d]
    (Hkv dividing H; Hkv = H for ordinary multi-head attention)."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    o = np.empty((B, H, N, v.shape[3]))
    lse = np.empty((B, H, N))

    def one(bh):
        b, h = bh
        hk = kv_head(h, H, Hkv)
        o[b, h], lse[b, h] = head_forward(q[b, h], k[b, hk], v[b, hk], scale, causal, block_mask,
                                          _key_len(seqlens_k, b))

    _map_heads(one, B, H, workers)
    return o, lse


def attention_backward(q, k, v, do, scale, causal=False, block_mask=None, seqlens_k=None, workers=None):
    """dQ [B,H,N,d] and dK, dV [B,Hkv,N,d] in float64 (the full gradient; N x N fp64 per head in
    memory). With Hkv < H, dK and dV of a K/V head sum the contributions of its query heads."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    dq = np.empty_like(q)
    dk_h = np.empty((B, H, k.shape[2], k.shape[3]))  # per query head, summed over each group below
    dv_h = np.empty((B, H, v.shape[2], v.shape[3]))

    def one(bh):
        b, h = bh
        L = _key_len(seqlens_k, b)
        hk = kv_head(h, H, Hkv)
        args = (q[b, h], k[b, hk], v[b, hk], do[b, h], scale, causal, block_mask, L)
        dq[b, h] = head_dq(*args)
        dk_h[b, h], dv_h[b, h] = head_dkdv(*args)

    _map_heads(one, B, H, workers)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            dk[b, kv_head(h, H, Hkv)] += dk_h[b, h]
            dv[b, kv_head(h, H, Hkv)] += dv_h[b, h]
    return dq, dk, dv


def attention_backward_block(q, k, v, o, lse, do, scale, causal=False):
    """One block of keys' share of the gradients, given each query row's final O and log-sum-exp
    over all of its keys: the pieces that a sequence-sharded backward pass adds up.

    q, o, do [B,H,Nq,d] and lse [B,H,Nq] belong to the query rows; k, v [B,Hkv,Nk,d] are one block
    of their keys. P_ij = exp(s_ij - LSE_i) on the block's valid keys (the row's softmax over all
    keys, restricted to the block); D_i = sum_k dO_ik O_ik (the whole row's D, from the final O);
    dP = dO V^T and dS = P * (dP - D). By the chain rule of L = sum(dO * O), the block's dV = P^T dO
    and dK = c dS^T Q, and its share of dQ is c dS K. Over a partition of the keys the shares of dQ
    add up to attention_backward's dQ, and each block's dK, dV are that block's rows of it.
    `causal` is the square (own-block) case; dK, dV of a K/V head sum its group's query heads."""
    q, k, v, o, lse, do = (_as64(x) for x in (q, k, v, o, lse, do))
    B, H, Nq, _ = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    valid = valid_matrix(np.arange(Nq), Nk, causal, offset=Nk - Nq)
    for b in range(B):
        for h in range(H):
            hk = kv_head(h, H, Hkv)
            lrow = lse[b, h][:, None]
            live = valid & np.isfinite(lrow)  # a row with no valid key anywhere has no gradient
            s = scores(q[b, h], k[b, hk], scale)
            p = np.where(live, np.exp(np.where(live, s - np.where(np.isfinite(lrow), lrow, 0.0), 0.0)), 0.0)
            dp = do[b, h] @ v[b, hk].T
            D = np.sum(do[b, h] * o[b, h], axis=1, keepdims=True)
            ds = p * (dp - D)
            dq[b, h] = scale * (ds @ k[b, hk])
            dk[b, hk] += scale * (ds.T @ q[b, h])
            dv[b, hk] += p.T @ do[b, h]
    return dq, dk, dv


def tile_grid(N, causal=False, block_mask=None, key_len=None, tile=TILE):
    """bool [nb, nb]: (query tile I, key tile J) holds at least one valid (i, j) pair, for one head.

    A fused kernel that skips exactly the blocks with no valid pair visits the True entries:
    row sums are the key tiles a query tile visits (forward), column sums the query tiles a key
    tile visits (backward).
    """
    nb = (N + tile - 1) // tile
    grid = np.zeros((nb, nb), dtype=bool)
    for it in range(nb):
        r = np.arange(it * tile, min(N, (it + 1) * tile))
        cols_any = valid_matrix(r, N, causal, block_mask, key_len, tile).any(axis=0)
        for jt in range(nb):
            grid[it, jt] = cols_any[jt * tile : (jt + 1) * tile].any()
    return grid


# ----------------------------------------------------------------------------- packed sequences


def attention_forward_varlen(q, k, v, cu_q, cu_k, scale, causal=False):
    """Packed batch: q [rows_q, H, d], k and v [rows_k, Hkv, d]; sequence b owns query rows
    cu_q[b]..cu_q[b+1] and keys cu_k[b]..cu_k[b+1]. Each (sequence, head) is the definition above
    on its own rows (causal aligned to the bottom-right corner). Returns O [rows_q, H, d] and LSE
    [H, rows_q] in float64; rows outside every sequence are left 0 and -inf."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    cu_q, cu_k = np.asarray(cu_q, dtype=np.int64), np.asarray(cu_k, dtype=np.int64)
    H, Hkv = q.shape[1], k.shape[1]
    o = np.zeros((q.shape[0], H, v.shape[2]))
    lse = np.full((H, q.shape[0]), -np.inf)
    for b in range(cu_q.shape[0] - 1):
        qa, qe, ka, ke = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if qe <= qa:
            continue
        for h in range(H):
            hk = kv_head(h, H, Hkv)
            o[qa:qe, h], lse[h, qa:qe] = head_forward(q[qa:qe, h], k[ka:ke, hk], v[ka:ke, hk], scale, causal)
    return o, lse


def attention_backward_varlen(q, k, v, do, cu_q, cu_k, scale, causal=False):
    """Gradients of L = sum(dO * O) for a packed batch (layout as attention_forward_varlen):
    dQ [rows_q, H, d], dK and dV [rows_k, Hkv, d] (summed over each K/V head's query heads);
    rows outside every sequence are 0."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    cu_q, cu_k = np.asarray(cu_q, dtype=np.int64), np.asarray(cu_k, dtype=np.int64)
    H, Hkv = q.shape[1], k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(cu_q.shape[0] - 1):
        qa, qe, ka, ke = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if qe <= qa or ke <= ka:
            continue
        for h in range(H):
            hk = kv_head(h, H, Hkv)
            args = (q[qa:qe, h], k[ka:ke, hk], v[ka:ke, hk], do[qa:qe, h], scale, causal)
            dq[qa:qe, h] = head_dq(*args)
            dkh, dvh = head_dkdv(*args)
            dk[ka:ke, hk] += dkh
            dv[ka:ke, hk] += dvh
    return dq, dk, dv

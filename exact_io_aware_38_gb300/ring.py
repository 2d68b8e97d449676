"""Sequence-sharded ring attention (forward and backward) built on the library's kernels.

The commentary on the FlashAttention paper notes that the online softmax is associative over
pieces of the key space, which is what lets ring attention shard a long sequence across devices:
rank r holds the r-th contiguous block of the queries, keys and values; in W steps every key/value
block passes every rank (rank r receives from r - 1 and sends to r + 1), and each rank folds the
attention of its queries over the block it holds into a running (O, LSE) with the log-sum-exp
merge of fa_merge_partials. Causal attention with equal blocks: the rank's own block is causal
(the square case), blocks from lower ranks are seen whole, blocks from higher ranks are skipped
(the rotation still passes them on). Each received block lands in a local buffer before it is
used (point-to-point copies, no multicast).

The backward pass follows the same schedule. With each query row's final O and log-sum-exp over
all keys, one (query block, key block) pair's share of the gradients is exactly what the fused
backward kernel computes for that pair: P = exp(c S - LSE) is the row's softmax restricted to the
block and D = rowsum(dO * O) is the whole row's. So each step runs fa_bwd_varlen on the block it
holds; the library adds each share in fp32 into the rank's dQ accumulator and the dK, dV
accumulators that travel with the K/V block (fa_bwd_varlen_accumulate), so no share is rounded to
bf16 before it is summed. After the last step a rank holds block rank + 1 and its accumulators, so
one more rotation delivers every block's dK, dV to its owner.

Out of scope: load balancing of the causal case (e.g. zig-zag block orders), overlap of the
rotation with the compute.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

import exact_io_aware_38_gb300 as fa


def ring_schedule(rank: int, world: int, causal: bool):
    """(step, source block, causal flag or None to skip) for each of the W steps of `rank`."""
    out = []
    for step in range(world):
        src = (rank - step) % world
        if causal and src > rank:
            out.append((step, src, None))
        else:
            out.append((step, src, bool(causal and src == rank)))
    return out


def rotate(tensors, group=None):
    """Send the tensors to rank + 1 and receive the same shapes from rank - 1 (ring order)."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    nxt, prv = (rank + 1) % world, (rank - 1) % world
    recv = [torch.empty_like(t) for t in tensors]
    ops = [dist.P2POp(dist.isend, t, nxt, group) for t in tensors]
    ops += [dist.P2POp(dist.irecv, t, prv, group) for t in recv]
    for req in dist.batch_isend_irecv(ops):
        req.wait()
    return recv


def ring_forward(q, k, v, *, causal=False, scale=None, group=None, partial=None, merge=None, finalize=None,
                 rotate_fn=None):
    """O, LSE of this rank's query block ([B, N_block, H, d] views) over the whole sharded
    sequence. `partial`, `merge`, `finalize` and `rotate_fn` default to the library's kernels and
    torch.distributed point-to-point copies (they are parameters so the ring's bookkeeping can be
    exercised without a GPU)."""
    partial = partial or (lambda q_, k_, v_, c_: fa.fwd_partial(q_, k_, v_, causal=c_, scale=scale))
    merge = merge or (lambda acc, part: fa.merge_partials(q, k, acc, part))
    finalize = finalize or (lambda acc: fa.finalize_partials(q, k, acc))
    rotate_fn = rotate_fn or rotate
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    kv = [k, v]
    acc = None
    for step, _src, c in ring_schedule(rank, world, causal):
        if c is not None:
            part = partial(q, kv[0], kv[1], c)
            acc = part if acc is None else merge(acc, part)
        if step + 1 < world:
            kv = rotate_fn(kv, group)
    return finalize(acc)


def ring_backward(q, k, v, o, lse, do, *, causal=False, scale=None, group=None, partial_bwd=None, rotate_fn=None):
    """dQ, dK, dV of this rank's blocks ([B, N_block, H, d] views, as for ring_forward; o and lse
    are ring_forward's results for this rank's queries, do the gradient of o). `partial_bwd`
    (q, k_blk, v_blk, o, lse, do, causal, dq_acc, dk_acc, dv_acc) adds one block pair's shares into
    the accumulators in place; it and `rotate_fn` default to the library's accumulating backward
    kernel and torch.distributed point-to-point copies."""
    partial_bwd = partial_bwd or (lambda q_, k_, v_, o_, l_, do_, c_, aq, ak, av: fa.bwd_varlen_accumulate(
        q_, k_, v_, o_, l_, do_, aq, ak, av, causal=c_, scale=scale))
    rotate_fn = rotate_fn or rotate
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    acc = torch.float32 if q.dtype in (torch.bfloat16, torch.float16) else q.dtype  # sums of the shares
    kv = [k, v]
    dq = torch.zeros(q.shape, dtype=acc, device=q.device)
    dkv = [torch.zeros(k.shape, dtype=acc, device=k.device), torch.zeros(v.shape, dtype=acc, device=v.device)]
    for step, _src, c in ring_schedule(rank, world, causal):
        if c is not None:
            partial_bwd(q, kv[0], kv[1], o, lse, do, c, dq, dkv[0], dkv[1])
        if step + 1 < world:
            moved = rotate_fn(kv + dkv, group)  # the block and its accumulators travel together
            kv, dkv = moved[:2], moved[2:]
    if world > 1:
        dkv = rotate_fn(dkv, group)  # block rank + 1's accumulators to their owner; ours arrive
    return dq.to(q.dtype), dkv[0].to(k.dtype), dkv[1].to(v.dtype)

"""Ulysses sequence parallelism around the block-sparse attention, pipelined by head group.

The deep-dive ("HeyGen Avatar IV on Trillium TPU", sections on one mesh with two
shardings and on keeping the all-to-all out of the way) runs the video sequence
sharded over the chips of a host.  Attention needs every key of a head, so an
all-to-all turns the sequence shards into head shards before the attention
kernel and a second one turns the output back.  Issued as one exchange, that
collective sat on the compute stream; split by head group into independent
exchange / attention / exchange chains whose exchanges are started
asynchronously, it overlapped the attention of the other groups and its window
on the compute stream shrank about five-fold.

Here P ranks (one process per GPU, ``torch.distributed``) each hold a
contiguous 1/P of the sequence of every head, [B, H, L/P, D].  Rank r owns
heads [r * H/P, (r+1) * H/P) for the attention; those are cut into G groups.
For each group an asynchronous all-to-all gathers the group's heads over the
whole sequence ([B, H/(P*G), L, D]), the attention runs on them (through the
C ABI on GPU ranks), and an asynchronous all-to-all sends each rank its
sequence shard of the group's output back.  The exchange of group g + 1 is in
flight while group g computes, and group g's return exchange while g + 1
computes.  With NCCL each collective is ordered after the work already queued
on the current stream, so the return exchange starts when the group's
attention is done, with no host synchronisation.

The exchanges move bytes only: bf16 rows travel as 32-bit words (D must be
even), so any backend that moves float32 moves them (gloo has no 16-bit
all-to-all).  This is the data path's only collective; one GPU per process.
"""
from __future__ import annotations

from typing import Callable, Optional

import numpy as np


def _dist():
    import torch.distributed as dist
    return dist


def _words(x):
    """A byte-preserving float32 view of a contiguous tensor whose last dim has an even number of 16-bit
    elements (or is already 32-bit)."""
    import torch
    if x.element_size() == 4:
        return x.view(torch.float32)
    assert x.element_size() == 2 and x.shape[-1] % 2 == 0, "16-bit rows of even length"
    return x.view(torch.float32)


def head_group_slices(H: int, world: int, groups: int):
    """Per rank r and group g, the global heads it computes: r * H/P + [g * Hg, (g+1) * Hg)."""
    if H % (world * groups) != 0:
        raise ValueError(f"H = {H} heads do not split into {world} ranks x {groups} groups")
    Hp, Hg = H // world, H // (world * groups)
    return [[slice(r * Hp + g * Hg, r * Hp + (g + 1) * Hg) for g in range(groups)] for r in range(world)]


def seq_to_heads_start(x_seq, g: int, groups: int, world: int, pg=None):
    """Start the exchange of group g: x_seq [B, H, Ls, D] (this rank's sequence shard) ->
    (work, recv) where, once work is done, ``finish_seq_to_heads(recv)`` is [B, Hg, P * Ls, D]: this
    rank's group-g heads over the whole sequence, shards in rank order."""
    import torch
    B, H, Ls, D = x_seq.shape
    Hp, Hg = H // world, H // (world * groups)
    # chunk j (for rank j) = heads j * Hp + g * Hg .. + Hg of the local shard
    send = x_seq.view(B, world, Hp, Ls, D)[:, :, g * Hg:(g + 1) * Hg].permute(1, 0, 2, 3, 4).contiguous()
    recv = torch.empty_like(send)  # [P (source rank), B, Hg, Ls, D]
    work = _dist().all_to_all_single(_words(recv), _words(send), group=pg, async_op=True)
    return work, recv


def finish_seq_to_heads(recv):
    P, B, Hg, Ls, D = recv.shape
    return recv.permute(1, 2, 0, 3, 4).reshape(B, Hg, P * Ls, D)


def heads_to_seq_start(o_heads, world: int, pg=None):
    """Start the return exchange of one group: o_heads [B, Hg, L, D] -> (work, recv) where recv
    [P (source rank), B, Hg, L/P, D] holds, from rank i, its group's heads over this rank's shard."""
    import torch
    B, Hg, L, D = o_heads.shape
    Ls = L // world
    send = o_heads.view(B, Hg, world, Ls, D).permute(2, 0, 1, 3, 4).contiguous()
    recv = torch.empty_like(send)
    work = _dist().all_to_all_single(_words(recv), _words(send), group=pg, async_op=True)
    return work, recv


def place_group_output(out_seq, recv, g: int, groups: int):
    """Write a finished return exchange of group g into out_seq [B, H, Ls, D]."""
    P, B, Hg, Ls, D = recv.shape
    Hp = out_seq.shape[1] // P
    view = out_seq.view(B, P, Hp, Ls, D)
    view[:, :, g * Hg:(g + 1) * Hg] = recv.permute(1, 0, 2, 3, 4)


def ulysses_attention(q_seq, k_seq, v_seq, attend: Callable, groups: int = 1, pg=None):
    """Attention of sequence-sharded Q [B, H, L/P, D] and K, V [B, H, L_kv/P, D] over P ranks.

    ``attend(q, k, v, heads)`` computes the attention of the global heads ``heads`` (a slice)
    for [B, Hg, L, D] inputs and returns O [B, Hg, L, D] (e.g. ``bsattn_group_attend``).
    Returns this rank's output shard [B, H, L/P, D].  Every rank calls it with the same shapes."""
    import torch
    dist = _dist()
    world = dist.get_world_size(pg)
    rank = dist.get_rank(pg)
    H = q_seq.shape[1]
    mine = head_group_slices(H, world, groups)[rank]
    out = torch.empty_like(q_seq)
    # all exchanges of the inputs are started up front (each group's waits only on its own)
    pending = [tuple(seq_to_heads_start(t, g, groups, world, pg) for t in (q_seq, k_seq, v_seq))
               for g in range(groups)]
    back = []
    for g in range(groups):
        for work, _ in pending[g]:
            work.wait()
        q, k, v = (finish_seq_to_heads(recv) for _, recv in pending[g])
        o = attend(q, k, v, mine[g])
        back.append(heads_to_seq_start(o.contiguous(), world, pg))
    for g, (work, recv) in enumerate(back):
        work.wait()
        place_group_output(out, recv, g, groups)
    return out


def bsattn_group_attend(block_mask, block_size: int, scale: Optional[float] = None, flags: int = 0):
    """An ``attend`` for ulysses_attention that runs the C-ABI path on the rank's GPU: the shared
    frame mask, or for a per-head mask [H, nb, nb_kv] the group's own slice."""
    from . import bsattn
    m = np.asarray(block_mask)

    def attend(q, k, v, heads: slice):
        mask = m[heads] if m.ndim == 3 else m
        return bsattn.attention(q, k, v, mask, block_size, scale, flags)
    return attend

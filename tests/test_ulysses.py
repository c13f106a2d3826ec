"""Head-grouped Ulysses exchange around the attention, on two gloo ranks (CPU, no GPU).

The deep-dive ("HeyGen Avatar IV on Trillium TPU", section on keeping the
all-to-all out of the way) turns sequence shards into head shards with an
all-to-all before the attention and back after it, split by head group so the
exchanges overlap the other groups' attention.  Here each rank holds half of
the sequence of every head; the attention of a head group is the fp64 oracle
(rounded to bf16) on CPU, standing in for the kernel.  The sharded result must
equal the oracle on the whole, unsharded problem bit for bit: the oracle
computes every row on its own, so only a misplaced head, shard or group would
change a value.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _problem(per_head):
    from block_sparse_video_row_b300 import synth
    B, H, D, frames, bs = 2, 8, 64, 4, 48
    L = frames * bs
    q = synth.tensor_bf16(31, synth.TAG_Q, B, H, L, D)
    k = synth.tensor_bf16(31, synth.TAG_K, B, H, L, D)
    v = synth.tensor_bf16(31, synth.TAG_V, B, H, L, D)
    mask = synth.mixed_head_masks(frames, H) if per_head else synth.window_mask(frames, 1, True)
    return q, k, v, mask, bs, 0.125


def _oracle_attend(mask, bs, scale):
    import oracle
    from block_sparse_video_row_b300 import synth

    def attend(q, k, v, heads):
        m = mask[heads] if mask.ndim == 3 else mask
        bits = [t.contiguous().view(torch.int16).numpy().view(np.uint16) for t in (q, k, v)]
        o, _, _ = oracle.attention(bits[0], bits[1], bits[2], m, bs, scale, nthreads=1)
        o16 = synth.f32_to_bf16_bits(o.astype(np.float32)).reshape(q.shape)
        return torch.from_numpy(o16.view(np.int16)).view(torch.bfloat16)
    return attend


def _rank_main(rank, world, port, per_head, groups, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from block_sparse_video_row_b300 import ulysses
    q, k, v, mask, bs, scale = _problem(per_head)
    L = q.shape[2]
    Ls = L // world
    shard = [torch.from_numpy(np.ascontiguousarray(t[:, :, rank * Ls:(rank + 1) * Ls]).view(np.int16))
             .view(torch.bfloat16) for t in (q, k, v)]
    # the exchange alone: group g's heads of this rank over the whole sequence
    heads = ulysses.head_group_slices(q.shape[1], world, groups)[rank]
    for g in range(groups):
        work, recv = ulysses.seq_to_heads_start(shard[0], g, groups, world)
        work.wait()
        got = ulysses.finish_seq_to_heads(recv).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, q[:, heads[g]]), (rank, g)
    o = ulysses.ulysses_attention(*shard, _oracle_attend(mask, bs, scale), groups=groups)
    out[rank] = o.view(torch.int16).numpy().view(np.uint16).copy()
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("per_head,groups", [(False, 1), (False, 2), (True, 4)])
def test_ulysses_two_ranks_equal_the_unsharded_attention(per_head, groups):
    import oracle
    from block_sparse_video_row_b300 import synth
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), per_head, groups, out), nprocs=world,
                           start_method="spawn")
        res = dict(out)
    q, k, v, mask, bs, scale = _problem(per_head)
    B, H, L, D = q.shape
    want, _, _ = oracle.attention(q, k, v, mask, bs, scale)
    want = synth.f32_to_bf16_bits(want.astype(np.float32)).reshape(B, H, L, D)
    got = np.concatenate([res[r] for r in range(world)], axis=2)
    assert np.array_equal(got, want)


def test_head_groups_must_divide_the_heads():
    from block_sparse_video_row_b300 import ulysses
    with pytest.raises(ValueError):
        ulysses.head_group_slices(24, 2, 5)
    s = ulysses.head_group_slices(24, 2, 3)
    assert s[1][2] == slice(20, 24) and s[0][0] == slice(0, 4)

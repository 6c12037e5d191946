"""Ulysses sequence parallelism around the attention forward, with CFG parallel.

The sns.style article on TensorRT LLM VisualGen and FLUX 3 Image Klein (its
multi-GPU and deployment paragraphs) runs the Base model on 8 GPUs as two
CFG groups (cfg_size 2: the conditional and unconditional halves of the
batch, no communication inside attention) of four Ulysses ranks each
(ulysses_size 4).  Between attention layers every Ulysses rank holds a slice
of the token sequence; attention needs whole sequences, so an all-to-all
turns the sequence shards into head shards before the forward (each rank
then holds H/u heads over all L tokens) and the inverse all-to-all turns the
output back into sequence shards.  The attention itself is the unchanged
library forward on H/u heads: heads are independent, so the sharded result
is the unsharded one, head by head.

Layouts (contiguous, [B, H, L, d] as the forward takes them; u = ulysses size,
r = this rank's index in its Ulysses group):

    sequence shard r:  x_r = x[:, :, r*L/u : (r+1)*L/u, :]        [B, H, L/u, d]
    head shard r:      y_r = y[:, r*H/u : (r+1)*H/u, :, :]        [B, H/u, L, d]

seq_to_head(x_r) = head shard r of the full x; head_to_seq is its inverse.
Each is one torch.distributed.all_to_all_single (NCCL between GPUs, gloo on
CPU) between two local permutations: the send buffer is the shard cut into
u blocks along the heads ([u, B, H/u, L/u, d]), and block s received from
rank s is the sequence chunk s of this rank's heads.  The permutations are
torch copies (memory layout only; no arithmetic), the exchange is the
collective, the attention is the library's kernel.

Requirements: H and L divisible by u (the pages' shapes: H = 24, L = 4608,
16896, 33280 for u = 2, 4, 8); for CFG parallel, the batch divisible by
cfg_size.
"""
from __future__ import annotations

import math

__all__ = ["pack_seq_to_head", "unpack_seq_to_head", "pack_head_to_seq", "unpack_head_to_seq",
           "seq_to_head", "head_to_seq", "attention", "ParallelGroups", "make_groups"]


def _check(x, u: int, dim: int, what: str):
    if x.dim() != 4:
        raise ValueError(f"{what} must be a [B, H, L, d] tensor")
    if u < 1 or x.shape[dim] % u:
        raise ValueError(f"{what}: dimension {dim} ({x.shape[dim]}) is not divisible by {u}")


# ----------------------------------------------------------------- local permutations
def pack_seq_to_head(x_r, u: int):
    """Send buffer of seq_to_head: [B, H, L/u, d] -> [u, B, H/u, L/u, d], block g
    holding head group g (for Ulysses rank g)."""
    _check(x_r, u, 1, "sequence shard")
    B, H, Ls, d = x_r.shape
    return x_r.reshape(B, u, H // u, Ls, d).permute(1, 0, 2, 3, 4).contiguous()


def unpack_seq_to_head(recv, u: int):
    """Receive buffer of seq_to_head -> head shard: [u, B, H/u, L/u, d] (block s
    = sequence chunk s from rank s) -> [B, H/u, L, d]."""
    _, B, Hs, Ls, d = recv.shape
    return recv.permute(1, 2, 0, 3, 4).reshape(B, Hs, u * Ls, d).contiguous()


def pack_head_to_seq(y_r, u: int):
    """Send buffer of head_to_seq: [B, H/u, L, d] -> [u, B, H/u, L/u, d], block s
    holding sequence chunk s (for Ulysses rank s)."""
    _check(y_r, u, 2, "head shard")
    B, Hs, L, d = y_r.shape
    return y_r.reshape(B, Hs, u, L // u, d).permute(2, 0, 1, 3, 4).contiguous()


def unpack_head_to_seq(recv, u: int):
    """Receive buffer of head_to_seq -> sequence shard: [u, B, H/u, L/u, d] (block
    g = head group g from rank g) -> [B, H, L/u, d]."""
    _, B, Hs, Ls, d = recv.shape
    return recv.permute(1, 0, 2, 3, 4).reshape(B, u * Hs, Ls, d).contiguous()


# ----------------------------------------------------------------- collectives
def _all_to_all(send, group):
    import torch
    import torch.distributed as dist
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send, group=group)
    return recv


def _group_size(group) -> int:
    import torch.distributed as dist
    return dist.get_world_size(group)


def seq_to_head(x_r, group=None):
    """Sequence shard [B, H, L/u, d] of this rank -> its head shard [B, H/u, L, d]."""
    u = _group_size(group)
    if u == 1:
        return x_r
    return unpack_seq_to_head(_all_to_all(pack_seq_to_head(x_r, u), group), u)


def head_to_seq(y_r, group=None):
    """Head shard [B, H/u, L, d] of this rank -> its sequence shard [B, H, L/u, d]."""
    u = _group_size(group)
    if u == 1:
        return y_r
    return unpack_head_to_seq(_all_to_all(pack_head_to_seq(y_r, u), group), u)


def attention(q_r, k_r, v_r, scale: float | None = None, group=None, forward=None):
    """Ulysses attention: sequence shards in, sequence shards out.

    q_r: [B, H, Lq/u, d], k_r and v_r: [B, H, Lk/u, d] (this rank's chunks of
    the joint sequence), bf16.  Returns this rank's chunk [B, H, Lq/u, d] of
    softmax(q k^T * scale) v over the whole sequence.  ``forward`` is the
    per-rank attention on [B, H/u, L, d] tensors (default: the library's
    CUDA forward); scale defaults to 1/sqrt(d).
    """
    if forward is None:
        from . import forward as forward
    if scale is None:
        scale = 1.0 / math.sqrt(q_r.shape[-1])
    qh, kh, vh = (seq_to_head(t, group) for t in (q_r, k_r, v_r))
    return head_to_seq(forward(qh, kh, vh, scale), group)


# ----------------------------------------------------------------- CFG x Ulysses groups
class ParallelGroups:
    """This rank's place in a cfg_size x ulysses_size layout: ranks
    c*u .. c*u + u - 1 form Ulysses group c, which takes batch slice c of the
    CFG batch (B / cfg_size elements)."""

    def __init__(self, rank: int, cfg_size: int, ulysses_size: int, ulysses_group):
        self.rank = rank
        self.cfg_size = cfg_size
        self.ulysses_size = ulysses_size
        self.cfg_index = rank // ulysses_size
        self.ulysses_rank = rank % ulysses_size
        self.ulysses_group = ulysses_group

    def batch_slice(self, B: int) -> slice:
        if B % self.cfg_size:
            raise ValueError(f"batch {B} is not divisible by cfg_size {self.cfg_size}")
        n = B // self.cfg_size
        return slice(self.cfg_index * n, (self.cfg_index + 1) * n)

    def seq_slice(self, L: int) -> slice:
        if L % self.ulysses_size:
            raise ValueError(f"sequence {L} is not divisible by ulysses_size {self.ulysses_size}")
        n = L // self.ulysses_size
        return slice(self.ulysses_rank * n, (self.ulysses_rank + 1) * n)


def make_groups(cfg_size: int, ulysses_size: int) -> ParallelGroups:
    """Create the Ulysses process groups of an initialised default group of
    cfg_size * ulysses_size ranks (every rank must call this, in the same order)."""
    import torch.distributed as dist
    world, rank = dist.get_world_size(), dist.get_rank()
    if cfg_size * ulysses_size != world:
        raise ValueError(f"cfg_size {cfg_size} x ulysses_size {ulysses_size} != world {world}")
    mine = None
    for c in range(cfg_size):
        ranks = list(range(c * ulysses_size, (c + 1) * ulysses_size))
        g = dist.new_group(ranks)
        if rank in ranks:
            mine = g
    return ParallelGroups(rank, cfg_size, ulysses_size, mine)

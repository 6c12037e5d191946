"""Ulysses sequence parallelism (with CFG parallel) on CPU ranks over gloo.

The sns.style article on TensorRT LLM VisualGen and FLUX 3 Image Klein runs
Base on 8 GPUs as cfg_size 2 x ulysses_size 4 (multi-GPU and deployment
paragraphs).  These tests run the layout exchange of that scheme with real
all-to-all collectives between processes (gloo, world sizes 2 and 4):

* seq_to_head gives each rank exactly its heads of the unsharded tensor, over
  the whole sequence, bit for bit; head_to_seq brings the sequence shard back
  bit for bit;
* the whole sharded layer, with the FP64 oracle as the per-rank attention,
  returns each rank's rows of the oracle's unsharded result bit for bit
  (attention rows are independent per (batch, head, query)).

The per-rank forward on the GPU is checked against the oracle in
tests/test_ulysses_gpu.py (one GPU, the exchange emulated by the same
permutations).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bf16_tensor(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _oracle_forward(q, k, v, scale):
    """Per-rank attention for the test: the FP64 oracle on the bf16 bit patterns."""
    import torch
    import oracle
    bits = [t.contiguous().view(torch.int16).numpy().view(np.uint16) for t in (q, k, v)]
    return torch.from_numpy(oracle.attention(*bits, scale, n_threads=1))


def _worker(rank, world, port, cfg, u, results):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import workloads as W
    from diffusion_transformer_joint_causal_b300 import ulysses
    import oracle
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        g = ulysses.make_groups(cfg, u)
        B, H, Lq, Lk, d = 2 * cfg, 12, 24, 40, 16
        rng = np.random.default_rng(77)
        qb = W.random_bf16(rng, (B, H, Lq, d))
        kb = W.random_bf16(rng, (B, H, Lk, d))
        vb = W.random_bf16(rng, (B, H, Lk, d))
        q, k, v = _bf16_tensor(qb), _bf16_tensor(kb), _bf16_tensor(vb)
        bs, hs = g.batch_slice(B), slice(g.ulysses_rank * H // u, (g.ulysses_rank + 1) * H // u)
        q_r = q[bs, :, g.seq_slice(Lq)].contiguous()
        k_r = k[bs, :, g.seq_slice(Lk)].contiguous()
        v_r = v[bs, :, g.seq_slice(Lk)].contiguous()
        # layout exchange, both directions, bit for bit
        q_h = ulysses.seq_to_head(q_r, g.ulysses_group)
        k_h = ulysses.seq_to_head(k_r, g.ulysses_group)
        assert torch.equal(q_h.view(torch.int16), q[bs, hs].contiguous().view(torch.int16))
        assert torch.equal(k_h.view(torch.int16), k[bs, hs].contiguous().view(torch.int16))
        back = ulysses.head_to_seq(q_h, g.ulysses_group)
        assert torch.equal(back.view(torch.int16), q_r.view(torch.int16))
        # the whole layer with the oracle as the per-rank attention
        scale = float(np.float32(1 / np.sqrt(d)))
        out_r = ulysses.attention(q_r, k_r, v_r, scale, g.ulysses_group, forward=_oracle_forward)
        want = oracle.attention(qb, kb, vb, scale, n_threads=1)[bs, :, g.seq_slice(Lq)]
        assert out_r.shape == want.shape
        assert np.array_equal(out_r.numpy(), want)
        results[rank] = "ok"
        dist.barrier()
    except Exception as e:   # reported to the parent, which fails the test
        results[rank] = repr(e)
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("cfg,u", [(1, 2), (1, 4), (2, 2)], ids=["u2", "u4", "cfg2xu2"])
def test_ulysses_exchange_and_layer_on_gloo(cfg, u):
    world = cfg * u
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), cfg, u, results), nprocs=world, join=True)
        res = dict(results)
    assert res == {r: "ok" for r in range(world)}, res


def test_local_permutations_invert_each_other():
    sys.path.insert(0, ROOT)
    import torch
    from diffusion_transformer_joint_causal_b300 import ulysses
    u, B, H, L, d = 4, 2, 8, 12, 4
    x = torch.arange(B * H * L * d, dtype=torch.float32).reshape(u, B, H, L // u, d)
    # emulate the exchange on one process: rank r receives block r of every rank's send buffer
    shards = [x[r] for r in range(u)]                      # sequence shards [B, H, L/u, d]
    sends = [ulysses.pack_seq_to_head(s, u) for s in shards]
    heads = [ulysses.unpack_seq_to_head(torch.stack([sends[s][r] for s in range(u)]), u)
             for r in range(u)]
    full = torch.cat(shards, dim=2)                         # [B, H, L, d]
    for r in range(u):
        assert torch.equal(heads[r], full[:, r * H // u:(r + 1) * H // u])
    sends = [ulysses.pack_head_to_seq(h, u) for h in heads]
    back = [ulysses.unpack_head_to_seq(torch.stack([sends[g][r] for g in range(u)]), u)
            for r in range(u)]
    for r in range(u):
        assert torch.equal(back[r], shards[r])


def test_indivisible_shapes_are_rejected():
    sys.path.insert(0, ROOT)
    import torch
    from diffusion_transformer_joint_causal_b300 import ulysses
    with pytest.raises(ValueError):
        ulysses.pack_seq_to_head(torch.zeros(1, 6, 4, 8), 4)      # H = 6, u = 4
    with pytest.raises(ValueError):
        ulysses.pack_head_to_seq(torch.zeros(1, 2, 10, 8), 4)     # L = 10, u = 4

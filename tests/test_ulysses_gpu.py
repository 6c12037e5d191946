"""Ulysses head shards through the CUDA forward on one GPU.

The pages' 8-GPU layout for Base at 2048x2048 is cfg_size 2 x ulysses_size 4
(sns.style article on TensorRT LLM VisualGen and FLUX 3 Image Klein,
multi-GPU and deployment paragraphs): each of the 8 ranks runs the forward on
one batch element and 6 of the 24 heads over the whole joint sequence.  Here
the 8 ranks are emulated one after another on one GPU: each rank's sequence
shards go through the same send/receive permutations as the all-to-all path
(the exchange itself, a copy of blocks, is done by indexing), the library's
forward runs on the head shard, and the output shards are reassembled.  The
result must meet the bf16 bar against the FP64 oracle on the seeded row
sample, and, with the split tail off, equal the unsharded forward bit for bit
(every head's arithmetic is the same whichever rank runs it).  The collective
itself is tested between processes in tests/test_ulysses_gloo.py.
"""
import numpy as np
import pytest

import workloads as W
from gpu_util import assert_close, oracle_sampled, to_device, to_host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dit():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_transformer_joint_causal_b300 as lib
    from diffusion_transformer_joint_causal_b300 import build
    build.build()
    lib.create()
    yield lib
    assert lib.get_device_error() == 0


def _emulated_layer(dit, q, k, v, scale, cfg, u, workspace):
    """Output of cfg x u emulated ranks, reassembled to [B, H, Lq, d]."""
    import torch
    from diffusion_transformer_joint_causal_b300 import ulysses
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    nb = B // cfg
    out = torch.empty_like(q)
    for c in range(cfg):
        bs = slice(c * nb, (c + 1) * nb)
        shards = {name: [t[bs, :, r * L // u:(r + 1) * L // u].contiguous() for r in range(u)]
                  for name, t, L in (("q", q, Lq), ("k", k, Lk), ("v", v, Lk))}
        sends = {n: [ulysses.pack_seq_to_head(s, u) for s in shards[n]] for n in shards}
        outs = []
        for r in range(u):   # rank r of the Ulysses group: receive block r from every rank
            qh, kh, vh = (ulysses.unpack_seq_to_head(torch.stack([sends[n][s][r] for s in range(u)]), u)
                          for n in ("q", "k", "v"))
            outs.append(dit.forward(qh, kh, vh, scale, workspace=workspace))
        back = [ulysses.pack_head_to_seq(o, u) for o in outs]
        for r in range(u):
            out[bs, :, r * Lq // u:(r + 1) * Lq // u] = ulysses.unpack_head_to_seq(
                torch.stack([back[g][r] for g in range(u)]), u)
    return out


@pytest.mark.parametrize("name,cfg,u", [("2048px_t2i_cfg", 2, 4), ("1024px", 1, 8),
                                        ("2048px_i2i_ref", 1, 4)])
def test_emulated_ranks_match_oracle_and_unsharded(dit, name, cfg, u):
    import torch
    w = W.workload(name)
    qh, kh, vh = W.make_qkv(w)
    q, k, v = to_device(qh), to_device(kh), to_device(vh)
    sharded = _emulated_layer(dit, q, k, v, w.scale, cfg, u, "auto")
    torch.cuda.synchronize()
    bh = np.repeat(np.arange(w.B * w.H), 64)
    rows = np.concatenate([W.sample_rows(w, b, h)[::4] for b in range(w.B) for h in range(w.H)])
    got = to_host_f64(sharded.view(w.B * w.H, w.Lq, w.d)[torch.from_numpy(bh).cuda(),
                                                           torch.from_numpy(rows).cuda()])
    assert_close(got, oracle_sampled(qh, kh, vh, w.scale, bh, rows), f"{name} cfg{cfg} x u{u}")
    unsplit = _emulated_layer(dit, q, k, v, w.scale, cfg, u, None)
    whole = dit.forward(q, k, v, w.scale, workspace=None)
    torch.cuda.synchronize()
    assert torch.equal(unsplit.view(torch.int16), whole.view(torch.int16))

"""Failure detection on the GPU without a fault: a bounded wait runs out.

The self-test kernel waits on a barrier that nothing completes; it must give
up after its limit, set the device error word (read back as TIMEOUT), and
leave the context usable for a following attention call.
"""
import numpy as np
import pytest

import workloads as W
from gpu_util import assert_close, oracle_full, to_device, to_host_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_transformer_joint_causal_b300 as dit
    from diffusion_transformer_joint_causal_b300 import build
    build.build()
    dit.create()
    assert dit.get_device_error() == 0
    assert dit.check_wait_timeout(20000) == 0          # 20 ms limit
    assert dit.get_device_error() == 6                 # TIMEOUT
    assert dit.get_device_error() == 0                 # read clears it
    rng = np.random.default_rng(3)
    q = W.random_bf16(rng, (1, 2, 300, 128))
    k = W.random_bf16(rng, (1, 2, 300, 128))
    v = W.random_bf16(rng, (1, 2, 300, 128))
    out = dit.forward(to_device(q), to_device(k), to_device(v), 0.088)
    torch.cuda.synchronize()
    assert dit.get_device_error() == 0
    assert_close(to_host_f64(out), oracle_full(q, k, v, 0.088), "after timeout")


def test_timeout_recorded_while_another_stream_reads_is_kept():
    # The read-and-clear of the error word is one atomic exchange: a TIMEOUT
    # that a kernel on stream s1 records while dit_attn_get_device_error runs
    # on an idle stream s2 is reported exactly once, never lost.
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_transformer_joint_causal_b300 as dit
    dit.create()
    assert dit.get_device_error() == 0
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    seen = []
    assert dit.check_wait_timeout(50000, s1) == 0      # gives up after 50 ms
    for _ in range(200):
        seen.append(dit.get_device_error(s2))
    seen.append(dit.get_device_error(s1))               # waits for the s1 kernel
    seen.append(dit.get_device_error(s2))
    assert seen.count(6) == 1 and all(x in (0, 6) for x in seen), seen

"""Failure paths that never fault the GPU (GPU): a bounded wait that runs out and an invalid
CE target are both reported through the status word, and the context stays usable."""
import math

import torch

import pytest
import synth_inputs as si
import tensor_transformer_layer_way_gb300 as ttl

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    assert ttl.device_status() == 0
    assert ttl.selftest_wait_timeout(2000) == ttl.TTL_ERR_TIMEOUT
    assert ttl.device_status() == 0          # cleared by the read
    bufs = [torch.ones((8, 8), device="cuda", dtype=torch.bfloat16) for _ in range(2)]
    ttl.shard_all_reduce(bufs)
    assert bufs[1][3, 3].item() == 2.0


def test_ce_target_out_of_range_sets_device_error():
    t, T, h, V = 2, 16, 64, 2 * 64
    inp = si.ce_inputs(T, h, V, seed=0)
    target = inp["target"].clone()
    target[5] = V + 3
    Ws = [w.contiguous().cuda() for w in inp["W"].chunk(t, 0)]
    out = ttl.vocab_parallel_ce(inp["H"].cuda(), Ws, target.cuda(), flags=ttl.CE_FORWARD_ONLY)
    assert ttl.device_status() == ttl.TTL_ERR_DEVICE
    loss_tok = out["stats"].reshape(3 * t + 2, T)[3 * t + 1]
    assert math.isnan(loss_tok[5].item()) and not math.isnan(loss_tok[4].item())
    assert ttl.device_status() == 0

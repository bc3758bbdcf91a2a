"""Reduce-scatter / all-gather / all-reduce over t shard buffers vs the oracle (GPU).

The oracle's mirror sums in fp32 in buffer order and rounds once, so the comparison is
bit for bit; the fp64 sum is within one bf16 ulp of it (checked by the oracle's own pins).
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
import tensor_transformer_layer_way_gb300 as ttl
from oracle import collectives
from parity import dev, f32

pytestmark = pytest.mark.gpu


def _bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def _run(mode, bufs_dev, bias_dev):
    if mode == "rs":
        ttl.shard_reduce_scatter(bufs_dev, bias_dev)
    elif mode == "ag":
        ttl.shard_all_gather(bufs_dev)
    else:
        ttl.shard_all_reduce(bufs_dev, bias_dev)
    assert ttl.device_status() == 0


@pytest.mark.parametrize("t", [1, 2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("mode", ["rs", "ag", "ar"])
@pytest.mark.parametrize("bias", [False, True])
def test_small_ragged_bit_exact(t, mode, bias):
    if mode == "ag" and bias:
        pytest.skip("all-gather takes no bias")
    T, h = 7 * t, 40                       # slabs of 7 rows; 5 vectors per row
    bufs = si.partial_sum_buffers(t, T, h, seed=100 + t)
    b = si.randn_bf16(si.generator(5), (h,), 1.0) if bias else None
    host = [f32(x) for x in bufs]
    ref = {"rs": lambda: collectives.reduce_scatter_mirror(host, None if b is None else f32(b)),
           "ag": lambda: collectives.all_gather_mirror(host),
           "ar": lambda: collectives.all_reduce_mirror(host, None if b is None else f32(b))}[mode]()
    d = dev(bufs)
    _run(mode, d, None if b is None else b.cuda())
    for j in range(t):
        np.testing.assert_array_equal(_bits(f32(d[j])), _bits(ref[j]), err_msg=f"buffer {j}")


def test_fused_all_reduce_equals_reduce_scatter_then_all_gather():
    t, T, h = 8, 8 * 33, 264
    bufs = si.partial_sum_buffers(t, T, h, seed=9)
    d1 = dev(bufs)
    d2 = dev(bufs)
    ttl.shard_all_reduce(d1)
    ttl.shard_reduce_scatter(d2)
    ttl.shard_all_gather(d2)
    for j in range(t):
        assert torch.equal(d1[j], d2[j])


def test_printed_two_card_example():
    bufs = [torch.tensor([[1.0], [2.0]]).repeat(1, 8).to(torch.bfloat16),
            torch.tensor([[3.0], [4.0]]).repeat(1, 8).to(torch.bfloat16)]
    d = dev(bufs)
    ttl.shard_reduce_scatter(d)
    assert d[0][0, 0].item() == 4.0 and d[1][1, 0].item() == 6.0      # owned halves
    assert d[0][1, 0].item() == 2.0 and d[1][0, 0].item() == 3.0      # untouched halves
    ttl.shard_all_gather(d)
    for j in range(2):
        assert d[j][:, 0].float().tolist() == [4.0, 6.0]


def test_empty_is_noop():
    d = [torch.empty((0, 16), device="cuda", dtype=torch.bfloat16) for _ in range(2)]
    ttl.shard_all_reduce(d)


@pytest.mark.parametrize("t", [2, 4, 8, 16])
def test_full_size_sweep_sampled(t):
    """b=1, s=4096, h=8192 partial sums (64 MiB each), as timed by the bench: the literal
    reduce-scatter then all-gather, and the fused all-reduce the MLP and attention blocks call.
    Sampled rows against the oracle's mirror bit for bit; whole buffers against each other."""
    cfg = si.REDUCE_SWEEP
    bufs = si.partial_sum_buffers(t, cfg.T, cfg.h, seed=cfg.seed)
    rows = torch.arange(0, cfg.T, cfg.T // 32)[:32]           # 32 rows, spread over every slab,
    rows[-1] = cfg.T - 1                                      # the last row included
    host_rows = [f32(x[rows]) for x in bufs]
    ref = collectives.all_reduce_mirror(host_rows)[0]
    d = dev(bufs)
    ttl.shard_reduce_scatter(d)
    slab = cfg.T // t
    for k, r in enumerate(rows.tolist()):
        owner = r // slab
        np.testing.assert_array_equal(_bits(f32(d[owner][r])), _bits(ref[k]))
        other = (owner + 1) % t
        assert torch.equal(d[other][r].cpu(), bufs[other][r])
    ttl.shard_all_gather(d)
    for j in range(1, t):
        assert torch.equal(d[0], d[j])
    for k, r in enumerate(rows.tolist()):
        np.testing.assert_array_equal(_bits(f32(d[t - 1][r])), _bits(ref[k]))
    fused = dev(bufs)
    del bufs
    ttl.shard_all_reduce(fused)
    assert ttl.device_status() == 0
    for j in range(t):
        assert torch.equal(fused[j], d[0]), f"fused all-reduce buffer {j} differs from RS + AG"
    r = rows.cuda()
    for j in (0, t - 1):
        np.testing.assert_array_equal(_bits(f32(fused[j][r])), _bits(ref), err_msg=f"fused buffer {j}")
    del d, fused
    torch.cuda.empty_cache()

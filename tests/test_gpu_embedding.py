"""Vocab-parallel embedding lookup and backward vs the oracle (GPU)."""
import numpy as np
import pytest
import torch

import synth_inputs as si
import tensor_transformer_layer_way_gb300 as ttl
from oracle import embedding
from parity import assert_fp32_close, dev, f32, f64

pytestmark = pytest.mark.gpu


def _inputs(t, T, h, V, seed):
    g = si.generator(seed)
    E = si.randn_bf16(g, (V, h), 1.0)
    ids = torch.randint(0, V, (T,), generator=g, dtype=torch.int64)
    ids[: T // 4] = ids[T // 4]                       # repeated ids
    dY = si.randn_bf16(g, (T, h), 1.0)
    return E, ids, dY


@pytest.mark.parametrize("t,T,h,V", [(1, 64, 64, 96), (2, 130, 136, 2 * 40), (8, 257, 256, 8 * 24)])
@pytest.mark.parametrize("literal", [True, False])
def test_lookup_bit_exact_every_buffer(t, T, h, V, literal):
    E, ids, _ = _inputs(t, T, h, V, seed=t + T)
    shards = dev([e.contiguous() for e in E.chunk(t, 0)])
    out = ttl.vocab_parallel_embedding_fwd(dev(ids), shards, literal=literal)
    assert ttl.device_status() == 0
    ref = embedding.vocab_parallel_embedding(ids.numpy(), f64(E), t)["out"]
    for i in range(t):
        np.testing.assert_array_equal(f64(out[i]), ref)
        assert torch.equal(out[i], out[0])


@pytest.mark.parametrize("t,T,h,V", [(2, 130, 136, 2 * 40), (8, 300, 256, 8 * 24)])
def test_backward_accumulates_owned_rows(t, T, h, V):
    E, ids, dY = _inputs(t, T, h, V, seed=7)
    Vs = V // t
    dE = [torch.zeros((Vs, h), device="cuda") for _ in range(t)]
    ttl.vocab_parallel_embedding_bwd(dev(ids), dev(dY), dE)
    assert ttl.device_status() == 0
    ref = embedding.vocab_parallel_embedding_backward(ids.numpy(), f64(dY), V, t)
    for i in range(t):
        assert_fp32_close(f32(dE[i]), ref[i], f"dE[{i}]")


def test_full_size_qwen3_vocab():
    """151936 x 4096 table in 8 shards of 18992 rows, 8192 token ids; every token's row is
    compared bit for bit, the gradient on the rows of 64 sampled tokens."""
    t, T, h, V = 8, 8192, 4096, 151936
    g = si.generator(6)
    E = si.randn_bf16(g, (V, h), 0.02)
    ids = torch.randint(0, V, (T,), generator=g, dtype=torch.int64)
    dY = si.randn_bf16(g, (T, h), 1.0)
    shards = dev([e.contiguous() for e in E.chunk(t, 0)])
    idd = dev(ids)
    lit = ttl.vocab_parallel_embedding_fwd(idd, shards, literal=True)
    fus = ttl.vocab_parallel_embedding_fwd(idd, shards, literal=False)
    assert ttl.device_status() == 0
    ref = E[ids]
    for i in range(t):
        assert torch.equal(lit[i].cpu(), ref) and torch.equal(fus[i], lit[i])
    Vs = V // t
    dE = [torch.zeros((Vs, h), device="cuda") for _ in range(t)]
    ttl.vocab_parallel_embedding_bwd(idd, dev(dY), dE)
    assert ttl.device_status() == 0
    rows = si.sample_indices(T, 64, 6).tolist()
    dYd = dY.double()
    for tok in rows:
        v = int(ids[tok])
        want = dYd[ids == v].sum(0).numpy()
        got = f32(dE[v // Vs][v % Vs])
        assert_fp32_close(got, want, f"dE row {v}")


def test_out_of_range_id_sets_device_error():
    t, T, h, V = 2, 16, 64, 2 * 8
    E, ids, _ = _inputs(t, T, h, V, seed=1)
    ids[3] = V + 5
    shards = dev([e.contiguous() for e in E.chunk(t, 0)])
    out = ttl.vocab_parallel_embedding_fwd(dev(ids), shards, literal=False)
    assert ttl.device_status() == ttl.TTL_ERR_DEVICE
    assert torch.count_nonzero(out[0][3]).item() == 0
    assert ttl.device_status() == 0

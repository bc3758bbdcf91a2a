"""Pins of the oracle's vocab-parallel embedding (CPU only)."""
import numpy as np
import pytest
import torch

from conftest import golden
from oracle import embedding


def test_hand_worked_example():
    g = golden("embedding_lookup_small.json")
    E = np.array(g["E"], float)
    r = embedding.vocab_parallel_embedding(g["ids"], E, g["t"])
    assert r["partials"][0].tolist() == g["partial_shard0"]
    assert r["partials"][1].tolist() == g["partial_shard1"]
    assert r["out"].tolist() == g["out"]
    dE = embedding.vocab_parallel_embedding_backward(g["ids"], np.array(g["dY"], float), E.shape[0], g["t"])
    assert dE[0].tolist() == g["dE_shard0"] and dE[1].tolist() == g["dE_shard1"]


@pytest.mark.parametrize("t", [1, 2, 8])
def test_sharded_equals_torch_embedding_and_its_gradient(t):
    rng = np.random.default_rng(t)
    V, h, T = 8 * 12, 5, 40
    E = rng.standard_normal((V, h))
    ids = rng.integers(0, V, T)
    ids[:4] = ids[4]                                   # repeated ids accumulate
    r = embedding.vocab_parallel_embedding(ids, E, t)
    Et = torch.tensor(E, requires_grad=True)
    out = torch.nn.functional.embedding(torch.tensor(ids), Et)
    np.testing.assert_array_equal(r["out"], out.detach().numpy())
    np.testing.assert_array_equal(embedding.embedding_unsharded(ids, E), r["out"])
    # exactly one shard contributes a nonzero row per token
    nz = np.stack([np.any(p != 0, axis=1) for p in r["partials"]]).sum(axis=0)
    assert np.all(nz == 1)
    dY = rng.standard_normal((T, h))
    (out * torch.tensor(dY)).sum().backward()
    dE = np.concatenate(embedding.vocab_parallel_embedding_backward(ids, dY, V, t), axis=0)
    np.testing.assert_allclose(dE, Et.grad.numpy(), rtol=1e-13, atol=1e-13)

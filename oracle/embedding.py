"""Vocab-parallel embedding lookup and its backward, in float64.

Test infrastructure only (see the package docstring).

Source: the TP/SP page "v4:Tensor Parallel 与 Sequence Parallel", section "Embedding 和 LM head:按
vocab 切": the embedding table is split by vocabulary rows into t shards (151936 / 8 = 18992
ids each); a shard outputs 0 for every token whose id it does not own, and an all-reduce
sums the shards' outputs so that each token ends up with exactly its own row.

Readings where the page is silent: shard i owns ids ``[i V/t, (i+1) V/t)``; the backward
follows the f/g placement of the same page (g after the lookup: its backward is the
identity), so every shard sees the full output gradient and accumulates, for each id it
owns, the sum of the gradient rows of the tokens that carry that id.
"""
from __future__ import annotations

import numpy as np


def shard_lookup(ids, E_shard, v0: int) -> np.ndarray:
    """One shard's partial output: ``E_shard[id - v0]`` for owned ids, 0 for the rest."""
    ids = np.asarray(ids, dtype=np.int64)
    E_shard = np.asarray(E_shard, dtype=np.float64)
    Vs, h = E_shard.shape
    out = np.zeros((ids.shape[0], h))
    local = ids - v0
    own = (local >= 0) & (local < Vs)
    out[own] = E_shard[local[own]]
    return out


def vocab_parallel_embedding(ids, E, t: int) -> dict:
    """Literal sharded lookup: t partial outputs and their sum (the all-reduce)."""
    E = np.asarray(E, dtype=np.float64)
    V = E.shape[0]
    if V % t:
        raise ValueError("t must divide V")
    Vs = V // t
    partials = [shard_lookup(ids, E[i * Vs:(i + 1) * Vs], i * Vs) for i in range(t)]
    out = partials[0].copy()
    for p in partials[1:]:
        out = out + p
    return {"partials": partials, "out": out}


def embedding_unsharded(ids, E) -> np.ndarray:
    """The single-device definition: row ``E[id]`` for every token."""
    return np.asarray(E, dtype=np.float64)[np.asarray(ids, dtype=np.int64)]


def vocab_parallel_embedding_backward(ids, dY, V: int, t: int) -> list:
    """Per shard ``dE_i[v] = sum of dY[tok] over tokens with id == i V/t + v`` (t x [V/t, h])."""
    ids = np.asarray(ids, dtype=np.int64)
    dY = np.asarray(dY, dtype=np.float64)
    Vs = V // t
    out = []
    for i in range(t):
        g = np.zeros((Vs, dY.shape[1]))
        for tok in range(ids.shape[0]):
            v = ids[tok] - i * Vs
            if 0 <= v < Vs:
                g[v] += dY[tok]
        out.append(g)
    return out

"""Vocab-parallel LM head and cross-entropy from three numbers per token.

Test infrastructure only (see the package docstring).

Source: the TP/SP page "v4:Tensor Parallel 与 Sequence Parallel", section
"Embedding 和 LM head:按 vocab 切": the vocabulary is split by rows into t shards
(151936 / 8 = 18992 ids each); the LM head is column-parallel over the vocabulary; the
cross-entropy never gathers the logits, each token combines only three numbers across
shards: the max, the sum of exponentials and the target logit.

Readings where the page is silent: shard i owns ids ``[i V/t, (i+1) V/t)``; the loss is the
mean over all tokens with no ignore index, smoothing or extra terms; each shard's sum of
exponentials is taken relative to its own max and rescaled by ``exp(m_i - M)`` when
combined (one exchange of three numbers); the logits gradient is the textbook
``(softmax - onehot) / T``.
"""
from __future__ import annotations

import numpy as np


def lm_head_logits(H, W_shard) -> np.ndarray:
    """Column-parallel LM head on one vocab shard: ``Z_i = H W_i^T`` (``W_i [V/t, h]``)."""
    return np.asarray(H, dtype=np.float64) @ np.asarray(W_shard, dtype=np.float64).T


def shard_stats(Z_i, target, v0: int) -> tuple:
    """Per token, on shard i whose ids start at ``v0``: ``m_i = max_v Z_i``,
    ``s_i = sum_v exp(Z_i - m_i)``, and ``y_i`` = the target logit if the target id is on
    this shard, else 0."""
    Z_i = np.asarray(Z_i, dtype=np.float64)
    target = np.asarray(target, dtype=np.int64)
    m = Z_i.max(axis=1)
    s = np.exp(Z_i - m[:, None]).sum(axis=1)
    Vs = Z_i.shape[1]
    local = target - v0
    own = (local >= 0) & (local < Vs)
    y = np.zeros(Z_i.shape[0])
    rows = np.nonzero(own)[0]
    y[rows] = Z_i[rows, local[rows]]
    return m, s, y


def combine(stats) -> dict:
    """Combine the t shards' (m_i, s_i, y_i): ``M = max_i m_i``,
    ``S = sum_i s_i exp(m_i - M)``, ``z_y = sum_i y_i``, ``loss_t = log S + M - z_y``."""
    ms = np.stack([st[0] for st in stats])
    ss = np.stack([st[1] for st in stats])
    ys = np.stack([st[2] for st in stats])
    M = ms.max(axis=0)
    S = (ss * np.exp(ms - M[None, :])).sum(axis=0)
    zy = ys.sum(axis=0)
    loss_tok = np.log(S) + M - zy
    return {"M": M, "S": S, "z_target": zy, "lse": M + np.log(S), "loss_tok": loss_tok,
            "loss": loss_tok.mean()}


def dlogits_shard(Z_i, target, v0: int, lse, n_tokens: int) -> np.ndarray:
    """``dZ_i[t, v] = (exp(Z_i[t, v] - lse_t) - [v0 + v == target_t]) / n_tokens``."""
    Z_i = np.asarray(Z_i, dtype=np.float64)
    d = np.exp(Z_i - np.asarray(lse)[:, None])
    local = np.asarray(target, dtype=np.int64) - v0
    Vs = Z_i.shape[1]
    rows = np.nonzero((local >= 0) & (local < Vs))[0]
    d[rows, local[rows]] -= 1.0
    return d / n_tokens


def vocab_parallel_ce(H, W, target, t: int, rows=None) -> dict:
    """The whole sharded path on (optionally) a subset of token rows.

    Per shard: logits, three statistics; combine; per-shard dlogits; and the f-backward sum
    ``dH = sum_i dZ_i W_i``.  ``n_tokens`` for the mean is always the full token count.
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    target = np.asarray(target, dtype=np.int64)
    T = H.shape[0]
    V = W.shape[0]
    if V % t:
        raise ValueError("t must divide V")
    Vs = V // t
    if rows is None:
        rows = np.arange(T)
    Hs = H[rows]
    tg = target[rows]
    Zs = [lm_head_logits(Hs, W[i * Vs:(i + 1) * Vs]) for i in range(t)]
    stats = [shard_stats(Zs[i], tg, i * Vs) for i in range(t)]
    comb = combine(stats)
    dZ = [dlogits_shard(Zs[i], tg, i * Vs, comb["lse"], T) for i in range(t)]
    dH = dZ[0] @ W[0:Vs]
    for i in range(1, t):
        dH = dH + dZ[i] @ W[i * Vs:(i + 1) * Vs]
    return {"Z": Zs, "stats": stats, "dZ": dZ, "dH": dH, **comb}


def cross_entropy_unsharded(logits, target) -> dict:
    """Textbook cross-entropy on full logits ``[T, V]``: mean of ``logsumexp - z_target``,
    gradient ``(softmax - onehot) / T``."""
    Z = np.asarray(logits, dtype=np.float64)
    target = np.asarray(target, dtype=np.int64)
    T = Z.shape[0]
    m = Z.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(Z - m).sum(axis=1, keepdims=True)))[:, 0]
    loss_tok = lse - Z[np.arange(T), target]
    p = np.exp(Z - lse[:, None])
    p[np.arange(T), target] -= 1.0
    return {"loss_tok": loss_tok, "loss": loss_tok.mean(), "dZ": p / T, "lse": lse}

"""GTP_remat weight path: shards, gather, prefetch chain, wgrad reduce-scatter, deferred finalize.

Test infrastructure only (see the package docstring).

Source: the GTP page "Generalized Tensor Parallelism(GTP)是什么?":
  * concepts "GTP_remat", "Prefetch chain", "Deferred finalize": the TP slice of a weight is
    split again; each rank keeps one piece; an all-gather rebuilds the full TP slice right
    before the GEMM and it is released afterwards; gathers follow the forward order and the
    next layer's gather is issued while the current layer computes; the weight-gradient
    reduce-scatter result is merged into main_grad one backward layer later;
  * Fig. 1 and the list under "all-gather 和 weight gradient 怎么藏在计算后面": AG(W_{i+1})
    runs beside GEMM(W_i); the chain head's gather is exposed and the other L-1 are hidden;
    every weight's first gather is synchronous (cold start); backward walks the chain in
    reverse, overlapping layer i-1's gather with layer i's dgrad; the wgrad reduce-scatter
    is asynchronous with finalize deferred one step, and the last one is synchronous
    because nothing follows it;
  * the follow-up "GTP_remat 里的各个 rank 算的是同一份数据吗?": by default the GTP_remat
    ranks process independent samples;
  * the "手算一遍" paragraph: h = 8192 square bf16 weight = 128 MiB, TP = 4 -> 32 MiB,
    GTP_remat = 8 -> 4 MiB resident, a 32x reduction.

Readings where the page is silent: the TP slice ``[K, N]`` is split by rows into g blocks of
``K/g`` rows (shard j = rows ``[j K/g, (j+1) K/g)``); on one device the g "ranks" of the
wgrad reduce-scatter are the g contiguous token groups of the batch; staging and main_grad
are float32, and finalize adds (main_grad accumulates).
"""
from __future__ import annotations

import numpy as np


def shard_rows(W, g: int) -> list:
    """Split a TP slice ``[K, N]`` into g row blocks ``[K/g, N]`` (the resident shards)."""
    W = np.asarray(W)
    K = W.shape[0]
    if K % g:
        raise ValueError("g must divide K")
    w = K // g
    return [W[j * w:(j + 1) * w].copy() for j in range(g)]


def gather(shards) -> np.ndarray:
    """All-gather of the g shards: the full TP slice, shard j's rows at block j."""
    return np.concatenate([np.asarray(s) for s in shards], axis=0)


def forward_gemm(X, W) -> np.ndarray:
    """The layer GEMM on the gathered slice, ``Y = X W``."""
    return np.asarray(X, dtype=np.float64) @ np.asarray(W, dtype=np.float64)


def dgrad_gemm(dY, W) -> np.ndarray:
    """Backward data GEMM on the gathered slice, ``dX = dY W^T``."""
    return np.asarray(dY, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def wgrad_reduce_scatter(X, dY, g: int) -> list:
    """Literal GTP wgrad: logical rank r holds token group r (rows ``[r M/g, (r+1) M/g)``) and
    computes a full-slice partial ``X_r^T dY_r``; the reduce-scatter sums the g partials and
    hands row block j of the sum to rank j.  Returns the g staging blocks ``[K/g, N]``."""
    X = np.asarray(X, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    M = X.shape[0]
    if M % g:
        raise ValueError("g must divide the token count")
    w = M // g
    partials = [X[r * w:(r + 1) * w].T @ dY[r * w:(r + 1) * w] for r in range(g)]
    K = X.shape[1]
    kb = K // g
    staging = []
    for j in range(g):
        acc = partials[0][j * kb:(j + 1) * kb].copy()
        for r in range(1, g):
            acc = acc + partials[r][j * kb:(j + 1) * kb]
        staging.append(acc)
    return staging


def forward_chain_schedule(L: int, warm: bool) -> list:
    """Event list of one forward pass over an L-layer chain (Fig. 1).

    Cold pass (``warm`` False): every weight's first gather is synchronous, so each GEMM
    waits for its own gather and nothing overlaps.  Warm pass: the head gather AG(W_0) is
    exposed; AG(W_{l+1}) is issued beside GEMM(W_l), so L-1 gathers are hidden.
    Each event is ``(kind, layer, overlapped_with)``.
    """
    ev = []
    if not warm:
        for l in range(L):
            ev.append(("gather_sync", l, None))
            ev.append(("gemm", l, None))
        return ev
    ev.append(("gather_sync", 0, None))
    for l in range(L):
        if l + 1 < L:
            ev.append(("gather_async", l + 1, ("gemm", l)))
        ev.append(("gemm", l, None))
    return ev


def backward_chain_schedule(L: int) -> list:
    """Event list of one backward pass (reverse order).

    Layer L-1's gather is the head; AG(W_{l-1}) overlaps dgrad of layer l.  The wgrad
    reduce-scatter of layer l is asynchronous and its finalize runs one backward layer
    later (at layer l-1); layer 0 is last, nothing follows it, so its reduce-scatter and
    finalize are synchronous.
    """
    ev = [("gather_sync", L - 1, None)]
    for l in range(L - 1, -1, -1):
        if l - 1 >= 0:
            ev.append(("gather_async", l - 1, ("dgrad", l)))
        ev.append(("dgrad", l, None))
        ev.append(("wgrad_rs_sync" if l == 0 else "wgrad_rs_async", l, None))
        if l + 1 < L:
            ev.append(("finalize", l + 1, None))
        if l == 0:
            ev.append(("finalize", 0, None))
    return ev


def deferred_finalize(main_grad, staging_per_layer) -> dict:
    """Apply the backward schedule's finalize events to main_grad.

    ``main_grad[l][j]`` and ``staging_per_layer[l][j]`` are float64 arrays.  Backward visits
    layers L-1, ..., 0.  At the step of layer l the finalize of layer l+1 runs (deferred one
    layer); at the last step (l = 0) layer 0 is finalized at once.  Returns the final
    main_grad and, for each step l, the sorted list of layers already finalized after it.
    """
    L = len(staging_per_layer)
    mg = [[np.asarray(b, dtype=np.float64).copy() for b in layer] for layer in main_grad]
    done = []
    updated_after_step = {}
    for l in range(L - 1, -1, -1):
        targets = ([l + 1] if l + 1 < L else []) + ([0] if l == 0 else [])
        for k in targets:
            for j, s in enumerate(staging_per_layer[k]):
                mg[k][j] = mg[k][j] + np.asarray(s, dtype=np.float64)
            done.append(k)
        updated_after_step[l] = sorted(done)
    return {"main_grad": mg, "updated_after_step": updated_after_step}


def immediate_finalize(main_grad, staging_per_layer) -> list:
    """Finalize right after each layer's wgrad (no deferral); the same final values."""
    mg = [[np.asarray(b, dtype=np.float64).copy() for b in layer] for layer in main_grad]
    for l in range(len(staging_per_layer) - 1, -1, -1):
        for j, s in enumerate(staging_per_layer[l]):
            mg[l][j] = mg[l][j] + np.asarray(s, dtype=np.float64)
    return mg


def resident_weight_bytes(h: int, tp: int, g: int, bytes_per_elem: int = 2) -> dict:
    """Memory accounting of the "手算一遍" paragraph for one square ``[h, h]`` weight."""
    full = h * h * bytes_per_elem
    tp_slice = full // tp
    resident = tp_slice // g
    return {"full": full, "tp_slice": tp_slice, "resident": resident,
            "reduction": full // resident}

"""All-reduce = reduce-scatter + all-gather over t full-shape partial-sum buffers.

Test infrastructure only (see the package docstring).

Sources:
  * TP-communication page "TP 的 communication:一层几次?每次多少数据?", concept
    "Ring all-reduce" (data cut into t blocks; reduce-scatter, then all-gather) and
    Fig. 2 (two cards, [1,2] and [3,4]: after the reduce-scatter GPU0 holds the summed
    first half 4 and GPU1 the summed second half 6; after the all-gather both hold [4,6]).
  * TP/SP page "v4:Tensor Parallel 与 Sequence Parallel", section "SP": the row-parallel
    all-reduce becomes a reduce-scatter that leaves each card its own s/t tokens, an
    all-gather rebuilds the full sequence, and all-reduce = reduce-scatter + all-gather.

Reading: buffer r owns token slab r, rows ``[r T/t, (r+1) T/t)`` (Fig. 2: GPU0 ends with
the first half).  The pages do not fix the arithmetic of the sum; the reading taken is a
float32 accumulation in buffer order 0, 1, ..., t-1 followed by one round-to-nearest-even
to bf16.  ``*_exact`` functions give the float64 sum; ``*_mirror`` functions perform that
float32/bf16 sequence so that a bit-for-bit comparison is possible.
"""
from __future__ import annotations

import numpy as np

from .numerics import round_to_bf16


def slab_rows(T: int, t: int, r: int) -> slice:
    """Token slab owned by buffer r."""
    if T % t:
        raise ValueError("t must divide the token count")
    w = T // t
    return slice(r * w, (r + 1) * w)


def all_reduce_exact(bufs, bias=None) -> np.ndarray:
    """float64 ``sum_j P_j`` (+ the row bias once)."""
    s = np.asarray(bufs[0], dtype=np.float64).copy()
    for b in bufs[1:]:
        s = s + np.asarray(b, dtype=np.float64)
    if bias is not None:
        s = s + np.asarray(bias, dtype=np.float64)
    return s


def _sum_fp32_in_order(parts, bias=None) -> np.ndarray:
    acc = np.asarray(parts[0], dtype=np.float32).copy()
    for p in parts[1:]:
        acc = (acc + np.asarray(p, dtype=np.float32)).astype(np.float32)
    if bias is not None:
        acc = (acc + np.asarray(bias, dtype=np.float32)).astype(np.float32)
    return acc


def reduce_scatter_mirror(bufs, bias=None) -> list:
    """Reduce-scatter in place: buffer r's slab r becomes bf16(fp32 sum over buffers, in
    order), every other slab of every buffer is left as it was.  Inputs and outputs are
    float32 arrays holding bf16 values."""
    t = len(bufs)
    T = np.asarray(bufs[0]).shape[0]
    out = [np.asarray(b, dtype=np.float32).copy() for b in bufs]
    for r in range(t):
        sl = slab_rows(T, t, r)
        out[r][sl] = round_to_bf16(_sum_fp32_in_order([np.asarray(b)[sl] for b in bufs], bias))
    return out


def all_gather_mirror(bufs) -> list:
    """All-gather in place: slab r of buffer r is copied into slab r of every buffer."""
    t = len(bufs)
    T = np.asarray(bufs[0]).shape[0]
    src = [np.asarray(b, dtype=np.float32) for b in bufs]
    out = [b.copy() for b in src]
    for r in range(t):
        sl = slab_rows(T, t, r)
        for j in range(t):
            out[j][sl] = src[r][sl]
    return out


def all_reduce_mirror(bufs, bias=None) -> list:
    """All-reduce as the two phases in sequence: reduce-scatter, then all-gather."""
    return all_gather_mirror(reduce_scatter_mirror(bufs, bias))


def ring_all_reduce_steps(vectors) -> dict:
    """The ring schedule of Fig. 2 written out for t ranks, one chunk per rank.

    Rank r starts with vector r, cut into t chunks.  Reduce-scatter: in step k
    (k = 0..t-2) rank r sends chunk ``(r - k - 1) mod t`` to rank r+1, which adds it to
    its own copy of that chunk.  After t-1 steps rank r holds the complete sum of chunk r
    (Fig. 2: GPU0 sends its second half, GPU1 its first, and GPU0 ends with the first
    half's sum).  All-gather: in step k rank r passes chunk ``(r - k) mod t`` on, and the
    receiver overwrites its copy; after t-1 steps every rank holds every sum.
    Returns the per-rank state after the reduce-scatter and after the all-gather,
    and how many chunks each rank sent.
    """
    t = len(vectors)
    state = [np.asarray(v, dtype=np.float64).copy() for v in vectors]
    n = state[0].shape[0]
    if n % t:
        raise ValueError("t must divide the vector length")
    w = n // t

    def chunk(i):
        return slice((i % t) * w, (i % t + 1) * w)

    sent = [0] * t
    for k in range(t - 1):
        msgs = [(r, (r - k - 1) % t, state[r][chunk(r - k - 1)].copy()) for r in range(t)]
        for r, c, data in msgs:
            dst = (r + 1) % t
            state[dst][chunk(c)] = state[dst][chunk(c)] + data
            sent[r] += 1
    after_rs = [s.copy() for s in state]
    for k in range(t - 1):
        msgs = [(r, (r - k) % t, state[r][chunk(r - k)].copy()) for r in range(t)]
        for r, c, data in msgs:
            dst = (r + 1) % t
            state[dst][chunk(c)] = data
            sent[r] += 1
    return {"after_reduce_scatter": after_rs, "after_all_gather": state,
            "chunks_sent": sent, "chunk_len": w}

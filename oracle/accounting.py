"""Closed forms for the communication and memory accounting the pages derive.

Test infrastructure only (see the package docstring).  These give the units the bench and
the tests reason with; each is pinned to the numbers the pages print.

Sources: TP-communication page "TP 的 communication:一层几次?每次多少数据?", section
"推导 / 关键公式" (count = 2 forward + 2 backward per layer; ``S = b s h x 2`` bytes;
``T_AR ~ 2(t-1)/t * S / B``; per layer per rank ``8 b s h (t-1)/t`` elements; FLOPs per
communicated byte ``24 b s h^2 / t  /  (2 x 2 b s h x 2(t-1)/t) = 3h/(t-1)``) and section
"手算例子" (the t = 2 / 80 MB / 40 GB/s exercise and the b=1, s=4096, h=8192 table).
"""
from __future__ import annotations


def allreduces_per_layer() -> int:
    """Two g all-reduces in forward (attention out-proj, fc2) plus two f in backward."""
    return 2 + 2


def partial_sum_bytes(b: int, s: int, h: int, bytes_per_elem: int = 2) -> int:
    """``S = b s h`` elements of bf16."""
    return b * s * h * bytes_per_elem


def ring_bytes_per_rank(t: int, S: float) -> float:
    """Bytes each rank sends in a ring all-reduce: ``2 (t-1)/t * S``."""
    return 2.0 * (t - 1) / t * S


def allreduce_time(t: int, S: float, B: float) -> float:
    """``T_AR ~ 2 (t-1)/t * S / B`` seconds for per-rank bandwidth ``B`` bytes/s."""
    return ring_bytes_per_rank(t, S) / B


def elements_moved_per_layer(b: int, s: int, h: int, t: int) -> float:
    """Forward + backward elements each rank moves per layer: ``8 b s h (t-1)/t``."""
    return 8.0 * b * s * h * (t - 1) / t


def flops_per_comm_byte(b: int, s: int, h: int, t: int) -> float:
    """Per-rank GEMM FLOPs of one layer (``24 b s h^2 / t``) over its forward all-reduce
    bytes (``2 x 2(t-1)/t x 2 b s h``); algebraically ``3h/(t-1)``."""
    flops = 24.0 * b * s * h * h / t
    comm = 2.0 * ring_bytes_per_rank(t, partial_sum_bytes(b, s, h))
    return flops / comm

"""Pins of the oracle's reduce-scatter / all-gather / all-reduce (CPU only)."""
import numpy as np
import pytest

from conftest import golden
from oracle import collectives, numerics


def test_two_card_figure():
    g = golden("ring_allreduce_2card.json")
    vecs = [np.array(v, float) for v in g["inputs"]]
    ring = collectives.ring_all_reduce_steps(vecs)
    owned = [ring["after_reduce_scatter"][r][r] for r in range(2)]
    assert owned == g["after_reduce_scatter_owned"]
    assert [s.tolist() for s in ring["after_all_gather"]] == g["after_all_gather"]
    assert ring["chunks_sent"] == [g["chunks_sent_per_rank"]] * 2
    # The same semantics written as slab ownership over [T=2, 1] buffers.
    bufs = [np.array(v, np.float32).reshape(2, 1) for v in g["inputs"]]
    rs = collectives.reduce_scatter_mirror(bufs)
    assert [float(rs[r][r, 0]) for r in range(2)] == g["after_reduce_scatter_owned"]
    # slabs a buffer does not own are untouched by the reduce-scatter
    assert float(rs[0][1, 0]) == 2.0 and float(rs[1][0, 0]) == 3.0
    ar = collectives.all_reduce_mirror(bufs)
    assert [b[:, 0].tolist() for b in ar] == g["after_all_gather"]


@pytest.mark.parametrize("t", [2, 3, 4, 8, 16])
def test_ring_schedule_equals_slab_semantics(t):
    rng = np.random.default_rng(t)
    T = 4 * t
    vecs = [rng.integers(-8, 9, T).astype(float) for _ in range(t)]   # sums stay bf16-exact
    ring = collectives.ring_all_reduce_steps(vecs)
    bufs = [v.astype(np.float32).reshape(T, 1) for v in vecs]
    rs = collectives.reduce_scatter_mirror(bufs)
    for r in range(t):
        sl = collectives.slab_rows(T, t, r)
        np.testing.assert_array_equal(ring["after_reduce_scatter"][r][sl], rs[r][sl, 0])
    ar = collectives.all_reduce_mirror(bufs)
    total = np.sum(vecs, axis=0)
    for r in range(t):
        np.testing.assert_array_equal(ring["after_all_gather"][r], total)
        np.testing.assert_array_equal(ar[r][:, 0], total)
    # each rank sends 2(t-1) chunks of S/t: 2(t-1)/t of the data
    assert ring["chunks_sent"] == [2 * (t - 1)] * t


def test_mirror_is_fp32_in_order_then_one_rounding():
    # Values chosen so the order of the fp32 sum matters: 2^24 + 1 - 2^24.
    a = np.full((3, 1), 2.0 ** 24, np.float32)
    b = np.full((3, 1), 1.0, np.float32)
    c = np.full((3, 1), -(2.0 ** 24), np.float32)
    out = collectives.all_reduce_mirror([a, b, c])
    assert float(out[0][0, 0]) == 0.0          # (2^24 + 1) rounds to 2^24 in fp32 first
    out2 = collectives.all_reduce_mirror([a, c, b])
    assert float(out2[0][0, 0]) == 1.0


@pytest.mark.parametrize("t", [1, 2, 4, 8, 16])
def test_mirror_within_one_bf16_ulp_of_exact_sum(t):
    rng = np.random.default_rng(100 + t)
    T, h = 2 * t, 64
    bufs = [numerics.round_to_bf16(rng.standard_normal((T, h)).astype(np.float32)) for _ in range(t)]
    ar = collectives.all_reduce_mirror(bufs)
    exact = collectives.all_reduce_exact(bufs)
    ulp = np.abs(np.spacing(exact.astype(np.float32))) * 2.0 ** 16
    assert np.all(np.abs(ar[0] - exact) <= ulp + 1e-30)
    for r in range(t):
        np.testing.assert_array_equal(ar[r], ar[0])
    if t == 1:
        np.testing.assert_array_equal(ar[0], bufs[0])


def test_all_gather_leaves_owned_slabs_and_copies_bits():
    rng = np.random.default_rng(7)
    t, T, h = 4, 8, 5
    bufs = [numerics.round_to_bf16(rng.standard_normal((T, h)).astype(np.float32)) for _ in range(t)]
    ag = collectives.all_gather_mirror(bufs)
    for r in range(t):
        sl = collectives.slab_rows(T, t, r)
        for j in range(t):
            np.testing.assert_array_equal(ag[j][sl].view(np.uint32), bufs[r][sl].view(np.uint32))


def test_bias_added_once():
    bufs = [np.ones((4, 3), np.float32) for _ in range(4)]
    b = np.array([10.0, 20.0, 30.0], np.float32)
    ar = collectives.all_reduce_mirror(bufs, bias=b)
    np.testing.assert_array_equal(ar[2][0], [14.0, 24.0, 34.0])
    np.testing.assert_array_equal(collectives.all_reduce_exact(bufs, b)[0], [14.0, 24.0, 34.0])

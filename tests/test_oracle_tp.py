"""Pins of the oracle's TP linears and MLP block (CPU only).

Each check ties the oracle to something other than itself: numbers the pages print,
the single-device definition, torch's own activation routines, finite differences of a
scalar loss, or scalar triple loops on tiny inputs.
"""
import numpy as np
import pytest
import torch

from conftest import golden
from oracle import numerics, tp_mlp

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


# ---------------------------------------------------------------- printed examples

def test_column_and_row_split_2x2_printed_example():
    g = golden("tp_split_2x2.json")
    X = np.array(g["X"], float)
    A = np.array(g["A"], float)
    col = tp_mlp.column_parallel_forward(X, tp_mlp.split_columns(A, 2))
    assert [c.tolist() for c in col] == g["column_split"]["outputs"]
    assert np.concatenate(col, axis=1).tolist() == g["XA"]
    X_sl = [X[:, 0:1], X[:, 1:2]]
    parts = tp_mlp.row_parallel_partials(X_sl, tp_mlp.split_rows(A, 2))
    assert [p.tolist() for p in parts] == g["row_split"]["partials"]
    assert (parts[0] + parts[1]).tolist() == g["row_split"]["sum"]


def test_column_parallel_t3_printed_table():
    g = golden("column_parallel_t3.json")
    X = np.array(g["X"], float)
    W = np.array(g["W"], float)
    dY = np.array(g["dY"], float)
    Wsh = tp_mlp.split_columns(W, 3)
    Y = tp_mlp.column_parallel_forward(X, Wsh)
    assert [float(y[0, 0]) for y in Y] == g["Y_per_shard"]
    dY_sh = tp_mlp.split_columns(dY, 3)
    assert [float(d[0, 0]) for d in dY_sh] == g["dY_per_shard"]
    dW, pieces, dX = tp_mlp.column_parallel_backward(X, Wsh, dY_sh)
    assert [d[:, 0].tolist() for d in dW] == g["dW_per_shard"]
    assert [p[0].tolist() for p in pieces] == g["dX_pieces"]
    assert dX[0].tolist() == g["dX_all_reduced"]



def test_row_parallel_backward_2x2_example_and_finite_differences():
    """Row layer backward (table "Column 和 Row 各在哪里通信": dY is full on every shard, both
    gradients are local).  The printed 2x2 row split X = [1, 2], A = [[1,2],[3,4]] is run
    backwards with dY = [1, 1]: dX_i = dY A_i^T gives [3] and [7], dA_i = X_i^T dY gives
    [[1, 1]] and [[2, 2]].  Then central differences of sum_i sum(P_i * dY) on a random case, and
    the invariant that the dX slices side by side are the unsharded dY A^T."""
    g = golden("tp_split_2x2.json")
    X = np.array(g["X"], float)
    A = np.array(g["A"], float)
    X_sl = [X[:, 0:1], X[:, 1:2]]
    dY = np.array([[1.0, 1.0]])
    dW, dX = tp_mlp.row_parallel_backward(X_sl, tp_mlp.split_rows(A, 2), dY)
    assert [d.tolist() for d in dX] == [[[3.0]], [[7.0]]]
    assert [d.tolist() for d in dW] == [[[1.0, 1.0]], [[2.0, 2.0]]]

    rng = np.random.default_rng(41)
    T, k, n, t = 3, 6, 4, 3
    Xf = rng.standard_normal((T, k))
    W = rng.standard_normal((k, n))
    dY = rng.standard_normal((T, n))
    Wsh = tp_mlp.split_rows(W, t)
    X_sl = [Xf[:, i * (k // t):(i + 1) * (k // t)] for i in range(t)]
    dW, dX = tp_mlp.row_parallel_backward(X_sl, Wsh, dY)

    def loss(xs, ws):
        return sum(np.sum(p * dY) for p in tp_mlp.row_parallel_partials(xs, ws))
    eps = 1e-6
    for i in range(t):
        for idx in np.ndindex(X_sl[i].shape):
            a = [x.copy() for x in X_sl]; a[i][idx] += eps
            b = [x.copy() for x in X_sl]; b[i][idx] -= eps
            assert abs((loss(a, Wsh) - loss(b, Wsh)) / (2 * eps) - dX[i][idx]) < 1e-7
        for idx in np.ndindex(Wsh[i].shape):
            a = [w.copy() for w in Wsh]; a[i][idx] += eps
            b = [w.copy() for w in Wsh]; b[i][idx] -= eps
            assert abs((loss(X_sl, a) - loss(X_sl, b)) / (2 * eps) - dW[i][idx]) < 1e-7
    np.testing.assert_allclose(np.concatenate(dX, axis=1), dY @ W.T, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(np.concatenate(dW, axis=0), Xf.T @ dY, rtol=1e-13, atol=1e-14)


def test_relu_counterexample_row_then_column_is_wrong():
    g = golden("relu_counterexample.json")
    relu = lambda x: np.maximum(x, 0.0)  # noqa: E731
    parts = [np.array(p, float) for p in g["partials"]]
    assert relu(parts[0] + parts[1]) == g["act_of_sum"]
    assert tp_mlp.row_then_column_wrong(parts, relu) == g["sum_of_act"]


def test_ffn_columns_per_shard_table():
    g = golden("tp_degree_table.json")
    W = np.zeros((2, g["f"]))
    for row in g["rows"]:
        sh = tp_mlp.split_columns(W, row["t"])
        assert all(s.shape[1] == row["ffn_cols"] for s in sh)
        assert g["heads"] // row["t"] == row["heads"]


# ---------------------------------------------------------------- activations vs torch + closed forms

def test_gelu_tanh_matches_torch_and_closed_forms():
    x = np.linspace(-8, 8, 2001)
    ref = torch.nn.functional.gelu(torch.tensor(x, dtype=torch.float64), approximate="tanh").numpy()
    np.testing.assert_allclose(numerics.gelu_tanh(x), ref, rtol=1e-14, atol=1e-15)
    assert numerics.gelu_tanh(0.0) == 0.0
    # GeLU(x) - GeLU(-x) = x for the tanh form (tanh is odd).
    np.testing.assert_allclose(numerics.gelu_tanh(x) - numerics.gelu_tanh(-x), x, atol=1e-13)
    # Close to the exact erf form everywhere (the approximation error is below 1e-3).
    exact = torch.nn.functional.gelu(torch.tensor(x, dtype=torch.float64)).numpy()
    assert np.abs(numerics.gelu_tanh(x) - exact).max() < 1e-3


def test_activation_derivatives_vs_autograd_and_finite_differences():
    x = torch.linspace(-6, 6, 1201, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.gelu(x, approximate="tanh").sum().backward()
    np.testing.assert_allclose(numerics.gelu_tanh_grad(x.detach().numpy()), x.grad.numpy(),
                               rtol=1e-12, atol=1e-14)
    x.grad = None
    torch.nn.functional.silu(x).sum().backward()
    np.testing.assert_allclose(numerics.silu_grad(x.detach().numpy()), x.grad.numpy(),
                               rtol=1e-12, atol=1e-14)
    xs = np.linspace(-5, 5, 101)
    h = 1e-6
    for f, df in ((numerics.gelu_tanh, numerics.gelu_tanh_grad), (numerics.silu, numerics.silu_grad)):
        fd = (f(xs + h) - f(xs - h)) / (2 * h)
        np.testing.assert_allclose(df(xs), fd, rtol=1e-7, atol=1e-8)
    assert numerics.silu(0.0) == 0.0
    assert numerics.silu_grad(0.0) == 0.5
    np.testing.assert_allclose(numerics.silu(xs),
                               torch.nn.functional.silu(torch.tensor(xs)).numpy(), rtol=1e-14)


def test_round_to_bf16_matches_torch_and_ties_to_even():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10 ** rng.uniform(-30, 30, 100000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, np.inf, -np.inf, 3.3895314e38, 1e-40], np.float32)])
    v = v[np.isfinite(v) | np.isinf(v)]
    ref = torch.tensor(v).to(torch.bfloat16).to(torch.float32).numpy()
    got = numerics.round_to_bf16(v)
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))
    one = np.float32(1.0)
    assert numerics.round_to_bf16(np.float32(1 + 2 ** -8)) == one               # tie -> even (down)
    assert numerics.round_to_bf16(np.float32(1 + 3 * 2 ** -8)) == np.float32(1 + 2 ** -6)  # tie -> even (up)
    assert numerics.round_to_bf16(np.float32(1 + 2 ** -8 + 2 ** -20)) == np.float32(1 + 2 ** -7)
    assert np.isnan(numerics.round_to_bf16(np.float32(np.nan)))


# ---------------------------------------------------------------- brute force on tiny inputs

def _gemm_loops(A, B):
    n, k = len(A), len(A[0])
    m = len(B[0])
    return [[sum(A[i][p] * B[p][j] for p in range(k)) for j in range(m)] for i in range(n)]


def test_mlp_forward_against_scalar_loops():
    rng = np.random.default_rng(3)
    T, h, f, t = 3, 4, 8, 2
    X = rng.integers(-3, 4, (T, h)).astype(float)
    A = rng.integers(-2, 3, (h, f)).astype(float)
    B = rng.integers(-2, 3, (f, h)).astype(float)
    fwd = tp_mlp.tp_mlp_forward(X, {"A": A, "B": B}, t, "gelu_tanh")
    U = _gemm_loops(X.tolist(), A.tolist())
    Hl = [[float(numerics.gelu_tanh(u)) for u in row] for row in U]
    Z = _gemm_loops(Hl, B.tolist())
    np.testing.assert_allclose(fwd["Z"], np.array(Z), rtol=1e-13, atol=1e-12)
    # shard i's U is columns [i f/t, (i+1) f/t) of the loop result
    for i in range(t):
        np.testing.assert_array_equal(fwd["U"][i], np.array(U)[:, i * f // t:(i + 1) * f // t])


# ---------------------------------------------------------------- sharded == unsharded (the pages' verification recipe)

@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
@pytest.mark.parametrize("t", [1, 2, 4])
@pytest.mark.parametrize("bias", [False, True])
def test_sharded_equals_unsharded(act, t, bias):
    if act == "swiglu" and bias:
        pytest.skip("SwiGLU block carries no bias")
    rng = np.random.default_rng(10 + t)
    T, h, f = 6, 8, 16
    X = rng.standard_normal((T, h))
    dY = rng.standard_normal((T, h))
    if act == "gelu_tanh":
        W = {"A": rng.standard_normal((h, f)) * 0.5, "B": rng.standard_normal((f, h)) * 0.5}
    else:
        W = {"Wg": rng.standard_normal((h, f)) * 0.5, "Wu": rng.standard_normal((h, f)) * 0.5,
             "Wd": rng.standard_normal((f, h)) * 0.5}
    b1 = rng.standard_normal(f) if bias else None
    b2 = rng.standard_normal(h) if bias else None
    fwd = tp_mlp.tp_mlp_forward(X, W, t, act, b1, b2)
    np.testing.assert_allclose(fwd["Z"], tp_mlp.mlp_forward_unsharded(X, W, act, b1, b2),
                               rtol=1e-12, atol=1e-12)
    bwd = tp_mlp.tp_mlp_backward(X, W, t, act, dY, fwd)
    ref = tp_mlp.mlp_backward_unsharded(X, W, act, dY, b1)
    np.testing.assert_allclose(bwd["dX"], ref["dX"], rtol=1e-12, atol=1e-12)
    names = ("dA", "dB") if act == "gelu_tanh" else ("dWg", "dWu", "dWd")
    for n in names:
        full = np.concatenate(bwd[n], axis=0 if n in ("dB", "dWd") else 1)
        np.testing.assert_allclose(full, ref[n], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bwd["db2"], ref["db2"], rtol=1e-12)
    if bias:
        np.testing.assert_allclose(np.concatenate(bwd["db1"]), ref["db1"], rtol=1e-12, atol=1e-12)
        # row bias once: adding it on every shard would add it t times
        if t > 1:
            wrong = sum(P + b2 for P in fwd["P"])
            assert not np.allclose(wrong, fwd["Z"])


# ---------------------------------------------------------------- gradients by finite differences

@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
def test_backward_matches_finite_differences(act):
    rng = np.random.default_rng(5)
    T, h, f, t = 3, 4, 8, 2
    X = rng.standard_normal((T, h))
    dY = rng.standard_normal((T, h))
    if act == "gelu_tanh":
        W = {"A": rng.standard_normal((h, f)) * 0.7, "B": rng.standard_normal((f, h)) * 0.7}
    else:
        W = {"Wg": rng.standard_normal((h, f)) * 0.7, "Wu": rng.standard_normal((h, f)) * 0.7,
             "Wd": rng.standard_normal((f, h)) * 0.7}
    b1 = rng.standard_normal(f) if act == "gelu_tanh" else None

    def loss(Xv, Wv, b1v):
        return float((tp_mlp.tp_mlp_forward(Xv, Wv, t, act, b1v)["Z"] * dY).sum())

    fwd = tp_mlp.tp_mlp_forward(X, W, t, act, b1)
    bwd = tp_mlp.tp_mlp_backward(X, W, t, act, dY, fwd)
    eps = 1e-6

    def fd(arr, setter):
        g = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a = arr.copy(); a[idx] += eps
            b = arr.copy(); b[idx] -= eps
            g[idx] = (setter(a) - setter(b)) / (2 * eps)
        return g

    np.testing.assert_allclose(bwd["dX"], fd(X, lambda a: loss(a, W, b1)), rtol=1e-6, atol=1e-7)
    for name, axis in (("A", 1), ("B", 0)) if act == "gelu_tanh" else (("Wg", 1), ("Wu", 1), ("Wd", 0)):
        num = fd(W[name], lambda a: loss(X, {**W, name: a}, b1))
        got = np.concatenate(bwd["d" + name], axis=axis)
        np.testing.assert_allclose(got, num, rtol=1e-6, atol=1e-7)
    if b1 is not None:
        np.testing.assert_allclose(np.concatenate(bwd["db1"]), fd(b1, lambda a: loss(X, W, a)),
                                   rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
@pytest.mark.parametrize("t", [1, 2, 4])
def test_sequence_parallel_block_equals_tensor_parallel_block(act, t):
    """SP only changes how the all-reduce is split (reduce-scatter + all-gather), so its slabs
    are the slabs of the TP block's results, and the slab traffic per card is the same."""
    from oracle import accounting
    rng = np.random.default_rng(40 + t)
    T, h, f = 4 * t, 6, 8
    X = rng.standard_normal((T, h))
    dZ = rng.standard_normal((T, h))
    if act == "gelu_tanh":
        W = {"A": rng.standard_normal((h, f)), "B": rng.standard_normal((f, h))}
    else:
        W = {"Wg": rng.standard_normal((h, f)), "Wu": rng.standard_normal((h, f)), "Wd": rng.standard_normal((f, h))}
    w = T // t
    Xs = [X[r * w:(r + 1) * w] for r in range(t)]
    dZs = [dZ[r * w:(r + 1) * w] for r in range(t)]
    sp = tp_mlp.sp_mlp_forward(Xs, W, t, act)
    ref = tp_mlp.mlp_forward_unsharded(X, W, act)
    for r in range(t):
        np.testing.assert_allclose(sp["Z_slabs"][r], ref[r * w:(r + 1) * w], rtol=1e-12, atol=1e-12)
    spb = tp_mlp.sp_mlp_backward(Xs, W, t, act, dZs, sp)
    refb = tp_mlp.mlp_backward_unsharded(X, W, act, dZ)
    for r in range(t):
        np.testing.assert_allclose(spb["dX_slabs"][r], refb["dX"][r * w:(r + 1) * w], rtol=1e-12, atol=1e-12)
    name = "dA" if act == "gelu_tanh" else "dWg"
    np.testing.assert_allclose(np.concatenate(spb[name], axis=1), refb[name], rtol=1e-12, atol=1e-12)
    # all-reduce = reduce-scatter + all-gather: 56 + 56 = 112 MiB per card at t = 8
    g = golden("tp_comm_table.json")
    S = accounting.partial_sum_bytes(1, 4096, 8192)
    assert accounting.ring_bytes_per_rank(8, S) / 2 / 2 ** 20 == g["sp_split_MiB_t8"][0]


def test_sampled_evaluation_equals_full():
    rng = np.random.default_rng(9)
    T, h, f = 16, 8, 24
    X = rng.standard_normal((T, h))
    dY = rng.standard_normal((T, h))
    Wg, Wu, Wd = (rng.standard_normal(s) * 0.5 for s in ((h, f), (h, f), (f, h)))
    rows = np.array([0, 5, 15])
    fcols = np.array([1, 7, 23])
    s = tp_mlp.swiglu_mlp_sampled(X, Wg, Wu, Wd, dY, rows, fcols)
    full = tp_mlp.mlp_backward_unsharded(X, {"Wg": Wg, "Wu": Wu, "Wd": Wd}, "swiglu", dY)
    Z = tp_mlp.mlp_forward_unsharded(X, {"Wg": Wg, "Wu": Wu, "Wd": Wd}, "swiglu")
    np.testing.assert_allclose(s["Z"], Z[rows], rtol=1e-12)
    np.testing.assert_allclose(s["dX"], full["dX"][rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dWg"], full["dWg"][:, fcols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dWu"], full["dWu"][:, fcols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s["dWd"], full["dWd"][fcols], rtol=1e-12, atol=1e-12)
    A, B = rng.standard_normal((h, f)), rng.standard_normal((f, h))
    g = tp_mlp.gelu_mlp_sampled(X, A, B, dY, rows, fcols)
    fullg = tp_mlp.mlp_backward_unsharded(X, {"A": A, "B": B}, "gelu_tanh", dY)
    np.testing.assert_allclose(g["Z"], tp_mlp.mlp_forward_unsharded(X, {"A": A, "B": B}, "gelu_tanh")[rows], rtol=1e-12)
    np.testing.assert_allclose(g["dX"], fullg["dX"][rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dA"], fullg["dA"][:, fcols], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dB"], fullg["dB"][fcols], rtol=1e-12, atol=1e-12)

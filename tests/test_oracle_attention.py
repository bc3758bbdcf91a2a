"""Pins of the oracle's tensor-parallel attention block (CPU only)."""
import numpy as np
import pytest
import torch

from conftest import golden
from oracle import attention


def test_core_matches_torch_sdpa_and_its_gradients():
    rng = np.random.default_rng(0)
    T, n_q, n_kv, d = 9, 4, 2, 8
    Q = rng.standard_normal((T, n_q * d))
    K = rng.standard_normal((T, n_kv * d))
    V = rng.standard_normal((T, n_kv * d))
    dO = rng.standard_normal((T, n_q * d))
    core = attention.attention_core(Q, K, V, n_q, n_kv, d)
    Qt = torch.tensor(Q, requires_grad=True)
    Kt = torch.tensor(K, requires_grad=True)
    Vt = torch.tensor(V, requires_grad=True)
    q = Qt.reshape(T, n_q, d).transpose(0, 1)
    k = Kt.reshape(T, n_kv, d).transpose(0, 1).repeat_interleave(n_q // n_kv, 0)
    v = Vt.reshape(T, n_kv, d).transpose(0, 1).repeat_interleave(n_q // n_kv, 0)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    O = o.transpose(0, 1).reshape(T, n_q * d)
    np.testing.assert_allclose(core["O"], O.detach().numpy(), rtol=1e-12, atol=1e-12)
    (O * torch.tensor(dO)).sum().backward()
    g = attention.attention_core_backward(Q, K, V, core["P"], dO, n_q, n_kv, d)
    np.testing.assert_allclose(g["dQ"], Qt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dK"], Kt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dV"], Vt.grad.numpy(), rtol=1e-10, atol=1e-12)
    # causal: the first token attends only to itself
    np.testing.assert_allclose(core["O"][0, :d], V[0, :d], rtol=1e-14)
    for p in core["P"]:
        assert np.all(np.triu(p, 1) == 0) and np.allclose(p.sum(1), 1.0)


@pytest.mark.parametrize("t", [1, 2, 4])
def test_sharded_block_equals_unsharded(t):
    rng = np.random.default_rng(t)
    T, h, n_q, n_kv, d = 10, 12, 8, 4, 4
    W = {"Wq": rng.standard_normal((h, n_q * d)) * 0.5, "Wk": rng.standard_normal((h, n_kv * d)) * 0.5,
         "Wv": rng.standard_normal((h, n_kv * d)) * 0.5, "Wo": rng.standard_normal((n_q * d, h)) * 0.5}
    X = rng.standard_normal((T, h))
    dY = rng.standard_normal((T, h))
    fwd = attention.tp_attention_forward(X, W, t, n_q, n_kv, d)
    np.testing.assert_allclose(fwd["Y"], attention.attention_unsharded(X, W, n_q, n_kv, d), rtol=1e-12, atol=1e-12)
    bwd = attention.tp_attention_backward(X, W, t, n_q, n_kv, d, dY, fwd)
    Xt = torch.tensor(X, requires_grad=True)
    Wt = {k: torch.tensor(v, requires_grad=True) for k, v in W.items()}
    q = (Xt @ Wt["Wq"]).reshape(T, n_q, d).transpose(0, 1)
    k = (Xt @ Wt["Wk"]).reshape(T, n_kv, d).transpose(0, 1).repeat_interleave(n_q // n_kv, 0)
    v = (Xt @ Wt["Wv"]).reshape(T, n_kv, d).transpose(0, 1).repeat_interleave(n_q // n_kv, 0)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(0, 1).reshape(T, -1)
    ((o @ Wt["Wo"]) * torch.tensor(dY)).sum().backward()
    np.testing.assert_allclose(bwd["dX"], Xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    for name, axis in (("Wq", 1), ("Wk", 1), ("Wv", 1), ("Wo", 0)):
        np.testing.assert_allclose(np.concatenate(bwd["d" + name], axis=axis), Wt[name].grad.numpy(),
                                   rtol=1e-10, atol=1e-12)


def test_heads_per_shard_printed_counts():
    g = golden("attention_heads_qwen3.json")
    d = 128
    for row in g["per_shard"]:
        cq = attention.head_columns(g["n_q"], d, row["t"], 0)
        ck = attention.head_columns(g["n_kv"], d, row["t"], 0)
        assert (cq.stop - cq.start) // d == row["q_heads"]
        assert (ck.stop - ck.start) // d == row["kv_heads"]
    with pytest.raises(ValueError):
        attention.tp_attention_forward(np.zeros((2, 4)), {}, 3, 32, 8, 1)   # 3 does not divide 32


def _torch_block_grads(X, W, dY, n_q, n_kv):
    """Autograd of the unsharded block through torch's causal scaled_dot_product_attention."""
    T = X.shape[0]
    d = W["Wq"].shape[1] // n_q
    Xt = torch.tensor(X, requires_grad=True)
    Wt = {k: torch.tensor(v) for k, v in W.items()}
    q = (Xt @ Wt["Wq"]).reshape(T, n_q, d).transpose(0, 1)
    k = (Xt @ Wt["Wk"]).reshape(T, n_kv, d).transpose(0, 1).repeat_interleave(n_q // n_kv, 0)
    v = (Xt @ Wt["Wv"]).reshape(T, n_kv, d).transpose(0, 1).repeat_interleave(n_q // n_kv, 0)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(0, 1).reshape(T, -1)
    Y = o @ Wt["Wo"]
    (Y * torch.tensor(dY)).sum().backward()
    return Y.detach().numpy(), Xt.grad.numpy()


def test_row_functions_match_torch_autograd():
    rng = np.random.default_rng(5)
    T, h, n_q, n_kv, d = 11, 10, 6, 2, 4
    W = {"Wq": rng.standard_normal((h, n_q * d)) * 0.5, "Wk": rng.standard_normal((h, n_kv * d)) * 0.5,
         "Wv": rng.standard_normal((h, n_kv * d)) * 0.5, "Wo": rng.standard_normal((n_q * d, h)) * 0.5}
    X = rng.standard_normal((T, h))
    dY = rng.standard_normal((T, h))
    Y, dX = _torch_block_grads(X, W, dY, n_q, n_kv)
    rows = np.array([0, 3, 7, 10])
    np.testing.assert_allclose(attention.forward_rows(X, W, n_q, n_kv, d, rows), Y[rows], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(attention.backward_rows_dx(X, W, dY, n_q, n_kv, d, rows), dX[rows],
                               rtol=1e-10, atol=1e-12)
    # the first query sees only itself: its output is its own value row through W_O
    V0 = X[0] @ W["Wv"]
    o0 = np.concatenate([V0[(c // (n_q // n_kv)) * d:(c // (n_q // n_kv) + 1) * d] for c in range(n_q)])
    np.testing.assert_allclose(attention.forward_rows(X, W, n_q, n_kv, d, [0])[0], o0 @ W["Wo"], rtol=1e-13)


def test_gradient_of_rows_beyond_the_last_nonzero_dY_row_is_zero():
    """With dY zero below row m the block's gradients equal those of the first m tokens alone
    (causality): dX rows >= m vanish and the weight gradients match the truncated block."""
    rng = np.random.default_rng(6)
    T, m, h, n_q, n_kv, d, t = 12, 5, 8, 4, 2, 4, 2
    W = {"Wq": rng.standard_normal((h, n_q * d)), "Wk": rng.standard_normal((h, n_kv * d)),
         "Wv": rng.standard_normal((h, n_kv * d)), "Wo": rng.standard_normal((n_q * d, h))}
    X = rng.standard_normal((T, h))
    dY = rng.standard_normal((T, h))
    dY[m:] = 0
    full = attention.tp_attention_backward(X, W, t, n_q, n_kv, d, dY, attention.tp_attention_forward(X, W, t, n_q, n_kv, d))
    cut = attention.tp_attention_backward(X[:m], W, t, n_q, n_kv, d, dY[:m],
                                          attention.tp_attention_forward(X[:m], W, t, n_q, n_kv, d))
    assert np.all(full["dX"][m:] == 0)
    np.testing.assert_allclose(full["dX"][:m], cut["dX"], rtol=1e-10, atol=1e-12)
    for k in ("dWq", "dWk", "dWv", "dWo"):
        for i in range(t):
            np.testing.assert_allclose(full[k][i], cut[k][i], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- the bf16 rounding mirror

def _mirror_case(seed=8):
    rng = np.random.default_rng(seed)
    T, h, n_q, n_kv, d, t = 24, 16, 4, 2, 8, 2
    W = {"Wq": rng.standard_normal((h, n_q * d)) / 4, "Wk": rng.standard_normal((h, n_kv * d)) / 4,
         "Wv": rng.standard_normal((h, n_kv * d)) / 4, "Wo": rng.standard_normal((n_q * d, h)) / 6}
    X = rng.standard_normal((T, h))
    dY = rng.standard_normal((T, h))
    return X, W, dY, t, n_q, n_kv, d


def _block(X, W, dY, t, n_q, n_kv, d, mirror):
    f = attention.tp_attention_forward(X, W, t, n_q, n_kv, d, mirror=mirror)
    b = attention.tp_attention_backward(X, W, t, n_q, n_kv, d, dY, f, mirror=mirror)
    return f, b


def _outputs(f, b, t):
    out = {"Y": f["Y"], "dX": b["dX"]}
    for i in range(t):
        for k in ("Q", "K", "V", "O"):
            out[f"{k}{i}"] = f[k][i]
        for c, p in enumerate(f["P"][i]):
            out[f"P{i}_{c}"] = p
        for k in ("dWq", "dWk", "dWv", "dWo"):
            out[f"{k}{i}"] = b[k][i]
    return out


def test_mirror_with_rounding_switched_off_is_the_float64_block(monkeypatch):
    """The mirror adds nothing but roundings: with the rounding replaced by the identity it
    returns exactly the float64 block, output for output."""
    X, W, dY, t, n_q, n_kv, d = _mirror_case()
    ref = _outputs(*_block(X, W, dY, t, n_q, n_kv, d, False), t)
    monkeypatch.setattr(attention, "round_to_bf16", lambda a: np.asarray(a, dtype=np.float64))
    got = _outputs(*_block(X, W, dY, t, n_q, n_kv, d, True), t)
    for k in ref:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)


def test_mirror_outputs_are_bf16_values_near_the_float64_block():
    """Every mirrored output is a bf16 value (the rounding happened), and the chain of roundings
    moves each output by a few bf16 half-ulps: relative Frobenius distance from the float64
    block between 1e-4 and 2e-2 (about 2^-9 per rounding; the cancellation in dS = P (dP - D)
    amplifies the errors of dP and D, most in the query-side gradients of short sequences)."""
    from oracle import numerics
    X, W, dY, t, n_q, n_kv, d = _mirror_case()
    ref = _outputs(*_block(X, W, dY, t, n_q, n_kv, d, False), t)
    got = _outputs(*_block(X, W, dY, t, n_q, n_kv, d, True), t)
    for k, v in got.items():
        np.testing.assert_array_equal(numerics.round_to_bf16(v).astype(np.float64), v, err_msg=k)
        rf = np.linalg.norm(v - ref[k]) / np.linalg.norm(ref[k])
        assert 1e-4 < rf < 2e-2, (k, rf)


def test_mirror_forward_rows_equal_the_mirrored_block():
    X, W, dY, t, n_q, n_kv, d = _mirror_case(9)
    f = attention.tp_attention_forward(X, W, t, n_q, n_kv, d, mirror=True)
    rows = np.array([0, 5, 17, 23])
    got = attention.forward_rows(X, W, n_q, n_kv, d, rows, t=t, mirror=True)
    # the same roundings on row-wise products: equal up to a rare one-ulp flip where the
    # float64 product lands within its last bits of a bf16 rounding boundary
    assert np.linalg.norm(got - f["Y"][rows]) <= 1e-3 * np.linalg.norm(f["Y"][rows])
    assert np.mean(got == f["Y"][rows]) > 0.95

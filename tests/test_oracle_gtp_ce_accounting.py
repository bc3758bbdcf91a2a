"""Pins of the oracle's GTP, vocab-parallel CE and accounting functions (CPU only)."""
import math

import numpy as np
import pytest
import torch

from conftest import golden
from oracle import accounting, gtp, tp_mlp, vocab_ce

MiB = 1 << 20


# ---------------------------------------------------------------- GTP

def test_gtp_memory_paragraph():
    g = golden("gtp_memory.json")
    acc = gtp.resident_weight_bytes(g["h"], g["tp"], g["g"])
    assert acc["full"] == g["full_MiB"] * MiB
    assert acc["tp_slice"] == g["tp_slice_MiB"] * MiB
    assert acc["resident"] == g["resident_MiB"] * MiB
    assert acc["reduction"] == g["reduction"]


def test_gather_rebuilds_slice_bit_exact():
    rng = np.random.default_rng(0)
    W = rng.standard_normal((64, 12)).astype(np.float32)
    sh = gtp.shard_rows(W, 8)
    assert all(s.shape == (8, 12) for s in sh)
    np.testing.assert_array_equal(gtp.gather(sh).view(np.uint32), W.view(np.uint32))


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_wgrad_reduce_scatter_equals_row_blocks_of_full_wgrad(g):
    rng = np.random.default_rng(g)
    M, K, N = 16, 24, 5
    X = rng.standard_normal((M, K))
    dY = rng.standard_normal((M, N))
    st = gtp.wgrad_reduce_scatter(X, dY, g)
    full = X.T @ dY
    for j in range(g):
        np.testing.assert_allclose(st[j], full[j * K // g:(j + 1) * K // g], rtol=1e-12, atol=1e-12)
    # brute force one element with scalar loops
    j, r, c = g - 1, K // g - 1, N - 1
    ref = sum(X[m, j * K // g + r] * dY[m, c] for m in range(M))
    assert math.isclose(st[j][r, c], ref, rel_tol=1e-12, abs_tol=1e-12)


def test_chain_schedules_hide_l_minus_1_gathers():
    L = 8
    warm = gtp.forward_chain_schedule(L, warm=True)
    hidden = [e for e in warm if e[0] == "gather_async"]
    exposed = [e for e in warm if e[0] == "gather_sync"]
    assert len(hidden) == L - 1 and len(exposed) == 1 and exposed[0][1] == 0
    assert all(e[2] == ("gemm", e[1] - 1) for e in hidden)          # AG(W_{l+1}) || GEMM(W_l)
    cold = gtp.forward_chain_schedule(L, warm=False)
    assert sum(e[0] == "gather_sync" for e in cold) == L             # cold start: all synchronous
    bwd = gtp.backward_chain_schedule(L)
    assert [e[1] for e in bwd if e[0] == "dgrad"] == list(range(L - 1, -1, -1))
    assert all(e[2] == ("dgrad", e[1] + 1) for e in bwd if e[0] == "gather_async")
    rs = [e for e in bwd if e[0].startswith("wgrad_rs")]
    assert [e[0] for e in rs].count("wgrad_rs_sync") == 1 and rs[-1] == ("wgrad_rs_sync", 0, None)


def test_deferred_finalize_visibility_and_result():
    rng = np.random.default_rng(4)
    L, g = 4, 2
    mg0 = [[rng.standard_normal((3, 2)) for _ in range(g)] for _ in range(L)]
    st = [[rng.standard_normal((3, 2)) for _ in range(g)] for _ in range(L)]
    d = gtp.deferred_finalize(mg0, st)
    imm = gtp.immediate_finalize(mg0, st)
    for l in range(L):
        for j in range(g):
            np.testing.assert_allclose(d["main_grad"][l][j], mg0[l][j] + st[l][j], rtol=1e-15)
            np.testing.assert_allclose(imm[l][j], d["main_grad"][l][j], rtol=1e-15)
    # after backward step l, layers > l are finalized except the one just computed; l = 0 all
    assert d["updated_after_step"][L - 1] == []
    assert d["updated_after_step"][L - 2] == [L - 1]
    assert d["updated_after_step"][1] == list(range(2, L))
    assert d["updated_after_step"][0] == list(range(L))



# GTP GEMMs on the gathered slice (GTP page, concepts "GTP_remat" and "Prefetch chain": the
# gathered TP slice is an ordinary GEMM operand, forward X W and backward dY W^T).

def _triple_loop(A, B):
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    C = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += float(A[m, k]) * float(B[k, n])
            C[m, n] = acc
    return C


def test_gtp_forward_gemm_printed_example_and_scalar_loops():
    g = golden("tp_split_2x2.json")
    assert gtp.forward_gemm(np.array(g["X"], float), np.array(g["A"], float)).tolist() == g["XA"]
    rng = np.random.default_rng(21)
    M, K, N = 3, 8, 5                                   # M, K, N all different
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((K, N))
    Y = gtp.forward_gemm(X, W)
    assert Y.shape == (M, N)
    np.testing.assert_allclose(Y, _triple_loop(X, W), rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_gtp_forward_on_gathered_shards_is_the_row_split_sum(g):
    """Shard j holds rows j of the slice, i.e. the row-split weight of the TP/SP page's block
    identity [X_1, X_2][A_1; A_2] = X_1 A_1 + X_2 A_2: the GEMM on the gathered slice must equal
    the sum of the per-shard partials on the matching column blocks of X."""
    rng = np.random.default_rng(30 + g)
    M, K, N = 5, 16, 3
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((K, N))
    sh = gtp.shard_rows(W, g)
    kb = K // g
    parts = tp_mlp.row_parallel_partials([X[:, j * kb:(j + 1) * kb] for j in range(g)], sh)
    np.testing.assert_allclose(gtp.forward_gemm(X, gtp.gather(sh)), sum(parts), rtol=1e-12, atol=1e-13)
    # the slice as one column-parallel shard gives the same output
    np.testing.assert_allclose(gtp.forward_gemm(X, gtp.gather(sh)),
                               tp_mlp.column_parallel_forward(X, [W])[0], rtol=1e-13, atol=1e-14)


def test_gtp_dgrad_gemm_scalar_loops_and_finite_differences():
    """dgrad is the gradient of sum(Y * dY) with respect to X, for Y = X W: checked by central
    differences of the forward GEMM (a square, non-symmetric W would hide W in place of W^T
    from a shape check, so both a square and a rectangular case run)."""
    rng = np.random.default_rng(22)
    for (M, K, N) in [(4, 5, 5), (3, 6, 4)]:
        X = rng.standard_normal((M, K))
        W = rng.standard_normal((K, N))
        dY = rng.standard_normal((M, N))
        dX = gtp.dgrad_gemm(dY, W)
        assert dX.shape == (M, K)
        np.testing.assert_allclose(dX, _triple_loop(dY, np.ascontiguousarray(W.T)), rtol=1e-13, atol=1e-14)
        eps = 1e-6
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            a = X.copy(); a[idx] += eps
            b = X.copy(); b[idx] -= eps
            num[idx] = (np.sum(gtp.forward_gemm(a, W) * dY) - np.sum(gtp.forward_gemm(b, W) * dY)) / (2 * eps)
        np.testing.assert_allclose(dX, num, rtol=1e-7, atol=1e-8)
    # torch autograd of the same scalar
    Xt = torch.tensor(X, requires_grad=True)
    (Xt @ torch.tensor(W) * torch.tensor(dY)).sum().backward()
    np.testing.assert_allclose(gtp.dgrad_gemm(dY, W), Xt.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_gtp_dgrad_on_gathered_shards_equals_per_shard_row_blocks():
    """dX = dY W^T on the gathered slice: its column block j equals dY shard_j^T, the backward of
    shard j's rows alone (what a rank that holds only shard j could compute)."""
    rng = np.random.default_rng(23)
    M, K, N, g = 4, 16, 6, 8
    dY = rng.standard_normal((M, N))
    W = rng.standard_normal((K, N))
    sh = gtp.shard_rows(W, g)
    dX = gtp.dgrad_gemm(dY, gtp.gather(sh))
    kb = K // g
    for j in range(g):
        np.testing.assert_allclose(dX[:, j * kb:(j + 1) * kb], _triple_loop(dY, np.ascontiguousarray(sh[j].T)),
                                   rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- vocab-parallel CE

def test_vocab_shard_sizes():
    g = golden("vocab_shard.json")
    assert g["V"] // g["t"] == g["ids_per_shard"] and g["V"] % g["t"] == 0
    logits_bytes = g["tokens"] * g["V"] * 4
    assert abs(logits_bytes / 1e9 - g["logits_GB_approx"]) < 0.05
    assert abs(logits_bytes / g["t"] / 1e9 - g["logits_per_shard_GB_approx"]) < 0.01


@pytest.mark.parametrize("t", [1, 2, 8])
def test_sharded_ce_equals_textbook_and_torch(t):
    rng = np.random.default_rng(t)
    T, h, V = 12, 6, 40
    H = rng.standard_normal((T, h))
    W = rng.standard_normal((V, h)) * 0.8
    target = rng.integers(0, V, T)
    r = vocab_ce.vocab_parallel_ce(H, W, target, t)
    logits = H @ W.T
    ref = vocab_ce.cross_entropy_unsharded(logits, target)
    np.testing.assert_allclose(r["loss_tok"], ref["loss_tok"], rtol=1e-12)
    np.testing.assert_allclose(np.concatenate(r["dZ"], axis=1), ref["dZ"], rtol=1e-12, atol=1e-15)
    lt = torch.tensor(logits, requires_grad=True)
    tl = torch.nn.functional.cross_entropy(lt, torch.tensor(target), reduction="mean")
    tl.backward()
    assert math.isclose(r["loss"], tl.item(), rel_tol=1e-12)
    np.testing.assert_allclose(ref["dZ"], lt.grad.numpy(), rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(r["dH"], ref["dZ"] @ W, rtol=1e-12, atol=1e-14)



def test_ce_shard_helpers_directly():
    """The per-shard pieces on their own: the logits GEMM against scalar loops (W is [V, h], so
    Z_i = H W_i^T), and one shard's dlogits against torch's gradient columns of that shard."""
    rng = np.random.default_rng(13)
    T, h, V, t = 4, 3, 10, 2
    H = rng.standard_normal((T, h))
    W = rng.standard_normal((V, h))
    target = np.array([0, 9, 5, 4])
    Vs = V // t
    Z1 = vocab_ce.lm_head_logits(H, W[Vs:])
    np.testing.assert_allclose(Z1, _triple_loop(H, np.ascontiguousarray(W[Vs:].T)), rtol=1e-13, atol=1e-14)
    lt = torch.tensor(H @ W.T, requires_grad=True)
    torch.nn.functional.cross_entropy(lt, torch.tensor(target), reduction="mean").backward()
    lse = np.log(np.exp(H @ W.T).sum(axis=1))
    for i in range(t):
        Zi = vocab_ce.lm_head_logits(H, W[i * Vs:(i + 1) * Vs])
        d = vocab_ce.dlogits_shard(Zi, target, i * Vs, lse, T)
        np.testing.assert_allclose(d, lt.grad.numpy()[:, i * Vs:(i + 1) * Vs], rtol=1e-10, atol=1e-15)


def test_ce_special_cases_and_invariants():
    T, V, t = 5, 24, 4
    z = np.zeros((T, V))
    target = np.array([0, 5, 6, 23, 11])
    comb = vocab_ce.combine([vocab_ce.shard_stats(z[:, i * 6:(i + 1) * 6], target, i * 6) for i in range(t)])
    np.testing.assert_allclose(comb["loss_tok"], math.log(V), rtol=1e-15)
    assert math.isclose(math.log(151936), 11.931215, rel_tol=1e-7)
    rng = np.random.default_rng(2)
    H = rng.standard_normal((T, 3))
    W = rng.standard_normal((V, 3))
    r = vocab_ce.vocab_parallel_ce(H, W, target, t)
    dZ = np.concatenate(r["dZ"], axis=1)
    np.testing.assert_allclose(dZ.sum(axis=1), 0.0, atol=1e-15)
    p = np.exp(H @ W.T - r["lse"][:, None])
    np.testing.assert_allclose(dZ[np.arange(T), target], (p[np.arange(T), target] - 1) / T, rtol=1e-12)
    # exactly one shard owns each target
    owners = np.stack([(st[2] != 0) for st in r["stats"]]).sum(axis=0)
    assert np.all(owners == 1)


def test_ce_dH_by_finite_differences():
    rng = np.random.default_rng(11)
    T, h, V, t = 3, 4, 8, 2
    H = rng.standard_normal((T, h))
    W = rng.standard_normal((V, h))
    target = rng.integers(0, V, T)
    r = vocab_ce.vocab_parallel_ce(H, W, target, t)
    eps = 1e-6
    num = np.zeros_like(H)
    for idx in np.ndindex(H.shape):
        a = H.copy(); a[idx] += eps
        b = H.copy(); b[idx] -= eps
        num[idx] = (vocab_ce.vocab_parallel_ce(a, W, target, t)["loss"]
                    - vocab_ce.vocab_parallel_ce(b, W, target, t)["loss"]) / (2 * eps)
    np.testing.assert_allclose(r["dH"], num, rtol=1e-6, atol=1e-9)


def test_ce_row_subset_uses_full_token_count():
    rng = np.random.default_rng(12)
    T, h, V, t = 10, 4, 16, 4
    H = rng.standard_normal((T, h))
    W = rng.standard_normal((V, h))
    target = rng.integers(0, V, T)
    full = vocab_ce.vocab_parallel_ce(H, W, target, t)
    rows = np.array([1, 4, 9])
    sub = vocab_ce.vocab_parallel_ce(H, W, target, t, rows=rows)
    np.testing.assert_allclose(sub["loss_tok"], full["loss_tok"][rows], rtol=1e-13)
    np.testing.assert_allclose(sub["dH"], full["dH"][rows], rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- accounting closed forms

def test_tp_comm_table():
    g = golden("tp_comm_table.json")
    S = accounting.partial_sum_bytes(g["b"], g["s"], g["h"])
    assert S == g["S_MiB"] * MiB
    for row in g["rows"]:
        assert accounting.ring_bytes_per_rank(row["t"], S) == row["traffic_MiB"] * MiB
        f = accounting.flops_per_comm_byte(g["b"], g["s"], g["h"], row["t"])
        assert math.isclose(f, 3 * g["h"] / (row["t"] - 1), rel_tol=1e-12)
        assert round(f) == row["flops_per_byte"]          # the table prints rounded values
    assert accounting.allreduces_per_layer() == g["allreduces_per_layer"]
    half = accounting.ring_bytes_per_rank(8, S) / 2
    assert [half / MiB, half / MiB] == g["sp_split_MiB_t8"]
    el = accounting.elements_moved_per_layer(1, 4096, 8192, 8)
    # four all-reduces per layer, each 2(t-1)/t of S bytes = S/2 elements
    assert el == accounting.allreduces_per_layer() * accounting.ring_bytes_per_rank(8, S) / 2


def test_allreduce_time_exercise():
    g = golden("allreduce_time_exercise.json")
    T = accounting.allreduce_time(g["t"], g["S_MB"] * 1e6, g["B_GBps"] * 1e9)
    assert math.isclose(T * 1e3, g["T_ms"], rel_tol=1e-12)

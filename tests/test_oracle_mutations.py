"""Planted mistakes in the oracle (CPU only): each must be caught by one of the pins.

These show the pins are strong enough: a dropped term, a wrong sign, a transposed operand
or a wrong owner index anywhere in the oracle makes at least one pin test fail.
"""
import numpy as np
import pytest

import test_oracle_collectives as tcol
import test_oracle_gtp_ce_accounting as tgce
import test_oracle_tp as ttp
from oracle import collectives, gtp, numerics, tp_mlp, vocab_ce


def _expect_failure(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_dropped_term_in_gelu_derivative_is_caught(monkeypatch):
    def bad(x):
        x = np.asarray(x, dtype=np.float64)
        u = numerics.SQRT_2_OVER_PI * (x + numerics.GELU_C * x ** 3)
        return 0.5 * (1.0 + np.tanh(u))          # second product-rule term dropped
    monkeypatch.setattr(numerics, "gelu_tanh_grad", bad)
    monkeypatch.setattr(tp_mlp, "gelu_tanh_grad", bad)
    _expect_failure(ttp.test_activation_derivatives_vs_autograd_and_finite_differences)
    _expect_failure(ttp.test_backward_matches_finite_differences, "gelu_tanh")


def test_wrong_swiglu_derivative_sign_is_caught(monkeypatch):
    def bad(x):
        s = numerics.sigmoid(x)
        return s * (1.0 - np.asarray(x) * (1.0 - s))
    monkeypatch.setattr(tp_mlp, "silu_grad", bad)
    _expect_failure(ttp.test_backward_matches_finite_differences, "swiglu")


def test_reversed_shard_ownership_is_caught(monkeypatch):
    orig = tp_mlp.split_columns

    def bad(W, t):
        return orig(W, t)[::-1]
    monkeypatch.setattr(tp_mlp, "split_columns", bad)
    _expect_failure(ttp.test_column_parallel_t3_printed_table)


def test_transposed_wgrad_operand_is_caught(monkeypatch):
    def bad(X, W_shards, dY_shards):
        X = np.asarray(X, float)
        dW = [np.asarray(d, float).T @ X for d in dY_shards]      # dY^T X instead of X^T dY
        pieces = [np.asarray(d, float) @ np.asarray(W, float).T for d, W in zip(dY_shards, W_shards)]
        return dW, pieces, sum(pieces)
    monkeypatch.setattr(tp_mlp, "column_parallel_backward", bad)
    _expect_failure(ttp.test_column_parallel_t3_printed_table)


def test_off_by_one_slab_owner_is_caught(monkeypatch):
    orig = collectives.slab_rows

    def bad(T, t, r):
        return orig(T, t, (r + 1) % t)
    monkeypatch.setattr(collectives, "slab_rows", bad)
    _expect_failure(tcol.test_two_card_figure)


def test_ce_combine_without_rescale_is_caught(monkeypatch):
    def bad(stats):
        ms = np.stack([s[0] for s in stats]); ss = np.stack([s[1] for s in stats])
        ys = np.stack([s[2] for s in stats])
        M = ms.max(axis=0); S = ss.sum(axis=0); zy = ys.sum(axis=0)   # forgot exp(m_i - M)
        lt = np.log(S) + M - zy
        return {"M": M, "S": S, "z_target": zy, "lse": M + np.log(S), "loss_tok": lt, "loss": lt.mean()}
    monkeypatch.setattr(vocab_ce, "combine", bad)
    _expect_failure(tgce.test_sharded_ce_equals_textbook_and_torch, 8)


def test_gtp_reduce_scatter_wrong_block_is_caught(monkeypatch):
    orig = gtp.wgrad_reduce_scatter

    def bad(X, dY, g):
        st = orig(X, dY, g)
        return st[1:] + st[:1]
    monkeypatch.setattr(gtp, "wgrad_reduce_scatter", bad)
    _expect_failure(tgce.test_wgrad_reduce_scatter_equals_row_blocks_of_full_wgrad, 4)


def test_finalize_not_deferred_is_caught(monkeypatch):
    def bad(main_grad, staging):
        mg = gtp.immediate_finalize(main_grad, staging)
        L = len(staging)
        return {"main_grad": mg, "updated_after_step": {l: list(range(l, L)) for l in range(L)}}
    monkeypatch.setattr(gtp, "deferred_finalize", bad)
    _expect_failure(tgce.test_deferred_finalize_visibility_and_result)


def test_embedding_wrong_owner_offset_is_caught(monkeypatch):
    import test_oracle_embedding as temb
    from oracle import embedding
    orig = embedding.shard_lookup

    def bad(ids, E_shard, v0):
        return orig(ids, E_shard, v0 + 1)                  # off-by-one id offset
    monkeypatch.setattr(embedding, "shard_lookup", bad)
    _expect_failure(temb.test_hand_worked_example)


def test_attention_without_causal_mask_is_caught(monkeypatch):
    import test_oracle_attention as tatt
    from oracle import attention

    def bad(S):
        S = np.asarray(S, dtype=np.float64)
        E = np.exp(S - S.max(axis=1, keepdims=True))
        return E / E.sum(axis=1, keepdims=True)               # every key, no mask
    monkeypatch.setattr(attention, "causal_softmax", bad)
    _expect_failure(tatt.test_core_matches_torch_sdpa_and_its_gradients)


def test_attention_backward_missing_rowsum_term_is_caught(monkeypatch):
    import test_oracle_attention as tatt
    from oracle import attention
    def bad(Q, K, V, P, dO, n_q, n_kv, d):
        # softmax backward written as dS = P dP / sqrt(d): the - rowsum(dO O) term dropped
        Q, K, V, dO = (np.asarray(a, dtype=np.float64) for a in (Q, K, V, dO))
        grp = n_q // n_kv
        dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
        for c in range(n_q):
            g = c // grp
            cs, gs = slice(c * d, (c + 1) * d), slice(g * d, (g + 1) * d)
            p = np.asarray(P[c])
            ds = p * (dO[:, cs] @ V[:, gs].T) / np.sqrt(d)
            dQ[:, cs] = ds @ K[:, gs]
            dK[:, gs] += ds.T @ Q[:, cs]
            dV[:, gs] += p.T @ dO[:, cs]
        return {"dQ": dQ, "dK": dK, "dV": dV}
    monkeypatch.setattr(attention, "attention_core_backward", bad)
    _expect_failure(tatt.test_core_matches_torch_sdpa_and_its_gradients)


def test_bf16_rounding_by_truncation_is_caught(monkeypatch):
    def bad(x):
        f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
        return ((f.view(np.uint32) >> 16) << 16).astype(np.uint32).view(np.float32)
    monkeypatch.setattr(numerics, "round_to_bf16", bad)
    _expect_failure(ttp.test_round_to_bf16_matches_torch_and_ties_to_even)


def test_row_softmax_without_normalisation_is_caught(monkeypatch):
    import test_oracle_attention as tatt
    from oracle import attention

    def bad(s):
        return np.exp(s - s.max())                                # the division by the sum dropped
    monkeypatch.setattr(attention, "_softmax_vec", bad)
    _expect_failure(tatt.test_row_functions_match_torch_autograd)


def test_gtp_dgrad_without_transpose_is_caught(monkeypatch):
    def bad(dY, W):
        return np.asarray(dY, float) @ np.asarray(W, float)      # W instead of W^T (square case)
    monkeypatch.setattr(gtp, "dgrad_gemm", bad)
    _expect_failure(tgce.test_gtp_dgrad_gemm_scalar_loops_and_finite_differences)


def test_gtp_forward_with_transposed_slice_is_caught(monkeypatch):
    def bad(X, W):
        return np.asarray(X, float) @ np.asarray(W, float).T
    monkeypatch.setattr(gtp, "forward_gemm", bad)
    _expect_failure(tgce.test_gtp_forward_gemm_printed_example_and_scalar_loops)


def test_row_backward_with_wrong_shard_weight_is_caught(monkeypatch):
    def bad(X_slices, W_shards, dY):
        dY = np.asarray(dY, float)
        dW = [np.asarray(x, float).T @ dY for x in X_slices]
        dX = [dY @ np.asarray(w, float).T for w in W_shards[::-1]]   # shard order reversed
        return dW, dX
    monkeypatch.setattr(tp_mlp, "row_parallel_backward", bad)
    _expect_failure(ttp.test_row_parallel_backward_2x2_example_and_finite_differences)

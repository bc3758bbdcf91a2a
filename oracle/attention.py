"""Tensor-parallel attention block (heads split across shards), forward and backward, float64.

Test infrastructure only (see the package docstring).

Source: the TP/SP page "v4:Tensor Parallel 与 Sequence Parallel", section "Attention:按 head 切":
every head is computed on its own; W_Q, W_K, W_V are column-parallel by head so each card
finishes its heads' attention without communication; W_O is row-parallel, followed by one
all-reduce; the head counts must be divisible by t.  Qwen3 has 32 query heads and 8 KV heads
(GQA), so at t = 8 each card holds 4 query heads and 1 KV head.  The TP-communication page's
Fig. 1 draws the same f -> column -> local -> row -> g shape for attention.

Readings where the pages are silent: scaled dot-product attention with scale 1/sqrt(d) and a
causal mask (a decoder language model), one sequence of T tokens, no rotary embedding, no
QK-normalisation, no biases; query head j uses KV head j // (n_q / n_kv); shard i owns query
heads [i n_q/t, (i+1) n_q/t) and KV heads [i n_kv/t, (i+1) n_kv/t) (contiguous blocks of
head-major columns, head c at columns [c d, (c+1) d)).

Rounding mirror (``mirror=True``): the pages fix no precision for the intermediates.  The
plain functions keep every intermediate in float64.  With ``mirror=True`` the same arithmetic
rounds to bf16 (round to nearest even, via float32) at each point where a bf16 tensor is
materialised in the bf16 data path: the projections Q, K, V; the probabilities P; the head
outputs O; the W_O partials; dO; the score gradients dS; dQ, dK, dV (dK and dV after the sum
over the group's query heads); the weight gradients; the dX partials; and the two all-reduced
sums Y and dX.  Everything between those points stays float64.  It is a diagnostic for the
chain of roundings, not a bit-exact model of any kernel.
"""
from __future__ import annotations

import numpy as np

from .numerics import round_to_bf16


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def _rounder(mirror: bool):
    """bf16 rounding of a float64 array (identity unless ``mirror``)."""
    if not mirror:
        return lambda a: a
    return lambda a: round_to_bf16(a).astype(np.float64)


def causal_softmax(S) -> np.ndarray:
    """Row softmax of S [T, T] over the keys j <= i (the rest get probability 0)."""
    S = _f64(S)
    T = S.shape[0]
    mask = np.tril(np.ones((T, T), dtype=bool))
    Z = np.where(mask, S, -np.inf)
    m = Z.max(axis=1, keepdims=True)
    E = np.where(mask, np.exp(Z - m), 0.0)
    return E / E.sum(axis=1, keepdims=True)


def attention_core(Q, K, V, n_q: int, n_kv: int, d: int, mirror: bool = False) -> dict:
    """Causal multi-head attention with grouped KV heads.  Q [T, n_q d], K/V [T, n_kv d].
    Returns per-head probabilities ``P[c]`` [T, T] and the output O [T, n_q d]."""
    r = _rounder(mirror)
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    T = Q.shape[0]
    grp = n_q // n_kv
    O = np.zeros((T, n_q * d))
    P = []
    for c in range(n_q):
        g = c // grp
        q = Q[:, c * d:(c + 1) * d]
        k = K[:, g * d:(g + 1) * d]
        v = V[:, g * d:(g + 1) * d]
        p = r(causal_softmax(q @ k.T / np.sqrt(d)))
        P.append(p)
        O[:, c * d:(c + 1) * d] = r(p @ v)
    return {"P": P, "O": O}


def attention_core_backward(Q, K, V, P, dO, n_q: int, n_kv: int, d: int, mirror: bool = False) -> dict:
    """Backward of :func:`attention_core`: dP = dO_c V_g^T, dS = P (dP - rowsum(dO_c O_c)) / sqrt(d)
    (softmax backward, the masked entries have P = 0), dQ_c = dS K_g, and the KV gradients
    summed over the query heads of each group: dK_g += dS^T Q_c, dV_g += P^T dO_c."""
    r = _rounder(mirror)
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    T = Q.shape[0]
    grp = n_q // n_kv
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for c in range(n_q):
        g = c // grp
        cs, gs = slice(c * d, (c + 1) * d), slice(g * d, (g + 1) * d)
        p = _f64(P[c])
        do = dO[:, cs]
        o = r(p @ V[:, gs])
        dp = do @ V[:, gs].T
        Dr = (do * o).sum(axis=1, keepdims=True)
        ds = r(p * (dp - Dr) / np.sqrt(d))
        dQ[:, cs] = r(ds @ K[:, gs])
        dK[:, gs] += ds.T @ Q[:, cs]
        dV[:, gs] += p.T @ do
    return {"dQ": dQ, "dK": r(dK), "dV": r(dV)}


def head_columns(n_heads: int, d: int, t: int, i: int) -> slice:
    """Columns of shard i's heads in a head-major [*, n_heads d] matrix."""
    w = n_heads // t
    return slice(i * w * d, (i + 1) * w * d)


def tp_attention_forward(X, W: dict, t: int, n_q: int, n_kv: int, d: int, mirror: bool = False) -> dict:
    """Literal sharded block: per shard i, Q_i K_i V_i = X W{q,k,v}_i (its heads), local attention
    over its 4 query heads and 1 KV head, the partial P_i = O_i Wo_i; the g all-reduce sums them."""
    if n_q % t or n_kv % t:
        raise ValueError("t must divide both head counts")
    r = _rounder(mirror)
    X = _f64(X)
    out = {"Q": [], "K": [], "V": [], "P": [], "O": [], "part": []}
    for i in range(t):
        cq, ck = head_columns(n_q, d, t, i), head_columns(n_kv, d, t, i)
        Qi = r(X @ _f64(W["Wq"])[:, cq])
        Ki = r(X @ _f64(W["Wk"])[:, ck])
        Vi = r(X @ _f64(W["Wv"])[:, ck])
        core = attention_core(Qi, Ki, Vi, n_q // t, n_kv // t, d, mirror)
        out["Q"].append(Qi)
        out["K"].append(Ki)
        out["V"].append(Vi)
        out["P"].append(core["P"])
        out["O"].append(core["O"])
        out["part"].append(r(core["O"] @ _f64(W["Wo"])[cq, :]))
    Y = out["part"][0].copy()
    for p in out["part"][1:]:
        Y = Y + p
    out["Y"] = r(Y)
    return out


def tp_attention_backward(X, W: dict, t: int, n_q: int, n_kv: int, d: int, dY, fwd: dict,
                          mirror: bool = False) -> dict:
    """Backward: g is the identity (dY full on every shard); dWo_i = O_i^T dY, dO_i = dY Wo_i^T;
    the local attention backward; dW{q,k,v}_i = X^T d{Q,K,V}_i; the dX partials
    d{Q,K,V}_i W{q,k,v}_i^T are all-reduced (f backward)."""
    r = _rounder(mirror)
    X, dY = _f64(X), _f64(dY)
    res = {"dWq": [], "dWk": [], "dWv": [], "dWo": [], "dX_part": []}
    for i in range(t):
        cq, ck = head_columns(n_q, d, t, i), head_columns(n_kv, d, t, i)
        Woi = _f64(W["Wo"])[cq, :]
        res["dWo"].append(r(fwd["O"][i].T @ dY))
        dO = r(dY @ Woi.T)
        g = attention_core_backward(fwd["Q"][i], fwd["K"][i], fwd["V"][i], fwd["P"][i], dO, n_q // t, n_kv // t, d,
                                    mirror)
        res["dWq"].append(r(X.T @ g["dQ"]))
        res["dWk"].append(r(X.T @ g["dK"]))
        res["dWv"].append(r(X.T @ g["dV"]))
        res["dX_part"].append(r(g["dQ"] @ _f64(W["Wq"])[:, cq].T + g["dK"] @ _f64(W["Wk"])[:, ck].T
                                + g["dV"] @ _f64(W["Wv"])[:, ck].T))
    dX = res["dX_part"][0].copy()
    for p in res["dX_part"][1:]:
        dX = dX + p
    res["dX"] = r(dX)
    return res


def attention_unsharded(X, W: dict, n_q: int, n_kv: int, d: int) -> np.ndarray:
    """The single-device block ``attention(X Wq, X Wk, X Wv) Wo``."""
    X = _f64(X)
    core = attention_core(X @ _f64(W["Wq"]), X @ _f64(W["Wk"]), X @ _f64(W["Wv"]), n_q, n_kv, d)
    return core["O"] @ _f64(W["Wo"])


def _softmax_vec(s) -> np.ndarray:
    e = np.exp(s - s.max())
    return e / e.sum()


def forward_rows(X, W: dict, n_q: int, n_kv: int, d: int, rows, t: int = 1, mirror: bool = False) -> np.ndarray:
    """Rows ``rows`` of the block output, each on its own: under the causal mask output row i
    depends on the tokens 0..i only, so it needs query i, the keys and values up to i and W_O.
    For sampled checks of shapes too large for :func:`attention_unsharded`.  ``t`` only matters
    with ``mirror``: the W_O partials of the t shards are rounded before their sum."""
    rnd = _rounder(mirror)
    X = _f64(X)
    rows = np.asarray(rows, dtype=np.int64)
    m = int(rows.max()) + 1
    K = rnd(X[:m] @ _f64(W["Wk"]))
    V = rnd(X[:m] @ _f64(W["Wv"]))
    Wq, Wo = _f64(W["Wq"]), _f64(W["Wo"])
    grp = n_q // n_kv
    out = np.zeros((len(rows), Wo.shape[1]))
    for r, i in enumerate(rows):
        q = rnd(X[i] @ Wq)
        o = np.zeros(n_q * d)
        for c in range(n_q):
            g = c // grp
            cs, gs = slice(c * d, (c + 1) * d), slice(g * d, (g + 1) * d)
            p = rnd(_softmax_vec(K[:i + 1, gs] @ q[cs] / np.sqrt(d)))
            o[cs] = rnd(p @ V[:i + 1, gs])
        qc = n_q * d // t
        out[r] = rnd(sum(rnd(o[j * qc:(j + 1) * qc] @ Wo[j * qc:(j + 1) * qc]) for j in range(t)))
    return out


def backward_rows_dx(X, W: dict, dY, n_q: int, n_kv: int, d: int, rows) -> np.ndarray:
    """Rows ``rows`` of the input gradient dX = dQ Wq^T + dK Wk^T + dV Wv^T, each on its own.
    Row i of dQ needs query i's softmax row; rows i of dK and dV collect, over every query
    q >= i, the entries dS_c[q, i] Q_c[q] and P_c[q, i] dO_c[q] of the group's query heads.
    The work grows with T - min(rows): sample rows near the end of long sequences."""
    X, dY = _f64(X), _f64(dY)
    rows = np.asarray(rows, dtype=np.int64)
    T = X.shape[0]
    Wq, Wk, Wv, Wo = (_f64(W[k]) for k in ("Wq", "Wk", "Wv", "Wo"))
    K, V = X @ Wk, X @ Wv
    grp = n_q // n_kv
    dQ = {int(i): np.zeros(n_q * d) for i in rows}
    dK = {int(i): np.zeros(n_kv * d) for i in rows}
    dV = {int(i): np.zeros(n_kv * d) for i in rows}
    for q in range(int(rows.min()), T):
        Qq = X[q] @ Wq
        dOq = dY[q] @ Wo.T
        for c in range(n_q):
            g = c // grp
            cs, gs = slice(c * d, (c + 1) * d), slice(g * d, (g + 1) * d)
            Kg, Vg = K[:q + 1, gs], V[:q + 1, gs]
            p = _softmax_vec(Kg @ Qq[cs] / np.sqrt(d))
            o = p @ Vg
            ds = p * (Vg @ dOq[cs] - dOq[cs] @ o) / np.sqrt(d)
            if q in dQ:
                dQ[q][cs] = ds @ Kg
            for i in dK:
                if i <= q:
                    dK[i][gs] += ds[i] * Qq[cs]
                    dV[i][gs] += p[i] * dOq[cs]
    return np.stack([dQ[int(i)] @ Wq.T + dK[int(i)] @ Wk.T + dV[int(i)] @ Wv.T for i in rows])

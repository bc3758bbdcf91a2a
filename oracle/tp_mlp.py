"""Column/row-parallel linears and the TP MLP block, forward and backward, in float64.

Test infrastructure only (see the package docstring).

Source: the TP/SP page "v4:Tensor Parallel 与 Sequence Parallel":
  * section "TP 的数学:分块矩阵乘法" -- column split ``X[A_1,A_2] = [XA_1, XA_2]`` and
    row split ``[X_1,X_2][A_1;A_2] = X_1A_1 + X_2A_2``;
  * table "Column 和 Row 各在哪里通信" -- column: weight ``[k, n/t]``, full X in,
    output columns, backward all-reduce of dX; row: weight ``[k/t, n]``, input slice
    ``X_i``, full-shape partial sum, forward all-reduce, no backward communication;
  * table "完整流程:column parallel,t = 3" -- ``dW_i = X^T dY_i``, ``dX = sum_i dY_i c_i^T``;
  * the f/g pseudocode -- f: identity forward, all-reduce backward; g: all-reduce
    forward, identity backward;
  * section "MLP:先 column,再 row" -- ``Z = GeLU(XA_1)B_1 + GeLU(XA_2)B_2``, SwiGLU's
    gate and up both column-split with the product taken locally;
  * "自测", the bias question -- column bias split with the columns, row bias added
    once after the all-reduce.

Shard i owns the contiguous column block ``[i n/t, (i+1) n/t)`` of a column-split
weight and the same row block of a row-split weight ("GPU i 拿第 i 列" in the t = 3
table).  Weights are in math orientation ``[in, out]`` (the table's ``weight [k, n]``).
"""
from __future__ import annotations

import numpy as np

from .numerics import gelu_tanh, gelu_tanh_grad, silu, silu_grad


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def split_columns(W, t: int) -> list:
    """Shard i = columns ``[i n/t, (i+1) n/t)`` of ``W [k, n]`` (each shard ``[k, n/t]``)."""
    W = _f64(W)
    n = W.shape[1]
    if n % t:
        raise ValueError("t must divide the column count")
    w = n // t
    return [W[:, i * w:(i + 1) * w].copy() for i in range(t)]


def split_rows(W, t: int) -> list:
    """Shard i = rows ``[i k/t, (i+1) k/t)`` of ``W [k, n]`` (each shard ``[k/t, n]``)."""
    W = _f64(W)
    k = W.shape[0]
    if k % t:
        raise ValueError("t must divide the row count")
    w = k // t
    return [W[i * w:(i + 1) * w, :].copy() for i in range(t)]


def split_vector(b, t: int) -> list:
    b = _f64(b)
    w = b.shape[0] // t
    return [b[i * w:(i + 1) * w].copy() for i in range(t)]


# --------------------------------------------------------------------------
# Single linears (the worked examples of "TP 的数学" and the t = 3 table).
# --------------------------------------------------------------------------


def column_parallel_forward(X, W_shards, b_shards=None) -> list:
    """Each shard: ``Y_i = X W_i (+ b_i)``, its own output columns.  No communication."""
    X = _f64(X)
    out = []
    for i, Wi in enumerate(W_shards):
        Yi = X @ _f64(Wi)
        if b_shards is not None:
            Yi = Yi + _f64(b_shards[i])
        out.append(Yi)
    return out


def row_parallel_partials(X_slices, W_shards) -> list:
    """Each shard: the full-shape partial ``P_i = X_i W_i``; they still need a sum."""
    return [_f64(Xi) @ _f64(Wi) for Xi, Wi in zip(X_slices, W_shards)]


def column_parallel_backward(X, W_shards, dY_shards):
    """Column backward: ``dW_i = X^T dY_i`` (local), dX pieces ``dY_i W_i^T`` and their sum
    (the all-reduce in f's backward).  Returns ``(dW_list, dX_pieces, dX)``."""
    X = _f64(X)
    dW = [X.T @ _f64(dYi) for dYi in dY_shards]
    pieces = [_f64(dYi) @ _f64(Wi).T for dYi, Wi in zip(dY_shards, W_shards)]
    dX = pieces[0].copy()
    for p in pieces[1:]:
        dX = dX + p
    return dW, pieces, dX


def row_parallel_backward(X_slices, W_shards, dY):
    """Row backward: dY is already full on every shard (g's backward is identity), so
    ``dX_i = dY W_i^T`` and ``dW_i = X_i^T dY`` are both local.  Returns ``(dW, dX_slices)``."""
    dY = _f64(dY)
    dW = [_f64(Xi).T @ dY for Xi in X_slices]
    dX = [dY @ _f64(Wi).T for Wi in W_shards]
    return dW, dX


# --------------------------------------------------------------------------
# The MLP block: f -> column fc1 -> local activation -> row fc2 -> g.
# --------------------------------------------------------------------------


def tp_mlp_forward(X, weights: dict, t: int, act: str, b1=None, b2=None) -> dict:
    """Literal sharded forward.

    GeLU:   ``U_i = X A_i + b1_i``; ``H_i = GeLU(U_i)``; ``P_i = H_i B_i``.
    SwiGLU: ``G_i = X Wg_i``; ``V_i = X Wu_i``; ``H_i = SiLU(G_i) * V_i``; ``P_i = H_i Wd_i``.
    g forward: ``Z = sum_i P_i``, then the row bias ``b2`` once.
    Returns every per-shard intermediate plus ``Z``.
    """
    X = _f64(X)
    out = {"U": [], "G": [], "V": [], "H": [], "P": []}
    if act == "gelu_tanh":
        A_sh = split_columns(weights["A"], t)
        B_sh = split_rows(weights["B"], t)
        b1_sh = split_vector(b1, t) if b1 is not None else None
        for i in range(t):
            Ui = X @ A_sh[i]
            if b1_sh is not None:
                Ui = Ui + b1_sh[i]
            Hi = gelu_tanh(Ui)
            out["U"].append(Ui)
            out["H"].append(Hi)
            out["P"].append(Hi @ B_sh[i])
    elif act == "swiglu":
        Wg_sh = split_columns(weights["Wg"], t)
        Wu_sh = split_columns(weights["Wu"], t)
        Wd_sh = split_rows(weights["Wd"], t)
        for i in range(t):
            Gi = X @ Wg_sh[i]
            Vi = X @ Wu_sh[i]
            Hi = silu(Gi) * Vi
            out["G"].append(Gi)
            out["V"].append(Vi)
            out["H"].append(Hi)
            out["P"].append(Hi @ Wd_sh[i])
    else:
        raise ValueError(act)
    Z = out["P"][0].copy()
    for Pi in out["P"][1:]:
        Z = Z + Pi
    if b2 is not None:
        Z = Z + _f64(b2)
    out["Z"] = Z
    return out


def tp_mlp_backward(X, weights: dict, t: int, act: str, dY, fwd: dict) -> dict:
    """Literal sharded backward.

    g backward is the identity: every shard sees the full ``dY``.
    Row fc2 (local):   ``dB_i = H_i^T dY``; ``dH_i = dY B_i^T``.
    Activation:        GeLU ``dU_i = dH_i * GeLU'(U_i)``;
                       SwiGLU ``dG_i = dH_i * V_i * SiLU'(G_i)``, ``dV_i = dH_i * SiLU(G_i)``.
    Column fc1:        ``dA_i = X^T dU_i`` (local); ``dX_i = dU_i A_i^T`` is a partial.
    f backward:        ``dX = sum_i dX_i``.
    Bias gradients:    ``db1_i = sum over tokens of dU_i``; ``db2 = sum over tokens of dY``
                       (once: the row bias is not split).
    """
    X = _f64(X)
    dY = _f64(dY)
    res = {"dX_part": [], "db1": []}
    if act == "gelu_tanh":
        A_sh = split_columns(weights["A"], t)
        B_sh = split_rows(weights["B"], t)
        res.update(dA=[], dB=[], dU=[])
        for i in range(t):
            res["dB"].append(fwd["H"][i].T @ dY)
            dHi = dY @ B_sh[i].T
            dUi = dHi * gelu_tanh_grad(fwd["U"][i])
            res["dU"].append(dUi)
            res["db1"].append(dUi.sum(axis=0))
            res["dA"].append(X.T @ dUi)
            res["dX_part"].append(dUi @ A_sh[i].T)
    elif act == "swiglu":
        Wg_sh = split_columns(weights["Wg"], t)
        Wu_sh = split_columns(weights["Wu"], t)
        Wd_sh = split_rows(weights["Wd"], t)
        res.update(dWg=[], dWu=[], dWd=[], dG=[], dV=[])
        for i in range(t):
            Gi, Vi = fwd["G"][i], fwd["V"][i]
            res["dWd"].append(fwd["H"][i].T @ dY)
            dHi = dY @ Wd_sh[i].T
            dGi = dHi * Vi * silu_grad(Gi)
            dVi = dHi * silu(Gi)
            res["dG"].append(dGi)
            res["dV"].append(dVi)
            res["dWg"].append(X.T @ dGi)
            res["dWu"].append(X.T @ dVi)
            res["dX_part"].append(dGi @ Wg_sh[i].T + dVi @ Wu_sh[i].T)
    else:
        raise ValueError(act)
    dX = res["dX_part"][0].copy()
    for p in res["dX_part"][1:]:
        dX = dX + p
    res["dX"] = dX
    res["db2"] = dY.sum(axis=0)
    return res


def mlp_forward_unsharded(X, weights: dict, act: str, b1=None, b2=None) -> np.ndarray:
    """The single-device definition ``Z = act(X A + b1) B + b2`` (SwiGLU:
    ``(SiLU(X Wg) * (X Wu)) Wd``), the right-hand side the sharded form must equal."""
    X = _f64(X)
    if act == "gelu_tanh":
        U = X @ _f64(weights["A"])
        if b1 is not None:
            U = U + _f64(b1)
        Z = gelu_tanh(U) @ _f64(weights["B"])
    else:
        Z = (silu(X @ _f64(weights["Wg"])) * (X @ _f64(weights["Wu"]))) @ _f64(weights["Wd"])
    if b2 is not None:
        Z = Z + _f64(b2)
    return Z


def mlp_backward_unsharded(X, weights: dict, act: str, dY, b1=None) -> dict:
    """Single-device gradients of ``sum(Z * dY)`` w.r.t. X, the weights and the biases."""
    X = _f64(X)
    dY = _f64(dY)
    if act == "gelu_tanh":
        A, B = _f64(weights["A"]), _f64(weights["B"])
        U = X @ A
        if b1 is not None:
            U = U + _f64(b1)
        H = gelu_tanh(U)
        dH = dY @ B.T
        dU = dH * gelu_tanh_grad(U)
        return {"dX": dU @ A.T, "dA": X.T @ dU, "dB": H.T @ dY,
                "db1": dU.sum(axis=0), "db2": dY.sum(axis=0)}
    Wg, Wu, Wd = _f64(weights["Wg"]), _f64(weights["Wu"]), _f64(weights["Wd"])
    G = X @ Wg
    V = X @ Wu
    H = silu(G) * V
    dH = dY @ Wd.T
    dG = dH * V * silu_grad(G)
    dV = dH * silu(G)
    return {"dX": dG @ Wg.T + dV @ Wu.T, "dWg": X.T @ dG, "dWu": X.T @ dV, "dWd": H.T @ dY,
            "db2": dY.sum(axis=0)}


def sp_mlp_forward(X_slabs, weights: dict, t: int, act: str) -> dict:
    """Sequence-parallel MLP block, literal: the block's input arrives as t token slabs; an
    all-gather rebuilds the full sequence before the column layer, the row layer's partial
    sums are reduce-scattered so shard r keeps only the sum of its own token slab.

    Source: the TP/SP page, section "SP": after the row-parallel layer the all-reduce
    becomes a reduce-scatter that leaves each card its own s/t tokens, and an all-gather
    before the next column-parallel layer rebuilds the full sequence.
    Returns the tp_mlp_forward intermediates plus ``Z_slabs``."""
    X = np.concatenate([_f64(x) for x in X_slabs], axis=0)          # all-gather
    fwd = tp_mlp_forward(X, weights, t, act)
    T = X.shape[0]
    w = T // t
    fwd["Z_slabs"] = []
    for r in range(t):                                                # reduce-scatter
        acc = fwd["P"][0][r * w:(r + 1) * w].copy()
        for P in fwd["P"][1:]:
            acc = acc + P[r * w:(r + 1) * w]
        fwd["Z_slabs"].append(acc)
    return fwd


def sp_mlp_backward(X_slabs, weights: dict, t: int, act: str, dZ_slabs, fwd: dict) -> dict:
    """Backward of :func:`sp_mlp_forward`: the reduce-scatter's backward is an all-gather of
    the output-gradient slabs, the all-gather's backward a reduce-scatter of the dX partials.
    Returns the tp_mlp_backward results plus ``dX_slabs``."""
    X = np.concatenate([_f64(x) for x in X_slabs], axis=0)
    dZ = np.concatenate([_f64(d) for d in dZ_slabs], axis=0)         # all-gather of dZ
    bwd = tp_mlp_backward(X, weights, t, act, dZ, fwd)
    T = X.shape[0]
    w = T // t
    bwd["dX_slabs"] = []
    for r in range(t):                                                # reduce-scatter of dX
        acc = bwd["dX_part"][0][r * w:(r + 1) * w].copy()
        for p in bwd["dX_part"][1:]:
            acc = acc + p[r * w:(r + 1) * w]
        bwd["dX_slabs"].append(acc)
    return bwd


def row_then_column_wrong(partials, act):
    """The order the "MLP:先 column,再 row" section rules out: the activation applied to
    each rank's partial sum and the results added, instead of to the sum."""
    out = act(_f64(partials[0]))
    for p in partials[1:]:
        out = out + act(_f64(p))
    return out


# --------------------------------------------------------------------------
# Row-sampled evaluation for the large workloads: the same definitions, evaluated
# only at selected token rows or selected hidden (FFN) columns.  Exact, not approximate.
# --------------------------------------------------------------------------


def swiglu_mlp_sampled(X, Wg, Wu, Wd, dY, rows, fcols) -> dict:
    """SwiGLU MLP outputs at sampled positions, from the unsharded definitions.

    ``rows``: token rows for Z and dX (full width h).
    ``fcols``: FFN columns (global indices into f) for dWg/dWu columns and dWd rows.
    Returns ``Z[rows]``, ``dX[rows]``, ``dWg[:, fcols]``, ``dWu[:, fcols]``, ``dWd[fcols, :]``.
    """
    X = _f64(X)
    dY = _f64(dY)
    Wg = _f64(Wg)
    Wu = _f64(Wu)
    Wd = _f64(Wd)
    Xr = X[rows]
    Gr = Xr @ Wg
    Vr = Xr @ Wu
    Z = (silu(Gr) * Vr) @ Wd
    dHr = dY[rows] @ Wd.T
    dGr = dHr * Vr * silu_grad(Gr)
    dVr = dHr * silu(Gr)
    dX = dGr @ Wg.T + dVr @ Wu.T
    # Columns of the FFN dimension need every token.
    Gc = X @ Wg[:, fcols]
    Vc = X @ Wu[:, fcols]
    dHc = dY @ Wd[fcols, :].T
    dGc = dHc * Vc * silu_grad(Gc)
    dVc = dHc * silu(Gc)
    Hc = silu(Gc) * Vc
    return {"Z": Z, "dX": dX, "dWg": X.T @ dGc, "dWu": X.T @ dVc, "dWd": Hc.T @ dY}


def gelu_mlp_sampled(X, A, B, dY, rows, fcols) -> dict:
    """GeLU MLP outputs at sampled token rows and sampled FFN columns (exact)."""
    X = _f64(X)
    dY = _f64(dY)
    A = _f64(A)
    B = _f64(B)
    Ur = X[rows] @ A
    Z = gelu_tanh(Ur) @ B
    dUr = (dY[rows] @ B.T) * gelu_tanh_grad(Ur)
    dX = dUr @ A.T
    Uc = X @ A[:, fcols]
    dUc = (dY @ B[fcols, :].T) * gelu_tanh_grad(Uc)
    return {"Z": Z, "dX": dX, "dA": X.T @ dUc, "dB": gelu_tanh(Uc).T @ dY}

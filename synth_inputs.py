"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and names shapes.  It holds none of the
tensor-parallel arithmetic: no splitting into shards, no products, no sums.
Both the CUDA path and the CPU oracle are fed from here, so that each
comparison sees the very same bf16 values.

Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
in a fixed order (X, then each full weight in the order listed, then dY, then
targets), as ``randn * std`` rounded once to bf16.  The shapes follow the
pages' workloads: the toy MLP of the "MLP: column then row" section
(h=256, 4h=1024), the b=1, s=4096, h=8192 layer output of the TP
communication page's worked table, the Qwen3-8B layer (h=4096, SwiGLU width
12288, vocab 151936, 32 query and 8 KV heads of dimension 128) of the TP/SP page, and
the h=8192, TP=4, GTP_remat=8 square weight of the GTP page's memory example.
"""
from __future__ import annotations

import dataclasses

import torch

# --------------------------------------------------------------------------
# Named workloads.  Each is a plain record of shapes and a seed.
# --------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class MlpShape:
    name: str
    t: int            # logical shard count
    T: int            # tokens
    h: int            # model width
    f: int            # FFN width (unsharded)
    act: str          # "gelu_tanh" or "swiglu"
    seed: int


@dataclasses.dataclass(frozen=True)
class ReduceShape:
    name: str
    T: int
    h: int
    ts: tuple
    seed: int


@dataclasses.dataclass(frozen=True)
class GtpShape:
    name: str
    L: int            # layers in the chain
    h: int            # square weight side
    tp: int           # TP degree (the TP slice is [h, h/tp])
    g: int            # GTP_remat degree (shards per TP slice)
    T: int            # tokens
    seed: int


@dataclasses.dataclass(frozen=True)
class CeShape:
    name: str
    t: int
    T: int
    h: int
    V: int
    seed: int


TP_MLP_GELU_T2 = MlpShape("tp_mlp_gelu_t2_T128_h256_f1024", t=2, T=128, h=256, f=1024,
                          act="gelu_tanh", seed=0)
REDUCE_SWEEP = ReduceShape("partial_sum_reduce_T4096_h8192", T=4096, h=8192, ts=(2, 4, 8, 16), seed=2)
QWEN3_8B_SWIGLU_T8 = MlpShape("qwen3_8b_swiglu_mlp_t8_T8192_h4096_f12288", t=8, T=8192, h=4096,
                              f=12288, act="swiglu", seed=3)
GTP_CHAIN = GtpShape("gtp_chain_L8_h8192_tp4_g8_T4096", L=8, h=8192, tp=4, g=8, T=4096, seed=4)
VOCAB_CE_T8 = CeShape("vocab_parallel_ce_t8_T8192_h4096_V151936", t=8, T=8192, h=4096, V=151936, seed=5)


@dataclasses.dataclass(frozen=True)
class AttnShape:
    name: str
    t: int
    T: int
    h: int
    n_q: int          # query heads
    n_kv: int         # key/value heads (grouped-query attention)
    d: int            # head dimension
    seed: int


QWEN3_8B_ATTN_T8 = AttnShape("qwen3_8b_attention_t8_T8192_h4096_q32_kv8_d128", t=8, T=8192, h=4096,
                             n_q=32, n_kv=8, d=128, seed=6)


# --------------------------------------------------------------------------
# Drawing helpers.
# --------------------------------------------------------------------------


def generator(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(int(seed))


def randn_bf16(gen: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    """``randn * std`` drawn in fp32 and rounded once to bf16 (CPU tensor)."""
    x = torch.randn(tuple(shape), generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def small_int_bf16(gen: torch.Generator, shape, lo: int = -3, hi: int = 3) -> torch.Tensor:
    """Uniform small integers in [lo, hi] as bf16.  Products and sums of these stay
    exactly representable, so integer-valued cases compare bit for bit."""
    return torch.randint(lo, hi + 1, tuple(shape), generator=gen, dtype=torch.int32).to(torch.bfloat16)


def mlp_inputs(T: int, h: int, f: int, act: str, seed: int, *, bias: bool = False,
               w_std: float = 0.02, ints: bool = False) -> dict:
    """Full (unsharded) MLP block inputs.

    GeLU: ``X [T,h]``, ``A [h,f]``, ``B [f,h]``, ``dY [T,h]``.
    SwiGLU: ``X``, ``Wg [h,f]``, ``Wu [h,f]``, ``Wd [f,h]``, ``dY``.
    Optional biases ``b1 [f]`` (column layer) and ``b2 [h]`` (row layer).
    ``ints`` draws every tensor as small integers (weights in [-2, 2]).
    """
    g = generator(seed)

    def act_(shape):
        return small_int_bf16(g, shape) if ints else randn_bf16(g, shape, 1.0)

    def w_(shape):
        return small_int_bf16(g, shape, -2, 2) if ints else randn_bf16(g, shape, w_std)

    out = {"X": act_((T, h))}
    if act == "gelu_tanh":
        out["A"] = w_((h, f))
        out["B"] = w_((f, h))
    elif act == "swiglu":
        out["Wg"] = w_((h, f))
        out["Wu"] = w_((h, f))
        out["Wd"] = w_((f, h))
    else:
        raise ValueError(act)
    if bias:
        out["b1"] = w_((f,)) if ints else randn_bf16(g, (f,), 0.1)
        out["b2"] = w_((h,)) if ints else randn_bf16(g, (h,), 0.1)
    out["dY"] = act_((T, h))
    return out


def partial_sum_buffers(t: int, T: int, h: int, seed: int, *, ints: bool = False) -> list:
    """``t`` full-shape ``[T,h]`` bf16 buffers ~N(0,1), buffer 0 first."""
    g = generator(seed)
    if ints:
        return [small_int_bf16(g, (T, h), -8, 8) for _ in range(t)]
    return [randn_bf16(g, (T, h), 1.0) for _ in range(t)]


def gtp_inputs(L: int, K: int, N: int, T: int, seed: int, *, w_std: float = 0.02,
               ints: bool = False) -> dict:
    """GTP chain: ``X [T,K]``, per layer a TP slice ``W_l [K,N]`` and ``dY_l [T,N]``."""
    g = generator(seed)
    if ints:
        X = small_int_bf16(g, (T, K))
        W = [small_int_bf16(g, (K, N), -2, 2) for _ in range(L)]
        dY = [small_int_bf16(g, (T, N)) for _ in range(L)]
    else:
        X = randn_bf16(g, (T, K), 1.0)
        W = [randn_bf16(g, (K, N), w_std) for _ in range(L)]
        dY = [randn_bf16(g, (T, N), 1.0) for _ in range(L)]
    return {"X": X, "W": W, "dY": dY}


def ce_inputs(T: int, h: int, V: int, seed: int, *, w_std: float = 0.02) -> dict:
    """LM head + CE: ``H [T,h]`` ~N(0,1), ``W [V,h]`` ~N(0,w_std), targets uniform in [0,V)."""
    g = generator(seed)
    H = randn_bf16(g, (T, h), 1.0)
    W = randn_bf16(g, (V, h), w_std)
    target = torch.randint(0, V, (T,), generator=g, dtype=torch.int64)
    return {"H": H, "W": W, "target": target}


def attn_inputs(T: int, h: int, n_q: int, n_kv: int, d: int, seed: int, *, w_std: float | None = None,
                dY_rows: int | None = None) -> dict:
    """Attention block: ``X [T,h]`` ~N(0,1), ``Wq [h,n_q d]``, ``Wk``, ``Wv [h,n_kv d]``,
    ``Wo [n_q d,h]`` ~N(0,w_std) (default 1/sqrt(h), so projected entries are ~N(0,1)) and
    ``dY [T,h]`` ~N(0,1).  ``dY_rows = m`` keeps dY only on the first m rows (zeros below)."""
    g = generator(seed)
    w_std = h ** -0.5 if w_std is None else w_std
    out = {"X": randn_bf16(g, (T, h), 1.0)}
    out["Wq"] = randn_bf16(g, (h, n_q * d), w_std)
    out["Wk"] = randn_bf16(g, (h, n_kv * d), w_std)
    out["Wv"] = randn_bf16(g, (h, n_kv * d), w_std)
    out["Wo"] = randn_bf16(g, (n_q * d, h), (n_q * d) ** -0.5)
    dY = randn_bf16(g, (T, h), 1.0)
    if dY_rows is not None:
        dY[dY_rows:] = 0
    out["dY"] = dY
    return out


def sample_indices(n_total: int, n_sample: int, seed: int) -> torch.Tensor:
    """Sorted distinct indices in [0, n_total), always including the first and last."""
    g = generator(seed + 7919)
    n_sample = min(n_sample, n_total)
    perm = torch.randperm(n_total, generator=g)[:n_sample]
    return torch.unique(torch.cat([perm, torch.tensor([0, n_total - 1])]))

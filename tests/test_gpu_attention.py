"""Head-split TP attention block, forward and backward through the C ABI, vs the fp64 oracle
and its bf16 rounding mirror (GPU).  Small shapes are compared element by element; the
Qwen3-8B shape (T=8192, h=4096, 32 query / 8 KV heads of 128, t=8) on sampled rows and through
causality properties."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import synth_inputs as si
import tensor_transformer_layer_way_gb300 as ttl
from oracle import attention
from parity import (ATTN_FP64_MAX_ABS_FRAC, ATTN_FP64_REL_FRO, ATTN_MIRROR_MAX_ABS_FRAC, ATTN_MIRROR_REL_FRO,
                    dev, f64, gemm_errors)

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _split(inp, t, n_q, n_kv, d):
    qc, kc = n_q // t * d, n_kv // t * d
    Wq = [inp["Wq"][:, i * qc:(i + 1) * qc].contiguous() for i in range(t)]
    Wk = [inp["Wk"][:, i * kc:(i + 1) * kc].contiguous() for i in range(t)]
    Wv = [inp["Wv"][:, i * kc:(i + 1) * kc].contiguous() for i in range(t)]
    Wo = [inp["Wo"][i * qc:(i + 1) * qc, :].contiguous() for i in range(t)]
    return dev(Wq), dev(Wk), dev(Wv), dev(Wo)


def _run(inp, t, n_q, n_kv, d, backward=True):
    Wq, Wk, Wv, Wo = _split(inp, t, n_q, n_kv, d)
    X = dev(inp["X"])
    fwd = ttl.tp_attn_fwd(X, Wq, Wk, Wv, Wo, n_q=n_q, n_kv=n_kv, d=d)
    bwd = None
    if backward:
        bwd = ttl.tp_attn_bwd(X, dev(inp["dY"]), Wq, Wk, Wv, Wo, fwd, n_q=n_q, n_kv=n_kv, d=d)
    torch.cuda.synchronize()
    assert ttl.device_status() == 0
    return fwd, bwd


class _Errors:
    """Collects each output's errors against the float64 oracle and, where given, against the
    rounding mirror, and checks them: the mirror at the GEMM bounds, float64 at the attention
    bounds (single projections: the GEMM bounds against both).  Prints the table."""

    def __init__(self):
        self.rows = []

    def add(self, got, ref, name, mirror=None, gemm=False):
        rf, maf = gemm_errors(got, ref, name)
        mrf, mmaf = gemm_errors(got, mirror, name) if mirror is not None else (None, None)
        self.rows.append((name, rf, maf, mrf, mmaf, gemm))

    def check(self):
        for name, rf, maf, mrf, mmaf, gemm in self.rows:
            m = f"  mirror {mrf:.3e} / {mmaf:.3e}" if mrf is not None else ""
            print(f"{name:14s} fp64 rel_fro {rf:.3e}  max_abs/max {maf:.3e}{m}")
        for name, rf, maf, mrf, mmaf, gemm in self.rows:
            lim_rf = 5e-3 if gemm else ATTN_FP64_REL_FRO
            lim_ma = 2e-2 if gemm else ATTN_FP64_MAX_ABS_FRAC
            assert rf <= lim_rf, f"{name}: relative Frobenius error {rf:.3e} > {lim_rf} (fp64)"
            assert maf <= lim_ma, f"{name}: max-abs error {maf:.3e} of max|ref| > {lim_ma} (fp64)"
            if mrf is not None:
                assert mrf <= ATTN_MIRROR_REL_FRO, f"{name}: relative Frobenius error {mrf:.3e} > " \
                                                   f"{ATTN_MIRROR_REL_FRO} (mirror)"
                assert mmaf <= ATTN_MIRROR_MAX_ABS_FRAC, f"{name}: max-abs error {mmaf:.3e} of max|ref| > " \
                                                         f"{ATTN_MIRROR_MAX_ABS_FRAC} (mirror)"


def _W64(inp):
    return {k: f64(inp[k]) for k in ("Wq", "Wk", "Wv", "Wo")}


def _check_p_band(P, T):
    """Row q of every head's P is zero for q < j < min(T, round_up(q + 1, 128)) (the rest of
    its query tile's diagonal tile)."""
    j = torch.arange(T, device=P.device)
    q = j[:, None]
    band = (j[None, :] > q) & (j[None, :] < torch.clamp((q // 128 + 1) * 128, max=T))
    assert torch.all(P[:, band] == 0)


SMALL = [
    # t, T, h, n_q, n_kv, d
    (2, 256, 256, 4, 2, 128),     # GQA groups of 2, one 256-row tile
    (1, 328, 192, 4, 1, 64),      # one KV head (MQA), ragged T (per-head maps), d = 64
    (4, 512, 256, 8, 4, 128),     # four shards, two tile rows
    (2, 136, 128, 2, 2, 64),      # one query head per KV head, ragged T below two tiles
    (2, 64, 64, 4, 2, 64),        # every GEMM at most 128 rows: single-CTA tiles
    (8, 392, 128, 8, 8, 64),      # eight shards of one head each, ragged T
    (1, 200, 128, 4, 2, 128),     # two KV heads per shard: K|V projections span two paired tiles
    (2, 264, 256, 8, 4, 64),      # two KV heads per shard at d = 64, ragged T
]


@pytest.mark.parametrize("t,T,h,n_q,n_kv,d", SMALL)
def test_small_blocks_match_oracle(t, T, h, n_q, n_kv, d):
    inp = si.attn_inputs(T, h, n_q, n_kv, d, seed=T + 7 * t + n_q)
    fwd, bwd = _run(inp, t, n_q, n_kv, d)
    W = _W64(inp)
    X, dY = f64(inp["X"]), f64(inp["dY"])
    rf = attention.tp_attention_forward(X, W, t, n_q, n_kv, d)
    rb = attention.tp_attention_backward(X, W, t, n_q, n_kv, d, dY, rf)
    mf = attention.tp_attention_forward(X, W, t, n_q, n_kv, d, mirror=True)
    mb = attention.tp_attention_backward(X, W, t, n_q, n_kv, d, dY, mf, mirror=True)
    lower = np.tril(np.ones((T, T), dtype=bool))
    err = _Errors()
    for i in range(t):
        for k in ("Q", "K", "V"):
            err.add(f64(fwd[k][i]), rf[k][i], f"{k}[{i}]", mf[k][i], gemm=True)
        err.add(f64(fwd["O"][i]), rf["O"][i], f"O[{i}]", mf["O"][i])
        for c in range(n_q // t):
            Pg = f64(fwd["P"][i][c])
            err.add(Pg[lower], rf["P"][i][c][lower], f"P[{i}][{c}]", mf["P"][i][c][lower])
        _check_p_band(fwd["P"][i], T)
        assert torch.equal(fwd["Y"][i], fwd["Y"][0])
        for k in ("dWq", "dWk", "dWv", "dWo"):
            err.add(f64(bwd[k][i]), rb[k][i], f"{k}[{i}]", mb[k][i])
        assert torch.equal(bwd["dX"][i], bwd["dX"][0])
    err.add(f64(fwd["Y"][0]), rf["Y"], "Y", mf["Y"])
    err.add(f64(bwd["dX"][0]), rb["dX"], "dX", mb["dX"])
    err.check()


def test_probability_rows_sum_to_one():
    t, T, h, n_q, n_kv, d = 2, 512, 128, 4, 2, 64
    inp = si.attn_inputs(T, h, n_q, n_kv, d, seed=99)
    fwd, _ = _run(inp, t, n_q, n_kv, d, backward=False)
    lower = torch.tril(torch.ones(T, T, dtype=torch.bool, device="cuda"))
    for P in fwd["P"]:
        s = torch.where(lower, P.float(), 0.0).sum(-1)
        # bf16 rounding of each of up to T probabilities: |sum - 1| <= T * 2^-9 * max p; far less in practice
        assert torch.all((s - 1).abs() < 1e-2), (s - 1).abs().max()
        assert torch.all(P[:, 0, 0] == 1)          # the first query sees only itself


def test_empty_sequence():
    t, h, n_q, n_kv, d = 2, 64, 4, 2, 64
    inp = si.attn_inputs(8, h, n_q, n_kv, d, seed=1)
    Wq, Wk, Wv, Wo = _split(inp, t, n_q, n_kv, d)
    X = torch.empty(0, h, device="cuda", dtype=torch.bfloat16)
    fwd = ttl.tp_attn_fwd(X, Wq, Wk, Wv, Wo, n_q=n_q, n_kv=n_kv, d=d)
    out = ttl.attn_bwd_buffers(t, 0, h, n_q, n_kv, d)
    for k in ("dWq", "dWk", "dWv", "dWo"):
        for w in out[k]:
            w.fill_(1.0)
    bwd = ttl.tp_attn_bwd(X, X, Wq, Wk, Wv, Wo, fwd, n_q=n_q, n_kv=n_kv, d=d, out=out)
    torch.cuda.synchronize()
    for k in ("dWq", "dWk", "dWv", "dWo"):
        for w in bwd[k]:
            assert torch.count_nonzero(w) == 0


def test_bad_shapes_are_rejected():
    T, h, d = 64, 64, 64
    inp = si.attn_inputs(T, h, 6, 3, d, seed=2)
    # 2 shards cannot split 3 KV heads; the binding slices 2 * 64 and 1 * 64 columns per shard
    Wq, Wk, Wv, Wo = _split(inp, 2, 6, 2, d)
    with pytest.raises(ttl.TTLError) as e:
        ttl.tp_attn_fwd(dev(inp["X"]), Wq, Wk, Wv, Wo, n_q=6, n_kv=3, d=d)
    assert e.value.code == ttl.TTL_ERR_SHAPE


def test_single_cta_tiles_in_a_child_process():
    """The same small cases with the CTA-pair tiles switched off (128-row tiles, whose causal
    k-ranges and skipped tiles differ from the 256-row ones)."""
    env = dict(os.environ, TTL_GEMM_CTA_PAIR="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_attention.py"), "-k",
                        "test_small_blocks_match_oracle and (256-256 or 328-192 or 512-256)"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "3 passed" in r.stdout, r.stdout[-2000:]


def test_repeatable_bit_for_bit():
    """Three runs on the same inputs give the same bits in every output: a shape with several
    waves of CTAs in each core (the forward and dQ cores 512 CTAs, the dK/dV core 128), so a race
    between a core's roles or its CTAs would show as a difference between runs."""
    t, T, h, n_q, n_kv, d = 8, 2048, 1024, 32, 8, 128
    inp = si.attn_inputs(T, h, n_q, n_kv, d, seed=11)
    runs = [_run(inp, t, n_q, n_kv, d) for _ in range(3)]
    f0, b0 = runs[0]
    j = torch.arange(T, device=f0["P"][0].device)
    written = j[None, :] < torch.clamp((j[:, None] // 128 + 1) * 128, max=T)   # P's stored band
    for fwd, bwd in runs[1:]:
        for k in ("Q", "K", "V", "O", "Y"):
            for i in range(t):
                assert torch.equal(fwd[k][i], f0[k][i]), f"{k}[{i}] differs between runs"
        for i in range(t):
            assert torch.equal(fwd["P"][i][:, written], f0["P"][i][:, written]), f"P[{i}] differs between runs"
        for k in ("dWq", "dWk", "dWv", "dWo", "dX"):
            for i in range(t):
                assert torch.equal(bwd[k][i], b0[k][i]), f"{k}[{i}] differs between runs"
    del runs, f0, b0
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ Qwen3-8B shape, t = 8

@pytest.fixture(scope="module")
def qwen3():
    s = si.QWEN3_8B_ATTN_T8
    inp = si.attn_inputs(s.T, s.h, s.n_q, s.n_kv, s.d, s.seed)
    return s, inp


def test_qwen3_forward_sampled_rows(qwen3):
    s, inp = qwen3
    fwd, _ = _run(inp, s.t, s.n_q, s.n_kv, s.d, backward=False)
    rows = si.sample_indices(s.T, 24, s.seed).numpy()
    ref = attention.forward_rows(f64(inp["X"]), _W64(inp), s.n_q, s.n_kv, s.d, rows)
    mir = attention.forward_rows(f64(inp["X"]), _W64(inp), s.n_q, s.n_kv, s.d, rows, t=s.t, mirror=True)
    for i in range(s.t):
        assert torch.equal(fwd["Y"][i], fwd["Y"][0])
    err = _Errors()
    err.add(f64(fwd["Y"][0][rows]), ref, "Y[sampled]", mir)
    err.check()
    for i in (0, s.t - 1):
        Ps = fwd["P"][i][:, rows, :].float()
        for r, q in enumerate(rows):
            z = min(s.T, (q // 128 + 1) * 128)
            assert torch.all((Ps[:, r, :q + 1].sum(-1) - 1).abs() < 1e-2)
            assert torch.all(Ps[:, r, q + 1:z] == 0)
    del fwd
    torch.cuda.empty_cache()


def test_qwen3_backward_last_rows(qwen3):
    s, inp = qwen3
    fwd, bwd = _run(inp, s.t, s.n_q, s.n_kv, s.d)
    rows = np.array([s.T - 6, s.T - 3, s.T - 2, s.T - 1])
    ref = attention.backward_rows_dx(f64(inp["X"]), _W64(inp), f64(inp["dY"]), s.n_q, s.n_kv, s.d, rows)
    for i in range(s.t):
        assert torch.equal(bwd["dX"][i], bwd["dX"][0])
    err = _Errors()
    err.add(f64(bwd["dX"][0][rows]), ref, "dX[last rows]")
    err.check()
    del fwd, bwd
    torch.cuda.empty_cache()


def test_qwen3_backward_with_dY_on_the_first_rows_only():
    """dY zero below row m: every gradient equals that of the first m tokens alone, which the
    oracle computes in full; the dX rows from m on are exactly zero."""
    s = si.QWEN3_8B_ATTN_T8
    m = 72
    inp = si.attn_inputs(s.T, s.h, s.n_q, s.n_kv, s.d, s.seed, dY_rows=m)
    fwd, bwd = _run(inp, s.t, s.n_q, s.n_kv, s.d)
    W = _W64(inp)
    X, dY = f64(inp["X"])[:m], f64(inp["dY"])[:m]
    rf = attention.tp_attention_forward(X, W, s.t, s.n_q, s.n_kv, s.d)
    rb = attention.tp_attention_backward(X, W, s.t, s.n_q, s.n_kv, s.d, dY, rf)
    mf = attention.tp_attention_forward(X, W, s.t, s.n_q, s.n_kv, s.d, mirror=True)
    mb = attention.tp_attention_backward(X, W, s.t, s.n_q, s.n_kv, s.d, dY, mf, mirror=True)
    assert torch.count_nonzero(bwd["dX"][0][m:]) == 0
    err = _Errors()
    err.add(f64(bwd["dX"][0][:m]), rb["dX"], "dX[:m]", mb["dX"])
    for i in range(s.t):
        for k in ("dWq", "dWk", "dWv", "dWo"):
            err.add(f64(bwd[k][i]), rb[k][i], f"{k}[{i}]", mb[k][i])
    err.check()
    del fwd, bwd
    torch.cuda.empty_cache()

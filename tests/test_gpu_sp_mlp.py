"""Sequence-parallel MLP block (all-gather and reduce-scatter folded into the GEMMs) vs the
oracle's literal SP block (GPU)."""
import pytest
import torch

import synth_inputs as si
import tensor_transformer_layer_way_gb300 as ttl
from oracle import tp_mlp
from parity import assert_gemm_close, cols, dev, f64, rows

pytestmark = pytest.mark.gpu


def _setup(act, t, T, h, f, seed):
    inp = si.mlp_inputs(T, h, f, act, seed)
    if act == "gelu_tanh":
        A, B, Au = dev(cols(inp["A"], t)), dev(rows(inp["B"], t)), None
        W = {"A": f64(inp["A"]), "B": f64(inp["B"])}
    else:
        A, B, Au = dev(cols(inp["Wg"], t)), dev(rows(inp["Wd"], t)), dev(cols(inp["Wu"], t))
        W = {k: f64(inp[k]) for k in ("Wg", "Wu", "Wd")}
    Xs = dev([x.contiguous() for x in inp["X"].chunk(t, 0)])
    dZs = dev([d.contiguous() for d in inp["dY"].chunk(t, 0)])
    return inp, A, B, Au, W, Xs, dZs


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
@pytest.mark.parametrize("t,T", [(1, 256), (2, 512), (4, 512), (8, 1024), (8, 2048)])
def test_sp_block_matches_oracle(act, t, T):
    h, f = 136, 96 * 8
    inp, A, B, Au, W, Xs, dZs = _setup(act, t, T, h, f, seed=t + T)
    fwd = ttl.sp_mlp_fwd(Xs, A, B, act=act, A_up=Au)
    bwd = ttl.sp_mlp_bwd(Xs, dZs, A, B, fwd, act=act, A_up=Au)
    assert ttl.device_status() == 0
    w = T // t
    X64 = [f64(inp["X"])[r * w:(r + 1) * w] for r in range(t)]
    dZ64 = [f64(inp["dY"])[r * w:(r + 1) * w] for r in range(t)]
    rf = tp_mlp.sp_mlp_forward(X64, W, t, act)
    rb = tp_mlp.sp_mlp_backward(X64, W, t, act, dZ64, rf)
    for r in range(t):
        assert_gemm_close(f64(fwd["Z_slabs"][r]), rf["Z_slabs"][r], f"Z slab {r}")
        assert_gemm_close(f64(bwd["dX_slabs"][r]), rb["dX_slabs"][r], f"dX slab {r}")
    names = ("dA", "dB") if act == "gelu_tanh" else ("dWg", "dWd")
    for i in range(t):
        assert_gemm_close(f64(fwd["H"][i]), rf["H"][i], f"H[{i}]")
        assert_gemm_close(f64(bwd["dA"][i]), rb[names[0]][i], f"{names[0]}[{i}]")
        assert_gemm_close(f64(bwd["dB"][i]), rb[names[1]][i], f"{names[1]}[{i}]")
        if act == "swiglu":
            assert_gemm_close(f64(bwd["dA_up"][i]), rb["dWu"][i], f"dWu[{i}]")


def test_sp_equals_tp_block_on_the_same_inputs():
    act, t, T, h, f = "swiglu", 4, 1024, 256, 1024
    inp, A, B, Au, W, Xs, dZs = _setup(act, t, T, h, f, seed=9)
    sp = ttl.sp_mlp_fwd(Xs, A, B, act=act, A_up=Au)
    spb = ttl.sp_mlp_bwd(Xs, dZs, A, B, sp, act=act, A_up=Au)
    X, dY = dev(inp["X"]), dev(inp["dY"])
    tp = ttl.tp_mlp_fwd(X, A, B, act=act, A_up=Au)
    tpb = ttl.tp_mlp_bwd(X, dY, A, B, tp, act=act, A_up=Au)
    assert ttl.device_status() == 0
    for i in range(t):
        assert torch.equal(sp["H"][i], tp["H"][i])          # fc1 reads the same rows, same order
        assert_gemm_close(f64(spb["dA"][i]), f64(tpb["dA"][i]), f"dA[{i}]")
        assert_gemm_close(f64(spb["dB"][i]), f64(tpb["dB"][i]), f"dB[{i}]")
    assert_gemm_close(f64(torch.cat(sp["Z_slabs"])), f64(tp["Z"][0]), "Z")
    assert_gemm_close(f64(torch.cat(spb["dX_slabs"])), f64(tpb["dX"][0]), "dX")


def test_qwen3_8b_sp_full_size_sampled():
    """The Qwen3-8B SwiGLU block, t = 8, 8192 tokens in slabs of 1024."""
    cfg = si.QWEN3_8B_SWIGLU_T8
    inp, A, B, Au, _, Xs, dZs = _setup(cfg.act, cfg.t, cfg.T, cfg.h, cfg.f, seed=cfg.seed)
    fwd = ttl.sp_mlp_fwd(Xs, A, B, act=cfg.act, A_up=Au)
    bwd = ttl.sp_mlp_bwd(Xs, dZs, A, B, fwd, act=cfg.act, A_up=Au)
    assert ttl.device_status() == 0
    rws = si.sample_indices(cfg.T, 128, cfg.seed).numpy()
    fcols = si.sample_indices(cfg.f, 32, cfg.seed + 1).numpy()
    ref = tp_mlp.swiglu_mlp_sampled(f64(inp["X"]), f64(inp["Wg"]), f64(inp["Wu"]), f64(inp["Wd"]),
                                    f64(inp["dY"]), rws, fcols)
    Z = torch.cat(fwd["Z_slabs"])
    dX = torch.cat(bwd["dX_slabs"])
    r = torch.as_tensor(rws).cuda()
    assert_gemm_close(f64(Z[r]), ref["Z"], "Z rows")
    assert_gemm_close(f64(dX[r]), ref["dX"], "dX rows")
    fs = cfg.f // cfg.t
    dWg = torch.stack([bwd["dA"][c // fs][:, c % fs] for c in fcols.tolist()], 1)
    dWd = torch.stack([bwd["dB"][c // fs][c % fs, :] for c in fcols.tolist()], 0)
    assert_gemm_close(f64(dWg), ref["dWg"], "dWg cols")
    assert_gemm_close(f64(dWd), ref["dWd"], "dWd rows")


def test_slab_rows_must_be_multiples_of_128():
    t, T, h, f = 2, 2 * 100, 64, 128
    inp, A, B, Au, _, Xs, _ = _setup("gelu_tanh", t, T, h, f, seed=1)
    with pytest.raises(ttl.TTLError) as e:
        ttl.sp_mlp_fwd(Xs, A, B, act="gelu_tanh")
    assert e.value.code == ttl.TTL_ERR_SHAPE

"""TP MLP block forward + backward through the C ABI vs the fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import synth_inputs as si
import tensor_transformer_layer_way_gb300 as ttl
from oracle import tp_mlp
from parity import assert_gemm_close, cols, dev, f64, rows

pytestmark = pytest.mark.gpu


def _shards(inp, act, t):
    if act == "gelu_tanh":
        return dict(A=dev(cols(inp["A"], t)), B=dev(rows(inp["B"], t)), A_up=None)
    return dict(A=dev(cols(inp["Wg"], t)), B=dev(rows(inp["Wd"], t)), A_up=dev(cols(inp["Wu"], t)))


def _weights64(inp, act):
    keys = ("A", "B") if act == "gelu_tanh" else ("Wg", "Wu", "Wd")
    return {k: f64(inp[k]) for k in keys}


def _run(inp, act, t, bias=False):
    sh = _shards(inp, act, t)
    X, dY = dev(inp["X"]), dev(inp["dY"])
    b1 = dev(cols(inp["b1"][None, :], t)) if bias else None
    b1 = [b[0].contiguous() for b in b1] if bias else None
    b2 = dev(inp["b2"]) if bias else None
    fwd = ttl.tp_mlp_fwd(X, sh["A"], sh["B"], act=act, A_up=sh["A_up"], b1=b1, b2=b2)
    bwd = ttl.tp_mlp_bwd(X, dY, sh["A"], sh["B"], fwd, act=act, A_up=sh["A_up"], bias=bias)
    assert ttl.device_status() == 0
    return fwd, bwd


def _check_full(inp, act, t, fwd, bwd, bias=False):
    W = _weights64(inp, act)
    X, dY = f64(inp["X"]), f64(inp["dY"])
    b1 = f64(inp["b1"]) if bias else None
    b2 = f64(inp["b2"]) if bias else None
    rf = tp_mlp.tp_mlp_forward(X, W, t, act, b1, b2)
    rb = tp_mlp.tp_mlp_backward(X, W, t, act, dY, rf)
    for i in range(t):
        assert_gemm_close(f64(fwd["Z"][i]), rf["Z"], f"Z[{i}]")
        assert_gemm_close(f64(bwd["dX"][i]), rb["dX"], f"dX[{i}]")
        assert torch.equal(fwd["Z"][i], fwd["Z"][0]) and torch.equal(bwd["dX"][i], bwd["dX"][0])
        assert_gemm_close(f64(fwd["H"][i]), rf["H"][i], f"H[{i}]")
        if act == "gelu_tanh":
            assert_gemm_close(f64(fwd["U"][i]), rf["U"][i], f"U[{i}]")
            assert_gemm_close(f64(bwd["dA"][i]), rb["dA"][i], f"dA[{i}]")
            assert_gemm_close(f64(bwd["dB"][i]), rb["dB"][i], f"dB[{i}]")
            if bias:
                assert_gemm_close(f64(bwd["db1"][i]), rb["db1"][i], f"db1[{i}]")
        else:
            assert_gemm_close(f64(fwd["U"][i]), rf["G"][i], f"G[{i}]")
            assert_gemm_close(f64(fwd["V"][i]), rf["V"][i], f"V[{i}]")
            assert_gemm_close(f64(bwd["dA"][i]), rb["dWg"][i], f"dWg[{i}]")
            assert_gemm_close(f64(bwd["dA_up"][i]), rb["dWu"][i], f"dWu[{i}]")
            assert_gemm_close(f64(bwd["dB"][i]), rb["dWd"][i], f"dWd[{i}]")
    if bias:
        assert_gemm_close(f64(bwd["db2"]), rb["db2"], "db2")


def test_toy_mlp_t2_gelu_seed0():
    """The t=2 tanh-GeLU block of the "MLP: column then row" section, X [128,256], 4h=1024."""
    cfg = si.TP_MLP_GELU_T2
    inp = si.mlp_inputs(cfg.T, cfg.h, cfg.f, cfg.act, cfg.seed)
    fwd, bwd = _run(inp, cfg.act, cfg.t)
    _check_full(inp, cfg.act, cfg.t, fwd, bwd)


@pytest.mark.parametrize("act", ["gelu_tanh", "swiglu"])
@pytest.mark.parametrize("t", [1, 2, 4])
def test_ragged_shapes(act, t):
    T, h, f = 200, 136, 96 * 4            # T and h not multiples of the 128/256 tiles
    inp = si.mlp_inputs(T, h, f, act, seed=11 + t)
    fwd, bwd = _run(inp, act, t)
    _check_full(inp, act, t, fwd, bwd)


@pytest.mark.parametrize("t", [1, 2, 4])
def test_gelu_with_bias_row_bias_added_once(t):
    T, h, f = 64, 128, 512
    inp = si.mlp_inputs(T, h, f, "gelu_tanh", seed=21, bias=True)
    fwd, bwd = _run(inp, "gelu_tanh", t, bias=True)
    _check_full(inp, "gelu_tanh", t, fwd, bwd, bias=True)


def test_sharded_matches_unsharded_t1():
    T, h, f = 256, 256, 1024
    inp = si.mlp_inputs(T, h, f, "swiglu", seed=5)
    f1, b1 = _run(inp, "swiglu", 1)
    f8, b8 = _run(inp, "swiglu", 8)
    assert_gemm_close(f64(f8["Z"][3]), f64(f1["Z"][0]), "Z t=8 vs t=1")
    assert_gemm_close(f64(b8["dX"][5]), f64(b1["dX"][0]), "dX t=8 vs t=1")
    assert_gemm_close(torch.cat([x.float() for x in b8["dA"]], 1).numpy(force=True), f64(b1["dA"][0]), "dWg")


def test_zero_tokens():
    t, h, f = 2, 64, 128
    inp = si.mlp_inputs(0, h, f, "gelu_tanh", seed=1)
    fwd, bwd = _run(inp, "gelu_tanh", t)
    for i in range(t):
        assert torch.count_nonzero(bwd["dA"][i]).item() == 0
        assert torch.count_nonzero(bwd["dB"][i]).item() == 0


def test_repeatable_bit_for_bit():
    inp = si.mlp_inputs(256, 256, 1024, "swiglu", seed=2)
    f1, b1 = _run(inp, "swiglu", 4)
    f2, b2 = _run(inp, "swiglu", 4)
    for k in ("Z", "H"):
        for a, b in zip(f1[k], f2[k]):
            assert torch.equal(a, b)
    for k in ("dX", "dA", "dA_up", "dB"):
        for a, b in zip(b1[k], b2[k]):
            assert torch.equal(a, b)


def test_qwen3_8b_swiglu_t8_full_size_sampled():
    """X [8192,4096], gate/up [4096,12288] in 1536-column shards, down in 1536-row shards: the
    launch configuration the bench times.  256 token rows of Z and dX and 64 FFN columns of
    every weight gradient are computed exactly by the oracle."""
    cfg = si.QWEN3_8B_SWIGLU_T8
    inp = si.mlp_inputs(cfg.T, cfg.h, cfg.f, cfg.act, cfg.seed)
    fwd, bwd = _run(inp, cfg.act, cfg.t)
    rows_ = si.sample_indices(cfg.T, 256, cfg.seed).numpy()
    fcols = si.sample_indices(cfg.f, 64, cfg.seed + 1).numpy()
    ref = tp_mlp.swiglu_mlp_sampled(f64(inp["X"]), f64(inp["Wg"]), f64(inp["Wu"]), f64(inp["Wd"]), f64(inp["dY"]),
                                    rows_, fcols)
    fs = cfg.f // cfg.t
    r = torch.as_tensor(rows_)
    assert_gemm_close(f64(fwd["Z"][0][r.cuda()]), ref["Z"], "Z rows")
    assert_gemm_close(f64(bwd["dX"][7][r.cuda()]), ref["dX"], "dX rows")
    dWg = torch.stack([bwd["dA"][c // fs][:, c % fs] for c in fcols.tolist()], 1)
    dWu = torch.stack([bwd["dA_up"][c // fs][:, c % fs] for c in fcols.tolist()], 1)
    dWd = torch.stack([bwd["dB"][c // fs][c % fs, :] for c in fcols.tolist()], 0)
    assert_gemm_close(f64(dWg), ref["dWg"], "dWg cols")
    assert_gemm_close(f64(dWu), ref["dWu"], "dWu cols")
    assert_gemm_close(f64(dWd), ref["dWd"], "dWd rows")
    for i in range(1, cfg.t):
        assert torch.equal(fwd["Z"][0], fwd["Z"][i])
        assert torch.equal(bwd["dX"][0], bwd["dX"][i])


_CHILD = r"""
import os, sys
root, out = sys.argv[1], sys.argv[2]
sys.path[:0] = [root, os.path.join(root, "tests")]
import torch
import synth_inputs as si
import test_gpu_mlp as m
inp = si.mlp_inputs(520, 392, 640, "swiglu", seed=31)
fwd, bwd = m._run(inp, "swiglu", 2)
ce = m._ce_case()
torch.save({"fwd": {k: [x.cpu() for x in v] for k, v in fwd.items() if isinstance(v, list)},
            "bwd": {k: [x.cpu() for x in v] for k, v in bwd.items() if isinstance(v, list)},
            "ce": {k: ([x.cpu() for x in v] if isinstance(v, list) else v.cpu()) for k, v in ce.items() if v is not None}},
           out)
"""


def _ce_case():
    """Vocab-parallel CE, t = 2, 600-column shards (fp32 logits and the fused partials take the
    wide tiles when allowed), ragged T."""
    import tensor_transformer_layer_way_gb300 as ttl_
    g = torch.Generator().manual_seed(41)
    T, h, V = 300, 256, 1200
    H = torch.randn((T, h), generator=g).to(torch.bfloat16).cuda()
    W = [(torch.randn((V // 2, h), generator=g) * 0.05).to(torch.bfloat16).cuda() for _ in range(2)]
    target = torch.randint(0, V, (T,), generator=g).cuda()
    out = ttl_.vocab_parallel_ce(H, W, target, fused_stats=True)
    torch.cuda.synchronize()
    assert ttl_.device_status() == 0
    return {k: v for k, v in out.items() if k != "ws"}


def test_wide_tiles_give_the_same_bits_as_256_column_tiles(tmp_path):
    """Every GEMM output element is the same chain of K = 16 MMAs whichever tile width the
    launch uses, rounded once, so the 256x512 tiles (this process) and the 256x256 tiles (a
    child process with TTL_GEMM_WIDE=0) must agree bit for bit: on a SwiGLU block whose fc1,
    fc2, weight-gradient and dX launches all qualify for the wide tiles (ragged T = 520), and
    on a vocab-parallel CE (fp32 logits, the fused partials, the loss, dlogits and dH)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = str(tmp_path / "narrow.pt")
    env = dict(os.environ, TTL_GEMM_WIDE="0")
    subprocess.run([sys.executable, "-c", _CHILD, root, out], env=env, check=True, timeout=600)
    narrow = torch.load(out)
    inp = si.mlp_inputs(520, 392, 640, "swiglu", seed=31)
    fwd, bwd = _run(inp, "swiglu", 2)
    for part, res in (("fwd", fwd), ("bwd", bwd)):
        for k, lst in narrow[part].items():
            for i, x in enumerate(lst):
                assert torch.equal(res[k][i].cpu(), x), f"{part} {k}[{i}] differs between tile widths"
    ce = _ce_case()
    for k, v in narrow["ce"].items():
        got = ce[k]
        if isinstance(v, list):
            for i, x in enumerate(v):
                assert torch.equal(got[i].cpu(), x), f"ce {k}[{i}] differs between tile widths"
        else:
            assert torch.equal(got.cpu(), v), f"ce {k} differs between tile widths"

"""Vocab-parallel LM head + cross-entropy vs the oracle (GPU)."""
import numpy as np
import pytest
import torch

import synth_inputs as si
import tensor_transformer_layer_way_gb300 as ttl
from oracle import vocab_ce
from parity import assert_fp32_close, assert_gemm_close, dev, f32, f64

pytestmark = pytest.mark.gpu


def _assert_sumexp_close(got, ref, Z, name):
    """Per-token sum-exp s = sum_v exp(z_v - m) against the oracle.  It inherits the logits'
    error: d(log s) = sum_v softmax_v dz_v (the shift by the max cancels), so |ds / s| <= max_v
    |dz_v|, which the logits check bounds by 1e-5 * max|z|.  A 4-ulp allowance covers the
    exponentials' own rounding.  At K = 4096 the tensor cores' fp32 accumulation moves the
    logits by a few 1e-5, so the plain 1e-5 relative bound is not attainable for s, while the
    loss (log s + m - z_y) still meets it."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = (1e-5 * np.abs(Z).max() + 4 * 2.0 ** -24) * ref
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"{name}: max relative error {(err / ref).max():.3e} > {(bound / ref).max():.3e}"


def _run(H, W, target, t, flags=0, fused=True):
    Ws = dev([w.contiguous() for w in W.chunk(t, 0)])
    out = ttl.vocab_parallel_ce(dev(H), Ws, dev(target), flags=flags, fused_stats=fused)
    return out


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("t,T,h,V", [(1, 64, 64, 512), (4, 100, 64, 4 * 296), (8, 130, 136, 8 * 48),
                                     (2, 300, 64, 2 * 600)])
def test_small_full_parity(t, T, h, V, fused):
    inp = si.ce_inputs(T, h, V, seed=t + T)
    out = _run(inp["H"], inp["W"], inp["target"], t, fused=fused)
    assert ttl.device_status() == 0
    ref = vocab_ce.vocab_parallel_ce(f64(inp["H"]), f64(inp["W"]), inp["target"].numpy(), t)
    Vs = V // t
    stats = f32(out["stats"]).reshape(3 * t + 2, T)
    for i in range(t):
        assert_fp32_close(f32(out["logits"][i]), ref["Z"][i], f"logits[{i}]")
        assert_fp32_close(stats[3 * i], ref["stats"][i][0], f"max[{i}]")
        assert_fp32_close(stats[3 * i + 1], ref["stats"][i][1], f"sumexp[{i}]")
        assert_fp32_close(stats[3 * i + 2], ref["stats"][i][2], f"target logit[{i}]")
        assert_gemm_close(f64(out["dlogits"][i]), ref["dZ"][i], f"dlogits[{i}]")
    assert_fp32_close(stats[3 * t], ref["lse"], "lse")
    assert_fp32_close(stats[3 * t + 1], ref["loss_tok"], "loss per token")
    assert abs(out["loss"].item() - ref["loss"]) <= 1e-5 * abs(ref["loss"])
    assert_gemm_close(f64(out["dH"]), ref["dH"], "dH")
    del Vs


def test_fp32_dlogits_in_place_and_forward_only():
    t, T, h, V = 2, 64, 64, 2 * 136
    inp = si.ce_inputs(T, h, V, seed=1)
    out = _run(inp["H"], inp["W"], inp["target"], t, flags=ttl.CE_FP32_DLOGITS)
    ref = vocab_ce.vocab_parallel_ce(f64(inp["H"]), f64(inp["W"]), inp["target"].numpy(), t)
    for i in range(t):
        assert_fp32_close(f32(out["logits"][i]), ref["dZ"][i], f"fp32 dlogits[{i}]", rel=1e-5)
    fo = _run(inp["H"], inp["W"], inp["target"], t, flags=ttl.CE_FORWARD_ONLY)
    assert abs(fo["loss"].item() - ref["loss"]) <= 1e-5 * abs(ref["loss"])


def test_all_zero_logits_give_log_v():
    t, T, h, V = 8, 32, 64, 8 * 64
    H = torch.zeros((T, h), dtype=torch.bfloat16)
    W = si.randn_bf16(si.generator(0), (V, h))
    target = torch.randint(0, V, (T,), generator=si.generator(1))
    out = _run(H, W, target, t, flags=ttl.CE_FP32_DLOGITS)
    assert abs(out["loss"].item() - np.log(V)) <= 1e-5 * np.log(V)
    # fp32 dlogits: each row sums to zero up to fp32 rounding of V terms
    dZ32 = torch.cat(out["logits"], 1).double()
    assert dZ32.sum(1).abs().max().item() <= 1e-6 / T
    # bf16 dlogits: the target entry (1/V - 1)/T carries one bf16 rounding (2^-9 relative)
    dZ = torch.cat([d.double() for d in out["dlogits"]], 1)
    assert dZ.sum(1).abs().max().item() <= 2.0 ** -8 / T


def test_fused_and_separate_statistics_agree():
    t, T, h, V = 8, 256, 128, 8 * 520
    inp = si.ce_inputs(T, h, V, seed=3)
    a = _run(inp["H"], inp["W"], inp["target"], t, fused=True)
    b = _run(inp["H"], inp["W"], inp["target"], t, fused=False)
    assert ttl.device_status() == 0
    for i in range(t):
        assert torch.equal(a["logits"][i], b["logits"][i])
    sa = f32(a["stats"]).reshape(3 * t + 2, T)
    sb = f32(b["stats"]).reshape(3 * t + 2, T)
    for i in range(t):
        np.testing.assert_array_equal(sa[3 * i], sb[3 * i])            # maxima are exact
        np.testing.assert_array_equal(sa[3 * i + 2], sb[3 * i + 2])    # target logits are copies
        assert_fp32_close(sa[3 * i + 1], sb[3 * i + 1], f"sumexp[{i}]")
    assert abs(a["loss"].item() - b["loss"].item()) <= 1e-5 * abs(b["loss"].item())


@pytest.mark.parametrize("fused", [True, False])
def test_vocab_parallel_ce_full_size_sampled(fused):
    """H [8192, 4096], W [151936, 4096] in 8 vocab shards of 18992 rows (fp32 logits 4.98 GB).
    On sampled token rows, for every shard: the fp32 logits over all 18992 columns (the last
    256-wide tile holds only 48 of them), the three statistics, and the bf16 dlogits; then the
    combined statistics, the per-token loss and dH.  The mean loss is checked as the mean of
    the per-token losses, which the oracle pins on the sample."""
    cfg = si.VOCAB_CE_T8
    inp = si.ce_inputs(cfg.T, cfg.h, cfg.V, cfg.seed)
    out = _run(inp["H"], inp["W"], inp["target"], cfg.t, fused=fused)
    assert ttl.device_status() == 0
    rows = si.sample_indices(cfg.T, 48, cfg.seed).numpy()
    ref = vocab_ce.vocab_parallel_ce(f64(inp["H"]), f64(inp["W"]), inp["target"].numpy(), cfg.t, rows=rows)
    stats = f32(out["stats"]).reshape(3 * cfg.t + 2, cfg.T)
    r = torch.as_tensor(rows).cuda()
    Vs = cfg.V // cfg.t
    tail = (Vs // 256) * 256                       # first column of the ragged last tile
    assert Vs - tail == 48
    for i in range(cfg.t):
        Z = f32(out["logits"][i][r])
        assert_fp32_close(Z, ref["Z"][i], f"logits[{i}] rows")
        assert_fp32_close(Z[:, tail:], ref["Z"][i][:, tail:], f"logits[{i}] rows, ragged last tile")
        assert_fp32_close(stats[3 * i][rows], ref["stats"][i][0], f"max[{i}] rows")
        _assert_sumexp_close(stats[3 * i + 1][rows], ref["stats"][i][1], ref["Z"][i], f"sumexp[{i}] rows")
        assert_fp32_close(stats[3 * i + 2][rows], ref["stats"][i][2], f"target logit[{i}] rows")
        assert_gemm_close(f64(out["dlogits"][i][r]), ref["dZ"][i], f"dlogits[{i}] rows")
    assert_fp32_close(stats[3 * cfg.t][rows], ref["lse"], "lse (sampled rows)")
    assert_fp32_close(stats[3 * cfg.t + 1][rows], ref["loss_tok"], "loss per token (sampled rows)")
    loss_tok = stats[3 * cfg.t + 1].astype(np.float64)
    assert abs(out["loss"].item() - loss_tok.mean()) <= 1e-5 * abs(loss_tok.mean())
    assert_gemm_close(f64(out["dH"][r]), ref["dH"], "dH rows")
    del out
    torch.cuda.empty_cache()

"""Shared helpers for the GPU parity tests: shard splitting on the host, device transfer,
and the tolerances the comparisons use.

Tolerances (bf16 operands, fp32 accumulation):
  * bf16 GEMM outputs: relative Frobenius error <= 5e-3 and max-abs error <= 2e-2 * max|ref|;
  * fp32 reductions and the CE loss: relative error <= 1e-5;
  * gathers, scatters, copies and the ordered bf16 reductions: bit-exact.
"""
import numpy as np
import torch

REL_FRO = 5e-3
MAX_ABS_FRAC = 2e-2
REL_FP32 = 1e-5


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def cols(W, t):
    w = W.shape[1] // t
    return [W[:, i * w:(i + 1) * w].contiguous() for i in range(t)]


def rows(W, t):
    w = W.shape[0] // t
    return [W[i * w:(i + 1) * w, :].contiguous() for i in range(t)]


def dev(x, device="cuda"):
    if isinstance(x, (list, tuple)):
        return [dev(v, device) for v in x]
    return x.to(device)


def assert_gemm_close(got, ref, name=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    rf = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    ma = np.abs(got - ref).max() if got.size else 0.0
    lim = MAX_ABS_FRAC * (np.abs(ref).max() if ref.size else 0.0)
    assert rf <= REL_FRO, f"{name}: relative Frobenius error {rf:.3e} > {REL_FRO}"
    assert ma <= lim, f"{name}: max-abs error {ma:.3e} > {lim:.3e}"


def assert_fp32_close(got, ref, name="", rel=REL_FP32):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    scale = max(np.abs(ref).max() if ref.size else 0.0, 1e-30)
    err = np.abs(got - ref).max() if got.size else 0.0
    assert err <= rel * scale, f"{name}: max error {err:.3e} > {rel:.1e} * {scale:.3e}"

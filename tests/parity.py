"""Shared helpers for the GPU parity tests: shard splitting on the host, device transfer,
and the tolerances the comparisons use.

Tolerances (bf16 operands, fp32 accumulation):
  * bf16 GEMM outputs: relative Frobenius error <= 5e-3 and max-abs error <= 2e-2 * max|ref|;
  * fp32 reductions and the CE loss: relative error <= 1e-5;
  * gathers, scatters, copies and the ordered bf16 reductions: bit-exact;
  * the attention block's outputs sit at the end of a chain of up to seven bf16 roundings
    (Q/K/V, P, O, dO, dS, dQ/dK/dV, the output itself).  They are compared twice:
      - against the oracle's rounding mirror (the same float64 arithmetic rounded to bf16 where
        the bf16 data path materialises a tensor) at the GEMM bounds above, 5e-3 and 2e-2;
      - against the plain float64 oracle at relative Frobenius error <= 1.05e-2 and max-abs
        <= 2e-2 * max|ref|.  The 1.05e-2 is the triangle inequality over the two measured legs:
        5e-3 allowed between the kernels and the mirror, plus 5.5e-3 for the mirror's own
        distance from float64 (largest measured over the eight small test blocks: 5.14e-3, on
        dWk; the cancellation in dS = P (dP - D) amplifies the roundings of dP and D).
"""
import numpy as np
import torch

REL_FRO = 5e-3
MAX_ABS_FRAC = 2e-2
REL_FP32 = 1e-5
ATTN_MIRROR_REL_FRO = 5e-3
ATTN_MIRROR_MAX_ABS_FRAC = 2e-2
ATTN_FP64_REL_FRO = 5e-3 + 5.5e-3
ATTN_FP64_MAX_ABS_FRAC = 2e-2


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


def gemm_errors(got, ref, name=""):
    """(relative Frobenius error, max-abs error / max|ref|) of got against ref."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    rf = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    ma = np.abs(got - ref).max() if got.size else 0.0
    return rf, ma / max(np.abs(ref).max() if ref.size else 0.0, 1e-300)


def assert_gemm_close(got, ref, name="", rel_fro=REL_FRO, max_abs_frac=MAX_ABS_FRAC):
    rf, maf = gemm_errors(got, ref, name)
    assert rf <= rel_fro, f"{name}: relative Frobenius error {rf:.3e} > {rel_fro}"
    assert maf <= max_abs_frac, f"{name}: max-abs error {maf:.3e} of max|ref| > {max_abs_frac}"


def assert_fp32_close(got, ref, name="", rel=REL_FP32):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    scale = max(np.abs(ref).max() if ref.size else 0.0, 1e-30)
    err = np.abs(got - ref).max() if got.size else 0.0
    assert err <= rel * scale, f"{name}: max error {err:.3e} > {rel:.1e} * {scale:.3e}"

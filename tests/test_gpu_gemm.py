"""tcgen05 GEMM core against the oracle's linear (GPU)."""
import numpy as np
import pytest
import torch

import synth_inputs as si
import tensor_transformer_layer_way_gb300 as ttl
from oracle import tp_mlp
from oracle.numerics import round_to_bf16
from parity import assert_gemm_close, f64

pytestmark = pytest.mark.gpu

SHAPES = [(128, 256, 64), (300, 264, 200), (1, 8, 8), (520, 776, 1000), (256, 512, 4096)]


def _operands(M, N, K, a_kmajor, b_kmajor, ints, seed):
    g = si.generator(seed)
    if ints:
        A = si.small_int_bf16(g, (M, K), -2, 2)
        B = si.small_int_bf16(g, (K, N), -2, 2)
    else:
        A = si.randn_bf16(g, (M, K))
        B = si.randn_bf16(g, (K, N), 0.05)
    A_st = A if a_kmajor else A.t().contiguous()       # stored [M,K] or [K,M]
    B_st = B.t().contiguous() if b_kmajor else B        # stored [N,K] or [K,N]
    return A, B, A_st.cuda(), B_st.cuda()


@pytest.mark.parametrize("a_kmajor,b_kmajor", [(True, True), (True, False), (False, True), (False, False)])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_integer_inputs_exact(M, N, K, a_kmajor, b_kmajor):
    A, B, Ad, Bd = _operands(M, N, K, a_kmajor, b_kmajor, True, M + N + K)
    D = torch.full((M, N), float("nan"), device="cuda", dtype=torch.float32)
    if not a_kmajor and M % 8:
        # A stored [K, M] has rows of M bf16: not a multiple of 16 bytes, which TMA cannot
        # address; the library must refuse before launching anything.
        with pytest.raises(ttl.TTLError) as e:
            ttl.gemm(Ad, Bd, D, a_kmajor=a_kmajor, b_kmajor=b_kmajor)
        assert e.value.code == ttl.TTL_ERR_ALIGN
        return
    ttl.gemm(Ad, Bd, D, a_kmajor=a_kmajor, b_kmajor=b_kmajor)
    assert ttl.device_status() == 0
    ref = tp_mlp.column_parallel_forward(f64(A), [f64(B)])[0]
    np.testing.assert_array_equal(D.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("a_kmajor,b_kmajor", [(True, True), (True, False), (False, True), (False, False)])
def test_gemm_random_bf16_output(a_kmajor, b_kmajor):
    M, N, K = 384, 520, 1032
    A, B, Ad, Bd = _operands(M, N, K, a_kmajor, b_kmajor, False, 7)
    D = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
    ttl.gemm(Ad, Bd, D, a_kmajor=a_kmajor, b_kmajor=b_kmajor)
    assert ttl.device_status() == 0
    ref = tp_mlp.column_parallel_forward(f64(A), [f64(B)])[0]
    assert_gemm_close(f64(D), ref, "D")


def test_gemm_empty_contraction_gives_zeros():
    A = torch.empty((16, 0), device="cuda", dtype=torch.bfloat16)
    B = torch.empty((24, 0), device="cuda", dtype=torch.bfloat16)
    D = torch.full((16, 24), 3.0, device="cuda", dtype=torch.float32)
    ttl.gemm(A, B, D)
    assert torch.count_nonzero(D).item() == 0


def test_gemm_deterministic():
    A, B, Ad, Bd = _operands(640, 1024, 2048, True, False, False, 3)
    D1 = torch.empty((640, 1024), device="cuda", dtype=torch.float32)
    D2 = torch.empty_like(D1)
    ttl.gemm(Ad, Bd, D1, b_kmajor=False)
    ttl.gemm(Ad, Bd, D2, b_kmajor=False)
    assert torch.equal(D1, D2)


@pytest.mark.parametrize("a_kmajor,b_kmajor", [(True, True), (True, False), (False, True), (False, False)])
@pytest.mark.parametrize("M,N,K", [(520, 776, 1000), (256, 512, 4096), (296, 1032, 192), (1024, 264, 512)])
def test_gemm_integer_inputs_bf16_output_exact(M, N, K, a_kmajor, b_kmajor):
    """bf16 outputs (the 256 x 512 tiles with the TMA-store epilogue take these launches when
    N > 256) of small-integer products: every fp32 sum is exact, so D must equal the exact
    product rounded once to bf16, element for element, ragged rows and columns included."""
    A, B, Ad, Bd = _operands(M, N, K, a_kmajor, b_kmajor, True, 3 * M + N + K)
    D = torch.full((M, N), float("nan"), device="cuda", dtype=torch.bfloat16)
    ttl.gemm(Ad, Bd, D, a_kmajor=a_kmajor, b_kmajor=b_kmajor)
    assert ttl.device_status() == 0
    ref = tp_mlp.column_parallel_forward(f64(A), [f64(B)])[0]
    np.testing.assert_array_equal(f64(D), round_to_bf16(ref).astype(np.float64))

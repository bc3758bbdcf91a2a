"""GTP_remat weight path vs the oracle (GPU): gather, slot and folded GEMMs, wgrad
reduce-scatter into fp32 staging, one-layer-deferred finalize."""
import numpy as np
import pytest
import torch

import synth_inputs as si
import tensor_transformer_layer_way_gb300 as ttl
from oracle import gtp
from parity import assert_fp32_close, assert_gemm_close, dev, f32, f64

pytestmark = pytest.mark.gpu


def _shards(W, g):
    return dev([s.contiguous() for s in W.chunk(g, 0)])


@pytest.mark.parametrize("g", [1, 4, 8])
def test_gather_bit_exact_and_event(g):
    K, N = 64 * g, 136
    W = si.randn_bf16(si.generator(g), (K, N), 0.02)
    sh = _shards(W, g)
    slot = torch.empty((K, N), device="cuda", dtype=torch.bfloat16)
    side = torch.cuda.Stream()
    ev = torch.cuda.Event()
    with torch.cuda.stream(side):
        ttl.gtp_gather(sh, slot, stream=side, done_event=ev)
    torch.cuda.current_stream().wait_event(ev)
    assert torch.equal(slot.cpu(), W)
    np.testing.assert_array_equal(f32(slot).view(np.uint32),
                                  gtp.gather([f32(s) for s in sh]).view(np.uint32))


@pytest.mark.parametrize("g,M,K,N", [(4, 192, 256, 128), (8, 100, 512, 264), (2, 384, 128 * 2, 520)])
def test_forward_and_dgrad_slot_and_folded(g, M, K, N):
    inp = si.gtp_inputs(1, K, N, M, seed=K + N)
    W = inp["W"][0]
    sh = _shards(W, g)
    X = dev(inp["X"])
    dY = dev(inp["dY"][0])
    slot = torch.empty((K, N), device="cuda", dtype=torch.bfloat16)
    ttl.gtp_gather(sh, slot)
    Y_slot = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
    Y_fold = torch.empty_like(Y_slot)
    ttl.gtp_gather_gemm(X, sh, Y_slot, slot=slot)
    ttl.gtp_gather_gemm(X, sh, Y_fold)
    dX_slot = torch.empty((M, K), device="cuda", dtype=torch.bfloat16)
    dX_fold = torch.empty_like(dX_slot)
    ttl.gtp_gather_gemm(dY, sh, dX_slot, slot=slot, transpose_w=True)
    ttl.gtp_gather_gemm(dY, sh, dX_fold, transpose_w=True)
    assert ttl.device_status() == 0
    assert torch.equal(Y_slot, Y_fold)
    assert torch.equal(dX_slot, dX_fold)
    assert_gemm_close(f64(Y_slot), gtp.forward_gemm(f64(inp["X"]), f64(W)), "Y")
    assert_gemm_close(f64(dX_slot), gtp.dgrad_gemm(f64(inp["dY"][0]), f64(W)), "dX")


def test_gather_gemm_integer_exact():
    g, M, K, N = 4, 130, 256, 72
    inp = si.gtp_inputs(1, K, N, M, seed=3, ints=True)
    sh = _shards(inp["W"][0], g)
    Y = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
    ttl.gtp_gather_gemm(dev(inp["X"]), sh, Y)
    ref = gtp.forward_gemm(f64(inp["X"]), f64(inp["W"][0]))
    # sums of at most 256 products of |x|<=3, |w|<=2 stay below 2^11: exact in bf16 only up to 256
    mask = np.abs(ref) <= 256
    np.testing.assert_array_equal(f64(Y)[mask], ref[mask])


@pytest.mark.parametrize("g", [1, 2, 8])
def test_wgrad_reduce_scatter_staging(g):
    M, K, N = 256, 64 * g * 2, 200
    inp = si.gtp_inputs(1, K, N, M, seed=g)
    staging = [torch.full((K // g, N), float("nan"), device="cuda") for _ in range(g)]
    ttl.gtp_wgrad_rs_finalize(dev(inp["X"]), dev(inp["dY"][0]), staging)
    assert ttl.device_status() == 0
    ref = gtp.wgrad_reduce_scatter(f64(inp["X"]), f64(inp["dY"][0]), g)
    for j in range(g):
        assert_fp32_close(f32(staging[j]), ref[j], f"staging[{j}]", rel=2e-5)


def test_deferred_finalize_chain_matches_oracle_schedule():
    L, g, M, K, N = 4, 4, 128, 256, 64
    inp = si.gtp_inputs(L, K, N, M, seed=17)
    X = dev(inp["X"])
    dYs = dev(inp["dY"])
    mg0 = [[torch.randn((K // g, N), generator=si.generator(100 + l * g + j)) for j in range(g)] for l in range(L)]
    mg = [[m.cuda() for m in layer] for layer in mg0]
    staging = [[torch.empty((K // g, N), device="cuda") for _ in range(g)] for _ in range(L)]
    seen = {}
    for l in range(L - 1, -1, -1):
        prev = l + 1 if l + 1 < L else None
        ttl.gtp_wgrad_rs_finalize(X, dYs[l], staging[l],
                                  staging_prev=staging[prev] if prev is not None else None,
                                  main_grad_prev=mg[prev] if prev is not None else None,
                                  sync=(l == 0), main_grad_cur=mg[0] if l == 0 else None)
        torch.cuda.synchronize()
        seen[l] = sorted(k for k in range(L)
                         if not torch.equal(mg[k][0].cpu(), mg0[k][0]))
    assert ttl.device_status() == 0
    st_ref = [gtp.wgrad_reduce_scatter(f64(inp["X"]), f64(inp["dY"][l]), g) for l in range(L)]
    ref = gtp.deferred_finalize([[m.double().numpy() for m in layer] for layer in mg0], st_ref)
    assert seen == ref["updated_after_step"]
    for l in range(L):
        for j in range(g):
            assert_fp32_close(f32(mg[l][j]), ref["main_grad"][l][j], f"main_grad[{l}][{j}]", rel=2e-5)


def test_full_size_chain_layer_sampled():
    """One layer of the h=8192, TP=4, GTP_remat=8 chain: TP slice [8192, 2048] as 8 shards of
    [1024, 2048] (4 MiB each), X [4096, 8192]."""
    cfg = si.GTP_CHAIN
    K, N, M, g = cfg.h, cfg.h // cfg.tp, cfg.T, cfg.g
    inp = si.gtp_inputs(1, K, N, M, seed=cfg.seed)
    W = inp["W"][0]
    sh = _shards(W, g)
    assert sh[0].numel() * 2 == 4 * 2 ** 20
    X, dY = dev(inp["X"]), dev(inp["dY"][0])
    slot = torch.empty((K, N), device="cuda", dtype=torch.bfloat16)
    ttl.gtp_gather(sh, slot)
    assert torch.equal(slot.cpu(), W)
    Y = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
    Yf = torch.empty_like(Y)
    ttl.gtp_gather_gemm(X, sh, Y, slot=slot)
    ttl.gtp_gather_gemm(X, sh, Yf)
    assert torch.equal(Y, Yf)
    dX = torch.empty((M, K), device="cuda", dtype=torch.bfloat16)
    ttl.gtp_gather_gemm(dY, sh, dX, transpose_w=True)
    staging = [torch.empty((K // g, N), device="cuda") for _ in range(g)]
    ttl.gtp_wgrad_rs_finalize(X, dY, staging)
    assert ttl.device_status() == 0
    r = si.sample_indices(M, 128, 4).numpy()
    Xs, dYs, W64 = f64(inp["X"]), f64(inp["dY"][0]), f64(W)
    assert_gemm_close(f64(Y)[r], gtp.forward_gemm(Xs[r], W64), "Y rows")
    assert_gemm_close(f64(dX)[r], gtp.dgrad_gemm(dYs[r], W64), "dX rows")
    kr = si.sample_indices(K, 64, 5).numpy()
    full_rows = (Xs[:, kr].T @ dYs)           # rows kr of X^T dY, every token
    got = np.stack([f32(staging[k // (K // g)][k % (K // g)]) for k in kr.tolist()])
    assert_fp32_close(got, full_rows, "staging rows", rel=2e-5)


def test_prefetch_chain_runner_matches_direct_and_oracle():
    """The two-slot side-stream chain (warm, cold and folded) gives the same bits as direct
    calls, and its deferred finalize leaves main_grad = initial + staging, as the oracle's
    schedule does."""
    from tensor_transformer_layer_way_gb300 import chain
    L, g, M, K, N = 5, 4, 192, 512, 136
    inp = si.gtp_inputs(L, K, N, M, seed=23)
    shards = [_shards(W, g) for W in inp["W"]]
    X = dev(inp["X"])
    dYs = dev(inp["dY"])
    slots = [torch.empty((K, N), device="cuda", dtype=torch.bfloat16) for _ in range(2)]
    runner = chain.GtpChain(ttl, torch, shards, slots)
    Yc = [torch.empty((M, N), device="cuda", dtype=torch.bfloat16) for _ in range(L)]
    Yw = [torch.empty_like(y) for y in Yc]
    Yf = [torch.empty_like(y) for y in Yc]
    runner.forward(X, Yc, cold=True)
    runner.forward(X, Yw)
    runner.forward(X, Yf, folded=True)
    dX = [torch.empty((M, K), device="cuda", dtype=torch.bfloat16) for _ in range(L)]
    staging = [[torch.empty((K // g, N), device="cuda") for _ in range(g)] for _ in range(L)]
    mg = [[torch.zeros((K // g, N), device="cuda") for _ in range(g)] for _ in range(L)]
    runner.backward(X, dYs, dX, staging, mg)
    torch.cuda.synchronize()
    assert ttl.device_status() == 0
    for l in range(L):
        assert torch.equal(Yc[l], Yw[l]) and torch.equal(Yc[l], Yf[l])
        direct = torch.empty_like(dX[l])
        ttl.gtp_gather_gemm(dYs[l], shards[l], direct, transpose_w=True)
        assert torch.equal(direct, dX[l])
        assert_gemm_close(f64(Yw[l]), gtp.forward_gemm(f64(inp["X"]), f64(inp["W"][l])), f"Y[{l}]")
    st_ref = [gtp.wgrad_reduce_scatter(f64(inp["X"]), f64(inp["dY"][l]), g) for l in range(L)]
    ref = gtp.deferred_finalize([[np.zeros((K // g, N)) for _ in range(g)] for _ in range(L)], st_ref)
    for l in range(L):
        for j in range(g):
            assert_fp32_close(f32(mg[l][j]), ref["main_grad"][l][j], f"main_grad[{l}][{j}]", rel=2e-5)


def test_trace_records_launches():
    K, N, g = 256, 64, 4
    sh = _shards(si.randn_bf16(si.generator(0), (K, N)), g)
    slot = torch.empty((K, N), device="cuda", dtype=torch.bfloat16)
    ttl.trace_enable(True, 64)
    ttl.gtp_gather(sh, slot)
    recs = ttl.trace_read(64)
    ttl.trace_enable(False)
    assert len(recs) == 1 and recs[0][0] == "gtp_gather" and recs[0][1] > 0 and recs[0][3] == 2 * K * N * 2


def test_finalize_is_one_fp32_add_and_the_finalize_stream_changes_no_bit():
    """Each main_grad element after the chain is exactly initial + staging in fp32 (one IEEE
    addition), and the chain with its deferred finalizes on a stream of their own, or with its
    weight gradients on a stream of their own too, gives the same bits as with everything on
    the compute stream."""
    from tensor_transformer_layer_way_gb300 import chain
    L, g, M, K, N = 3, 4, 256, 512, 320
    inp = si.gtp_inputs(L, K, N, M, seed=23)
    X = dev(inp["X"])
    dYs = dev(inp["dY"])
    shards = [_shards(w, g) for w in inp["W"]]
    slots = [torch.empty((K, N), device="cuda", dtype=torch.bfloat16) for _ in range(2)]
    mg0 = [[torch.randn((K // g, N), generator=si.generator(200 + l * g + j)) for j in range(g)] for l in range(L)]

    def run(fin, wgs=False):
        runner = chain.GtpChain(ttl, torch, shards, slots)
        mg = [[m.cuda() for m in layer] for layer in mg0]
        staging = [[torch.empty((K // g, N), device="cuda") for _ in range(g)] for _ in range(L)]
        dX = torch.empty((M, K), device="cuda", dtype=torch.bfloat16)
        runner.backward(X, dYs, dX, staging, mg, finalize_stream=fin, wgrad_stream=wgs)
        torch.cuda.synchronize()
        assert ttl.device_status() == 0
        return mg, staging, dX

    mg_a, st_a, dx_a = run(True)
    mg_b, st_b, dx_b = run(False)
    mg_c, st_c, dx_c = run(True, True)
    assert torch.equal(dx_a, dx_b) and torch.equal(dx_a, dx_c)
    for l in range(L):
        for j in range(g):
            expect = (mg0[l][j].numpy() + f32(st_a[l][j])).astype(np.float32)
            np.testing.assert_array_equal(f32(mg_a[l][j]).view(np.uint32), expect.view(np.uint32),
                                          err_msg=f"main_grad[{l}][{j}]")
            assert torch.equal(st_a[l][j], st_b[l][j])
            assert torch.equal(mg_a[l][j], mg_b[l][j]), f"finalize stream: main_grad[{l}][{j}]"
            assert torch.equal(st_a[l][j], st_c[l][j]) and torch.equal(mg_a[l][j], mg_c[l][j]), f"wgrad stream [{l}][{j}]"
    with pytest.raises(ttl.TTLError):
        ttl.gtp_finalize(st_a[0], st_a[0])       # staging and main_grad alias

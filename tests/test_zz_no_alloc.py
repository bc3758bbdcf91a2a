"""ttl_tp_mlp_bwd_static_ws, the MLP backward for callers that cannot allocate device memory
(e.g. a program whose device memory is all owned by another allocator, or a loop that must
not pay for cudaMalloc and its implicit device-wide synchronisation).  It uses the library's
built-in scratch array instead of a caller workspace, and must give what ttl_tp_mlp_bwd gives.

This file is collected last so that a run that stops at the first failure has already run
every other test; it also passes on its own in a fresh process (GPU)."""
import ctypes

import pytest
import torch

import synth_inputs as si
import tensor_transformer_layer_way_gb300 as ttl
from parity import assert_gemm_close, cols, dev, f64, rows

pytestmark = pytest.mark.gpu


def _case(act, t, T, h, f, seed):
    inp = si.mlp_inputs(T, h, f, act, seed)
    if act == "gelu_tanh":
        A, B, Au = dev(cols(inp["A"], t)), dev(rows(inp["B"], t)), None
    else:
        A, B, Au = dev(cols(inp["Wg"], t)), dev(rows(inp["Wd"], t)), dev(cols(inp["Wu"], t))
    X, dY = dev(inp["X"]), dev(inp["dY"])
    fwd = ttl.tp_mlp_fwd(X, A, B, act=act, A_up=Au)
    return X, dY, A, B, Au, fwd


def _compare(ref, got, act):
    keys = ["dA", "dB", "dX"] + (["dA_up"] if act == "swiglu" else [])
    for k in keys:
        for i, (r, g) in enumerate(zip(ref[k], got[k])):
            assert_gemm_close(f64(g), f64(r), f"{k}[{i}]")


def _dirty_scratch(act):
    """One call on a different, larger problem (the other activation, another seed, 2 MiB of
    scratch or more), so that the scratch holds values unrelated to the checked case."""
    other = "swiglu" if act == "gelu_tanh" else "gelu_tanh"
    t, T, h, f = 2, 512, 128, 2048
    X, dY, A, B, Au, fwd = _case(other, t, T, h, f, seed=77)
    out = ttl.mlp_bwd_buffers(t, other, T, h, f, X.device)
    ttl.tp_mlp_bwd_static_ws(X, dY, A, B, fwd, act=other, A_up=Au, out=out)
    torch.cuda.synchronize()
    assert ttl.device_status() == 0


@pytest.mark.parametrize("act,t,T,h,f", [("gelu_tanh", 2, 128, 256, 1024), ("swiglu", 4, 200, 136, 384)])
def test_static_scratch_matches_workspace_entry_point_twice(act, t, T, h, f):
    """Two checked calls in a row, each after a call on another problem has left different
    values in the scratch, so a read of a scratch element before this call writes it would
    show up as a mismatch."""
    X, dY, A, B, Au, fwd = _case(act, t, T, h, f, seed=31)
    ref = ttl.tp_mlp_bwd(X, dY, A, B, fwd, act=act, A_up=Au)
    for _ in range(2):
        _dirty_scratch(act)
        out = ttl.mlp_bwd_buffers(t, act, T, h, f, X.device)
        ttl.tp_mlp_bwd_static_ws(X, dY, A, B, fwd, act=act, A_up=Au, out=out)
        torch.cuda.synchronize()
        assert ttl.device_status() == 0
        _compare(ref, out, act)


def test_shape_beyond_the_scratch_is_rejected_before_running():
    t, T, h, f = 2, 8192, 64, 2048          # needs T*f*2 = 32 MiB of scratch
    assert ttl.tp_mlp_bwd_workspace_size(t, "gelu_tanh", T, h, f) > ttl.STATIC_WS_BYTES
    arr = (ctypes.c_void_p * t)(*[0x10000 * (i + 1) for i in range(t)])
    rc = ttl.lib().ttl_tp_mlp_bwd_static_ws(t, 0, T, h, f, 0x10000, 0x20000, arr, None, arr, arr, None, arr,
                                           arr, None, arr, None, None, arr, None)
    assert rc == ttl.TTL_ERR_UNSUPPORTED
    assert "built-in area" in ttl.last_error()

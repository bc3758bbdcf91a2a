"""ctypes binding over ``libttl.so``: argument marshalling only.

Every function here checks tensor dtypes/devices/shapes, turns tensors into device
pointers (and lists of tensors into host arrays of device pointers), passes the current
torch CUDA stream, and calls the C entry point of the same name.  All arithmetic runs in
the library's CUDA kernels; there is no Python or CPU fallback.  torch is used only for
device memory, streams and events.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libttl.so")

TTL_OK = 0
TTL_ERR_ARG = 1
TTL_ERR_SHAPE = 2
TTL_ERR_ALIGN = 3
TTL_ERR_CUDA = 4
TTL_ERR_TIMEOUT = 5
TTL_ERR_DEVICE = 6
TTL_ERR_UNSUPPORTED = 7
TTL_MAX_SHARDS = 16
ACT = {"gelu_tanh": 0, "swiglu": 1}
CE_FP32_DLOGITS = 1
CE_FORWARD_ONLY = 2

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int

# name -> (restype, argtypes); mirrors include/ttl.h
_SIGS = {
    "ttl_last_error": (ctypes.c_char_p, []),
    "ttl_version": (_int, []),
    "ttl_device_status": (_int, [_vp, ctypes.POINTER(_int)]),
    "ttl_selftest_wait_timeout": (_int, [_i64, _vp]),
    "ttl_trace_enable": (_int, [_int, _int]),
    "ttl_trace_read": (_int, [_int, ctypes.POINTER(_int), ctypes.POINTER(ctypes.c_float),
                              ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_int)]),
    "ttl_gemm": (_int, [_i64, _i64, _i64, _vp, _i64, _int, _vp, _i64, _int, _vp, _i64, _int, _vp]),
    "ttl_shard_reduce_scatter": (_int, [_int, _i64, _i64, _vp, _vp, _vp]),
    "ttl_shard_all_gather": (_int, [_int, _i64, _i64, _vp, _vp]),
    "ttl_shard_all_reduce": (_int, [_int, _i64, _i64, _vp, _vp, _vp]),
    "ttl_tp_mlp_fwd": (_int, [_int, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ttl_tp_mlp_bwd_workspace_size": (ctypes.c_size_t, [_int, _int, _i64, _i64, _i64]),
    "ttl_tp_mlp_bwd": (_int, [_int, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                              _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "ttl_tp_mlp_bwd_static_ws": (_int, [_int, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _vp, _vp, _vp, _vp, _vp, _vp]),
    "ttl_gtp_gather": (_int, [_int, _i64, _i64, _vp, _vp, _vp, _vp]),
    "ttl_gtp_gather_gemm": (_int, [_int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _int, _vp]),
    "ttl_gtp_wgrad_rs_finalize": (_int, [_int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _int, _vp, _vp]),
    "ttl_gtp_finalize": (_int, [_int, _i64, _i64, _vp, _vp, _vp]),
    "ttl_vocab_parallel_ce": (_int, [_int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                     ctypes.c_size_t, _int, _vp]),
    "ttl_vocab_parallel_ce_workspace_size": (ctypes.c_size_t, [_int, _i64, _i64, _i64]),
    "ttl_sp_mlp_fwd": (_int, [_int, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ttl_sp_mlp_bwd_workspace_size": (ctypes.c_size_t, [_int, _int, _i64, _i64, _i64]),
    "ttl_sp_mlp_bwd": (_int, [_int, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                              _vp, _vp, ctypes.c_size_t, _vp]),
    "ttl_vocab_parallel_embedding_fwd": (_int, [_int, _i64, _i64, _i64, _vp, _vp, _vp, _int, _vp]),
    "ttl_vocab_parallel_embedding_bwd": (_int, [_int, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "ttl_tp_attn_fwd_workspace_size": (ctypes.c_size_t, [_int, _i64, _int, _int, _int]),
    "ttl_tp_attn_fwd": (_int, [_int, _i64, _i64, _int, _int, _int] + [_vp] * 11 + [_vp, ctypes.c_size_t, _vp]),
    "ttl_tp_attn_bwd_workspace_size": (ctypes.c_size_t, [_int, _i64, _int, _int, _int]),
    "ttl_tp_attn_bwd": (_int, [_int, _i64, _i64, _int, _int, _int] + [_vp] * 16 + [_vp, ctypes.c_size_t, _vp]),
}

_lib = None


class TTLError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"ttl error {code}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                              "(python -m tensor_transformer_layer_way_gb300._build)")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def exported_symbols() -> list:
    return list(_SIGS)


def last_error() -> str:
    return lib().ttl_last_error().decode(errors="replace")


def _check(rc: int):
    if rc != TTL_OK:
        raise TTLError(rc, last_error())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _p(t):
    return None if t is None else t.data_ptr()


def _arr(ts):
    if ts is None:
        return None
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _need(t, name, dtype=torch.bfloat16, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _need_list(ts, name, n, dtype=torch.bfloat16, shape=None):
    if ts is None or len(ts) != n:
        raise ValueError(f"{name} must be a list of {n} tensors")
    for i, t in enumerate(ts):
        _need(t, f"{name}[{i}]", dtype, shape)
    return ts


# ------------------------------------------------------------------ housekeeping

def version() -> int:
    return lib().ttl_version()


def device_status(stream=None) -> int:
    """Synchronise the stream and read/clear the device status word (0 = no error)."""
    out = ctypes.c_int(0)
    _check(lib().ttl_device_status(_stream(stream), ctypes.byref(out)))
    return out.value


def selftest_wait_timeout(timeout_us: int, stream=None) -> int:
    """Runs the bounded-wait self test; returns the status code the kernel recorded."""
    return lib().ttl_selftest_wait_timeout(int(timeout_us), _stream(stream))


KERNEL_KINDS = ["gemm", "reduce", "gather", "gtp_gather", "finalize", "ce_stats", "ce_small", "ce_dlogits", "other",
                "embed", "softmax", "attn_core"]


def trace_enable(on: bool = True, capacity: int = 65536):
    """Bracket every library kernel launch with CUDA events (see ttl_trace_enable)."""
    _check(lib().ttl_trace_enable(int(on), int(capacity)))


def trace_read(max_records: int = 65536) -> list:
    """Per-launch records ``(kind, ms, flops, bytes)`` since tracing was enabled."""
    n = max(0, int(max_records))
    kind = (ctypes.c_int * max(n, 1))()
    ms = (ctypes.c_float * max(n, 1))()
    fl = (ctypes.c_double * max(n, 1))()
    by = (ctypes.c_double * max(n, 1))()
    cnt = ctypes.c_int(0)
    _check(lib().ttl_trace_read(n, kind, ms, fl, by, ctypes.byref(cnt)))
    return [(KERNEL_KINDS[kind[i]], float(ms[i]), float(fl[i]), float(by[i])) for i in range(min(n, cnt.value))]


# ------------------------------------------------------------------ GEMM core

def gemm(A, B, D, *, a_kmajor=True, b_kmajor=True, stream=None):
    """``D = op(A) op(B)``; A is [M,K] (a_kmajor) or [K,M]; B is [N,K] (b_kmajor) or [K,N]."""
    _need(A, "A")
    _need(B, "B")
    if D.dtype not in (torch.bfloat16, torch.float32) or not D.is_cuda or not D.is_contiguous():
        raise TypeError("D must be a contiguous CUDA bf16 or fp32 tensor")
    M, K = (A.shape[0], A.shape[1]) if a_kmajor else (A.shape[1], A.shape[0])
    N, Kb = (B.shape[0], B.shape[1]) if b_kmajor else (B.shape[1], B.shape[0])
    if K != Kb or tuple(D.shape) != (M, N):
        raise ValueError("gemm: inconsistent shapes")
    _check(lib().ttl_gemm(M, N, K, _p(A), A.shape[1], int(a_kmajor), _p(B), B.shape[1], int(b_kmajor),
                          _p(D), N, int(D.dtype == torch.float32), _stream(stream)))
    return D


# ------------------------------------------------------------------ partial-sum reduction

def _bufs(bufs):
    t = len(bufs)
    _need_list(bufs, "bufs", t, shape=bufs[0].shape)
    if bufs[0].dim() != 2:
        raise ValueError("buffers must be 2-D [rows, cols]")
    return t, bufs[0].shape[0], bufs[0].shape[1]


def shard_reduce_scatter(bufs, bias=None, stream=None):
    t, rows, cols = _bufs(bufs)
    if bias is not None:
        _need(bias, "bias", shape=(cols,))
    _check(lib().ttl_shard_reduce_scatter(t, rows, cols, _arr(bufs), _p(bias), _stream(stream)))
    return bufs


def shard_all_gather(bufs, stream=None):
    t, rows, cols = _bufs(bufs)
    _check(lib().ttl_shard_all_gather(t, rows, cols, _arr(bufs), _stream(stream)))
    return bufs


def shard_all_reduce(bufs, bias=None, stream=None):
    t, rows, cols = _bufs(bufs)
    if bias is not None:
        _need(bias, "bias", shape=(cols,))
    _check(lib().ttl_shard_all_reduce(t, rows, cols, _arr(bufs), _p(bias), _stream(stream)))
    return bufs


# ------------------------------------------------------------------ TP MLP block

def mlp_fwd_buffers(t, act, T, h, f, device="cuda"):
    """Allocates (with torch) the per-shard outputs tp_mlp_fwd writes."""
    fs = f // t
    e = dict(device=device, dtype=torch.bfloat16)
    out = {"U": [torch.empty(T, fs, **e) for _ in range(t)],
           "H": [torch.empty(T, fs, **e) for _ in range(t)],
           "Z": [torch.empty(T, h, **e) for _ in range(t)]}
    out["V"] = [torch.empty(T, fs, **e) for _ in range(t)] if act == "swiglu" else None
    return out


def tp_mlp_fwd(X, A, B, *, act="gelu_tanh", A_up=None, b1=None, b2=None, out=None, stream=None):
    """Forward of the TP MLP block over len(A) shards.  Returns dict U, V, H, Z (lists)."""
    t = len(A)
    T, h = X.shape
    fs = A[0].shape[1]
    f = fs * t
    _need(X, "X")
    _need_list(A, "A", t, shape=(h, fs))
    _need_list(B, "B", t, shape=(fs, h))
    if act == "swiglu":
        _need_list(A_up, "A_up", t, shape=(h, fs))
    if b1 is not None:
        _need_list(b1, "b1", t, shape=(fs,))
    if b2 is not None:
        _need(b2, "b2", shape=(h,))
    if out is None:
        out = mlp_fwd_buffers(t, act, T, h, f, X.device)
    _check(lib().ttl_tp_mlp_fwd(t, ACT[act], T, h, f, _p(X), _arr(A), _arr(A_up), _arr(B), _arr(b1), _p(b2),
                                _arr(out["U"]), _arr(out["V"]), _arr(out["H"]), _arr(out["Z"]), _stream(stream)))
    return out


def tp_mlp_bwd_workspace_size(t, act, T, h, f) -> int:
    return int(lib().ttl_tp_mlp_bwd_workspace_size(t, ACT[act], T, h, f))


def mlp_bwd_buffers(t, act, T, h, f, device="cuda", bias=False):
    fs = f // t
    e = dict(device=device, dtype=torch.bfloat16)
    out = {"dA": [torch.empty(h, fs, **e) for _ in range(t)],
           "dB": [torch.empty(fs, h, **e) for _ in range(t)],
           "dX": [torch.empty(T, h, **e) for _ in range(t)]}
    out["dA_up"] = [torch.empty(h, fs, **e) for _ in range(t)] if act == "swiglu" else None
    out["db1"] = [torch.empty(fs, **e) for _ in range(t)] if bias and act == "gelu_tanh" else None
    out["db2"] = torch.empty(h, **e) if bias else None
    ws = tp_mlp_bwd_workspace_size(t, act, T, h, f)
    out["ws"] = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
    return out


def tp_mlp_bwd(X, dY, A, B, fwd, *, act="gelu_tanh", A_up=None, out=None, bias=False, stream=None):
    """Backward of the TP MLP block.  ``fwd`` is the dict tp_mlp_fwd returned.
    Returns dict dA, dA_up, dB, db1, db2, dX (dX all-reduced in every buffer)."""
    t = len(A)
    T, h = X.shape
    fs = A[0].shape[1]
    f = fs * t
    _need(X, "X")
    _need(dY, "dY", shape=(T, h))
    if out is None:
        out = mlp_bwd_buffers(t, act, T, h, f, X.device, bias)
    ws = out["ws"]
    _check(lib().ttl_tp_mlp_bwd(t, ACT[act], T, h, f, _p(X), _p(dY), _arr(A), _arr(A_up), _arr(B), _arr(fwd["U"]),
                                _arr(fwd["V"]), _arr(fwd["H"]), _arr(out["dA"]), _arr(out["dA_up"]), _arr(out["dB"]),
                                _arr(out["db1"]), _p(out["db2"]), _arr(out["dX"]), _p(ws), ws.numel(),
                                _stream(stream)))
    return out


def sp_mlp_fwd(X_slabs, A, B, *, act="gelu_tanh", A_up=None, out=None, stream=None):
    """Sequence-parallel MLP forward: token slabs in ([T/t, h] each), token slabs out, the
    all-gather and reduce-scatter folded into the GEMMs.  Returns dict U, V, H, Z_slabs."""
    t = len(A)
    slab, h = X_slabs[0].shape
    T = slab * t
    fs = A[0].shape[1]
    f = fs * t
    _need_list(X_slabs, "X_slabs", t, shape=(slab, h))
    _need_list(A, "A", t, shape=(h, fs))
    _need_list(B, "B", t, shape=(fs, h))
    if act == "swiglu":
        _need_list(A_up, "A_up", t, shape=(h, fs))
    if out is None:
        out = mlp_fwd_buffers(t, act, T, h, f, X_slabs[0].device)
        del out["Z"]                      # SP writes only the t output slabs
        out["Z_slabs"] = [torch.empty((slab, h), device=X_slabs[0].device, dtype=torch.bfloat16) for _ in range(t)]
    _check(lib().ttl_sp_mlp_fwd(t, ACT[act], T, h, f, _arr(X_slabs), _arr(A), _arr(A_up), _arr(B), _arr(out["U"]),
                                _arr(out["V"]), _arr(out["H"]), _arr(out["Z_slabs"]), _stream(stream)))
    return out


def sp_mlp_bwd(X_slabs, dZ_slabs, A, B, fwd, *, act="gelu_tanh", A_up=None, out=None, stream=None):
    """Sequence-parallel MLP backward.  Returns dict dA, dA_up, dB, dX_slabs."""
    t = len(A)
    slab, h = X_slabs[0].shape
    T = slab * t
    fs = A[0].shape[1]
    f = fs * t
    _need_list(dZ_slabs, "dZ_slabs", t, shape=(slab, h))
    dev = X_slabs[0].device
    if out is None:
        e = dict(device=dev, dtype=torch.bfloat16)
        out = {"dA": [torch.empty(h, fs, **e) for _ in range(t)], "dB": [torch.empty(fs, h, **e) for _ in range(t)],
               "dA_up": [torch.empty(h, fs, **e) for _ in range(t)] if act == "swiglu" else None,
               "dX_slabs": [torch.empty(slab, h, **e) for _ in range(t)]}
        ws = int(lib().ttl_sp_mlp_bwd_workspace_size(t, ACT[act], T, h, f))
        out["ws"] = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
    ws = out["ws"]
    _check(lib().ttl_sp_mlp_bwd(t, ACT[act], T, h, f, _arr(X_slabs), _arr(dZ_slabs), _arr(A), _arr(A_up), _arr(B),
                                _arr(fwd["U"]), _arr(fwd["V"]), _arr(fwd["H"]), _arr(out["dA"]), _arr(out["dA_up"]),
                                _arr(out["dB"]), _arr(out["dX_slabs"]), _p(ws), ws.numel(), _stream(stream)))
    return out


# The size of the library's built-in scratch, TTL_STATIC_WS_BYTES in include/ttl.h (a CPU test
# checks that the two agree).
STATIC_WS_BYTES = 16 << 20


def tp_mlp_bwd_static_ws(X, dY, A, B, fwd, *, act="gelu_tanh", A_up=None, out, stream=None):
    """tp_mlp_bwd using the library's built-in 16 MiB scratch instead of a caller workspace,
    for callers that cannot allocate device memory.  ``out`` (dA, dA_up, dB, db1, db2, dX) must be
    provided.  Calls that overlap on the GPU share the scratch and race.  The call runs with
    X's device current, because the library takes the scratch of the current device."""
    t = len(A)
    T, h = X.shape
    f = A[0].shape[1] * t
    _need(X, "X")
    _need(dY, "dY", shape=(T, h))
    with torch.cuda.device(X.device):
        _check(lib().ttl_tp_mlp_bwd_static_ws(t, ACT[act], T, h, f, _p(X), _p(dY), _arr(A), _arr(A_up), _arr(B),
                                              _arr(fwd["U"]), _arr(fwd["V"]), _arr(fwd["H"]), _arr(out["dA"]),
                                              _arr(out["dA_up"]), _arr(out["dB"]), _arr(out["db1"]),
                                              _p(out["db2"]), _arr(out["dX"]), _stream(stream)))
    return out


# ------------------------------------------------------------------ GTP_remat

def gtp_gather(shards, slot, *, stream=None, done_event=None):
    """Gather g row shards [K/g, N] into slot [K, N]; records ``done_event`` (torch) after."""
    g = len(shards)
    Kg, N = shards[0].shape
    _need_list(shards, "shards", g, shape=(Kg, N))
    _need(slot, "slot", shape=(Kg * g, N))
    s = torch.cuda.current_stream() if stream is None else stream
    _check(lib().ttl_gtp_gather(g, Kg * g, N, _arr(shards), _p(slot), s.cuda_stream, None))
    if done_event is not None:
        done_event.record(s)
    return slot


def gtp_gather_gemm(X, shards, Y, *, slot=None, slot_ready=None, transpose_w=False, stream=None):
    """transpose_w False: Y[M,N] = X[M,K] W;  True: Y[M,K] = X[M,N] W^T.  W is the TP slice held
    as ``shards`` (g x [K/g, N]); with ``slot`` the gathered copy is read instead (after the
    stream waits on the torch event ``slot_ready``)."""
    g = len(shards)
    Kg, N = shards[0].shape
    K = Kg * g
    M = X.shape[0]
    _need(X, "X", shape=(M, N if transpose_w else K))
    _need(Y, "Y", shape=(M, K if transpose_w else N))
    if slot is None:
        _need_list(shards, "shards", g, shape=(Kg, N))
    else:
        _need(slot, "slot", shape=(K, N))
    s = torch.cuda.current_stream() if stream is None else stream
    if slot_ready is not None:
        s.wait_event(slot_ready)
    _check(lib().ttl_gtp_gather_gemm(g, M, K, N, _p(X), _arr(shards), _p(slot), None, _p(Y), int(transpose_w),
                                     s.cuda_stream))
    return Y


def gtp_wgrad_rs_finalize(X, dY, staging_cur, *, staging_prev=None, main_grad_prev=None, sync=False,
                          main_grad_cur=None, stream=None):
    g = len(staging_cur)
    M, K = X.shape
    N = dY.shape[1]
    _need(X, "X")
    _need(dY, "dY", shape=(M, N))
    _need_list(staging_cur, "staging_cur", g, torch.float32, (K // g, N))
    if staging_prev is not None:
        _need_list(staging_prev, "staging_prev", g, torch.float32, (K // g, N))
        _need_list(main_grad_prev, "main_grad_prev", g, torch.float32, (K // g, N))
    if sync:
        _need_list(main_grad_cur, "main_grad_cur", g, torch.float32, (K // g, N))
    _check(lib().ttl_gtp_wgrad_rs_finalize(g, M, K, N, _p(X), _p(dY), _arr(staging_cur), _arr(staging_prev),
                                           _arr(main_grad_prev), int(sync), _arr(main_grad_cur) if sync else None,
                                           _stream(stream)))


def gtp_finalize(staging, main_grad, *, stream=None):
    """main_grad[j] += staging[j] for the g fp32 shards [K/g, N] (on ``stream``, a torch stream)."""
    g = len(staging)
    Kg, N = staging[0].shape
    _need_list(staging, "staging", g, torch.float32, (Kg, N))
    _need_list(main_grad, "main_grad", g, torch.float32, (Kg, N))
    s = torch.cuda.current_stream() if stream is None else stream
    _check(lib().ttl_gtp_finalize(g, Kg * g, N, _arr(staging), _arr(main_grad), s.cuda_stream))


# ------------------------------------------------------------------ vocab-parallel CE

def ce_workspace_size(t, T, h, V) -> int:
    return int(lib().ttl_vocab_parallel_ce_workspace_size(t, T, h, V))


def ce_buffers(t, T, h, V, device="cuda", fused_stats=True):
    """Allocates (with torch) the CE outputs and, for fused statistics, its workspace."""
    Vs = V // t
    out = {"logits": [torch.empty(T, Vs, device=device, dtype=torch.float32) for _ in range(t)],
           "dlogits": [torch.empty(T, Vs, device=device, dtype=torch.bfloat16) for _ in range(t)],
           "stats": torch.empty((3 * t + 2) * T, device=device, dtype=torch.float32),
           "loss": torch.empty(1, device=device, dtype=torch.float32),
           "dH": torch.empty(T, h, device=device, dtype=torch.bfloat16), "ws": None}
    if fused_stats:
        out["ws"] = torch.empty(max(ce_workspace_size(t, T, h, V), 16), device=device, dtype=torch.uint8)
    return out


def vocab_parallel_ce(H, W, target, *, out=None, flags=0, fused_stats=True, stream=None):
    """Vocab-parallel LM head + CE over len(W) vocab shards (each [V/t, h]).  fused_stats: the
    LM-head GEMM epilogue computes the per-row statistics (needs the workspace ce_buffers
    allocates); otherwise a separate pass re-reads the logits.
    Returns dict logits, dlogits, stats, loss, dH (and ws)."""
    t = len(W)
    T, h = H.shape
    Vs = W[0].shape[0]
    V = Vs * t
    _need(H, "H")
    _need_list(W, "W", t, shape=(Vs, h))
    _need(target, "target", torch.int64, (T,))
    if out is None:
        out = ce_buffers(t, T, h, V, H.device, fused_stats)
    fwd_only = bool(flags & CE_FORWARD_ONLY)
    ws = out.get("ws") if fused_stats else None
    _check(lib().ttl_vocab_parallel_ce(t, T, h, V, _p(H), _arr(W), _p(target), _arr(out["logits"]),
                                       None if fwd_only else _arr(out["dlogits"]), _p(out["stats"]),
                                       _p(out["loss"]), None if fwd_only else _p(out["dH"]), _p(ws),
                                       0 if ws is None else ws.numel(), int(flags), _stream(stream)))
    return out


# ------------------------------------------------------------------ vocab-parallel embedding

def vocab_parallel_embedding_fwd(ids, E, *, out=None, literal=True, stream=None):
    """Lookup with the table split into len(E) vocab shards ([V/t, h] each).  Returns the t
    output buffers [T, h], each holding every token's row (literal: masked lookups + the
    all-reduce; otherwise one fused gather pass with the same bits)."""
    t = len(E)
    Vs, h = E[0].shape
    T = ids.shape[0]
    _need(ids, "ids", torch.int64, (T,))
    _need_list(E, "E", t, shape=(Vs, h))
    if out is None:
        out = [torch.empty((T, h), device=ids.device, dtype=torch.bfloat16) for _ in range(t)]
    _need_list(out, "out", t, shape=(T, h))
    _check(lib().ttl_vocab_parallel_embedding_fwd(t, T, h, Vs * t, _p(ids), _arr(E), _arr(out), int(bool(literal)),
                                                  _stream(stream)))
    return out


def vocab_parallel_embedding_bwd(ids, dY, dE, *, stream=None):
    """Accumulates dY rows into the owning shard's fp32 gradient dE[i] ([V/t, h])."""
    t = len(dE)
    Vs, h = dE[0].shape
    T = ids.shape[0]
    _need(ids, "ids", torch.int64, (T,))
    _need(dY, "dY", shape=(T, h))
    _need_list(dE, "dE", t, torch.float32, (Vs, h))
    _check(lib().ttl_vocab_parallel_embedding_bwd(t, T, h, Vs * t, _p(ids), _p(dY), _arr(dE), _stream(stream)))
    return dE


# ------------------------------------------------------------------ TP attention block

def attn_fwd_buffers(t, T, h, n_q, n_kv, d, device="cuda"):
    """Output, saved-activation and workspace buffers of tp_attn_fwd."""
    qc, kc = n_q // t * d, n_kv // t * d
    e = dict(device=device, dtype=torch.bfloat16)
    out = {"Q": [torch.empty(T, qc, **e) for _ in range(t)], "K": [torch.empty(T, kc, **e) for _ in range(t)],
           "V": [torch.empty(T, kc, **e) for _ in range(t)], "O": [torch.empty(T, qc, **e) for _ in range(t)],
           "P": [torch.empty(n_q // t, T, T, **e) for _ in range(t)], "Y": [torch.empty(T, h, **e) for _ in range(t)]}
    ws = int(lib().ttl_tp_attn_fwd_workspace_size(t, T, n_q, n_kv, d))
    out["ws"] = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
    return out


def tp_attn_fwd(X, Wq, Wk, Wv, Wo, *, n_q, n_kv, d, out=None, stream=None):
    """Forward of the head-split attention block over len(Wq) shards.
    Returns dict Q, K, V, P, O (saved per shard) and Y (all-reduced in every buffer)."""
    t = len(Wq)
    T, h = X.shape
    qc, kc = n_q // t * d, n_kv // t * d
    _need(X, "X")
    _need_list(Wq, "Wq", t, shape=(h, qc))
    _need_list(Wk, "Wk", t, shape=(h, kc))
    _need_list(Wv, "Wv", t, shape=(h, kc))
    _need_list(Wo, "Wo", t, shape=(qc, h))
    if out is None:
        out = attn_fwd_buffers(t, T, h, n_q, n_kv, d, X.device)
    ws = out["ws"]
    _check(lib().ttl_tp_attn_fwd(t, T, h, n_q, n_kv, d, _p(X), _arr(Wq), _arr(Wk), _arr(Wv), _arr(Wo),
                                 _arr(out["Q"]), _arr(out["K"]), _arr(out["V"]), _arr(out["P"]), _arr(out["O"]),
                                 _arr(out["Y"]), _p(ws), ws.numel(), _stream(stream)))
    return out


def attn_bwd_buffers(t, T, h, n_q, n_kv, d, device="cuda"):
    qc, kc = n_q // t * d, n_kv // t * d
    e = dict(device=device, dtype=torch.bfloat16)
    out = {"dWq": [torch.empty(h, qc, **e) for _ in range(t)], "dWk": [torch.empty(h, kc, **e) for _ in range(t)],
           "dWv": [torch.empty(h, kc, **e) for _ in range(t)], "dWo": [torch.empty(qc, h, **e) for _ in range(t)],
           "dX": [torch.empty(T, h, **e) for _ in range(t)]}
    ws = int(lib().ttl_tp_attn_bwd_workspace_size(t, T, n_q, n_kv, d))
    out["ws"] = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
    return out


def tp_attn_bwd(X, dY, Wq, Wk, Wv, Wo, fwd, *, n_q, n_kv, d, out=None, stream=None):
    """Backward of tp_attn_fwd (``fwd`` is the dict it returned).
    Returns dict dWq, dWk, dWv, dWo and dX (all-reduced in every buffer)."""
    t = len(Wq)
    T, h = X.shape
    _need(X, "X")
    _need(dY, "dY", shape=(T, h))
    if out is None:
        out = attn_bwd_buffers(t, T, h, n_q, n_kv, d, X.device)
    ws = out["ws"]
    _check(lib().ttl_tp_attn_bwd(t, T, h, n_q, n_kv, d, _p(X), _p(dY), _arr(Wq), _arr(Wk), _arr(Wv), _arr(Wo),
                                 _arr(fwd["Q"]), _arr(fwd["K"]), _arr(fwd["V"]), _arr(fwd["P"]), _arr(fwd["O"]),
                                 _arr(out["dWq"]), _arr(out["dWk"]), _arr(out["dWv"]), _arr(out["dWo"]),
                                 _arr(out["dX"]), _p(ws), ws.numel(), _stream(stream)))
    return out

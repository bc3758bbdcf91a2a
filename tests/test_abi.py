"""The C ABI library builds, loads and exports every declared symbol; host-side argument
validation returns the documented status codes before anything touches a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import __graft_entry__ as entry

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    entry.build()
    import tensor_transformer_layer_way_gb300 as ttl
    return ttl.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "ttl.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ttl_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    import tensor_transformer_layer_way_gb300 as ttl
    declared = _declared()
    assert len(declared) >= 15
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(ttl.exported_symbols()) == declared


def test_version_and_error_text(lib):
    assert lib.ttl_version() == 100
    assert isinstance(lib.ttl_last_error(), bytes)


P = ctypes.c_void_p


def _arr(*vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def test_reduce_validation(lib):
    A16, B16 = 0x10000, 0x20000
    assert lib.ttl_shard_all_reduce(0, 8, 8, _arr(A16), None, None) == 1          # t < 1
    assert lib.ttl_shard_all_reduce(17, 8, 8, _arr(A16), None, None) == 1         # t > 16
    assert lib.ttl_shard_all_reduce(2, 8, 8, None, None, None) == 1               # null array
    assert lib.ttl_shard_all_reduce(2, 8, 8, _arr(A16, None), None, None) == 1    # null buffer
    assert lib.ttl_shard_all_reduce(2, 8, 12, _arr(A16, B16), None, None) == 2    # cols % 8
    assert lib.ttl_shard_reduce_scatter(3, 8, 8, _arr(A16, B16, 0x30000), None, None) == 2  # t does not divide rows
    assert lib.ttl_shard_all_gather(2, 8, 8, _arr(A16, B16 + 2), None) == 3       # misaligned
    assert lib.ttl_shard_all_reduce(2, 8, 8, _arr(A16, A16), None, None) == 1     # aliasing buffers
    assert b"alias" in lib.ttl_last_error()
    assert lib.ttl_shard_all_reduce(2, -1, 8, _arr(A16, B16), None, None) == 1    # negative
    assert lib.ttl_shard_all_reduce(2, 0, 8, _arr(A16, B16), None, None) == 0     # empty: no-op, no GPU needed


def test_mlp_validation(lib):
    X = 0x10000
    sh = _arr(0x20000, 0x30000)
    args = [None] * 10
    # t does not divide f
    assert lib.ttl_tp_mlp_fwd(3, 0, 16, 64, 128, X, _arr(1, 2, 3), None, _arr(1, 2, 3), None, None,
                              _arr(1, 2, 3), None, _arr(1, 2, 3), _arr(1, 2, 3), None) == 2
    # unknown activation
    assert lib.ttl_tp_mlp_fwd(2, 7, 16, 64, 128, X, sh, None, sh, None, None, sh, None, sh, sh, None) == 1
    # SwiGLU without the up weights
    assert lib.ttl_tp_mlp_fwd(2, 1, 16, 64, 128, X, sh, None, sh, None, None, sh, sh, sh, sh, None) == 1
    # misaligned X
    assert lib.ttl_tp_mlp_fwd(2, 0, 16, 64, 128, X + 4, sh, None, sh, None, None, sh, None, sh, sh, None) == 3
    # f/t not a multiple of 8
    assert lib.ttl_tp_mlp_fwd(2, 0, 16, 64, 12, X, sh, None, sh, None, None, sh, None, sh, sh, None) == 2
    # zero tokens: nothing to do
    assert lib.ttl_tp_mlp_fwd(2, 0, 0, 64, 128, X, sh, None, sh, None, None, sh, None, sh, sh, None) == 0
    del args
    assert lib.ttl_tp_mlp_bwd_workspace_size(2, 0, 16, 64, 128) == 2 * 256 * ((16 * 64 * 2 + 255) // 256)
    assert lib.ttl_tp_mlp_bwd_workspace_size(2, 1, 16, 64, 128) == 2 * lib.ttl_tp_mlp_bwd_workspace_size(2, 0, 16, 64, 128)
    # workspace too small
    assert lib.ttl_tp_mlp_bwd(2, 0, 16, 64, 128, X, X, sh, None, sh, sh, None, sh, sh, None, sh, None, None, sh,
                              0x40000, 16, None) == 1


def test_gtp_and_ce_validation(lib):
    sh = _arr(*[0x10000 * (i + 1) for i in range(8)])
    assert lib.ttl_gtp_gather(0, 64, 64, sh, 0x90000, None, None) == 1            # g < 1
    assert lib.ttl_gtp_gather(8, 60, 64, sh, 0x90000, None, None) == 2            # g does not divide K
    assert lib.ttl_gtp_gather(8, 64 * 8, 64, sh, 0x90008, None, None) == 3        # misaligned slot
    assert lib.ttl_gtp_gather_gemm(8, 16, 512, 64, 0x90000, sh, None, None, 0xA0000, 2, None) == 1
    assert lib.ttl_gtp_wgrad_rs_finalize(8, 16, 512, 64, 0x90000, 0xA0000, sh, sh, None, 0, None, None) == 1
    assert lib.ttl_gtp_finalize(0, 512, 64, sh, sh, None) == 1                    # g < 1
    assert lib.ttl_gtp_finalize(8, 60, 64, sh, sh, None) == 2                     # g does not divide K
    assert lib.ttl_gtp_finalize(8, 512, 64, sh, None, None) == 1                  # null main_grad
    assert lib.ttl_gtp_finalize(8, 512, 64, sh, sh, None) == 1                    # staging aliases main_grad
    W = _arr(0x10000, 0x20000)
    L = _arr(0x30000, 0x40000)
    # t does not divide V
    assert lib.ttl_vocab_parallel_ce(2, 8, 64, 33, 0x90000, W, 0xA0000, L, L, 0xB0000, 0xC0000, 0xD0000,
                                     None, 0, 0, None) == 2
    # unknown flag
    assert lib.ttl_vocab_parallel_ce(2, 8, 64, 32, 0x90000, W, 0xA0000, L, L, 0xB0000, 0xC0000, 0xD0000,
                                     None, 0, 8, None) == 1
    # workspace too small for the fused statistics
    need = lib.ttl_vocab_parallel_ce_workspace_size(2, 8, 64, 32)
    # 8 tokens x 2 shards x 2 half tiles x 8 bytes (256), 8 target logits (32 -> 256), a counter (256)
    assert need == 256 + 256 + 256
    assert lib.ttl_vocab_parallel_ce(2, 8, 64, 32, 0x90000, W, 0xA0000, L, L, 0xB0000, 0xC0000, 0xD0000,
                                     0xE0000, need - 1, 0, None) == 1
    # embedding: t does not divide V, misaligned ids
    assert lib.ttl_vocab_parallel_embedding_fwd(2, 8, 64, 33, 0x10000, W, L, 1, None) == 2
    assert lib.ttl_vocab_parallel_embedding_fwd(2, 8, 64, 32, 0x10004, W, L, 1, None) == 3
    assert lib.ttl_vocab_parallel_embedding_bwd(2, 8, 64, 32, 0x10000, 0x20000, None, None) == 1
    # zero tokens would write the loss with a device copy: not on a CPU host, so only shape checks here
    assert lib.ttl_gemm(8, 12, 16, 0x10000, 16, 1, 0x20000, 16, 1, 0x30000, 12, 0, None) == 2


def test_attention_validation(lib):
    sh = _arr(0x10000, 0x20000)
    X, ws = 0x90000, 0xA0000
    fwd = lib.ttl_tp_attn_fwd
    ten = [sh] * 10   # Wq Wk Wv Wo Q K V P O Y

    def call(t, T, h, nq, nkv, d, x=X, arrs=ten, w=ws, wb=1 << 40):
        return fwd(t, T, h, nq, nkv, d, x, *arrs, w, wb, None)
    assert call(3, 64, 64, 32, 8, 128) == 2          # t does not divide the head counts
    assert call(2, 64, 64, 8, 3, 128) == 2           # t does not divide n_kv
    assert call(2, 64, 64, 6, 4, 128) == 2           # n_kv does not divide n_q
    assert call(2, 64, 64, 8, 2, 96) == 2            # head dimension not 64 or 128
    assert call(2, 64, 64, 8, 2, 256) == 2
    assert call(2, 60, 64, 8, 2, 128) == 2           # T not a multiple of 8
    assert call(2, 64, 64, 8, 2, 128, x=X + 2) == 3  # misaligned X
    assert call(2, 64, 64, 8, 2, 128, arrs=[sh] * 9 + [None]) == 1   # Y missing
    assert call(2, 0, 64, 8, 2, 128) == 0            # no tokens: nothing to do
    # the fused forward keeps scores and statistics on chip
    assert lib.ttl_tp_attn_fwd_workspace_size(2, 64, 8, 2, 128) == 0
    # D per row (fp32), then per shard dO, dQ [64, 512], dK, dV [64, 128]
    per = 2 * (64 * 512 * 2) + 2 * (64 * 128 * 2)
    assert lib.ttl_tp_attn_bwd_workspace_size(2, 64, 8, 2, 128) == 512 * 4 + 2 * per
    assert lib.ttl_tp_attn_bwd_workspace_size(3, 64, 8, 2, 128) == 0    # invalid shape
    bwd = lib.ttl_tp_attn_bwd
    assert bwd(2, 64, 64, 8, 2, 128, X, X, *([sh] * 9), sh, sh, sh, None, sh, ws, 1 << 40, None) == 1  # dWo missing
    assert bwd(2, 64, 64, 8, 2, 128, X, X, *([sh] * 9), sh, sh, sh, sh, sh, ws, 16, None) == 1         # workspace


def test_selftest_bounds(lib):
    assert lib.ttl_selftest_wait_timeout(0, None) == 1
    assert lib.ttl_selftest_wait_timeout(2_000_000, None) == 1


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import tensor_transformer_layer_way_gb300._binding as b
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(b, "_lib", None)
    with pytest.raises(ImportError):
        b.lib()


def test_every_declaration_is_documented():
    # Each entry point carries the contract right above it: a comment block (its own, or its
    # section's when declarations share one) with nothing but blank lines between them.
    lines = open(os.path.join(ROOT, "include", "ttl.h")).read().splitlines()
    for i, line in enumerate(lines):
        m = re.match(r"^(?:int|size_t|const char\*)\s+(ttl_[a-z0-9_]+)\s*\(", line)
        if not m:
            continue
        j = i - 1
        # blank lines, and the lines of declarations grouped under the same comment
        while j >= 0 and (not lines[j].strip() or not lines[j].lstrip().startswith(("/*", "*", "#", "}"))
                          and not lines[j].rstrip().endswith("*/")):
            j -= 1
        assert j >= 0 and lines[j].rstrip().endswith("*/"), f"{m.group(1)} has no comment block above it"


def test_static_scratch_size_matches_the_header():
    import re
    import tensor_transformer_layer_way_gb300 as ttl
    hdr = open(os.path.join(ROOT, "include", "ttl.h")).read()
    m = re.search(r"#define\s+TTL_STATIC_WS_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", hdr)
    assert m, "TTL_STATIC_WS_BYTES not found in include/ttl.h"
    assert ttl.STATIC_WS_BYTES == int(m.group(1)) << int(m.group(2))


def test_package_exports_every_binding_of_a_library_call():
    """Each Python wrapper named after a C entry point (the name minus ``ttl_``) is reachable
    from the package itself."""
    import tensor_transformer_layer_way_gb300 as pkg
    from tensor_transformer_layer_way_gb300 import _binding
    hdr = open(os.path.join(ROOT, "include", "ttl.h")).read()
    import re
    for name in re.findall(r"\bttl_([a-z0-9_]+)\s*\(", hdr):
        if hasattr(_binding, name) and callable(getattr(_binding, name)):
            assert hasattr(pkg, name), f"{name} is not exported by the package"

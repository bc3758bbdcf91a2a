"""GB300-native tensor-parallel transformer-block math (sm_103a).

The t tensor-parallel shards of the method are t device buffers on one GPU; the hot path
(column/row-parallel GEMMs with fused activations, the partial-sum all-reduce, the GTP_remat
weight path, vocab-parallel cross-entropy and embedding, the head-split attention block) runs
in the hand-written CUDA kernels of ``_lib/libttl.so`` behind the C ABI in ``include/ttl.h``.
This package is the thin Python binding over that ABI.
"""
from ._binding import (  # noqa: F401
    ACT, CE_FORWARD_ONLY, attn_bwd_buffers, attn_fwd_buffers, CE_FP32_DLOGITS, LIB_PATH, STATIC_WS_BYTES, TTL_ERR_ALIGN, TTL_ERR_ARG, TTL_ERR_CUDA, TTL_ERR_DEVICE,
    TTL_ERR_SHAPE, TTL_ERR_TIMEOUT, TTL_ERR_UNSUPPORTED, TTL_MAX_SHARDS, TTL_OK, TTLError, ce_buffers, device_status,
    exported_symbols, gemm, gtp_finalize, gtp_gather, gtp_gather_gemm, gtp_wgrad_rs_finalize, last_error, lib, mlp_bwd_buffers,
    mlp_fwd_buffers, selftest_wait_timeout, sp_mlp_bwd, sp_mlp_fwd, shard_all_gather, shard_all_reduce, shard_reduce_scatter, tp_mlp_bwd,
    tp_attn_bwd, tp_attn_fwd, tp_mlp_bwd_static_ws, tp_mlp_bwd_workspace_size, tp_mlp_fwd, trace_enable, trace_read, version,
    vocab_parallel_ce, vocab_parallel_embedding_bwd, vocab_parallel_embedding_fwd)

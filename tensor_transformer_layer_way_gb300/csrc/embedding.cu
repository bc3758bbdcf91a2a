// Vocab-parallel embedding lookup (forward and backward) on t logical vocab shards of one GPU.
//
// Source: "v4:Tensor Parallel 与 Sequence Parallel", section "Embedding 和 LM head:按 vocab
// 切": the table is split by vocabulary rows (shard i owns ids [i V/t, (i+1) V/t)); a shard
// outputs 0 for tokens whose id it does not own, and an all-reduce of the t outputs gives
// every token exactly its own row.
//
// Forward, two ways with the same bits:
//   literal: each shard writes its masked lookup (owned row or zeros) into its buffer, then
//            the on-device all-reduce sums the t buffers (one nonzero term per element);
//   fused:   one pass reads each token's row from the owning shard and writes it into all t
//            buffers -- the all-reduce's result without its (2t+1) S of traffic.
// Backward: the all-reduce's backward is the identity, so each shard accumulates, for every
// token it owns, that token's gradient row into its fp32 table gradient (vector atomics).
// All kernels are HBM streams over 16-byte vectors, one CTA per token row.

#include "ttl_device.cuh"
#include "ttl_internal.h"

namespace ttl {

struct EmbedTables {
  const uint4* e[kMaxShards];
};

struct EmbedOut {
  uint4* o[kMaxShards];
};

struct EmbedGrad {
  float4* g[kMaxShards];
};

// grid (T, t): shard i's masked lookup for token `tok` (h8 = h / 8 vectors per row).
__global__ void __launch_bounds__(256) embed_partial_kernel(const __grid_constant__ EmbedTables E,
                                                            const __grid_constant__ EmbedOut O, const int64_t* ids,
                                                            int64_t h8, int64_t Vs, int64_t V, int* status) {
  const int64_t tok = blockIdx.x;
  const int i = blockIdx.y;
  const int64_t id = ids[tok];
  if ((id < 0 || id >= V) && i == 0 && threadIdx.x == 0) atomicCAS(status, 0, TTL_ERR_DEVICE);
  const int64_t local = id - static_cast<int64_t>(i) * Vs;
  const bool own = id >= 0 && id < V && local >= 0 && local < Vs;
  uint4* dst = O.o[i] + tok * h8;
  const uint4* src = own ? E.e[i] + local * h8 : nullptr;
  for (int64_t k = threadIdx.x; k < h8; k += blockDim.x) dst[k] = own ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
}

// grid T: token `tok`'s row from its owning shard into every output buffer.
__global__ void __launch_bounds__(256) embed_gather_kernel(const __grid_constant__ EmbedTables E,
                                                           const __grid_constant__ EmbedOut O, const int64_t* ids,
                                                           int t, int64_t h8, int64_t Vs, int64_t V, int* status) {
  const int64_t tok = blockIdx.x;
  const int64_t id = ids[tok];
  const bool valid = id >= 0 && id < V;
  if (!valid && threadIdx.x == 0) atomicCAS(status, 0, TTL_ERR_DEVICE);
  const int owner = valid ? static_cast<int>(id / Vs) : 0;
  const uint4* src = E.e[owner] + (valid ? (id - owner * Vs) : 0) * h8;
  for (int64_t k = threadIdx.x; k < h8; k += blockDim.x) {
    const uint4 v = valid ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
    for (int j = 0; j < t; ++j) __stcs(O.o[j] + tok * h8 + k, v);
  }
}

// grid T: dE_owner[id - owner V/t] += dY[tok] (fp32, 4-wide vector atomics).
__global__ void __launch_bounds__(256) embed_grad_kernel(const __grid_constant__ EmbedGrad G, const int64_t* ids,
                                                         const uint4* dY, int64_t h8, int64_t Vs, int64_t V,
                                                         int* status) {
  const int64_t tok = blockIdx.x;
  const int64_t id = ids[tok];
  if (id < 0 || id >= V) {
    if (threadIdx.x == 0) atomicCAS(status, 0, TTL_ERR_DEVICE);
    return;
  }
  const int owner = static_cast<int>(id / Vs);
  float4* dst = G.g[owner] + (id - owner * Vs) * h8 * 2;
  for (int64_t k = threadIdx.x; k < h8; k += blockDim.x) {
    const uint4 v = __ldcs(dY + tok * h8 + k);
    atomicAdd(dst + 2 * k, make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y)));
    atomicAdd(dst + 2 * k + 1, make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)));
  }
}

namespace {

int check_common(int t, int64_t T, int64_t h, int64_t V, const int64_t* ids, const char* name) {
  if (t < 1 || t > kMaxShards) return set_error(TTL_ERR_ARG, "%s: t=%d outside [1,%d]", name, t, kMaxShards);
  if (T < 0 || h < 0 || V < 0) return set_error(TTL_ERR_ARG, "%s: negative shape", name);
  if (V % t) return set_error(TTL_ERR_SHAPE, "%s: t=%d must divide V=%lld", name, t, (long long)V);
  if (h % 8) return set_error(TTL_ERR_SHAPE, "%s: h must be a multiple of 8", name);
  if (T > 0 && !ids) return set_error(TTL_ERR_ARG, "%s: ids is null", name);
  if (ids && (reinterpret_cast<uintptr_t>(ids) & 7)) return set_error(TTL_ERR_ALIGN, "%s: ids not 8-byte aligned", name);
  if (T >= (int64_t(1) << 31)) return set_error(TTL_ERR_SHAPE, "%s: T beyond 2^31", name);
  return TTL_OK;
}

int check_array(const void* const* a, int t, const char* what) {
  if (!a) return set_error(TTL_ERR_ARG, "%s: null shard array", what);
  for (int i = 0; i < t; ++i) {
    if (!a[i]) return set_error(TTL_ERR_ARG, "%s[%d] is null", what, i);
    if (!aligned16(a[i])) return set_error(TTL_ERR_ALIGN, "%s[%d] not 16-byte aligned", what, i);
  }
  return TTL_OK;
}

}  // namespace
}  // namespace ttl

using namespace ttl;

extern "C" int ttl_vocab_parallel_embedding_fwd(int t, int64_t T, int64_t h, int64_t V, const int64_t* ids,
                                                const ttl_bf16* const* E, ttl_bf16* const* out, int literal,
                                                void* stream) {
  const char* name = "ttl_vocab_parallel_embedding_fwd";
  int rc = check_common(t, T, h, V, ids, name);
  if (rc) return rc;
  if (literal != 0 && literal != 1) return set_error(TTL_ERR_ARG, "%s: literal must be 0 or 1", name);
  if (T == 0 || h == 0) return TTL_OK;
  if (V == 0) return set_error(TTL_ERR_SHAPE, "%s: empty vocabulary", name);
  if ((rc = check_array(reinterpret_cast<const void* const*>(E), t, "E"))) return rc;
  if ((rc = check_array(reinterpret_cast<const void* const*>(out), t, "out"))) return rc;
  if ((rc = require_sm103())) return rc;
  int* status = device_status_ptr();
  if (!status) return TTL_ERR_CUDA;
  EmbedTables tab;
  EmbedOut o;
  for (int i = 0; i < kMaxShards; ++i) {
    tab.e[i] = i < t ? reinterpret_cast<const uint4*>(E[i]) : nullptr;
    o.o[i] = i < t ? reinterpret_cast<uint4*>(out[i]) : nullptr;
  }
  const int64_t Vs = V / t;
  const int64_t h8 = h / 8;
  const int threads = h8 >= 256 ? 256 : static_cast<int>((h8 + 31) / 32 * 32);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const double row_bytes = static_cast<double>(h) * 2.0;
  if (!literal) {
    TraceScope trace(s, TTL_K_EMBED, 0.0, static_cast<double>(T) * row_bytes * (1.0 + t));
    embed_gather_kernel<<<static_cast<unsigned>(T), threads, 0, s>>>(tab, o, ids, t, h8, Vs, V, status);
    return cuda_check(cudaGetLastError(), "embed_gather_kernel launch");
  }
  {
    TraceScope trace(s, TTL_K_EMBED, 0.0, static_cast<double>(T) * row_bytes * (1.0 + t));
    embed_partial_kernel<<<dim3(static_cast<unsigned>(T), t), threads, 0, s>>>(tab, o, ids, h8, Vs, V, status);
    if ((rc = cuda_check(cudaGetLastError(), "embed_partial_kernel launch"))) return rc;
  }
  // g: the all-reduce of the t masked lookups.
  return shard_all_reduce_internal(t, T, h, out, nullptr, s);
}

extern "C" int ttl_vocab_parallel_embedding_bwd(int t, int64_t T, int64_t h, int64_t V, const int64_t* ids,
                                                const ttl_bf16* dY, float* const* dE, void* stream) {
  const char* name = "ttl_vocab_parallel_embedding_bwd";
  int rc = check_common(t, T, h, V, ids, name);
  if (rc) return rc;
  if (T == 0 || h == 0) return TTL_OK;
  if (V == 0) return set_error(TTL_ERR_SHAPE, "%s: empty vocabulary", name);
  if (!dY) return set_error(TTL_ERR_ARG, "%s: dY is null", name);
  if (!aligned16(dY)) return set_error(TTL_ERR_ALIGN, "%s: dY not 16-byte aligned", name);
  if ((rc = check_array(reinterpret_cast<const void* const*>(dE), t, "dE"))) return rc;
  if ((rc = require_sm103())) return rc;
  int* status = device_status_ptr();
  if (!status) return TTL_ERR_CUDA;
  EmbedGrad G;
  for (int i = 0; i < kMaxShards; ++i) G.g[i] = i < t ? reinterpret_cast<float4*>(dE[i]) : nullptr;
  const int64_t h8 = h / 8;
  const int threads = h8 >= 256 ? 256 : static_cast<int>((h8 + 31) / 32 * 32);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  TraceScope trace(s, TTL_K_EMBED, 0.0, static_cast<double>(T) * h * (2.0 + 8.0));
  embed_grad_kernel<<<static_cast<unsigned>(T), threads, 0, s>>>(G, ids, reinterpret_cast<const uint4*>(dY), h8,
                                                                 V / t, V, status);
  return cuda_check(cudaGetLastError(), "embed_grad_kernel launch");
}

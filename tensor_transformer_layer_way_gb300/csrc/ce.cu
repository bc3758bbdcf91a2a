// Vocab-parallel LM head + cross-entropy on t logical vocab shards of one GPU.
//
// Source: "v4:Tensor Parallel 与 Sequence Parallel", section "Embedding 和 LM head:按 vocab
// 切": the LM head is column-parallel over the vocabulary (shard i owns ids
// [i V/t, (i+1) V/t)); the loss never gathers the logits -- each token combines only three
// numbers across shards: the max, the sum of exponentials and the target logit.
//
// Steps (one launch each):
//   1. logits   Z_i = H W_i^T, fp32, all shards in one grouped tcgen05 GEMM
//   2. stats    per (token, shard) row: m_i = max, s_i = sum exp(z - m_i), y_i = target logit
//               (one CTA per row, float4 loads, online max/sum, warp-shuffle reductions)
//   3. combine  per token: M = max m_i, S = sum s_i exp(m_i - M), lse = M + log S,
//               loss_t = lse - sum y_i
//   4. mean     loss = mean_t loss_t (one CTA, fixed order, fp64 partials)
//   With a workspace, step 1's epilogue leaves per-tile (max, sum exp) partials, and steps 2-4
//   are one launch: a CTA per token merges every shard's partials (a warp per shard), combines
//   the shards, and the last CTA to finish takes the mean.
//   5. dlogits  dZ_i = (exp(z - lse) - [v == target]) / T -> bf16 (and fp32 in place if asked)
//   6. dH       sum_i dZ_i W_i as ONE GEMM whose K loop walks the t shards in order, so the
//               f-backward reduction of the column-parallel head happens in the accumulator.

#include <math.h>

#include "ttl_device.cuh"
#include "ttl_internal.h"

namespace ttl {

struct CeShards {
  const float* z[kMaxShards];
};

__device__ __forceinline__ void online_update(float& m, float& s, float x) {
  if (x > m) {
    s = s * __expf(m - x) + 1.0f;
    m = x;
  } else {
    s += __expf(x - m);
  }
}

__device__ __forceinline__ void online_merge(float& m, float& s, float m2, float s2) {
  if (m2 > m) {
    s = s * __expf(m - m2) + s2;
    m = m2;
  } else if (m2 > -INFINITY) {
    s += s2 * __expf(m2 - m);
  }
}

// grid (T, t), 256 threads: row `tok` of shard `i`.
__global__ void __launch_bounds__(256) ce_stats_kernel(const __grid_constant__ CeShards S, const int64_t* target, int64_t T, int64_t Vs,
                                                       float* stats) {
  const int64_t tok = blockIdx.x;
  const int i = blockIdx.y;
  const float* row = S.z[i] + tok * Vs;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  const int64_t n4 = Vs / 4;
  float m = -INFINITY, s = 0.0f;
  for (int64_t k = threadIdx.x; k < n4; k += blockDim.x) {
    const float4 v = __ldcs(row4 + k);
    const float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    if (mx > m) {
      s *= __expf(m - mx);
      m = mx;
    }
    s += __expf(v.x - m) + __expf(v.y - m) + __expf(v.z - m) + __expf(v.w - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    online_merge(m, s, m2, s2);
  }
  __shared__ float sm[8], ss[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sm[warp] = m;
    ss[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = sm[0], Ssum = ss[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) online_merge(M, Ssum, sm[w], ss[w]);
    const int64_t tg = target[tok] - static_cast<int64_t>(i) * Vs;
    const float y = (tg >= 0 && tg < Vs) ? row[tg] : 0.0f;
    stats[(3 * i + 0) * T + tok] = M;
    stats[(3 * i + 1) * T + tok] = Ssum;
    stats[(3 * i + 2) * T + tok] = y;
  }
}

// Fused path, one launch for statistics, combine and mean.  grid T, 32 t threads: warp i merges
// shard i's per-tile partials for token `tok` and writes its three numbers; warp 0 then combines
// the shards exactly as ce_combine_kernel does.  Every CTA counts itself done on `ticket` after a
// fence; the CTA that draws the last ticket sums all T per-token losses in fp64 in a fixed order
// (independent of which CTA is last) and writes the mean.  `ticket` must be 0 at launch.
__global__ void __launch_bounds__(32 * kMaxShards) ce_stats_combine_mean_kernel(
    const float2* part, const float* ztarget, const int64_t* target, int64_t T, int64_t Vs, int64_t V, int tps,
    int64_t ntot, float* stats, float* loss, unsigned int* ticket, int* status) {
  const int t = static_cast<int>(blockDim.x >> 5);
  const int64_t tok = blockIdx.x;
  const int i = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  __shared__ float sm[kMaxShards], ss[kMaxShards];
  __shared__ double red[32 * kMaxShards];
  __shared__ bool last;
  {
    const float2* p = part + tok * ntot + static_cast<int64_t>(i) * tps;
    float m = -INFINITY, s = 0.0f;
    // Every load of a batch is issued before the first merge, so a lane has up to 8
    // independent 8-byte loads in flight.
    constexpr int U = 8;
    for (int j0 = lane; j0 < tps; j0 += 32 * U) {
      float2 q[U];
#pragma unroll
      for (int u = 0; u < U; ++u) q[u] = j0 + 32 * u < tps ? __ldcs(p + j0 + 32 * u) : make_float2(-INFINITY, 0.0f);
#pragma unroll
      for (int u = 0; u < U; ++u) online_merge(m, s, q[u].x, q[u].y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      online_merge(m, s, m2, s2);
    }
    if (lane == 0) {
      const int64_t tg = target[tok];
      const bool own = tg >= 0 && tg < V && tg / Vs == i;
      stats[(3 * i + 0) * T + tok] = m;
      stats[(3 * i + 1) * T + tok] = s;
      stats[(3 * i + 2) * T + tok] = own ? ztarget[tok] : 0.0f;
      sm[i] = m;
      ss[i] = s;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int64_t tg = target[tok];
    float M = -INFINITY;
    for (int k = 0; k < t; ++k) M = fmaxf(M, sm[k]);
    float Ssum = 0.0f;
    for (int k = 0; k < t; ++k) Ssum += ss[k] * expf(sm[k] - M);
    const bool ok = tg >= 0 && tg < V;
    const float zy = ok ? ztarget[tok] : 0.0f;
    const float lse = M + logf(Ssum);
    float lt = lse - zy;
    if (!ok) {
      atomicCAS(status, 0, TTL_ERR_DEVICE);
      lt = __int_as_float(0x7fc00000);
    }
    stats[(3 * t) * T + tok] = lse;
    stats[(3 * t + 1) * T + tok] = lt;
    __threadfence();
    last = atomicAdd(ticket, 1u) == static_cast<unsigned int>(gridDim.x) - 1u;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const float* lt = stats + (3 * t + 1) * T;
  double a = 0.0;
  for (int64_t k = threadIdx.x; k < T; k += blockDim.x) a += static_cast<double>(__ldcg(lt + k));
  red[threadIdx.x] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    double sum = 0.0;
    for (int k = 0; k < static_cast<int>(blockDim.x); ++k) sum += red[k];
    *loss = static_cast<float>(sum / static_cast<double>(T));
  }
}

__global__ void ce_combine_kernel(int t, int64_t T, int64_t V, const int64_t* target, float* stats, int* status) {
  const int64_t tok = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (tok >= T) return;
  float M = -INFINITY;
  for (int i = 0; i < t; ++i) M = fmaxf(M, stats[(3 * i) * T + tok]);
  float Ssum = 0.0f, zy = 0.0f;
  for (int i = 0; i < t; ++i) {
    Ssum += stats[(3 * i + 1) * T + tok] * expf(stats[(3 * i) * T + tok] - M);
    zy += stats[(3 * i + 2) * T + tok];
  }
  const float lse = M + logf(Ssum);
  const int64_t tg = target[tok];
  float loss = lse - zy;
  if (tg < 0 || tg >= V) {
    atomicCAS(status, 0, TTL_ERR_DEVICE);
    loss = __int_as_float(0x7fc00000);
  }
  stats[(3 * t) * T + tok] = lse;
  stats[(3 * t + 1) * T + tok] = loss;
}

// One CTA of 1024 threads: each thread sums a strided subset in fp64, then a fixed tree.
__global__ void __launch_bounds__(1024) ce_mean_kernel(const float* loss_tok, int64_t T, float* loss) {
  __shared__ double part[1024];
  double a = 0.0;
  for (int64_t k = threadIdx.x; k < T; k += blockDim.x) a += static_cast<double>(loss_tok[k]);
  part[threadIdx.x] = a;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = T > 0 ? static_cast<float>(part[0] / static_cast<double>(T)) : 0.0f;
}

struct DlogitsShards {
  float* z[kMaxShards];
  __nv_bfloat16* d[kMaxShards];
};

// One float4 of logits (columns 4k..4k+3) -> dZ.
__device__ __forceinline__ void ce_dlogits_vec(float4 v, int64_t k, float* row, __nv_bfloat16* drow, float L,
                                               float invT, int64_t tg, int write_f32) {
  float r[4] = {__expf(v.x - L), __expf(v.y - L), __expf(v.z - L), __expf(v.w - L)};
  const int64_t c0 = k * 4;
#pragma unroll
  for (int q = 0; q < 4; ++q) r[q] = (r[q] - (tg == c0 + q ? 1.0f : 0.0f)) * invT;
  uint2 packed;
  packed.x = pack_bf16x2(r[0], r[1]);
  packed.y = pack_bf16x2(r[2], r[3]);
  __stcs(reinterpret_cast<uint2*>(drow) + k, packed);
  if (write_f32) __stcs(reinterpret_cast<float4*>(row) + k, make_float4(r[0], r[1], r[2], r[3]));
}

// grid (T, t): dZ = (exp(z - lse) - onehot) / T.  Each thread issues kDlU independent 16-byte
// loads before it computes, so enough bytes are in flight to cover HBM latency.
constexpr int kDlU = 4;
__global__ void __launch_bounds__(256) ce_dlogits_kernel(const __grid_constant__ DlogitsShards S, const int64_t* target, int64_t T,
                                                         int64_t Vs, const float* lse, int write_f32) {
  const int64_t tok = blockIdx.x;
  const int i = blockIdx.y;
  float* row = S.z[i] + tok * Vs;
  __nv_bfloat16* drow = S.d[i] + tok * Vs;
  const float L = lse[tok];
  const float invT = 1.0f / static_cast<float>(T);
  const int64_t tg = target[tok] - static_cast<int64_t>(i) * Vs;
  const int64_t n4 = Vs / 4;
  const int64_t step = blockDim.x;
  int64_t k = threadIdx.x;
  for (; k + (kDlU - 1) * step < n4; k += kDlU * step) {
    float4 v[kDlU];
#pragma unroll
    for (int u = 0; u < kDlU; ++u) v[u] = __ldcs(reinterpret_cast<const float4*>(row) + k + u * step);
#pragma unroll
    for (int u = 0; u < kDlU; ++u) ce_dlogits_vec(v[u], k + u * step, row, drow, L, invT, tg, write_f32);
  }
  for (; k < n4; k += step) ce_dlogits_vec(__ldcs(reinterpret_cast<const float4*>(row) + k), k, row, drow, L, invT, tg, write_f32);
}

}  // namespace ttl

using namespace ttl;

namespace {
// Fused-statistics workspace: per token, one (max, sum exp) pair per half GEMM n-tile
// (kGemmBN / 2 vocabulary columns) of every shard, then one target logit per token.
int64_t ce_tiles_per_shard(int64_t Vs) { return 2 * ((Vs + kGemmBN - 1) / kGemmBN); }
size_t ce_part_bytes(int t, int64_t T, int64_t Vs) {
  return (static_cast<size_t>(T) * static_cast<size_t>(t * ce_tiles_per_shard(Vs)) * 8 + 255) & ~size_t(255);
}
size_t ce_ztarget_bytes(int64_t T) { return (static_cast<size_t>(T) * 4 + 255) & ~size_t(255); }
}  // namespace

extern "C" size_t ttl_vocab_parallel_ce_workspace_size(int t, int64_t T, int64_t h, int64_t V) {
  (void)h;
  if (t < 1 || t > kMaxShards || T < 0 || V < 0 || V % t) return 0;
  return ce_part_bytes(t, T, V / t) + ce_ztarget_bytes(T) + 256;   // + the fused launch's ticket
}

extern "C" int ttl_vocab_parallel_ce(int t, int64_t T, int64_t h, int64_t V, const ttl_bf16* H,
                                     const ttl_bf16* const* W, const int64_t* target, float* const* logits,
                                     ttl_bf16* const* dlogits, float* stats, float* loss, ttl_bf16* dH, void* ws,
                                     size_t ws_bytes, int flags, void* stream) {
  const char* name = "ttl_vocab_parallel_ce";
  if (t < 1 || t > kMaxShards) return set_error(TTL_ERR_ARG, "%s: t=%d outside [1,%d]", name, t, kMaxShards);
  if (T < 0 || h < 0 || V < 0) return set_error(TTL_ERR_ARG, "%s: negative shape", name);
  if (flags & ~(TTL_CE_FP32_DLOGITS | TTL_CE_FORWARD_ONLY)) return set_error(TTL_ERR_ARG, "%s: unknown flags", name);
  if (V % t) return set_error(TTL_ERR_SHAPE, "%s: t=%d must divide V=%lld", name, t, (long long)V);
  const int64_t Vs = V / t;
  if (Vs % 8 || h % 8) return set_error(TTL_ERR_SHAPE, "%s: V/t and h must be multiples of 8", name);
  if (T > 0 && (h == 0 || V == 0)) return set_error(TTL_ERR_SHAPE, "%s: h and V must be positive", name);
  if (T >= (int64_t(1) << 31) || Vs >= (int64_t(1) << 31) || h >= (int64_t(1) << 31))
    return set_error(TTL_ERR_SHAPE, "%s: extent beyond 2^31", name);
  const bool fwd_only = flags & TTL_CE_FORWARD_ONLY;
  if (!H || !W || !target || !logits || !stats || !loss) return set_error(TTL_ERR_ARG, "%s: null pointer", name);
  if (!fwd_only && (!dlogits || !dH)) return set_error(TTL_ERR_ARG, "%s: dlogits and dH are required", name);
  if (!aligned16(H) || !aligned16(stats) || (!fwd_only && !aligned16(dH)))
    return set_error(TTL_ERR_ALIGN, "%s: H, stats and dH must be 16-byte aligned", name);
  if (reinterpret_cast<uintptr_t>(target) & 7) return set_error(TTL_ERR_ALIGN, "%s: target not 8-byte aligned", name);
  for (int i = 0; i < t; ++i) {
    if (!W[i] || !logits[i] || (!fwd_only && !dlogits[i])) return set_error(TTL_ERR_ARG, "%s: null shard pointer", name);
    if (!aligned16(W[i]) || !aligned16(logits[i]) || (!fwd_only && !aligned16(dlogits[i])))
      return set_error(TTL_ERR_ALIGN, "%s: shard %d pointer not 16-byte aligned", name, i);
  }
  const bool fused = ws != nullptr;
  if (fused) {
    const size_t need = ttl_vocab_parallel_ce_workspace_size(t, T, h, V);
    if (ws_bytes < need)
      return set_error(TTL_ERR_ARG, "%s: workspace of %zu bytes needed, %zu given", name, need, ws_bytes);
    if (!aligned16(ws)) return set_error(TTL_ERR_ALIGN, "%s: workspace not 16-byte aligned", name);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int rc;
  if (T == 0) {
    // No tokens: the mean over an empty set is taken as 0 and dH has no rows.
    const float zero = 0.0f;
    return cuda_check(cudaMemcpyAsync(loss, &zero, sizeof(float), cudaMemcpyHostToDevice, s), "cudaMemcpyAsync");
  }
  if ((rc = require_sm103())) return rc;
  int* status = device_status_ptr();
  if (!status) return TTL_ERR_CUDA;
  const int tps = static_cast<int>(ce_tiles_per_shard(Vs));
  const int64_t ntot = static_cast<int64_t>(t) * tps;
  float2* part = fused ? static_cast<float2*>(ws) : nullptr;
  float* ztarget = fused ? reinterpret_cast<float*>(static_cast<char*>(ws) + ce_part_bytes(t, T, Vs)) : nullptr;

  // 1. logits Z_i = H W_i^T (fp32).  With a workspace, the epilogue also leaves per-tile
  //    (max, sum exp) partials and the target logit, so step 2 need not re-read the logits.
  {
    GemmBatch batch;
    const int mh = batch.add_map(H, T, h, h, false);
    for (int i = 0; i < t; ++i) {
      const int mw = batch.add_map(W[i], Vs, h, h, false);
      Problem* p = batch.add_problem(T, Vs, false, false, fused ? EPI_F32_CE : EPI_F32, false, i > 0);
      if (batch.error()) return batch.error();
      p->out0 = logits[i];
      p->ld_out = Vs;
      if (fused) {
        p->aux0 = target;
        p->ext0 = static_cast<int64_t>(i) * Vs;
        p->out1 = part;
        p->ext1 = ntot;
        p->out2 = ztarget;
      }
      if ((rc = batch.add_seg(p, mh, 0, mw, -1, 0, h))) return rc;
    }
    if ((rc = batch.launch(s))) return rc;
  }

  // 2-4. per-shard statistics, combine, mean.
  if (fused) {
    unsigned int* ticket = reinterpret_cast<unsigned int*>(static_cast<char*>(ws) + ce_part_bytes(t, T, Vs) +
                                                           ce_ztarget_bytes(T));
    if ((rc = cuda_check(cudaMemsetAsync(ticket, 0, sizeof(unsigned int), s), "cudaMemsetAsync(ticket)"))) return rc;
    TraceScope trace(s, TTL_K_CE_STATS, 0.0,
                     static_cast<double>(T) * (ntot * 8.0 + 4.0 + 8.0 + 3.0 * t * 4.0 + 2.0 * 4.0 + 4.0));
    ce_stats_combine_mean_kernel<<<static_cast<unsigned>(T), 32 * t, 0, s>>>(part, ztarget, target, T, Vs, V, tps,
                                                                             ntot, stats, loss, ticket, status);
    if ((rc = cuda_check(cudaGetLastError(), "ce_stats_combine_mean_kernel launch"))) return rc;
  } else {
    CeShards cs;
    for (int i = 0; i < kMaxShards; ++i) cs.z[i] = i < t ? logits[i] : nullptr;
    {
      TraceScope trace(s, TTL_K_CE_STATS, 0.0, static_cast<double>(T) * V * 4.0);
      ce_stats_kernel<<<dim3(static_cast<unsigned>(T), t), 256, 0, s>>>(cs, target, T, Vs, stats);
      if ((rc = cuda_check(cudaGetLastError(), "ce_stats_kernel launch"))) return rc;
    }
    {
      TraceScope trace(s, TTL_K_CE_SMALL, 0.0, static_cast<double>(T) * (3.0 * t + 2.0) * 4.0);
      ce_combine_kernel<<<static_cast<unsigned>((T + 255) / 256), 256, 0, s>>>(t, T, V, target, stats, status);
      if ((rc = cuda_check(cudaGetLastError(), "ce_combine_kernel launch"))) return rc;
    }
    {
      TraceScope trace(s, TTL_K_CE_SMALL, 0.0, static_cast<double>(T) * 4.0);
      ce_mean_kernel<<<1, 1024, 0, s>>>(stats + (3 * t + 1) * T, T, loss);
      if ((rc = cuda_check(cudaGetLastError(), "ce_mean_kernel launch"))) return rc;
    }
  }
  if (fwd_only) return TTL_OK;

  // 5. dlogits.
  DlogitsShards ds;
  for (int i = 0; i < kMaxShards; ++i) {
    ds.z[i] = i < t ? logits[i] : nullptr;
    ds.d[i] = i < t ? reinterpret_cast<__nv_bfloat16*>(dlogits[i]) : nullptr;
  }
  {
    const double wb = (flags & TTL_CE_FP32_DLOGITS) ? 6.0 : 2.0;
    TraceScope trace(s, TTL_K_CE_DLOGITS, 0.0, static_cast<double>(T) * V * (4.0 + wb));
    ce_dlogits_kernel<<<dim3(static_cast<unsigned>(T), t), 256, 0, s>>>(ds, target, T, Vs, stats + 3 * t * T,
                                                                        (flags & TTL_CE_FP32_DLOGITS) ? 1 : 0);
    if ((rc = cuda_check(cudaGetLastError(), "ce_dlogits_kernel launch"))) return rc;
  }

  // 6. dH = sum_i dZ_i W_i: one accumulator, K loop over the shards in order.
  GemmBatch batch;
  Problem* p = batch.add_problem(T, h, false, true, EPI_BF16, false);
  if (batch.error()) return batch.error();
  p->out0 = dH;
  p->ld_out = h;
  for (int i = 0; i < t; ++i) {
    const int md = batch.add_map(dlogits[i], T, Vs, Vs, false);
    const int mw = batch.add_map(W[i], Vs, h, h, true);
    if ((rc = batch.add_seg(p, md, 0, mw, -1, 0, Vs))) return rc;
  }
  return batch.launch(s);
}

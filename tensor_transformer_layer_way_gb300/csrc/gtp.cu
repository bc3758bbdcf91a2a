// GTP_remat weight path on one GPU.  A TP slice W [K, N] is kept as g row shards
// (shard j = rows [j K/g, (j+1) K/g), each its own allocation).  Before the layer GEMM
// the slice is rebuilt (gathered) and released after; the next layer's gather is issued
// on a side stream while the current GEMM runs; the weight gradient is reduce-scattered
// back into per-shard fp32 staging and merged into main_grad one backward layer later.
//
// Source: "Generalized Tensor Parallelism(GTP)是什么?" -- concepts "GTP_remat",
// "Prefetch chain", "Deferred finalize"; Fig. 1 (AG(W_{i+1}) beside GEMM(W_i), the chain
// head exposed); the list under "all-gather 和 weight gradient 怎么藏在计算后面" (cold start,
// reverse chain in backward, asynchronous reduce-scatter with finalize deferred one step,
// the last one synchronous); the follow-up on GTP_remat ranks seeing independent samples.
//
// Two ways to feed the GEMM: (1) an explicit gather kernel into a slot buffer (what the
// chain prefetches on the side stream), or (2) the gather folded into the GEMM's TMA loads:
// every shard gets its own tensor map and the K loop (forward) or the output column range
// (dgrad) walks the shards, so no slot is materialised.

#include "ttl_device.cuh"
#include "ttl_internal.h"

namespace ttl {

struct GatherSet {
  const uint4* p[kMaxShards];
};

// Block b of a grid of G handles the contiguous vector range [b c, min(n, (b + 1) c)) with
// c = ceil(n / G): every block gets the same work (the last one at most c less), so a launch
// that is all one wave has no tail.
__device__ __forceinline__ void block_range(int64_t n, int64_t& begin, int64_t& end) {
  const int64_t per = (n + gridDim.x - 1) / gridDim.x;
  begin = static_cast<int64_t>(blockIdx.x) * per;
  end = begin + per < n ? begin + per : n;
}

// slot vector v belongs to shard v / vps at offset v % vps (16-byte vectors).  Each thread keeps
// U independent loads in flight.
__global__ void __launch_bounds__(256) gtp_gather_kernel(const __grid_constant__ GatherSet S, uint4* slot, int64_t nvec, int64_t vps) {
  constexpr int U = 4;
  int64_t begin, end;
  block_range(nvec, begin, end);
  for (int64_t base = begin + threadIdx.x; base < end; base += static_cast<int64_t>(blockDim.x) * U) {
    uint4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + static_cast<int64_t>(u) * blockDim.x;
      if (v < end) {
        const int j = static_cast<int>(v / vps);
        x[u] = __ldcs(S.p[j] + (v - j * vps));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + static_cast<int64_t>(u) * blockDim.x;
      if (v < end) slot[v] = x[u];
    }
  }
}

struct FinalizeSet {
  float4* mg[kMaxShards];
  const float4* st[kMaxShards];
};

// main_grad[j] += staging[j] over g shards of nvec4_per float4 vectors each.
__global__ void __launch_bounds__(256) gtp_finalize_kernel(const __grid_constant__ FinalizeSet S, int g, int64_t nvec4_per) {
  constexpr int U = 4;
  const int64_t total = nvec4_per * g;
  int64_t begin, end;
  block_range(total, begin, end);
  for (int64_t base = begin + threadIdx.x; base < end; base += static_cast<int64_t>(blockDim.x) * U) {
    float4 a[U], b[U];
    int j[U];
    int64_t o[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + static_cast<int64_t>(u) * blockDim.x;
      j[u] = v < end ? static_cast<int>(v / nvec4_per) : 0;
      o[u] = v - j[u] * nvec4_per;
      if (v < end) {
        a[u] = S.mg[j[u]][o[u]];
        b[u] = __ldcs(S.st[j[u]] + o[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + static_cast<int64_t>(u) * blockDim.x;
      if (v < end) {
        float4 r = a[u];
        r.x += b[u].x;
        r.y += b[u].y;
        r.z += b[u].z;
        r.w += b[u].w;
        S.mg[j[u]][o[u]] = r;
      }
    }
  }
}

namespace {

// One wave of 256-thread blocks (as many per SM as the kernel's registers allow, from the
// occupancy query), fewer if n is small; the kernels split n evenly over the blocks.
unsigned grid_for(int64_t n, int blocks_per_sm) {
  const int64_t want = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms()) * blocks_per_sm;
  return static_cast<unsigned>(want < 1 ? 1 : (want > cap ? cap : want));
}

template <typename Kernel>
int resident_blocks(Kernel kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, 0) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    n = 1;
  }
  return n;
}

int check_shards(int g, const void* const* arr, const char* what) {
  if (!arr) return set_error(TTL_ERR_ARG, "%s: null shard array", what);
  for (int j = 0; j < g; ++j) {
    if (!arr[j]) return set_error(TTL_ERR_ARG, "%s[%d] is null", what, j);
    if (!aligned16(arr[j])) return set_error(TTL_ERR_ALIGN, "%s[%d] not 16-byte aligned", what, j);
  }
  return TTL_OK;
}

int check_gkn(int g, int64_t K, int64_t N, const char* name) {
  if (g < 1 || g > kMaxShards) return set_error(TTL_ERR_ARG, "%s: g=%d outside [1,%d]", name, g, kMaxShards);
  if (K < 0 || N < 0) return set_error(TTL_ERR_ARG, "%s: negative shape", name);
  if (K % g) return set_error(TTL_ERR_SHAPE, "%s: g=%d must divide K=%lld", name, g, (long long)K);
  if ((K / g) % 8 || N % 8) return set_error(TTL_ERR_SHAPE, "%s: K/g and N must be multiples of 8", name);
  if (K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return set_error(TTL_ERR_SHAPE, "%s: extent beyond 2^31", name);
  return TTL_OK;
}

int finalize(int g, int64_t rows, int64_t N, const float* const* staging, float* const* main_grad, cudaStream_t s) {
  if (rows == 0 || N == 0) return TTL_OK;
  FinalizeSet S;
  for (int j = 0; j < kMaxShards; ++j) {
    S.mg[j] = nullptr;
    S.st[j] = nullptr;
  }
  for (int j = 0; j < g; ++j) {
    S.mg[j] = reinterpret_cast<float4*>(main_grad[j]);
    S.st[j] = reinterpret_cast<const float4*>(staging[j]);
  }
  const int64_t n4 = rows * N / 4;
  TraceScope trace(s, TTL_K_FINALIZE, 0.0, 3.0 * 16.0 * static_cast<double>(n4) * g);
  static const int bps = resident_blocks(gtp_finalize_kernel);
  gtp_finalize_kernel<<<grid_for(n4 * g, bps), 256, 0, s>>>(S, g, n4);
  return cuda_check(cudaGetLastError(), "gtp_finalize_kernel launch");
}

}  // namespace
}  // namespace ttl

using namespace ttl;

extern "C" int ttl_gtp_gather(int g, int64_t K, int64_t N, const ttl_bf16* const* shards, ttl_bf16* slot, void* stream,
                              void* done_event) {
  const char* name = "ttl_gtp_gather";
  int rc = check_gkn(g, K, N, name);
  if (rc) return rc;
  if ((rc = check_shards(g, reinterpret_cast<const void* const*>(shards), "shards"))) return rc;
  if (!slot) return set_error(TTL_ERR_ARG, "%s: slot is null", name);
  if (!aligned16(slot)) return set_error(TTL_ERR_ALIGN, "%s: slot not 16-byte aligned", name);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K > 0 && N > 0) {
    if ((rc = require_sm103())) return rc;
    GatherSet S;
    for (int j = 0; j < kMaxShards; ++j) S.p[j] = nullptr;
    for (int j = 0; j < g; ++j) S.p[j] = reinterpret_cast<const uint4*>(shards[j]);
    const int64_t nvec = K * N / 8;
    TraceScope trace(s, TTL_K_GTP_GATHER, 0.0, 2.0 * 16.0 * static_cast<double>(nvec));
    static const int bps = resident_blocks(gtp_gather_kernel);
    gtp_gather_kernel<<<grid_for(nvec, bps), 256, 0, s>>>(S, reinterpret_cast<uint4*>(slot), nvec, nvec / g);
    if ((rc = cuda_check(cudaGetLastError(), "gtp_gather_kernel launch"))) return rc;
  }
  if (done_event) return cuda_check(cudaEventRecord(static_cast<cudaEvent_t>(done_event), s), "cudaEventRecord");
  return TTL_OK;
}

extern "C" int ttl_gtp_gather_gemm(int g, int64_t M, int64_t K, int64_t N, const ttl_bf16* X,
                                   const ttl_bf16* const* shards, const ttl_bf16* slot, void* slot_ready_event,
                                   ttl_bf16* Y, int transpose_w, void* stream) {
  const char* name = "ttl_gtp_gather_gemm";
  int rc = check_gkn(g, K, N, name);
  if (rc) return rc;
  if (M < 0) return set_error(TTL_ERR_ARG, "%s: negative M", name);
  if (transpose_w != 0 && transpose_w != 1) return set_error(TTL_ERR_ARG, "%s: transpose_w must be 0 or 1", name);
  if (!X || !Y) return set_error(TTL_ERR_ARG, "%s: X or Y is null", name);
  if (!aligned16(X) || !aligned16(Y)) return set_error(TTL_ERR_ALIGN, "%s: X or Y not 16-byte aligned", name);
  if (slot) {
    if (!aligned16(slot)) return set_error(TTL_ERR_ALIGN, "%s: slot not 16-byte aligned", name);
  } else if ((rc = check_shards(g, reinterpret_cast<const void* const*>(shards), "shards"))) {
    return rc;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (slot && slot_ready_event &&
      (rc = cuda_check(cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(slot_ready_event), 0), "cudaStreamWaitEvent")))
    return rc;
  const int64_t Kg = K / g;
  const int64_t out_cols = transpose_w ? K : N;
  const int64_t contr = transpose_w ? N : K;
  if (M == 0 || out_cols == 0) return TTL_OK;
  if (contr == 0) return fill_zero(Y, static_cast<size_t>(M * out_cols) * 2, s);

  GemmBatch batch;
  const int mx = batch.add_map(X, M, contr, contr, false);
  if (!transpose_w) {
    // Y = X W: W is the B operand stored [K, N] (N-major).
    Problem* p = batch.add_problem(M, N, false, true, EPI_BF16, false);
    if (batch.error()) return batch.error();
    p->out0 = Y;
    p->ld_out = N;
    if (slot) {
      const int mw = batch.add_map(slot, K, N, N, true);
      if ((rc = batch.add_seg(p, mx, 0, mw, -1, 0, K))) return rc;
    } else {
      // Folded gather: K segment j reads X columns [j K/g, ...) against shard j.
      for (int j = 0; j < g; ++j) {
        const int mw = batch.add_map(shards[j], Kg, N, N, true);
        if ((rc = batch.add_seg(p, mx, j * Kg, mw, -1, 0, Kg))) return rc;
      }
    }
  } else {
    // dX = dY W^T: W^T is the B operand; W stored [K, N] is K-major for it (N = contraction).
    if (slot) {
      const int mw = batch.add_map(slot, K, N, N, false);
      Problem* p = batch.add_problem(M, K, false, false, EPI_BF16, false);
      if (batch.error()) return batch.error();
      p->out0 = Y;
      p->ld_out = K;
      if ((rc = batch.add_seg(p, mx, 0, mw, -1, 0, N))) return rc;
    } else {
      // Folded gather: output columns [j K/g, (j+1) K/g) come from shard j.
      for (int j = 0; j < g; ++j) {
        const int mw = batch.add_map(shards[j], Kg, N, N, false);
        Problem* p = batch.add_problem(M, Kg, false, false, EPI_BF16, false, j > 0);
        if (batch.error()) return batch.error();
        p->out0 = Y + j * Kg;
        p->ld_out = K;
        if ((rc = batch.add_seg(p, mx, 0, mw, -1, 0, N))) return rc;
      }
    }
  }
  return batch.launch(s);
}

extern "C" int ttl_gtp_wgrad_rs_finalize(int g, int64_t M, int64_t K, int64_t N, const ttl_bf16* X, const ttl_bf16* dY,
                                         float* const* staging_cur, const float* const* staging_prev,
                                         float* const* main_grad_prev, int sync, float* const* main_grad_cur,
                                         void* stream) {
  const char* name = "ttl_gtp_wgrad_rs_finalize";
  int rc = check_gkn(g, K, N, name);
  if (rc) return rc;
  if (M < 0) return set_error(TTL_ERR_ARG, "%s: negative M", name);
  if (!X || !dY) return set_error(TTL_ERR_ARG, "%s: X or dY is null", name);
  if (!aligned16(X) || !aligned16(dY)) return set_error(TTL_ERR_ALIGN, "%s: X or dY not 16-byte aligned", name);
  if ((rc = check_shards(g, reinterpret_cast<const void* const*>(staging_cur), "staging_cur"))) return rc;
  if ((staging_prev == nullptr) != (main_grad_prev == nullptr))
    return set_error(TTL_ERR_ARG, "%s: staging_prev and main_grad_prev must be given together", name);
  if (staging_prev) {
    if ((rc = check_shards(g, reinterpret_cast<const void* const*>(staging_prev), "staging_prev"))) return rc;
    if ((rc = check_shards(g, reinterpret_cast<const void* const*>(main_grad_prev), "main_grad_prev"))) return rc;
  }
  if (sync && (rc = check_shards(g, reinterpret_cast<const void* const*>(main_grad_cur), "main_grad_cur"))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t Kg = K / g;
  if (Kg > 0 && N > 0 && (rc = require_sm103())) return rc;

  // Deferred finalize of the layer processed one backward step earlier.
  if (staging_prev && (rc = finalize(g, Kg, N, staging_prev, main_grad_prev, s))) return rc;

  // wgrad reduce-scattered into shards: staging_j = rows of X^T dY owned by shard j.  The
  // sum over the g token groups' partials is the GEMM's own contraction over the M tokens.
  if (Kg > 0 && N > 0) {
    if (M == 0) {
      for (int j = 0; j < g; ++j)
        if ((rc = fill_zero(staging_cur[j], static_cast<size_t>(Kg * N) * 4, s))) return rc;
    } else {
      GemmBatch batch;
      const int mx = batch.add_map(X, M, K, K, true);    // A = X^T: X stored [M tokens, K] is M-major
      const int md = batch.add_map(dY, M, N, N, true);   // B = dY stored [M tokens, N] is N-major
      for (int j = 0; j < g; ++j) {
        Problem* p = batch.add_problem(Kg, N, true, true, EPI_F32, false);
        if (batch.error()) return batch.error();
        p->a_m0 = static_cast<int32_t>(j * Kg);
        p->out0 = staging_cur[j];
        p->ld_out = N;
        if ((rc = batch.add_seg(p, mx, 0, md, -1, 0, M))) return rc;
      }
      if ((rc = batch.launch(s))) return rc;
    }
  }

  // The last backward layer: nothing follows it, so its finalize happens now.
  if (sync) return finalize(g, Kg, N, const_cast<const float* const*>(staging_cur), main_grad_cur, s);
  return TTL_OK;
}

extern "C" int ttl_gtp_finalize(int g, int64_t K, int64_t N, const float* const* staging, float* const* main_grad,
                                void* stream) {
  const char* name = "ttl_gtp_finalize";
  int rc = check_gkn(g, K, N, name);
  if (rc) return rc;
  if ((rc = check_shards(g, reinterpret_cast<const void* const*>(staging), "staging"))) return rc;
  if ((rc = check_shards(g, reinterpret_cast<const void* const*>(main_grad), "main_grad"))) return rc;
  for (int j = 0; j < g; ++j)
    for (int k = 0; k < g; ++k)
      if (static_cast<const void*>(staging[j]) == static_cast<const void*>(main_grad[k]))
        return set_error(TTL_ERR_ARG, "%s: staging[%d] and main_grad[%d] alias", name, j, k);
  const int64_t Kg = K / g;
  if (Kg == 0 || N == 0) return TTL_OK;
  if ((rc = require_sm103())) return rc;
  return finalize(g, Kg, N, staging, main_grad, static_cast<cudaStream_t>(stream));
}

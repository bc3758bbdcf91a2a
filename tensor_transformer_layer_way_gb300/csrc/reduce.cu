// On-device partial-sum reduction over t logical shard buffers held in one GPU's HBM:
// reduce-scatter, all-gather and the fused all-reduce (= reduce-scatter + all-gather),
// plus the column sums that give bias gradients.
//
// Each buffer is a full-shape partial sum [rows, cols] bf16; buffer r owns the token slab
// rows [r*rows/t, (r+1)*rows/t) (TP-communication page, Fig. 2: GPU0 ends with the first
// half).  Every element is read as bf16, summed in fp32 in buffer order 0..t-1 (plus the
// row bias once), and rounded once to bf16 with round-to-nearest-even.  The kernels are
// HBM-bound streams: 16-byte vectors, consecutive threads on consecutive vectors, every
// shard's load for a vector issued before the adds, grid sized to fill every SM.

#include "ttl_device.cuh"
#include "ttl_internal.h"

namespace ttl {

struct ShardSet {
  __nv_bfloat16* p[kMaxShards];
};

__device__ __forceinline__ uint4 ld_stream(const __nv_bfloat16* base, int64_t v) {
  return __ldcs(reinterpret_cast<const uint4*>(base) + v);
}

__device__ __forceinline__ void st_stream(__nv_bfloat16* base, int64_t v, uint4 x) {
  __stcs(reinterpret_cast<uint4*>(base) + v, x);
}

__device__ __forceinline__ void acc_add(float (&a)[8], uint4 x) {
  a[0] += bf16_lo(x.x); a[1] += bf16_hi(x.x);
  a[2] += bf16_lo(x.y); a[3] += bf16_hi(x.y);
  a[4] += bf16_lo(x.z); a[5] += bf16_hi(x.z);
  a[6] += bf16_lo(x.w); a[7] += bf16_hi(x.w);
}

__device__ __forceinline__ void acc_init(float (&a)[8], uint4 x) {
  a[0] = bf16_lo(x.x); a[1] = bf16_hi(x.x);
  a[2] = bf16_lo(x.y); a[3] = bf16_hi(x.y);
  a[4] = bf16_lo(x.z); a[5] = bf16_hi(x.z);
  a[6] = bf16_lo(x.w); a[7] = bf16_hi(x.w);
}

__device__ __forceinline__ uint4 acc_pack(const float (&a)[8]) {
  uint4 r;
  r.x = pack_bf16x2(a[0], a[1]);
  r.y = pack_bf16x2(a[2], a[3]);
  r.z = pack_bf16x2(a[4], a[5]);
  r.w = pack_bf16x2(a[6], a[7]);
  return r;
}

// Reduce-scatter (AR = false) or all-reduce (AR = true).  nvec = rows*cols/8 vectors,
// vps = vectors per slab, cvec = vectors per row (for the bias column).
template <int T, bool AR>
__global__ void __launch_bounds__(256) shard_reduce_kernel(const __grid_constant__ ShardSet S, const __nv_bfloat16* bias, int64_t nvec,
                                                           int64_t vps, int64_t cvec) {
  constexpr int U = T >= 8 ? 1 : 8 / T;  // vectors per thread per step: >= 8 loads in flight
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x * U;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * U + threadIdx.x; base < nvec; base += step) {
    uint4 in[U][T];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + static_cast<int64_t>(u) * blockDim.x;
      if (v < nvec) {
#pragma unroll
        for (int j = 0; j < T; ++j) in[u][j] = ld_stream(S.p[j], v);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + static_cast<int64_t>(u) * blockDim.x;
      if (v < nvec) {
        float a[8];
        acc_init(a, in[u][0]);
#pragma unroll
        for (int j = 1; j < T; ++j) acc_add(a, in[u][j]);
        if (bias) acc_add(a, *reinterpret_cast<const uint4*>(bias + (v % cvec) * 8));
        const uint4 r = acc_pack(a);
        if (AR) {
#pragma unroll
          for (int j = 0; j < T; ++j) st_stream(S.p[j], v, r);
        } else {
          const int owner = static_cast<int>(v / vps);
          st_stream(S.p[owner], v, r);
        }
      }
    }
  }
}

// All-gather: vector v of slab s is copied from buffer s into every other buffer.
template <int T>
__global__ void __launch_bounds__(256) shard_gather_kernel(const __grid_constant__ ShardSet S, int64_t nvec, int64_t vps) {
  constexpr int U = 4;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x * U;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * U + threadIdx.x; base < nvec; base += step) {
    uint4 x[U];
    int owner[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + static_cast<int64_t>(u) * blockDim.x;
      owner[u] = v < nvec ? static_cast<int>(v / vps) : 0;
      if (v < nvec) x[u] = ld_stream(S.p[owner[u]], v);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + static_cast<int64_t>(u) * blockDim.x;
      if (v < nvec) {
#pragma unroll
        for (int j = 0; j < T; ++j)
          if (j != owner[u]) st_stream(S.p[j], v, x[u]);
      }
    }
  }
}

// Column sums of a [rows, cols] bf16 matrix into bf16 [cols] (fp32 accumulation, fixed
// order: thread y sums rows y, y+8, ...; then the 8 partials are added in order y=0..7).
__global__ void __launch_bounds__(256) column_sum_kernel(const __nv_bfloat16* x, int64_t rows, int64_t cols,
                                                         int64_t ld, __nv_bfloat16* out) {
  __shared__ float part[8][32][8];
  const int64_t cv = static_cast<int64_t>(blockIdx.x) * 32 + threadIdx.x;  // column vector index
  const bool ok = cv * 8 < cols;
  float a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (ok) {
    for (int64_t r = threadIdx.y; r < rows; r += 8) acc_add(a, *reinterpret_cast<const uint4*>(x + r * ld + cv * 8));
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) part[threadIdx.y][threadIdx.x][k] = a[k];
  __syncthreads();
  if (threadIdx.y == 0 && ok) {
    float s[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) s[k] = part[0][threadIdx.x][k];
    for (int y = 1; y < 8; ++y)
#pragma unroll
      for (int k = 0; k < 8; ++k) s[k] += part[y][threadIdx.x][k];
    *reinterpret_cast<uint4*>(out + cv * 8) = acc_pack(s);
  }
}

int column_sum_bf16(const void* x, int64_t rows, int64_t cols, int64_t ld, void* out, cudaStream_t s) {
  if (cols == 0) return TTL_OK;
  if (rows == 0) return fill_zero(out, static_cast<size_t>(cols) * 2, s);
  const unsigned blocks = static_cast<unsigned>((cols / 8 + 31) / 32);
  TraceScope trace(s, TTL_K_OTHER, 0.0, static_cast<double>(rows) * cols * 2.0);
  column_sum_kernel<<<blocks, dim3(32, 8), 0, s>>>(static_cast<const __nv_bfloat16*>(x), rows, cols, ld,
                                                  static_cast<__nv_bfloat16*>(out));
  return cuda_check(cudaGetLastError(), "column_sum_kernel launch");
}

// ------------------------------------------------------------------ launch helpers

namespace {

enum class Mode { RS, AG, AR };

unsigned grid_for(int64_t nvec, int per_thread) {
  const int64_t want = (nvec + 256LL * per_thread - 1) / (256LL * per_thread);
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;  // 8 x 256 threads fill an SM
  return static_cast<unsigned>(want < 1 ? 1 : (want > cap ? cap : want));
}

template <int T>
void launch_t(Mode m, const ShardSet& S, const __nv_bfloat16* bias, int64_t nvec, int64_t vps, int64_t cvec,
              cudaStream_t s) {
  constexpr int U = T >= 8 ? 1 : 8 / T;
  if (m == Mode::RS) shard_reduce_kernel<T, false><<<grid_for(nvec, U), 256, 0, s>>>(S, bias, nvec, vps, cvec);
  else if (m == Mode::AR) shard_reduce_kernel<T, true><<<grid_for(nvec, U), 256, 0, s>>>(S, bias, nvec, vps, cvec);
  else shard_gather_kernel<T><<<grid_for(nvec, 4), 256, 0, s>>>(S, nvec, vps);
}

int run(Mode m, int t, int64_t rows, int64_t cols, ttl_bf16* const* bufs, const ttl_bf16* bias, void* stream,
        const char* name) {
  if (t < 1 || t > kMaxShards) return set_error(TTL_ERR_ARG, "%s: t=%d outside [1,%d]", name, t, kMaxShards);
  if (rows < 0 || cols < 0) return set_error(TTL_ERR_ARG, "%s: negative shape", name);
  if (!bufs) return set_error(TTL_ERR_ARG, "%s: null buffer array", name);
  if (cols % 8) return set_error(TTL_ERR_SHAPE, "%s: cols=%lld must be a multiple of 8", name, (long long)cols);
  // Slab ownership needs t | rows; the fused all-reduce writes every row of every buffer and
  // accepts any row count.
  if (m != Mode::AR && rows % t)
    return set_error(TTL_ERR_SHAPE, "%s: t=%d must divide rows=%lld", name, t, (long long)rows);
  if (rows == 0 || cols == 0) return TTL_OK;   // empty buffers (their pointers may be null)
  ShardSet S;
  for (int j = 0; j < kMaxShards; ++j) S.p[j] = nullptr;
  for (int j = 0; j < t; ++j) {
    if (!bufs[j]) return set_error(TTL_ERR_ARG, "%s: buffer %d is null", name, j);
    if (!aligned16(bufs[j])) return set_error(TTL_ERR_ALIGN, "%s: buffer %d not 16-byte aligned", name, j);
    for (int k = 0; k < j; ++k)
      if (bufs[k] == bufs[j]) return set_error(TTL_ERR_ARG, "%s: buffers %d and %d alias", name, k, j);
    S.p[j] = reinterpret_cast<__nv_bfloat16*>(bufs[j]);
  }
  if (bias && !aligned16(bias)) return set_error(TTL_ERR_ALIGN, "%s: bias not 16-byte aligned", name);
  int rc = require_sm103();
  if (rc) return rc;
  const int64_t nvec = rows * cols / 8;
  const int64_t vps = nvec / t;
  const int64_t cvec = cols / 8;
  const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(bias);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Algorithmic HBM bytes: RS reads t slabs per owned slab and writes it, (t+1) S in all;
  // AR reads t S and writes t S; AG reads S and writes (t-1) S.
  const double S_bytes = static_cast<double>(rows) * cols * 2.0;
  const double bytes = m == Mode::RS ? (t + 1) * S_bytes : m == Mode::AR ? 2.0 * t * S_bytes : t * S_bytes;
  TraceScope trace(s, m == Mode::AG ? TTL_K_GATHER : TTL_K_REDUCE, 0.0, bytes);
  switch (t) {
    case 1: launch_t<1>(m, S, b, nvec, vps, cvec, s); break;
    case 2: launch_t<2>(m, S, b, nvec, vps, cvec, s); break;
    case 3: launch_t<3>(m, S, b, nvec, vps, cvec, s); break;
    case 4: launch_t<4>(m, S, b, nvec, vps, cvec, s); break;
    case 5: launch_t<5>(m, S, b, nvec, vps, cvec, s); break;
    case 6: launch_t<6>(m, S, b, nvec, vps, cvec, s); break;
    case 7: launch_t<7>(m, S, b, nvec, vps, cvec, s); break;
    case 8: launch_t<8>(m, S, b, nvec, vps, cvec, s); break;
    case 9: launch_t<9>(m, S, b, nvec, vps, cvec, s); break;
    case 10: launch_t<10>(m, S, b, nvec, vps, cvec, s); break;
    case 11: launch_t<11>(m, S, b, nvec, vps, cvec, s); break;
    case 12: launch_t<12>(m, S, b, nvec, vps, cvec, s); break;
    case 13: launch_t<13>(m, S, b, nvec, vps, cvec, s); break;
    case 14: launch_t<14>(m, S, b, nvec, vps, cvec, s); break;
    case 15: launch_t<15>(m, S, b, nvec, vps, cvec, s); break;
    default: launch_t<16>(m, S, b, nvec, vps, cvec, s); break;
  }
  return cuda_check(cudaGetLastError(), name);
}

}  // namespace

int shard_all_reduce_internal(int t, int64_t rows, int64_t cols, ttl_bf16* const* bufs, const ttl_bf16* bias,
                              cudaStream_t s) {
  // t = 1 with no bias is the identity (bf16 -> fp32 -> bf16 is exact): skip the pass.
  if (t == 1 && !bias) return TTL_OK;
  return run(Mode::AR, t, rows, cols, bufs, bias, s, "shard_all_reduce");
}

}  // namespace ttl

extern "C" int ttl_shard_reduce_scatter(int t, int64_t rows, int64_t cols, ttl_bf16* const* bufs,
                                        const ttl_bf16* bias, void* stream) {
  return ttl::run(ttl::Mode::RS, t, rows, cols, bufs, bias, stream, "ttl_shard_reduce_scatter");
}

extern "C" int ttl_shard_all_gather(int t, int64_t rows, int64_t cols, ttl_bf16* const* bufs, void* stream) {
  return ttl::run(ttl::Mode::AG, t, rows, cols, bufs, nullptr, stream, "ttl_shard_all_gather");
}

extern "C" int ttl_shard_all_reduce(int t, int64_t rows, int64_t cols, ttl_bf16* const* bufs, const ttl_bf16* bias,
                                    void* stream) {
  return ttl::run(ttl::Mode::AR, t, rows, cols, bufs, bias, stream, "ttl_shard_all_reduce");
}

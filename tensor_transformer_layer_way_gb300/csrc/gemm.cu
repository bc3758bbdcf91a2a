// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05) for sm_103a.
//
// One launch computes a list of problems (e.g. the t shards of a column-parallel layer,
// or the t shards' dgrad and wgrad) so that the narrow per-shard GEMMs fill the GPU
// together.  Work is cut into tiles of TILE_M rows x 256 (wide: 512) accumulator columns,
// walked by persistent workers with a static stride.  Roles (192 threads per CTA; wide: 320):
//   warp 0      TMA producer: one thread issues cp.async.bulk.tensor loads of this CTA's
//               A rows and B columns for each 64-wide K block into a shared-memory ring;
//   warp 1      MMA issuer: allocates 512 TMEM columns (two 128 x 256 fp32 accumulators,
//               double-buffered; wide: one 128 x 512) and one thread issues tcgen05.mma per
//               16-wide K step;
//   warps 2..   epilogue (4 warps; wide: 8): tcgen05.ld the accumulator rows, apply the fused
//               op (bias, GeLU, SwiGLU, their derivatives, cross-entropy partials) and store
//               bf16/fp32 to global memory.
//
// Three variants share the code:
//   single CTA  (PAIR = false): TILE_M = 128, MMA M=128 N=256, 4 stages of 48 KiB.
//   CTA pair    (PAIR = true) : a cluster of two CTAs on two SMs computes a 256 x 256 tile
//               with tcgen05.mma.cta_group::2 (M=256 N=256).  Each CTA holds its own 128 A
//               rows and 128 of the 256 B columns, so the B tile is read from HBM/L2 and
//               shared memory once per pair; each stage is 32 KiB and 7 stages fit.  Both
//               CTAs' TMA loads complete on the leader CTA's full barrier, the leader alone
//               issues MMAs, and its commits arrive on both CTAs' barriers (multicast).
//   wide pair   (WIDE = true) : 256 x 512 tiles (bf16, SwiGLU-forward and fp32 outputs, see
//               launch() for which launches qualify).  Each K step issues two
//               independent N=256 MMAs into the halves of one 512-column accumulator: MMAs
//               into one accumulator wait for each other, two chains overlap, and the operand
//               bytes per MMA drop by a quarter (each stage: 16 KiB of A, 32 KiB of B per CTA,
//               4 stages).  With TMEM full the epilogue cannot overlap the next tile's MMAs, so
//               8 epilogue warps empty the accumulator into shared-memory staging (partly the
//               ring slots of the next tile's k-blocks 2 and 3) and write it with TMA stores.
//
// Every mbarrier wait is bounded in wall time; a timeout records TTL_ERR_TIMEOUT, all roles
// leave their loops, in-flight copies and MMAs are waited for (again bounded), TMEM is
// released and the kernel returns.
//
// Shared-memory operand layouts (128-byte swizzle, 1024-byte aligned stages):
//   K-major operand  : box {64 K, 128 rows}; row r at r*128 B; 8-row atoms 1024 B apart
//                      (SBO = 1024).  K step of 16 = +32 B on the descriptor start.
//   MN-major operand : boxes {64 MN, 64 K} side by side 8 KiB apart (LBO = 8192);
//                      K row k at k*128 B (SBO = 1024).  K step of 16 = +2048 B.

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "ttl_device.cuh"
#include "ttl_internal.h"

namespace ttl {

constexpr int BN = kGemmBN;        // accumulator columns per tile
constexpr int BK = 64;             // K per stage
constexpr int TMEM_COLS = 2 * BN;  // two accumulators
constexpr int GROUP_M = 16;
constexpr int STG_BOX = 4096;      // wide epilogue: one TMA store box, 32 rows x 64 bf16 columns

// WIDE (a CTA pair only): 256 x 512 output tiles, two N = 256 MMAs per K step into the two
// halves of a single 512-column accumulator, plain bf16 epilogue through TMA stores.
template <bool PAIR, bool WIDE = false>
struct Cfg {
  static_assert(!WIDE || PAIR, "the wide tile is a CTA-pair tile");
  static constexpr int TILE_M = PAIR ? 256 : 128;     // rows per tile (both CTAs of a pair)
  static constexpr int TILE_N = WIDE ? 2 * BN : BN;   // output columns per (unpaired) tile
  static constexpr int TILE_NP = WIDE ? BN : BN / 2;  // output columns per paired tile
  static constexpr int B_COLS = WIDE ? 256 : PAIR ? 128 : 256;   // B columns held by one CTA
  static constexpr int A_BYTES = 128 * BK * 2;        // 16 KiB
  static constexpr int B_BYTES = B_COLS * BK * 2;     // 16 or 32 KiB
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = WIDE ? 4 : PAIR ? 7 : 4;
  static constexpr int TX_BYTES = PAIR ? 2 * STAGE : STAGE;   // counted on the (leader's) full barrier
  // producer warp, MMA warp, then the epilogue warps: one per TMEM lane quadrant, two in the
  // wide kernel (one per 256-column half of the accumulator)
  static constexpr int THREADS = WIDE ? 320 : 192;
  static constexpr int EPI_WARPS = THREADS / 32 - 2;
  static constexpr int SCHED_BYTES = 1280;   // the shared copy of the tile schedule
  // Wide epilogue staging: 32 boxes, 12 in each of the two ring slots it borrows at a tile's
  // end and 8 in a region of their own after the barriers and the schedule.
  static constexpr int STG_OFF = STAGES * STAGE + 2048;
  static constexpr int SMEM = WIDE ? STG_OFF + 8 * STG_BOX + 1024 /*align slack*/
                                   : STAGES * STAGE + 1024 /*align slack*/ + 256 /*barriers*/ + SCHED_BYTES;
  static_assert(SMEM <= 232448, "shared memory beyond the per-CTA limit");
  static_assert(!WIDE || (STAGE % STG_BOX == 0 && STAGE / STG_BOX == 12), "wide staging layout");
};

struct TileCoord {
  int p, tm, tn;
};

// The tile schedule, copied into shared memory at kernel start.  Decoding a tile from the
// parameter block (about 32 KiB, far more than the constant cache holds) misses that cache at
// every tile change, while the tensor pipe runs dry.
struct SchedTable {
  int32_t g_start[kMaxProblems], g_tm[kMaxProblems], g_tn[kMaxProblems], g_first[kMaxProblems],
      g_count[kMaxProblems];
  int32_t p_tn0[kMaxProblems];
  int32_t p_kb[kMaxProblems];      // k-blocks of each of the problem's tiles (all segments)
  uint32_t p_flags[kMaxProblems];  // bit 0: A MN-major, bit 1: B MN-major, bit 2: 128-column MMAs
  // Per group, what the MMA thread needs when every problem of the group has the same k-block
  // count and flags: bit 31 set, flags in bits 0..2, k-blocks from bit 3.  The MMA thread then
  // skips the full tile decode, which at a tile change leaves the tensor pipe waiting.
  uint32_t g_mma[kMaxProblems];
  int32_t ngroups;
};
static_assert(sizeof(SchedTable) <= Cfg<true>::SCHED_BYTES, "schedule table beyond its space");
static_assert(256 + Cfg<true>::SCHED_BYTES <= 2048, "barriers and schedule overlap the wide staging");

// Linear tile index -> (problem, m-tile, n-tile).  Inside a tile group the order is: bands
// of GROUP_M m-tiles; within a band, n-tiles across all of the group's problems; within
// an n-tile, the band's m-tiles.  Persistent workers taking consecutive indices therefore
// share A rows (same band) and B columns (same n-tile) in L2.
// `gi` is the caller's running group index: a worker visits increasing tile indices, so the
// search for the tile's group resumes where the previous one ended.
__device__ __forceinline__ TileCoord decode_tile_s(const SchedTable& S, int tile, int& gi) {
#pragma unroll 1
  while (gi + 1 < S.ngroups && tile >= S.g_start[gi + 1]) ++gi;
  const int local = tile - S.g_start[gi];
  const int per_band = GROUP_M * S.g_tn[gi];
  const int band = local / per_band;
  const int first_m = band * GROUP_M;
  const int gm = min(GROUP_M, S.g_tm[gi] - first_m);
  const int r = local - band * per_band;
  const int tn = r / gm;
  int lo = S.g_first[gi], hi = S.g_first[gi] + S.g_count[gi] - 1;
#pragma unroll 1
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (S.p_tn0[mid] <= tn) lo = mid;
    else hi = mid - 1;
  }
  TileCoord c;
  c.p = lo;
  c.tm = first_m + r % gm;
  c.tn = tn - S.p_tn0[lo];
  return c;
}
static_assert(sizeof(GemmParams) <= 32764, "kernel parameter block beyond the 32 KiB limit");

// ------------------------------------------------------------------ epilogue math

// The epilogue math uses the fast exponential intrinsic: its results are rounded to bf16
// right after, so a few ulp of fp32 error are invisible.
// tanh(u) = 1 - 2 / (exp(2u) + 1), which saturates correctly to +-1 at large |u|.
__device__ __forceinline__ float tanh_fast(float u) { return 1.0f - __fdividef(2.0f, __expf(2.0f * u) + 1.0f); }

__device__ __forceinline__ float gelu_tanh_f(float x) {
  const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
  return 0.5f * x * (1.0f + tanh_fast(u));
}

__device__ __forceinline__ float gelu_tanh_grad_f(float x) {
  const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
  const float th = tanh_fast(u);
  const float du = 0.7978845608028654f * (1.0f + 3.0f * 0.044715f * x * x);
  return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * du;
}

__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// Stores 32 consecutive bf16 values of one row (columns col0..col0+31), masking at N.  A whole,
// 32-byte aligned chunk goes out as two 32-byte stores: each one fills an L2 sector, where a
// 16-byte store fills half of one (this thread's row is the only one in the sector).  The same
// change to the fp32 stores (CE logits) gained nothing and is not made.
__device__ __forceinline__ void store_row32_bf16(void* base, int64_t ld, int row, int col0, int N,
                                                 const float* v) {
  __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(base) + static_cast<int64_t>(row) * ld + col0;
  if (col0 + 32 <= N && (reinterpret_cast<uintptr_t>(p) & 31u) == 0) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    st_global_v8(p, w);
    st_global_v8(p + 16, w + 8);
    return;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (col0 + q * 8 < N) {
      uint4 w;
      w.x = pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]);
      w.y = pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]);
      w.z = pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]);
      w.w = pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]);
      *reinterpret_cast<uint4*>(p + q * 8) = w;
    }
  }
}

__device__ __forceinline__ void store_row32_f32(void* base, int64_t ld, int row, int col0, int N,
                                                const float* v) {
  float* p = reinterpret_cast<float*>(base) + static_cast<int64_t>(row) * ld + col0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (col0 + q * 4 < N) {
      *reinterpret_cast<float4*>(p + q * 4) = make_float4(v[q * 4], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
    }
  }
}

__device__ __forceinline__ void load_row32_bf16(const void* base, int64_t ld, int row, int col0, int N, float* v) {
  const __nv_bfloat16* p = reinterpret_cast<const __nv_bfloat16*>(base) + static_cast<int64_t>(row) * ld + col0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w = make_uint4(0, 0, 0, 0);
    if (col0 + q * 8 < N) w = *reinterpret_cast<const uint4*>(p + q * 8);
    v[q * 8 + 0] = bf16_lo(w.x);
    v[q * 8 + 1] = bf16_hi(w.x);
    v[q * 8 + 2] = bf16_lo(w.y);
    v[q * 8 + 3] = bf16_hi(w.y);
    v[q * 8 + 4] = bf16_lo(w.z);
    v[q * 8 + 5] = bf16_hi(w.z);
    v[q * 8 + 6] = bf16_lo(w.w);
    v[q * 8 + 7] = bf16_hi(w.w);
  }
}

// Per-row state an epilogue carries across the chunks of one tile.
struct EpiState {
  float m = -INFINITY, s = 0.0f;   // EPI_F32_CE: running max and sum
  int64_t ce_tgt = -1;             // EPI_F32_CE: target column relative to the tile's first
};

// The epilogue of one 32-column chunk (chunk `ch` of the tile starting at column n_base) of
// this thread's row; r holds the fp32 accumulator bits.
__device__ __forceinline__ void epilogue_chunk(const Problem& pr, int row, int n_base, int ch,
                                               const uint32_t (&r)[32], EpiState& st) {
  const int col0 = n_base + ch * 32;
  if (col0 >= pr.N) return;
  const int epi = pr.epi;
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  if (epi == EPI_F32) {
    store_row32_f32(pr.out0, pr.ld_out, row, col0, pr.N, v);
  } else if (epi == EPI_F32_CE) {
    store_row32_f32(pr.out0, pr.ld_out, row, col0, pr.N, v);
    const int nv = min(32, pr.N - col0);
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nv) mx = fmaxf(mx, v[j]);
    if (mx > st.m) {
      st.s *= __expf(st.m - mx);
      st.m = mx;
    }
    float se = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < nv) se += __expf(v[j] - st.m);
      if (st.ce_tgt == ch * 32 + j && j < nv) reinterpret_cast<float*>(pr.out2)[row] = v[j];
    }
    st.s += se;
  } else if (epi == EPI_BF16 || epi == EPI_GELU_FWD) {
    if (pr.bias0) {
      float b[32];
      load_row32_bf16(pr.bias0, 0, 0, col0, pr.N, b);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] += b[j];
    }
    store_row32_bf16(pr.out0, pr.ld_out, row, col0, pr.N, v);
    if (epi == EPI_GELU_FWD) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = gelu_tanh_f(v[j]);
      store_row32_bf16(pr.out1, pr.ld_out, row, col0, pr.N, v);
    }
  } else if (epi == EPI_GELU_BWD) {
    float x[32];
    load_row32_bf16(pr.aux0, pr.ld_aux, row, col0, pr.N, x);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= gelu_tanh_grad_f(x[j]);
    store_row32_bf16(pr.out0, pr.ld_out, row, col0, pr.N, v);
  } else if (epi == EPI_SWIGLU_BWD) {
    float gg[32], vv[32], dg[32];
    load_row32_bf16(pr.aux0, pr.ld_aux, row, col0, pr.N, gg);
    load_row32_bf16(pr.aux1, pr.ld_aux, row, col0, pr.N, vv);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float sg = sigmoid_f(gg[j]);
      dg[j] = v[j] * vv[j] * sg * (1.0f + gg[j] * (1.0f - sg));
      v[j] = v[j] * gg[j] * sg;
    }
    store_row32_bf16(pr.out0, pr.ld_out, row, col0, pr.N, dg);
    store_row32_bf16(pr.out1, pr.ld_out, row, col0, pr.N, v);
  }
}

// Applies the problem's epilogue to one accumulator tile slice held in this CTA's TMEM
// (128 rows; this thread owns one row) and stores it.  `half` selects the accumulator columns
// [half BN/2, (half + 1) BN/2) (a paired tile: output columns [half BN/4, (half + 1) BN/4) of
// both halves); an epilogue warp calls it for half 0, then half 1.
__device__ __forceinline__ void epilogue_tile(const Problem& pr, uint32_t tbase, int row, int n_base_paired,
                                              int n_base, int half) {
  const bool row_ok = row < pr.M;
  const int epi = pr.epi;
  if (pr.paired) {
#pragma unroll 1
    for (int ch = half * (BN / 4 / 32); ch < (half + 1) * (BN / 4 / 32); ++ch) {
      uint32_t g[32], u[32];
      __syncwarp();
      tmem_ld_32x32b_x32(tbase + ch * 32, g);
      tmem_ld_32x32b_x32(tbase + BN / 2 + ch * 32, u);
      tmem_ld_wait();
      const int col0 = n_base_paired + ch * 32;
      if (row_ok && col0 < pr.N) {
        float gv[32], uv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          gv[j] = __uint_as_float(g[j]);
          uv[j] = __uint_as_float(u[j]);
        }
        store_row32_bf16(pr.out0, pr.ld_out, row, col0, pr.N, gv);
        store_row32_bf16(pr.out1, pr.ld_out, row, col0, pr.N, uv);
        if (epi == EPI_SWIGLU_FWD) {
          float hv[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) hv[j] = gv[j] * sigmoid_f(gv[j]) * uv[j];
          store_row32_bf16(pr.out2, pr.ld_out, row, col0, pr.N, hv);
        }
      }
    }
    return;
  }
  EpiState st;
  if (epi == EPI_F32_CE && row_ok) st.ce_tgt = reinterpret_cast<const int64_t*>(pr.aux0)[row] - pr.ext0 - n_base;
  // Two 32-column chunks per TMEM round trip: both loads are in flight before the one wait.
#pragma unroll 1
  for (int ch = half * (BN / 2 / 32); ch < (half + 1) * (BN / 2 / 32); ch += 2) {
    if (n_base + ch * 32 >= pr.N) break;   // the same for the whole warp: nothing left to store
    uint32_t r0[32], r1[32];
    __syncwarp();
    tmem_ld_32x32b_x32(tbase + ch * 32, r0);
    tmem_ld_32x32b_x32(tbase + ch * 32 + 32, r1);
    tmem_ld_wait();
    if (row_ok) {
      epilogue_chunk(pr, row, n_base, ch, r0, st);
      epilogue_chunk(pr, row, n_base, ch + 1, r1, st);
    }
  }
  // One (max, sum) partial per row and half tile (BN / 2 columns): index 2 tile + half.
  if (epi == EPI_F32_CE && row_ok) {
    const int64_t chunk = pr.cbase + 2 * (n_base / BN) + half;   // 128-column chunk of this half tile
    reinterpret_cast<float2*>(pr.out1)[static_cast<int64_t>(row) * pr.ext1 + chunk] = make_float2(st.m, st.s);
  }
}

// ------------------------------------------------------------------ the kernel

template <bool PAIR, bool WIDE = false>
__global__ void __launch_bounds__(Cfg<PAIR, WIDE>::THREADS, 1) gemm_tcgen05_kernel(const __grid_constant__ GemmParams P) {
  using C = Cfg<PAIR, WIDE>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Stages must sit on 1024-byte boundaries for the 128-byte swizzle atoms.  The offset is
  // the same in both CTAs of a pair, which the pair MMA's shared descriptors rely on.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE);
  uint64_t* empty_bar = full_bar + C::STAGES;
  uint64_t* tfull_bar = empty_bar + C::STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* done_bar = tempty_bar + 2;
  uint64_t* stg_bar = done_bar + 1;   // wide: the epilogue has handed its borrowed ring slots back
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stg_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  SchedTable* sched = reinterpret_cast<SchedTable*>(smem + C::STAGES * C::STAGE + 256);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;   // 0 = leader of the pair
  const bool leader = rank == 0;
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int nunits = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], (PAIR ? 2 : 1) * C::EPI_WARPS);   // every epilogue warp of the pair arrives
    }
    mbar_init(done_bar, 1);
    mbar_init(stg_bar, C::EPI_WARPS);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) {
    for (int i = lane; i < P.nmaps; i += 32) tma_prefetch_map(&P.maps[i]);
  }
  for (int i = threadIdx.x; i < kMaxProblems; i += blockDim.x) {
    if (i < P.ngroups) {
      const TileGroup& g = P.groups[i];
      sched->g_start[i] = g.tile_start;
      sched->g_tm[i] = g.tiles_m;
      sched->g_tn[i] = g.tiles_n;
      sched->g_first[i] = g.first;
      sched->g_count[i] = g.count;
    }
    if (i < P.nprob) {
      const Problem& pr = P.probs[i];
      int kb = 0;
      for (int s = 0; s < pr.nseg; ++s) kb += pr.seg[s].kblocks;
      sched->p_tn0[i] = pr.tn0;
      sched->p_kb[i] = kb;
      sched->p_flags[i] = (pr.a_mn ? 1u : 0u) | (pr.b_mn ? 2u : 0u) | (pr.half_n ? 4u : 0u);
    }
  }
  if (threadIdx.x < P.ngroups) {
    const TileGroup& g = P.groups[threadIdx.x];
    uint32_t word = 0;
    bool uniform = true;
    for (int j = g.first; j < g.first + g.count; ++j) {
      const Problem& pr = P.probs[j];
      int kb = 0;
      for (int s = 0; s < pr.nseg; ++s) kb += pr.seg[s].kblocks;
      const uint32_t w = (pr.a_mn ? 1u : 0u) | (pr.b_mn ? 2u : 0u) | (pr.half_n ? 4u : 0u) |
                         (static_cast<uint32_t>(kb) << 3);
      if (j == g.first) word = w;
      else if (w != word) uniform = false;
    }
    sched->g_mma[threadIdx.x] = (uniform && g.count > 0 && (word >> 3) < (1u << 28)) ? (word | 0x80000000u) : 0u;
  }
  if (threadIdx.x == 0) sched->ngroups = P.ngroups;
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  if (PAIR) cluster_sync_all();   // the peer's barriers must be initialised before any remote signal
  else __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  int* status = P.status;
  const uint64_t tmo = P.timeout_ns;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      int gi = 0;
      int tile_seq = 0;   // tiles this worker has loaded so far
      for (int tile = unit; ok && tile < P.total_tiles; tile += nunits, ++tile_seq) {
        const TileCoord c = decode_tile_s(*sched, tile, gi);
        int lkb = 0;      // k-block index within the tile, over its segments
        const Problem& pr = P.probs[c.p];
        int am = pr.a_m0 + c.tm * C::TILE_M + static_cast<int>(rank) * 128;
        int slab = 0;
        if (pr.a_slab_rows > 0) {   // rows of token slab `slab` come from its own map
          slab = am / pr.a_slab_rows;
          am -= slab * pr.a_slab_rows;
        }
        for (int s = 0; ok && s < pr.nseg; ++s) {
          const Seg& sg = pr.seg[s];
          const CUtensorMap* ma = &P.maps[sg.map_a + slab];
          const CUtensorMap* mb0 = &P.maps[sg.map_b];
          const CUtensorMap* mb1 = pr.paired ? &P.maps[sg.map_b2] : mb0;
          const int bnb = pr.b_n0 + sg.b_n1;
          const int bn0 = pr.paired ? bnb + c.tn * C::TILE_NP : bnb + c.tn * C::TILE_N;
          // The second half of the B columns: a pair's second CTA supplies columns
          // [N/2, N) of the MMA (64 of a 128-column one); paired tiles share coordinates.
          const int bn1 = pr.paired ? bn0 : bn0 + (pr.half_n ? BN / 4 : BN / 2);
          const bool b_half = !PAIR && pr.half_n;   // one CTA, 128 columns: no second B box
          for (int kb = 0; kb < sg.kblocks; ++kb, ++lkb) {
            // Wide: the previous tile's epilogue borrowed the ring slots of this tile's k-blocks
            // 2 and 3 (every tile has at least 3) as staging; wait until it hands them back.
            if (WIDE && lkb == 2 && tile_seq > 0 &&
                !mbar_wait(stg_bar, static_cast<uint32_t>(tile_seq - 1) & 1u, abort_flag, status, tmo)) {
              ok = false;
              break;
            }
            if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, status, tmo)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + stage * C::STAGE;
            uint8_t* sb = sa + C::A_BYTES;
            const int ka = sg.a_k0 + kb * BK;
            const int kbb = sg.b_k0 + kb * BK;
            if (PAIR) {
              // Both CTAs' copies complete on the leader's full barrier, which the leader
              // arms with the bytes of the whole pair.
              if (leader) mbar_arrive_expect_tx(&full_bar[stage], C::TX_BYTES);
              const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
              if (!pr.a_mn) {
                tma_load_2d_pair(sa, ma, fb, ka, am);
              } else {
                tma_load_2d_pair(sa, ma, fb, am, ka);
                tma_load_2d_pair(sa + 8192, ma, fb, am + 64, ka);
              }
              if (WIDE) {
                // This CTA's 128 columns of each 256-column accumulator half: [r 128, r 128 + 128)
                // of the first half, then the same of the second half 16 KiB further on (a paired
                // tile: the same columns of map_b2).
                const int bw = bn0 + static_cast<int>(rank) * (BN / 2);
                const int bw2 = pr.paired ? bw : bw + BN;
                if (!pr.b_mn) {
                  tma_load_2d_pair(sb, mb0, fb, kbb, bw);
                  tma_load_2d_pair(sb + 16384, mb1, fb, kbb, bw2);
                } else {
                  tma_load_2d_pair(sb, mb0, fb, bw, kbb);
                  tma_load_2d_pair(sb + 8192, mb0, fb, bw + 64, kbb);
                  tma_load_2d_pair(sb + 16384, mb1, fb, bw2, kbb);
                  tma_load_2d_pair(sb + 24576, mb1, fb, bw2 + 64, kbb);
                }
              } else {
                const CUtensorMap* mb = rank ? mb1 : mb0;
                const int bn = rank ? bn1 : bn0;
                if (!pr.b_mn) {
                  tma_load_2d_pair(sb, mb, fb, kbb, bn);
                } else {
                  tma_load_2d_pair(sb, mb, fb, bn, kbb);
                  tma_load_2d_pair(sb + 8192, mb, fb, bn + 64, kbb);
                }
              }
            } else {
              mbar_arrive_expect_tx(&full_bar[stage], b_half ? C::TX_BYTES - 16384 : C::TX_BYTES);
              if (!pr.a_mn) {
                tma_load_2d(sa, ma, &full_bar[stage], ka, am);
              } else {
                tma_load_2d(sa, ma, &full_bar[stage], am, ka);
                tma_load_2d(sa + 8192, ma, &full_bar[stage], am + 64, ka);
              }
              if (!pr.b_mn) {
                tma_load_2d(sb, mb0, &full_bar[stage], kbb, bn0);
                if (!b_half) tma_load_2d(sb + 16384, mb1, &full_bar[stage], kbb, bn1);
              } else {
                tma_load_2d(sb, mb0, &full_bar[stage], bn0, kbb);
                tma_load_2d(sb + 8192, mb0, &full_bar[stage], bn0 + 64, kbb);
                if (!b_half) {
                  tma_load_2d(sb + 16384, mb1, &full_bar[stage], bn1, kbb);
                  tma_load_2d(sb + 24576, mb1, &full_bar[stage], bn1 + 64, kbb);
                }
              }
            }
            ++issued;
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // No copy may still be landing in shared memory when the CTA leaves: wait for the
      // completion of the last min(issued, STAGES) loads (bounded).  In a pair the leader's
      // full barriers count the follower's copies too, and the follower leaves only after
      // the leader (cluster barrier below).
      if (leader) {
        const int pending = issued < C::STAGES ? issued : C::STAGES;
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < pending; ++i) {
          if (--s < 0) {
            s = C::STAGES - 1;
            ph ^= 1u;
          }
          int dummy_abort = 0;
          mbar_wait(&full_bar[s], ph, reinterpret_cast<volatile int*>(&dummy_abort), status, tmo);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (leader)
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const uint32_t sbase = smem_u32(smem);
      int gi = 0;
      for (int tile = unit; ok && tile < P.total_tiles; tile += nunits) {
#pragma unroll 1
        while (gi + 1 < sched->ngroups && tile >= sched->g_start[gi + 1]) ++gi;
        uint32_t fl;
        int nkb;
        const uint32_t gw = sched->g_mma[gi];
        if (gw & 0x80000000u) {
          fl = gw & 7u;
          nkb = static_cast<int>((gw >> 3) & 0x0FFFFFFFu);
        } else {
          const int pi = decode_tile_s(*sched, tile, gi).p;
          fl = sched->p_flags[pi];
          nkb = sched->p_kb[pi];
        }
        const bool a_mn = fl & 1u, b_mn = fl & 2u;
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, status, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + (WIDE ? 0u : static_cast<uint32_t>(acc * BN));
        const uint32_t idesc = idesc_bf16_f32(C::TILE_M, (fl & 4u) ? BN / 2 : BN, a_mn, b_mn);
        const uint32_t a_step = a_mn ? 2048u : 32u;
        const uint32_t b_step = b_mn ? 2048u : 32u;
        const uint32_t a_lbo = a_mn ? 8192u : 16u;
        const uint32_t b_lbo = b_mn ? 8192u : 16u;
        uint32_t accumulate = 0;
        {   // the tile's k-blocks over all its segments, in order
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&full_bar[stage], phase, abort_flag, status, tmo)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t sa = sbase + stage * C::STAGE;
            const uint64_t ad0 = smem_desc_sw128(sa, a_lbo, 1024);
            const uint64_t bd0 = smem_desc_sw128(sa + C::A_BYTES, b_lbo, 1024);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t adesc = desc_advance(ad0, kk * a_step);
              const uint64_t bdesc = desc_advance(bd0, kk * b_step);
              if (PAIR) {
                umma_bf16_pair(d_tmem, adesc, bdesc, idesc, accumulate);
                // Wide: the second half into accumulator columns [256, 512); the two chains
                // are independent, so neither MMA waits for the other's accumulator.
                if (WIDE) umma_bf16_pair(d_tmem + BN, adesc, desc_advance(bdesc, 16384), idesc, accumulate);
              } else {
                umma_bf16(d_tmem, adesc, bdesc, idesc, accumulate);
              }
              accumulate = 1;
            }
            // Frees this stage in both CTAs once the MMAs reading it are done.
            if (PAIR) umma_commit_pair(&empty_bar[stage], 0x3);
            else umma_commit(&empty_bar[stage]);
            if (++stage == C::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) break;
        if (PAIR) umma_commit_pair(&tfull_bar[acc], 0x3);
        else umma_commit(&tfull_bar[acc]);
        if (WIDE) {
          acc_phase ^= 1u;   // one accumulator: the next tile waits for this tile's epilogue
        } else if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs issued by this thread must finish before TMEM is released.
      if (PAIR) umma_commit_pair(done_bar, 0x1);
      else umma_commit(done_bar);
      int dummy_abort = 0;
      mbar_wait(done_bar, 0, reinterpret_cast<volatile int*>(&dummy_abort), status, tmo);
    }
    __syncwarp();
  } else if (WIDE) {
    // ---------------------------------------------------------------- wide epilogue warps
    // Two warps per TMEM lane quadrant, one per 256-column half.  A warp moves its 32 rows x
    // 256 columns from TMEM through registers (rounded to bf16) into four swizzled 32 x 64 staging
    // boxes, hands the accumulator back, then writes the boxes with TMA stores.  The staging
    // lives in the two ring slots that the next tile's k-blocks 2 and 3 will use (both free once
    // this tile's MMAs are done; the producer waits for stg_bar before refilling them) and in a
    // region of its own, so the accumulator is free again after the TMEM reads alone.
    const int ew = warp - 2;                // 0 .. EPI_WARPS - 1
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    const int h2 = ew >> 2;                 // accumulator half
    const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty_bar[0]), 0);
    uint32_t acc_phase = 0;
    int gi = 0;
    int64_t kb_end = 0;                     // k-blocks loaded through the current tile
    for (int tile = unit; tile < P.total_tiles; tile += nunits) {
      const TileCoord c = decode_tile_s(*sched, tile, gi);
      const Problem& pr = P.probs[c.p];
      kb_end += sched->p_kb[c.p];
      const bool ready = mbar_wait(&tfull_bar[0], acc_phase, abort_flag, status, tmo);
      if (!__all_sync(0xffffffffu, ready)) break;
      tc_fence_after_sync();
      // Boxes in a warp's own region (warps 6 and 7) are not lent by the producer: the plain
      // path hands such a warp's share back before its stores have read them, so it waits for
      // them here, before it writes the boxes again.
      const bool lent = 4 * ew < 24;
      if (!lent) {
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
      }
      uint8_t* const slot_a = smem + static_cast<int>((kb_end + 2) % C::STAGES) * C::STAGE;
      uint8_t* const slot_b = smem + static_cast<int>((kb_end + 3) % C::STAGES) * C::STAGE;
      // Staging box j of this warp: boxes 0..11 in slot_a, 12..23 in slot_b, 24..31 in the own region.
      auto box = [&](int j) -> uint8_t* {
        const int b = 4 * ew + j;
        return b < 12 ? slot_a + b * STG_BOX : b < 24 ? slot_b + (b - 12) * STG_BOX : smem + C::STG_OFF + (b - 24) * STG_BOX;
      };
      const int y = c.tm * C::TILE_M + static_cast<int>(rank) * 128 + q * 32;   // first row of this warp
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      if (pr.paired) {
        // SwiGLU forward: accumulator columns [0, 256) hold G and [256, 512) hold V of the tile's
        // 256 output columns; this warp takes output columns [h2 128, h2 128 + 128).  G and V go
        // to boxes 0, 1 and 2, 3; H = SiLU(G) V (from the fp32 values) waits in registers and
        // takes G's boxes once their stores have read them.
        const int col0 = c.tn * C::TILE_NP + h2 * 128;
        uint32_t hq[64];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int sub = 0; sub < 2; ++sub) {
            uint32_t g[32], u[32];
            __syncwarp();
            const uint32_t cg = tq + static_cast<uint32_t>(h2 * 128 + j * 64 + sub * 32);
            tmem_ld_32x32b_x32(cg, g);
            tmem_ld_32x32b_x32(cg + BN, u);
            tmem_ld_wait();
            uint8_t* rg = box(j) + lane * 128;
            uint8_t* rv = box(2 + j) + lane * 128;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float gv[8], uv[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                gv[e] = __uint_as_float(g[8 * k + e]);
                uv[e] = __uint_as_float(u[8 * k + e]);
              }
              const int pos = ((sub * 4 + k) ^ (lane & 7)) << 4;
              *reinterpret_cast<uint4*>(rg + pos) = make_uint4(pack_bf16x2(gv[0], gv[1]), pack_bf16x2(gv[2], gv[3]),
                                                               pack_bf16x2(gv[4], gv[5]), pack_bf16x2(gv[6], gv[7]));
              *reinterpret_cast<uint4*>(rv + pos) = make_uint4(pack_bf16x2(uv[0], uv[1]), pack_bf16x2(uv[2], uv[3]),
                                                               pack_bf16x2(uv[4], uv[5]), pack_bf16x2(uv[6], uv[7]));
#pragma unroll
              for (int e = 0; e < 4; ++e)
                hq[j * 32 + sub * 16 + k * 4 + e] =
                    pack_bf16x2(gv[2 * e] * sigmoid_f(gv[2 * e]) * uv[2 * e],
                                gv[2 * e + 1] * sigmoid_f(gv[2 * e + 1]) * uv[2 * e + 1]);
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (y < pr.M) {
#pragma unroll 1
            for (int j = 0; j < 2; ++j) {
              if (col0 + j * 64 >= pr.N) break;
              tma_store_2d(&P.maps[pr.omap], box(j), col0 + j * 64, y);
              tma_store_2d(&P.maps[pr.omap + 1], box(2 + j), col0 + j * 64, y);
            }
          }
          bulk_commit_group();
          bulk_wait_group_read<0>();
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint8_t* rowp = box(j) + lane * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4*>(rowp + ((k ^ (lane & 7)) << 4)) =
                make_uint4(hq[j * 32 + 4 * k], hq[j * 32 + 4 * k + 1], hq[j * 32 + 4 * k + 2], hq[j * 32 + 4 * k + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (y < pr.M) {
#pragma unroll 1
            for (int j = 0; j < 2; ++j) {
              if (col0 + j * 64 >= pr.N) break;
              tma_store_2d(&P.maps[pr.omap + 2], box(j), col0 + j * 64, y);
            }
          }
          bulk_commit_group();
          bulk_wait_group_read<0>();   // the boxes may be overwritten: hand the borrowed slots back
          mbar_arrive(stg_bar);
        }
        __syncwarp();
        acc_phase ^= 1u;
        continue;
      }
      const int col0 = c.tn * C::TILE_N + h2 * BN;   // output column of this warp's first box
      const uint32_t tb = tq + static_cast<uint32_t>(h2 * BN);
      if (pr.epi == EPI_F32 || pr.epi == EPI_F32_CE) {
        // fp32: 256 columns are 8 boxes of 32 rows x 32 columns, staged in two rounds of 128
        // columns through this warp's four boxes; round 1 reuses them once round 0's stores
        // have read them, and TMEM is released after round 1's last read.  The cross-entropy
        // variant folds each round's 128 columns into one (max, sum exp) partial per row.
        const bool ce = pr.epi == EPI_F32_CE;
        const int row = y + lane;
        const bool row_ok = row < pr.M;
        const int64_t tgt = (ce && row_ok) ? reinterpret_cast<const int64_t*>(pr.aux0)[row] - pr.ext0 : -1;
        const int nchunks = 2 * ((pr.N + BN - 1) / BN);   // partials this problem owns per row
#pragma unroll 1
        for (int r = 0; r < 2; ++r) {
          float m = -INFINITY, sum = 0.0f;
#pragma unroll 1
          for (int sub = 0; sub < 2; ++sub) {
            uint32_t r0[32], r1[32];
            __syncwarp();
            tmem_ld_32x32b_x32(tb + r * 128 + sub * 64, r0);
            tmem_ld_32x32b_x32(tb + r * 128 + sub * 64 + 32, r1);
            tmem_ld_wait();
            if (r == 1 && sub == 1) {
              // The last TMEM read of this warp: the MMA may start the next tile.
              tc_fence_before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);
            }
            if (r == 1 && sub == 0) {   // round 0's boxes must have been read by their stores
              if (lane == 0) bulk_wait_group_read<0>();
              __syncwarp();
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t* w = hh ? r1 : r0;
              const int colc = col0 + r * 128 + sub * 64 + hh * 32;   // problem column of w[0]
              if (ce) {
                const int nv = min(32, pr.N - colc);
                if (nv > 0) {
                  float mx = -INFINITY;
#pragma unroll
                  for (int e = 0; e < 32; ++e)
                    if (e < nv) mx = fmaxf(mx, __uint_as_float(w[e]));
                  if (mx > m) {
                    sum *= __expf(m - mx);
                    m = mx;
                  }
                  float se = 0.0f;
#pragma unroll
                  for (int e = 0; e < 32; ++e)
                    if (e < nv) se += __expf(__uint_as_float(w[e]) - m);
                  sum += se;
                  if (tgt >= colc && tgt < colc + nv) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                      if (tgt == colc + e) reinterpret_cast<float*>(pr.out2)[row] = __uint_as_float(w[e]);
                  }
                }
              }
              uint8_t* rowp = box(2 * sub + hh) + lane * 128;
#pragma unroll
              for (int k = 0; k < 8; ++k)
                *reinterpret_cast<uint4*>(rowp + ((k ^ (lane & 7)) << 4)) =
                    make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
            }
          }
          if (ce && row_ok) {
            const int chunk = 4 * c.tn + 2 * h2 + r;   // 128-column chunk of the problem
            if (chunk < nchunks)
              reinterpret_cast<float2*>(pr.out1)[static_cast<int64_t>(row) * pr.ext1 + pr.cbase + chunk] =
                  make_float2(m, sum);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (y < pr.M) {
#pragma unroll 1
              for (int b = 0; b < 4; ++b) {
                const int x = col0 + r * 128 + b * 32;
                if (x >= pr.N) break;
                tma_store_2d(&P.maps[pr.omap], box(b), x, y);
              }
            }
            bulk_commit_group();
          }
          __syncwarp();
        }
        if (lane == 0) {
          bulk_wait_group_read<0>();   // the boxes may be overwritten: hand the borrowed slots back
          mbar_arrive(stg_bar);
        }
        __syncwarp();
        acc_phase ^= 1u;
        continue;
      }
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        uint32_t r0[32], r1[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tb + j * 64, r0);
        tmem_ld_32x32b_x32(tb + j * 64 + 32, r1);
        tmem_ld_wait();
        if (j == 3) {
          // Every TMEM read of this warp is complete (tcgen05.wait::ld): the MMA may start the next tile.
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);
        }
        float v[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          v[i] = __uint_as_float(r0[i]);
          v[32 + i] = __uint_as_float(r1[i]);
        }
        // Row `lane` of the box: 128 bytes, 16-byte chunk k at position k ^ (row mod 8) (the
        // 128-byte swizzle of the output tensor map).
        uint8_t* rowp = box(j) + lane * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 w = make_uint4(pack_bf16x2(v[8 * k], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                                     pack_bf16x2(v[8 * k + 4], v[8 * k + 5]), pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
          *reinterpret_cast<uint4*>(rowp + ((k ^ (lane & 7)) << 4)) = w;
        }
        // Each box is stored as soon as it is written, so the stores run beside the next reads.
        fence_proxy_async_smem();   // generic-proxy writes before the TMA engine's reads
        __syncwarp();
        if (lane == 0 && y < pr.M && col0 + j * 64 < pr.N) tma_store_2d(&P.maps[pr.omap], box(j), col0 + j * 64, y);
      }
      if (lane == 0) {
        bulk_commit_group();
        if (lent) bulk_wait_group_read<0>();   // the boxes may be overwritten: hand the borrowed slots back
        mbar_arrive(stg_bar);
      }
      __syncwarp();
      acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_group_all();   // every store complete before shared memory goes away
    __syncwarp();
    tc_fence_before_sync();
  } else {
    // ---------------------------------------------------------------- epilogue warps
    // One warp per TMEM lane quadrant, storing both halves of the accumulator columns in turn.
    // (Two warps per quadrant finished each tile sooner but ran as a denser burst, which slowed
    // the next tile's first MMAs on the schedulers they share with the MMA and producer warps.)
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint32_t tempty_leader0 = PAIR ? mapa_shared(smem_u32(&tempty_bar[0]), 0) : 0u;
    // (The saved pre-activations of a backward epilogue are not prefetched to L2 a tile
    // ahead: measured on the fc2 dgrad, the prefetches added 0.5 GB of DRAM reads, lines
    // evicted before use, and made the launch 2% slower.)
    int gi = 0;
    for (int tile = unit; tile < P.total_tiles; tile += nunits) {
      const TileCoord c = decode_tile_s(*sched, tile, gi);
      const Problem& pr = P.probs[c.p];
      const bool ready = mbar_wait(&tfull_bar[acc], acc_phase, abort_flag, status, tmo);
      if (!__all_sync(0xffffffffu, ready)) break;
      tc_fence_after_sync();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      const int row = c.tm * C::TILE_M + static_cast<int>(rank) * 128 + row_in_tile;
      for (int half = 0; half < 2; ++half) epilogue_tile(pr, tbase, row, c.tn * (BN / 2), c.tn * BN, half);
      tc_fence_before_sync();
      __syncwarp();
      // This warp's accumulator reads are complete (tcgen05.wait::ld in the epilogue): the
      // MMA may overwrite the buffer.  Relaxed: the tile's global stores need not drain first.
      if (lane == 0) {
        if (PAIR) mbar_arrive_cluster_relaxed(tempty_leader0 + acc * 8u);
        else mbar_arrive_relaxed(&tempty_bar[acc]);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    tc_fence_before_sync();
  }

  // Both CTAs of a pair leave together: the leader's MMAs read the follower's shared memory
  // and write its TMEM, so neither may release them while the other still works.
  if (PAIR) cluster_sync_all();
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    if (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

namespace {

using EncodeTiledFn = decltype(&cuTensorMapEncodeTiled);

// The driver's tensor-map encoder, looked up through the runtime so that the library does
// not link libcuda (it then loads on machines without a driver, e.g. for symbol checks).
EncodeTiledFn encode_tiled_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct DevState {
  bool attrs = false;
  int pair_clusters = 0;   // co-resident CTA pairs (0 = not queried / none)
  int wide_clusters = 0;   // the same for the wide kernel
};

int device_setup(int device, DevState** out) {
  static std::mutex mu;
  static DevState st[64];
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return set_error(TTL_ERR_CUDA, "device index out of range");
  DevState& s = st[device];
  if (!s.attrs) {
    int rc = cuda_check(cudaFuncSetAttribute(gemm_tcgen05_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg<false>::SMEM),
                        "cudaFuncSetAttribute(gemm smem)");
    if (rc) return rc;
    rc = cuda_check(cudaFuncSetAttribute(gemm_tcgen05_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<true>::SMEM),
                    "cudaFuncSetAttribute(gemm pair smem)");
    if (rc) return rc;
    rc = cuda_check(cudaFuncSetAttribute(gemm_tcgen05_kernel<true, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<true, true>::SMEM),
                    "cudaFuncSetAttribute(gemm wide smem)");
    if (rc) return rc;
    // How many CTA pairs can be resident at once (one CTA per SM).
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * 512, 1, 1);
    cfg.blockDim = dim3(Cfg<true>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg<true>::SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tcgen05_kernel<true>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    s.pair_clusters = n;
    cfg.blockDim = dim3(Cfg<true, true>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg<true, true>::SMEM;
    n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tcgen05_kernel<true, true>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    s.wide_clusters = n;
    s.attrs = true;
  }
  *out = &s;
  return TTL_OK;
}

// TTL_GEMM_CTA_PAIR=0 selects the single-CTA tiles for every launch (for comparisons).
bool pair_allowed() {
  static int v = -1;
  if (v < 0) {
    const char* e = std::getenv("TTL_GEMM_CTA_PAIR");
    v = (e && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}

// TTL_GEMM_WIDE=0 keeps every launch on the 256-column tiles (for comparisons).
bool wide_allowed() {
  static int v = -1;
  if (v < 0) {
    const char* e = std::getenv("TTL_GEMM_WIDE");
    v = (e && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}

}  // namespace

int encode_map_bf16(CUtensorMap* out, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows) {
  if (!aligned16(ptr) || (ld * 2) % 16 != 0 || cols % 8 != 0 || rows <= 0 || cols <= 0)
    return set_error(TTL_ERR_ALIGN, "tensor map %p: pointer, row stride (%lld) and width (%lld) must be 16-byte aligned",
                     ptr, (long long)ld, (long long)cols);
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return set_error(TTL_ERR_CUDA, "cuTensorMapEncodeTiled not available from the CUDA driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return cu_check(enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                  "cuTensorMapEncodeTiled");
}

int encode_map_f32(CUtensorMap* out, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                   int box_rows) {
  if (!aligned16(ptr) || (ld * 4) % 16 != 0 || cols % 4 != 0 || rows <= 0 || cols <= 0)
    return set_error(TTL_ERR_ALIGN, "tensor map %p: pointer, row stride (%lld) and width (%lld) must be 16-byte aligned",
                     ptr, (long long)ld, (long long)cols);
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return set_error(TTL_ERR_CUDA, "cuTensorMapEncodeTiled not available from the CUDA driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return cu_check(enc(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                  "cuTensorMapEncodeTiled(f32)");
}

int encode_map_bf16_3d(CUtensorMap* out, const void* ptr, int64_t d0, int64_t d1, int64_t d2, int64_t ld1,
                       int64_t ld2, int box0, int box1) {
  if (!aligned16(ptr) || (ld1 * 2) % 16 != 0 || (ld2 * 2) % 16 != 0 || d0 % 8 != 0 || d0 <= 0 || d1 <= 0 || d2 <= 0)
    return set_error(TTL_ERR_ALIGN, "tensor map %p: pointer, strides and width must be 16-byte aligned", ptr);
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return set_error(TTL_ERR_CUDA, "cuTensorMapEncodeTiled not available from the CUDA driver");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d0), static_cast<cuuint64_t>(d1), static_cast<cuuint64_t>(d2)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld1) * 2, static_cast<cuuint64_t>(ld2) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box0), static_cast<cuuint32_t>(box1), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return cu_check(enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                  "cuTensorMapEncodeTiled(3d)");
}

GemmBatch::GemmBatch() : p_(new GemmParams), nmaps_(0), err_(TTL_OK), flops_(0.0), bytes_(0.0) {
  std::memset(static_cast<void*>(p_), 0, sizeof(GemmParams));
}

GemmBatch::~GemmBatch() { delete p_; }

int GemmBatch::add_map(const void* ptr, int64_t rows, int64_t cols, int64_t ld, bool mn_major) {
  if (err_) return -1;
  if (nmaps_ >= kMaxMaps) {
    err_ = set_error(TTL_ERR_ARG, "GEMM batch: too many operands (max %d)", kMaxMaps);
    return -1;
  }
  if (!aligned16(ptr) || (ld * 2) % 16 != 0 || cols % 8 != 0) {
    err_ = set_error(TTL_ERR_ALIGN, "GEMM operand %p: pointer, row stride (%lld) and width (%lld) must be 16-byte aligned",
                     ptr, (long long)ld, (long long)cols);
    return -1;
  }
  if (rows <= 0 || cols <= 0) {
    err_ = set_error(TTL_ERR_SHAPE, "GEMM operand with empty extent");
    return -1;
  }
  for (int i = 0; i < nmaps_; ++i) {
    const MapKey& k = keys_[i];
    if (k.ptr == ptr && k.rows == rows && k.cols == cols && k.ld == ld && k.mn == mn_major) return i;
  }
  keys_[nmaps_] = MapKey{ptr, rows, cols, ld, mn_major};
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64, mn_major ? 64u : 128u};
  cuuint32_t estr[2] = {1, 1};
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) {
    err_ = set_error(TTL_ERR_CUDA, "cuTensorMapEncodeTiled not available from the CUDA driver");
    return -1;
  }
  CUresult r = enc(&p_->maps[nmaps_], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    err_ = cu_check(r, "cuTensorMapEncodeTiled");
    return -1;
  }
  return nmaps_++;
}

int GemmBatch::add_maps_consecutive(const void* const* ptrs, int n, int64_t rows, int64_t cols, int64_t ld,
                                    bool mn_major) {
  if (err_) return -1;
  if (n < 1 || nmaps_ + n > kMaxMaps) {
    err_ = set_error(TTL_ERR_ARG, "GEMM batch: no room for %d consecutive operands", n);
    return -1;
  }
  const int first = nmaps_;
  for (int i = 0; i < n; ++i) {
    // A distinct key per slot keeps add_map's de-duplication from folding these together.
    const int before = nmaps_;
    keys_[nmaps_] = MapKey{nullptr, -1, -1, -1, false};
    const int idx = add_map(ptrs[i], rows, cols, ld, mn_major);
    if (idx < 0) return -1;
    if (idx != before) {   // de-duplicated onto an earlier map: encode a private copy here
      p_->maps[nmaps_] = p_->maps[idx];
      keys_[nmaps_] = MapKey{nullptr, -1, -1, -1, false};
      ++nmaps_;
    }
  }
  return first;
}

Problem* GemmBatch::add_problem(int64_t M, int64_t N, bool a_mn, bool b_mn, int epi, bool paired, bool join) {
  if (err_) return nullptr;
  if (join && (p_->nprob == 0 || p_->probs[p_->nprob - 1].M != M))
    join = false;   // a group needs the same M; otherwise start a new one.  Its problems may
                    // mix paired and unpaired tiles: each tile is decoded against its own problem.
  if (p_->nprob >= kMaxProblems) {
    err_ = set_error(TTL_ERR_ARG, "GEMM batch: too many problems (max %d)", kMaxProblems);
    return nullptr;
  }
  if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) {
    err_ = set_error(TTL_ERR_SHAPE, "GEMM extent beyond 2^31");
    return nullptr;
  }
  Problem* p = &p_->probs[p_->nprob++];
  std::memset(static_cast<void*>(p), 0, sizeof(Problem));
  p->M = static_cast<int32_t>(M);
  p->N = static_cast<int32_t>(N);
  p->a_mn = a_mn;
  p->b_mn = b_mn;
  p->epi = static_cast<uint8_t>(epi);
  p->paired = paired;
  p->join = join;
  return p;
}

int GemmBatch::add_seg(Problem* p, int map_a, int64_t a_k0, int map_b, int map_b2, int64_t b_k0, int64_t K,
                       int64_t b_n1) {
  if (err_) return err_;
  if (!p || map_a < 0 || map_b < 0 || (p->paired && map_b2 < 0)) return err_ = set_error(TTL_ERR_ARG, "bad GEMM segment");
  if (p->nseg >= kMaxSegs) return err_ = set_error(TTL_ERR_ARG, "GEMM problem: too many K segments");
  if (K <= 0) return err_ = set_error(TTL_ERR_SHAPE, "GEMM segment with empty K");
  Seg& s = p->seg[p->nseg++];
  s.map_a = static_cast<int16_t>(map_a);
  s.map_b = static_cast<int16_t>(map_b);
  s.map_b2 = static_cast<int16_t>(map_b2 < 0 ? map_b : map_b2);
  s.a_k0 = static_cast<int32_t>(a_k0);
  s.b_k0 = static_cast<int32_t>(b_k0);
  s.kblocks = static_cast<int32_t>((K + BK - 1) / BK);
  s.b_n1 = static_cast<int32_t>(b_n1);
  const double ncols = p->paired ? 2.0 * p->N : static_cast<double>(p->N);
  flops_ += 2.0 * p->M * ncols * static_cast<double>(K);
  bytes_ += 2.0 * (static_cast<double>(p->M) * K + ncols * K);
  if (p->nseg == 1) {
    const int nout = p->epi == EPI_SWIGLU_FWD ? 3 : (p->epi == EPI_GELU_FWD || p->epi == EPI_SWIGLU_BWD) ? 2 : 1;
    const int naux = p->epi == EPI_SWIGLU_BWD ? 2 : p->epi == EPI_GELU_BWD ? 1 : 0;
    const double esz = (p->epi == EPI_F32 || p->epi == EPI_F32_CE) ? 4.0 : 2.0;
    bytes_ += static_cast<double>(p->M) * p->N * (esz * nout + 2.0 * naux);
  }
  return TTL_OK;
}

int GemmBatch::flush(cudaStream_t stream) {
  if (err_) return err_;
  const int rc = p_->nprob ? launch(stream) : TTL_OK;
  std::memset(static_cast<void*>(p_), 0, sizeof(GemmParams));
  nmaps_ = 0;
  flops_ = 0.0;
  bytes_ = 0.0;
  return rc;
}

int GemmBatch::launch(cudaStream_t stream) {
  if (err_) return err_;
  int max_m = 0;
  for (int i = 0; i < p_->nprob; ++i) {
    Problem& p = p_->probs[i];
    if (p.nseg == 0) return set_error(TTL_ERR_ARG, "GEMM problem %d has no K segment", i);
    // Every TMA x coordinate (innermost, in elements) must be a multiple of 8 bf16 = 16 bytes.
    bool aligned = (p.a_m0 % 8 == 0) && (p.b_n0 % 8 == 0);
    for (int k = 0; k < p.nseg; ++k)
      aligned = aligned && p.seg[k].a_k0 % 8 == 0 && p.seg[k].b_k0 % 8 == 0 && p.seg[k].b_n1 % 8 == 0;
    if (!aligned) return set_error(TTL_ERR_ALIGN, "GEMM problem %d: operand offsets must be multiples of 8", i);
    if (p.M > max_m) max_m = p.M;
  }
  int rc = require_sm103();
  if (rc) return rc;
  int dev = 0;
  if ((rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice"))) return rc;
  DevState* ds = nullptr;
  if ((rc = device_setup(dev, &ds))) return rc;
  // CTA pairs (256-row tiles) unless every problem is at most 128 rows tall, or a problem's
  // A rows come in token slabs that a 256-row tile would straddle.
  bool pair = pair_allowed() && ds->pair_clusters > 0 && max_m > 128;
  for (int i = 0; i < p_->nprob; ++i) {
    const Problem& p = p_->probs[i];
    if (p.a_slab_rows <= 0) continue;
    if (p.a_slab_rows % 128 || (p.a_m0 + p.M) > p.a_slab_rows * kMaxShards || p.a_m0 % p.a_slab_rows)
      return set_error(TTL_ERR_SHAPE, "GEMM problem %d: token slabs of %d rows must be multiples of 128", i,
                       p.a_slab_rows);
    if (p.a_slab_rows % 256) pair = false;
  }
  // The wide kernel (256 x 512 tiles, TMA-store epilogue) takes launches whose problems all
  // have one of its epilogues (plain bf16 without bias, the SwiGLU forward, fp32, fp32 with the
  // cross-entropy partials), more than 256 columns (SwiGLU: 128) and at least 3 k-blocks (its
  // epilogue borrows the ring slots of the next tile's k-blocks 2 and 3), and whose outputs a
  // tensor map can address.
  int out_maps = 0;   // the wide epilogue's output tensor maps: one per problem, three for SwiGLU
  for (int i = 0; i < p_->nprob; ++i) out_maps += p_->probs[i].paired ? 3 : 1;
  bool wide = pair && wide_allowed() && ds->wide_clusters > 0 && nmaps_ + out_maps <= kMaxMaps;
  for (int i = 0; wide && i < p_->nprob; ++i) {
    const Problem& p = p_->probs[i];
    int kb = 0;
    for (int k = 0; k < p.nseg; ++k) kb += p.seg[k].kblocks;
    const bool plain = p.epi == EPI_BF16 && !p.paired && p.N > BN && (p.ld_out * 2) % 16 == 0;
    const bool swiglu = p.epi == EPI_SWIGLU_FWD && p.paired && p.N > BN / 2 && aligned16(p.out1) &&
                        aligned16(p.out2) && (p.ld_out * 2) % 16 == 0;
    const bool f32 = (p.epi == EPI_F32 || p.epi == EPI_F32_CE) && !p.paired && p.N > BN && (p.ld_out * 4) % 16 == 0;
    wide = (plain || swiglu || f32) && !p.bias0 && p.N % 8 == 0 && kb >= 3 && aligned16(p.out0) && p.ld_out >= p.N;
  }
  const int tile_m = pair ? Cfg<true>::TILE_M : Cfg<false>::TILE_M;
  const int tile_n = wide ? Cfg<true, true>::TILE_N : BN;
  int total = 0;
  p_->ngroups = 0;
  for (int i = 0; i < p_->nprob; ++i) {
    Problem& p = p_->probs[i];
    const int tn = p.paired ? (wide ? Cfg<true, true>::TILE_NP : BN / 2) : tile_n;
    p.tiles_m = (p.M + tile_m - 1) / tile_m;
    p.tiles_n = (p.N + tn - 1) / tn;
    p.half_n = !p.paired && p.N <= BN / 2;
    if (!p.join || p_->ngroups == 0) {
      TileGroup& g = p_->groups[p_->ngroups++];
      g.tile_start = total;
      g.tiles_m = p.tiles_m;
      g.tiles_n = 0;
      g.first = i;
      g.count = 0;
    }
    TileGroup& g = p_->groups[p_->ngroups - 1];
    // Cross-entropy partials: two per 256-column tile of every earlier problem of the group,
    // whichever tile width the launch uses.
    p.cbase = g.count == 0 ? 0 : p_->probs[i - 1].cbase + 2 * ((p_->probs[i - 1].N + BN - 1) / BN);
    p.tn0 = g.tiles_n;
    g.tiles_n += p.tiles_n;
    g.count += 1;
    total += p.tiles_m * p.tiles_n;
  }
  p_->total_tiles = total;
  if (wide) {
    for (int i = 0; i < p_->nprob; ++i) {
      Problem& p = p_->probs[i];
      // 32-row x 128-byte boxes (64 bf16 or 32 fp32 columns), the staging layout of the wide
      // epilogue; a SwiGLU tile writes G, V and H through three consecutive maps.
      p.omap = static_cast<uint8_t>(nmaps_);
      if (p.epi == EPI_F32 || p.epi == EPI_F32_CE) {
        if ((rc = encode_map_f32(&p_->maps[nmaps_++], p.out0, p.M, p.N, p.ld_out, 32, 32))) return rc;
        continue;
      }
      void* const outs[3] = {p.out0, p.out1, p.out2};
      for (int k = 0; k < (p.paired ? 3 : 1); ++k)
        if ((rc = encode_map_bf16(&p_->maps[nmaps_++], outs[k], p.M, p.N, p.ld_out, 64, 32))) return rc;
    }
  }
  p_->nmaps = nmaps_;
  if (total == 0) return TTL_OK;
  p_->status = device_status_ptr();
  if (!p_->status) return TTL_ERR_CUDA;
  p_->timeout_ns = 2000000000ull;  // 2 s per wait: far beyond any legitimate stall
  TraceScope trace(stream, TTL_K_GEMM, flops_, bytes_);
  if (!pair) {
    const int grid = total < num_sms() ? total : num_sms();
    gemm_tcgen05_kernel<false><<<grid, Cfg<false>::THREADS, Cfg<false>::SMEM, stream>>>(*p_);
    return cuda_check(cudaGetLastError(), "gemm_tcgen05_kernel launch");
  }
  const int max_pairs = wide ? ds->wide_clusters : ds->pair_clusters;
  const int pairs = total < max_pairs ? total : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(wide ? Cfg<true, true>::THREADS : Cfg<true>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = wide ? Cfg<true, true>::SMEM : Cfg<true>::SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (wide)
    return cuda_check(cudaLaunchKernelEx(&cfg, gemm_tcgen05_kernel<true, true>, *p_), "gemm_tcgen05_kernel<wide> launch");
  return cuda_check(cudaLaunchKernelEx(&cfg, gemm_tcgen05_kernel<true>, *p_), "gemm_tcgen05_kernel<pair> launch");
}

}  // namespace ttl

// ------------------------------------------------------------------ C entry point

extern "C" int ttl_gemm(int64_t M, int64_t N, int64_t K, const ttl_bf16* A, int64_t lda, int a_kmajor,
                        const ttl_bf16* B, int64_t ldb, int b_kmajor, void* D, int64_t ldd, int d_fp32,
                        void* stream) {
  using namespace ttl;
  if (M < 0 || N < 0 || K < 0) return set_error(TTL_ERR_ARG, "ttl_gemm: negative extent");
  if (M == 0 || N == 0) return TTL_OK;
  if (!D) return set_error(TTL_ERR_ARG, "ttl_gemm: null D");
  if (N % 8 || K % 8) return set_error(TTL_ERR_SHAPE, "ttl_gemm: N and K must be multiples of 8");
  if (!aligned16(D) || (ldd * (d_fp32 ? 4 : 2)) % 16) return set_error(TTL_ERR_ALIGN, "ttl_gemm: D not 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K > 0 && (!A || !B)) return set_error(TTL_ERR_ARG, "ttl_gemm: null operand");
  if (K == 0) {
    // Empty contraction: D = 0.
    if (ldd == N) return fill_zero(D, static_cast<size_t>(M * N) * (d_fp32 ? 4 : 2), s);
    for (int64_t r = 0; r < M; ++r) {
      int rc = fill_zero(static_cast<char*>(D) + r * ldd * (d_fp32 ? 4 : 2), N * (d_fp32 ? 4 : 2), s);
      if (rc) return rc;
    }
    return TTL_OK;
  }
  GemmBatch b;
  const int ma = a_kmajor ? b.add_map(A, M, K, lda, false) : b.add_map(A, K, M, lda, true);
  const int mb = b_kmajor ? b.add_map(B, N, K, ldb, false) : b.add_map(B, K, N, ldb, true);
  Problem* p = b.add_problem(M, N, !a_kmajor, !b_kmajor, d_fp32 ? EPI_F32 : EPI_BF16, false);
  if (b.error()) return b.error();
  p->out0 = D;
  p->ld_out = ldd;
  b.add_seg(p, ma, 0, mb, -1, 0, K);
  return b.launch(s);
}

// The forward core of the head-split attention block in one kernel: for every (shard, query
// head, 128-query tile) one CTA computes the causal softmax probabilities P of its rows and
// O = P V, with the scores held in tensor memory and never written to HBM.
//
// Source: "v4:Tensor Parallel 与 Sequence Parallel", section "Attention:按 head 切" (each card
// computes its heads' attention alone).  The attention itself is causal scaled dot-product
// attention, scale 1/sqrt(d), query head j reading KV head j / (n_q / n_kv).
//
// Two passes over the key tiles 0..qt of query tile qt (128 keys each):
//   pass 1: S = Q K^T (tcgen05, fp32 in TMEM), two key tiles per 256-column MMA group; per row the
//           max and the sum of 2^(s log2e/sqrt(d) - max) over the keys <= the query -- exact row
//           statistics, so P needs no later rescaling;
//   pass 2: S again; P = 2^(s log2e/sqrt(d) - M - log2 sum) as bf16, written to tensor memory (the
//           A operand of O += P V) and to a shared tile that a TMA store writes to HBM (saved
//           for the backward).
// The probabilities the backward reads are therefore written once; nothing re-reads them here.
//
// Roles (352 threads): warp 0 issues TMA loads (Q once; then the pairs (K_0, K_1), (K_2, K_3), ...
// for pass 1, each filling two adjacent slots, and K_0, K_1, V_0, K_2, V_1, ... -- K a tile ahead
// of V -- for pass 2 through a 4-slot ring); warp 1 issues the MMAs; warp 10 issues the TMA stores of P; warps 2..9 run the
// softmax: two warps per TMEM lane quadrant, each on half of a score group's keys (and, at the
// end, half of O's d columns).  In pass 2 the MMA warp
// issues whichever is ready first, the next S or the next P V, so the softmax of tile j
// overlaps the previous tile's P V, and it never waits for a store.  Every wait is bounded
// (TTL_ERR_TIMEOUT on expiry).
//
// Layouts: Q, K tiles K-major (d contiguous, 64-column 128-byte-swizzled boxes of 128 rows);
// V tiles MN-major (64 d x 64 keys boxes).  Pass 1: TMEM columns [0,256) and [256,512) are its two
// 256-key score buffers.  Pass 2: [0,128) and [128,256) are the two score buffers, [256, 256 + d)
// the O accumulator, [384,448) and [448,512) the two P buffers (bf16, keys 2i and 2i + 1 in
// column i).  The MMAs here are bound by shared-memory bandwidth, so P V
// reads P from tensor memory; the shared copy of P only feeds the coalesced TMA store.

#include <cmath>
#include <cstring>
#include <mutex>

#include "ttl_device.cuh"
#include "ttl_internal.h"

namespace ttl {
namespace {

constexpr int kBQ = 128;            // queries per CTA
constexpr int kBKV = 128;           // keys per tile
constexpr int kRing = 4;            // K / V slots
constexpr int kThreads = 320;
// Every core adds a warp of its own for its P traffic (the forward's stores, the backward's
// loads): a second polling thread inside the producer warp would run interleaved with it.
constexpr int kCoreThreads = kThreads + 32;
constexpr int kTmemCols = 512;

struct CoreParams {
  CUtensorMap q[kMaxShards];   // Q_i [T, n_q/t d], box 64 x 128
  CUtensorMap k[kMaxShards];   // K_i [T, n_kv/t d], box 64 x 128
  CUtensorMap v[kMaxShards];   // V_i [T, n_kv/t d], box 64 x 64 (MN-major B operand)
  CUtensorMap pm[kMaxShards];  // P_i as [n_q/t][T][T], box 64 x 128 x 1 (TMA stores of P tiles)
  __nv_bfloat16* O[kMaxShards];   // [T, n_q/t d]
  int t, nql, grp, T, ntq;         // ntq = query tiles per head
  float k_log2;                    // log2(e) / sqrt(d)
  int* status;
  uint64_t timeout_ns;
};

template <int D>
struct CoreCfg {
  static constexpr int KB = D / 64;                       // 64-wide d blocks
  static constexpr int Q_BYTES = KB * kBQ * 128;          // 16 KiB per d block
  static constexpr int SLOT = KB * kBKV * 128;            // a K tile or a V tile
  static constexpr int OFF_Q = 0;
  static constexpr int P_BYTES = kBQ * kBKV * 2;          // 32 KiB: a P tile on its way to HBM
  static constexpr int OFF_RING = OFF_Q + Q_BYTES;
  static constexpr int OFF_P = OFF_RING + kRing * SLOT;
  // float2 [2][128] row-statistics exchange between the two passes, in the P buffers (which
  // pass 2 only writes after every softmax warp has read it)
  static constexpr int OFF_XCH = OFF_P;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;       // barriers + alignment slack
  static_assert(SMEM <= 232448, "shared memory beyond the per-CTA limit");
  // tensor memory: two score buffers, O, two P buffers (bf16, two per 32-bit column)
  static constexpr int T_O = 2 * kBKV;
  static constexpr int T_P = 2 * kBKV + 128;
  static_assert(T_P + 2 * (kBKV / 2) <= kTmemCols, "tensor memory layout");
};


__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Bulk tensor store shared -> global of one box; completion tracked by bulk async-groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* smem_src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}


// Folds 64 scores of one row (r0: keys 0..31, r1: keys 32..63 of the chunk, fp32 bits) into
// the row's running max m and sum l of 2^(s k - m); only the first nv keys count (nv <= 0: none).
__device__ __forceinline__ void row_stats64(const uint32_t (&r0)[32], const uint32_t (&r1)[32], int nv, float k,
                                            float& m, float& l) {
  if (nv >= 64) {   // below the diagonal: no mask
    // Three-input max and packed fp32 pairs: the same values and sums as the scalar form
    // (four running maxima, four partial sums over the same elements), fewer instructions.
    float x0 = -INFINITY, x1 = -INFINITY, x2 = -INFINITY, x3 = -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      x0 = fmax3(x0, __uint_as_float(r0[e]), __uint_as_float(r0[e + 2]));
      x1 = fmax3(x1, __uint_as_float(r0[e + 1]), __uint_as_float(r0[e + 3]));
      x2 = fmax3(x2, __uint_as_float(r1[e]), __uint_as_float(r1[e + 2]));
      x3 = fmax3(x3, __uint_as_float(r1[e + 1]), __uint_as_float(r1[e + 3]));
    }
    const float mnew = fmaxf(m, fmaxf(fmaxf(x0, x1), fmaxf(x2, x3)) * k);
    const float nm = -mnew;
    const uint64_t k2 = f2_pack(k, k), nm2 = f2_pack(nm, nm);
    uint64_t s01 = 0, s23 = 0;   // (s0, s1) and (s2, s3), all 0.0f
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const float2 a = f2_unpack(ffma2(f2_pack(__uint_as_float(r0[e]), __uint_as_float(r0[e + 1])), k2, nm2));
      const float2 b = f2_unpack(ffma2(f2_pack(__uint_as_float(r1[e]), __uint_as_float(r1[e + 1])), k2, nm2));
      s01 = fadd2(s01, f2_pack(ex2_approx(a.x), ex2_approx(a.y)));
      s23 = fadd2(s23, f2_pack(ex2_approx(b.x), ex2_approx(b.y)));
    }
    const float2 p01 = f2_unpack(s01), p23 = f2_unpack(s23);
    l = l * ex2_approx(m - mnew) + ((p01.x + p01.y) + (p23.x + p23.y));
    m = mnew;
  } else if (nv > 0) {
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      mx = fmaxf(mx, e < nv ? __uint_as_float(r0[e]) : -INFINITY);
      mx = fmaxf(mx, e + 32 < nv ? __uint_as_float(r1[e]) : -INFINITY);
    }
    const float mnew = fmaxf(m, mx * k);
    const float nm = -mnew;
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      s0 += e < nv ? ex2_approx(fmaf(__uint_as_float(r0[e]), k, nm)) : 0.0f;
      s1 += e + 32 < nv ? ex2_approx(fmaf(__uint_as_float(r1[e]), k, nm)) : 0.0f;
    }
    l = l * ex2_approx(m - mnew) + (s0 + s1);
    m = mnew;
  }
}

template <int D>
__global__ void __launch_bounds__(kCoreThreads, 1) attn_fwd_core_kernel(const __grid_constant__ CoreParams P) {
  using C = CoreCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sRing = smem + C::OFF_RING;
  uint8_t* sP = smem + C::OFF_P;
  float2* xch = reinterpret_cast<float2*>(smem + C::OFF_XCH);
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* ring_full = q_full + 1;
  uint64_t* ring_empty = ring_full + kRing;
  uint64_t* s_full = ring_empty + kRing;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* p_empty = p_full + 2;
  uint64_t* o_full = p_empty + 2;
  uint64_t* done_bar = o_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert((1 + 2 * kRing + 8 + 2) * 8 + 8 <= 256, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Heaviest query tiles first: block b takes tile ntq - 1 - b / (t n_q/t) of head b % (t n_q/t).
  const int heads = P.t * P.nql;
  const int qt = P.ntq - 1 - static_cast<int>(blockIdx.x) / heads;
  const int hh = static_cast<int>(blockIdx.x) % heads;
  const int shard = hh / P.nql;
  const int c = hh % P.nql;                 // query head within the shard
  const int g = c / P.grp;                  // its KV head within the shard
  const int q0 = qt * kBQ;
  const int ntiles = qt + 1;   // key tiles 0..qt (qt * 128 < T)
  const int npairs = (ntiles + 1) >> 1;   // pass-1 score groups of two key tiles
  const int p1_pos = 2 * npairs;          // ring positions of pass 1
  // Pass-2 ring positions: K_0, K_1, V_0, K_2, V_1, ..., K_(n-1), V_(n-2), V_(n-1).  V_j's slot
  // frees only when P_(j-2) V_(j-2) is done, and the producer fills positions in order, so with
  // K_(j+1) behind V_j the score tile S_(j+1) would wait for that P V; K one tile ahead of V
  // breaks the chain.  Each slot still fills and frees in position order.
  auto p2_k_pos = [&](int j) { return p1_pos + (j == 0 ? 0 : 2 * j - 1); };
  auto p2_v_pos = [&](int j) { return p1_pos + (j == ntiles - 1 ? 2 * ntiles - 1 : 2 * j + 2); };
  int* status = P.status;
  const uint64_t tmo = P.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], 8);   // every softmax warp
      mbar_init(&p_full[b], 8);
      mbar_init(&p_empty[b], 2);   // the P V MMAs (TMEM P) and the TMA store (shared P) have read it
    }
    mbar_init(o_full, 1);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&P.q[shard]);
    tma_prefetch_map(&P.k[shard]);
    tma_prefetch_map(&P.v[shard]);
    tma_prefetch_map(&P.pm[shard]);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
      for (int kb = 0; kb < C::KB; ++kb) tma_load_2d(sQ + kb * 16384, &P.q[shard], q_full, c * D + kb * 64, q0);
      // ring sequence: pass 1 the pairs (K_0, K_1), (K_2, K_3), ... two positions each; pass 2
      // K_0, K_1, V_0, K_2, V_1, ..., K_(n-1), V_(n-2), V_(n-1)
      const int nseq = p1_pos + 2 * ntiles;
      int issued = 0;
      for (int seq = 0; ok && seq < nseq; ++seq) {
        const int slot = seq % kRing;
        const uint32_t ph = static_cast<uint32_t>(seq / kRing) & 1u;
        if (!mbar_wait(&ring_empty[slot], ph ^ 1u, abort_flag, status, tmo)) {
          ok = false;
          break;
        }
        uint8_t* dst = sRing + slot * C::SLOT;
        mbar_arrive_expect_tx(&ring_full[slot], C::SLOT);
        if (seq < p1_pos) {
          // Pass-1 pair m fills the slot pair starting at slot 2m % kRing (even, so the two slots
          // are adjacent) as one 256-row K-major operand: box (K_{2m+x}, d block kb) at byte
          // kb * 32 KiB + x * 16 KiB.  Position 2m + h carries the boxes in [h SLOT, (h+1) SLOT).
          // A K_{2m+1} past the last tile lies above the diagonal (or past T: zero fill); its
          // scores are masked.
          const int m = seq >> 1, h = seq & 1;
          uint8_t* pair_base = dst - h * C::SLOT;
          for (int kb = 0; kb < C::KB; ++kb)
            for (int x = 0; x < 2; ++x) {
              const int off = kb * 32768 + x * 16384;
              if (off / C::SLOT == h)
                tma_load_2d(pair_base + off, &P.k[shard], &ring_full[slot], g * D + kb * 64, (2 * m + x) * kBKV);
            }
          ++issued;
          continue;
        }
        // Pass 2 order: K_0, then K_(j+1) before V_j (K runs a tile ahead, see p2_k_pos).
        const int k2 = seq - p1_pos;
        const bool is_v = k2 != 0 && (k2 == 2 * ntiles - 1 || (k2 & 1) == 0);
        const int j = k2 == 0 ? 0 : (k2 == 2 * ntiles - 1 ? ntiles - 1 : (is_v ? k2 / 2 - 1 : (k2 + 1) / 2));
        if (!is_v) {
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_2d(dst + kb * 16384, &P.k[shard], &ring_full[slot], g * D + kb * 64, j * kBKV);
        } else {
          // two 64-key blocks, each KB boxes of 64 d x 64 keys
          for (int kk = 0; kk < 2; ++kk)
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_2d(dst + (kk * C::KB + kb) * 8192, &P.v[shard], &ring_full[slot], g * D + kb * 64,
                          j * kBKV + kk * 64);
        }
        ++issued;
      }
      // No copy may still be landing when the CTA leaves: wait (bounded) for the last loads.
      int dummy_abort = 0;
      mbar_wait(q_full, 0, reinterpret_cast<volatile int*>(&dummy_abort), status, tmo);
      const int pending = issued < kRing ? issued : kRing;
      for (int i = issued - pending; i < issued; ++i)
        mbar_wait(&ring_full[i % kRing], static_cast<uint32_t>(i / kRing) & 1u,
                  reinterpret_cast<volatile int*>(&dummy_abort), status, tmo);
    }
    __syncwarp();
  } else if (warp == kThreads / 32) {
    // ------------------------------------------------------------------ P stores (own warp)
    if (lane == 0) {
      // P_j leaves for HBM (two 64-key boxes) as soon as the softmax has written it.  This thread
      // alone waits for each store to have read the shared tile, so the MMA warp never waits on
      // a store; its arrival is the second one the P buffer needs (the first: the P V MMAs).
      bool ok = true;
      for (int j = 0; ok && j < ntiles; ++j) {
        const int b = j & 1;
        ok = mbar_wait(&p_full[b], static_cast<uint32_t>(j >> 1) & 1u, abort_flag, status, tmo);
        if (!ok) break;
        tma_store_3d(&P.pm[shard], sP + b * C::P_BYTES, j * kBKV, q0, c);
        tma_store_3d(&P.pm[shard], sP + b * C::P_BYTES + 16384, j * kBKV + 64, q0, c);
        bulk_commit_group();
        bulk_wait_group_read<0>();
        mbar_arrive(&p_empty[b]);
      }
      bulk_wait_group_all();   // every store complete before the CTA's shared memory goes away
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0, abort_flag, status, tmo);
      tc_fence_after_sync();
      const uint32_t ring0 = smem_u32(sRing);
      const uint64_t qd = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint32_t idesc_s = idesc_bf16_f32(kBQ, kBKV, false, false);
      const uint32_t idesc_o = idesc_bf16_f32(kBQ, D, false, true);
      int sj = 0;            // S tiles issued (both passes), selects the score buffer
      // Pass 2's S_ns, issued once the caller has seen its K tile loaded and its score buffer free.
      // The K slot is released by a softmax thread once S_ns is complete (one commit fewer here).
      auto issue_s = [&](int slot) {
        const int b = sj & 1;
        const uint64_t kd = smem_desc_sw128(ring0 + slot * C::SLOT, 16, 1024);
        for (int kb = 0; kb < C::KB; ++kb) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = desc_advance(qd, kb * 16384 + kk * 32);
            const uint64_t bd = desc_advance(kd, kb * 16384 + kk * 32);
            umma_bf16(tmem_base + b * kBKV, ad, bd, idesc_s, (kb | kk) ? 1u : 0u);
          }
        }
        umma_commit(&s_full[b]);
        ++sj;
        return true;
      };
      // Ring position pos (the producer's load order) lives in slot pos % kRing.
      auto wait_pos = [&](int pos) {
        const int slot = pos % kRing;
        if (!mbar_wait(&ring_full[slot], static_cast<uint32_t>(pos / kRing) & 1u, abort_flag, status, tmo))
          return -1;
        tc_fence_after_sync();
        return slot;
      };
      // pass 1: scores only, 256 keys per group (K_2m, K_2m+1 at positions 2m, 2m + 1) into a
      // 256-column score buffer at column 256 b: O and the P buffers are not used yet, so the
      // whole tensor memory holds two such buffers.  Twice the work per MMA instruction halves
      // this thread's waits, commits and bookkeeping per key.
      const uint32_t idesc_w = idesc_bf16_f32(kBQ, 2 * kBKV, false, false);
      for (int m = 0; ok && m < npairs; ++m) {
        const int s0 = wait_pos(2 * m);
        const int s1 = s0 < 0 ? -1 : wait_pos(2 * m + 1);
        const int b = sj & 1;
        ok = s1 >= 0 && mbar_wait(&s_empty[b], (static_cast<uint32_t>(sj >> 1) & 1u) ^ 1u, abort_flag, status, tmo);
        if (!ok) break;
        tc_fence_after_sync();
        const uint64_t kd = smem_desc_sw128(ring0 + s0 * C::SLOT, 16, 1024);
        for (int kb = 0; kb < C::KB; ++kb) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = desc_advance(qd, kb * 16384 + kk * 32);
            const uint64_t bd = desc_advance(kd, kb * 32768 + kk * 32);
            umma_bf16(tmem_base + b * 2 * kBKV, ad, bd, idesc_w, (kb | kk) ? 1u : 0u);
          }
        }
        umma_commit(&s_full[b]);   // a softmax thread releases both K slots once this completes
        ++sj;
      }
      // Pass 2's score buffers (columns [0, 256)) overlap pass 1's buffer 0, whose last group may
      // be the one just issued: wait until the softmax has read it.
      if (ok) ok = mbar_wait(&s_empty[(sj - 1) & 1], static_cast<uint32_t>((sj - 1) >> 1) & 1u, abort_flag, status, tmo);
      // pass 2: issue whichever is ready first -- the next score tile S_ns (K_ns at ring position
      // p1 + 2 ns, a free score buffer) or the next P_np V_np (V_np at p1 + 2 np + 1, P_np
      // written) -- so that a P V never waits behind a late K tile, nor an S behind a late softmax.
      int ns = 0, np = 0;
      // The wall-clock timeout is measured from the start of an idle stretch: the timer is read
      // when polling first finds nothing to issue, never on the path between two MMA groups
      // (a read costs about 200 cycles, during which the tensor pipe would run dry).
      uint64_t t_idle = 0;
      bool idle = false;
      while (ok && np < ntiles) {
        bool progress = false;
        if (ns < ntiles) {
          const int pos = p2_k_pos(ns);
          const int slot = pos % kRing;
          const int b = sj & 1;
          if (mbar_test_wait(&ring_full[slot], static_cast<uint32_t>(pos / kRing) & 1u) &&
              mbar_test_wait(&s_empty[b], (static_cast<uint32_t>(sj >> 1) & 1u) ^ 1u)) {
            tc_fence_after_sync();
            ok = issue_s(slot);   // both conditions hold: no wait inside
            ++ns;
            progress = true;
          }
        }
        if (ok && np < ns) {
          const int pos = p2_v_pos(np);
          const int vslot = pos % kRing;
          const int b = np & 1;
          if (mbar_test_wait(&ring_full[vslot], static_cast<uint32_t>(pos / kRing) & 1u) &&
              mbar_test_wait(&p_full[b], static_cast<uint32_t>(np >> 1) & 1u)) {
            tc_fence_after_sync();
            // O += P_np V_np with P from tensor memory (A operand, 8 columns per 16 keys)
            const uint64_t vd = smem_desc_sw128(ring0 + vslot * C::SLOT, 8192, 1024);
            for (int kk2 = 0; kk2 < 2; ++kk2) {          // 64-key blocks
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t at = tmem_base + C::T_P + b * (kBKV / 2) + (kk2 * 4 + kk) * 8;
                const uint64_t bd = desc_advance(vd, kk2 * C::KB * 8192 + kk * 2048);
                umma_bf16_ts(tmem_base + C::T_O, at, bd, idesc_o, (np | kk2 | kk) ? 1u : 0u);
              }
            }
            umma_commit(&ring_empty[vslot]);
            umma_commit(&p_empty[b]);                  // the MMAs have read P_np
            ++np;
            progress = true;
          }
        }
        if (progress) {
          idle = false;
        } else if (*abort_flag) {
          ok = false;
        } else if (!idle) {
          idle = true;
          t_idle = globaltimer_ns();
        } else if (globaltimer_ns() - t_idle > tmo) {
          if (status) atomicCAS(status, 0, TTL_ERR_TIMEOUT);
          *abort_flag = 1;
          ok = false;
        }
      }
      if (ok) umma_commit(o_full);
      // Every MMA issued here must finish before TMEM is released.
      umma_commit(done_bar);
      int dummy_abort = 0;
      mbar_wait(done_bar, 0, reinterpret_cast<volatile int*>(&dummy_abort), status, tmo);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;          // pass 2: keys [64 half, 64 half + 64) of each tile
    const int r = quad * 32 + lane;            // row within the query tile
    const int q = q0 + r;                      // query index
    const bool row_ok = q < P.T;
    const float k = P.k_log2;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    bool ok = true;
    int sj = 0;
    // pass 1: running max and sum over the keys <= q, 256 keys per score group (this warp: 128
    // of them, in two chunks of 64)
    float m = -INFINITY, l = 0.0f;
    for (int pg = 0; pg < npairs; ++pg, ++sj) {
      const int b = sj & 1;
      ok = ok && mbar_wait(&s_full[b], static_cast<uint32_t>(sj >> 1) & 1u, abort_flag, status, tmo);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      // The group's MMAs are complete, so its two K tiles (ring positions 2 pg, 2 pg + 1) are free.
      if (warp == 2 && lane == 0) {
        mbar_arrive(&ring_empty[(2 * pg) % kRing]);
        mbar_arrive(&ring_empty[(2 * pg + 1) % kRing]);
      }
      tc_fence_after_sync();
      uint32_t ra[32], rb[32], rc[32], rd[32];
      const uint32_t col = lane_base + b * 2 * kBKV + half * kBKV;
      tmem_ld_32x32b_x32(col, ra);
      tmem_ld_32x32b_x32(col + 32, rb);
      tmem_ld_32x32b_x32(col + 64, rc);
      tmem_ld_32x32b_x32(col + 96, rd);
      tmem_ld_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[b]);
      const int key0 = pg * 2 * kBKV + half * kBKV;
      row_stats64(ra, rb, q - key0 + 1, k, m, l);
      row_stats64(rc, rd, q - key0 - 63, k, m, l);
    }
    // combine the two halves of each row (every softmax warp reaches this barrier)
    xch[half * kBQ + r] = make_float2(m, l);
    named_bar_sync(1, 256);
    {
      const float2 o = xch[(1 - half) * kBQ + r];
      const float M = fmaxf(m, o.x);
      const float L = (m == -INFINITY ? 0.0f : l * ex2_approx(m - M)) +
                      (o.x == -INFINITY ? 0.0f : o.y * ex2_approx(o.x - M));
      m = M;
      l = L;
    }
    named_bar_sync(1, 256);   // every half has read the exchange before P overwrites it
    // P = 2^(s k - m) / l = 2^(s k - (m + log2 l)): the normalisation rides in the exponent.  A row
    // past the end of the sequence (never stored) gets finite values.
    const float nm = row_ok ? -(m + __log2f(l)) : 0.0f;
    // pass 2: probabilities, into the TMEM P buffer the MMA warp feeds to P V, and into a
    // 128-byte-swizzled shared tile that the MMA warp stores to HBM by TMA
    uint8_t* my_row = sP + half * 16384 + (r >> 3) * 1024 + (r & 7) * 128;
    const uint32_t p_tmem = lane_base + C::T_P + half * 32;
    for (int j = 0; ok && j < ntiles; ++j, ++sj) {
      const int b = sj & 1;
      ok = mbar_wait(&s_full[b], static_cast<uint32_t>(sj >> 1) & 1u, abort_flag, status, tmo);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      // S_j is complete: its K tile's ring slot is free.
      if (warp == 2 && lane == 0) mbar_arrive(&ring_empty[p2_k_pos(j) % kRing]);
      tc_fence_after_sync();
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(lane_base + b * kBKV + half * 64, r0);
      tmem_ld_32x32b_x32(lane_base + b * kBKV + half * 64 + 32, r1);
      tmem_ld_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[b]);
      const int nv = q - (j * kBKV + half * 64) + 1;
      uint32_t w[32];   // keys 2i, 2i + 1 of this warp's 64 in word i
      if (nv >= 64) {   // below the diagonal: no mask
        const uint64_t k2 = f2_pack(k, k), nm2 = f2_pack(nm, nm);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t a0 = i < 16 ? r0[2 * i] : r1[2 * i - 32];
          const uint32_t a1 = i < 16 ? r0[2 * i + 1] : r1[2 * i - 31];
          const float2 x = f2_unpack(ffma2(f2_pack(__uint_as_float(a0), __uint_as_float(a1)), k2, nm2));
          w[i] = pack_bf16x2(ex2_approx(x.x), ex2_approx(x.y));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t a0 = i < 16 ? r0[2 * i] : r1[2 * i - 32];
          const uint32_t a1 = i < 16 ? r0[2 * i + 1] : r1[2 * i - 31];
          w[i] = pack_bf16x2(2 * i < nv ? ex2_approx(fmaf(__uint_as_float(a0), k, nm)) : 0.0f,
                             2 * i + 1 < nv ? ex2_approx(fmaf(__uint_as_float(a1), k, nm)) : 0.0f);
        }
      }
      // the P buffers are free once the P V and the store that read them two tiles ago are done
      const int pb = j & 1;
      ok = mbar_wait(&p_empty[pb], static_cast<uint32_t>((j >> 1) & 1) ^ 1u, abort_flag, status, tmo);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      tmem_st_32x32b_x32(p_tmem + pb * (kBKV / 2), w);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(my_row + pb * C::P_BYTES + ((u ^ (r & 7)) << 4)) =
            make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
    }
    // O = (sum_j P_j V_j): this warp stores its half of the d columns
    if (ok) ok = mbar_wait(o_full, 0, abort_flag, status, tmo);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after_sync();
      __nv_bfloat16* Orow = P.O[shard] + static_cast<int64_t>(row_ok ? q : 0) * (P.nql * D) + c * D + half * (D / 2);
#pragma unroll
      for (int cc = 0; cc < D / 2; cc += 32) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(lane_base + C::T_O + half * (D / 2) + cc, o);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(Orow + cc + u * 8) = make_uint4(
                pack_bf16x2(__uint_as_float(o[u * 8 + 0]), __uint_as_float(o[u * 8 + 1])),
                pack_bf16x2(__uint_as_float(o[u * 8 + 2]), __uint_as_float(o[u * 8 + 3])),
                pack_bf16x2(__uint_as_float(o[u * 8 + 4]), __uint_as_float(o[u * 8 + 5])),
                pack_bf16x2(__uint_as_float(o[u * 8 + 6]), __uint_as_float(o[u * 8 + 7])));
        }
      }
    }
    tc_fence_before_sync();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ backward core

struct BwdParams {
  CUtensorMap dO[kMaxShards];    // dO_i [T, n_q/t d], box 64 x 128 (A of dP)
  CUtensorMap v[kMaxShards];     // V_i [T, n_kv/t d], box 64 x 128 (K-major B of dP = dO V^T)
  CUtensorMap kmn[kMaxShards];   // K_i [T, n_kv/t d], box 64 x 64 (MN-major B of dQ = dS K)
  CUtensorMap p[kMaxShards];     // P_i as [n_q/t][T][T], box 64 x 128 x 1 (loads)
  __nv_bfloat16* dQ[kMaxShards];  // [T, n_q/t d]
  const float* D;                 // rowsum(dO O), [t][n_q/t][T]
  int t, nql, grp, T, ntq;
  float scale;                    // 1 / sqrt(d)
  int* status;
  uint64_t timeout_ns;
};

template <int D>
struct BwdCfg {
  static constexpr int KB = D / 64;
  static constexpr int RING = 5;                          // V / K slots
  static constexpr int A_BYTES = KB * kBQ * 128;          // the dO tile
  static constexpr int SLOT = KB * kBKV * 128;            // a V tile or a K tile
  static constexpr int P_BYTES = kBQ * kBKV * 2;          // a P tile, read by the dS warps alone
  static constexpr int OFF_A = 0;
  static constexpr int OFF_RING = OFF_A + A_BYTES;
  static constexpr int OFF_P = OFF_RING + RING * SLOT;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static_assert(SMEM <= 232448, "shared memory beyond the per-CTA limit");
  // tensor memory: two dP buffers, the dQ accumulator, two dS buffers (bf16, keys 2i and 2i + 1
  // in column i: the A operand of dQ += dS K)
  static constexpr int T_DQ = 2 * kBKV;
  static constexpr int T_DS = 2 * kBKV + D;
  static_assert(T_DS + 2 * (kBKV / 2) <= kTmemCols, "tensor memory layout");
};

// Asks L2 to fetch one box ahead of its load (HBM latency hidden without shared memory).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// dQ: for every (shard, query head, 128-query tile) over the key tiles 0..qt (128 keys each):
//   dP_j = dO_c V_j^T (tcgen05, TMEM); the P_j tile arrives by TMA into a shared buffer; the
//   dS warps read it (each thread its own row) and write dS_j = P_j (dP_j - D) / sqrt(d) (P is
//   zero above the diagonal, so is dS) into tensor memory, where dQ += dS_j K_j reads it as the
//   A operand.  dQ accumulates in TMEM and is stored at the end.  The P tile is free as soon as
//   the dS warps hold it in registers, so one buffer suffices, and the shared memory it saves
//   holds a fifth V / K slot: the ring's loads get more lead.
// Roles (352 threads): warp 0 loads dO, then V_j / K_j through the 5-slot ring; warp 10 loads
// the P tiles; warp 1 issues the MMAs (dP_j, then dQ_(j-1)); warps 2..9 compute dS, two per
// TMEM lane quadrant.
template <int D>
__global__ void __launch_bounds__(kCoreThreads, 1) attn_bwd_core_kernel(const __grid_constant__ BwdParams P) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sRing = smem + C::OFF_RING;
  uint8_t* sP = smem + C::OFF_P;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* ring_full = a_full + 1;
  uint64_t* ring_empty = ring_full + C::RING;
  uint64_t* dp_full = ring_empty + C::RING;
  uint64_t* dp_empty = dp_full + 2;
  uint64_t* pb_full = dp_empty + 2;            // the P tile in shared memory
  uint64_t* pb_empty = pb_full + 1;
  uint64_t* ds_full = pb_empty + 1;            // [2] dS in tensor memory
  uint64_t* ds_empty = ds_full + 2;            // [2]
  uint64_t* dq_full = ds_empty + 2;
  uint64_t* done_bar = dq_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert((1 + 2 * C::RING + 4 + 2 + 4 + 2) * 8 + 8 <= 256, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int heads = P.t * P.nql;
  const int qt = P.ntq - 1 - static_cast<int>(blockIdx.x) / heads;
  const int hh = static_cast<int>(blockIdx.x) % heads;
  const int shard = hh / P.nql;
  const int c = hh % P.nql;
  const int g = c / P.grp;
  const int q0 = qt * kBQ;
  const int ntiles = qt + 1;
  int* status = P.status;
  const uint64_t tmo = P.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    for (int s = 0; s < C::RING; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&dp_full[b], 1);
      mbar_init(&dp_empty[b], 8);
      mbar_init(&ds_full[b], 8);
      mbar_init(&ds_empty[b], 1);   // the dQ MMAs have read dS
    }
    mbar_init(pb_full, 1);
    mbar_init(pb_empty, 8);         // the eight dS warps have read the P tile
    mbar_init(dq_full, 1);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&P.dO[shard]);
    tma_prefetch_map(&P.v[shard]);
    tma_prefetch_map(&P.kmn[shard]);
    tma_prefetch_map(&P.p[shard]);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- dO, then V_j / K_j
      bool ok = true;
      mbar_arrive_expect_tx(a_full, C::A_BYTES);
      for (int kb = 0; kb < C::KB; ++kb) tma_load_2d(sA + kb * 16384, &P.dO[shard], a_full, c * D + kb * 64, q0);
      int issued = 0;
      for (int pos = 0; ok && pos < 2 * ntiles; ++pos) {
        const int slot = pos % C::RING;
        if (!mbar_wait(&ring_empty[slot], (static_cast<uint32_t>(pos / C::RING) & 1u) ^ 1u, abort_flag, status, tmo)) {
          ok = false;
          break;
        }
        uint8_t* dst = sRing + slot * C::SLOT;
        const int j = pos >> 1;
        mbar_arrive_expect_tx(&ring_full[slot], C::SLOT);
        if ((pos & 1) == 0) {   // V_j, K-major
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_2d(dst + kb * 16384, &P.v[shard], &ring_full[slot], g * D + kb * 64, j * kBKV);
        } else {                // K_j, MN-major: two 64-key blocks of KB boxes
          for (int kk = 0; kk < 2; ++kk)
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_2d(dst + (kk * C::KB + kb) * 8192, &P.kmn[shard], &ring_full[slot], g * D + kb * 64,
                          j * kBKV + kk * 64);
        }
        ++issued;
      }
      int dummy_abort = 0;
      mbar_wait(a_full, 0, reinterpret_cast<volatile int*>(&dummy_abort), status, tmo);
      const int pending = issued < C::RING ? issued : C::RING;
      for (int i = issued - pending; i < issued; ++i)
        mbar_wait(&ring_full[i % C::RING], static_cast<uint32_t>(i / C::RING) & 1u,
                  reinterpret_cast<volatile int*>(&dummy_abort), status, tmo);
    }
    __syncwarp();
  } else if (warp == kThreads / 32) {
    // ------------------------------------------------------------------ P tiles (own warp)
    if (lane == 0) {
      bool ok = true;
      int started = 0;   // P tiles whose load was issued
      for (int j = 0; j < 2 && j < ntiles; ++j) {
        tma_prefetch_3d(&P.p[shard], j * kBKV, q0, c);
        tma_prefetch_3d(&P.p[shard], j * kBKV + 64, q0, c);
      }
      for (int j = 0; ok && j < ntiles; ++j) {
        if (j + 2 < ntiles) {   // two tiles ahead into L2
          tma_prefetch_3d(&P.p[shard], (j + 2) * kBKV, q0, c);
          tma_prefetch_3d(&P.p[shard], (j + 2) * kBKV + 64, q0, c);
        }
        if (!mbar_wait(pb_empty, (static_cast<uint32_t>(j) & 1u) ^ 1u, abort_flag, status, tmo)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(pb_full, C::P_BYTES);
        tma_load_3d(sP, &P.p[shard], pb_full, j * kBKV, q0, c);
        tma_load_3d(sP + 16384, &P.p[shard], pb_full, j * kBKV + 64, q0, c);
        ++started;
      }
      // No copy may still be landing when the CTA leaves: wait (bounded) for the latest load (an
      // earlier one completed before the buffer could be reused).
      int dummy_abort = 0;
      if (started > 0)
        mbar_wait(pb_full, static_cast<uint32_t>(started - 1) & 1u, reinterpret_cast<volatile int*>(&dummy_abort),
                  status, tmo);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(a_full, 0, abort_flag, status, tmo);
      tc_fence_after_sync();
      const uint64_t dod = smem_desc_sw128(smem_u32(sA), 16, 1024);   // the dO tile (A of dP)
      const uint32_t ring0 = smem_u32(sRing);
      const uint32_t idesc_dp = idesc_bf16_f32(kBQ, kBKV, false, false);
      const uint32_t idesc_dq = idesc_bf16_f32(kBQ, D, false, true);
      auto wait_pos = [&](int pos) {
        const int slot = pos % C::RING;
        if (!mbar_wait(&ring_full[slot], static_cast<uint32_t>(pos / C::RING) & 1u, abort_flag, status, tmo))
          return -1;
        tc_fence_after_sync();
        return slot;
      };
      for (int j = 0; ok && j <= ntiles; ++j) {
        if (j < ntiles) {   // dP_j = dO V_j^T into score buffer j & 1
          const int b = j & 1;
          const int vslot = wait_pos(2 * j);
          if (vslot < 0 ||
              !mbar_wait(&dp_empty[b], (static_cast<uint32_t>(j >> 1) & 1u) ^ 1u, abort_flag, status, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t vd = smem_desc_sw128(ring0 + vslot * C::SLOT, 16, 1024);
          for (int kb = 0; kb < C::KB; ++kb) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = desc_advance(dod, kb * 16384 + kk * 32);
              const uint64_t bd = desc_advance(vd, kb * 16384 + kk * 32);
              umma_bf16(tmem_base + b * kBKV, ad, bd, idesc_dp, (kb | kk) ? 1u : 0u);
            }
          }
          umma_commit(&ring_empty[vslot]);
          umma_commit(&dp_full[b]);
        }
        if (j > 0) {        // dQ += dS_(j-1) K_(j-1)
          const int jp = j - 1;
          const int b = jp & 1;
          const int kslot = wait_pos(2 * jp + 1);
          if (kslot < 0 || !mbar_wait(&ds_full[b], static_cast<uint32_t>(jp >> 1) & 1u, abort_flag, status, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t kd = smem_desc_sw128(ring0 + kslot * C::SLOT, 8192, 1024);
          const uint32_t t_ds = tmem_base + C::T_DS + b * (kBKV / 2);
          for (int kk2 = 0; kk2 < 2; ++kk2) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {   // keys 64 kk2 + 16 kk .. +15: dS columns 32 kk2 + 8 kk
              const uint64_t bd = desc_advance(kd, kk2 * C::KB * 8192 + kk * 2048);
              umma_bf16_ts(tmem_base + C::T_DQ, t_ds + kk2 * 32 + kk * 8, bd, idesc_dq, (jp | kk2 | kk) ? 1u : 0u);
            }
          }
          umma_commit(&ring_empty[kslot]);
          umma_commit(&ds_empty[b]);                 // the MMAs have read dS_(j-1)
        }
      }
      if (ok) umma_commit(dq_full);
      umma_commit(done_bar);
      int dummy_abort = 0;
      mbar_wait(done_bar, 0, reinterpret_cast<volatile int*>(&dummy_abort), status, tmo);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ dS warps
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;
    const int q = q0 + r;
    const bool row_ok = q < P.T;
    const float Dq = row_ok ? P.D[(static_cast<int64_t>(shard) * P.nql + c) * P.T + q] : 0.0f;
    const float scale = P.scale;
    const uint64_t nDs2 = f2_pack(-Dq * scale, -Dq * scale), scale2 = f2_pack(scale, scale);
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    const uint8_t* my_row = sP + half * 16384 + (r >> 3) * 1024 + (r & 7) * 128;
    bool ok = true;
    for (int j = 0; ok && j < ntiles; ++j) {
      const int b = j & 1;
      ok = mbar_wait(&dp_full[b], static_cast<uint32_t>(j >> 1) & 1u, abort_flag, status, tmo);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(lane_base + b * kBKV + half * 64, r0);
      tmem_ld_32x32b_x32(lane_base + b * kBKV + half * 64 + 32, r1);
      tmem_ld_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dp_empty[b]);
      ok = mbar_wait(pb_full, static_cast<uint32_t>(j) & 1u, abort_flag, status, tmo);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      uint32_t pv[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 pw = *reinterpret_cast<const uint4*>(my_row + ((u ^ (r & 7)) << 4));
        pv[4 * u] = pw.x;
        pv[4 * u + 1] = pw.y;
        pv[4 * u + 2] = pw.z;
        pv[4 * u + 3] = pw.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(pb_empty);   // P_j is in registers: the tile may be refilled
      // dS = (dP scale - D scale) P, two columns per packed fp32 instruction (one fma and one
      // multiply per pair).  P is zero above the diagonal.
      uint32_t ds[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int col = 2 * e;
        const uint64_t dp2 = f2_pack(__uint_as_float(col < 32 ? r0[col] : r1[col - 32]),
                                     __uint_as_float(col < 32 ? r0[col + 1] : r1[col - 31]));
        const uint64_t p2 = f2_pack(bf16_lo(pv[e]), bf16_hi(pv[e]));
        const float2 d2 = f2_unpack(fmul2(ffma2(dp2, scale2, nDs2), p2));
        ds[e] = pack_bf16x2(d2.x, d2.y);
      }
      if (j >= 2) {
        ok = mbar_wait(&ds_empty[b], (static_cast<uint32_t>(j >> 1) & 1u) ^ 1u, abort_flag, status, tmo);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
      }
      tmem_st_32x32b_x32(lane_base + C::T_DS + b * (kBKV / 2) + half * 32, ds);
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_full[b]);
    }
    if (ok) ok = mbar_wait(dq_full, 0, abort_flag, status, tmo);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after_sync();
      __nv_bfloat16* out = P.dQ[shard] + static_cast<int64_t>(row_ok ? q : 0) * (P.nql * D) + c * D + half * (D / 2);
#pragma unroll
      for (int cc = 0; cc < D / 2; cc += 32) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(lane_base + C::T_DQ + half * (D / 2) + cc, o);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(out + cc + u * 8) = make_uint4(
                pack_bf16x2(__uint_as_float(o[u * 8 + 0]), __uint_as_float(o[u * 8 + 1])),
                pack_bf16x2(__uint_as_float(o[u * 8 + 2]), __uint_as_float(o[u * 8 + 3])),
                pack_bf16x2(__uint_as_float(o[u * 8 + 4]), __uint_as_float(o[u * 8 + 5])),
                pack_bf16x2(__uint_as_float(o[u * 8 + 6]), __uint_as_float(o[u * 8 + 7])));
        }
      }
    }
    tc_fence_before_sync();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ dK and dV

struct KvParams {
  CUtensorMap q[kMaxShards];    // Q_i [T, n_q/t d], box 64 x 128 (MN-major B of dK)
  CUtensorMap dO[kMaxShards];   // dO_i [T, n_q/t d], box 64 x 128 (A of dP, MN-major B of dV)
  CUtensorMap v[kMaxShards];    // V_i [T, n_kv/t d], box 64 x 128 (K-major B of dP)
  CUtensorMap p[kMaxShards];    // P_i as [n_q/t][T][T], box 64 x 128 x 1
  __nv_bfloat16* dK[kMaxShards];  // [T, n_kv/t d]
  __nv_bfloat16* dV[kMaxShards];
  const float* D;                 // rowsum(dO O), [t][n_q/t][T]
  int t, nql, nkvl, grp, T, ntq;
  float scale;
  int* status;
  uint64_t timeout_ns;
};

template <int D>
struct KvCfg {
  static constexpr int KB = D / 64;
  static constexpr int V_BYTES = KB * kBKV * 128;         // the CTA's V tile
  static constexpr int SLOT = KB * kBQ * 128;             // a Q tile or a dO tile
  static constexpr int P_BYTES = kBQ * kBKV * 2;          // a P tile, overwritten in place by dS
  static constexpr int DO_SLOTS = 2;                      // dO_j: read by dP_j and dV_j
  static constexpr int P_BUFS = 3;                        // P_j, then dS_j: read until dK_j
  static constexpr int OFF_V = 0;
  static constexpr int OFF_DO = OFF_V + V_BYTES;
  static constexpr int OFF_Q = OFF_DO + DO_SLOTS * SLOT;  // one Q slot: Q_j is read by dK_j alone
  static constexpr int OFF_P = OFF_Q + SLOT;
  static constexpr int OFF_BAR = OFF_P + P_BUFS * P_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static_assert(SMEM <= 232448, "shared memory beyond the per-CTA limit");
};

// dK and dV: for every (shard, KV head g, 128-key tile kt), over the pairs (query head c of the
// group, query tile qt >= kt, the last tile first), with the queries as rows of every score tile:
//   dP = dO_c V^T (TMEM); the saved P tile arrives by TMA; dV += P^T dO_c reads it as an
//   MN-major operand; the softmax warps then overwrite it in place with
//   dS = P (dP - D) / sqrt(d) (zero above the diagonal, where P is zero); dK += dS^T Q_c.
// Neither P^T nor dS^T is ever formed: the MMAs read the [queries x keys] tiles as MN-major A
// operands, and the [queries x d] Q and dO tiles loaded K-major double as MN-major B operands.
// Roles (352 threads): warp 0 loads V once, then dO_(j+1) and Q_j (dO one pair ahead: dP_j needs
// dO_j at the start of pair j, dK_j needs Q_j only a pair later, so dO takes two slots and Q one);
// warp 10 loads P_j into three P buffers (a P buffer is busy from its load until dK_j has read
// dS_j, about two pairs); warp 1 issues dP_j, dV_j, then dK_(j-1); warps 2..9 compute dS (two per
// TMEM lane quadrant) and at the end store dK and dV.
template <int D>
__global__ void __launch_bounds__(kCoreThreads, 1) attn_bwd_kv_kernel(const __grid_constant__ KvParams P) {
  using C = KvCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sP = smem + C::OFF_P;
  uint64_t* v_full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* do_full = v_full + 1;              // [DO_SLOTS]
  uint64_t* do_empty = do_full + C::DO_SLOTS;  // [DO_SLOTS]
  uint64_t* q_full = do_empty + C::DO_SLOTS;
  uint64_t* q_empty = q_full + 1;
  uint64_t* dp_full = q_empty + 1;             // [2] the dP buffers in TMEM
  uint64_t* dp_empty = dp_full + 2;            // [2]
  uint64_t* pb_full = dp_empty + 2;            // [P_BUFS]
  uint64_t* pb_empty = pb_full + C::P_BUFS;    // [P_BUFS]
  uint64_t* pv_done = pb_empty + C::P_BUFS;    // [P_BUFS]
  uint64_t* ds_full = pv_done + C::P_BUFS;     // [P_BUFS]
  uint64_t* acc_full = ds_full + C::P_BUFS;
  uint64_t* done_bar = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert((1 + 2 * C::DO_SLOTS + 2 + 4 + 4 * C::P_BUFS + 2) * 8 + 8 <= 256, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Heaviest key tiles first: block b takes key tile b / (t n_kv/t) of KV head b % (t n_kv/t).
  const int kvheads = P.t * P.nkvl;
  const int kt = static_cast<int>(blockIdx.x) / kvheads;
  const int hh = static_cast<int>(blockIdx.x) % kvheads;
  const int shard = hh / P.nkvl;
  const int g = hh % P.nkvl;
  const int k0 = kt * kBKV;
  const int nqt = P.ntq - kt;               // query tiles kt .. ntq-1
  const int npairs = nqt * P.grp;           // pair j: query tile kt + j / grp, head g grp + j % grp
  int* status = P.status;
  const uint64_t tmo = P.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(v_full, 1);
    for (int s = 0; s < C::DO_SLOTS; ++s) {
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 1);   // one commit after dV_j, the tile's last MMA
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);          // one commit after dK_j
    for (int b = 0; b < 2; ++b) {
      mbar_init(&dp_full[b], 1);
      mbar_init(&dp_empty[b], 8);
    }
    for (int b = 0; b < C::P_BUFS; ++b) {
      mbar_init(&pb_full[b], 1);
      mbar_init(&pb_empty[b], 1);
      mbar_init(&pv_done[b], 1);
      mbar_init(&ds_full[b], 8);
    }
    mbar_init(acc_full, 1);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&P.q[shard]);
    tma_prefetch_map(&P.dO[shard]);
    tma_prefetch_map(&P.v[shard]);
    tma_prefetch_map(&P.p[shard]);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // Query-tile row and query head of pair j.  The query tiles run from the last one down to kt:
  // every CTA of a shard then reads the same dO and Q tiles at about the same time, whatever its
  // key tile, and finds most of them in L2 (dK/dV core 0.736 -> 0.723 ms at the Qwen3 shape
  // against the upward order).
  auto pair_row = [&](int j) { return (P.ntq - 1 - j / P.grp) * kBQ; };
  auto pair_head = [&](int j) { return g * P.grp + j % P.grp; };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- V, then dO_(j+1) / Q_j
      bool ok = true;
      mbar_arrive_expect_tx(v_full, C::V_BYTES);
      for (int kb = 0; kb < C::KB; ++kb) tma_load_2d(sV + kb * 16384, &P.v[shard], v_full, g * D + kb * 64, k0);
      auto load_do = [&](int j) {
        const int s = j % C::DO_SLOTS;
        if (!mbar_wait(&do_empty[s], (static_cast<uint32_t>(j / C::DO_SLOTS) & 1u) ^ 1u, abort_flag, status, tmo))
          return false;
        mbar_arrive_expect_tx(&do_full[s], C::SLOT);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_2d(sDO + s * C::SLOT + kb * 16384, &P.dO[shard], &do_full[s], pair_head(j) * D + kb * 64,
                      pair_row(j));
        return true;
      };
      auto load_q = [&](int j) {
        if (!mbar_wait(q_empty, (static_cast<uint32_t>(j) & 1u) ^ 1u, abort_flag, status, tmo)) return false;
        mbar_arrive_expect_tx(q_full, C::SLOT);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_2d(sQ + kb * 16384, &P.q[shard], q_full, pair_head(j) * D + kb * 64, pair_row(j));
        return true;
      };
      // Order: dO_0, then for every j: dO_(j+1), Q_j -- Q_j's slot frees only once dK_(j-1) is done.
      int n_do = 0, n_q = 0;
      if (npairs > 0) {
        ok = load_do(0);
        if (ok) n_do = 1;
      }
      for (int j = 0; ok && j < npairs; ++j) {
        if (j + 1 < npairs) {
          ok = load_do(j + 1);
          if (!ok) break;
          ++n_do;
        }
        ok = load_q(j);
        if (!ok) break;
        ++n_q;
      }
      // No copy may still be landing when the CTA leaves: wait (bounded) for the latest phase of
      // every buffer (an earlier load on a buffer completed before the buffer could be reused).
      int dummy_abort = 0;
      volatile int* da = reinterpret_cast<volatile int*>(&dummy_abort);
      mbar_wait(v_full, 0, da, status, tmo);
      for (int s = 0; s < C::DO_SLOTS; ++s) {
        const int jl = n_do - 1 - ((n_do - 1 - s) % C::DO_SLOTS + C::DO_SLOTS) % C::DO_SLOTS;
        if (jl >= 0) mbar_wait(&do_full[s], static_cast<uint32_t>(jl / C::DO_SLOTS) & 1u, da, status, tmo);
      }
      if (n_q > 0) mbar_wait(q_full, static_cast<uint32_t>(n_q - 1) & 1u, da, status, tmo);
    }
    __syncwarp();
  } else if (warp == kThreads / 32) {
    // ------------------------------------------------------------------ P tiles (own warp)
    if (lane == 0) {
      bool ok = true;
      int started = 0;
      auto prefetch_pair = [&](int j) {
        tma_prefetch_3d(&P.p[shard], k0, pair_row(j), pair_head(j));
        tma_prefetch_3d(&P.p[shard], k0 + 64, pair_row(j), pair_head(j));
      };
      for (int j = 0; j < 3 && j < npairs; ++j) prefetch_pair(j);
      for (int j = 0; ok && j < npairs; ++j) {
        const int b = j % C::P_BUFS;
        if (j + 3 < npairs) prefetch_pair(j + 3);   // three pairs ahead into L2
        if (!mbar_wait(&pb_empty[b], (static_cast<uint32_t>(j / C::P_BUFS) & 1u) ^ 1u, abort_flag, status, tmo)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&pb_full[b], C::P_BYTES);
        tma_load_3d(sP + b * C::P_BYTES, &P.p[shard], &pb_full[b], k0, pair_row(j), pair_head(j));
        tma_load_3d(sP + b * C::P_BYTES + 16384, &P.p[shard], &pb_full[b], k0 + 64, pair_row(j), pair_head(j));
        ++started;
      }
      int dummy_abort = 0;
      for (int b = 0; b < C::P_BUFS; ++b) {
        const int jl = started - 1 - ((started - 1 - b) % C::P_BUFS + C::P_BUFS) % C::P_BUFS;   // last on b
        if (jl >= 0)
          mbar_wait(&pb_full[b], static_cast<uint32_t>(jl / C::P_BUFS) & 1u,
                    reinterpret_cast<volatile int*>(&dummy_abort), status, tmo);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(v_full, 0, abort_flag, status, tmo);
      tc_fence_after_sync();
      const uint64_t vkd = smem_desc_sw128(smem_u32(sV), 16, 1024);   // V, K-major B of dP
      const uint32_t do0 = smem_u32(sDO);
      const uint32_t qaddr = smem_u32(sQ);
      const uint32_t paddr = smem_u32(sP);
      const uint32_t idesc_dp = idesc_bf16_f32(kBQ, kBKV, false, false);   // [queries x keys]
      const uint32_t idesc_acc = idesc_bf16_f32(kBKV, D, true, true);      // [keys x d], A and B MN-major
      const uint32_t t_dk = tmem_base + 2 * kBKV;
      const uint32_t t_dv = tmem_base + 2 * kBKV + D;
      for (int j = 0; ok && j <= npairs; ++j) {
        if (j < npairs) {
          const int b = j & 1;
          const int ds = j % C::DO_SLOTS;
          const int pbuf = j % C::P_BUFS;
          // dP_j = dO_j V^T  [queries x keys]
          if (!mbar_wait(&do_full[ds], static_cast<uint32_t>(j / C::DO_SLOTS) & 1u, abort_flag, status, tmo) ||
              !mbar_wait(&dp_empty[b], (static_cast<uint32_t>(j >> 1) & 1u) ^ 1u, abort_flag, status, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t daddr = do0 + ds * C::SLOT;
          const uint64_t dd = smem_desc_sw128(daddr, 16, 1024);
          for (int kb = 0; kb < C::KB; ++kb) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = desc_advance(dd, kb * 16384 + kk * 32);
              const uint64_t bd = desc_advance(vkd, kb * 16384 + kk * 32);
              umma_bf16(tmem_base + b * kBKV, ad, bd, idesc_dp, (kb | kk) ? 1u : 0u);
            }
          }
          umma_commit(&dp_full[b]);
          // dV += P_j^T dO_j: A = P tile read MN-major (keys contiguous), B = dO tile read MN-major
          if (!mbar_wait(&pb_full[pbuf], static_cast<uint32_t>(j / C::P_BUFS) & 1u, abort_flag, status, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t pmd = smem_desc_sw128(paddr + pbuf * C::P_BYTES, 16384, 1024);
          const uint64_t dmd = smem_desc_sw128(daddr, 16384, 1024);
#pragma unroll
          for (int kq = 0; kq < kBQ / 16; ++kq) {   // K = the 128 queries, 16 per MMA
            const uint64_t ad = desc_advance(pmd, kq * 2048);
            const uint64_t bd = desc_advance(dmd, kq * 2048);
            umma_bf16(t_dv, ad, bd, idesc_acc, (j | kq) ? 1u : 0u);
          }
          umma_commit(&pv_done[pbuf]);
          umma_commit(&do_empty[ds]);               // the dO tile's last MMA (dP's are earlier)
        }
        if (ok && j > 0) {
          // dK += dS_(j-1)^T Q_(j-1): A = dS (in the P buffer) MN-major, B = Q tile MN-major
          const int jp = j - 1;
          const int pbuf = jp % C::P_BUFS;
          if (!mbar_wait(q_full, static_cast<uint32_t>(jp) & 1u, abort_flag, status, tmo) ||
              !mbar_wait(&ds_full[pbuf], static_cast<uint32_t>(jp / C::P_BUFS) & 1u, abort_flag, status, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t smd = smem_desc_sw128(paddr + pbuf * C::P_BYTES, 16384, 1024);
          const uint64_t qmd = smem_desc_sw128(qaddr, 16384, 1024);
#pragma unroll
          for (int kq = 0; kq < kBQ / 16; ++kq) {
            const uint64_t ad = desc_advance(smd, kq * 2048);
            const uint64_t bd = desc_advance(qmd, kq * 2048);
            umma_bf16(t_dk, ad, bd, idesc_acc, (jp | kq) ? 1u : 0u);
          }
          umma_commit(&pb_empty[pbuf]);
          umma_commit(q_empty);
        }
      }
      if (ok) umma_commit(acc_full);
      umma_commit(done_bar);
      int dummy_abort = 0;
      mbar_wait(done_bar, 0, reinterpret_cast<volatile int*>(&dummy_abort), status, tmo);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ dS warps
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;            // query row within the pair's query tile
    const float scale = P.scale;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    uint8_t* my_row = sP + half * 16384 + (r >> 3) * 1024 + (r & 7) * 128;
    bool ok = true;
    for (int j = 0; ok && j < npairs; ++j) {
      const int b = j & 1;
      const int pbuf = j % C::P_BUFS;
      const int q = pair_row(j) + r;
      const int c = pair_head(j);
      const float Dq = q < P.T ? P.D[(static_cast<int64_t>(shard) * P.nql + c) * P.T + q] : 0.0f;
      const uint64_t nDs2 = f2_pack(-Dq * scale, -Dq * scale), scale2 = f2_pack(scale, scale);
      ok = mbar_wait(&dp_full[b], static_cast<uint32_t>(j >> 1) & 1u, abort_flag, status, tmo);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(lane_base + b * kBKV + half * 64, r0);
      tmem_ld_32x32b_x32(lane_base + b * kBKV + half * 64 + 32, r1);
      tmem_ld_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dp_empty[b]);
      // dV's MMA has read P_j: it may now be overwritten by dS_j
      ok = mbar_wait(&pv_done[pbuf], static_cast<uint32_t>(j / C::P_BUFS) & 1u, abort_flag, status, tmo);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint8_t* row = my_row + pbuf * C::P_BYTES;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint4* unit = reinterpret_cast<uint4*>(row + ((u ^ (r & 7)) << 4));
        const uint4 pw = *unit;
        const uint32_t pv[4] = {pw.x, pw.y, pw.z, pw.w};
        // dS = (dP scale - D scale) P, two columns per packed fp32 instruction (one fma and one
        // multiply per pair).  P is zero above the diagonal.
        uint32_t o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = u * 8 + 2 * e;
          const uint64_t dp2 = f2_pack(__uint_as_float(col < 32 ? r0[col] : r1[col - 32]),
                                       __uint_as_float(col < 32 ? r0[col + 1] : r1[col - 31]));
          const uint64_t p2 = f2_pack(bf16_lo(pv[e]), bf16_hi(pv[e]));
          const float2 d2 = f2_unpack(fmul2(ffma2(dp2, scale2, nDs2), p2));
          o4[e] = pack_bf16x2(d2.x, d2.y);
        }
        *unit = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_full[pbuf]);
    }
    // dK and dV rows (keys): this warp stores half of the d columns of each
    if (ok) ok = mbar_wait(acc_full, 0, abort_flag, status, tmo);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after_sync();
      const int key = k0 + r;
      const bool key_ok = key < P.T;
      const int64_t off = static_cast<int64_t>(key_ok ? key : 0) * (P.nkvl * D) + g * D + half * (D / 2);
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        __nv_bfloat16* out = (w == 0 ? P.dK[shard] : P.dV[shard]) + off;
#pragma unroll
        for (int cc = 0; cc < D / 2; cc += 32) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(lane_base + 2 * kBKV + w * D + half * (D / 2) + cc, o);
          tmem_ld_wait();
          if (key_ok) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<uint4*>(out + cc + u * 8) = make_uint4(
                  pack_bf16x2(__uint_as_float(o[u * 8 + 0]), __uint_as_float(o[u * 8 + 1])),
                  pack_bf16x2(__uint_as_float(o[u * 8 + 2]), __uint_as_float(o[u * 8 + 3])),
                  pack_bf16x2(__uint_as_float(o[u * 8 + 4]), __uint_as_float(o[u * 8 + 5])),
                  pack_bf16x2(__uint_as_float(o[u * 8 + 6]), __uint_as_float(o[u * 8 + 7])));
          }
        }
      }
    }
    tc_fence_before_sync();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

// Raises a core kernel's dynamic shared-memory limit, once per kernel and device (thread-safe).
enum CoreKernelSlot { kFwd128, kFwd64, kBwd128, kBwd64, kKv128, kKv64, kCoreKernelSlots };
constexpr int kMaxCoreDevices = 64;
static int set_core_smem(const void* fn, int slot, int bytes, const char* what) {
  static std::mutex mu;
  static bool done[kCoreKernelSlots][kMaxCoreDevices] = {};
  int dev = 0;
  int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= kMaxCoreDevices) return set_error(TTL_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (done[slot][dev]) return TTL_OK;
  rc = cuda_check(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes), what);
  if (!rc) done[slot][dev] = true;
  return rc;
}

int attn_fwd_core(int t, int64_t T, int nql, int grp, int d, const void* const* Q, const void* const* K,
                  const void* const* V, void* const* Pout, void* const* Oout, int64_t qc, int64_t kc,
                  cudaStream_t stream) {
  if (d != 64 && d != 128) return set_error(TTL_ERR_SHAPE, "attention core: head dimension %d is not 64 or 128", d);
  int rc = require_sm103();
  if (rc) return rc;
  CoreParams* p = new CoreParams;
  std::memset(static_cast<void*>(p), 0, sizeof(CoreParams));
  for (int i = 0; i < t && !rc; ++i) {
    rc = encode_map_bf16(&p->q[i], Q[i], T, qc, qc, 64, 128);
    if (!rc) rc = encode_map_bf16(&p->k[i], K[i], T, kc, kc, 64, 128);
    if (!rc) rc = encode_map_bf16(&p->v[i], V[i], T, kc, kc, 64, 64);
    if (!rc) rc = encode_map_bf16_3d(&p->pm[i], Pout[i], T, T, nql, T, T * T, 64, 128);
    p->O[i] = static_cast<__nv_bfloat16*>(Oout[i]);
  }
  if (rc) {
    delete p;
    return rc;
  }
  p->t = t;
  p->nql = nql;
  p->grp = grp;
  p->T = static_cast<int>(T);
  p->ntq = static_cast<int>((T + kBQ - 1) / kBQ);
  p->k_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  p->status = device_status_ptr();
  p->timeout_ns = 2000000000ull;
  if (!p->status) {
    delete p;
    return TTL_ERR_CUDA;
  }
  const unsigned blocks = static_cast<unsigned>(t) * nql * p->ntq;
  const double tri = static_cast<double>(T) * (T + 1) / 2.0;
  // Algorithmic work: S = Q K^T and P V over the causal triangle (the second score pass is a
  // recomputation and is not counted); bytes: Q, K, V read once, P and O written once.
  TraceScope tr(stream, TTL_K_ATTN_CORE, 2.0 * 2.0 * tri * d * t * nql,
                2.0 * tri * t * nql + 2.0 * T * (2.0 * qc + 2.0 * kc) * t);
  if (d == 128) {
    if ((rc = set_core_smem(reinterpret_cast<const void*>(attn_fwd_core_kernel<128>), kFwd128, CoreCfg<128>::SMEM,
                            "cudaFuncSetAttribute(attn core)"))) {
      delete p;
      return rc;
    }
    attn_fwd_core_kernel<128><<<blocks, kCoreThreads, CoreCfg<128>::SMEM, stream>>>(*p);
  } else {
    if ((rc = set_core_smem(reinterpret_cast<const void*>(attn_fwd_core_kernel<64>), kFwd64, CoreCfg<64>::SMEM,
                            "cudaFuncSetAttribute(attn core)"))) {
      delete p;
      return rc;
    }
    attn_fwd_core_kernel<64><<<blocks, kCoreThreads, CoreCfg<64>::SMEM, stream>>>(*p);
  }
  delete p;
  return cuda_check(cudaGetLastError(), "attn_fwd_core_kernel launch");
}


int attn_bwd_core(int t, int64_t T, int nql, int grp, int d, const void* const* dO, const void* const* V,
                  const void* const* K, const void* const* Pin, void* const* dQ, const float* Drow, int64_t qc,
                  int64_t kc, cudaStream_t stream) {
  if (d != 64 && d != 128) return set_error(TTL_ERR_SHAPE, "attention core: head dimension %d is not 64 or 128", d);
  int rc = require_sm103();
  if (rc) return rc;
  BwdParams* p = new BwdParams;
  std::memset(static_cast<void*>(p), 0, sizeof(BwdParams));
  for (int i = 0; i < t && !rc; ++i) {
    rc = encode_map_bf16(&p->dO[i], dO[i], T, qc, qc, 64, 128);
    if (!rc) rc = encode_map_bf16(&p->v[i], V[i], T, kc, kc, 64, 128);
    if (!rc) rc = encode_map_bf16(&p->kmn[i], K[i], T, kc, kc, 64, 64);
    if (!rc) rc = encode_map_bf16_3d(&p->p[i], Pin[i], T, T, nql, T, T * T, 64, 128);
    p->dQ[i] = static_cast<__nv_bfloat16*>(dQ[i]);
  }
  if (rc) {
    delete p;
    return rc;
  }
  p->D = Drow;
  p->t = t;
  p->nql = nql;
  p->grp = grp;
  p->T = static_cast<int>(T);
  p->ntq = static_cast<int>((T + kBQ - 1) / kBQ);
  p->scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  p->status = device_status_ptr();
  p->timeout_ns = 2000000000ull;
  if (!p->status) {
    delete p;
    return TTL_ERR_CUDA;
  }
  const unsigned blocks = static_cast<unsigned>(t) * nql * p->ntq;
  const double tri = static_cast<double>(T) * (T + 1) / 2.0;
  // Algorithmic work: dP = dO V^T and dQ = dS K over the causal triangle; bytes: P read, dO, V,
  // K read and dQ written once.
  TraceScope tr(stream, TTL_K_ATTN_CORE, 2.0 * 2.0 * tri * d * t * nql,
                2.0 * tri * t * nql + 2.0 * T * (2.0 * qc + 2.0 * kc) * t);
  if (d == 128) {
    if ((rc = set_core_smem(reinterpret_cast<const void*>(attn_bwd_core_kernel<128>), kBwd128, BwdCfg<128>::SMEM,
                            "cudaFuncSetAttribute(attn bwd core)"))) {
      delete p;
      return rc;
    }
    attn_bwd_core_kernel<128><<<blocks, kCoreThreads, BwdCfg<128>::SMEM, stream>>>(*p);
  } else {
    if ((rc = set_core_smem(reinterpret_cast<const void*>(attn_bwd_core_kernel<64>), kBwd64, BwdCfg<64>::SMEM,
                            "cudaFuncSetAttribute(attn bwd core)"))) {
      delete p;
      return rc;
    }
    attn_bwd_core_kernel<64><<<blocks, kCoreThreads, BwdCfg<64>::SMEM, stream>>>(*p);
  }
  delete p;
  return cuda_check(cudaGetLastError(), "attn_bwd_core_kernel launch");
}


int attn_bwd_kv(int t, int64_t T, int nql, int nkvl, int grp, int d, const void* const* Q, const void* const* dO,
                const void* const* V, const void* const* Pin, void* const* dK, void* const* dV, const float* Drow,
                int64_t qc, int64_t kc, cudaStream_t stream) {
  if (d != 64 && d != 128) return set_error(TTL_ERR_SHAPE, "attention core: head dimension %d is not 64 or 128", d);
  int rc = require_sm103();
  if (rc) return rc;
  KvParams* p = new KvParams;
  std::memset(static_cast<void*>(p), 0, sizeof(KvParams));
  for (int i = 0; i < t && !rc; ++i) {
    rc = encode_map_bf16(&p->q[i], Q[i], T, qc, qc, 64, 128);
    if (!rc) rc = encode_map_bf16(&p->dO[i], dO[i], T, qc, qc, 64, 128);
    if (!rc) rc = encode_map_bf16(&p->v[i], V[i], T, kc, kc, 64, 128);
    if (!rc) rc = encode_map_bf16_3d(&p->p[i], Pin[i], T, T, nql, T, T * T, 64, 128);
    p->dK[i] = static_cast<__nv_bfloat16*>(dK[i]);
    p->dV[i] = static_cast<__nv_bfloat16*>(dV[i]);
  }
  if (rc) {
    delete p;
    return rc;
  }
  p->D = Drow;
  p->t = t;
  p->nql = nql;
  p->nkvl = nkvl;
  p->grp = grp;
  p->T = static_cast<int>(T);
  p->ntq = static_cast<int>((T + kBQ - 1) / kBQ);
  p->scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  p->status = device_status_ptr();
  p->timeout_ns = 2000000000ull;
  if (!p->status) {
    delete p;
    return TTL_ERR_CUDA;
  }
  const unsigned blocks = static_cast<unsigned>(t) * nkvl * p->ntq;
  const double tri = static_cast<double>(T) * (T + 1) / 2.0;
  // Algorithmic work: dV = P^T dO and dK = dS^T Q over the causal triangle (the dP it recomputes
  // is not counted); bytes: P read once, Q, dO, V read once, dK and dV written once.
  TraceScope tr(stream, TTL_K_ATTN_CORE, 2.0 * 2.0 * tri * d * t * nql,
                2.0 * tri * t * nql + 2.0 * T * (2.0 * qc + 3.0 * kc) * t);
  if (d == 128) {
    if ((rc = set_core_smem(reinterpret_cast<const void*>(attn_bwd_kv_kernel<128>), kKv128, KvCfg<128>::SMEM,
                            "cudaFuncSetAttribute(attn kv core)"))) {
      delete p;
      return rc;
    }
    attn_bwd_kv_kernel<128><<<blocks, kCoreThreads, KvCfg<128>::SMEM, stream>>>(*p);
  } else {
    if ((rc = set_core_smem(reinterpret_cast<const void*>(attn_bwd_kv_kernel<64>), kKv64, KvCfg<64>::SMEM,
                            "cudaFuncSetAttribute(attn kv core)"))) {
      delete p;
      return rc;
    }
    attn_bwd_kv_kernel<64><<<blocks, kCoreThreads, KvCfg<64>::SMEM, stream>>>(*p);
  }
  delete p;
  return cuda_check(cudaGetLastError(), "attn_bwd_kv_kernel launch");
}

}  // namespace ttl

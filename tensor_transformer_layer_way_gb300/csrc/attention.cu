// Tensor-parallel attention block on t logical shards of one GPU, heads split across shards.
//
// Source: "v4:Tensor Parallel 与 Sequence Parallel", section "Attention:按 head 切": heads are
// independent, so W_Q, W_K, W_V are column-split by head and each shard finishes the attention
// of its own heads without communication; W_O is row-split and followed by one all-reduce;
// the head counts must be divisible by t (Qwen3: 32 query / 8 KV heads, 4 + 1 per shard at
// t = 8).  The TP-communication page's Fig. 1 draws the same f -> column -> local -> row -> g
// shape.  The pages do not spell out the attention itself; this file computes causal scaled
// dot-product attention with scale 1/sqrt(d), query head j reading KV head j / (n_q / n_kv).
//
// The projections, W_O and the projection gradients run in the tcgen05 GEMM; the attention
// itself runs in three fused kernels (attention_core.cu) with every score tile in tensor memory:
//   forward : QKV (3t problems) -> core: S = Q_c K_g^T, exact row statistics, P = softmax(S /
//             sqrt(d)) (bf16, saved), O_c = P_c V_g -> Y_i = O_i Wo_i -> all-reduce
//   backward: {dO_i = dY Wo_i^T, dWo_i = O_i^T dY} -> D = rowsum(dO_c O_c)
//             -> query-tile core: dP = dO_c V_g^T, dS = P (dP - D) / sqrt(d), dQ_c = dS_c K_g
//             -> key-tile core: the same dP and dS, dK_g = sum_c dS_c^T Q_c, dV_g = sum_c P_c^T dO_c
//             -> {dW_i = X^T d{Q,K,V}_i, dX_i = dQ_i Wq_i^T + dK_i Wk_i^T + dV_i Wv_i^T} -> all-reduce
// Only P goes through HBM (written once, read by both backward cores); dS never does.
// Row q of P is written for every key j < min(T, round_up(q + 1, 128)) (its query tile's
// diagonal tile), with exact zeros above the diagonal.

#include <cmath>

#include "ttl_device.cuh"
#include "ttl_internal.h"

namespace ttl {
namespace {

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int kRowWarps = 8;   // rows (one per warp) per CTA of the row kernels

// Per-shard pointers of the row kernels.
struct AttnRows {
  const __nv_bfloat16* dO[kMaxShards];   // [T, n_q/t d]
  const __nv_bfloat16* o[kMaxShards];    // [T, n_q/t d]
};

__device__ __forceinline__ void unpack8_bf16(uint4 w, float* v) {
  v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}

// One warp per (shard, query) row, covering all of the shard's query heads (their nql d columns
// are contiguous): D[(i nql + c) T + q] = sum over head c's d columns of dO[q, .] O[q, .] (the
// rowsum term of the softmax backward).  Each 256-column sweep loads 512 contiguous bytes per
// operand; the d / 8 lanes of one head then reduce among themselves.
__global__ void __launch_bounds__(kRowWarps * 32) attn_rowdot_kernel(const __grid_constant__ AttnRows R,
                                                                     float* __restrict__ D, int64_t rows,
                                                                     int64_t T, int64_t nql, int d) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  if (row >= rows) return;   // rows = t T: the whole warp leaves together
  const int lane = threadIdx.x & 31;
  const int i = static_cast<int>(row / T);
  const int64_t q = row - i * T;
  const int64_t cols = nql * d;
  const __nv_bfloat16* a = R.dO[i] + q * cols;
  const __nv_bfloat16* o = R.o[i] + q * cols;
  const int lph = d / 8;     // lanes per head in a sweep (8 or 16)
  for (int64_t base = 0; base < cols; base += 256) {
    const int64_t k0 = base + lane * 8;
    float acc = 0.0f;
    if (k0 < cols) {
      float x[8], y[8];
      unpack8_bf16(*reinterpret_cast<const uint4*>(a + k0), x);
      unpack8_bf16(*reinterpret_cast<const uint4*>(o + k0), y);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc = fmaf(x[j], y[j], acc);
    }
    for (int off = lph >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (k0 < cols && (lane & (lph - 1)) == 0) D[(static_cast<int64_t>(i) * nql + k0 / d) * T + q] = acc;
  }
}

struct Shape {
  int t;
  int64_t T, h;
  int n_q, n_kv, d;
  int64_t nql, nkvl, grp;   // query heads, KV heads per shard; query heads per KV head
  int64_t qc, kc;           // columns of Q_i and of K_i / V_i
};

int check_shape(int t, int64_t T, int64_t h, int n_q, int n_kv, int d, const char* name, Shape* out) {
  if (t < 1 || t > kMaxShards) return set_error(TTL_ERR_ARG, "%s: t=%d outside [1,%d]", name, t, kMaxShards);
  if (T < 0 || h < 0 || n_q < 1 || n_kv < 1 || d < 1) return set_error(TTL_ERR_ARG, "%s: bad shape", name);
  if (n_q % t || n_kv % t)
    return set_error(TTL_ERR_SHAPE, "%s: t=%d must divide the head counts %d and %d", name, t, n_q, n_kv);
  if (n_q % n_kv) return set_error(TTL_ERR_SHAPE, "%s: n_kv=%d must divide n_q=%d", name, n_kv, n_q);
  if (d != 64 && d != 128) return set_error(TTL_ERR_SHAPE, "%s: head dimension %d is not 64 or 128", name, d);
  if (T % 8 || h % 8 || h == 0)
    return set_error(TTL_ERR_SHAPE, "%s: T and h must be multiples of 8 (16-byte rows), h > 0", name);
  if (T >= (int64_t(1) << 28) || h >= (int64_t(1) << 31) || static_cast<int64_t>(n_q / t) * T >= (int64_t(1) << 31))
    return set_error(TTL_ERR_SHAPE, "%s: extent beyond 2^31", name);
  Shape& s = *out;
  s.t = t; s.T = T; s.h = h; s.n_q = n_q; s.n_kv = n_kv; s.d = d;
  s.nql = n_q / t; s.nkvl = n_kv / t; s.grp = n_q / n_kv;
  s.qc = s.nql * d; s.kc = s.nkvl * d;
  return TTL_OK;
}

int check_ptrs(const void* const* arr, int t, const char* what) {
  if (!arr) return set_error(TTL_ERR_ARG, "%s: null shard array", what);
  for (int i = 0; i < t; ++i) {
    if (!arr[i]) return set_error(TTL_ERR_ARG, "%s[%d] is null", what, i);
    if (!aligned16(arr[i])) return set_error(TTL_ERR_ALIGN, "%s[%d] not 16-byte aligned", what, i);
  }
  return TTL_OK;
}

const __nv_bfloat16* bf(const ttl_bf16* p) { return reinterpret_cast<const __nv_bfloat16*>(p); }

// Backward workspace: D = rowsum(dO O) [t n_q/t T] fp32, then per shard dO, dQ ([T, n_q/t d]),
// dK, dV ([T, n_kv/t d]).
size_t bwd_d_bytes(const Shape& s) { return round256(static_cast<size_t>(s.t * s.nql * s.T) * 4); }
size_t bwd_shard_bytes(const Shape& s) {
  const size_t tok = static_cast<size_t>(s.T) * 2;
  return 2 * round256(tok * s.qc) + 2 * round256(tok * s.kc);
}

}  // namespace
}  // namespace ttl

using namespace ttl;

extern "C" size_t ttl_tp_attn_fwd_workspace_size(int t, int64_t T, int n_q, int n_kv, int d) {
  Shape s;
  if (check_shape(t, T, 8, n_q, n_kv, d, "ttl_tp_attn_fwd_workspace_size", &s)) return 0;
  return 0;   // the fused forward core keeps its scores and statistics on chip
}

extern "C" size_t ttl_tp_attn_bwd_workspace_size(int t, int64_t T, int n_q, int n_kv, int d) {
  Shape s;
  if (check_shape(t, T, 8, n_q, n_kv, d, "ttl_tp_attn_bwd_workspace_size", &s)) return 0;
  return bwd_d_bytes(s) + bwd_shard_bytes(s) * static_cast<size_t>(t);
}

extern "C" int ttl_tp_attn_fwd(int t, int64_t T, int64_t h, int n_q, int n_kv, int d, const ttl_bf16* X,
                               const ttl_bf16* const* Wq, const ttl_bf16* const* Wk, const ttl_bf16* const* Wv,
                               const ttl_bf16* const* Wo, ttl_bf16* const* Q_save, ttl_bf16* const* K_save,
                               ttl_bf16* const* V_save, ttl_bf16* const* P_save, ttl_bf16* const* O_save,
                               ttl_bf16* const* Y, void* ws, size_t ws_bytes, void* stream) {
  const char* name = "ttl_tp_attn_fwd";
  Shape s;
  int rc = check_shape(t, T, h, n_q, n_kv, d, name, &s);
  if (rc) return rc;
  if (T == 0) return TTL_OK;   // no tokens: every output is empty
  if (!X) return set_error(TTL_ERR_ARG, "%s: X is null", name);
  if (!aligned16(X)) return set_error(TTL_ERR_ALIGN, "%s: X not 16-byte aligned", name);
  using CP = const void* const*;
  const struct { CP p; const char* n; } arrs[] = {
      {reinterpret_cast<CP>(Wq), "Wq"},         {reinterpret_cast<CP>(Wk), "Wk"},
      {reinterpret_cast<CP>(Wv), "Wv"},         {reinterpret_cast<CP>(Wo), "Wo"},
      {reinterpret_cast<CP>(Q_save), "Q_save"}, {reinterpret_cast<CP>(K_save), "K_save"},
      {reinterpret_cast<CP>(V_save), "V_save"}, {reinterpret_cast<CP>(P_save), "P_save"},
      {reinterpret_cast<CP>(O_save), "O_save"}, {reinterpret_cast<CP>(Y), "Y"}};
  for (const auto& a : arrs)
    if ((rc = check_ptrs(a.p, t, a.n))) return rc;
  (void)ws;
  (void)ws_bytes;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  GemmBatch batch;

  // Column-parallel projections: Q_i = X Wq_i in one launch (one tile group over X; wide tiles
  // where Q is wider than 256 columns), then K_i, V_i = X Wk_i, X Wv_i as one paired problem
  // per shard in a second launch (each 256-column accumulator tile holds 128 columns of K_i
  // and the same 128 of V_i, so the narrow KV heads run as full-width MMAs).  Kept apart, the
  // paired problems do not hold the Q problems back to the 256-column tiles.
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(2, 1) && (rc = batch.flush(st))) return rc;
    const int mx = batch.add_map(X, T, h, h, false);
    const int mq = batch.add_map(Wq[i], h, s.qc, s.qc, true);
    Problem* p = batch.add_problem(T, s.qc, false, true, EPI_BF16, false, true);
    if (batch.error()) return batch.error();
    p->out0 = Q_save[i];
    p->ld_out = s.qc;
    if ((rc = batch.add_seg(p, mx, 0, mq, -1, 0, h))) return rc;
  }
  if ((rc = batch.flush(st))) return rc;
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(3, 1) && (rc = batch.flush(st))) return rc;
    const int mx = batch.add_map(X, T, h, h, false);
    const int mk = batch.add_map(Wk[i], h, s.kc, s.kc, true);
    const int mv = batch.add_map(Wv[i], h, s.kc, s.kc, true);
    Problem* p = batch.add_problem(T, s.kc, false, true, EPI_PAIR_BF16, true, true);
    if (batch.error()) return batch.error();
    p->out0 = K_save[i];
    p->out1 = V_save[i];
    p->ld_out = s.kc;
    if ((rc = batch.add_seg(p, mx, 0, mk, mv, 0, h))) return rc;
  }
  if ((rc = batch.flush(st))) return rc;

  // The fused core: scores, softmax and P V for every (shard, head, 128-query tile).
  {
    using CP = const void* const*;
    using VP = void* const*;
    if ((rc = attn_fwd_core(t, T, static_cast<int>(s.nql), static_cast<int>(s.grp), d, reinterpret_cast<CP>(Q_save),
                            reinterpret_cast<CP>(K_save), reinterpret_cast<CP>(V_save), reinterpret_cast<VP>(P_save),
                            reinterpret_cast<VP>(O_save), s.qc, s.kc, st)))
      return rc;
  }

  // Row-parallel W_O: the full-shape partial Y_i = O_i Wo_i.
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(2, 1) && (rc = batch.flush(st))) return rc;
    const int mo = batch.add_map(O_save[i], T, s.qc, s.qc, false);
    const int mw = batch.add_map(Wo[i], s.qc, h, h, true);
    Problem* p = batch.add_problem(T, h, false, true, EPI_BF16, false);
    if (batch.error()) return batch.error();
    p->out0 = Y[i];
    p->ld_out = h;
    if ((rc = batch.add_seg(p, mo, 0, mw, -1, 0, s.qc))) return rc;
  }
  if ((rc = batch.flush(st))) return rc;

  // g forward: all-reduce of the partials.
  return shard_all_reduce_internal(t, T, h, Y, nullptr, st);
}

extern "C" int ttl_tp_attn_bwd(int t, int64_t T, int64_t h, int n_q, int n_kv, int d, const ttl_bf16* X,
                               const ttl_bf16* dY, const ttl_bf16* const* Wq, const ttl_bf16* const* Wk,
                               const ttl_bf16* const* Wv, const ttl_bf16* const* Wo, const ttl_bf16* const* Q_save,
                               const ttl_bf16* const* K_save, const ttl_bf16* const* V_save,
                               const ttl_bf16* const* P_save, const ttl_bf16* const* O_save, ttl_bf16* const* dWq,
                               ttl_bf16* const* dWk, ttl_bf16* const* dWv, ttl_bf16* const* dWo,
                               ttl_bf16* const* dX, void* ws, size_t ws_bytes, void* stream) {
  const char* name = "ttl_tp_attn_bwd";
  Shape s;
  int rc = check_shape(t, T, h, n_q, n_kv, d, name, &s);
  if (rc) return rc;
  using CP = const void* const*;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  {
    const struct { CP p; const char* n; } outs[] = {{reinterpret_cast<CP>(dWq), "dWq"},
                                                    {reinterpret_cast<CP>(dWk), "dWk"},
                                                    {reinterpret_cast<CP>(dWv), "dWv"},
                                                    {reinterpret_cast<CP>(dWo), "dWo"}};
    for (const auto& a : outs)
      if ((rc = check_ptrs(a.p, t, a.n))) return rc;
  }
  if (T == 0) {   // no tokens: the weight gradients are empty sums
    for (int i = 0; i < t; ++i) {
      if ((rc = fill_zero(dWq[i], h * s.qc * 2, st))) return rc;
      if ((rc = fill_zero(dWk[i], h * s.kc * 2, st))) return rc;
      if ((rc = fill_zero(dWv[i], h * s.kc * 2, st))) return rc;
      if ((rc = fill_zero(dWo[i], s.qc * h * 2, st))) return rc;
    }
    return TTL_OK;
  }
  if (!X || !dY) return set_error(TTL_ERR_ARG, "%s: X or dY is null", name);
  if (!aligned16(X) || !aligned16(dY)) return set_error(TTL_ERR_ALIGN, "%s: X or dY not 16-byte aligned", name);
  {
    const struct { CP p; const char* n; } arrs[] = {
        {reinterpret_cast<CP>(Wq), "Wq"},         {reinterpret_cast<CP>(Wk), "Wk"},
        {reinterpret_cast<CP>(Wv), "Wv"},         {reinterpret_cast<CP>(Wo), "Wo"},
        {reinterpret_cast<CP>(Q_save), "Q_save"}, {reinterpret_cast<CP>(K_save), "K_save"},
        {reinterpret_cast<CP>(V_save), "V_save"}, {reinterpret_cast<CP>(P_save), "P_save"},
        {reinterpret_cast<CP>(O_save), "O_save"}, {reinterpret_cast<CP>(dX), "dX"}};
    for (const auto& a : arrs)
      if ((rc = check_ptrs(a.p, t, a.n))) return rc;
  }
  const size_t need = ttl_tp_attn_bwd_workspace_size(t, T, n_q, n_kv, d);
  if (!ws || ws_bytes < need)
    return set_error(TTL_ERR_ARG, "%s: workspace of %zu bytes needed, %zu given", name, need, ws_bytes);
  if (!aligned16(ws)) return set_error(TTL_ERR_ALIGN, "%s: workspace not 16-byte aligned", name);

  // Workspace: D for every (shard, head, query) row, then per shard dO_i, dQ_i, dK_i, dV_i.
  const size_t b_q = round256(static_cast<size_t>(T) * 2 * s.qc), b_k = round256(static_cast<size_t>(T) * 2 * s.kc);
  float* Drow = static_cast<float*>(ws);
  auto base = [&](int i) {
    return static_cast<char*>(ws) + bwd_d_bytes(s) + bwd_shard_bytes(s) * static_cast<size_t>(i);
  };
  auto dO_of = [&](int i) { return reinterpret_cast<__nv_bfloat16*>(base(i)); };
  auto dQ_of = [&](int i) { return reinterpret_cast<__nv_bfloat16*>(base(i) + b_q); };
  auto dK_of = [&](int i) { return reinterpret_cast<__nv_bfloat16*>(base(i) + 2 * b_q); };
  auto dV_of = [&](int i) { return reinterpret_cast<__nv_bfloat16*>(base(i) + 2 * b_q + b_k); };
  GemmBatch batch;

  // g backward is the identity: dO_i = dY Wo_i^T (one tile group over dY) and dWo_i = O_i^T dY.
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(2, 1) && (rc = batch.flush(st))) return rc;
    const int md = batch.add_map(dY, T, h, h, false);
    const int mw = batch.add_map(Wo[i], s.qc, h, h, false);
    Problem* p = batch.add_problem(T, s.qc, false, false, EPI_BF16, false, true);
    if (batch.error()) return batch.error();
    p->out0 = dO_of(i);
    p->ld_out = s.qc;
    if ((rc = batch.add_seg(p, md, 0, mw, -1, 0, h))) return rc;
  }
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(2, 1) && (rc = batch.flush(st))) return rc;
    const int mo = batch.add_map(O_save[i], T, s.qc, s.qc, true);
    const int md = batch.add_map(dY, T, h, h, true);
    Problem* p = batch.add_problem(s.qc, h, true, true, EPI_BF16, false);
    if (batch.error()) return batch.error();
    p->out0 = dWo[i];
    p->ld_out = h;
    if ((rc = batch.add_seg(p, mo, 0, md, -1, 0, T))) return rc;
  }
  if ((rc = batch.flush(st))) return rc;

  // D = rowsum(dO_c O_c) for every (shard, head, query) row; one warp per (shard, query).
  {
    AttnRows R = {};
    for (int i = 0; i < t; ++i) {
      R.dO[i] = dO_of(i);
      R.o[i] = bf(O_save[i]);
    }
    const int64_t rows = static_cast<int64_t>(t) * T;
    TraceScope tr(st, TTL_K_SOFTMAX, 0.0, static_cast<double>(rows) * s.nql * (4.0 * d + 4.0));
    attn_rowdot_kernel<<<static_cast<unsigned>((rows + kRowWarps - 1) / kRowWarps), kRowWarps * 32, 0, st>>>(
        R, Drow, rows, T, s.nql, d);
    if ((rc = cuda_check(cudaGetLastError(), "attn_rowdot_kernel launch"))) return rc;
  }

  // The backward cores: dQ per (shard, query head, 128-query tile) and dK, dV per (shard, KV
  // head, 128-key tile), each recomputing dP = dO V^T in TMEM and dS = P (dP - D) / sqrt(d) on
  // chip from the saved P.
  {
    using CP = const void* const*;
    const void* dOs[kMaxShards];
    void* dQs[kMaxShards];
    void* dKs[kMaxShards];
    void* dVs[kMaxShards];
    for (int i = 0; i < t; ++i) {
      dOs[i] = dO_of(i);
      dQs[i] = dQ_of(i);
      dKs[i] = dK_of(i);
      dVs[i] = dV_of(i);
    }
    if ((rc = attn_bwd_core(t, T, static_cast<int>(s.nql), static_cast<int>(s.grp), d, dOs,
                            reinterpret_cast<CP>(V_save), reinterpret_cast<CP>(K_save), reinterpret_cast<CP>(P_save),
                            dQs, Drow, s.qc, s.kc, st)))
      return rc;
    if ((rc = attn_bwd_kv(t, T, static_cast<int>(s.nql), static_cast<int>(s.nkvl), static_cast<int>(s.grp), d,
                          reinterpret_cast<CP>(Q_save), dOs, reinterpret_cast<CP>(V_save), reinterpret_cast<CP>(P_save),
                          dKs, dVs, Drow, s.qc, s.kc, st)))
      return rc;
  }

  // Column-parallel projections backward: dWk_i and dWv_i = X^T dK_i, X^T dV_i as one paired
  // problem per shard (one launch, a tile group over X^T), then dWq_i = X^T dQ_i (a tile group
  // over X^T) and the dX partials dQ_i Wq_i^T + dK_i Wk_i^T + dV_i Wv_i^T (three K segments) in
  // one launch that the paired problems do not hold back to the 256-column tiles.
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(3, 1) && (rc = batch.flush(st))) return rc;
    const int mx = batch.add_map(X, T, h, h, true);
    const int mk = batch.add_map(dK_of(i), T, s.kc, s.kc, true);
    const int mv = batch.add_map(dV_of(i), T, s.kc, s.kc, true);
    Problem* p = batch.add_problem(h, s.kc, true, true, EPI_PAIR_BF16, true, true);
    if (batch.error()) return batch.error();
    p->out0 = dWk[i];
    p->out1 = dWv[i];
    p->ld_out = s.kc;
    if ((rc = batch.add_seg(p, mx, 0, mk, mv, 0, T))) return rc;
  }
  if ((rc = batch.flush(st))) return rc;
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(2, 1) && (rc = batch.flush(st))) return rc;
    const int mx = batch.add_map(X, T, h, h, true);
    const int mq = batch.add_map(dQ_of(i), T, s.qc, s.qc, true);
    Problem* p = batch.add_problem(h, s.qc, true, true, EPI_BF16, false, true);
    if (batch.error()) return batch.error();
    p->out0 = dWq[i];
    p->ld_out = s.qc;
    if ((rc = batch.add_seg(p, mx, 0, mq, -1, 0, T))) return rc;
  }
  for (int i = 0; i < t; ++i) {
    const __nv_bfloat16* G[3] = {dQ_of(i), dK_of(i), dV_of(i)};
    const ttl_bf16* const* W[3] = {Wq, Wk, Wv};
    if (!batch.has_room(6, 1) && (rc = batch.flush(st))) return rc;
    Problem* p = batch.add_problem(T, h, false, false, EPI_BF16, false);
    if (batch.error()) return batch.error();
    p->out0 = dX[i];
    p->ld_out = h;
    for (int w = 0; w < 3; ++w) {
      const int64_t cols = w == 0 ? s.qc : s.kc;
      const int mg = batch.add_map(G[w], T, cols, cols, false);
      const int mw = batch.add_map(W[w][i], h, cols, cols, false);
      if (batch.error()) return batch.error();
      if ((rc = batch.add_seg(p, mg, 0, mw, -1, 0, cols))) return rc;
    }
  }
  if ((rc = batch.flush(st))) return rc;

  // f backward: all-reduce of the dX partials.
  return shard_all_reduce_internal(t, T, h, dX, nullptr, st);
}

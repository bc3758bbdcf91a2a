// The tensor-parallel MLP block on t logical shards of one GPU:
//   f -> column-parallel fc1 (+ GeLU or SwiGLU, fused in the GEMM epilogue)
//     -> row-parallel fc2 (full-shape partial sums, one per shard buffer)
//     -> g: on-device all-reduce of the partials.
// Backward: g is the identity, fc2's dgrad and wgrad are local, the activation derivative
// is fused into fc2's dgrad epilogue, fc1's wgrad is local, and f all-reduces dX.
//
// Source: "v4:Tensor Parallel 与 Sequence Parallel" -- "TP 的数学:分块矩阵乘法",
// table "Column 和 Row 各在哪里通信", table "完整流程:column parallel,t = 3", the f/g
// pseudocode, "MLP:先 column,再 row" (GeLU(XA_1)B_1 + GeLU(XA_2)B_2; SwiGLU gate and up
// both column-split), and the bias answer under "自测" (row bias added once after the sum).
//
// Launches per call (t shards batched into one persistent GEMM launch each):
//   forward : fc1 (t problems) -> fc2 (t problems) -> all-reduce
//   backward: fc2 dgrad + act' (t) -> {fc2 wgrad, fc1 wgrad, fc1 dgrad} (3t or 4t)
//             -> all-reduce of dX (+ column sums for the bias gradients)

#include "ttl_internal.h"

namespace ttl {
namespace {

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

int check_ptrs(const void* const* arr, int t, const char* what, bool required) {
  if (!arr) return required ? set_error(TTL_ERR_ARG, "%s: null shard array", what) : TTL_OK;
  for (int i = 0; i < t; ++i) {
    if (!arr[i]) return set_error(TTL_ERR_ARG, "%s[%d] is null", what, i);
    if (!aligned16(arr[i])) return set_error(TTL_ERR_ALIGN, "%s[%d] not 16-byte aligned", what, i);
  }
  return TTL_OK;
}

int check_common(int t, int act, int64_t T, int64_t h, int64_t f, const char* name) {
  if (t < 1 || t > kMaxShards) return set_error(TTL_ERR_ARG, "%s: t=%d outside [1,%d]", name, t, kMaxShards);
  if (act != TTL_ACT_GELU_TANH && act != TTL_ACT_SWIGLU) return set_error(TTL_ERR_ARG, "%s: unknown act %d", name, act);
  if (T < 0 || h < 0 || f < 0) return set_error(TTL_ERR_ARG, "%s: negative shape", name);
  if (f % t) return set_error(TTL_ERR_SHAPE, "%s: t=%d must divide f=%lld", name, t, (long long)f);
  if (h % 8 || (f / t) % 8)
    return set_error(TTL_ERR_SHAPE, "%s: h and f/t must be multiples of 8 (16-byte rows)", name);
  if (T > 0 && (h == 0 || f == 0)) return set_error(TTL_ERR_SHAPE, "%s: h and f must be positive", name);
  if (T >= (int64_t(1) << 31) || h >= (int64_t(1) << 31) || f >= (int64_t(1) << 31))
    return set_error(TTL_ERR_SHAPE, "%s: extent beyond 2^31", name);
  return TTL_OK;
}

}  // namespace
}  // namespace ttl

using namespace ttl;

extern "C" int ttl_tp_mlp_fwd(int t, int act, int64_t T, int64_t h, int64_t f, const ttl_bf16* X,
                              const ttl_bf16* const* A, const ttl_bf16* const* A_up, const ttl_bf16* const* B,
                              const ttl_bf16* const* b1, const ttl_bf16* b2, ttl_bf16* const* U_save,
                              ttl_bf16* const* V_save, ttl_bf16* const* Hact, ttl_bf16* const* Z, void* stream) {
  const char* name = "ttl_tp_mlp_fwd";
  int rc = check_common(t, act, T, h, f, name);
  if (rc) return rc;
  if (T == 0) return TTL_OK;   // no tokens: every output is empty (its pointer may be null)
  const bool swiglu = act == TTL_ACT_SWIGLU;
  if (!X) return set_error(TTL_ERR_ARG, "%s: X is null", name);
  if (!aligned16(X)) return set_error(TTL_ERR_ALIGN, "%s: X not 16-byte aligned", name);
  using CP = const void* const*;
  if ((rc = check_ptrs(reinterpret_cast<CP>(A), t, "A", true))) return rc;
  if ((rc = check_ptrs(reinterpret_cast<CP>(B), t, "B", true))) return rc;
  if ((rc = check_ptrs(reinterpret_cast<CP>(U_save), t, "U_save", true))) return rc;
  if ((rc = check_ptrs(reinterpret_cast<CP>(Hact), t, "Hact", true))) return rc;
  if ((rc = check_ptrs(reinterpret_cast<CP>(Z), t, "Z", true))) return rc;
  if (swiglu) {
    if ((rc = check_ptrs(reinterpret_cast<CP>(A_up), t, "A_up", true))) return rc;
    if ((rc = check_ptrs(reinterpret_cast<CP>(V_save), t, "V_save", true))) return rc;
    if (b1) return set_error(TTL_ERR_ARG, "%s: the SwiGLU block takes no column bias", name);
  } else if ((rc = check_ptrs(reinterpret_cast<CP>(b1), t, "b1", false))) {
    return rc;
  }
  if (b2 && !aligned16(b2)) return set_error(TTL_ERR_ALIGN, "%s: b2 not 16-byte aligned", name);
  if (T == 0) return TTL_OK;

  const int64_t fs = f / t;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemmBatch batch;

  // fc1, column-parallel: U_i = X A_i (+ b1_i), activation fused in the epilogue.
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(swiglu ? 3 : 2, 1) && (rc = batch.flush(s))) return rc;
    const int mx = batch.add_map(X, T, h, h, false);
    const int ma = batch.add_map(A[i], h, fs, fs, true);
    const int mu = swiglu ? batch.add_map(A_up[i], h, fs, fs, true) : -1;
    Problem* p = batch.add_problem(T, fs, false, true, swiglu ? EPI_SWIGLU_FWD : EPI_GELU_FWD, swiglu, i > 0);
    if (batch.error()) return batch.error();
    p->out0 = U_save[i];
    p->out1 = swiglu ? static_cast<void*>(V_save[i]) : static_cast<void*>(Hact[i]);
    p->out2 = swiglu ? static_cast<void*>(Hact[i]) : nullptr;
    p->bias0 = (!swiglu && b1) ? b1[i] : nullptr;
    p->ld_out = fs;
    if ((rc = batch.add_seg(p, mx, 0, ma, mu, 0, h))) return rc;
  }
  if ((rc = batch.flush(s))) return rc;

  // fc2, row-parallel: P_i = H_i B_i, a full-shape partial in Z[i].
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(2, 1) && (rc = batch.flush(s))) return rc;
    const int mh = batch.add_map(Hact[i], T, fs, fs, false);
    const int mb = batch.add_map(B[i], fs, h, h, true);
    Problem* p = batch.add_problem(T, h, false, true, EPI_BF16, false);
    if (batch.error()) return batch.error();
    p->out0 = Z[i];
    p->ld_out = h;
    if ((rc = batch.add_seg(p, mh, 0, mb, -1, 0, fs))) return rc;
  }
  if ((rc = batch.flush(s))) return rc;

  // g forward: all-reduce of the partials; the row bias is added once, after the sum.
  return shard_all_reduce_internal(t, T, h, Z, b2, s);
}

extern "C" size_t ttl_tp_mlp_bwd_workspace_size(int t, int act, int64_t T, int64_t h, int64_t f) {
  if (t < 1 || t > kMaxShards || T < 0 || f < 0 || f % t) return 0;
  (void)h;
  const size_t per = round256(static_cast<size_t>(T) * static_cast<size_t>(f / t) * 2);
  return per * static_cast<size_t>(t) * (act == TTL_ACT_SWIGLU ? 2 : 1);
}

extern "C" int ttl_tp_mlp_bwd(int t, int act, int64_t T, int64_t h, int64_t f, const ttl_bf16* X, const ttl_bf16* dY,
                              const ttl_bf16* const* A, const ttl_bf16* const* A_up, const ttl_bf16* const* B,
                              const ttl_bf16* const* U_save, const ttl_bf16* const* V_save,
                              const ttl_bf16* const* Hact, ttl_bf16* const* dA, ttl_bf16* const* dA_up,
                              ttl_bf16* const* dB, ttl_bf16* const* db1, ttl_bf16* db2, ttl_bf16* const* dX, void* ws,
                              size_t ws_bytes, void* stream) {
  const char* name = "ttl_tp_mlp_bwd";
  int rc = check_common(t, act, T, h, f, name);
  if (rc) return rc;
  const bool swiglu = act == TTL_ACT_SWIGLU;
  const int64_t fs = f / t;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  using CP = const void* const*;
  if (T == 0) {
    // No tokens: every weight and bias gradient is an empty sum; token-sized buffers are
    // empty and may be null.
    if ((rc = check_ptrs(reinterpret_cast<CP>(dA), t, "dA", true))) return rc;
    if ((rc = check_ptrs(reinterpret_cast<CP>(dB), t, "dB", true))) return rc;
    if (swiglu && (rc = check_ptrs(reinterpret_cast<CP>(dA_up), t, "dA_up", true))) return rc;
    if (!swiglu && (rc = check_ptrs(reinterpret_cast<CP>(db1), t, "db1", false))) return rc;
    if (db2 && !aligned16(db2)) return set_error(TTL_ERR_ALIGN, "%s: db2 not 16-byte aligned", name);
    for (int i = 0; i < t; ++i) {
      if ((rc = fill_zero(dA[i], h * fs * 2, s))) return rc;
      if (swiglu && (rc = fill_zero(dA_up[i], h * fs * 2, s))) return rc;
      if ((rc = fill_zero(dB[i], fs * h * 2, s))) return rc;
      if (db1 && (rc = fill_zero(db1[i], fs * 2, s))) return rc;
    }
    return db2 ? fill_zero(db2, h * 2, s) : TTL_OK;
  }
  if (!X || !dY) return set_error(TTL_ERR_ARG, "%s: X or dY is null", name);
  if (!aligned16(X) || !aligned16(dY)) return set_error(TTL_ERR_ALIGN, "%s: X or dY not 16-byte aligned", name);
  if ((rc = check_ptrs(reinterpret_cast<CP>(A), t, "A", true))) return rc;
  if ((rc = check_ptrs(reinterpret_cast<CP>(B), t, "B", true))) return rc;
  if ((rc = check_ptrs(reinterpret_cast<CP>(U_save), t, "U_save", true))) return rc;
  if ((rc = check_ptrs(reinterpret_cast<CP>(Hact), t, "Hact", true))) return rc;
  if ((rc = check_ptrs(reinterpret_cast<CP>(dA), t, "dA", true))) return rc;
  if ((rc = check_ptrs(reinterpret_cast<CP>(dB), t, "dB", true))) return rc;
  if ((rc = check_ptrs(reinterpret_cast<CP>(dX), t, "dX", true))) return rc;
  if (swiglu) {
    if ((rc = check_ptrs(reinterpret_cast<CP>(A_up), t, "A_up", true))) return rc;
    if ((rc = check_ptrs(reinterpret_cast<CP>(V_save), t, "V_save", true))) return rc;
    if ((rc = check_ptrs(reinterpret_cast<CP>(dA_up), t, "dA_up", true))) return rc;
    if (db1) return set_error(TTL_ERR_ARG, "%s: the SwiGLU block has no column bias", name);
  } else if ((rc = check_ptrs(reinterpret_cast<CP>(db1), t, "db1", false))) {
    return rc;
  }
  if (db2 && !aligned16(db2)) return set_error(TTL_ERR_ALIGN, "%s: db2 not 16-byte aligned", name);
  const size_t need = ttl_tp_mlp_bwd_workspace_size(t, act, T, h, f);
  if (need && (!ws || ws_bytes < need))
    return set_error(TTL_ERR_ARG, "%s: workspace of %zu bytes needed, %zu given", name, need, ws_bytes);
  if (need && !aligned16(ws)) return set_error(TTL_ERR_ALIGN, "%s: workspace not 16-byte aligned", name);

  const size_t per = round256(static_cast<size_t>(T) * static_cast<size_t>(fs) * 2);
  auto ws_slot = [&](int k) { return static_cast<void*>(static_cast<char*>(ws) + per * static_cast<size_t>(k)); };
  // GeLU: dU_i = ws_slot(i).  SwiGLU: dG_i = ws_slot(i), dV_i = ws_slot(t + i).
  GemmBatch batch;

  // fc2 dgrad with the activation derivative fused: dH_i = dY B_i^T, then
  // GeLU: dU_i = dH_i * GeLU'(U_i);  SwiGLU: dG_i = dH_i * V_i * SiLU'(G_i), dV_i = dH_i * SiLU(G_i).
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(2, 1) && (rc = batch.flush(s))) return rc;
    const int md = batch.add_map(dY, T, h, h, false);
    const int mb = batch.add_map(B[i], fs, h, h, false);
    Problem* p = batch.add_problem(T, fs, false, false, swiglu ? EPI_SWIGLU_BWD : EPI_GELU_BWD, false, i > 0);
    if (batch.error()) return batch.error();
    p->out0 = ws_slot(i);
    p->out1 = swiglu ? ws_slot(t + i) : nullptr;
    p->aux0 = U_save[i];
    p->aux1 = swiglu ? static_cast<const void*>(V_save[i]) : nullptr;
    p->ld_out = fs;
    p->ld_aux = fs;
    if ((rc = batch.add_seg(p, md, 0, mb, -1, 0, h))) return rc;
  }
  if ((rc = batch.flush(s))) return rc;

  // Weight gradients (all local), one launch for all shards.  Problems that share an operand
  // sit next to each other in the tile order -- every X^T wgrad, then every dY one -- and all
  // of them contract over the T tokens, so the persistent CTAs stay on neighbouring tiles of
  // equal cost and the shared operand is served from L2.
  // dA_i = X^T dU_i (SwiGLU: dWg_i = X^T dG_i and dWu_i = X^T dV_i).
  for (int k = 0; k < (swiglu ? 2 : 1); ++k) {
    for (int i = 0; i < t; ++i) {
      if (!batch.has_room(2, 1) && (rc = batch.flush(s))) return rc;
      const int ma = batch.add_map(X, T, h, h, true);
      const int mb = batch.add_map(ws_slot(k * t + i), T, fs, fs, true);
      Problem* p = batch.add_problem(h, fs, true, true, EPI_BF16, false, k + i > 0);
      if (batch.error()) return batch.error();
      p->out0 = k == 0 ? static_cast<void*>(dA[i]) : static_cast<void*>(dA_up[i]);
      p->ld_out = fs;
      if ((rc = batch.add_seg(p, ma, 0, mb, -1, 0, T))) return rc;
    }
  }
  // dB_i = H_i^T dY: A = H_i stored [T, f/t] (M-major), B = dY stored [T, h] (N-major).
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(2, 1) && (rc = batch.flush(s))) return rc;
    const int ma = batch.add_map(Hact[i], T, fs, fs, true);
    const int mb = batch.add_map(dY, T, h, h, true);
    Problem* p = batch.add_problem(fs, h, true, true, EPI_BF16, false);
    if (batch.error()) return batch.error();
    p->out0 = dB[i];
    p->ld_out = h;
    if ((rc = batch.add_seg(p, ma, 0, mb, -1, 0, T))) return rc;
  }
  if ((rc = batch.flush(s))) return rc;

  // dX partials, one launch: dX_i = dU_i A_i^T (SwiGLU: dG_i Wg_i^T + dV_i Wu_i^T, one
  // accumulator, two K segments).
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(swiglu ? 4 : 2, 1) && (rc = batch.flush(s))) return rc;
    const int mdu = batch.add_map(ws_slot(i), T, fs, fs, false);
    const int mwa = batch.add_map(A[i], h, fs, fs, false);
    Problem* p = batch.add_problem(T, h, false, false, EPI_BF16, false);
    if (batch.error()) return batch.error();
    p->out0 = dX[i];
    p->ld_out = h;
    if ((rc = batch.add_seg(p, mdu, 0, mwa, -1, 0, fs))) return rc;
    if (swiglu) {
      const int mdv = batch.add_map(ws_slot(t + i), T, fs, fs, false);
      const int mwu = batch.add_map(A_up[i], h, fs, fs, false);
      if (batch.error()) return batch.error();
      if ((rc = batch.add_seg(p, mdv, 0, mwu, -1, 0, fs))) return rc;
    }
  }
  if ((rc = batch.flush(s))) return rc;

  // Bias gradients: db1_i = column sums of dU_i; db2 = column sums of dY, once.
  if (db1)
    for (int i = 0; i < t; ++i)
      if ((rc = column_sum_bf16(ws_slot(i), T, fs, fs, db1[i], s))) return rc;
  if (db2 && (rc = column_sum_bf16(dY, T, h, h, db2, s))) return rc;

  // f backward: all-reduce of the dX partials.
  return shard_all_reduce_internal(t, T, h, dX, nullptr, s);
}

// Sequence-parallel MLP block with its collectives folded into the GEMMs.
//
// Source: "v4:Tensor Parallel 与 Sequence Parallel", section "SP": after a row-parallel layer
// the all-reduce becomes a reduce-scatter (each card keeps its own s/t tokens), and an
// all-gather before the next column-parallel layer rebuilds the full sequence; the TP
// communication page's "怎么优化 TP 的 all-reduce" answer pairs this with splitting the GEMM
// so the all-gather / reduce-scatter overlap it.
//
// Here the block's input and output are t token slabs [T/t, h] and no collective kernel runs:
//   all-gather    -> fc1's A operand is read through one tensor map per slab; a 256-row tile
//                    takes its rows from the slab that holds them;
//   reduce-scatter-> fc2's output slab r is ONE accumulator whose K loop walks the t shards'
//                    H_i[slab r] W_i, so no full-shape partial ever reaches HBM.
// Backward: the reduce-scatter's backward (an all-gather of the dZ slabs) is folded into the
// dgrad's A loads and into the K segments of the weight gradients, and the all-gather's
// backward (a reduce-scatter of the dX partials) into the dX GEMM's K loop over shards.
// Summing the shards inside the fp32 accumulator skips the bf16 rounding of each partial
// that the literal block applies; the results agree within the GEMM tolerance.

#include "ttl_internal.h"

namespace ttl {
namespace {

int check_arr(const void* const* a, int n, const char* what, bool required) {
  if (!a) return required ? set_error(TTL_ERR_ARG, "%s: null array", what) : TTL_OK;
  for (int i = 0; i < n; ++i) {
    if (!a[i]) return set_error(TTL_ERR_ARG, "%s[%d] is null", what, i);
    if (!aligned16(a[i])) return set_error(TTL_ERR_ALIGN, "%s[%d] not 16-byte aligned", what, i);
  }
  return TTL_OK;
}

int check_sp(int t, int act, int64_t T, int64_t h, int64_t f, const char* name) {
  if (t < 1 || t > kMaxShards) return set_error(TTL_ERR_ARG, "%s: t=%d outside [1,%d]", name, t, kMaxShards);
  if (act != TTL_ACT_GELU_TANH && act != TTL_ACT_SWIGLU) return set_error(TTL_ERR_ARG, "%s: unknown act %d", name, act);
  if (T < 0 || h < 0 || f < 0) return set_error(TTL_ERR_ARG, "%s: negative shape", name);
  if (f % t || T % t) return set_error(TTL_ERR_SHAPE, "%s: t=%d must divide f and T", name, t);
  if (h % 8 || (f / t) % 8) return set_error(TTL_ERR_SHAPE, "%s: h and f/t must be multiples of 8", name);
  if (T > 0 && ((T / t) % 128)) return set_error(TTL_ERR_SHAPE, "%s: token slabs T/t must be multiples of 128", name);
  if (T > 0 && (h == 0 || f == 0)) return set_error(TTL_ERR_SHAPE, "%s: h and f must be positive", name);
  if (T >= (int64_t(1) << 31) || h >= (int64_t(1) << 31) || f >= (int64_t(1) << 31))
    return set_error(TTL_ERR_SHAPE, "%s: extent beyond 2^31", name);
  return TTL_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace ttl

using namespace ttl;

extern "C" int ttl_sp_mlp_fwd(int t, int act, int64_t T, int64_t h, int64_t f, const ttl_bf16* const* X_slabs,
                              const ttl_bf16* const* A, const ttl_bf16* const* A_up, const ttl_bf16* const* B,
                              ttl_bf16* const* U_save, ttl_bf16* const* V_save, ttl_bf16* const* Hact,
                              ttl_bf16* const* Z_slabs, void* stream) {
  const char* name = "ttl_sp_mlp_fwd";
  int rc = check_sp(t, act, T, h, f, name);
  if (rc) return rc;
  if (T == 0) return TTL_OK;
  const bool swiglu = act == TTL_ACT_SWIGLU;
  using CP = const void* const*;
  if ((rc = check_arr(reinterpret_cast<CP>(X_slabs), t, "X_slabs", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(A), t, "A", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(B), t, "B", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(U_save), t, "U_save", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(Hact), t, "Hact", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(Z_slabs), t, "Z_slabs", true))) return rc;
  if (swiglu) {
    if ((rc = check_arr(reinterpret_cast<CP>(A_up), t, "A_up", true))) return rc;
    if ((rc = check_arr(reinterpret_cast<CP>(V_save), t, "V_save", true))) return rc;
  }
  const int64_t fs = f / t, slab = T / t;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemmBatch batch;

  // fc1 with the all-gather folded: A = X read slab by slab.
  int mx = -1;
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(swiglu ? 2 : 1, 1)) {
      if ((rc = batch.flush(s))) return rc;
      mx = -1;
    }
    if (mx < 0) mx = batch.add_maps_consecutive(reinterpret_cast<CP>(X_slabs), t, slab, h, h, false);
    const int ma = batch.add_map(A[i], h, fs, fs, true);
    const int mu = swiglu ? batch.add_map(A_up[i], h, fs, fs, true) : -1;
    Problem* p = batch.add_problem(T, fs, false, true, swiglu ? EPI_SWIGLU_FWD : EPI_GELU_FWD, swiglu, i > 0);
    if (batch.error()) return batch.error();
    p->a_slab_rows = static_cast<int32_t>(slab);
    p->out0 = U_save[i];
    p->out1 = swiglu ? static_cast<void*>(V_save[i]) : static_cast<void*>(Hact[i]);
    p->out2 = swiglu ? static_cast<void*>(Hact[i]) : nullptr;
    p->ld_out = fs;
    if ((rc = batch.add_seg(p, mx, 0, ma, mu, 0, h))) return rc;
  }
  if ((rc = batch.flush(s))) return rc;

  // fc2 with the reduce-scatter folded: slab r = sum_i H_i[slab r] B_i in one accumulator.
  // (every slab problem reads the same 2t operands: only the first one registers new maps)
  for (int r = 0; r < t; ++r) {
    if (!batch.has_room(r == 0 ? 2 * t : 0, 1) && (rc = batch.flush(s))) return rc;
    Problem* p = batch.add_problem(slab, h, false, true, EPI_BF16, false);
    if (batch.error()) return batch.error();
    p->a_m0 = static_cast<int32_t>(r * slab);
    p->out0 = Z_slabs[r];
    p->ld_out = h;
    for (int i = 0; i < t; ++i) {
      const int mh = batch.add_map(Hact[i], T, fs, fs, false);
      const int mb = batch.add_map(B[i], fs, h, h, true);
      if ((rc = batch.add_seg(p, mh, 0, mb, -1, 0, fs))) return rc;
    }
  }
  return batch.flush(s);
}

extern "C" size_t ttl_sp_mlp_bwd_workspace_size(int t, int act, int64_t T, int64_t h, int64_t f) {
  if (t < 1 || t > kMaxShards || T < 0 || f < 0 || f % t) return 0;
  (void)h;
  return round256(static_cast<size_t>(T) * static_cast<size_t>(f / t) * 2) * static_cast<size_t>(t) *
         (act == TTL_ACT_SWIGLU ? 2 : 1);
}

extern "C" int ttl_sp_mlp_bwd(int t, int act, int64_t T, int64_t h, int64_t f, const ttl_bf16* const* X_slabs,
                              const ttl_bf16* const* dZ_slabs, const ttl_bf16* const* A,
                              const ttl_bf16* const* A_up, const ttl_bf16* const* B, const ttl_bf16* const* U_save,
                              const ttl_bf16* const* V_save, const ttl_bf16* const* Hact, ttl_bf16* const* dA,
                              ttl_bf16* const* dA_up, ttl_bf16* const* dB, ttl_bf16* const* dX_slabs, void* ws,
                              size_t ws_bytes, void* stream) {
  const char* name = "ttl_sp_mlp_bwd";
  int rc = check_sp(t, act, T, h, f, name);
  if (rc) return rc;
  const bool swiglu = act == TTL_ACT_SWIGLU;
  if (swiglu && 2 * t > kMaxSegs)
    return set_error(TTL_ERR_UNSUPPORTED, "%s: the SwiGLU dX contraction walks 2t segments; t <= %d", name, kMaxSegs / 2);
  using CP = const void* const*;
  if ((rc = check_arr(reinterpret_cast<CP>(dA), t, "dA", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(dB), t, "dB", true))) return rc;
  if (swiglu && (rc = check_arr(reinterpret_cast<CP>(dA_up), t, "dA_up", true))) return rc;
  const int64_t fs = f / t, slab = T / t;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    for (int i = 0; i < t; ++i) {
      if ((rc = fill_zero(dA[i], h * fs * 2, s))) return rc;
      if (swiglu && (rc = fill_zero(dA_up[i], h * fs * 2, s))) return rc;
      if ((rc = fill_zero(dB[i], fs * h * 2, s))) return rc;
    }
    return TTL_OK;
  }
  if ((rc = check_arr(reinterpret_cast<CP>(X_slabs), t, "X_slabs", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(dZ_slabs), t, "dZ_slabs", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(A), t, "A", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(B), t, "B", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(U_save), t, "U_save", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(Hact), t, "Hact", true))) return rc;
  if ((rc = check_arr(reinterpret_cast<CP>(dX_slabs), t, "dX_slabs", true))) return rc;
  if (swiglu) {
    if ((rc = check_arr(reinterpret_cast<CP>(A_up), t, "A_up", true))) return rc;
    if ((rc = check_arr(reinterpret_cast<CP>(V_save), t, "V_save", true))) return rc;
  }
  const size_t need = ttl_sp_mlp_bwd_workspace_size(t, act, T, h, f);
  if (!ws || ws_bytes < need)
    return set_error(TTL_ERR_ARG, "%s: workspace of %zu bytes needed, %zu given", name, need, ws_bytes);
  if (!aligned16(ws)) return set_error(TTL_ERR_ALIGN, "%s: workspace not 16-byte aligned", name);
  const size_t per = round256(static_cast<size_t>(T) * static_cast<size_t>(fs) * 2);
  auto ws_slot = [&](int k) { return static_cast<void*>(static_cast<char*>(ws) + per * static_cast<size_t>(k)); };
  GemmBatch batch;

  // fc2 dgrad with the activation derivative fused; A = dZ read slab by slab (the backward of
  // the reduce-scatter is this all-gather).
  int mdz = -1;
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(1, 1)) {
      if ((rc = batch.flush(s))) return rc;
      mdz = -1;
    }
    if (mdz < 0) mdz = batch.add_maps_consecutive(reinterpret_cast<CP>(dZ_slabs), t, slab, h, h, false);
    const int mb = batch.add_map(B[i], fs, h, h, false);
    Problem* p = batch.add_problem(T, fs, false, false, swiglu ? EPI_SWIGLU_BWD : EPI_GELU_BWD, false, i > 0);
    if (batch.error()) return batch.error();
    p->a_slab_rows = static_cast<int32_t>(slab);
    p->out0 = ws_slot(i);
    p->out1 = swiglu ? ws_slot(t + i) : nullptr;
    p->aux0 = U_save[i];
    p->aux1 = swiglu ? static_cast<const void*>(V_save[i]) : nullptr;
    p->ld_out = fs;
    p->ld_aux = fs;
    if ((rc = batch.add_seg(p, mdz, 0, mb, -1, 0, h))) return rc;
  }
  if ((rc = batch.flush(s))) return rc;

  // Weight gradients: the token contraction walks the slabs as K segments.
  //   dA_i = X^T dU_i  (SwiGLU: dWg_i = X^T dG_i, dWu_i = X^T dV_i): A = X slab r, B = dU_i rows of slab r
  int mxs = -1;
  for (int k = 0; k < (swiglu ? 2 : 1); ++k) {
    for (int i = 0; i < t; ++i) {
      if (!batch.has_room(1, 1)) {
        if ((rc = batch.flush(s))) return rc;
        mxs = -1;
      }
      if (mxs < 0) mxs = batch.add_maps_consecutive(reinterpret_cast<CP>(X_slabs), t, slab, h, h, true);
      const int mb = batch.add_map(ws_slot(k * t + i), T, fs, fs, true);
      Problem* p = batch.add_problem(h, fs, true, true, EPI_BF16, false, k + i > 0);
      if (batch.error()) return batch.error();
      p->out0 = k == 0 ? static_cast<void*>(dA[i]) : static_cast<void*>(dA_up[i]);
      p->ld_out = fs;
      for (int r = 0; r < t; ++r)
        if ((rc = batch.add_seg(p, mxs + r, 0, mb, -1, r * slab, slab))) return rc;
    }
  }
  //   dB_i = H_i^T dZ: A = H_i rows of slab r, B = dZ slab r.
  int mzs = -1;
  for (int i = 0; i < t; ++i) {
    if (!batch.has_room(1, 1)) {
      if ((rc = batch.flush(s))) return rc;
      mzs = -1;
    }
    if (mzs < 0) mzs = batch.add_maps_consecutive(reinterpret_cast<CP>(dZ_slabs), t, slab, h, h, true);
    const int ma = batch.add_map(Hact[i], T, fs, fs, true);
    Problem* p = batch.add_problem(fs, h, true, true, EPI_BF16, false);
    if (batch.error()) return batch.error();
    p->out0 = dB[i];
    p->ld_out = h;
    for (int r = 0; r < t; ++r)
      if ((rc = batch.add_seg(p, ma, r * slab, mzs + r, -1, 0, slab))) return rc;
  }
  if ((rc = batch.flush(s))) return rc;

  // dX with the reduce-scatter folded: slab r = sum_i dU_i[slab r] A_i^T (SwiGLU: both halves).
  for (int r = 0; r < t; ++r) {
    if (!batch.has_room(r == 0 ? (swiglu ? 4 * t : 2 * t) : 0, 1) && (rc = batch.flush(s))) return rc;
    Problem* p = batch.add_problem(slab, h, false, false, EPI_BF16, false);
    if (batch.error()) return batch.error();
    p->a_m0 = static_cast<int32_t>(r * slab);
    p->out0 = dX_slabs[r];
    p->ld_out = h;
    for (int i = 0; i < t; ++i) {
      const int md = batch.add_map(ws_slot(i), T, fs, fs, false);
      const int mw = batch.add_map(A[i], h, fs, fs, false);
      if ((rc = batch.add_seg(p, md, 0, mw, -1, 0, fs))) return rc;
      if (swiglu) {
        const int mv = batch.add_map(ws_slot(t + i), T, fs, fs, false);
        const int mu = batch.add_map(A_up[i], h, fs, fs, false);
        if ((rc = batch.add_seg(p, mv, 0, mu, -1, 0, fs))) return rc;
      }
    }
  }
  return batch.flush(s);
}

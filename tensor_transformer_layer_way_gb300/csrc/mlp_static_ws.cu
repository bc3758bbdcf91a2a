// ttl_tp_mlp_bwd_static_ws: the MLP backward for callers that cannot allocate device memory.
//
// ttl_tp_mlp_bwd needs a scratch area (the per-shard activation gradients) that its caller
// allocates.  Some callers have no way to do that: a host program whose device memory is
// owned entirely by another allocator (an inference or training runtime that reserved its
// pool up front and forbids further cudaMalloc), or a latency-critical loop that must not
// pay cudaMalloc's cost or its implicit device-wide synchronisation.  For them this file
// provides the scratch itself, as a fixed-size array in the library's own device memory.
//
// The array lives in every GPU that loads the library, from module load until the process
// exits.  Host code cannot use the array's name as a pointer (it is only a host-side handle
// for the symbol); the device address is looked up once per device with
// cudaGetSymbolAddress while that device is current, and then passed to the kernels.

#include <mutex>

#include "ttl_internal.h"

namespace ttl {
namespace {

// The scratch: TTL_STATIC_WS_BYTES bytes, 256-byte aligned, one copy per device.
static __device__ __align__(256) unsigned char g_mlp_bwd_static_ws[TTL_STATIC_WS_BYTES];

constexpr int kMaxDevs = 64;
std::mutex g_ws_mu;
void* g_ws_ptr[kMaxDevs] = {nullptr};

// Device address of the scratch on the current device (set up on first use per device).
int static_ws_ptr(void** out) {
  int dev = 0;
  int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= kMaxDevs) return set_error(TTL_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_ws_mu);
  if (!g_ws_ptr[dev]) {
    void* p = nullptr;
    rc = cuda_check(cudaGetSymbolAddress(&p, g_mlp_bwd_static_ws), "cudaGetSymbolAddress(static scratch)");
    if (rc) return rc;
    g_ws_ptr[dev] = p;
  }
  *out = g_ws_ptr[dev];
  return TTL_OK;
}

}  // namespace
}  // namespace ttl

extern "C" int ttl_tp_mlp_bwd_static_ws(int t, int act, int64_t T, int64_t h, int64_t f, const ttl_bf16* X,
                                        const ttl_bf16* dY, const ttl_bf16* const* A, const ttl_bf16* const* A_up,
                                        const ttl_bf16* const* B, const ttl_bf16* const* U_save,
                                        const ttl_bf16* const* V_save, const ttl_bf16* const* Hact,
                                        ttl_bf16* const* dA, ttl_bf16* const* dA_up, ttl_bf16* const* dB,
                                        ttl_bf16* const* db1, ttl_bf16* db2, ttl_bf16* const* dX, void* stream) {
  using namespace ttl;
  const size_t need = ttl_tp_mlp_bwd_workspace_size(t, act, T, h, f);
  if (need > static_cast<size_t>(TTL_STATIC_WS_BYTES))
    return set_error(TTL_ERR_UNSUPPORTED,
                     "ttl_tp_mlp_bwd_static_ws: this shape needs %zu bytes of scratch but the built-in area holds %zu; "
                     "use ttl_tp_mlp_bwd with a caller-provided workspace",
                     need, static_cast<size_t>(TTL_STATIC_WS_BYTES));
  void* ws = nullptr;
  int rc = static_ws_ptr(&ws);
  if (rc) return rc;
  // Every element of the scratch is written (by the fc2 dgrad epilogue) before it is read,
  // so nothing left over from an earlier call needs clearing.
  return ttl_tp_mlp_bwd(t, act, T, h, f, X, dY, A, A_up, B, U_save, V_save, Hact, dA, dA_up, dB, db1, db2, dX, ws,
                        static_cast<size_t>(TTL_STATIC_WS_BYTES), stream);
}

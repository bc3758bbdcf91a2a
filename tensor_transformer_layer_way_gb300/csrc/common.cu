// Host-side plumbing shared by every entry point: thread-local error text, the per-device
// status word that kernels write when a bounded wait runs out or an input is invalid,
// device queries, and the failure-path self test.

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ttl_device.cuh"
#include "ttl_internal.h"

namespace ttl {

namespace {
thread_local char g_last_error[512] = "no error";

// One status word per device.  Kernels receive its device address as a parameter.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int* g_status_ptr[kMaxDevices] = {nullptr};
int g_sms[kMaxDevices] = {0};
int g_cc[kMaxDevices] = {0};
}  // namespace

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return TTL_OK;
  return set_error(TTL_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

int cu_check(CUresult r, const char* what) {
  if (r == CUDA_SUCCESS) return TTL_OK;
  return set_error(TTL_ERR_CUDA, "%s: driver error %d", what, static_cast<int>(r));
}

static int current_device(int* dev) {
  int rc = cuda_check(cudaGetDevice(dev), "cudaGetDevice");
  if (rc) return rc;
  if (*dev < 0 || *dev >= kMaxDevices) return set_error(TTL_ERR_CUDA, "device index %d out of range", *dev);
  return TTL_OK;
}

int* device_status_ptr() {
  int dev = 0;
  if (current_device(&dev)) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cuda_check(cudaGetSymbolAddress(&p, g_status_word), "cudaGetSymbolAddress(status)")) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

static int query_device(int dev) {
  if (g_sms[dev]) return TTL_OK;
  cudaDeviceProp prop;
  int rc = cuda_check(cudaGetDeviceProperties(&prop, dev), "cudaGetDeviceProperties");
  if (rc) return rc;
  g_sms[dev] = prop.multiProcessorCount;
  g_cc[dev] = prop.major * 10 + prop.minor;
  return TTL_OK;
}

int num_sms() {
  int dev = 0;
  if (current_device(&dev)) return 1;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (query_device(dev)) return 1;
  return g_sms[dev];
}

int require_sm103() {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if ((rc = query_device(dev))) return rc;
  if (g_cc[dev] != 103)
    return set_error(TTL_ERR_UNSUPPORTED, "device %d has compute capability %d.%d; this library is built for sm_103a",
                     dev, g_cc[dev] / 10, g_cc[dev] % 10);
  return TTL_OK;
}

// ------------------------------------------------------------------ launch tracing

namespace {
struct TraceRec {
  cudaEvent_t start, stop;
  int kind;
  double flops, bytes;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
TraceRec* g_trace = nullptr;
int g_trace_cap = 0;
int g_trace_n = 0;

void trace_free() {
  for (int i = 0; i < g_trace_cap; ++i) {
    cudaEventDestroy(g_trace[i].start);
    cudaEventDestroy(g_trace[i].stop);
  }
  delete[] g_trace;
  g_trace = nullptr;
  g_trace_cap = 0;
  g_trace_n = 0;
}
}  // namespace

int trace_begin(cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  if (!g_trace_on || g_trace_n >= g_trace_cap) return -1;
  const int slot = g_trace_n++;
  cudaEventRecord(g_trace[slot].start, s);
  return slot;
}

void trace_end(int slot, cudaStream_t s, int kind, double flops, double bytes) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lock(g_trace_mu);
  if (!g_trace || slot >= g_trace_cap) return;
  g_trace[slot].kind = kind;
  g_trace[slot].flops = flops;
  g_trace[slot].bytes = bytes;
  cudaEventRecord(g_trace[slot].stop, s);
}

// ------------------------------------------------------------------ small kernels

__global__ void fill_zero_kernel(uint4* p, size_t n16, uint8_t* tail, size_t ntail) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16; i += stride)
    p[i] = make_uint4(0, 0, 0, 0);
  if (blockIdx.x == 0 && threadIdx.x < ntail) tail[threadIdx.x] = 0;
}

int fill_zero(void* ptr, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return TTL_OK;
  if (!aligned16(ptr)) return set_error(TTL_ERR_ALIGN, "fill_zero: pointer not 16-byte aligned");
  const size_t n16 = bytes / 16;
  const size_t ntail = bytes % 16;
  size_t blocks = (n16 + 255) / 256;
  const size_t cap = static_cast<size_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  fill_zero_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<uint4*>(ptr), n16, static_cast<uint8_t*>(ptr) + n16 * 16, ntail);
  return cuda_check(cudaGetLastError(), "fill_zero_kernel launch");
}

// One thread initialises an mbarrier that expects an arrival nobody makes, then waits on
// it with the same bounded wait the GEMM uses.
__global__ void wait_timeout_selftest_kernel(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_wait(&bar, 0, &abort_flag, status, timeout_ns);
  }
}

}  // namespace ttl

// ------------------------------------------------------------------ C entry points

extern "C" const char* ttl_last_error(void) { return ttl::g_last_error; }

extern "C" int ttl_version(void) { return 100; }

extern "C" int ttl_device_status(void* stream, int* status_out) {
  using namespace ttl;
  if (!status_out) return set_error(TTL_ERR_ARG, "ttl_device_status: null output");
  int rc = cuda_check(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "cudaStreamSynchronize");
  if (rc) return rc;
  int* p = device_status_ptr();
  if (!p) return TTL_ERR_CUDA;
  int v = 0;
  if ((rc = cuda_check(cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost), "read status word"))) return rc;
  if (v != 0) {
    const int zero = 0;
    if ((rc = cuda_check(cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice), "clear status word"))) return rc;
    set_error(v, "a kernel reported status %d", v);
  }
  *status_out = v;
  return TTL_OK;
}

extern "C" int ttl_trace_enable(int on, int capacity) {
  using namespace ttl;
  std::lock_guard<std::mutex> lock(g_trace_mu);
  if (!on) {
    g_trace_on = false;
    return TTL_OK;
  }
  if (capacity < 1 || capacity > (1 << 20)) return set_error(TTL_ERR_ARG, "trace capacity must be in [1, 2^20]");
  if (capacity != g_trace_cap) {
    trace_free();
    g_trace = new TraceRec[capacity];
    for (int i = 0; i < capacity; ++i) {
      g_trace[i] = TraceRec{nullptr, nullptr, TTL_K_OTHER, 0.0, 0.0};
      int rc = cuda_check(cudaEventCreate(&g_trace[i].start), "cudaEventCreate");
      if (!rc) rc = cuda_check(cudaEventCreate(&g_trace[i].stop), "cudaEventCreate");
      if (rc) {
        g_trace_cap = i + 1;
        trace_free();
        return rc;
      }
    }
    g_trace_cap = capacity;
  }
  g_trace_n = 0;
  g_trace_on = true;
  return TTL_OK;
}

extern "C" int ttl_trace_read(int max, int* kind, float* ms, double* flops, double* bytes, int* count) {
  using namespace ttl;
  if (!count || max < 0 || (max > 0 && (!kind || !ms || !flops || !bytes)))
    return set_error(TTL_ERR_ARG, "ttl_trace_read: bad arguments");
  std::lock_guard<std::mutex> lock(g_trace_mu);
  *count = g_trace_n;
  const int n = g_trace_n < max ? g_trace_n : max;
  for (int i = 0; i < n; ++i) {
    int rc = cuda_check(cudaEventSynchronize(g_trace[i].stop), "cudaEventSynchronize");
    if (rc) return rc;
    float t = 0.0f;
    if ((rc = cuda_check(cudaEventElapsedTime(&t, g_trace[i].start, g_trace[i].stop), "cudaEventElapsedTime")))
      return rc;
    kind[i] = g_trace[i].kind;
    ms[i] = t;
    flops[i] = g_trace[i].flops;
    bytes[i] = g_trace[i].bytes;
  }
  return TTL_OK;
}

extern "C" int ttl_selftest_wait_timeout(int64_t timeout_us, void* stream) {
  using namespace ttl;
  if (timeout_us < 1 || timeout_us > 1000000) return set_error(TTL_ERR_ARG, "timeout_us must be in [1, 1e6]");
  int rc = require_sm103();
  if (rc) return rc;
  int* st = device_status_ptr();
  if (!st) return TTL_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(st, static_cast<uint64_t>(timeout_us) * 1000u);
  if ((rc = cuda_check(cudaGetLastError(), "selftest launch"))) return rc;
  int status = 0;
  if ((rc = ttl_device_status(stream, &status))) return rc;
  return status;
}

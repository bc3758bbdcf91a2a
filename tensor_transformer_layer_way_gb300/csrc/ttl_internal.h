// Internal declarations shared by the library's translation units (host side) and the
// GEMM problem description that crosses into the kernel as a parameter block.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ttl.h"

namespace ttl {

constexpr int kMaxShards = TTL_MAX_SHARDS;

// ------------------------------------------------------------------ errors

// Records a formatted message for ttl_last_error() and returns `code`.
int set_error(int code, const char* fmt, ...);
// TTL_OK if e == cudaSuccess, else records the CUDA error string.
int cuda_check(cudaError_t e, const char* what);
// TTL_OK if r == CUDA_SUCCESS, else records the driver error.
int cu_check(CUresult r, const char* what);

// Device address of the current device's status word (looked up once per device).
int* device_status_ptr();
// Multiprocessor count of the current device (cached per device).
int num_sms();
// TTL_OK if the current device is sm_103 (compute capability 10.3).
int require_sm103();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch tracing (no-ops unless ttl_trace_enable(1, ...) was called).  trace_begin records
// the start event on `s` and returns a slot (or -1); trace_end records the stop event.
int trace_begin(cudaStream_t s);
void trace_end(int slot, cudaStream_t s, int kind, double flops, double bytes);

// RAII helper: brackets one launch.
struct TraceScope {
  int slot;
  cudaStream_t s;
  int kind;
  double flops, bytes;
  TraceScope(cudaStream_t st, int k, double f, double b) : slot(trace_begin(st)), s(st), kind(k), flops(f), bytes(b) {}
  ~TraceScope() { trace_end(slot, s, kind, flops, bytes); }
};

// ------------------------------------------------------------------ GEMM problem block

constexpr int kGemmBN = 256;   // accumulator columns per GEMM tile
constexpr int kMaxMaps = 96;
constexpr int kMaxProblems = 32;
constexpr int kMaxSegs = kMaxShards;

enum Epilogue : int {
  EPI_BF16 = 0,        // out0 = bf16(acc + bias0[n])
  EPI_F32 = 1,         // out0 = acc (fp32)
  EPI_GELU_FWD = 2,    // out0 = U = bf16(acc + bias0[n]); out1 = bf16(GeLU(acc + bias0[n]))
  EPI_SWIGLU_FWD = 3,  // paired tile: out0 = G, out1 = V, out2 = SiLU(G) * V
  EPI_GELU_BWD = 4,    // out0 = bf16(acc * GeLU'(aux0))                          (dU)
  EPI_SWIGLU_BWD = 5,  // out0 = bf16(acc * aux1 * SiLU'(aux0)), out1 = bf16(acc * SiLU(aux0))
  EPI_F32_CE = 6,      // out0 = acc (fp32 logits) and, per row and 128-column chunk c of the
                       // problem, the cross-entropy partials: out1[row * ext1 + cbase + c] =
                       // (max, sum exp(z - max)) over the chunk's columns (chunks counted 2 per
                       // 256-column tile, so every chunk below 2 ceil(N / 256) is written);
                       // out2[row] = the logit at target aux0[row] - ext0 when that column exists
  EPI_PAIR_BF16 = 7,   // paired tile: out0 = bf16(accumulator columns [0,128)) from map_b,
                       // out1 = bf16(columns [128,256)) from map_b2 (two narrow products as one
                       // full-width MMA, e.g. the K and V projections of a shard)
};

// One K-range of a problem: k-blocks of 64 read from map_a at K offset a_k0 and from
// map_b (and, for a paired tile, map_b2) at K offset b_k0; b_n1 is added to B's N
// coordinate for this segment only (e.g. one head's columns of a head-major operand).
struct Seg {
  int16_t map_a, map_b, map_b2, pad;
  int32_t a_k0, b_k0, kblocks, b_n1;
};

// One output matrix [M, N]; tiles of 128 rows x 256 accumulator columns.  A paired tile
// (SwiGLU forward, EPI_PAIR_BF16) covers 128 output columns: accumulator columns [0,128)
// come from map_b and [128,256) from map_b2 at the same N coordinates.
struct Problem {
  int32_t M, N;
  int32_t tiles_m, tiles_n;
  int32_t tn0;            // first n-tile of this problem within its group's n-tile range
  int32_t cbase;          // EPI_F32_CE: first partial of this problem in a row of out1 (set by launch())
  int32_t a_m0, b_n0;     // offsets added to the M coordinate of A and N coordinate of B
  int32_t a_slab_rows;    // > 0: A's rows live in consecutive maps seg.map_a + r, r = row / a_slab_rows
                          // (token slabs, e.g. an all-gather folded into the operand loads)
  uint8_t a_mn, b_mn;     // 1 = operand stored MN-major (A as [K,M], B as [K,N])
  uint8_t epi, nseg;
  uint8_t paired;
  uint8_t join;           // 1 = same tile group as the previous problem (shares its A rows)
  uint8_t omap;           // set by launch() for the wide kernel: the map of out0 its TMA stores use
  uint8_t half_n;         // set by launch() when N <= 128 (unpaired): the MMAs are 128 columns wide
  Seg seg[kMaxSegs];
  void* out0;
  void* out1;
  void* out2;
  const void* aux0;
  const void* aux1;
  const void* bias0;
  int64_t ld_out;         // row stride (elements) of out0/out1/out2
  int64_t ld_aux;         // row stride (elements) of aux0/aux1
  int64_t ext0, ext1;     // epilogue-specific integers (EPI_F32_CE: vocab offset, row stride of out1)
};

// Consecutive problems with the same M that read the same A rows form one tile group: its
// tiles are ordered band by band over M (GROUP_M tiles tall) and, inside a band, across the
// n-tiles of every problem of the group, so the band's A rows are read from HBM once.
struct TileGroup {
  int32_t tile_start;     // first linear tile index of the group
  int32_t tiles_m;        // m-tiles (common to the group's problems)
  int32_t tiles_n;        // n-tiles summed over the group's problems
  int32_t first, count;   // the group's problems: probs[first .. first + count)
};

struct GemmParams {
  CUtensorMap maps[kMaxMaps];
  Problem probs[kMaxProblems];
  TileGroup groups[kMaxProblems];
  int32_t ngroups;
  int32_t nprob;
  int32_t total_tiles;
  int32_t nmaps;
  int* status;
  uint64_t timeout_ns;
};
// The block travels as a __grid_constant__ kernel parameter (at most 32764 bytes).
static_assert(sizeof(GemmParams) <= 32764, "GEMM parameter block exceeds the kernel parameter limit");

// Host-side builder: collects tensor maps and problems, then launches the persistent
// tcgen05 GEMM kernel once for all of them.
class GemmBatch {
 public:
  GemmBatch();
  ~GemmBatch();
  // Registers a bf16 operand stored row-major [rows, cols] with row stride `ld` elements.
  // mn_major selects the 64x64 box of an MN-major operand; otherwise the 64x128 box of a
  // K-major one.  Returns the map index or -1 (error recorded).
  int add_map(const void* ptr, int64_t rows, int64_t cols, int64_t ld, bool mn_major);
  // Registers n operands as n consecutive maps (no de-duplication), e.g. the t token slabs
  // of an operand whose all-gather is folded into the loads.  Returns the first index or -1.
  int add_maps_consecutive(const void* const* ptrs, int n, int64_t rows, int64_t cols, int64_t ld, bool mn_major);
  // Adds a problem and returns it (nullptr if the batch is full).  Segments are appended
  // with add_seg(); tile counts are filled in by launch().
  // join = true puts the problem in the previous problem's tile group; use it when both
  // read the same A rows (same A tensor, same a_m0, same M).
  Problem* add_problem(int64_t M, int64_t N, bool a_mn, bool b_mn, int epi, bool paired, bool join = false);
  int add_seg(Problem* p, int map_a, int64_t a_k0, int map_b, int map_b2, int64_t b_k0, int64_t K,
              int64_t b_n1 = 0);
  int launch(cudaStream_t stream);
  int error() const { return err_; }
  // True if `maps` more operands and `probs` more problems still fit in this launch.
  bool has_room(int maps, int probs) const {
    return nmaps_ + maps <= kMaxMaps && p_->nprob + probs <= kMaxProblems;
  }
  // Launches what has been collected (if anything) and starts an empty batch.
  int flush(cudaStream_t stream);

 private:
  struct MapKey {
    const void* ptr;
    int64_t rows, cols, ld;
    bool mn;
  };
  GemmParams* p_;
  MapKey keys_[kMaxMaps];
  int nmaps_;
  int err_;
  double flops_;   // algorithmic FLOPs of the collected problems (2 M N K each)
  double bytes_;   // operand bytes read once + output bytes written once
};

// Encodes a 2-D tensor map of a row-major bf16 matrix [rows, cols] (row stride ld elements)
// with a box of box_cols x box_rows elements and 128-byte swizzle.  TTL_OK or an error code.
int encode_map_bf16(CUtensorMap* out, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                    int box_rows);

// The same for an fp32 matrix (row stride ld elements, a multiple of 4).
int encode_map_f32(CUtensorMap* out, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                   int box_rows);

// The same for a 3-D bf16 tensor [d2][d1][d0] (d0 contiguous; ld1, ld2 the strides of dims 1
// and 2 in elements) with a box of box0 x box1 x 1.
int encode_map_bf16_3d(CUtensorMap* out, const void* ptr, int64_t d0, int64_t d1, int64_t d2, int64_t ld1,
                       int64_t ld2, int box0, int box1);

// Forward core of the head-split attention block for t shards (one kernel launch): from Q_i
// [T, qc], K_i and V_i [T, kc] (qc = nql d, kc = nql d / grp) writes the probabilities P_i
// [nql, T, T] (row q up to key min(T, round_up(q + 1, 128)), zeros above the diagonal) and
// O_i [T, qc].  d is 64 or 128.
int attn_fwd_core(int t, int64_t T, int nql, int grp, int d, const void* const* Q, const void* const* K,
                  const void* const* V, void* const* Pout, void* const* Oout, int64_t qc, int64_t kc,
                  cudaStream_t stream);

// Backward cores of the head-split attention block (one launch each), from dO_i [T, qc],
// V_i, K_i [T, kc], Q_i [T, qc], the saved P_i [nql, T, T] and D = rowsum(dO O) [t][nql][T]
// (fp32): attn_bwd_core writes dQ_i = dS K [T, qc] with dS = P (dO V^T - D) / sqrt(d);
// attn_bwd_kv writes dK_i = sum over the group's heads of dS^T Q and dV_i = sum of P^T dO
// ([T, kc]).  Neither writes dS.  d is 64 or 128.
int attn_bwd_core(int t, int64_t T, int nql, int grp, int d, const void* const* dO, const void* const* V,
                  const void* const* K, const void* const* Pin, void* const* dQ, const float* Drow, int64_t qc,
                  int64_t kc, cudaStream_t stream);
int attn_bwd_kv(int t, int64_t T, int nql, int nkvl, int grp, int d, const void* const* Q, const void* const* dO,
                const void* const* V, const void* const* Pin, void* const* dK, void* const* dV, const float* Drow,
                int64_t qc, int64_t kc, cudaStream_t stream);

// Zero-fill helper (used where a contraction is empty).
int fill_zero(void* ptr, size_t bytes, cudaStream_t stream);

// Column sums of a [rows, cols] bf16 matrix (row stride ld) into bf16 [cols].
int column_sum_bf16(const void* x, int64_t rows, int64_t cols, int64_t ld, void* out, cudaStream_t s);

// In-place all-reduce over t shard buffers (validated like ttl_shard_all_reduce).
int shard_all_reduce_internal(int t, int64_t rows, int64_t cols, ttl_bf16* const* bufs, const ttl_bf16* bias,
                              cudaStream_t s);

}  // namespace ttl

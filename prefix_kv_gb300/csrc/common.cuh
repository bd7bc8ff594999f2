// Shared definitions of the CUDA side of the library.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "bca.h"

namespace bca {

constexpr int kHeadDim = 128;
constexpr int kBlockM = 128;   // query rows per work tile
constexpr int kBlockN = 128;   // keys per K/V tile

// Bounded device waits give up after this long and report BCA_ERR_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ void report_status(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Bounds-checked build (-DBCA_BOUNDS_CHECK, libbca_gb300_debug.so): the kernels test
// every computed global index, TMA coordinate and workspace or cache index against
// the extent of its buffer before the access.  A failed test skips the access and
// writes BCA_ERR_BOUNDS to the status word; it never traps.  It stands in for a
// memory checker.  In the release build BCA_IN_BOUNDS is the constant true and
// its condition is not evaluated.
#ifdef BCA_BOUNDS_CHECK
__device__ __forceinline__ bool bounds_ok(bool ok, int32_t* status) {
  if (!ok) report_status(status, BCA_ERR_BOUNDS);
  return ok;
}
#define BCA_IN_BOUNDS(status, cond) (::bca::bounds_ok((cond), (status)))
#else
#define BCA_IN_BOUNDS(status, cond) (true)
#endif

struct PrefillTile {  // one record per (sequence, 128-row query tile)
  int32_t k_hi;       // max visible-key end over the tile's valid rows (0: no work)
  int32_t k_min;      // min visible-key end over the tile's valid rows
  int32_t rows;       // valid query rows in the tile
  int32_t pad;
};

// ---- host-side launchers (defined in the .cu files) ----------------------------------
// Host-side argument checks of the prefill entry points (bca_prefill and its
// variants): BCA_OK when the call may proceed; batch == 0 or total_q == 0 pass
// (nothing to launch).
bca_status check_prefill_args(const void* q, const void* k, const void* v,
                              const int32_t* block_id, const int32_t* cu_seqlens_q,
                              const int32_t* cu_seqlens_k, int32_t batch, int32_t num_heads,
                              int32_t head_dim, int32_t total_q, int32_t total_k,
                              int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                              const void* out, const float* lse);

// A sequence whose offsets leave [0, total_q) / [0, total_k) fails with BCA_ERR_SEQLENS.
cudaError_t launch_schedule_prep(const int32_t* block_id, const int32_t* cu_q, const int32_t* cu_k,
                                 int batch, int total_q, int total_k, int tiles_per_seq,
                                 int32_t* row_end, PrefillTile* tiles, int32_t* status,
                                 cudaStream_t stream);

// Balanced decode tail: at most this many equal key ranges (one per SM), and one
// partial slot per piece, two per range: the unnormalised fp32 O rows of the two
// query tiles as [tile][32 column groups of 4][128 rows][4], then (m, l) per row
// as [tile][128 rows][2] (m in the log2 domain of the scaled scores).
constexpr int kMaxSegRanges = 256;
constexpr int kSegSlotO = 2 * 128 * kHeadDim;               // floats of O in a slot
constexpr int kSegSlotFloats = kSegSlotO + 2 * 128 * 2;
constexpr size_t kSegSlotBytes = static_cast<size_t>(kSegSlotFloats) * sizeof(float);

// Workspace bytes that let a decode launch run its last, partly filled wave as a
// balanced tail on the current device (0: this decode has no such tail).
size_t decode_tail_workspace_bytes(int batch, int num_heads, int max_seqlen_q, int max_prefix);

struct AttnLaunch {
  // tensors
  const void* q;          // [total_q, H, 128]
  const void* k;          // prefill: [total_k, H, 128]; decode: cache layer slab [H][cap][128]
  const void* v;
  const void* k2;         // decode: target K [total_q, H, 128]
  const void* v2;
  void* out;
  float* lse;
  // sizes
  int batch, num_heads, total_q, total_k, tiles_per_seq;
  int64_t capacity;
  float softmax_scale;
  // metadata (device)
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* row_end;
  const PrefillTile* tiles;
  const int32_t* cu_prefix;
  const int32_t* page_table;   // decode over a paged cache: [batch][max_pages], else null
  int max_pages;
  void* cache_k;               // prefill with cache append: layer base [H][capacity][128], else null
  void* cache_v;
  int32_t* status;
  // decode: workspace for the balanced tail (null: the key-split tail instead) and
  // the bound on the prefix lengths it plans with
  void* tail_ws;
  size_t tail_ws_bytes;
  int max_prefix;
};
int launch_attention(const AttnLaunch& a, bool decode, cudaStream_t stream);  // returns bca_status

}  // namespace bca

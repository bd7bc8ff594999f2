// bca_prefill_noalloc: block-causal prefill for callers that cannot allocate.
//
// Some callers cannot allocate device memory at all: a plugin inside an
// inference runtime that owns every byte of the GPU in a pre-planned arena and
// forbids allocations from the libraries it loads, or a latency-critical loop
// that must not take cudaMalloc's implicit device synchronisation.  They also
// cannot size and pass a workspace.  This entry point gives them the same
// computation as bca_prefill, with the schedule scratch (per-row visible-key
// ends and per-tile records) held in a fixed array that lives in this
// library's own device memory for as long as the library is loaded.
//
// Limits: total_q <= kNoAllocMaxRows and batch * ceil(max_seqlen_q / 128) <=
// kNoAllocMaxTiles; larger problems are rejected with BCA_ERR_WORKSPACE before
// anything is launched.  Every GPU that loads the library holds the 2 MiB
// array until the process exits.  All calls share it and it keeps the last
// call's contents; nothing in it needs to start at zero, because the schedule
// kernel of each call rewrites every entry the attention kernel of that call
// reads.  Two calls whose kernels may overlap on the GPU (other streams, or
// other host threads) race on the array: callers must serialise them.
#include "common.cuh"

namespace {

constexpr int kNoAllocMaxRows = 262144;   // query rows            (1 MiB of int32)
constexpr int kNoAllocMaxTiles = 65536;   // (sequence, 128-row tile) records (1 MiB)
constexpr size_t kRowBytes = static_cast<size_t>(kNoAllocMaxRows) * sizeof(int32_t);
constexpr size_t kScratchBytes =
    kRowBytes + static_cast<size_t>(kNoAllocMaxTiles) * sizeof(bca::PrefillTile);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// In host code g_noalloc_scratch names a host-side stand-in, not device memory.
// Its device address on the current device is looked up on every call (the
// lookup allocates nothing and is cheap): a cached address would go stale when
// the device is reset or its primary context is re-created, since the module,
// and with it the array, is then loaded again, possibly elsewhere.
cudaError_t scratch_for_current_device(void** out) {
  return cudaGetSymbolAddress(out, g_noalloc_scratch);
}

}  // namespace

extern "C" bca_status bca_prefill_noalloc(
    const void* q, const void* k, const void* v, const int32_t* block_id,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch, int32_t num_heads,
    int32_t head_dim, int32_t total_q, int32_t total_k, int32_t max_seqlen_q,
    int32_t max_seqlen_k, float softmax_scale, void* out, float* lse, int32_t* status_dev,
    void* stream) {
  using namespace bca;
  const bca_status arg = check_prefill_args(q, k, v, block_id, cu_seqlens_q, cu_seqlens_k, batch,
                                           num_heads, head_dim, total_q, total_k, max_seqlen_q,
                                           max_seqlen_k, softmax_scale, out, lse);
  if (arg != BCA_OK || batch == 0 || total_q == 0) return arg;
  const int tiles_per_seq = (max_seqlen_q + kBlockM - 1) / kBlockM;
  if (total_q > kNoAllocMaxRows ||
      static_cast<int64_t>(batch) * tiles_per_seq > kNoAllocMaxTiles)
    return BCA_ERR_WORKSPACE;  // larger than this entry point's fixed scratch

  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return BCA_ERR_CUDA;
  int32_t* row_end = static_cast<int32_t*>(scratch);
  PrefillTile* tiles =
      reinterpret_cast<PrefillTile*>(static_cast<unsigned char*>(scratch) + kRowBytes);

  auto s = static_cast<cudaStream_t>(stream);
  if (launch_schedule_prep(block_id, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                           tiles_per_seq, row_end, tiles, status_dev, s) != cudaSuccess)
    return BCA_ERR_CUDA;
  AttnLaunch a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.batch = batch;
  a.num_heads = num_heads;
  a.total_q = total_q;
  a.total_k = total_k;
  a.tiles_per_seq = tiles_per_seq;
  a.softmax_scale = softmax_scale;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.row_end = row_end;
  a.tiles = tiles;
  a.status = status_dev;
  return launch_attention(a, /*decode=*/false, s);
}

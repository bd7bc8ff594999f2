// The exported C ABI: argument validation, workspace carving and launches.
#include "kernels.cuh"

#include <cmath>

namespace {

using namespace bca;

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int tiles_for(int max_seqlen_q) { return (max_seqlen_q + kBlockM - 1) / kBlockM; }

struct PrefillWorkspace {
  int32_t* row_end;
  PrefillTile* tiles;
  size_t bytes;
};

PrefillWorkspace carve(void* base, int batch, int total_q, int max_seqlen_q) {
  PrefillWorkspace w{};
  const size_t row_bytes = round_up(static_cast<size_t>(total_q) * sizeof(int32_t));
  const size_t tile_bytes =
      round_up(static_cast<size_t>(batch) * tiles_for(max_seqlen_q) * sizeof(PrefillTile));
  w.bytes = row_bytes + tile_bytes;
  if (base != nullptr) {
    w.row_end = static_cast<int32_t*>(base);
    w.tiles = reinterpret_cast<PrefillTile*>(static_cast<uint8_t*>(base) + row_bytes);
  }
  return w;
}

}  // namespace

namespace bca {

bca_status check_prefill_args(const void* q, const void* k, const void* v,
                              const int32_t* block_id, const int32_t* cu_seqlens_q,
                              const int32_t* cu_seqlens_k, int32_t batch, int32_t num_heads,
                              int32_t head_dim, int32_t total_q, int32_t total_k,
                              int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                              const void* out, const float* lse) {
  if (head_dim != kHeadDim) return BCA_ERR_UNSUPPORTED;
  if (batch < 0 || num_heads <= 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 ||
      max_seqlen_k < 0 || max_seqlen_q > max_seqlen_k)
    return BCA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return BCA_ERR_INVALID_ARG;
  if (batch == 0 || total_q == 0) return BCA_OK;
  if (total_k == 0) return BCA_ERR_SEQLENS;
  if (!q || !k || !v || !block_id || !cu_seqlens_q || !cu_seqlens_k || !out || !lse)
    return BCA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return BCA_ERR_INVALID_ARG;
  if (num_heads > 65535 || batch > 65535 || tiles_for(max_seqlen_q) > 65535)
    return BCA_ERR_UNSUPPORTED;
  return BCA_OK;
}

}  // namespace bca

namespace {

// Decode over one layer's bf16 K and V ([H][capacity][128] each).
bca_status decode_layer(const void* q_tgt, const void* k_layer, const void* v_layer,
                        int64_t capacity, const int32_t* cu_prefix, const void* k_tgt,
                        const void* v_tgt, const int32_t* cu_seqlens_q, int32_t batch,
                        int32_t num_heads, int32_t total_q, int32_t max_seqlen_q,
                        float softmax_scale, void* out, float* lse, int32_t* status_dev,
                        cudaStream_t stream, int32_t max_prefix, void* tail_ws,
                        size_t tail_ws_bytes, const int32_t* page_table = nullptr,
                        int max_pages = 0) {
  AttnLaunch a{};
  a.tail_ws = tail_ws;
  a.tail_ws_bytes = tail_ws_bytes;
  a.max_prefix = max_prefix;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.q = q_tgt;
  // An empty cache (capacity 0) is never read, since every prefix must then be
  // empty; its tensor maps are pointed at q_tgt only to keep them valid.
  a.k = capacity > 0 ? k_layer : q_tgt;
  a.v = capacity > 0 ? v_layer : q_tgt;
  a.k2 = k_tgt;
  a.v2 = v_tgt;
  a.out = out;
  a.lse = lse;
  a.batch = batch;
  a.num_heads = num_heads;
  a.total_q = total_q;
  a.total_k = 0;
  a.tiles_per_seq = tiles_for(max_seqlen_q);
  a.capacity = capacity;
  a.softmax_scale = softmax_scale;
  a.cu_q = cu_seqlens_q;
  a.cu_prefix = cu_prefix;
  a.status = status_dev;
  return launch_attention(a, /*decode=*/true, stream);
}

// Argument checks shared by the decode entry points.
bca_status check_decode_args(const void* q_tgt, const void* cache_k, const void* cache_v,
                             int32_t layer, int32_t num_layers, int64_t capacity,
                             const int32_t* cu_prefix, const void* k_tgt, const void* v_tgt,
                             const int32_t* cu_seqlens_q, int32_t batch, int32_t num_heads,
                             int32_t head_dim, int32_t total_q, int32_t max_seqlen_q,
                             int32_t max_prefix, float softmax_scale, void* out, float* lse) {
  if (head_dim != kHeadDim) return BCA_ERR_UNSUPPORTED;
  if (batch < 0 || num_heads <= 0 || total_q < 0 || max_seqlen_q < 0 || max_prefix < 0 ||
      capacity < 0 || layer < 0 || num_layers <= 0 || layer >= num_layers)
    return BCA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return BCA_ERR_INVALID_ARG;
  if (batch == 0 || total_q == 0) return BCA_OK;
  if (!q_tgt || !k_tgt || !v_tgt || !cu_seqlens_q || !out || !lse || !cu_prefix)
    return BCA_ERR_INVALID_ARG;
  if (capacity > 0 && (!cache_k || !cache_v)) return BCA_ERR_INVALID_ARG;
  if (!aligned16(q_tgt) || !aligned16(k_tgt) || !aligned16(v_tgt) || !aligned16(out) ||
      !aligned16(cache_k) || !aligned16(cache_v))
    return BCA_ERR_INVALID_ARG;
  if (num_heads > 65535 || batch > 65535 || tiles_for(max_seqlen_q) > 65535)
    return BCA_ERR_UNSUPPORTED;
  return BCA_OK;
}

// A decode workspace is optional: null (with any size) runs the key-split tail;
// otherwise it must be 16-byte aligned and hold the balanced tail's slots.
bca_status check_tail_workspace(const void* workspace, size_t workspace_bytes, int32_t batch,
                                int32_t num_heads, int32_t max_seqlen_q, int32_t max_prefix) {
  if (workspace == nullptr) return BCA_OK;
  if (!aligned16(workspace) ||
      workspace_bytes < decode_tail_workspace_bytes(batch, num_heads, max_seqlen_q, max_prefix))
    return BCA_ERR_WORKSPACE;
  return BCA_OK;
}

// The FP8 decodes' workspace: their bf16 layers first (`used` bytes), then, when
// it has room for them, the balanced tail's slots (else the key-split tail runs).
void* tail_after(void* workspace, size_t workspace_bytes, size_t used, int32_t batch,
                 int32_t num_heads, int32_t max_seqlen_q, int32_t max_prefix, size_t* tail_bytes) {
  const size_t need = decode_tail_workspace_bytes(batch, num_heads, max_seqlen_q, max_prefix);
  *tail_bytes = 0;
  if (need == 0 || workspace == nullptr || !aligned16(workspace) || workspace_bytes < used ||
      workspace_bytes - used < need)
    return nullptr;
  *tail_bytes = workspace_bytes - used;
  return static_cast<uint8_t*>(workspace) + used;
}

// Bytes of one layer of a bf16 cache, rounded up to 256.
size_t bf16_layer_bytes(int32_t num_heads, int64_t capacity) {
  const size_t b = static_cast<size_t>(num_heads) * static_cast<size_t>(capacity) * kHeadDim * 2;
  return (b + 255) & ~static_cast<size_t>(255);
}

// Shared by the contiguous and paged FP8 appends (page_table null: contiguous).
bca_status append_fp8_impl(const void* k, const void* v, const int32_t* cu_seqlens_k,
                           const int32_t* cu_prefix, const int32_t* page_table, int max_pages,
                           int32_t batch, int32_t num_heads, int32_t head_dim, int32_t total_k,
                           int32_t mode, void* cache_k, void* cache_v, float* scale_k,
                           float* scale_v, int32_t layer, int32_t num_layers, int64_t capacity,
                           int32_t* status_dev, void* stream) {
  if (head_dim != kHeadDim) return BCA_ERR_UNSUPPORTED;
  if (mode != BCA_FP8_V && mode != BCA_FP8_KV) return BCA_ERR_INVALID_ARG;
  if (batch < 0 || num_heads <= 0 || total_k < 0 || capacity < 0 || layer < 0 ||
      num_layers <= 0 || layer >= num_layers)
    return BCA_ERR_INVALID_ARG;
  if (batch == 0) return BCA_OK;
  if (!k || !v || !cu_seqlens_k || !cu_prefix) return BCA_ERR_INVALID_ARG;
  const bool quant_k = mode == BCA_FP8_KV;
  if (capacity > 0 && (!cache_k || !cache_v || !scale_v || (quant_k && !scale_k)))
    return BCA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(cache_k) || !aligned16(cache_v) ||
      (reinterpret_cast<uintptr_t>(scale_v) & 3u) || (reinterpret_cast<uintptr_t>(scale_k) & 3u))
    return BCA_ERR_INVALID_ARG;
  const size_t rows = static_cast<size_t>(num_heads) * capacity;   // per layer
  if (rows > 0x7fffffffu) return BCA_ERR_UNSUPPORTED;   // (head, token) rows are 32-bit indices
  const size_t k_bytes = quant_k ? 1 : 2;
  cudaError_t e = launch_cache_append_fp8(
      k, v, cu_seqlens_k, cu_prefix, batch, num_heads, total_k, quant_k,
      static_cast<uint8_t*>(cache_k) + layer * rows * kHeadDim * k_bytes,
      static_cast<uint8_t*>(cache_v) + layer * rows * kHeadDim,
      quant_k ? scale_k + layer * rows : nullptr, scale_v + layer * rows, capacity, page_table,
      max_pages, status_dev, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* bca_status_string(bca_status s) {
  switch (s) {
    case BCA_OK: return "ok";
    case BCA_ERR_INVALID_ARG: return "invalid argument";
    case BCA_ERR_UNSUPPORTED: return "unsupported (head_dim != 128 or too many image runs)";
    case BCA_ERR_BLOCK_ID: return "invalid block ids (id < -1 or an id split over several runs)";
    case BCA_ERR_WORKSPACE: return "workspace missing or too small";
    case BCA_ERR_CAPACITY: return "prefix cache capacity exceeded";
    case BCA_ERR_CUDA: return "CUDA runtime error";
    case BCA_ERR_TIMEOUT: return "device wait timed out";
    case BCA_ERR_SEQLENS: return "invalid cu_seqlens / lengths";
    case BCA_ERR_BOUNDS: return "index outside its buffer (bounds-checked build)";
    default: return "unknown status";
  }
}

int32_t bca_version(void) { return 100; }

bca_status bca_read_device_status(const int32_t* status_dev, void* stream) {
  if (status_dev == nullptr) return BCA_ERR_INVALID_ARG;
  int32_t h = 0;
  auto s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&h, status_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return BCA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return BCA_ERR_CUDA;
  return h;
}

size_t bca_prefill_workspace_bytes(int32_t batch, int32_t total_q, int32_t max_seqlen_q) {
  if (batch < 0 || total_q < 0 || max_seqlen_q < 0) return 0;
  return carve(nullptr, batch, total_q, max_seqlen_q).bytes;
}

bca_status bca_schedule_prep(const int32_t* block_id, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q,
                             int32_t total_k, int32_t max_seqlen_q, int32_t* row_end,
                             int32_t* tiles, int32_t* status_dev, void* stream) {
  if (batch < 0 || max_seqlen_q < 0 || total_q < 0 || total_k < 0) return BCA_ERR_INVALID_ARG;
  if (batch == 0 || max_seqlen_q == 0) return BCA_OK;
  if (!block_id || !cu_seqlens_q || !cu_seqlens_k || !row_end || !tiles)
    return BCA_ERR_INVALID_ARG;
  if (batch > 65535) return BCA_ERR_UNSUPPORTED;
  cudaError_t e = launch_schedule_prep(block_id, cu_seqlens_q, cu_seqlens_k, batch, total_q,
                                       total_k, tiles_for(max_seqlen_q), row_end,
                                       reinterpret_cast<PrefillTile*>(tiles), status_dev,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}

}  // extern "C"

namespace {

// bca_prefill, with the prefix cache append fused in when cache_k is not null.
bca_status prefill_impl(const void* q, const void* k, const void* v, const int32_t* block_id,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                       int32_t num_heads, int32_t head_dim, int32_t total_q, int32_t total_k,
                       int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                       void* out, float* lse, void* workspace, size_t workspace_bytes,
                       const int32_t* cu_prefix, void* cache_k, void* cache_v, int64_t capacity,
                       const int32_t* page_table, int32_t max_pages, int32_t* status_dev,
                       void* stream) {
  const bca_status arg = check_prefill_args(q, k, v, block_id, cu_seqlens_q, cu_seqlens_k, batch,
                                           num_heads, head_dim, total_q, total_k, max_seqlen_q,
                                           max_seqlen_k, softmax_scale, out, lse);
  if (arg != BCA_OK || batch == 0 || total_q == 0) return arg;
  PrefillWorkspace w = carve(workspace, batch, total_q, max_seqlen_q);
  if (workspace == nullptr || workspace_bytes < w.bytes || !aligned16(workspace))
    return BCA_ERR_WORKSPACE;

  auto s = static_cast<cudaStream_t>(stream);
  const int tps = tiles_for(max_seqlen_q);
  if (launch_schedule_prep(block_id, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, tps,
                           w.row_end, w.tiles, status_dev, s) != cudaSuccess)
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
  a.tiles_per_seq = tps;
  a.softmax_scale = softmax_scale;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.row_end = w.row_end;
  a.tiles = w.tiles;
  a.status = status_dev;
  a.cu_prefix = cu_prefix;
  a.cache_k = cache_k;
  a.cache_v = cache_v;
  a.capacity = capacity;
  a.page_table = page_table;
  a.max_pages = max_pages;
  return launch_attention(a, /*decode=*/false, s);
}

}  // namespace

extern "C" {

bca_status bca_prefill(const void* q, const void* k, const void* v, const int32_t* block_id,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                       int32_t num_heads, int32_t head_dim, int32_t total_q, int32_t total_k,
                       int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                       void* out, float* lse, void* workspace, size_t workspace_bytes,
                       int32_t* status_dev, void* stream) {
  return prefill_impl(q, k, v, block_id, cu_seqlens_q, cu_seqlens_k, batch, num_heads, head_dim,
                      total_q, total_k, max_seqlen_q, max_seqlen_k, softmax_scale, out, lse,
                      workspace, workspace_bytes, nullptr, nullptr, nullptr, 0, nullptr, 0,
                      status_dev, stream);
}

bca_status bca_prefill_append(const void* q, const void* k, const void* v,
                              const int32_t* block_id, const int32_t* cu_seqlens_q,
                              const int32_t* cu_seqlens_k, int32_t batch, int32_t num_heads,
                              int32_t head_dim, int32_t total_q, int32_t total_k,
                              int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                              void* out, float* lse, void* workspace, size_t workspace_bytes,
                              const int32_t* cu_prefix, void* cache_k, void* cache_v,
                              int32_t layer, int32_t num_layers, int64_t capacity,
                              int32_t* status_dev, void* stream) {
  if (head_dim != kHeadDim) return BCA_ERR_UNSUPPORTED;
  if (capacity < 0 || layer < 0 || num_layers <= 0 || layer >= num_layers || num_heads <= 0)
    return BCA_ERR_INVALID_ARG;
  if (!cu_prefix || !cache_k || !cache_v || !aligned16(cache_k) || !aligned16(cache_v))
    return BCA_ERR_INVALID_ARG;
  const size_t layer_elems = static_cast<size_t>(num_heads) * capacity * kHeadDim;
  return prefill_impl(q, k, v, block_id, cu_seqlens_q, cu_seqlens_k, batch, num_heads, head_dim,
                      total_q, total_k, max_seqlen_q, max_seqlen_k, softmax_scale, out, lse,
                      workspace, workspace_bytes, cu_prefix,
                      static_cast<__nv_bfloat16*>(cache_k) + layer * layer_elems,
                      static_cast<__nv_bfloat16*>(cache_v) + layer * layer_elems, capacity,
                      nullptr, 0, status_dev, stream);
}

bca_status bca_prefill_append_paged(const void* q, const void* k, const void* v,
                                    const int32_t* block_id, const int32_t* cu_seqlens_q,
                                    const int32_t* cu_seqlens_k, int32_t batch, int32_t num_heads,
                                    int32_t head_dim, int32_t total_q, int32_t total_k,
                                    int32_t max_seqlen_q, int32_t max_seqlen_k,
                                    float softmax_scale, void* out, float* lse, void* workspace,
                                    size_t workspace_bytes, const int32_t* cu_prefix,
                                    const int32_t* page_table, int32_t max_pages, void* cache_k,
                                    void* cache_v, int32_t layer, int32_t num_layers,
                                    int32_t num_pages, int32_t* status_dev, void* stream) {
  if (head_dim != kHeadDim) return BCA_ERR_UNSUPPORTED;
  if (num_pages <= 0 || num_pages > (1 << 24) || max_pages < 0 || layer < 0 ||
      num_layers <= 0 || layer >= num_layers || num_heads <= 0)
    return BCA_ERR_INVALID_ARG;
  if (!cu_prefix || !page_table || !cache_k || !cache_v || !aligned16(cache_k) ||
      !aligned16(cache_v))
    return BCA_ERR_INVALID_ARG;
  const int64_t capacity = static_cast<int64_t>(num_pages) * kBlockN;
  const size_t layer_elems = static_cast<size_t>(num_heads) * capacity * kHeadDim;
  return prefill_impl(q, k, v, block_id, cu_seqlens_q, cu_seqlens_k, batch, num_heads, head_dim,
                      total_q, total_k, max_seqlen_q, max_seqlen_k, softmax_scale, out, lse,
                      workspace, workspace_bytes, cu_prefix,
                      static_cast<__nv_bfloat16*>(cache_k) + layer * layer_elems,
                      static_cast<__nv_bfloat16*>(cache_v) + layer * layer_elems, capacity,
                      page_table, max_pages, status_dev, stream);
}

size_t bca_prefix_decode_workspace_bytes(int32_t batch, int32_t num_heads, int32_t head_dim,
                                         int32_t max_seqlen_q, int32_t max_prefix) {
  if (head_dim != kHeadDim) return 0;
  return decode_tail_workspace_bytes(batch, num_heads, max_seqlen_q, max_prefix);
}

bca_status bca_prefix_decode(const void* q_tgt, const void* cache_k, const void* cache_v,
                             int32_t layer, int32_t num_layers, int64_t capacity,
                             const int32_t* cu_prefix, const void* k_tgt, const void* v_tgt,
                             const int32_t* cu_seqlens_q, int32_t batch, int32_t num_heads,
                             int32_t head_dim, int32_t total_q, int32_t max_seqlen_q,
                             int32_t max_prefix, float softmax_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, int32_t* status_dev,
                             void* stream) {
  bca_status st = check_decode_args(q_tgt, cache_k, cache_v, layer, num_layers, capacity,
                                    cu_prefix, k_tgt, v_tgt, cu_seqlens_q, batch, num_heads,
                                    head_dim, total_q, max_seqlen_q, max_prefix, softmax_scale,
                                    out, lse);
  if (st != BCA_OK || batch == 0 || total_q == 0) return st;
  st = check_tail_workspace(workspace, workspace_bytes, batch, num_heads, max_seqlen_q, max_prefix);
  if (st != BCA_OK) return st;
  const size_t layer_elems = static_cast<size_t>(num_heads) * capacity * kHeadDim;
  return decode_layer(q_tgt, static_cast<const __nv_bfloat16*>(cache_k) + layer * layer_elems,
                      static_cast<const __nv_bfloat16*>(cache_v) + layer * layer_elems, capacity,
                      cu_prefix, k_tgt, v_tgt, cu_seqlens_q, batch, num_heads, total_q,
                      max_seqlen_q, softmax_scale, out, lse, status_dev,
                      static_cast<cudaStream_t>(stream), max_prefix, workspace, workspace_bytes);
}

bca_status bca_prefix_decode_paged(const void* q_tgt, const void* cache_k, const void* cache_v,
                                   int32_t layer, int32_t num_layers, int32_t num_pages,
                                   const int32_t* cu_prefix, const int32_t* page_table,
                                   int32_t max_pages, const void* k_tgt, const void* v_tgt,
                                   const int32_t* cu_seqlens_q, int32_t batch, int32_t num_heads,
                                   int32_t head_dim, int32_t total_q, int32_t max_seqlen_q,
                                   int32_t max_prefix, float softmax_scale, void* out, float* lse,
                                   void* workspace, size_t workspace_bytes, int32_t* status_dev,
                                   void* stream) {
  if (num_pages <= 0 || num_pages > (1 << 24) || max_pages < 0) return BCA_ERR_INVALID_ARG;
  const int64_t capacity = static_cast<int64_t>(num_pages) * kBlockN;
  bca_status st = check_decode_args(q_tgt, cache_k, cache_v, layer, num_layers, capacity,
                                    cu_prefix, k_tgt, v_tgt, cu_seqlens_q, batch, num_heads,
                                    head_dim, total_q, max_seqlen_q, max_prefix, softmax_scale,
                                    out, lse);
  if (st != BCA_OK || batch == 0 || total_q == 0) return st;
  if (!page_table) return BCA_ERR_INVALID_ARG;
  st = check_tail_workspace(workspace, workspace_bytes, batch, num_heads, max_seqlen_q, max_prefix);
  if (st != BCA_OK) return st;
  const size_t layer_elems = static_cast<size_t>(num_heads) * capacity * kHeadDim;
  return decode_layer(q_tgt, static_cast<const __nv_bfloat16*>(cache_k) + layer * layer_elems,
                      static_cast<const __nv_bfloat16*>(cache_v) + layer * layer_elems, capacity,
                      cu_prefix, k_tgt, v_tgt, cu_seqlens_q, batch, num_heads, total_q,
                      max_seqlen_q, softmax_scale, out, lse, status_dev,
                      static_cast<cudaStream_t>(stream), max_prefix, workspace, workspace_bytes,
                      page_table, max_pages);
}

size_t bca_prefix_decode_fp8_workspace_bytes(int32_t mode, int32_t num_heads, int32_t head_dim,
                                             int64_t capacity) {
  if ((mode != BCA_FP8_V && mode != BCA_FP8_KV) || head_dim != kHeadDim || num_heads <= 0 ||
      capacity < 0)
    return 0;
  return (mode == BCA_FP8_KV ? 2 : 1) * bf16_layer_bytes(num_heads, capacity);
}

bca_status bca_prefix_cache_dequant_fp8(const void* codes, const float* scales,
                                        const int32_t* cu_prefix, int32_t batch,
                                        int32_t num_heads, int32_t head_dim, int32_t layer,
                                        int32_t num_layers, int64_t capacity, void* out,
                                        int32_t* status_dev, void* stream) {
  if (head_dim != kHeadDim) return BCA_ERR_UNSUPPORTED;
  if (batch < 0 || num_heads <= 0 || capacity < 0 || layer < 0 || num_layers <= 0 ||
      layer >= num_layers)
    return BCA_ERR_INVALID_ARG;
  if (batch == 0 || capacity == 0) return BCA_OK;
  // (heads are a grid dimension; 16 chunks per row index a head's rows in 32 bits)
  if (num_heads > 65535 || capacity >= (int64_t{1} << 28)) return BCA_ERR_UNSUPPORTED;
  if (!codes || !scales || !cu_prefix || !out) return BCA_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(out) || (reinterpret_cast<uintptr_t>(scales) & 3u))
    return BCA_ERR_INVALID_ARG;
  const size_t rows = static_cast<size_t>(num_heads) * capacity;   // (head, token) rows per layer
  const cudaError_t e = launch_cache_dequant_fp8(
      static_cast<const uint8_t*>(codes) + layer * rows * kHeadDim, scales + layer * rows,
      cu_prefix, batch, num_heads, capacity, out, status_dev, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}

bca_status bca_prefix_decode_fp8(const void* q_tgt, const void* cache_k, const void* cache_v,
                                 int32_t mode, const float* scale_k, const float* scale_v,
                                 int32_t layer, int32_t num_layers, int64_t capacity,
                                 const int32_t* cu_prefix, const void* k_tgt, const void* v_tgt,
                                 const int32_t* cu_seqlens_q, int32_t batch, int32_t num_heads,
                                 int32_t head_dim, int32_t total_q, int32_t max_seqlen_q,
                                 int32_t max_prefix, float softmax_scale, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, int32_t* status_dev,
                                 void* stream) {
  if (mode != BCA_FP8_V && mode != BCA_FP8_KV) return BCA_ERR_INVALID_ARG;
  bca_status st = check_decode_args(q_tgt, cache_k, cache_v, layer, num_layers, capacity,
                                    cu_prefix, k_tgt, v_tgt, cu_seqlens_q, batch, num_heads,
                                    head_dim, total_q, max_seqlen_q, max_prefix, softmax_scale,
                                    out, lse);
  if (st != BCA_OK || batch == 0 || total_q == 0) return st;
  const bool k8 = mode == BCA_FP8_KV;
  if (capacity > 0 && (!scale_v || (k8 && !scale_k))) return BCA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scale_v) & 3u) || (reinterpret_cast<uintptr_t>(scale_k) & 3u))
    return BCA_ERR_INVALID_ARG;
  const size_t need = bca_prefix_decode_fp8_workspace_bytes(mode, num_heads, head_dim, capacity);
  if (capacity > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
    return BCA_ERR_WORKSPACE;
  auto s = static_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(num_heads) * capacity;
  const void* k_layer = nullptr;
  const void* v_layer = nullptr;
  if (capacity > 0) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* v_exp = ws;
    st = bca_prefix_cache_dequant_fp8(cache_v, scale_v, cu_prefix, batch, num_heads, head_dim,
                                      layer, num_layers, capacity, v_exp, status_dev, stream);
    if (st != BCA_OK) return st;
    v_layer = v_exp;
    if (k8) {
      void* k_exp = ws + bf16_layer_bytes(num_heads, capacity);
      st = bca_prefix_cache_dequant_fp8(cache_k, scale_k, cu_prefix, batch, num_heads, head_dim,
                                        layer, num_layers, capacity, k_exp, status_dev, stream);
      if (st != BCA_OK) return st;
      k_layer = k_exp;
    } else {
      k_layer = static_cast<const __nv_bfloat16*>(cache_k) + layer * rows * kHeadDim;
    }
  }
  size_t tail_bytes = 0;
  void* tail = tail_after(workspace, workspace_bytes, capacity > 0 ? need : 0, batch, num_heads,
                          max_seqlen_q, max_prefix, &tail_bytes);
  return decode_layer(q_tgt, k_layer, v_layer, capacity, cu_prefix, k_tgt, v_tgt, cu_seqlens_q,
                      batch, num_heads, total_q, max_seqlen_q, softmax_scale, out, lse,
                      status_dev, s, max_prefix, tail, tail_bytes);
}

bca_status bca_prefix_cache_append(const void* k, const void* v, const int32_t* cu_seqlens_k,
                                   const int32_t* cu_prefix, int32_t batch, int32_t num_heads,
                                   int32_t head_dim, int32_t total_k, void* cache_k,
                                   void* cache_v, int32_t layer, int32_t num_layers,
                                   int64_t capacity, int32_t* status_dev, void* stream) {
  if (head_dim != kHeadDim) return BCA_ERR_UNSUPPORTED;
  if (batch < 0 || num_heads <= 0 || total_k < 0 || capacity < 0 || layer < 0 ||
      num_layers <= 0 || layer >= num_layers)
    return BCA_ERR_INVALID_ARG;
  if (batch == 0) return BCA_OK;
  if (!k || !v || !cu_seqlens_k || !cu_prefix) return BCA_ERR_INVALID_ARG;
  if (capacity > 0 && (!cache_k || !cache_v)) return BCA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(cache_k) || !aligned16(cache_v))
    return BCA_ERR_INVALID_ARG;
  const size_t layer_elems = static_cast<size_t>(num_heads) * capacity * kHeadDim;
  cudaError_t e = launch_cache_append(
      k, v, cu_seqlens_k, cu_prefix, batch, num_heads, total_k,
      static_cast<__nv_bfloat16*>(cache_k) + layer * layer_elems,
      static_cast<__nv_bfloat16*>(cache_v) + layer * layer_elems, capacity, nullptr, 0,
      status_dev, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}

bca_status bca_prefix_cache_append_paged(const void* k, const void* v,
                                         const int32_t* cu_seqlens_k, const int32_t* cu_prefix,
                                         const int32_t* page_table, int32_t max_pages,
                                         int32_t batch, int32_t num_heads, int32_t head_dim,
                                         int32_t total_k, void* cache_k, void* cache_v,
                                         int32_t layer, int32_t num_layers, int32_t num_pages,
                                         int32_t* status_dev, void* stream) {
  if (head_dim != kHeadDim) return BCA_ERR_UNSUPPORTED;
  if (batch < 0 || num_heads <= 0 || total_k < 0 || num_pages <= 0 || max_pages < 0 ||
      layer < 0 || num_layers <= 0 || layer >= num_layers || num_pages > (1 << 24))
    return BCA_ERR_INVALID_ARG;
  if (batch == 0) return BCA_OK;
  if (!k || !v || !cu_seqlens_k || !cu_prefix || !page_table || !cache_k || !cache_v)
    return BCA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(cache_k) || !aligned16(cache_v))
    return BCA_ERR_INVALID_ARG;
  const int64_t capacity = static_cast<int64_t>(num_pages) * kBlockN;
  const size_t layer_elems = static_cast<size_t>(num_heads) * capacity * kHeadDim;
  cudaError_t e = launch_cache_append(
      k, v, cu_seqlens_k, cu_prefix, batch, num_heads, total_k,
      static_cast<__nv_bfloat16*>(cache_k) + layer * layer_elems,
      static_cast<__nv_bfloat16*>(cache_v) + layer * layer_elems, capacity, page_table,
      max_pages, status_dev, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}

bca_status bca_pool_copy_rows(void* cache_k, void* cache_v, int32_t layer, int32_t num_layers,
                              int32_t num_heads, int32_t num_pages, int32_t src_page,
                              int32_t dst_page, int32_t n_rows, void* stream) {
  if (!cache_k || !cache_v || layer < 0 || num_layers <= 0 || layer >= num_layers ||
      num_heads <= 0 || num_pages <= 0 || num_pages > (1 << 24) || src_page < 0 ||
      src_page >= num_pages || dst_page < 0 || dst_page >= num_pages || n_rows < 0 ||
      n_rows > kBlockN)
    return BCA_ERR_INVALID_ARG;
  if (!aligned16(cache_k) || !aligned16(cache_v)) return BCA_ERR_INVALID_ARG;
  if (n_rows == 0 || src_page == dst_page) return BCA_OK;
  const int64_t capacity = static_cast<int64_t>(num_pages) * kBlockN;
  const size_t layer_elems = static_cast<size_t>(num_heads) * capacity * kHeadDim;
  const cudaError_t e = launch_cache_copy_rows(
      static_cast<__nv_bfloat16*>(cache_k) + layer * layer_elems,
      static_cast<__nv_bfloat16*>(cache_v) + layer * layer_elems, num_heads, capacity, src_page,
      dst_page, n_rows, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}

bca_status bca_prefix_cache_append_fp8(const void* k, const void* v, const int32_t* cu_seqlens_k,
                                       const int32_t* cu_prefix, int32_t batch, int32_t num_heads,
                                       int32_t head_dim, int32_t total_k, int32_t mode,
                                       void* cache_k, void* cache_v, float* scale_k,
                                       float* scale_v, int32_t layer, int32_t num_layers,
                                       int64_t capacity, int32_t* status_dev, void* stream) {
  return append_fp8_impl(k, v, cu_seqlens_k, cu_prefix, nullptr, 0, batch, num_heads, head_dim,
                         total_k, mode, cache_k, cache_v, scale_k, scale_v, layer, num_layers,
                         capacity, status_dev, stream);
}

bca_status bca_prefix_cache_append_fp8_paged(
    const void* k, const void* v, const int32_t* cu_seqlens_k, const int32_t* cu_prefix,
    const int32_t* page_table, int32_t max_pages, int32_t batch, int32_t num_heads,
    int32_t head_dim, int32_t total_k, int32_t mode, void* cache_k, void* cache_v,
    float* scale_k, float* scale_v, int32_t layer, int32_t num_layers, int32_t num_pages,
    int32_t* status_dev, void* stream) {
  if (num_pages <= 0 || num_pages > (1 << 24) || max_pages < 0 || !page_table)
    return BCA_ERR_INVALID_ARG;
  return append_fp8_impl(k, v, cu_seqlens_k, cu_prefix, page_table, max_pages, batch, num_heads,
                         head_dim, total_k, mode, cache_k, cache_v, scale_k, scale_v, layer,
                         num_layers, static_cast<int64_t>(num_pages) * kBlockN, status_dev,
                         stream);
}

size_t bca_prefix_decode_fp8_paged_workspace_bytes(int32_t num_heads, int32_t head_dim,
                                                   int64_t prefix_rows) {
  if (head_dim != kHeadDim || num_heads <= 0 || prefix_rows < 0) return 0;
  return 2 * bf16_layer_bytes(num_heads, prefix_rows);
}

bca_status bca_prefix_decode_fp8_paged(
    const void* q_tgt, const void* cache_k, const void* cache_v, int32_t mode,
    const float* scale_k, const float* scale_v, int32_t layer, int32_t num_layers,
    int32_t num_pages, const int32_t* cu_prefix, const int32_t* page_table, int32_t max_pages,
    int64_t prefix_rows, const void* k_tgt, const void* v_tgt, const int32_t* cu_seqlens_q,
    int32_t batch, int32_t num_heads, int32_t head_dim, int32_t total_q, int32_t max_seqlen_q,
    int32_t max_prefix, float softmax_scale, void* out, float* lse, void* workspace,
    size_t workspace_bytes, int32_t* status_dev, void* stream) {
  if (mode != BCA_FP8_V && mode != BCA_FP8_KV) return BCA_ERR_INVALID_ARG;
  if (num_pages <= 0 || num_pages > (1 << 24) || max_pages < 0 || prefix_rows < 0)
    return BCA_ERR_INVALID_ARG;
  if (prefix_rows >= (int64_t{1} << 28)) return BCA_ERR_UNSUPPORTED;
  const int64_t capacity = static_cast<int64_t>(num_pages) * kBlockN;
  bca_status st = check_decode_args(q_tgt, cache_k, cache_v, layer, num_layers, capacity,
                                    cu_prefix, k_tgt, v_tgt, cu_seqlens_q, batch, num_heads,
                                    head_dim, total_q, max_seqlen_q, max_prefix, softmax_scale,
                                    out, lse);
  if (st != BCA_OK || batch == 0 || total_q == 0) return st;
  const bool k8 = mode == BCA_FP8_KV;
  if (!page_table || !scale_v || (k8 && !scale_k)) return BCA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scale_v) & 3u) || (reinterpret_cast<uintptr_t>(scale_k) & 3u))
    return BCA_ERR_INVALID_ARG;
  const size_t need = bca_prefix_decode_fp8_paged_workspace_bytes(num_heads, head_dim,
                                                                   prefix_rows);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return BCA_ERR_WORKSPACE;
  auto s = static_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(num_heads) * capacity;   // (head, token) rows per layer
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* k_out = ws;
  void* v_out = ws + bf16_layer_bytes(num_heads, prefix_rows);
  const void* k_src = static_cast<const uint8_t*>(cache_k) + layer * rows * kHeadDim * (k8 ? 1 : 2);
  const void* v_src = static_cast<const uint8_t*>(cache_v) + layer * rows * kHeadDim;
  if (launch_cache_gather(k8, k_src, k8 ? scale_k + layer * rows : nullptr, cu_prefix,
                          page_table, max_pages, batch, num_heads, capacity, k_out, prefix_rows,
                          status_dev, s) != cudaSuccess ||
      launch_cache_gather(true, v_src, scale_v + layer * rows, cu_prefix, page_table, max_pages,
                          batch, num_heads, capacity, v_out, prefix_rows, status_dev, s) !=
          cudaSuccess)
    return BCA_ERR_CUDA;
  size_t tail_bytes = 0;
  void* tail = tail_after(workspace, workspace_bytes, need, batch, num_heads, max_seqlen_q,
                          max_prefix, &tail_bytes);
  return decode_layer(q_tgt, k_out, v_out, prefix_rows, cu_prefix, k_tgt, v_tgt, cu_seqlens_q,
                      batch, num_heads, total_q, max_seqlen_q, softmax_scale, out, lse,
                      status_dev, s, max_prefix, tail, tail_bytes);
}

bca_status bca_rope_positions(const int32_t* block_id, const int32_t* cu_seqlens, int32_t batch,
                              int32_t total, const int32_t* grid_w, int32_t n_ids,
                              int32_t* pos3, int32_t* status_dev, void* stream) {
  if (batch < 0 || total < 0 || n_ids < 0) return BCA_ERR_INVALID_ARG;
  if (batch == 0 || total == 0) return BCA_OK;
  if (!block_id || !cu_seqlens || !pos3 || (n_ids > 0 && !grid_w)) return BCA_ERR_INVALID_ARG;
  if (n_ids > 4096 || batch > 65535) return BCA_ERR_UNSUPPORTED;
  const cudaError_t e = launch_rope_positions(block_id, cu_seqlens, batch, total, grid_w, n_ids, pos3,
                                              status_dev, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}

bca_status bca_rope_table(const int32_t* pos3, int32_t total, float* table, void* stream) {
  if (total < 0) return BCA_ERR_INVALID_ARG;
  if (total == 0) return BCA_OK;
  if (!pos3 || !table || (reinterpret_cast<uintptr_t>(table) & 15u)) return BCA_ERR_INVALID_ARG;
  const cudaError_t e = launch_rope_table(pos3, total, table, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}

bca_status bca_qk_norm_rope_append(const void* q, const void* k, const void* v,
                                   const float* gamma_q, const float* gamma_k,
                                   const float* rope_table, const int32_t* cu_seqlens,
                                   const int32_t* cu_prefix, int32_t batch, int32_t num_heads,
                                   int32_t head_dim, int32_t total, float eps, void* q_out,
                                   void* k_out, void* cache_k, void* cache_v, int32_t layer,
                                   int32_t num_layers, int64_t capacity, int32_t* status_dev,
                                   void* stream) {
  if (head_dim != kHeadDim) return BCA_ERR_UNSUPPORTED;
  if (batch < 0 || num_heads <= 0 || total < 0 || !(eps >= 0.f) || !std::isfinite(eps))
    return BCA_ERR_INVALID_ARG;
  if (batch == 0 || total == 0) return BCA_OK;
  if (!q || !k || !rope_table || !cu_seqlens || !q_out || !k_out) return BCA_ERR_INVALID_ARG;
  const bool append = cu_prefix != nullptr;
  if (append && (!v || layer < 0 || num_layers <= 0 || layer >= num_layers || capacity < 0 ||
                 (capacity > 0 && (!cache_k || !cache_v))))
    return BCA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_out) || !aligned16(k_out) ||
      !aligned16(cache_k) || !aligned16(cache_v) || !aligned16(rope_table) ||
      !aligned16(gamma_q) || !aligned16(gamma_k))
    return BCA_ERR_INVALID_ARG;
  const size_t layer_elems = static_cast<size_t>(num_heads) * capacity * kHeadDim;
  void* ck = append && capacity > 0 ? static_cast<__nv_bfloat16*>(cache_k) + layer * layer_elems
                                    : nullptr;
  void* cv = append && capacity > 0 ? static_cast<__nv_bfloat16*>(cache_v) + layer * layer_elems
                                    : nullptr;
  const cudaError_t e = launch_qk_norm_rope(q, k, v, gamma_q, gamma_k, rope_table, cu_seqlens,
                                            cu_prefix, batch, num_heads, total, eps, q_out, k_out,
                                            ck, cv, capacity, status_dev,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}

}  // extern "C"

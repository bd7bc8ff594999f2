// bca_prefill_piecewise: the block-causal prefill as one exact attention call
// per segment, the path the default diffusers processor takes (Qwen-Image 2.1
// deployment notes, piecewise-attention paragraph; flozi.net "Two exact
// attention paths": one call for every text or image segment of the prefix
// and one for the target; a text segment is causal over itself, an image
// segment sees every earlier key and its whole block).
//
// It is a baseline for the single-launch bca_prefill, built on the same
// kernels: segment [a, e) of a sequence starting at s becomes its own problem
// with queries [a, e) over keys [s, e), the bottom-right alignment of the
// attention kernel putting query i at key position (e - s) - (e - a) + i.
// Its block ids are the sequence's ids [s, e): an image segment's queries
// share their id with the segment's keys and see them all; every earlier key
// is before them and visible by causality; a text segment's queries are
// causal.  Pieces run in stream order, so one scratch area serves them all.
// Each piece's LSE rows are scattered into the [H][total] output by one 2-D
// copy.  The segment table comes from host copies of block_id / cu_seqlens.
#include <cmath>
#include <vector>

#include "common.cuh"

namespace {

using namespace bca;

struct Piece {
  int a, e, s;   // query rows [a, e) of a sequence whose keys start at s (packed indices)
};

std::vector<Piece> pieces_of(const int32_t* bid, const int32_t* cu, int batch) {
  std::vector<Piece> out;
  for (int b = 0; b < batch; ++b) {
    int a = cu[b];
    while (a < cu[b + 1]) {
      int e = a + 1;
      while (e < cu[b + 1] && bid[e] == bid[a]) ++e;
      out.push_back({a, e, cu[b]});
      a = e;
    }
  }
  return out;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Scratch {
  size_t cu_off, row_off, tile_off, lse_off, bytes;
};

Scratch layout(size_t n_pieces, int max_q, int num_heads) {
  Scratch w{};
  w.cu_off = 0;
  w.row_off = round256(n_pieces * 4 * sizeof(int32_t));
  w.tile_off = w.row_off + round256(static_cast<size_t>(max_q) * sizeof(int32_t));
  const size_t tiles = (static_cast<size_t>(max_q) + kBlockM - 1) / kBlockM;
  w.lse_off = w.tile_off + round256(tiles * sizeof(PrefillTile));
  w.bytes = w.lse_off + round256(static_cast<size_t>(num_heads) * max_q * sizeof(float));
  return w;
}

bool valid_cu(const int32_t* cu, int batch) {
  if (cu[0] != 0) return false;
  for (int b = 0; b < batch; ++b)
    if (cu[b + 1] < cu[b]) return false;
  return true;
}

}  // namespace

extern "C" {

size_t bca_prefill_piecewise_workspace_bytes(const int32_t* block_id_host,
                                             const int32_t* cu_seqlens_host, int32_t batch,
                                             int32_t num_heads) {
  if (!block_id_host || !cu_seqlens_host || batch < 0 || num_heads <= 0 ||
      !valid_cu(cu_seqlens_host, batch))
    return 0;
  const std::vector<Piece> pcs = pieces_of(block_id_host, cu_seqlens_host, batch);
  int max_q = 1;
  for (const Piece& p : pcs) max_q = p.e - p.a > max_q ? p.e - p.a : max_q;
  return layout(pcs.size() > 0 ? pcs.size() : 1, max_q, num_heads).bytes;
}

bca_status bca_prefill_piecewise(const void* q, const void* k, const void* v,
                                 const int32_t* block_id, const int32_t* block_id_host,
                                 const int32_t* cu_seqlens_host, int32_t batch, int32_t num_heads,
                                 int32_t head_dim, int32_t total, float softmax_scale, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 int32_t* status_dev, void* stream) {
  if (head_dim != kHeadDim) return BCA_ERR_UNSUPPORTED;
  if (batch < 0 || num_heads <= 0 || total < 0) return BCA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return BCA_ERR_INVALID_ARG;
  if (batch == 0 || total == 0) return BCA_OK;
  if (!q || !k || !v || !block_id || !block_id_host || !cu_seqlens_host || !out || !lse)
    return BCA_ERR_INVALID_ARG;
  const auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return BCA_ERR_INVALID_ARG;
  if (!valid_cu(cu_seqlens_host, batch) || cu_seqlens_host[batch] != total)
    return BCA_ERR_SEQLENS;
  if (num_heads > 65535) return BCA_ERR_UNSUPPORTED;
  const std::vector<Piece> pcs = pieces_of(block_id_host, cu_seqlens_host, batch);
  int max_q = 1;
  for (const Piece& p : pcs) max_q = p.e - p.a > max_q ? p.e - p.a : max_q;
  const Scratch w = layout(pcs.size(), max_q, num_heads);
  if (workspace == nullptr || workspace_bytes < w.bytes || !aligned16(workspace))
    return BCA_ERR_WORKSPACE;

  auto st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto* d_cu = reinterpret_cast<int32_t*>(ws + w.cu_off);
  auto* row_end = reinterpret_cast<int32_t*>(ws + w.row_off);
  auto* tiles = reinterpret_cast<PrefillTile*>(ws + w.tile_off);
  auto* lse_tmp = reinterpret_cast<float*>(ws + w.lse_off);
  // per piece: cu_q = {0, e - a}, cu_k = {0, e - s}; one upload for all pieces
  std::vector<int32_t> h_cu(pcs.size() * 4);
  for (size_t i = 0; i < pcs.size(); ++i) {
    h_cu[4 * i + 0] = 0;
    h_cu[4 * i + 1] = pcs[i].e - pcs[i].a;
    h_cu[4 * i + 2] = 0;
    h_cu[4 * i + 3] = pcs[i].e - pcs[i].s;
  }
  if (cudaMemcpyAsync(d_cu, h_cu.data(), h_cu.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                      st) != cudaSuccess)
    return BCA_ERR_CUDA;
  const size_t row_bytes = static_cast<size_t>(num_heads) * kHeadDim * 2;   // one token, all heads
  for (size_t i = 0; i < pcs.size(); ++i) {
    const Piece& p = pcs[i];
    const int q_len = p.e - p.a, kv_len = p.e - p.s;
    const int tps = (q_len + kBlockM - 1) / kBlockM;
    if (launch_schedule_prep(block_id + p.s, d_cu + 4 * i, d_cu + 4 * i + 2, 1, q_len, kv_len,
                             tps, row_end, tiles, status_dev, st) != cudaSuccess)
      return BCA_ERR_CUDA;
    AttnLaunch a{};
    a.q = static_cast<const uint8_t*>(q) + p.a * row_bytes;
    a.k = static_cast<const uint8_t*>(k) + p.s * row_bytes;
    a.v = static_cast<const uint8_t*>(v) + p.s * row_bytes;
    a.out = static_cast<uint8_t*>(out) + p.a * row_bytes;
    a.lse = lse_tmp;
    a.batch = 1;
    a.num_heads = num_heads;
    a.total_q = q_len;
    a.total_k = kv_len;
    a.tiles_per_seq = tps;
    a.softmax_scale = softmax_scale;
    a.cu_q = d_cu + 4 * i;
    a.cu_k = d_cu + 4 * i + 2;
    a.row_end = row_end;
    a.tiles = tiles;
    a.status = status_dev;
    const int rc = launch_attention(a, /*decode=*/false, st);
    if (rc != BCA_OK) return static_cast<bca_status>(rc);
    if (cudaMemcpy2DAsync(lse + p.a, static_cast<size_t>(total) * sizeof(float), lse_tmp,
                          static_cast<size_t>(q_len) * sizeof(float),
                          static_cast<size_t>(q_len) * sizeof(float), num_heads,
                          cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return BCA_ERR_CUDA;
  }
  return BCA_OK;
}

}  // extern "C"

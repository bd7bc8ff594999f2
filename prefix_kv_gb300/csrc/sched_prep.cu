// Schedule preparation: the O(S) integer replacement of the O(S^2) block-causal mask.
//
// With every image id forming one contiguous run, row i of a sequence (key
// position p = kv_len - q_len + i, bottom-right alignment) sees exactly the key
// prefix [0, e), e = p + 1 for text and e = end of p's image run for an image
// token (10100.com, "Block-Causal mask": an image block [a, b) sees everything
// before it plus its own block).  Per 128-row query tile the attention kernel
// needs k_hi = max e (its K range, the per-M-block extension of the SenseNova-U1
// notes, "NEO-Unify 多模态 Prefill 的注意力") and k_min = min e (below it no key
// tile needs a mask).
//
// One CTA per sequence:
//   1. scan the block ids in chunks, collecting the (sorted) exclusive end of
//      every image run and its id; reject ids < -1;
//   2. reject an id that appears in two separate runs (flozi.net, "Block-causal
//      attention is the cache-enabling boundary": each image has its own id);
//   3. e per query row by binary search over the run ends; per-tile min/max.
#include "common.cuh"

namespace bca {
namespace {

constexpr int kPrepThreads = 512;
constexpr int kMaxRuns = 4096;

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

__global__ void __launch_bounds__(kPrepThreads)
    schedule_prep_kernel(const int32_t* __restrict__ bid, const int32_t* __restrict__ cu_q,
                         const int32_t* __restrict__ cu_k, int tiles_per_seq,
                         int32_t* __restrict__ row_end, PrefillTile* __restrict__ tiles,
                         int32_t* status) {
  __shared__ int run_end[kMaxRuns];
  __shared__ int run_id[kMaxRuns];
  __shared__ int warp_sum[kPrepThreads / 32];
  __shared__ int n_runs;
  __shared__ int err;
  __shared__ int red_max[kPrepThreads / 32], red_min[kPrepThreads / 32], red_cnt[kPrepThreads / 32];

  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31, wid = tid >> 5;
  const int k0 = cu_k[b];
  const int kv_len = cu_k[b + 1] - k0;
  const int q0 = cu_q[b];
  const int q_len = cu_q[b + 1] - q0;

  if (tid == 0) {
    n_runs = 0;
    err = 0;
    if (kv_len < 0 || q_len < 0 || q_len > kv_len || q_len > tiles_per_seq * kBlockM)
      err = BCA_ERR_SEQLENS;
  }
  __syncthreads();

  // ---- 1. image runs ------------------------------------------------------------
  if (err == 0) {
    for (int base = 0; base < kv_len; base += kPrepThreads) {
      const int j = base + tid;
      const bool in = j < kv_len;
      const int id = in ? bid[k0 + j] : -1;
      if (in && id < -1) err = BCA_ERR_BLOCK_ID;
      const bool is_end = in && id >= 0 && (j == kv_len - 1 || bid[k0 + j + 1] != id);
      const int incl = warp_incl_scan(is_end ? 1 : 0);
      if (lane == 31) warp_sum[wid] = incl;
      __syncthreads();
      if (wid == 0) {
        const int v = lane < kPrepThreads / 32 ? warp_sum[lane] : 0;
        const int s = warp_incl_scan(v);
        if (lane < kPrepThreads / 32) warp_sum[lane] = s - v;  // exclusive offsets
      }
      __syncthreads();
      const int rank = n_runs + warp_sum[wid] + incl - (is_end ? 1 : 0);
      if (is_end && rank < kMaxRuns) {
        run_end[rank] = j + 1;
        run_id[rank] = id;
      }
      __syncthreads();
      if (tid == kPrepThreads - 1) n_runs = rank + (is_end ? 1 : 0);
      __syncthreads();
    }
    if (tid == 0 && n_runs > kMaxRuns && err == 0) err = BCA_ERR_UNSUPPORTED;
    __syncthreads();

    // ---- 2. one run per id ----------------------------------------------------------
    if (err == 0) {
      const int R = n_runs;
      for (int a = tid; a < R; a += kPrepThreads) {
        const int id = run_id[a];
        for (int c = a + 1; c < R; ++c)
          if (run_id[c] == id) err = BCA_ERR_BLOCK_ID;
      }
    }
    __syncthreads();
  }

  if (err != 0) {
    if (tid == 0) report_status(status, err);
    for (int m = tid; m < tiles_per_seq; m += kPrepThreads)
      tiles[b * tiles_per_seq + m] = PrefillTile{0, 0, 0, 0};
    return;
  }

  // ---- 3. e per row, min / max per 128-row tile ------------------------------------
  const int R = n_runs;
  constexpr int kTilesPerPass = kPrepThreads / kBlockM;
  for (int m0 = 0; m0 < tiles_per_seq; m0 += kTilesPerPass) {
    const int m = m0 + tid / kBlockM;
    const int i = m * kBlockM + (tid % kBlockM);
    const bool valid = m < tiles_per_seq && i < q_len;
    int e = 0;
    if (valid) {
      const int pos = kv_len - q_len + i;
      const int id = bid[k0 + pos];
      if (id < 0) {
        e = pos + 1;
      } else {  // first run end > pos
        int lo = 0, hi = R;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (run_end[mid] > pos) hi = mid; else lo = mid + 1;
        }
        e = run_end[lo];
      }
      row_end[q0 + i] = e;
    }
    int vmax = valid ? e : 0;
    int vmin = valid ? e : 0x7fffffff;
    int cnt = valid ? 1 : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      vmax = max(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
      vmin = min(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
      cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    }
    if (lane == 0) {
      red_max[wid] = vmax;
      red_min[wid] = vmin;
      red_cnt[wid] = cnt;
    }
    __syncthreads();
    if (tid % kBlockM == 0 && m < tiles_per_seq) {
      const int w0 = tid / 32;
      int tmax = 0, tmin = 0x7fffffff, tcnt = 0;
      for (int w = w0; w < w0 + kBlockM / 32; ++w) {
        tmax = max(tmax, red_max[w]);
        tmin = min(tmin, red_min[w]);
        tcnt += red_cnt[w];
      }
      tiles[b * tiles_per_seq + m] =
          tcnt > 0 ? PrefillTile{tmax, tmin, tcnt, 0} : PrefillTile{0, 0, 0, 0};
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_schedule_prep(const int32_t* block_id, const int32_t* cu_q, const int32_t* cu_k,
                                 int batch, int tiles_per_seq, int32_t* row_end,
                                 PrefillTile* tiles, int32_t* status, cudaStream_t stream) {
  schedule_prep_kernel<<<batch, kPrepThreads, 0, stream>>>(block_id, cu_q, cu_k, tiles_per_seq,
                                                           row_end, tiles, status);
  return cudaGetLastError();
}

}  // namespace bca

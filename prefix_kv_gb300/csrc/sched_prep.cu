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
// A grid of (sequence, 1024-row chunk) CTAs of 1024 threads.  Every CTA of a
// sequence with rows to do runs steps 1 and 2 over the whole sequence (a few
// block-id reads from L2, so that no CTA waits on another), step 3 for its own rows:
//   1. stage 8192 block ids at a time in shared memory, mark the last position
//      of every image run (and reject ids < -1), and append the run ends, in
//      order, to a shared list with a block-wide scan;
//   2. reject an id that appears in two separate runs (flozi.net, "Block-causal
//      attention is the cache-enabling boundary": each image has its own id);
//   3. e per query row of the chunk by binary search over the run ends; min / max
//      of its eight 128-row tiles.
#include "common.cuh"
#include "ptx.cuh"

namespace bca {
namespace {

constexpr int kPrepThreads = 1024;
constexpr int kPerThread = 8;
constexpr int kChunk = kPrepThreads * kPerThread;  // positions or rows per pass
constexpr int kMaxRuns = 1024;  // image runs per sequence (BCA_ERR_UNSUPPORTED above)
constexpr int kWarps = kPrepThreads / 32;
constexpr int kTilesPerCta = kPrepThreads / kBlockM;   // one row per thread in step 3

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive prefix of `x` over the block; also returns the block total.
__device__ __forceinline__ int block_excl_scan(int x, int* warp_buf, int& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int incl = warp_incl_scan(x);
  if (lane == 31) warp_buf[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int v = warp_buf[lane];
    const int s = warp_incl_scan(v);
    warp_buf[lane] = s - v;
    if (lane == 31) warp_buf[kWarps] = s;
  }
  __syncthreads();
  const int r = warp_buf[wid] + incl - x;
  total = warp_buf[kWarps];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kPrepThreads)
    schedule_prep_kernel(const int32_t* __restrict__ bid, const int32_t* __restrict__ cu_q,
                         const int32_t* __restrict__ cu_k, int total_q, int total_k,
                         int tiles_per_seq, int32_t* __restrict__ row_end,
                         PrefillTile* __restrict__ tiles, int32_t* status) {
  __shared__ __align__(16) int ids[kChunk + 4];   // + the id past the chunk, padded
  __shared__ int run_end[kMaxRuns];
  __shared__ int run_id[kMaxRuns];
  __shared__ int warp_buf[kWarps + 1];
  __shared__ int red[3][kWarps];
  __shared__ int n_runs;
  __shared__ int err;

  // The attention grid launched next may start at once: it waits for this grid's
  // results where it reads them.
  grid_launch_dependents();
  const int b = blockIdx.x;
  const int chunk = blockIdx.y;   // query rows [chunk * 1024, chunk * 1024 + 1024)
  const int tid = threadIdx.x;
  const int lane = tid & 31, wid = tid >> 5;
  const int row = chunk * kPrepThreads + tid;   // this thread's query row in step 3
  const int k0 = cu_k[b];
  const int kv_len = cu_k[b + 1] - k0;
  const int q0 = cu_q[b];
  const int q_len = cu_q[b + 1] - q0;

  if (tid == 0) {
    n_runs = 0;
    err = 0;
    // the sequence's rows and keys must lie inside the packed arrays: nothing below
    // writes a row end or reads a block id before this check has passed
    if (kv_len < 0 || q_len < 0 || q_len > kv_len || q_len > tiles_per_seq * kBlockM ||
        q0 < 0 || k0 < 0 || q0 > total_q - q_len || k0 > total_k - kv_len)
      err = BCA_ERR_SEQLENS;
  }
  __syncthreads();
  // this CTA's eight tile records, zeroed (a chunk past the sequence's rows, or a
  // sequence that failed validation: the attention kernel skips zeroed tiles)
  auto zero_tiles = [&]() {
    if (tid < kTilesPerCta) {
      const int m = chunk * kTilesPerCta + tid;
      if (m < tiles_per_seq && BCA_IN_BOUNDS(status, b < static_cast<int>(gridDim.x)))
        tiles[b * tiles_per_seq + m] = PrefillTile{0, 0, 0, 0};
    }
  };
  if (err == 0 && chunk > 0 && chunk * kPrepThreads >= q_len) {
    zero_tiles();   // no rows here; the first chunk's CTA reports any bad id
    return;
  }
  const bool valid = err == 0 && row < q_len;
  // the row's own id, read now so that the load overlaps steps 1 and 2
  const int row_id = valid && BCA_IN_BOUNDS(status, k0 + kv_len - q_len + row < total_k)
                         ? bid[k0 + kv_len - q_len + row]
                         : -1;

  // ---- 1. image runs ------------------------------------------------------------
  if (err == 0) {
    for (int base = 0; base < kv_len; base += kChunk) {
      const int n = min(kChunk + 1, kv_len - base);  // + one id past the chunk
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        const int j = u * kPrepThreads + tid;
        if (j < n && BCA_IN_BOUNDS(status, k0 + base + j < total_k)) ids[j] = bid[k0 + base + j];
      }
      if (tid == 0 && kChunk < n && BCA_IN_BOUNDS(status, k0 + base + kChunk < total_k))
        ids[kChunk] = bid[k0 + base + kChunk];
      __syncthreads();
      // thread t looks at positions base + 8t .. base + 8t + 7 (read as two 16-byte
      // vectors plus the next id: scalar reads 8 words apart conflicted 8-way)
      int my[kPerThread + 1];
      {
        const int4 lo4 = *reinterpret_cast<const int4*>(&ids[tid * kPerThread]);
        const int4 hi4 = *reinterpret_cast<const int4*>(&ids[tid * kPerThread + 4]);
        my[0] = lo4.x; my[1] = lo4.y; my[2] = lo4.z; my[3] = lo4.w;
        my[4] = hi4.x; my[5] = hi4.y; my[6] = hi4.z; my[7] = hi4.w;
        my[8] = ids[tid * kPerThread + kPerThread];
      }
      int cnt = 0;
      unsigned ends = 0;
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        const int jl = tid * kPerThread + u;
        const int j = base + jl;
        if (j < kv_len) {
          const int id = my[u];
          if (id < -1) err = BCA_ERR_BLOCK_ID;
          if (id >= 0 && (j == kv_len - 1 || my[u + 1] != id)) {
            ends |= 1u << u;
            ++cnt;
          }
        }
      }
      int total;
      int rank = n_runs + block_excl_scan(cnt, warp_buf, total);
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        if (ends >> u & 1) {
          const int jl = tid * kPerThread + u;
          if (rank < kMaxRuns) {
            run_end[rank] = base + jl + 1;
            run_id[rank] = my[u];
          }
          ++rank;
        }
      }
      __syncthreads();
      if (tid == 0) n_runs += total;
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
    if (tid == 0 && chunk == 0) report_status(status, err);
    zero_tiles();
    return;
  }

  // ---- 3. e per row, min / max per 128-row tile ------------------------------------
  // Each warp owns 32 consecutive rows, each 128-row tile four consecutive warps.
  int e = 0;
  if (valid) {
    const int pos = kv_len - q_len + row;
    if (row_id < 0) {
      e = pos + 1;
    } else {  // first run end > pos
      int lo = 0, hi = n_runs;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (run_end[mid] > pos) hi = mid; else lo = mid + 1;
      }
      e = run_end[lo];
    }
    if (BCA_IN_BOUNDS(status, q0 + row >= 0 && q0 + row < total_q)) row_end[q0 + row] = e;
  }
  const int vmax = __reduce_max_sync(0xffffffffu, valid ? e : 0);
  const int vmin = __reduce_min_sync(0xffffffffu, valid ? e : 0x7fffffff);
  const int cnt = static_cast<int>(__reduce_add_sync(0xffffffffu, valid ? 1u : 0u));
  if (lane == 0) {
    red[0][wid] = vmax;
    red[1][wid] = vmin;
    red[2][wid] = cnt;
  }
  __syncthreads();
  if (tid < kTilesPerCta) {
    const int m = chunk * kTilesPerCta + tid;
    if (m < tiles_per_seq && BCA_IN_BOUNDS(status, b < static_cast<int>(gridDim.x))) {
      int tmax = 0, tmin = 0x7fffffff, tcnt = 0;
      for (int w = tid * (kBlockM / 32); w < (tid + 1) * (kBlockM / 32); ++w) {
        tmax = max(tmax, red[0][w]);
        tmin = min(tmin, red[1][w]);
        tcnt += red[2][w];
      }
      tiles[b * tiles_per_seq + m] = tcnt > 0 ? PrefillTile{tmax, tmin, tcnt, 0}
                                              : PrefillTile{0, 0, 0, 0};
    }
  }
}

}  // namespace

cudaError_t launch_schedule_prep(const int32_t* block_id, const int32_t* cu_q, const int32_t* cu_k,
                                 int batch, int total_q, int total_k, int tiles_per_seq,
                                 int32_t* row_end, PrefillTile* tiles, int32_t* status,
                                 cudaStream_t stream) {
  // at least one chunk, so that a sequence with rows but no tiles still reports
  const dim3 grid(batch, max(1, (tiles_per_seq + kTilesPerCta - 1) / kTilesPerCta));
  schedule_prep_kernel<<<grid, kPrepThreads, 0, stream>>>(block_id, cu_q, cu_k, total_q, total_k,
                                                          tiles_per_seq, row_end, tiles, status);
  return cudaGetLastError();
}

}  // namespace bca

// Q/K prologue of the attention: per-head RMS normalisation, three-axis RoPE
// and the append of the rotated prefix keys (and the values) to the cache.
//
// "Qwen-Image 2.1: Block-Causal Attention, Prefix KV Cache, and Turbo"
// (flozi.net): Q and K are RMS-normalised per head before RoPE (the paragraph
// on the 32 heads of width 128); "Three-axis RoPE preserves image geometry":
// the 128 dimensions split (16, 56, 56) across frame, height and width with
// base 10000, text advances one shared coordinate on all three axes, an image
// block keeps the frame coordinate the preceding text reached and lays its
// height/width coordinates on a grid centred on zero; RoPE changes Q and K,
// not V; "Timestep-zero conditioning makes the prefix invariant": the cache
// holds the post-RoPE prefix keys.
//
// Three kernels:
//   rope_positions_kernel  (frame, height, width) of every packed token; one
//                          1024-thread CTA per sequence, block scans.  Once
//                          per request.
//   rope_table_kernel      (cos, sin) of the 64 dimension pairs of every
//                          token, angles and sincos in double, stored fp32.
//                          Once per request; every layer and head reads it.
//   qk_norm_rope_kernel    per layer: 16 lanes per (token, head) row, 8 values
//                          each; fp32 RMS over the row by shuffles, weight,
//                          rotation of 4 interleaved pairs per lane, bf16 out;
//                          prefix tokens also write K_rot and V to the cache.
//                          HBM-bound.
// Conventions (readings where the page is silent): a running coordinate c
// starts at 0 per sequence; text takes (c, c, c) and advances c; an image of
// Hg x Wg tokens (row-major) takes frame c and (row - Hg/2, col - Wg/2), then
// advances c by one.  Pair k of axis a (d_a dims from offset o_a) turns by
// p_a * 10000^(-2k/d_a): (x, y) -> (x cos - y sin, x sin + y cos).
#include "kernels.cuh"
#include "ptx.cuh"

namespace bca {
namespace {

constexpr int kPosThreads = 1024;
constexpr int kPosWarps = kPosThreads / 32;

// Inclusive scan over the CTA of `x` under `op` (sum or max); the CTA total
// (or max) lands in `all`.
template <bool kMax>
__device__ __forceinline__ int block_incl_scan(int x, int* buf, int& all) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = kMax ? max(x, y) : x + y;
  }
  if (lane == 31) buf[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int v = buf[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v = kMax ? max(v, y) : v + y;
    }
    buf[lane] = v;                      // inclusive over warps
  }
  __syncthreads();
  if (wid > 0) x = kMax ? max(x, buf[wid - 1]) : x + buf[wid - 1];
  all = buf[kPosWarps - 1];
  __syncthreads();
  return x;
}

__global__ void __launch_bounds__(kPosThreads)
    rope_positions_kernel(const int32_t* __restrict__ bid, const int32_t* __restrict__ cu,
                          const int32_t* __restrict__ grid_w, int n_ids, int total,
                          int32_t* __restrict__ pos3, int32_t* status) {
  extern __shared__ int dyn[];
  int* cnt = dyn;                 // tokens of each image id in this sequence
  int* starts = dyn + n_ids;      // runs of each image id
  __shared__ int buf[kPosWarps];
  __shared__ int err;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int t0 = cu[b], t1 = cu[b + 1];
  for (int i = tid; i < n_ids; i += kPosThreads) {
    cnt[i] = 0;
    starts[i] = 0;
  }
  // the sequence's tokens must lie in [0, total): nothing is read or written otherwise
  if (tid == 0) err = (t1 < t0 || t0 < 0 || t1 > total) ? BCA_ERR_SEQLENS : 0;
  __syncthreads();
  // pass 1: image block sizes, one run per id
  for (int t = t0 + tid; t < t1; t += kPosThreads) {
    const int id = bid[t];
    if (id < -1 || id >= n_ids) {
      err = BCA_ERR_BLOCK_ID;
    } else if (id >= 0) {
      atomicAdd(&cnt[id], 1);
      if (t == t0 || bid[t - 1] != id) atomicAdd(&starts[id], 1);
    }
  }
  __syncthreads();
  for (int i = tid; i < n_ids; i += kPosThreads) {
    if (cnt[i] == 0) continue;
    const int w = grid_w[static_cast<int64_t>(b) * n_ids + i];
    if (starts[i] != 1 || w <= 0 || cnt[i] % w != 0) err = BCA_ERR_BLOCK_ID;
  }
  __syncthreads();
  if (err != 0) {
    if (tid == 0) report_status(status, err);
    return;
  }
  // pass 2: A(t) = number of tokens in [t0, t) that are text or start an image
  // block; text takes (A, A, A), an image token frame A(start of its block)
  int carry_a = 0, carry_start = -1;
  for (int c0 = t0; c0 < t1; c0 += kPosThreads) {
    const int t = c0 + tid;
    const bool valid = t < t1;
    const int id = valid ? bid[t] : -1;
    const bool start = valid && id >= 0 && (t == t0 || bid[t - 1] != id);
    const int f = valid && (id < 0 || start) ? 1 : 0;
    int sum_all, max_all;
    const int a_excl = block_incl_scan<false>(f, buf, sum_all) - f + carry_a;
    const int s = max(carry_start, block_incl_scan<true>(start ? t : -1, buf, max_all));
    if (valid) {
      int32_t* out = pos3 + static_cast<int64_t>(t) * 3;
      if (!BCA_IN_BOUNDS(status, t >= 0 && t < total)) {
        // skipped (bounds-checked build)
      } else if (id < 0) {
        out[0] = a_excl;
        out[1] = a_excl;
        out[2] = a_excl;
      } else {
        const int i = t - s;                              // index inside the block
        const int w = grid_w[static_cast<int64_t>(b) * n_ids + id];
        const int hg = cnt[id] / w;
        out[0] = a_excl - (t != s ? 1 : 0);
        out[1] = i / w - hg / 2;
        out[2] = i % w - w / 2;
      }
    }
    carry_a += sum_all;
    carry_start = max(carry_start, max_all);
  }
}

// (cos, sin) of pair j of token t at table[t * 64 + j].  The 64 inverse
// frequencies are computed once per CTA in double; each angle is reduced
// modulo 2 pi in double (error ~1e-12 for coordinates up to 1e5), and the
// remainder, |r| <= pi, goes through fp32 sincosf (error ~1e-7).
__global__ void __launch_bounds__(256)
    rope_table_kernel(const int32_t* __restrict__ pos3, int64_t total, float2* __restrict__ table) {
  __shared__ double inv_freq[64];
  if (threadIdx.x < 64) {
    const int j = threadIdx.x;
    const int axis = j < 8 ? 0 : (j < 36 ? 1 : 2);
    const int k = j - (axis == 0 ? 0 : (axis == 1 ? 8 : 36));
    const double d = axis == 0 ? 16.0 : 56.0;
    inv_freq[j] = pow(10000.0, -2.0 * k / d);
  }
  __syncthreads();
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  constexpr double kInvTwoPi = 0.15915494309189533576888376337251;
  const int64_t n = total * 64;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx >> 6;
    const int j = static_cast<int>(idx & 63);
    const int axis = j < 8 ? 0 : (j < 36 ? 1 : 2);
    const double theta = static_cast<double>(pos3[t * 3 + axis]) * inv_freq[j];
    const double r = fma(-rint(theta * kInvTwoPi), kTwoPi, theta);
    float s, c;
    sincosf(static_cast<float>(r), &s, &c);
    table[idx] = make_float2(c, s);
  }
}

constexpr int kPrologueThreads = 256;
constexpr int kMaxBatchSmem = 1024;

__device__ __forceinline__ void unpack8(uint4 r, float x[8]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// The lane's 8 weights (dimensions 8 * l16 ..), or ones without a weight.
__device__ __forceinline__ void load_gamma8(const float* __restrict__ g, int l16, float out[8]) {
  if (g == nullptr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = 1.f;
    return;
  }
  const float4 a = __ldg(reinterpret_cast<const float4*>(g) + 2 * l16);
  const float4 b = __ldg(reinterpret_cast<const float4*>(g) + 2 * l16 + 1);
  out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
  out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}

// 1 / sqrt(mean of squares over the 128 values of the row + eps); the 16 lanes
// of a row group hold 8 values each.
__device__ __forceinline__ float row_inv_rms(const float x[8], float eps) {
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  return 1.0f / sqrtf(ss * (1.0f / 128.0f) + eps);
}

// Normalise, weight and rotate the lane's 8 values; returns them as bf16.
__device__ __forceinline__ uint4 norm_rope8(const float x[8], float inv_rms, const float g[8],
                                            const float4 cs[2]) {
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = x[i] * inv_rms * g[i];
  const float c[4] = {cs[0].x, cs[0].z, cs[1].x, cs[1].z};
  const float s[4] = {cs[0].y, cs[0].w, cs[1].y, cs[1].w};
  uint32_t o[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float a = y[2 * p], bb = y[2 * p + 1];
    o[p] = pack_bf16x2(a * c[p] - bb * s[p], a * s[p] + bb * c[p]);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <bool kAppend>
__global__ void __launch_bounds__(kPrologueThreads, 4)
    qk_norm_rope_kernel(const uint4* q, const uint4* k, const uint4* __restrict__ v,
                        const float* __restrict__ gamma_q, const float* __restrict__ gamma_k,
                        const float4* __restrict__ table, const int32_t* __restrict__ cu_k,
                        const int32_t* __restrict__ cu_prefix, int batch, int num_heads,
                        int total, float eps, uint4* q_out, uint4* k_out, uint4* __restrict__ ck,
                        uint4* __restrict__ cv, int64_t capacity, int32_t* status) {
  __shared__ int s_ck[kMaxBatchSmem + 1];
  __shared__ int s_cp[kMaxBatchSmem + 1];
  __shared__ int s_bad;
  const bool in_smem = batch <= kMaxBatchSmem;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  if (kAppend && in_smem) {
    for (int i = threadIdx.x; i <= batch; i += blockDim.x) {
      s_ck[i] = cu_k[i];
      s_cp[i] = cu_prefix[i];
    }
  }
  __syncthreads();
  const int32_t* ckk = kAppend && in_smem ? s_ck : cu_k;
  const int32_t* cpp = kAppend && in_smem ? s_cp : cu_prefix;
  if (kAppend) {
    // the same checks as the plain append, by every CTA before any write
    for (int i = threadIdx.x; i < batch; i += blockDim.x) {
      const int pl = cpp[i + 1] - cpp[i];
      const int kl = ckk[i + 1] - ckk[i];
      if (pl < 0 || pl > kl || cpp[i] < 0) s_bad = BCA_ERR_SEQLENS;
    }
    if (threadIdx.x == 0 && static_cast<int64_t>(cpp[batch]) > capacity) s_bad = BCA_ERR_CAPACITY;
    __syncthreads();
    if (s_bad != 0) {
      if (blockIdx.x == 0 && threadIdx.x == 0) report_status(status, s_bad);
      return;
    }
  }
  const int l16 = threadIdx.x & 15;
  const int64_t rows = static_cast<int64_t>(total) * num_heads;
  const int64_t groups = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 4);
  // one 16-lane group per (token, head) row; whole warps stay in the loop for the shuffles
  for (int64_t r2 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       r2 * 2 < rows; r2 += groups / 2) {
    const int64_t row = r2 * 2 + ((threadIdx.x >> 4) & 1);
    const bool live = row < rows;
    const int64_t rr = live ? row : rows - 1;
    const int t = static_cast<int>(rr / num_heads);
    const int hh = static_cast<int>(rr - static_cast<int64_t>(t) * num_heads);
    int64_t crow = -1;                                     // cache row of a prefix token
    if (kAppend) {
      int lo = 0, hi = batch - 1;                          // sequence of token t
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ckk[mid] <= t) lo = mid; else hi = mid - 1;
      }
      const int j = t - ckk[lo];                           // position inside the sequence
      if (live && j < cpp[lo + 1] - cpp[lo])
        crow = static_cast<int64_t>(hh) * capacity + cpp[lo] + j;
    }
    // every load of the row first
    const uint4 qraw = __ldcs(q + rr * 16 + l16);
    const uint4 kraw = __ldcs(k + rr * 16 + l16);
    uint4 vraw = make_uint4(0, 0, 0, 0);
    if (kAppend && crow >= 0) vraw = __ldcs(v + rr * 16 + l16);
    float4 cs[2];
    cs[0] = table[static_cast<int64_t>(t) * 32 + 2 * l16];
    cs[1] = table[static_cast<int64_t>(t) * 32 + 2 * l16 + 1];
    float xq[8], xk[8], gq[8], gk[8];
    load_gamma8(gamma_q, l16, gq);      // L1-resident; reloaded per row to save registers
    load_gamma8(gamma_k, l16, gk);
    unpack8(qraw, xq);
    unpack8(kraw, xk);
    const float rq = row_inv_rms(xq, eps);
    const float rk = row_inv_rms(xk, eps);
    const uint4 qo = norm_rope8(xq, rq, gq, cs);
    const uint4 ko = norm_rope8(xk, rk, gk, cs);
    if (!live) continue;
    q_out[rr * 16 + l16] = qo;
    k_out[rr * 16 + l16] = ko;
    if (kAppend && crow >= 0 &&
        BCA_IN_BOUNDS(status, crow < static_cast<int64_t>(num_heads) * capacity)) {
      ck[crow * 16 + l16] = ko;
      cv[crow * 16 + l16] = vraw;
    }
  }
}

}  // namespace

cudaError_t launch_rope_positions(const int32_t* block_id, const int32_t* cu_seqlens, int batch,
                                  int total, const int32_t* grid_w, int n_ids, int32_t* pos3,
                                  int32_t* status, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(2) * n_ids * sizeof(int);
  rope_positions_kernel<<<batch, kPosThreads, smem, stream>>>(block_id, cu_seqlens, grid_w, n_ids,
                                                              total, pos3, status);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(const int32_t* pos3, int64_t total, float* table,
                              cudaStream_t stream) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // few CTAs: each computes the 64 double-precision frequencies once
  const int64_t n = total * 64;
  const int64_t want = (n + 255) / 256;
  const int blocks = static_cast<int>(want < 2 * sms ? want : 2 * sms);
  rope_table_kernel<<<blocks, 256, 0, stream>>>(pos3, total, reinterpret_cast<float2*>(table));
  return cudaGetLastError();
}

cudaError_t launch_qk_norm_rope(const void* q, const void* k, const void* v, const float* gamma_q,
                                const float* gamma_k, const float* table, const int32_t* cu_k,
                                const int32_t* cu_prefix, int batch, int num_heads, int total,
                                float eps, void* q_out, void* k_out, void* cache_k_layer,
                                void* cache_v_layer, int64_t capacity, int32_t* status,
                                cudaStream_t stream) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = sms * 8;
  const auto* q4 = static_cast<const uint4*>(q);
  const auto* k4 = static_cast<const uint4*>(k);
  const auto* v4 = static_cast<const uint4*>(v);
  const auto* t4 = reinterpret_cast<const float4*>(table);
  if (cu_prefix != nullptr) {
    qk_norm_rope_kernel<true><<<grid, kPrologueThreads, 0, stream>>>(
        q4, k4, v4, gamma_q, gamma_k, t4, cu_k, cu_prefix, batch, num_heads, total, eps,
        static_cast<uint4*>(q_out), static_cast<uint4*>(k_out),
        static_cast<uint4*>(cache_k_layer), static_cast<uint4*>(cache_v_layer), capacity, status);
  } else {
    qk_norm_rope_kernel<false><<<grid, kPrologueThreads, 0, stream>>>(
        q4, k4, v4, gamma_q, gamma_k, t4, cu_k, cu_prefix, batch, num_heads, total, eps,
        static_cast<uint4*>(q_out), static_cast<uint4*>(k_out), nullptr, nullptr, capacity,
        status);
  }
  return cudaGetLastError();
}

}  // namespace bca

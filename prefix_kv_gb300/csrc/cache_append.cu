// Prefix K/V cache append (the "extract" step).
//
// Sequence b's first P_b = cu_prefix[b+1] - cu_prefix[b] keys and values,
// packed [total_k, H, 128] bf16, are cloned into cache tokens cu_prefix[b]..
// of one layer's [H][capacity][128] slab (flozi.net, "Timestep-zero
// conditioning makes the prefix invariant": the extract step stores post-RoPE
// prefix K/V per layer as a clone; "The prefix cache is a compute-for-memory
// trade": two tensors of H x 128 values per token and layer).
//
// The copy is HBM-bound: each (token, head) row is 256 contiguous bytes on
// both sides, so one 16-thread group moves one row with 16-byte vectors;
// reads walk the packed tensor in order, writes land in 256-byte runs.
// Validation (capacity, prefix <= sequence) is done by every thread before it
// writes anything, so a failing call writes nothing.
#include "common.cuh"

namespace bca {
namespace {

constexpr int kAppendThreads = 256;
constexpr int kMaxBatchSmem = 1024;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kAppendThreads)
    cache_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                        const int32_t* __restrict__ cu_k, const int32_t* __restrict__ cu_prefix,
                        int batch, int num_heads, uint4* __restrict__ ck, uint4* __restrict__ cv,
                        int64_t capacity, int32_t* status) {
  __shared__ int s_cp[kMaxBatchSmem + 1];
  __shared__ int s_ck[kMaxBatchSmem + 1];
  __shared__ int s_bad;
  const bool in_smem = batch <= kMaxBatchSmem;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  if (in_smem) {
    for (int i = threadIdx.x; i <= batch; i += blockDim.x) {
      s_cp[i] = cu_prefix[i];
      s_ck[i] = cu_k[i];
    }
  }
  __syncthreads();
  const int32_t* cp = in_smem ? s_cp : cu_prefix;
  const int32_t* ckk = in_smem ? s_ck : cu_k;

  // validation: every CTA checks every sequence (batch is small)
  for (int i = threadIdx.x; i < batch; i += blockDim.x) {
    const int pl = cp[i + 1] - cp[i];
    const int kl = ckk[i + 1] - ckk[i];
    if (pl < 0 || pl > kl || cp[i] < 0) s_bad = BCA_ERR_SEQLENS;
  }
  if (threadIdx.x == 0 && static_cast<int64_t>(cp[batch]) > capacity) s_bad = BCA_ERR_CAPACITY;
  __syncthreads();
  if (s_bad != 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report_status(status, s_bad);
    return;
  }

  const int p0 = cp[0];
  const int64_t total_tok = cp[batch] - p0;
  const int64_t vec_per_tok = static_cast<int64_t>(num_heads) * 16;
  const int64_t total_vec = total_tok * vec_per_tok;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       base < total_vec; base += stride * kUnroll) {
    uint4 rk[kUnroll], rv[kUnroll];
    int64_t dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t idx = base + u * stride;
      dst[u] = -1;
      if (idx < total_vec) {
        const int c = static_cast<int>(idx / vec_per_tok) + p0;   // cache token
        const int rem = static_cast<int>(idx % vec_per_tok);
        const int hh = rem >> 4, x = rem & 15;
        int lo = 0, hi = batch - 1;                                 // sequence of c
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (cp[mid] <= c) lo = mid; else hi = mid - 1;
        }
        const int64_t src_tok = static_cast<int64_t>(ckk[lo]) + (c - cp[lo]);
        const int64_t src = (src_tok * num_heads + hh) * 16 + x;
        dst[u] = (static_cast<int64_t>(hh) * capacity + c) * 16 + x;
        rk[u] = __ldcs(k + src);
        rv[u] = __ldcs(v + src);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (dst[u] >= 0) {
        ck[dst[u]] = rk[u];
        cv[dst[u]] = rv[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_cache_append(const void* k, const void* v, const int32_t* cu_k,
                                const int32_t* cu_prefix, int batch, int num_heads,
                                void* cache_k_layer, void* cache_v_layer, int64_t capacity,
                                int32_t* status, cudaStream_t stream) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = sms * 8;
  cache_append_kernel<<<grid, kAppendThreads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), cu_k, cu_prefix, batch,
      num_heads, static_cast<uint4*>(cache_k_layer), static_cast<uint4*>(cache_v_layer), capacity,
      status);
  return cudaGetLastError();
}

}  // namespace bca

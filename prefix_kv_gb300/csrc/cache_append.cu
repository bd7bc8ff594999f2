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
// writes anything, so a failing call writes nothing.  With a page table the
// prefix token t of sequence b goes to cache token page_table[b][t/128]*128 +
// t%128 instead (one 128-token page per tile), every page id checked first.
// Further down: the row copy of a shared tail page, the FP8 E4M3 append, its
// expansion back to bf16, and the gather of paged layers for decode.
#include "kernels.cuh"
#include "ptx.cuh"

#include <algorithm>

namespace bca {
namespace {

constexpr int kAppendThreads = 256;
constexpr int kMaxBatchSmem = 1024;
constexpr int kUnroll = 4;

// Cache token of prefix token t of sequence b: contiguous (cu_prefix[b] + t) or,
// with a page table, page_table[b][t / 128] * 128 + t % 128.
__device__ __forceinline__ int64_t cache_token(const int32_t* __restrict__ page_table,
                                               int max_pages, const int32_t* cp, int b, int t) {
  if (page_table == nullptr) return static_cast<int64_t>(cp[b]) + t;
  return static_cast<int64_t>(page_table[static_cast<int64_t>(b) * max_pages + (t >> 7)]) * 128 +
         (t & 127);
}

// Every page entry a prefix needs lies in [0, capacity / 128) (paged caches).
__device__ int check_pages(const int32_t* __restrict__ page_table, int max_pages,
                           const int32_t* cp, int batch, int64_t capacity) {
  int bad = 0;
  const int64_t n_pages = capacity / 128;
  for (int b = 0; b < batch; ++b) {
    const int n = (cp[b + 1] - cp[b] + 127) / 128;
    if (n > max_pages) bad = BCA_ERR_CAPACITY;
    for (int j = threadIdx.x; j < n && j < max_pages; j += blockDim.x) {
      const int pg = page_table[static_cast<int64_t>(b) * max_pages + j];
      if (pg < 0 || pg >= n_pages) bad = BCA_ERR_CAPACITY;
    }
  }
  return bad;
}

__global__ void __launch_bounds__(kAppendThreads)
    cache_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                        const int32_t* __restrict__ cu_k, const int32_t* __restrict__ cu_prefix,
                        int batch, int num_heads, int total_k, uint4* __restrict__ ck,
                        uint4* __restrict__ cv,
                        int64_t capacity, const int32_t* __restrict__ page_table, int max_pages,
                        int32_t* status) {
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
    // the prefix's source keys [cu_k[i], cu_k[i] + pl) must lie in [0, total_k)
    if (pl < 0 || pl > kl || cp[i] < 0 || ckk[i] < 0 || ckk[i] > total_k - pl)
      s_bad = BCA_ERR_SEQLENS;
  }
  if (page_table == nullptr) {
    if (threadIdx.x == 0 && static_cast<int64_t>(cp[batch]) > capacity) s_bad = BCA_ERR_CAPACITY;
  } else if (check_pages(page_table, max_pages, cp, batch, capacity) != 0) {
    s_bad = BCA_ERR_CAPACITY;
  }
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
        const int64_t ctok = cache_token(page_table, max_pages, cp, lo, c - cp[lo]);
        if (BCA_IN_BOUNDS(status, src_tok >= 0 && src_tok < total_k && ctok >= 0 &&
                                      ctok < capacity)) {
          dst[u] = (static_cast<int64_t>(hh) * capacity + ctok) * 16 + x;
          rk[u] = __ldcs(k + src);
          rv[u] = __ldcs(v + src);
        }
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
                                const int32_t* cu_prefix, int batch, int num_heads, int total_k,
                                void* cache_k_layer, void* cache_v_layer, int64_t capacity,
                                const int32_t* page_table, int max_pages, int32_t* status,
                                cudaStream_t stream) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = sms * 8;
  cache_append_kernel<<<grid, kAppendThreads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), cu_k, cu_prefix, batch,
      num_heads, total_k, static_cast<uint4*>(cache_k_layer), static_cast<uint4*>(cache_v_layer),
      capacity, page_table, max_pages, status);
  return cudaGetLastError();
}

namespace {

// Rows [0, n_rows) of page src copied to page dst, every head, K and V.
__global__ void __launch_bounds__(256)
    cache_copy_rows_kernel(uint4* __restrict__ ck, uint4* __restrict__ cv, int num_heads,
                           int64_t capacity, int src_page, int dst_page, int n_rows) {
  const int64_t n = static_cast<int64_t>(num_heads) * n_rows * 16;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int x = static_cast<int>(i & 15);
    const int64_t rh = i >> 4;
    const int r = static_cast<int>(rh % n_rows);
    const int hh = static_cast<int>(rh / n_rows);
    const int64_t base = static_cast<int64_t>(hh) * capacity;
    const int64_t s = (base + static_cast<int64_t>(src_page) * 128 + r) * 16 + x;
    const int64_t d = (base + static_cast<int64_t>(dst_page) * 128 + r) * 16 + x;
    ck[d] = ck[s];
    cv[d] = cv[s];
  }
}

}  // namespace

cudaError_t launch_cache_copy_rows(void* cache_k_layer, void* cache_v_layer, int num_heads,
                                   int64_t capacity, int src_page, int dst_page, int n_rows,
                                   cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(num_heads) * n_rows * 16;
  const int blocks = static_cast<int>((n + 255) / 256 < 1216 ? (n + 255) / 256 : 1216);
  if (blocks == 0) return cudaSuccess;
  cache_copy_rows_kernel<<<blocks, 256, 0, stream>>>(static_cast<uint4*>(cache_k_layer),
                                                     static_cast<uint4*>(cache_v_layer), num_heads,
                                                     capacity, src_page, dst_page, n_rows);
  return cudaGetLastError();
}

}  // namespace bca

// ---------------------------------------------------------------------------
// FP8 E4M3 variant ("Qwen-Image 2.1 deployment notes", prefix-cache section:
// FP8 E4M3 with one FP32 scale per token and head, quantising K and V or V
// only).  Each (token, head) row of 128 values is scaled by its absmax onto
// the E4M3 range: scale = amax / 448, code = E4M3(x * (448 / amax)), rounded
// to nearest even and saturating, all arithmetic in fp32.  16 threads share a
// row (8 values each) and reduce amax with warp shuffles.
namespace bca {
namespace {

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantises the 8 bf16 values of one thread; returns the 8 codes as a uint2.
__device__ __forceinline__ uint2 quantize8(uint4 raw, float* scale_out) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float x[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  *scale_out = amax / 448.0f;
  const float inv = amax > 0.f ? 448.0f / amax : 0.f;
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    c[i] = e4m3x2(x[2 * i] * inv, x[2 * i + 1] * inv);
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

template <bool kQuantK>
__global__ void __launch_bounds__(256)
    cache_append_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                            const int32_t* __restrict__ cu_k, const int32_t* __restrict__ cu_prefix,
                            int batch, int num_heads, int total_k, void* __restrict__ ck,
                            uint2* __restrict__ cv,
                            float* __restrict__ sk, float* __restrict__ sv, int64_t capacity,
                            const int32_t* __restrict__ page_table, int max_pages,
                            int32_t* status) {
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < batch; i += blockDim.x) {
    const int pl = cu_prefix[i + 1] - cu_prefix[i];
    const int kl = cu_k[i + 1] - cu_k[i];
    if (pl < 0 || pl > kl || cu_prefix[i] < 0 || cu_k[i] < 0 || cu_k[i] > total_k - pl)
      s_bad = BCA_ERR_SEQLENS;
  }
  if (page_table == nullptr) {
    if (threadIdx.x == 0 && static_cast<int64_t>(cu_prefix[batch]) > capacity)
      s_bad = BCA_ERR_CAPACITY;
  } else if (check_pages(page_table, max_pages, cu_prefix, batch, capacity) != 0) {
    s_bad = BCA_ERR_CAPACITY;
  }
  __syncthreads();
  if (s_bad != 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report_status(status, s_bad);
    return;
  }
  const int p0 = cu_prefix[0];
  // (token, head) rows of the prefix region: at most capacity x heads < 2^31 (host check),
  // so the row arithmetic is 32-bit (a 64-bit division per row had made the kernel
  // bound by its instruction issue)
  const uint32_t rows = static_cast<uint32_t>(cu_prefix[batch] - p0) * static_cast<uint32_t>(num_heads);
  const uint32_t warps = gridDim.x * (blockDim.x >> 5);
  const int lane16 = threadIdx.x & 15;
  // Row (token, head) of the prefix region -> source vector and cache row.
  struct Where {
    int64_t src, dst_row;
    bool in;   // source token and cache row inside their buffers (bounds-checked build)
  };
  auto locate = [&](uint32_t row) {
    const uint32_t c_rel = row / static_cast<uint32_t>(num_heads);
    const int c = static_cast<int>(c_rel) + p0;                  // cache token
    const int hh = static_cast<int>(row - c_rel * static_cast<uint32_t>(num_heads));
    int lo = 0, hi = batch - 1;                                  // sequence of c
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu_prefix[mid] <= c) lo = mid; else hi = mid - 1;
    }
    const int64_t src_tok = static_cast<int64_t>(cu_k[lo]) + (c - cu_prefix[lo]);
    const int64_t ctok = cache_token(page_table, max_pages, cu_prefix, lo, c - cu_prefix[lo]);
    return Where{(src_tok * num_heads + hh) * 16 + lane16,
                 static_cast<int64_t>(hh) * capacity + ctok,
                 BCA_IN_BOUNDS(status, src_tok >= 0 && src_tok < total_k && ctok >= 0 &&
                                           ctok < capacity)};
  };
  // Two rows per warp (16 lanes each; all 32 lanes stay together for the shuffles)
  // and two such row pairs per pass, with all four loads issued before any
  // quantisation so that each lane keeps them in flight together.
  constexpr int kPairs = 2;
  for (uint32_t r2 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r2 * 2 < rows;
       r2 += kPairs * warps) {
    bool live[kPairs];
    int64_t src[kPairs], dst_row[kPairs];
    uint4 vraw[kPairs], kraw[kPairs];
#pragma unroll
    for (int u = 0; u < kPairs; ++u) {
      const uint32_t row = (r2 + u * warps) * 2 + ((threadIdx.x >> 4) & 1);
      live[u] = row < rows;
      const Where w = locate(live[u] ? row : rows - 1);
      if (!w.in) {   // skip the row (bounds-checked build); the lanes stay together
        live[u] = false;
        src[u] = 0;
        dst_row[u] = 0;
        vraw[u] = kraw[u] = make_uint4(0, 0, 0, 0);
        continue;
      }
      src[u] = w.src;
      dst_row[u] = w.dst_row;
      vraw[u] = __ldcs(v + src[u]);
      kraw[u] = __ldcs(k + src[u]);
    }
#pragma unroll
    for (int u = 0; u < kPairs; ++u) {
      float scale_v, scale_k;
      const uint2 qv = quantize8(vraw[u], &scale_v);
      if (live[u]) {
        cv[dst_row[u] * 16 + lane16] = qv;
        if (lane16 == 0) sv[dst_row[u]] = scale_v;
      }
      if constexpr (kQuantK) {
        const uint2 qk = quantize8(kraw[u], &scale_k);
        if (live[u]) {
          static_cast<uint2*>(ck)[dst_row[u] * 16 + lane16] = qk;
          if (lane16 == 0) sk[dst_row[u]] = scale_k;
        }
      } else {
        if (live[u]) static_cast<uint4*>(ck)[dst_row[u] * 16 + lane16] = kraw[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_cache_append_fp8(const void* k, const void* v, const int32_t* cu_k,
                                    const int32_t* cu_prefix, int batch, int num_heads,
                                    int total_k, bool quant_k, void* cache_k_layer, void* cache_v_layer,
                                    float* scale_k_layer, float* scale_v_layer, int64_t capacity,
                                    const int32_t* page_table, int max_pages, int32_t* status,
                                    cudaStream_t stream) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // One wave of the grid-stride loop: as many CTAs as fit on the SMs at once (the
  // kernel's registers allow 5 per SM, so 8 per SM ran as 1.6 uneven waves).
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, quant_k ? cache_append_fp8_kernel<true> : cache_append_fp8_kernel<false>, 256,
          0) != cudaSuccess ||
      per_sm <= 0)
    per_sm = 4;
  const int grid = sms * per_sm;
  if (quant_k) {
    cache_append_fp8_kernel<true><<<grid, 256, 0, stream>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), cu_k, cu_prefix, batch,
        num_heads, total_k, cache_k_layer, static_cast<uint2*>(cache_v_layer), scale_k_layer,
        scale_v_layer, capacity, page_table, max_pages, status);
  } else {
    cache_append_fp8_kernel<false><<<grid, 256, 0, stream>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), cu_k, cu_prefix, batch,
        num_heads, total_k, cache_k_layer, static_cast<uint2*>(cache_v_layer), scale_k_layer,
        scale_v_layer, capacity, page_table, max_pages, status);
  }
  return cudaGetLastError();
}

}  // namespace bca

// ---------------------------------------------------------------------------
// Expansion of the E4M3 cache back to bf16 for attention: every element of
// the stored prefix rows becomes bf16(fp32(value(code)) * scale), the
// dequantised value of the append's format, written in the bf16 cache layout.
// HBM-bound: a row is 128 code bytes plus one scale in, 256 bytes out.  Sixteen
// threads share a row, 8 codes each, so a warp's 8-byte loads read 256 and its
// 16-byte stores write 512 contiguous bytes; each thread loads kDequantUnroll
// such chunks (a grid stride apart) before expanding any.
namespace bca {
namespace {

constexpr int kDequantUnroll = 4;

// 8 E4M3 codes (the low byte first) times `scale`, rounded to 8 bf16 values.
__device__ __forceinline__ uint4 dequant8(uint2 raw, float scale) {
  const uint32_t w[2] = {raw.x, raw.y};
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const float2 f = e4m3x2_to_float2(static_cast<uint16_t>(w[q] >> (16 * hb)));
      o[2 * q + hb] = pack_bf16x2(f.x * scale, f.y * scale);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(256)
    cache_dequant_fp8_kernel(const uint2* __restrict__ codes, const float* __restrict__ scales,
                             const int32_t* __restrict__ cu_prefix, int batch, int num_heads,
                             int64_t capacity, uint4* __restrict__ out, int32_t* status) {
  const int p0 = cu_prefix[0], p1 = cu_prefix[batch];
  if (p0 < 0 || p1 < p0 || static_cast<int64_t>(p1) > capacity) {
    if (blockIdx.x == 0 && threadIdx.x == 0)
      report_status(status, p1 > capacity ? BCA_ERR_CAPACITY : BCA_ERR_SEQLENS);
    return;
  }
  // a grid of (chunk range, head): head h's prefix rows are contiguous, rows
  // h * capacity + p0 .. h * capacity + p1 - 1, 16 chunks of 8 codes each
  const int hh = blockIdx.y;
  const int64_t row0 = static_cast<int64_t>(hh) * capacity + p0;
  const uint32_t chunks = static_cast<uint32_t>(p1 - p0) * 16u;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < chunks;
       base += stride * kDequantUnroll) {
    uint2 raw[kDequantUnroll];
    float sc[kDequantUnroll];
    int64_t at[kDequantUnroll];   // chunk index in the layer, -1: none
#pragma unroll
    for (int u = 0; u < kDequantUnroll; ++u) {
      const uint32_t c = base + u * stride;
      at[u] = -1;
      if (c < chunks && BCA_IN_BOUNDS(status, hh < num_heads)) {
        const int64_t row = row0 + (c >> 4);
        at[u] = row * 16 + (c & 15);
        raw[u] = __ldcs(codes + at[u]);
        sc[u] = __ldg(scales + row);
      }
    }
#pragma unroll
    for (int u = 0; u < kDequantUnroll; ++u)
      if (at[u] >= 0) out[at[u]] = dequant8(raw[u], sc[u]);
  }
}

}  // namespace

cudaError_t launch_cache_dequant_fp8(const void* codes_layer, const float* scales_layer,
                                     const int32_t* cu_prefix, int batch, int num_heads,
                                     int64_t capacity, void* out_layer, int32_t* status,
                                     cudaStream_t stream) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // about one wave of 8 CTAs per SM over all heads
  const int per_head = std::max(1, (sms * 8 + num_heads - 1) / num_heads);
  cache_dequant_fp8_kernel<<<dim3(per_head, num_heads), 256, 0, stream>>>(
      static_cast<const uint2*>(codes_layer), scales_layer, cu_prefix, batch, num_heads, capacity,
      static_cast<uint4*>(out_layer), status);
  return cudaGetLastError();
}

}  // namespace bca

// ---------------------------------------------------------------------------
// Gather of a paged cache layer into a packed bf16 buffer (SenseNova-U1 /
// Prism-Infer notes, prefix KV reuse: a prefix hit gathers and dequantises the
// paged K/V in one batch).  Prefix token t of sequence b is read from cache
// token page_table[b][t / 128] * 128 + t % 128 of the [H][capacity][128]
// layer and written to row cu_prefix[b] + t of out [H][out_rows][128]: E4M3
// codes (kFp8) become bf16(fp32(value(code)) * scale), bf16 rows are copied.
namespace bca {
namespace {

template <bool kFp8>
__global__ void __launch_bounds__(256)
    cache_gather_kernel(const void* __restrict__ src, const float* __restrict__ scales,
                        const int32_t* __restrict__ cu_prefix, const int32_t* __restrict__ page_table,
                        int max_pages, int batch, int num_heads, int64_t capacity,
                        uint4* __restrict__ out, int64_t out_rows, int32_t* status) {
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < batch; i += blockDim.x)
    if (cu_prefix[i + 1] < cu_prefix[i] || cu_prefix[i] < 0) s_bad = BCA_ERR_SEQLENS;
  if (threadIdx.x == 0 && static_cast<int64_t>(cu_prefix[batch]) > out_rows)
    s_bad = BCA_ERR_CAPACITY;
  if (check_pages(page_table, max_pages, cu_prefix, batch, capacity) != 0) s_bad = BCA_ERR_CAPACITY;
  __syncthreads();
  if (s_bad != 0) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) report_status(status, s_bad);
    return;
  }
  // a grid of (chunk range, head); 16 chunks of 8 values per row, as in the expansion
  const int hh = blockIdx.y;
  const int p0 = cu_prefix[0];
  const uint32_t chunks = static_cast<uint32_t>(cu_prefix[batch] - p0) * 16u;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < chunks;
       base += stride * kDequantUnroll) {
    int64_t src_at[kDequantUnroll], dst_at[kDequantUnroll];   // -1: none
    uint2 raw8[kDequantUnroll];
    uint4 raw16[kDequantUnroll];
    float sc[kDequantUnroll];
#pragma unroll
    for (int u = 0; u < kDequantUnroll; ++u) {
      const uint32_t ch = base + u * stride;
      dst_at[u] = -1;
      if (ch >= chunks) continue;
      const int c = static_cast<int>(ch >> 4) + p0;   // packed prefix row
      int lo = 0, hi = batch - 1;                       // its sequence
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu_prefix[mid] <= c) lo = mid; else hi = mid - 1;
      }
      const int64_t src_row = static_cast<int64_t>(hh) * capacity +
                              cache_token(page_table, max_pages, cu_prefix, lo, c - cu_prefix[lo]);
      if (!BCA_IN_BOUNDS(status, hh < num_heads && src_row >= 0 &&
                                     src_row < static_cast<int64_t>(num_heads) * capacity &&
                                     c >= 0 && c < out_rows))
        continue;
      const int x = static_cast<int>(ch & 15);
      src_at[u] = src_row * 16 + x;
      dst_at[u] = (static_cast<int64_t>(hh) * out_rows + c) * 16 + x;
      if constexpr (kFp8) {
        raw8[u] = __ldcs(static_cast<const uint2*>(src) + src_at[u]);
        sc[u] = __ldg(scales + src_row);
      } else {
        raw16[u] = __ldcs(static_cast<const uint4*>(src) + src_at[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kDequantUnroll; ++u) {
      if (dst_at[u] < 0) continue;
      if constexpr (kFp8)
        out[dst_at[u]] = dequant8(raw8[u], sc[u]);
      else
        out[dst_at[u]] = raw16[u];
    }
  }
}

}  // namespace

cudaError_t launch_cache_gather(bool fp8, const void* src_layer, const float* scales_layer,
                                const int32_t* cu_prefix, const int32_t* page_table, int max_pages,
                                int batch, int num_heads, int64_t capacity, void* out,
                                int64_t out_rows, int32_t* status, cudaStream_t stream) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const dim3 grid(std::max(1, (sms * 8 + num_heads - 1) / num_heads), num_heads);
  if (fp8)
    cache_gather_kernel<true><<<grid, 256, 0, stream>>>(
        src_layer, scales_layer, cu_prefix, page_table, max_pages, batch, num_heads, capacity,
        static_cast<uint4*>(out), out_rows, status);
  else
    cache_gather_kernel<false><<<grid, 256, 0, stream>>>(
        src_layer, scales_layer, cu_prefix, page_table, max_pages, batch, num_heads, capacity,
        static_cast<uint4*>(out), out_rows, status);
  return cudaGetLastError();
}

}  // namespace bca

// Launchers of the kernels around the attention (cache append, FP8 cache,
// Q/K prologue), defined in their .cu files.  Kept apart from common.cuh so the
// attention kernel's sources change only when the attention kernel does.
#pragma once
#include "common.cuh"

namespace bca {

// page_table (device int32 [batch][max_pages]) or null for the contiguous cache
cudaError_t launch_cache_append(const void* k, const void* v, const int32_t* cu_k,
                                const int32_t* cu_prefix, int batch, int num_heads, int total_k,
                                void* cache_k_layer, void* cache_v_layer, int64_t capacity,
                                const int32_t* page_table, int max_pages, int32_t* status,
                                cudaStream_t stream);
// Rows [0, n_rows) of page src_page copied to page dst_page (every head, K and V).
cudaError_t launch_cache_copy_rows(void* cache_k_layer, void* cache_v_layer, int num_heads,
                                   int64_t capacity, int src_page, int dst_page, int n_rows,
                                   cudaStream_t stream);

cudaError_t launch_cache_append_fp8(const void* k, const void* v, const int32_t* cu_k,
                                    const int32_t* cu_prefix, int batch, int num_heads,
                                    int total_k, bool quant_k, void* cache_k_layer, void* cache_v_layer,
                                    float* scale_k_layer, float* scale_v_layer, int64_t capacity,
                                    const int32_t* page_table, int max_pages, int32_t* status,
                                    cudaStream_t stream);
// Paged layer rows (E4M3 with scales, or bf16) gathered into packed bf16 rows
// cu_prefix[b] + t of out [H][out_rows][128].
cudaError_t launch_cache_gather(bool fp8, const void* src_layer, const float* scales_layer,
                                const int32_t* cu_prefix, const int32_t* page_table, int max_pages,
                                int batch, int num_heads, int64_t capacity, void* out,
                                int64_t out_rows, int32_t* status, cudaStream_t stream);

// E4M3 cache rows cu_prefix[0] .. cu_prefix[batch]-1 of one layer ([H][cap][128]
// codes, [H][cap] scales) expanded to bf16 value * scale, same layout.
cudaError_t launch_cache_dequant_fp8(const void* codes_layer, const float* scales_layer,
                                     const int32_t* cu_prefix, int batch, int num_heads,
                                     int64_t capacity, void* out_layer, int32_t* status,
                                     cudaStream_t stream);

// Three-axis RoPE coordinates [total][3] (frame, height, width) of packed tokens.
cudaError_t launch_rope_positions(const int32_t* block_id, const int32_t* cu_seqlens, int batch,
                                  int total, const int32_t* grid_w, int n_ids, int32_t* pos3,
                                  int32_t* status, cudaStream_t stream);
// (cos, sin) of the 64 dimension pairs per token, float [total][64][2].
cudaError_t launch_rope_table(const int32_t* pos3, int64_t total, float* table,
                              cudaStream_t stream);
// RMS-normalise and rotate Q and K; with cu_prefix, also append K_rot / V of prefix tokens.
cudaError_t launch_qk_norm_rope(const void* q, const void* k, const void* v, const float* gamma_q,
                                const float* gamma_k, const float* table, const int32_t* cu_k,
                                const int32_t* cu_prefix, int batch, int num_heads, int total,
                                float eps, void* q_out, void* k_out, void* cache_k_layer,
                                void* cache_v_layer, int64_t capacity, int32_t* status,
                                cudaStream_t stream);

}  // namespace bca

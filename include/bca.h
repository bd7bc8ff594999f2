/*
 * bca.h -- block-causal attention with a prefix K/V cache, for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libbca_gb300.so.  Every pointer argument marked "device" is a CUDA
 * device pointer owned by the caller; the library never allocates device
 * memory except where an entry point says so.  All calls are asynchronous on
 * the given stream (a cudaStream_t passed as void*; NULL = legacy default
 * stream).  Host-side argument errors return a nonzero status before anything
 * is launched.  Errors that can only be seen on the device (block ids,
 * cu_seqlens contents, cache capacity, a bounded wait that ran out) are
 * written to *status_dev (first error wins) when status_dev is not NULL; read
 * them with bca_read_device_status().  status_dev must be zeroed by the
 * caller before first use; the library only ever writes nonzero codes to it.
 *
 * Tensor conventions (all row-major, contiguous):
 *   q, k, v, out   bf16 [total, H, 128]   token stride H*128 elements
 *   lse            fp32 [H, total_q]      natural log, over scaled scores
 *   cache_k/v      bf16 [num_layers][H][capacity][128]
 *   block_id       int32 [total_k]        -1 = text, >= 0 = image block id
 *   cu_seqlens_*   int32 [batch+1]        packed varlen offsets (device)
 * Device pointers must be 16-byte aligned.  head_dim must be 128.
 *
 * Source of the operations (page title, section):
 *   "Qwen-Image 2.1 deployment notes" (10100.com), "Block-Causal mask" and the
 *   piecewise-attention paragraph; "Qwen-Image 2.1: Block-Causal Attention,
 *   Prefix KV Cache, and Turbo" (flozi.net), sections "Block-causal attention
 *   is the cache-enabling boundary", "Timestep-zero conditioning makes the
 *   prefix invariant", "The prefix cache is a compute-for-memory trade" and
 *   "Two exact attention paths"; SenseNova-U1 inference-infra notes,
 *   "NEO-Unify 多模态 Prefill 的注意力" (per-M-block K-range extension).
 *
 * Beyond the prefill / decode / append path, the same library carries:
 *   - the prefill with the cache append fused in (one launch fewer):
 *     bca_prefill_append, bca_prefill_append_paged;
 *   - an FP8 E4M3 prefix cache with one fp32 scale per (token, head)
 *     (deployment notes, prefix-cache section): bca_prefix_cache_append_fp8,
 *     bca_prefix_cache_dequant_fp8, bca_prefix_decode_fp8;
 *   - the Q/K prologue, per-head RMS norm and three-axis RoPE fused with the
 *     cache append (flozi.net, "Three-axis RoPE preserves image geometry"):
 *     bca_rope_positions, bca_rope_table, bca_qk_norm_rope_append;
 *   - the piecewise prefill baseline (one call per segment):
 *     bca_prefill_piecewise;
 *   - a paged prefix cache with a host page pool (SenseNova-U1 / Prism-Infer
 *     notes, prefix KV reuse): bca_prefix_cache_append_paged,
 *     bca_prefix_decode_paged, their FP8 forms, bca_pool_copy_rows, bca_pool_*.
 */
#ifndef BCA_GB300_H
#define BCA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t bca_status;

enum {
  BCA_OK = 0,
  BCA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, negative size, bad scale      */
  BCA_ERR_UNSUPPORTED = 2,   /* head_dim != 128, more than 1024 image runs in a sequence */
  BCA_ERR_BLOCK_ID = 3,      /* id < -1, one image id split over separate runs, or (RoPE
                                coordinates) an id / image width that does not fit   */
  BCA_ERR_WORKSPACE = 4,     /* workspace NULL, misaligned or smaller than its
                                *_workspace_bytes                                     */
  BCA_ERR_CAPACITY = 5,      /* cache overflow: cu_prefix[batch] > capacity, or a page
                                id outside the pool                                   */
  BCA_ERR_CUDA = 6,          /* a CUDA runtime call failed (launch, attribute, ...)    */
  BCA_ERR_TIMEOUT = 7,       /* a bounded device wait ran out; outputs are undefined   */
  BCA_ERR_SEQLENS = 8,       /* cu_seqlens not monotone, q_len > kv_len, a length above
                                max_seqlen_*, or a cache prefix longer than its keys   */
  BCA_ERR_BOUNDS = 9         /* bounds-checked build only (libbca_gb300_debug.so): a
                                computed index, TMA coordinate or store address fell
                                outside its buffer; the access was skipped            */
};

/* Human-readable name of a status code (static string). */
const char* bca_status_string(bca_status s);

/* Library version, major*10000 + minor*100 + patch. */
int32_t bca_version(void);

/* Copies *status_dev to the host after synchronising `stream`; returns it
 * (BCA_ERR_CUDA if the copy itself failed). */
bca_status bca_read_device_status(const int32_t* status_dev, void* stream);

/* Self-test of the bounded device waits (no counterpart on the pages).  Launches
 * one CTA whose threads wait on an mbarrier that is never completed: one warp
 * with limit_ns (1 ns .. 1 s), the others with 50x that limit.  The first
 * gives up after limit_ns and writes BCA_ERR_TIMEOUT to *status_dev; the
 * others must see its abort flag and return at once, so the kernel ends after
 * about limit_ns.  If elapsed_ns_dev is not NULL the device-measured duration
 * (ns) is written there.  Faults nothing; the context stays usable. */
bca_status bca_selftest_wait_timeout(uint64_t limit_ns, int32_t* status_dev,
                                     uint64_t* elapsed_ns_dev, void* stream);

/* ------------------------------------------------------------------------ */
/* Schedule preparation (the O(S) replacement of the O(S^2) mask).
 *
 * For every query row r of sequence b (q_len = cu_q[b+1]-cu_q[b], kv_len =
 * cu_k[b+1]-cu_k[b], position p = kv_len - q_len + i: bottom-right alignment)
 * the visible keys are exactly [0, e(r)), e(r) = p+1 for a text row and the
 * exclusive end of p's image run for an image row ("an image block [a,b) sees
 * everything before it plus its own block", 10100.com, "Block-Causal mask").
 * Validates that every id >= 0 forms one contiguous run per sequence (at most
 * 1024 image runs per sequence; more gives BCA_ERR_UNSUPPORTED).
 *
 *   row_end  device int32 [total_q]  out: e(r), relative to the sequence's first key
 *   tiles    device int32 [batch * tiles_per_seq * 4] out, tiles_per_seq =
 *            ceil(max_seqlen_q / 128); record (b, m) = {k_hi = max e over
 *            the tile's valid rows, k_min = min e, valid rows, 0}; all zero
 *            for a tile past the sequence end or a sequence that failed
 *            validation.
 *   total_q, total_k  lengths of the packed query rows and keys (row_end and
 *            block_id hold that many entries).  A sequence with cu_q[b] < 0,
 *            cu_k[b] < 0, cu_q[b+1] > total_q or cu_k[b+1] > total_k fails with
 *            BCA_ERR_SEQLENS in *status_dev before any of its row ends is
 *            written or any of its block ids is read.
 */
bca_status bca_schedule_prep(const int32_t* block_id, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_k, int32_t batch, int32_t total_q,
                             int32_t total_k, int32_t max_seqlen_q, int32_t* row_end,
                             int32_t* tiles, int32_t* status_dev, void* stream);

/* Bytes of device workspace bca_prefill needs (row_end + tile records). */
size_t bca_prefill_workspace_bytes(int32_t batch, int32_t total_q, int32_t max_seqlen_q);

/* ------------------------------------------------------------------------ */
/* Block-causal multi-head attention forward over packed varlen sequences.
 *
 * visible(i, j) = (p_i >= j) or (bid[p_i] >= 0 and bid[p_i] == bid[j]) with
 * p_i = kv_len - q_len + i (10100.com "Block-Causal mask"; flozi.net
 * "Block-causal attention is the cache-enabling boundary"; bottom-right
 * alignment from 10100.com's piecewise-attention paragraph).
 *   out[r, h, :] = sum_j softmax_j(scale * q_r . k_j | visible) v_j      (bf16)
 *   lse[h, r]    = ln sum_j exp(scale * q_r . k_j | visible)             (fp32)
 * q: device bf16 [total_q, H, 128]; k, v: device bf16 [total_k, H, 128];
 * block_id: device int32 [total_k]; cu_seqlens_q/k: device int32 [batch+1];
 * out: device bf16 [total_q, H, 128]; lse: device fp32 [H, total_q];
 * workspace: device, >= bca_prefill_workspace_bytes(batch, total_q, max_seqlen_q).
 * A sequence that fails validation gets no output (its rows are left as they were).
 * Launches two or three kernels on `stream`: the schedule prep; the query-tile
 * pairs, which may start while the prep runs (programmatic dependent launch) and
 * read its records only once it has completed; and, for a pair grid of at most
 * four waves past two whole ones, the pairs of its last, partly filled wave as
 * key-split single tiles in a third grid that may start as the pairs drain.
 */
bca_status bca_prefill(const void* q, const void* k, const void* v, const int32_t* block_id,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                       int32_t batch, int32_t num_heads, int32_t head_dim,
                       int32_t total_q, int32_t total_k, int32_t max_seqlen_q,
                       int32_t max_seqlen_k, float softmax_scale, void* out, float* lse,
                       void* workspace, size_t workspace_bytes, int32_t* status_dev,
                       void* stream);

/* Prefill with the prefix cache append fused in: bca_prefill, and the cache
 * rows bca_prefix_cache_append would write (same arguments and layout:
 * cu_prefix device int32 [batch+1], cache_k/v device bf16
 * [num_layers][H][capacity][128], layer `layer`), written from the key and
 * value tiles the attention already reads (flozi.net "Timestep-zero
 * conditioning makes the prefix invariant": the first step clones the
 * post-RoPE prefix K/V into the cache).  One launch fewer than the two calls.
 * Errors as in the two calls: nothing is written to the cache when a prefix is
 * longer than its keys or a sequence with a prefix has no query rows
 * (BCA_ERR_SEQLENS), or cu_prefix[batch] > capacity (BCA_ERR_CAPACITY); a
 * sequence that fails block-id validation gets neither output nor cache rows.
 * With batch == 0 or total_q == 0 nothing is launched and nothing is written.
 */
bca_status bca_prefill_append(const void* q, const void* k, const void* v,
                              const int32_t* block_id, const int32_t* cu_seqlens_q,
                              const int32_t* cu_seqlens_k, int32_t batch, int32_t num_heads,
                              int32_t head_dim, int32_t total_q, int32_t total_k,
                              int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                              void* out, float* lse, void* workspace, size_t workspace_bytes,
                              const int32_t* cu_prefix, void* cache_k, void* cache_v,
                              int32_t layer, int32_t num_layers, int64_t capacity,
                              int32_t* status_dev, void* stream);

/* bca_prefill_append over a paged cache: the rows bca_prefix_cache_append_paged
 * would write (prefix token t of sequence b to cache token
 * page_table[b * max_pages + t / 128] * 128 + t % 128 of a pool of num_pages
 * 128-token pages per layer and head, cache_k/v device bf16
 * [num_layers][H][num_pages * 128][128]; page_table device int32).  Nothing is
 * written when a prefix needs more than max_pages pages or a page id lies
 * outside [0, num_pages) (BCA_ERR_CAPACITY), or on the errors of
 * bca_prefill_append.
 */
bca_status bca_prefill_append_paged(const void* q, const void* k, const void* v,
                                    const int32_t* block_id, const int32_t* cu_seqlens_q,
                                    const int32_t* cu_seqlens_k, int32_t batch, int32_t num_heads,
                                    int32_t head_dim, int32_t total_q, int32_t total_k,
                                    int32_t max_seqlen_q, int32_t max_seqlen_k,
                                    float softmax_scale, void* out, float* lse, void* workspace,
                                    size_t workspace_bytes, const int32_t* cu_prefix,
                                    const int32_t* page_table, int32_t max_pages, void* cache_k,
                                    void* cache_v, int32_t layer, int32_t num_layers,
                                    int32_t num_pages, int32_t* status_dev, void* stream);

/* Same computation as bca_prefill, for callers that cannot allocate device
 * memory or pass a workspace: for example a plugin inside a runtime that owns
 * all GPU memory in a pre-planned arena, or a loop that must not take
 * cudaMalloc's implicit synchronisation.  The pages have no counterpart of
 * this call; it only changes where the schedule scratch lives.
 *
 * The scratch is a fixed 2 MiB array in the library's own device memory, held
 * by every GPU that loads the library until the process exits.  Problems with
 * total_q > 262144 or batch * ceil(max_seqlen_q / 128) > 65536 are rejected
 * with BCA_ERR_WORKSPACE.  Every call looks up the array's device address on
 * the current device (cudaGetSymbolAddress; the first lookup on a device loads
 * the library's module there, so make the first call before any stream
 * capture).  Since the address is not cached, calls after a device reset or a
 * re-created primary context use the array's new location.  The call
 * allocates nothing.  All
 * calls share the array: calls whose kernels may overlap on the GPU (other
 * streams or host threads) race and must be serialised by the caller.
 * Arguments, layouts and errors are otherwise those of bca_prefill.
 */
bca_status bca_prefill_noalloc(const void* q, const void* k, const void* v,
                               const int32_t* block_id, const int32_t* cu_seqlens_q,
                               const int32_t* cu_seqlens_k, int32_t batch, int32_t num_heads,
                               int32_t head_dim, int32_t total_q, int32_t total_k,
                               int32_t max_seqlen_q, int32_t max_seqlen_k, float softmax_scale,
                               void* out, float* lse, int32_t* status_dev, void* stream);

/* Block-causal prefill as one exact attention call per segment, a baseline
 * for bca_prefill (Qwen-Image 2.1 deployment notes, piecewise-attention
 * paragraph; flozi.net "Two exact attention paths": the default diffusers
 * processor runs one call for every text or image segment of the prefix and
 * one for the target).  Segment [a, e) of sequence b (a maximal run of one
 * block id) is computed as its own problem: queries [a, e) over keys
 * [cu[b], e), a text segment causal over itself (bottom-right aligned), an
 * image segment unmasked; the results equal bca_prefill's.  Square sequences
 * only (the same cu_seqlens for q and k).  block_id: device int32 [total];
 * block_id_host / cu_seqlens_host: the same ids and offsets in host memory
 * (the segment table is built on the host).  q, k, v, out, lse as in
 * bca_prefill.  workspace: device memory of
 * bca_prefill_piecewise_workspace_bytes (16-byte aligned), reused by the
 * pieces in stream order.  Launches two or three kernels (as bca_prefill) and one
 * 2-D copy per segment. */
size_t bca_prefill_piecewise_workspace_bytes(const int32_t* block_id_host,
                                             const int32_t* cu_seqlens_host, int32_t batch,
                                             int32_t num_heads);
bca_status bca_prefill_piecewise(const void* q, const void* k, const void* v,
                                 const int32_t* block_id, const int32_t* block_id_host,
                                 const int32_t* cu_seqlens_host, int32_t batch, int32_t num_heads,
                                 int32_t head_dim, int32_t total, float softmax_scale, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 int32_t* status_dev, void* stream);

/* ------------------------------------------------------------------------ */
/* Prefix-cache "decode" (cached denoising steps): the target queries of every
 * sequence attend, with no mask, over [cached prefix K/V; their own K/V]
 * (flozi.net "Timestep-zero conditioning makes the prefix invariant": later
 * steps concatenate cached prefix K/V with fresh target K/V; "Two exact
 * attention paths": cached steps need no block-causal mask).
 *
 * q_tgt, k_tgt, v_tgt: device bf16 [total_q, H, 128] packed by cu_seqlens_q;
 * cache_k/v: device bf16 [num_layers][H][capacity][128]; sequence b's prefix
 * is cache tokens cu_prefix[b] .. cu_prefix[b+1]-1 of layer `layer`;
 * cu_prefix: device int32 [batch+1]; out/lse as in bca_prefill.
 * max_seqlen_q bounds every target length and max_prefix every prefix length
 * cu_prefix[b+1]-cu_prefix[b]; with the balanced tail below, a sequence whose
 * prefix and target tiles outnumber those of max_prefix and max_seqlen_q is
 * reported as BCA_ERR_SEQLENS.
 *
 * The query-tile pairs of all (sequence, head) run as one grid.  The pairs of a
 * last, partly filled wave run in a second grid that may start as the first
 * drains, in one of two ways:
 *  - workspace given (device memory of at least
 *    bca_prefix_decode_workspace_bytes, 16-byte aligned, else BCA_ERR_WORKSPACE):
 *    the balanced tail.  Those pairs' key tiles are cut into one equal range
 *    per SM; every piece leaves partial rows (unnormalised fp32 O, row max and
 *    row sum) in the workspace, and a third, small grid merges each pair's
 *    pieces into out and lse.  The workspace is scratch, free again once the
 *    stream passes the call; nothing in it needs initialising.
 *  - workspace NULL: when the wave would be at most half full, its pairs run
 *    as key-split single tiles (each tile's keys shared out between the two
 *    softmax warpgroups of one CTA), otherwise as plain pairs.
 * Both give the attention of the pages within the same tolerance; they round
 * differently, so their outputs are not bit-identical.
 */
bca_status bca_prefix_decode(const void* q_tgt, const void* cache_k, const void* cache_v,
                             int32_t layer, int32_t num_layers, int64_t capacity,
                             const int32_t* cu_prefix, const void* k_tgt, const void* v_tgt,
                             const int32_t* cu_seqlens_q, int32_t batch, int32_t num_heads,
                             int32_t head_dim, int32_t total_q, int32_t max_seqlen_q,
                             int32_t max_prefix, float softmax_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, int32_t* status_dev,
                             void* stream);

/* Workspace bytes that give the decodes (bca_prefix_decode and its paged and
 * FP8 forms) the balanced tail on the current device: two partial slots of
 * 133,120 bytes per SM when (batch, heads, max_seqlen_q, max_prefix) leave a
 * last, partly filled wave of query-tile pairs that is worth balancing; 0 when
 * they do not (the decode then needs no workspace) or the arguments are
 * invalid. */
size_t bca_prefix_decode_workspace_bytes(int32_t batch, int32_t num_heads, int32_t head_dim,
                                         int32_t max_seqlen_q, int32_t max_prefix);

/* ------------------------------------------------------------------------ */
/* Prefix cache append (the "extract" step): clone the first
 * cu_prefix[b+1]-cu_prefix[b] keys and values of every sequence b into cache
 * tokens cu_prefix[b].. of layer `layer` (flozi.net "Timestep-zero
 * conditioning makes the prefix invariant": the cache stores post-RoPE prefix
 * K/V per layer as a clone of the slices, not a view; "The prefix cache is a
 * compute-for-memory trade": two tensors per layer, H heads x 128 values).
 * k, v: device bf16 [total_k, H, 128] packed by cu_seqlens_k; cache_k/v:
 * device bf16 [num_layers][H][capacity][128].  Nothing is written when
 * cu_prefix[batch] > capacity (BCA_ERR_CAPACITY), or a prefix is longer than
 * its sequence or its source keys run past total_k (BCA_ERR_SEQLENS).
 */
bca_status bca_prefix_cache_append(const void* k, const void* v, const int32_t* cu_seqlens_k,
                                   const int32_t* cu_prefix, int32_t batch, int32_t num_heads,
                                   int32_t head_dim, int32_t total_k, void* cache_k,
                                   void* cache_v, int32_t layer, int32_t num_layers,
                                   int64_t capacity, int32_t* status_dev, void* stream);

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 prefix cache ("Qwen-Image 2.1 deployment notes", prefix-cache
 * section: the prefix cache is stored as FP8 E4M3 with one FP32 scale per token
 * and attention head, quantising K and V, or V only).  Each (token, head) row
 * of 128 values is scaled by its absolute maximum onto the E4M3 range, in fp32:
 *   scale = amax / 448;  code = E4M3(x * (448 / amax)), round to nearest even,
 *   saturating at +-448 (an all-zero row gets scale 0 and zero codes);
 * a dequantised value is bf16(fp32(value(code)) * scale).
 *   BCA_FP8_V : cache_k is bf16 [L][H][cap][128] (copied as in
 *               bca_prefix_cache_append), cache_v holds E4M3 codes
 *               uint8 [L][H][cap][128], scale_v fp32 [L][H][cap]; scale_k unused.
 *   BCA_FP8_KV: cache_k and cache_v hold E4M3 codes, scale_k and scale_v fp32.
 * Addressing, validation and errors are those of bca_prefix_cache_append; a layer
 * of H x capacity >= 2^31 rows is BCA_ERR_UNSUPPORTED. */
enum { BCA_FP8_V = 1, BCA_FP8_KV = 2 };

bca_status bca_prefix_cache_append_fp8(const void* k, const void* v, const int32_t* cu_seqlens_k,
                                       const int32_t* cu_prefix, int32_t batch, int32_t num_heads,
                                       int32_t head_dim, int32_t total_k, int32_t mode,
                                       void* cache_k, void* cache_v, float* scale_k,
                                       float* scale_v, int32_t layer, int32_t num_layers,
                                       int64_t capacity, int32_t* status_dev, void* stream);

/* Expansion of one layer of an E4M3 cache back to bf16: for the rows
 * cu_prefix[0] .. cu_prefix[batch]-1 of every head, out[h][t][d] =
 * bf16(fp32(value(codes[layer][h][t][d])) * scales[layer][h][t]), the
 * dequantised value defined above, rounded to nearest even.
 * codes: device uint8 [num_layers][H][capacity][128]; scales: device fp32
 * [num_layers][H][capacity]; out: device bf16 [H][capacity][128] for the one
 * layer (rows outside the range are not written).  cu_prefix: device int32
 * [batch+1].  When cu_prefix[batch] > capacity (BCA_ERR_CAPACITY) or the range
 * is negative (BCA_ERR_SEQLENS) nothing is written.  Pointers 16-byte aligned
 * (scales 4-byte).  More than 65535 heads or a capacity of 2^28 tokens or more
 * is BCA_ERR_UNSUPPORTED. */
bca_status bca_prefix_cache_dequant_fp8(const void* codes, const float* scales,
                                        const int32_t* cu_prefix, int32_t batch,
                                        int32_t num_heads, int32_t head_dim, int32_t layer,
                                        int32_t num_layers, int64_t capacity, void* out,
                                        int32_t* status_dev, void* stream);

/* Workspace bytes bca_prefix_decode_fp8 needs: one bf16 layer [H][capacity][128]
 * (256-byte rounded) per quantised tensor, i.e. one for BCA_FP8_V and two for
 * BCA_FP8_KV; 0 for invalid arguments. */
size_t bca_prefix_decode_fp8_workspace_bytes(int32_t mode, int32_t num_heads, int32_t head_dim,
                                             int64_t capacity);

/* Prefix-cache decode over an FP8 E4M3 cache written by
 * bca_prefix_cache_append_fp8 in the same mode ("Qwen-Image 2.1 deployment
 * notes", prefix-cache section).  Every cached key/value element enters the
 * attention as its dequantised value bf16(fp32(value(code)) * scale); target
 * K/V stay bf16.  The quantised tensors of the layer are first expanded
 * (bca_prefix_cache_dequant_fp8) into `workspace`, device memory of at least
 * bca_prefix_decode_fp8_workspace_bytes (16-byte aligned, else
 * BCA_ERR_WORKSPACE), then attended exactly as by bca_prefix_decode; the
 * workspace is scratch, free again once the stream passes the call.  When the
 * workspace holds bca_prefix_decode_workspace_bytes more bytes after those, the
 * decode uses them for its balanced tail (else its key-split tail).  mode,
 * cache_k, cache_v, scale_k and scale_v are laid out as in
 * bca_prefix_cache_append_fp8 (scale_k is not read in BCA_FP8_V mode).  All
 * other arguments, layouts and errors are those of bca_prefix_decode; an
 * unknown mode is BCA_ERR_INVALID_ARG. */
bca_status bca_prefix_decode_fp8(const void* q_tgt, const void* cache_k, const void* cache_v,
                                 int32_t mode, const float* scale_k, const float* scale_v,
                                 int32_t layer, int32_t num_layers, int64_t capacity,
                                 const int32_t* cu_prefix, const void* k_tgt, const void* v_tgt,
                                 const int32_t* cu_seqlens_q, int32_t batch, int32_t num_heads,
                                 int32_t head_dim, int32_t total_q, int32_t max_seqlen_q,
                                 int32_t max_prefix, float softmax_scale, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, int32_t* status_dev,
                                 void* stream);

/* ------------------------------------------------------------------------ */
/* Q/K prologue: per-head RMS normalisation, three-axis RoPE and the append of
 * the rotated prefix keys ("Qwen-Image 2.1: Block-Causal Attention, Prefix KV
 * Cache, and Turbo", flozi.net: Q and K are RMS-normalised per head before
 * RoPE; "Three-axis RoPE preserves image geometry": head dimensions split
 * (16, 56, 56) across frame, height and width, base 10000; "Timestep-zero
 * conditioning makes the prefix invariant": the cache holds post-RoPE K). */

/* Coordinates of every packed token, pos3: device int32 [total][3] = (frame,
 * height, width).  Per sequence a running coordinate c starts at 0; a text
 * token (block id -1) takes (c, c, c) and advances c by one; an image block
 * (one contiguous run of a non-negative id i) of n tokens with width
 * w = grid_w[b * n_ids + i] (n a multiple of w, height n / w, tokens row-major)
 * takes frame c and (row - height/2, column - width/2), then advances c by one.
 * block_id: device int32 [total]; cu_seqlens: device int32 [batch+1]; grid_w:
 * device int32 [batch][n_ids] (n_ids <= 4096, else BCA_ERR_UNSUPPORTED).  A
 * sequence with an id >= n_ids or < -1, an id in two runs, or a block whose
 * length is not a multiple of its width is reported as BCA_ERR_BLOCK_ID and
 * its coordinates are not written; so is (as BCA_ERR_SEQLENS) a sequence whose
 * tokens [cu_seqlens[b], cu_seqlens[b+1]) do not lie in [0, total). */
bca_status bca_rope_positions(const int32_t* block_id, const int32_t* cu_seqlens, int32_t batch,
                              int32_t total, const int32_t* grid_w, int32_t n_ids,
                              int32_t* pos3, int32_t* status_dev, void* stream);

/* Rotation table: table[t][j] = (cos, sin) of the angle of dimension pair j of
 * token t, fp32 [total][64][2] (16-byte aligned).  Pair j < 8 is frame pair
 * k = j, j < 36 height pair k = j - 8, else width pair k = j - 36; the angle is
 * coordinate * 10000^(-2k/d) with d = 16, 56, 56; computed in double. */
bca_status bca_rope_table(const int32_t* pos3, int32_t total, float* table, void* stream);

/* For every (token, head) row of q and k (device bf16 [total][H][128]):
 *   y = x / sqrt(mean(x^2) + eps) * gamma        (fp32; gamma = 1 when null)
 *   pair (y[2j], y[2j+1]) -> (y0 cos - y1 sin, y0 sin + y1 cos) by rope_table row t
 * written as bf16 to q_out / k_out (which may be q / k: in place is allowed).
 * gamma_q, gamma_k: device fp32 [128] (16-byte aligned) or null.  When cu_prefix (device int32
 * [batch+1]) is not null, the rotated keys and the values (v, device bf16
 * [total][H][128]) of the first cu_prefix[b+1]-cu_prefix[b] tokens of each
 * sequence are also written to cache tokens cu_prefix[b].. of layer `layer` of
 * cache_k / cache_v (bf16 [num_layers][H][capacity][128]); the cache K row is
 * bit-identical to the k_out row.  Validation and errors of the cache write are
 * those of bca_prefix_cache_append (nothing is written when they fail); with a
 * null cu_prefix, v and the cache arguments are not read. */
bca_status bca_qk_norm_rope_append(const void* q, const void* k, const void* v,
                                   const float* gamma_q, const float* gamma_k,
                                   const float* rope_table, const int32_t* cu_seqlens,
                                   const int32_t* cu_prefix, int32_t batch, int32_t num_heads,
                                   int32_t head_dim, int32_t total, float eps, void* q_out,
                                   void* k_out, void* cache_k, void* cache_v, int32_t layer,
                                   int32_t num_layers, int64_t capacity, int32_t* status_dev,
                                   void* stream);

/* ------------------------------------------------------------------------ */
/* Paged prefix cache (SenseNova-U1 / Prism-Infer notes, prefix KV reuse: the
 * cache is a pool of pages that requests with a common prefix share).  A page
 * holds 128 consecutive prefix tokens of one sequence for every head of a
 * layer: one layer of the pool is a bf16 cache [H][num_pages * 128][128], and
 * prefix token t of sequence b lives at token page_table[b * max_pages +
 * t / 128] * 128 + t % 128 (cache layout [num_layers][H][num_pages*128][128]).
 * cu_prefix (device int32 [batch+1]) gives only the prefix lengths here.  A
 * page entry outside [0, num_pages), or a prefix needing more than max_pages
 * pages, is reported as BCA_ERR_CAPACITY on the status word and nothing of
 * that call (append) or that sequence (decode) is written.  num_pages <= 2^24. */

/* bca_prefix_cache_append through a page table. */
bca_status bca_prefix_cache_append_paged(const void* k, const void* v,
                                         const int32_t* cu_seqlens_k, const int32_t* cu_prefix,
                                         const int32_t* page_table, int32_t max_pages,
                                         int32_t batch, int32_t num_heads, int32_t head_dim,
                                         int32_t total_k, void* cache_k, void* cache_v,
                                         int32_t layer, int32_t num_layers, int32_t num_pages,
                                         int32_t* status_dev, void* stream);

/* bca_prefix_decode with the prefix read through a page table (workspace as
 * there: NULL, or bca_prefix_decode_workspace_bytes for the balanced tail). */
bca_status bca_prefix_decode_paged(const void* q_tgt, const void* cache_k, const void* cache_v,
                                   int32_t layer, int32_t num_layers, int32_t num_pages,
                                   const int32_t* cu_prefix, const int32_t* page_table,
                                   int32_t max_pages, const void* k_tgt, const void* v_tgt,
                                   const int32_t* cu_seqlens_q, int32_t batch, int32_t num_heads,
                                   int32_t head_dim, int32_t total_q, int32_t max_seqlen_q,
                                   int32_t max_prefix, float softmax_scale, void* out, float* lse,
                                   void* workspace, size_t workspace_bytes, int32_t* status_dev,
                                   void* stream);

/* bca_prefix_cache_append_fp8 into a paged cache: codes and scales of prefix
 * token t of sequence b go to page token page_table[b * max_pages + t / 128] *
 * 128 + t % 128 of layer `layer` (codes [L][H][num_pages*128][128], scales
 * [L][H][num_pages*128]; in BCA_FP8_V mode cache_k is the bf16 paged cache). */
bca_status bca_prefix_cache_append_fp8_paged(
    const void* k, const void* v, const int32_t* cu_seqlens_k, const int32_t* cu_prefix,
    const int32_t* page_table, int32_t max_pages, int32_t batch, int32_t num_heads,
    int32_t head_dim, int32_t total_k, int32_t mode, void* cache_k, void* cache_v,
    float* scale_k, float* scale_v, int32_t layer, int32_t num_layers, int32_t num_pages,
    int32_t* status_dev, void* stream);

/* Workspace bytes of bca_prefix_decode_fp8_paged: two bf16 buffers
 * [H][prefix_rows][128] (256-byte rounded); 0 for invalid arguments. */
size_t bca_prefix_decode_fp8_paged_workspace_bytes(int32_t num_heads, int32_t head_dim,
                                                   int64_t prefix_rows);

/* Prefix decode over a paged FP8 cache.  The prefixes are first gathered through
 * the page table into the workspace, packed by cu_prefix (rows
 * cu_prefix[b] .. cu_prefix[b+1]-1 of [H][prefix_rows][128]): E4M3 tensors are
 * dequantised to bf16(fp32(value(code)) * scale), a bf16 K (BCA_FP8_V mode) is
 * copied.  Then the contiguous bf16 decode runs on the gathered rows.
 * prefix_rows >= cu_prefix[batch] bounds the gathered rows (a larger
 * cu_prefix[batch] is BCA_ERR_CAPACITY on the status word; prefix_rows >= 2^28
 * is BCA_ERR_UNSUPPORTED).  Workspace bytes
 * beyond bca_prefix_decode_fp8_paged_workspace_bytes serve the balanced tail as
 * in bca_prefix_decode_fp8.  Other arguments as in bca_prefix_decode_paged and
 * bca_prefix_decode_fp8. */
bca_status bca_prefix_decode_fp8_paged(
    const void* q_tgt, const void* cache_k, const void* cache_v, int32_t mode,
    const float* scale_k, const float* scale_v, int32_t layer, int32_t num_layers,
    int32_t num_pages, const int32_t* cu_prefix, const int32_t* page_table, int32_t max_pages,
    int64_t prefix_rows, const void* k_tgt, const void* v_tgt, const int32_t* cu_seqlens_q,
    int32_t batch, int32_t num_heads, int32_t head_dim, int32_t total_q, int32_t max_seqlen_q,
    int32_t max_prefix, float softmax_scale, void* out, float* lse, void* workspace,
    size_t workspace_bytes, int32_t* status_dev, void* stream);

/* Copy rows [0, n_rows) (n_rows <= 128) of page src_page to page dst_page, all
 * heads, K and V, of one layer: the copy of a shared tail page's common rows
 * into a page of its own. */
bca_status bca_pool_copy_rows(void* cache_k, void* cache_v, int32_t layer, int32_t num_layers,
                              int32_t num_heads, int32_t num_pages, int32_t src_page,
                              int32_t dst_page, int32_t n_rows, void* stream);

/* Host-side page pool (page ids only; thread-safe).  Rules kept (same notes):
 * a page joins the hit index only when its owner publishes it after the K/V
 * write completed; a page from bca_pool_alloc is unpublished, so a copied tail
 * page does not inherit the old entry's hash; idle cached pages (published,
 * no references) are lent to allocations, least recently released first, but
 * a referenced page is never reclaimed; capacity counts physical pages. */
typedef struct bca_page_pool bca_page_pool;
/* A pool of num_pages pages, all free; null for num_pages <= 0. */
bca_page_pool* bca_pool_create(int32_t num_pages);
void bca_pool_destroy(bca_page_pool* pool);
/* n pages with one reference each into pages_out: free pages first, then idle
 * cached pages (which leave the index).  BCA_ERR_CAPACITY, and nothing taken,
 * when fewer than n are free or idle. */
bca_status bca_pool_alloc(bca_page_pool* pool, int32_t n, int32_t* pages_out);
/* The longest run hashes[0..h) of published pages; each gains a reference and
 * its id goes to pages_out[i].  Returns h. */
int32_t bca_pool_match(bca_page_pool* pool, const uint64_t* hashes, int32_t n,
                       int32_t* pages_out);
/* Put a referenced, unpublished page into the index under `hash` (unique);
 * BCA_ERR_INVALID_ARG otherwise. */
bca_status bca_pool_publish(bca_page_pool* pool, int32_t page, uint64_t hash);
/* Drop one reference per listed page (a page may be listed more than once).
 * An unreferenced published page stays cached (idle); an unpublished one is
 * freed.  BCA_ERR_INVALID_ARG, and nothing changed, for a bad id or a drop
 * below zero. */
bca_status bca_pool_release(bca_page_pool* pool, const int32_t* pages, int32_t n);
/* Unique physical pages that are free, idle cached, and referenced. */
void bca_pool_stats(bca_page_pool* pool, int32_t* free_pages, int32_t* idle_cached,
                    int32_t* in_use);
/* References held on a page (-1 for a bad id). */
int32_t bca_pool_refs(bca_page_pool* pool, int32_t page);

#ifdef __cplusplus
}
#endif
#endif /* BCA_GB300_H */

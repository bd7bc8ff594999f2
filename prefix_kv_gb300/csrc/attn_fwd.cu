// Block-causal attention forward (prefill) and prefix-cache decode for sm_103a.
//
// One CTA computes one work item: head h and two consecutive 128-row query
// tiles (Q0, Q1) of sequence b, which share every K/V tile they both need.
// For each 128-key tile j of the item's K range:
//   S_i  = Q_i K_j^T                      tcgen05.mma, bf16 smem x smem -> fp32 TMEM
//   P_i  = exp2(S_i * scale*log2e - m_i)  softmax warpgroup i, one TMEM lane (row) per thread
//   O_i += P_i V_j                        tcgen05.mma, P_i read from TMEM, V_j from smem
// The MMA warp issues PV0(j), S0(j+1), PV1(j), S1(j+1), ... so that while one
// softmax warpgroup turns S into P the tensor core runs the other tile's MMAs.
// Because S_i(j+1) is issued after PV_i(j), the commit that signals S_i(j+1)
// also covers PV_i(j): the softmax may rescale O_i right after seeing S_i(j+1).
// The pairs of a short prefill grid's last, partly filled wave (and, when the
// caller gives no workspace, decode pairs that would fill less than half of a
// last wave) run in a second grid as single query tiles whose key range is
// split in two: warpgroup i runs the same loop over its part with its own K/V
// tiles, and warpgroup 0 merges the two partial rows, each against its own
// reference max, at the end.  Such an item takes ~0.6 of a pair's time, where
// a single tile on one warpgroup would take 0.7.
// With a workspace, the decode pairs of a last, partly filled wave are instead
// cut into as many equal key ranges as there are SMs (a range may end inside
// one pair and go on in the next; then it is two pieces).  Every piece runs as
// a pair item over its key tiles and leaves its unnormalised rows, reference
// max and row sum in the workspace; a merge grid combines the pieces of each
// pair.  The longer pieces launch first and the shorter ones after them,
// longest first.
// The reference max is taken exactly on the first K tile; afterwards P is
// formed against it directly and the max is only recomputed (with O and l
// rescaled) for a tile whose row sum would exceed 2^16.  O and l share the
// reference, so out = O / l is exact, and most tiles take no max at all.
//
// The K range of a prefill tile is [0, k_hi) where k_hi is the largest
// visible-key end e(r) of the tile's rows: a text row sees [0, p+1), an image
// row the keys up to the end of its image run (10100.com, "Block-Causal mask";
// per-M-block K-range extension as in the SenseNova-U1 notes, "NEO-Unify 多模态
// Prefill 的注意力").  Tiles entirely below min e(r) are mask-free; only the
// boundary tiles evaluate `key < e(r)`.  Decode reads the cached prefix tiles
// through one tensor map and the target tiles through another, and masks only
// the ragged end of each ("Two exact attention paths": cached steps need no
// block-causal mask).  Prefix tile j of sequence b starts at cache token
// cu_prefix[b] + 128 j, or with a page table at page_table[b][j] * 128 (a
// 128-token page is one tile).  The last softmax warpgroup to read S(j) hands
// the ring stages of V(j-1) and K(j) back to the producer (in a key-split item
// each warpgroup hands back its own).
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3  softmax + epilogue of Q0 (thread t owns TMEM lane t = query row t)
//   warps 4-7  softmax + epilogue of Q1
//   warp 8     TMEM allocator and MMA issuer
//   warp 9     TMA producer (Q0, Q1 once, then K_j, V_j into a ring of smem stages)
//   warp 10    V tail fix-up (zeroes V rows past the end of a key segment)
//   warp 11    prefix store (prefill with cache append: the CTA of each sequence's
//              last tile pair writes the prefix K/V tiles to the cache), else idle
// Launched at 168 registers per thread; the softmax warpgroups raise theirs to
// 208 and the control warpgroup drops to 88 (2*128*208 + 128*88 = 384*168).
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512); P_i is
// written over the first 64 columns of S_i once S_i has been read.
#include "common.cuh"
#include "ptx.cuh"

#include <cudaTypedefs.h>
#include <algorithm>
#include <mutex>

namespace bca {
namespace {

constexpr int kStages = 5;
constexpr int kTileBytes = kBlockN * kHeadDim * 2;  // 32 KB: 128 rows x 256 B
constexpr int kHalfBytes = kTileBytes / 2;          // one 64-column (128 B) half
constexpr int kThreads = 384;
constexpr int kRegsLaunch = 168, kRegsSoftmax = 208, kRegsControl = 88;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsControl == kThreads * kRegsLaunch, "register split");
constexpr int kWarpMma = 8;
constexpr int kWarpTma = 9;
constexpr int kWarpFix = 10;
constexpr int kWarpStore = 11;   // prefill with cache append: stores the prefix tiles
// Prefill kernels: one instance with the cache append into a contiguous cache when
// cache_k is set (or none), one with it through a page table.  (Three instances, one
// without any append code, measured 1.4% slower for the plain prefill: ptxas lays the
// shared code out differently.)
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;
constexpr float kSumLimit = 65536.0f;  // largest accepted tile row sum relative to m_ref

struct FwdSmem {
  uint8_t q[2][kTileBytes];
  uint8_t kv[kStages][kTileBytes];
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_final[2];
  uint64_t fix_req;     // MMA thread saw a tail V tile land: fix-up warp may zero it
  uint64_t v_fixed;     // fix-up warp zeroed the tail rows of that V tile
  uint64_t drain;
  uint64_t merge;       // key split: warpgroup 1 published its row maxima and sums
  uint64_t epi[2];      // query tile i's output rows are staged in q[i] for the TMA store
  uint32_t tmem_base;
  int abort;
  int fix_stage;        // the V tile to fix: its ring stage and first row past the segment
  int fix_from;
};
constexpr size_t kSmemBytes = sizeof(FwdSmem) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct FwdParams {
  int num_heads;
  int total_q;
  int total_k;                // prefill: rows of k and v
  int tiles_per_seq;
  float scale_log2;
  int64_t capacity;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* row_end;
  const PrefillTile* tiles;
  const int32_t* cu_prefix;
  const int32_t* page_table;  // decode, paged cache: page of prefix tile j of sequence b
  int max_pages;              //   at page_table[b * max_pages + j]; null: contiguous
  int head_groups;            // prefill: grid z = sequence * head_groups + group
  int batch;
  __nv_bfloat16* cache_k;     // prefill with cache append: one layer [H][capacity][128], else null
  __nv_bfloat16* cache_v;
  int decode_pairs_per_seq;   // decode: tile pairs per sequence (grid decoding)
  int decode_split_from;      // decode: first item split into single-tile items
  int64_t prefill_split_from; // prefill: the pair CTAs from this index on, counted with
                              //   the head in group fastest, then the sequence x head
                              //   group, then the tile pair (cheapest pairs last), are
                              //   done as two key-split single-tile items instead;
                              //   >= the grid size: none
  int prefill_x, prefill_y;   // prefill: x and y extents of the pair grid
  __nv_bfloat16* out;
  float* lse;
  int32_t* status;
  // Decode, balanced tail: the pairs decode_split_from.. (tail pairs t = 0, 1, ..),
  // seg_nkv key tiles each, laid end to end as seg_total = pairs * seg_nkv
  // iterations and cut into seg_ranges equal ranges; range c is part 0 (up to the
  // next pair boundary) and, if it crosses one, part 1.  Piece (c, part) leaves its
  // partial rows in slot 2c + part of seg_ws.  seg_order lists the ranges that
  // cross a boundary by ascending length of their longer part.
  int seg_ranges;
  int seg_nkv;
  int64_t seg_total;
  float* seg_ws;
  uint16_t seg_order[kMaxSegRanges];
};

// ---- balanced decode tail: ranges, pieces and partial slots ----------------------
// (the host plans with the same arithmetic)
__host__ __device__ __forceinline__ int64_t seg_start(int64_t c, int64_t total, int ranges) {
  return c * total / ranges;
}
// Part `part` of range c as virtual iterations [v0, v1); v1 <= v0 when absent.
__host__ __device__ __forceinline__ void seg_piece(int c, int part, int64_t total, int ranges,
                                                   int nkv, int64_t& v0, int64_t& v1) {
  const int64_t s = seg_start(c, total, ranges), e = seg_start(c + 1, total, ranges);
  const int64_t pb = (s / nkv + 1) * nkv;   // first pair boundary after s
  if (part == 0) {
    v0 = s;
    v1 = e < pb ? e : pb;
  } else {
    v0 = pb;
    v1 = e;
  }
}
// The longer part of range c (0 for a range inside one pair).
__host__ __device__ __forceinline__ int seg_long_part(int c, int64_t total, int ranges, int nkv) {
  int64_t a0, a1, b0, b1;
  seg_piece(c, 0, total, ranges, nkv, a0, a1);
  seg_piece(c, 1, total, ranges, nkv, b0, b1);
  return b1 - b0 > a1 - a0 ? 1 : 0;
}

// Prefill with cache append: the CTA of a sequence's last tile pair also writes the
// sequence's prefix K/V to the cache (it reads every key tile of the sequence).
__device__ __forceinline__ bool pair_appends(const FwdParams& p, int b, int m_base) {
  if (p.cache_k == nullptr) return false;
  const int q_len = p.cu_q[b + 1] - p.cu_q[b];
  return m_base == 2 * (((q_len + kBlockM - 1) / kBlockM - 1) / 2);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, kWaitLimitNs));
}

// One work item: head h, sequence b and its query tiles m_base .. m_base + n_qt - 1
// (kSplit: the single tile m_base for both softmax warpgroups, each over part
// of the key range; their partial results are merged at the end.  kSeg: a decode
// pair over its key tiles [seg_kt0, seg_kt1) only, whose unnormalised rows, row
// maxima and sums go to the partial slot seg_slot instead of out and lse).
template <bool kDecode, bool kSplit, bool kPagedAppend, bool kSeg = false>
__device__ __forceinline__ void attn_item(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                          const CUtensorMap& tm_v, const CUtensorMap& tm_k2,
                                          const CUtensorMap& tm_v2, const CUtensorMap& tm_o,
                                          const FwdParams& p, FwdSmem& sm,
                                          const int h, const int b, const int m_base,
                                          const int n_qt, const int seg_kt0 = 0,
                                          const int seg_kt1 = 0, float* seg_slot = nullptr) {
  static_assert(!(kSplit && kPagedAppend), "a key-split item never appends");
  static_assert(!kPagedAppend || !kDecode, "the cache append is a prefill option");
  static_assert(!kSeg || (kDecode && !kSplit), "a balanced-tail piece is a decode pair item");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Another CTA already gave up waiting: do not start new work.
  if (p.status != nullptr && *reinterpret_cast<volatile int32_t*>(p.status) == BCA_ERR_TIMEOUT)
    return;

  // ---- the work item (uniform over the CTA) ---------------------------------
  const int q_seq0 = p.cu_q[b];
  const int q_len = p.cu_q[b + 1] - q_seq0;
  if constexpr (kDecode) {
    // the sequence's query rows must lie in [0, total_q) (prefill sequences are
    // checked by the schedule prep, whose zeroed tile records end them below)
    if (q_seq0 < 0 || q_len < 0 || q_seq0 > p.total_q - q_len) {
      if (threadIdx.x == 0) report_status(p.status, BCA_ERR_SEQLENS);
      return;
    }
  }
  int rows_valid[2], nkt[2] = {0, 0};
  int k_min[2] = {0, 0}, k_hi[2] = {0, 0};
  for (int i = 0; i < 2; ++i) {
    const int m = m_base + (kSplit ? 0 : i);   // a key-split item's warpgroups share one tile
    rows_valid[i] = i < n_qt ? min(kBlockM, max(0, q_len - m * kBlockM)) : 0;
  }
  if (rows_valid[0] <= 0) return;

  int kv_seq0 = 0;     // prefill: first key of the sequence
  int n_pre = 0;       // decode: prefix keys
  int pre0 = 0;        // decode: first cache token of the prefix
  int n_pre_tiles = 0;
  int koff = 0;        // balanced-tail piece: its first key tile (0 otherwise)
  if constexpr (kDecode) {
    pre0 = p.cu_prefix[b];
    const int pre1 = p.cu_prefix[b + 1];
    n_pre = pre1 - pre0;
    n_pre_tiles = (n_pre + kBlockN - 1) / kBlockN;
    // contiguous: cache tokens [pre0, pre1) must lie in the cache; paged: every
    // page of the prefix must lie in the pool (capacity = pages * 128)
    bool bad = n_pre < 0;
    if (p.page_table == nullptr) {
      bad = bad || pre0 < 0 || static_cast<int64_t>(pre1) > p.capacity;
    } else if (!bad) {
      const int64_t n_pages = p.capacity / kBlockN;
      for (int j = threadIdx.x; j < n_pre_tiles; j += blockDim.x) {
        if (j >= p.max_pages) {
          bad = true;
          break;
        }
        const int pg = p.page_table[static_cast<int64_t>(b) * p.max_pages + j];
        if (pg < 0 || pg >= n_pages) bad = true;
      }
    }
    if (__syncthreads_or(bad)) {
      if (threadIdx.x == 0 && h == 0 && m_base == 0)
        report_status(p.status, n_pre < 0 ? BCA_ERR_SEQLENS : BCA_ERR_CAPACITY);
      if constexpr (kSeg) {
        // a row sum of -1 marks the slot's pair as failed for the merge
        if (threadIdx.x < 2 * kBlockM) seg_slot[kSegSlotO + 2 * threadIdx.x + 1] = -1.f;
      }
      return;
    }
    const int n_all = n_pre_tiles + (q_len + kBlockN - 1) / kBlockN;
    if constexpr (kSplit) {
      // warpgroup 1: key tiles [n_all - n_all / 2, n_all); warpgroup 0: the
      // rest (as many or one more; all of a single tile)
      nkt[1] = n_all / 2;
      nkt[0] = n_all - nkt[1];
    } else if constexpr (kSeg) {
      // the piece's key tiles of the pair, up to the sequence's last one (the merge
      // skips a piece that starts past it, as this one returns without a write)
      const int n_seg = min(seg_kt1, n_all) - seg_kt0;
      if (n_seg <= 0) return;
      koff = seg_kt0;
      for (int i = 0; i < 2; ++i) nkt[i] = rows_valid[i] > 0 ? n_seg : 0;
    } else {
      for (int i = 0; i < 2; ++i) nkt[i] = rows_valid[i] > 0 ? n_all : 0;
    }
  }
  // Row ends never decrease along a sequence, so a present Q1 needs at least as
  // many key tiles as Q0; keep that invariant explicitly (extra tiles would be
  // fully masked), since ring stages are released by Q1's softmax (below).
  // (Prefill: once the tile records have been read, after the set-up.)
  int nk = 0, k_hi_all = 0, koff1 = 0, n_kv_tiles = 0;
  auto derive_ranges = [&]() {
    if (!kSplit && nkt[1] > 0 && nkt[1] < nkt[0]) nkt[1] = nkt[0];
    nk = max(nkt[0], nkt[1]);
    k_hi_all = max(k_hi[0], k_hi[1]);
    koff1 = kSplit ? nkt[0] : 0;                  // first key tile of warpgroup 1
    n_kv_tiles = kSplit ? nkt[0] + nkt[1] : nk;   // distinct K/V tiles of the item
  };
  if constexpr (kDecode) derive_ranges();
  // valid keys left in K/V tile j's segment (>= 128: the tile is full)
  auto seg_left_of = [&](int j) {
    if constexpr (!kDecode) {
      return k_hi_all - j * kBlockN;
    } else {
      return j < n_pre_tiles ? n_pre - j * kBlockN : q_len - (j - n_pre_tiles) * kBlockN;
    }
  };
  // Prefill with cache append: the CTA of a sequence's last tile pair reads every key
  // tile of the sequence (its last row sees them all), and its store warp writes the
  // prefix ones to the cache; the stages it stores are released by that warp too.
  const bool appender = !kDecode && !kSplit && pair_appends(p, b, m_base);

  // ---- set-up -----------------------------------------------------------------
  bool q_armed = false;   // (TMA producer lane) the query loads were issued
  if (warp == kWarpTma && lane == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], appender ? 2 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], kSoftmaxThreads);
      mbar_init(&sm.o_final[i], 1);
    }
    mbar_init(&sm.fix_req, 1);
    mbar_init(&sm.v_fixed, 1);
    mbar_init(&sm.drain, 1);
    mbar_init(&sm.merge, kSoftmaxThreads);
    for (int i = 0; i < 2; ++i) mbar_init(&sm.epi[i], kSoftmaxThreads);
    sm.abort = 0;
    fence_mbar_init();
    // The query tiles are loaded at once, before the rest of the set-up: they
    // come from DRAM and are the first MMA's operands.
    const int n_q = !kSplit && rows_valid[1] > 0 ? 2 : 1;
    q_armed = BCA_IN_BOUNDS(p.status, h < p.num_heads && q_seq0 + m_base * kBlockM >= 0 &&
                                          q_seq0 + (m_base + n_q - 1) * kBlockM < p.total_q);
    if (q_armed) {
      mbar_arrive_expect_tx(&sm.q_full, n_q * kTileBytes);
      for (int i = 0; i < n_q; ++i) {
        const int row0 = q_seq0 + (m_base + i) * kBlockM;
        tma_load_3d(&tm_q, &sm.q_full, sm.q[i], 0, h, row0);
        tma_load_3d(&tm_q, &sm.q_full, sm.q[i] + kHalfBytes, 64, h, row0);
      }
    } else {
      sm.abort = 1;
    }
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if constexpr (kDecode) {
      tma_prefetch_desc(&tm_k2);
      tma_prefetch_desc(&tm_v2);
    }
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort;

  if constexpr (!kDecode) {
    // The tile records are written by the schedule prep launched just before this
    // grid, which may start this one early (programmatic dependent launch): the
    // set-up and query loads above overlap the prep, and nothing it writes is read
    // before this wait.
    // (A key-split item belongs to a grid launched after the pair grid, which it may
    // run beside: it reads the records without that wait.  It starts only after
    // every pair CTA has started.  The host splits only when at least two full waves
    // of pair CTAs keep their pairs (one CTA per SM at a time), none of which ends
    // before the prep has completed (those with nothing to do wait for it too), so
    // one of them has ended, after the prep, before the last could start; the pair
    // CTAs that hand their pair to the split grid return at once, wherever they sit
    // in launch order.  The records are read through L2.)
    if constexpr (!kSplit) {
      grid_dependency_wait();
      for (int i = 0; i < 2; ++i) {
        const int m = m_base + i;
        if (rows_valid[i] > 0 && m < p.tiles_per_seq && BCA_IN_BOUNDS(p.status, b < p.batch)) {
          const PrefillTile t = p.tiles[b * p.tiles_per_seq + m];
          k_hi[i] = t.k_hi;
          k_min[i] = t.k_min;
          nkt[i] = (t.k_hi + kBlockN - 1) / kBlockN;
        }
      }
    } else {
      // one query tile, its key tiles cut in two: warpgroup 0 takes the first half
      // (or one more), warpgroup 1 the rest
      if (rows_valid[0] > 0 && m_base < p.tiles_per_seq && BCA_IN_BOUNDS(p.status, b < p.batch)) {
        const int4 t = __ldcg(reinterpret_cast<const int4*>(p.tiles + b * p.tiles_per_seq + m_base));
        const int n_all = (t.x + kBlockN - 1) / kBlockN;
        nkt[1] = n_all / 2;
        nkt[0] = n_all - nkt[1];
        k_hi[0] = k_hi[1] = t.x;
        k_min[0] = k_min[1] = t.y;
      }
    }
    if (nkt[0] <= 0) {
      // an empty tile, or a sequence that failed validation: let the query loads
      // land before the CTA's shared memory is released, and free the TMEM
      if (warp == kWarpTma && lane == 0 && q_armed)
        mbar_wait(&sm.q_full, 0, abort_flag, kWaitLimitNs);
      if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
      return;
    }
    kv_seq0 = p.cu_k[b];
    derive_ranges();
  }

  auto give_up = [&]() {
    sm.abort = 1;
    report_status(p.status, BCA_ERR_TIMEOUT);
  };
  // ring position of load `idx` (K_j = 2j, V_j = 2j + 1)
  auto stage_of = [](int idx) { return idx % kStages; };
  auto phase_of = [](int idx) { return static_cast<uint32_t>((idx / kStages) & 1); };

  if (warp >= 8) {
   regs_decrease<kRegsControl>();
   if (warp == kWarpTma) {
    // =========================== TMA producer ===========================
    if (lane == 0) {
      uint32_t armed = 0;   // bit s: stage s has been loaded at least once
      uint32_t parity = 0;  // bit s: parity of the last load into stage s
      // Load number idx (ring stage idx % kStages) of K or V tile g.
      auto load = [&](int idx, bool is_v, int g) {
        const int s = stage_of(idx);
        const int r = idx / kStages;
        if (r > 0 && !mbar_wait(&sm.kv_empty[s], (r - 1) & 1, abort_flag, kWaitLimitNs)) {
          give_up();
          return false;
        }
        // the tile's map and its (dim 1, dim 2) coordinates
        const CUtensorMap* m;
        int c1, c2;
        bool in_map;   // the tile starts inside its tensor (always true in the release build)
        if constexpr (!kDecode) {
          m = is_v ? &tm_v : &tm_k;
          c1 = h;
          c2 = kv_seq0 + g * kBlockN;
          in_map = BCA_IN_BOUNDS(p.status, c2 >= 0 && c2 < p.total_k && h < p.num_heads);
        } else if (g < n_pre_tiles) {
          m = is_v ? &tm_v : &tm_k;
          c1 = p.page_table != nullptr
                   ? p.page_table[static_cast<int64_t>(b) * p.max_pages + g] * kBlockN
                   : pre0 + g * kBlockN;
          c2 = h;
          in_map = BCA_IN_BOUNDS(p.status, (p.page_table == nullptr || g < p.max_pages) &&
                                               c1 >= 0 && c1 < p.capacity && h < p.num_heads);
        } else {
          m = is_v ? &tm_v2 : &tm_k2;
          c1 = h;
          c2 = q_seq0 + (g - n_pre_tiles) * kBlockN;
          in_map = BCA_IN_BOUNDS(p.status, c2 >= 0 && c2 < p.total_q && h < p.num_heads);
        }
        if (!in_map) {
          *abort_flag = 1;
          return false;
        }
        mbar_arrive_expect_tx(&sm.kv_full[s], kTileBytes);
        armed |= 1u << s;
        parity = (parity & ~(1u << s)) | (static_cast<uint32_t>(r & 1) << s);
        uint8_t* dst = sm.kv[s];
        tma_load_3d(m, &sm.kv_full[s], dst, 0, c1, c2);
        tma_load_3d(m, &sm.kv_full[s], dst + kHalfBytes, 64, c1, c2);
        return true;
      };
      if constexpr (!kSplit) {
        // K_j, V_j shared by both query tiles: loads 2j and 2j + 1 (of key tile koff + j)
        for (int i = 0; i < 2 * nk; ++i)
          if (!load(i, i & 1, koff + (i >> 1))) break;
      } else {
        // Each warpgroup has its own tiles; loads follow the MMA thread's order of
        // use: K_0(0), K_1(0), then per step j: V_0(j), K_0(j+1), V_1(j), K_1(j+1).
        int idx = 0;
        bool go = true;
        for (int j = 0; j <= nk && go; ++j) {
          for (int i = 0; i < 2 && go; ++i) {
            const int g0 = i == 0 ? 0 : koff1;
            if (j >= 1 && j - 1 < nkt[i]) go = load(idx++, true, g0 + j - 1);
            if (go && j < nkt[i]) go = load(idx++, false, g0 + j);
          }
        }
      }
      // If anything went wrong, let every load in flight land before the CTA exits.
      if (*abort_flag) {
        for (int s = 0; s < kStages; ++s)
          if (armed >> s & 1) mbar_wait(&sm.kv_full[s], parity >> s & 1, nullptr, kWaitLimitNs / 4);
        if (q_armed) mbar_wait(&sm.q_full, 0, nullptr, kWaitLimitNs / 4);
      }
    }
   } else if (warp == kWarpMma) {
    // =========================== MMA issuer ===========================
    // One thread issues everything; waits are single-thread so no warp-wide
    // synchronisation sits between MMA groups.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBlockM, kHeadDim, 0, 1);
      // Operand layouts.  K-major (Q as A, K as B of S = Q K^T): 128 rows x 128
      // bf16 as two 128-byte-swizzled halves of 16 KB (columns 0-63, 64-127);
      // K-step kk starts at half kk / 4, byte 32 * (kk % 4).  MN-major (V as B
      // of O += P V): rows are keys, the 64-column halves along the head dim are
      // 16 KB apart (LBO), 8-key groups 1024 B apart (SBO); K-step kk starts at
      // key 16 kk (2048 B).  Descriptor start fields are in 16-byte units; a
      // ring stage is kTileBytes / 16 apart.
      // (a key-split item has its one query tile in q[0], used by both S MMAs)
      // Every descriptor shares its high word (stride, version, swizzle); the low
      // word holds the start address and the leading-byte offset, so each MMA
      // below costs one 32-bit add per shared-memory operand.
      const uint64_t desc_q0 = smem_desc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint32_t desc_hi = static_cast<uint32_t>(desc_q0 >> 32);
      const uint32_t q_lo0 = static_cast<uint32_t>(desc_q0);
      const uint32_t q_lo1 =
          static_cast<uint32_t>(smem_desc_sw128(smem_u32(sm.q[kSplit ? 0 : 1]), 16, 1024));
      const uint32_t k_lo0 = static_cast<uint32_t>(smem_desc_sw128(smem_u32(sm.kv[0]), 16, 1024));
      const uint32_t v_lo0 =
          static_cast<uint32_t>(smem_desc_sw128(smem_u32(sm.kv[0]), kHalfBytes, 1024));
      constexpr uint32_t kStageLo = kTileBytes >> 4;   // one ring stage, in 16-byte units
      auto issue_s = [&](int i, int stage) {  // S_i = Q_i K^T
        const uint32_t qa = i == 0 ? q_lo0 : q_lo1;
        const uint32_t kb = k_lo0 + static_cast<uint32_t>(stage) * kStageLo;
        const uint32_t d = tmem + kColS + i * 128;
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          constexpr uint32_t kHalfLo = kHalfBytes >> 4;
          const uint32_t off = (kk >> 2) * kHalfLo + (kk & 3) * 2;
          if (kk == 0)
            umma_ss<0>(d, qa + off, kb + off, desc_hi, idesc_qk);
          else
            umma_ss<1>(d, qa + off, kb + off, desc_hi, idesc_qk);
        }
        umma_commit(&sm.s_full[i]);
      };
      auto issue_pv = [&](int i, int stage, int j, bool last) {  // O_i += P_i V
        const uint32_t vb = v_lo0 + static_cast<uint32_t>(stage) * kStageLo;
        const uint32_t a = tmem + kColS + i * 128;
        const uint32_t d = tmem + kColO + i * 128;
        umma_ts<-1>(d, a, vb, desc_hi, idesc_pv, j > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < kBlockN / 16; ++kk)
          umma_ts<1>(d, a + kk * 8, vb + kk * (2048 >> 4), desc_hi, idesc_pv);
        if (last) umma_commit(&sm.o_final[i]);
      };

      // V tile g in stage s has landed; if its segment ends inside it, have the
      // fix-up warp zero the rows past the end before any PV reads it.
      int tails = 0;
      auto fix_tail = [&](int g, int s) {
        const int left = seg_left_of(g);
        if (left >= kBlockN) return true;
        sm.fix_stage = s;
        sm.fix_from = left;
        mbar_arrive(&sm.fix_req);
        return mbar_wait(&sm.v_fixed, (tails++) & 1, abort_flag, kWaitLimitNs);
      };
      auto landed = [&](int idx) {
        return mbar_wait(&sm.kv_full[stage_of(idx)], phase_of(idx), abort_flag, kWaitLimitNs);
      };

      bool ok = mbar_wait(&sm.q_full, 0, abort_flag, kWaitLimitNs);
      if constexpr (!kSplit) {
        if (ok && nk > 0) {
          ok = landed(0);
          if (ok) {
            for (int i = 0; i < 2; ++i)
              if (nkt[i] > 0) issue_s(i, stage_of(0));
          }
        }
        // Steady state: while both query tiles have a next key tile, every iteration
        // issues PV0, S0, PV1, S1 with no per-tile conditions; a loop body free of
        // branches on the tile counts measured 5.5% (prefill) and 3.7% (decode)
        // faster than the general loop below, which then finishes the item.
        int j = 0;
        const int n_both = min(nkt[0], nkt[1]) - 1;
        // V(j + 1) is checked (and its fix-up requested) before S1(j + 1) is issued,
        // while the pipe still holds PV1(j): between S1(j + 1) and PV0(j + 1), where
        // the pipe runs dry, only the wait for P0(j + 1) is left (1.0% prefill, 0.8%
        // decode).
        bool v_ready = false;   // V(j) landed and fixed ahead of iteration j
        if (n_both > 0 && ok) {
          ok = landed(1) && fix_tail(koff, stage_of(1));
          v_ready = true;
        }
        for (; j < n_both && ok; ++j) {
          const int vs = stage_of(2 * j + 1), ks = stage_of(2 * j + 2);
          if (!mbar_wait(&sm.p_full[0], j & 1, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(0, vs, j, false);
          if (!landed(2 * j + 2)) {
            ok = false;
            break;
          }
          issue_s(0, ks);
          if (!mbar_wait(&sm.p_full[1], j & 1, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(1, vs, j, false);
          if (!(landed(2 * j + 3) && fix_tail(koff + j + 1, stage_of(2 * j + 3)))) {
            ok = false;
            break;
          }
          issue_s(1, ks);
        }
        for (; j < nk && ok; ++j) {
          const int vs = stage_of(2 * j + 1), ks = stage_of(2 * j + 2);
          ok = (v_ready && j == n_both) || (landed(2 * j + 1) && fix_tail(koff + j, vs));
          bool k_next_ready = false;
          for (int i = 0; i < 2 && ok; ++i) {
            if (j < nkt[i]) {
              ok = mbar_wait(&sm.p_full[i], j & 1, abort_flag, kWaitLimitNs);
              if (!ok) break;
              tc_fence_after();
              issue_pv(i, vs, j, j == nkt[i] - 1);
            }
            if (j + 1 < nkt[i]) {
              if (!k_next_ready) {
                ok = landed(2 * j + 2);
                if (!ok) break;
                k_next_ready = true;
              }
              issue_s(i, ks);
            }
          }
        }
      } else {
        // Key split: every operand is used once, in the producer's load order; the
        // softmax warpgroup that owns it hands its stage back (see below).
        int c = 0;
        for (int i = 0; i < 2 && ok; ++i) {
          if (nkt[i] == 0) continue;
          ok = landed(c);
          if (ok) {
            issue_s(i, stage_of(c));
            ++c;
          }
        }
        for (int j = 0; j < nk && ok; ++j) {
          for (int i = 0; i < 2 && ok; ++i) {
            if (j < nkt[i]) {
              const int vs = stage_of(c);
              ok = landed(c) && fix_tail((i == 0 ? 0 : koff1) + j, vs) &&
                   mbar_wait(&sm.p_full[i], j & 1, abort_flag, kWaitLimitNs);
              if (!ok) break;
              tc_fence_after();
              issue_pv(i, vs, j, j == nkt[i] - 1);
              ++c;
            }
            if (j + 1 < nkt[i]) {
              ok = landed(c);
              if (!ok) break;
              issue_s(i, stage_of(c));
              ++c;
            }
          }
        }
      }
      if (!ok) give_up();
      // Drain: every MMA this thread issued must finish before TMEM is released.
      umma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, nullptr, kWaitLimitNs);
    }
    __syncwarp();
   } else if (warp == kWarpFix) {
    // ====================== V tail fix-up ======================
    // Keys past the end of a tile's segment may hold anything (another
    // sequence, unused cache capacity): zero those V rows so 0 * V stays 0.
    // The MMA thread names the stage and the first row to clear, after its own
    // wait on the tile's kv_full phase, so this warp never polls a ring barrier.
    int n_tails = 0;
    for (int g = koff; g < koff + n_kv_tiles; ++g) n_tails += seg_left_of(g) < kBlockN ? 1 : 0;
    for (int t = 0; t < n_tails; ++t) {
      if (!warp_wait(&sm.fix_req, t & 1, abort_flag)) {
        if (lane == 0) give_up();
        break;
      }
      const int fix_stage = *reinterpret_cast<volatile int*>(&sm.fix_stage);
      const int seg_left = *reinterpret_cast<volatile int*>(&sm.fix_from);
      uint8_t* vb = sm.kv[fix_stage];
      const int nrows = BCA_IN_BOUNDS(p.status, fix_stage >= 0 && fix_stage < kStages &&
                                                    seg_left >= 0 && seg_left < kBlockN)
                            ? kBlockN - seg_left
                            : 0;
      for (int idx = lane; idx < nrows * 16; idx += 32) {
        const int row = seg_left + (idx >> 4);
        const int chunk = idx & 15;
        *reinterpret_cast<uint4*>(vb + (chunk >> 3) * kHalfBytes + row * 128 + (chunk & 7) * 16) =
            make_uint4(0, 0, 0, 0);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.v_fixed);
    }
   } else if (warp == kWarpStore && appender) {
    // ============ prefix store (prefill with cache append) ============
    // Every sequence is checked first and nothing is written if one fails, as
    // in the standalone append: a prefix longer than its keys (or with no query
    // row to carry it), a negative offset, or the prefixes past the capacity
    // (paged: more pages than the table holds, or a page outside the pool).
    int bad = 0;
    for (int i = lane; i < p.batch; i += 32) {
      const int pl = p.cu_prefix[i + 1] - p.cu_prefix[i];
      const int kl = p.cu_k[i + 1] - p.cu_k[i];
      const int ql = p.cu_q[i + 1] - p.cu_q[i];
      if (pl < 0 || pl > kl || p.cu_prefix[i] < 0 || (pl > 0 && ql == 0)) bad = BCA_ERR_SEQLENS;
    }
    if constexpr (!kPagedAppend) {
      if (lane == 0 && static_cast<int64_t>(p.cu_prefix[p.batch]) > p.capacity)
        bad = bad != 0 ? bad : BCA_ERR_CAPACITY;
    } else {
      const int64_t n_pages = p.capacity / kBlockN;
      for (int i = 0; i < p.batch; ++i) {
        const int n = (p.cu_prefix[i + 1] - p.cu_prefix[i] + kBlockN - 1) / kBlockN;
        if (n > p.max_pages) bad = bad != 0 ? bad : BCA_ERR_CAPACITY;
        for (int jj = lane; jj < n && jj < p.max_pages; jj += 32) {
          const int pg = p.page_table[static_cast<int64_t>(i) * p.max_pages + jj];
          if (pg < 0 || pg >= n_pages) bad = bad != 0 ? bad : BCA_ERR_CAPACITY;
        }
      }
    }
    bad = __reduce_max_sync(0xffffffffu, bad);
    if (bad != 0 && lane == 0 && h == 0) report_status(p.status, bad);
    const int c0 = p.cu_prefix[b];
    const int n_pre_b = bad == 0 ? p.cu_prefix[b + 1] - c0 : 0;
    // Follow the ring in load order (K_j = 2j, V_j = 2j + 1): once a tile has
    // landed, store its prefix rows, then hand the stage back (the producer
    // waits for this arrival as well as the softmax's).
    for (int i = 0; i < 2 * nk; ++i) {
      const int s = stage_of(i);
      if (!warp_wait(&sm.kv_full[s], phase_of(i), abort_flag)) {
        if (lane == 0) give_up();
        break;
      }
      const int j = i >> 1;
      const bool is_v = i & 1;
      const int rows = min(kBlockN, n_pre_b - j * kBlockN);   // prefix rows in the tile
      // cache token of the tile's first row (a paged cache: one 128-token page)
      int64_t tok0 = static_cast<int64_t>(c0) + j * kBlockN;
      if constexpr (kPagedAppend) {
        if (rows > 0)
          tok0 = static_cast<int64_t>(p.page_table[static_cast<int64_t>(b) * p.max_pages + j]) *
                 kBlockN;
      }
      // the tile's cache rows [tok0, tok0 + rows) lie in the layer (bounds-checked build)
      const bool rows_in = rows <= 0 || BCA_IN_BOUNDS(p.status, tok0 >= 0 && tok0 + rows <= p.capacity &&
                                                                    h < p.num_heads &&
                                                                    (!kPagedAppend || j < p.max_pages));
      if (!rows_in) {
        // skip the tile
      } else if (rows == kBlockN) {
        // a whole tile: two TMA stores through the cache map (same 128-byte swizzled
        // layout as the loads), read out of shared memory before the stage is freed
        if (lane == 0) {
          const CUtensorMap* m = is_v ? &tm_v2 : &tm_k2;
          tma_store_3d(m, sm.kv[s], 0, static_cast<int>(tok0), h);
          tma_store_3d(m, sm.kv[s] + kHalfBytes, 64, static_cast<int>(tok0), h);
          bulk_commit_group();
          bulk_wait_read_all();
        }
      } else if (rows > 0) {
        // the prefix ends inside the tile: copy its rows with 16-byte accesses,
        // undoing the swizzle (chunk c of row r sits at chunk c ^ (r % 8))
        __nv_bfloat16* dst =
            (is_v ? p.cache_v : p.cache_k) + (static_cast<int64_t>(h) * p.capacity + tok0) * kHeadDim;
        for (int idx = lane; idx < rows * 16; idx += 32) {
          const int r = idx >> 4, c = idx & 15;
          const uint4 val = *reinterpret_cast<const uint4*>(
              sm.kv[s] + (c >> 3) * kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) * 16));
          *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(r) * kHeadDim + c * 8) = val;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.kv_empty[s]);
    }
    if (lane == 0) bulk_wait_read_all();   // the stages are read before the CTA ends
   }
  } else {
    regs_increase<kRegsSoftmax>();
    // =========================== softmax warpgroups ===========================
    const int qi = warp >> 2;               // which query tile
    const int wq = warp & 3;                // TMEM lane group
    const int row = wq * 32 + lane;         // == TMEM lane == row within the tile
    const int n_tiles = nkt[qi];
    // decode: this warpgroup's key tiles, counted from its first one (koff1 for
    // warpgroup 1 of a key-split item, koff in a balanced-tail piece): prefix tiles
    // before tgt0, keys left in the prefix
    const int kfirst = koff + (qi == 1 ? koff1 : 0);
    const int tgt0 = n_pre_tiles - kfirst;
    const int pre_left0 = n_pre - kfirst * kBlockN;
    const int row0 = q_seq0 + (m_base + (kSplit ? 0 : qi)) * kBlockM;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t s_addr = lane_addr + kColS + qi * 128;
    const uint32_t o_addr = lane_addr + kColO + qi * 128;
    const bool row_valid = row < rows_valid[qi];
    const bool releaser = !kSplit && (qi == 1 || nkt[1] == 0);
    int e_row = 0;
    if constexpr (!kDecode) {
      const bool e_in =
          row_valid && BCA_IN_BOUNDS(p.status, row0 + row >= 0 && row0 + row < p.total_q);
      if constexpr (kSplit)
        e_row = e_in ? __ldcg(p.row_end + row0 + row) : k_hi[qi];
      else
        e_row = e_in ? p.row_end[row0 + row] : k_hi[qi];
    }
    // first key tile of this warpgroup (warpgroup 1 of a key-split item: koff1)
    const int jg0 = kSplit && qi == 1 ? koff1 : 0;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY;   // reference max of the row, log2 domain
    float l_run = 0.f;
    bool ok = true;

    for (int j = 0; j < n_tiles; ++j) {
      ok = warp_wait(&sm.s_full[qi], j & 1, abort_flag);
      if (!ok) break;
      // The commit behind S_qi(j) covers every MMA issued before it.  For the
      // last tile in issue order (Q1, or Q0 alone) that includes all readers
      // of V_{j-1} and K_j, so their ring stages can be handed back to the
      // producer here, without a commit on the MMA thread's critical path.
      if constexpr (kSplit) {
        // Key split: each warpgroup releases its own K(j) and V(j-1), read only by
        // S(j) and PV(j-1), both covered by the commit behind S(j).  In the load
        // order K0(0), K1(0), then V0(j-1), K0(j), V1(j-1), K1(j) for j >= 1, they
        // are loads 4j-1 and 4j-2 (warpgroup 0), 4j+1 and 4j (warpgroup 1).
        if (wq == 0 && lane == 0) {
          if (j > 0) mbar_arrive(&sm.kv_empty[stage_of(qi == 0 ? 4 * j - 2 : 4 * j)]);
          mbar_arrive(&sm.kv_empty[stage_of(j == 0 ? qi : (qi == 0 ? 4 * j - 1 : 4 * j + 1))]);
        }
      }
      if (releaser && wq == 0 && lane == 0) {
        if (j > 0) mbar_arrive(&sm.kv_empty[stage_of(2 * j - 1)]);   // V_{j-1}
        mbar_arrive(&sm.kv_empty[stage_of(2 * j)]);                  // K_j
      }
      tc_fence_after();
      // S row as 64 register pairs: sp[c] = columns (2c, 2c+1)
      uint64_t sp[kBlockN / 2];
      tmem_ld128_pairs(s_addr, sp);
      // ---- mask (boundary tiles only) ----
      int lim;
      bool need_mask;
      if constexpr (!kDecode) {
        lim = e_row - (jg0 + j) * kBlockN;
        need_mask = (jg0 + j + 1) * kBlockN > k_min[qi];
      } else {
        lim = j < tgt0 ? pre_left0 - j * kBlockN : q_len - (j - tgt0) * kBlockN;
        need_mask = lim < kBlockN;
      }
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < kBlockN / 2; ++c) {
          const float lo = 2 * c < lim ? lo_f(sp[c]) : -INFINITY;
          const float hi = 2 * c + 1 < lim ? hi_f(sp[c]) : -INFINITY;
          sp[c] = pack2f(lo, hi);
        }
      }
      // Row max of the tile (log2 domain).
      auto tile_max = [&]() {
        float mxa[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mxa[u] = fmaxf(lo_f(sp[u]), hi_f(sp[u]));
#pragma unroll
        for (int c = 8; c < kBlockN / 2; c += 8) {
#pragma unroll
          for (int u = 0; u < 8; ++u) mxa[u] = fmax3(mxa[u], lo_f(sp[c + u]), hi_f(sp[c + u]));
        }
        return fmaxf(fmaxf(fmax3(mxa[0], mxa[1], mxa[2]), fmax3(mxa[3], mxa[4], mxa[5])),
                     fmaxf(mxa[6], mxa[7])) * sl2;
      };
      // P = exp2(S * scale*log2e - m_ref) -> bf16 into the first 64 columns of S_i;
      // returns the row sum of the fp32 values.
      auto write_p = [&]() {
        const uint64_t sl2v = pack2f(sl2, sl2);
        const uint64_t negm = pack2f(-m_ref, -m_ref);
        uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const uint64_t x = ffma2_b64(sp[half * 32 + c], sl2v, negm);
            const float p0 = ex2_approx(lo_f(x)), p1 = ex2_approx(hi_f(x));
            acc[c & 3] = fadd2_b64(acc[c & 3], pack2f(p0, p1));
            w[c] = pack_bf16x2(p0, p1);
          }
          tmem_st32(s_addr + half * 32, w);
        }
        tmem_st_wait();
        const uint64_t asum = fadd2_b64(fadd2_b64(acc[0], acc[1]), fadd2_b64(acc[2], acc[3]));
        return lo_f(asum) + hi_f(asum);
      };
      // The reference max m_ref is the exact row max after the first tile and is
      // only moved when a tile would make the row sum large (> 2^16 relative to
      // it): O and l share the reference, so out = O / l is exact either way and
      // in the common case no max needs to be taken at all.
      float alpha = 1.f;
      if (j == 0) {
        m_ref = tile_max();   // key 0 is visible to every row: finite
        if constexpr (kSplit && !kDecode) {
          // except in warpgroup 1 of a key-split prefill item, whose keys start at
          // tile koff1: a row that ends before them sees none, and any finite
          // reference gives it P = 0, l = 0, O = 0 for the merge
          if (m_ref == -INFINITY) m_ref = 0.f;
        }
      }
      float tsum = write_p();
      if (j > 0 && __any_sync(0xffffffffu, !(tsum <= kSumLimit))) {
        const float m_new = fmaxf(m_ref, tile_max());
        alpha = ex2_approx(m_ref - m_new);
        // O_i holds PV_i(0..j-1), all complete (covered by the S_i(j) commit)
        const uint64_t a2 = pack2f(alpha, alpha);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(o_addr + c * 32, r);
#pragma unroll
          for (int x = 0; x < 32; x += 2) {
            const uint64_t v = fmul2_b64(pack2f(__uint_as_float(r[x]), __uint_as_float(r[x + 1])), a2);
            r[x] = __float_as_uint(lo_f(v));
            r[x + 1] = __float_as_uint(hi_f(v));
          }
          tmem_st32(o_addr + c * 32, r);
        }
        m_ref = m_new;
        tsum = write_p();
      }
      l_run = l_run * alpha + tsum;
      tc_fence_before();
      mbar_arrive(&sm.p_full[qi]);
    }

    if constexpr (kSplit) {
      // Key split: warpgroup 1 hands its row maxima and sums to warpgroup 0, which
      // brings both partial rows to the larger max before adding O and l.  With a
      // single key tile warpgroup 1 has none, and there is nothing to merge.
      float* const ml = reinterpret_cast<float*>(sm.q[1]);   // q[1] holds no query here
      const bool use1 = nkt[1] > 0;
      if (qi == 1) {
        if (!ok) {
          if (lane == 0) give_up();
        } else if (use1) {
          ml[2 * row] = m_ref;
          ml[2 * row + 1] = l_run;
          mbar_arrive(&sm.merge);
        }
      } else {
        ok = ok && warp_wait(&sm.o_final[0], 0, abort_flag);
        if (use1)
          ok = ok && warp_wait(&sm.merge, 0, abort_flag) && warp_wait(&sm.o_final[1], 0, abort_flag);
        if (!ok) {
          if (lane == 0) give_up();
        } else {
          tc_fence_after();
          float m_fin = m_ref, l_fin = l_run, a0 = 1.f, a1 = 0.f;
          if (use1) {
            const float m1 = ml[2 * row], l1 = ml[2 * row + 1];
            m_fin = fmaxf(m_ref, m1);
            a0 = ex2_approx(m_ref - m_fin);
            a1 = ex2_approx(m1 - m_fin);
            l_fin = l_run * a0 + l1 * a1;
          }
          const float inv_l = 1.f / l_fin;
          const float c0 = a0 * inv_l, c1 = a1 * inv_l;
          __nv_bfloat16* orow =
              p.out + (static_cast<size_t>(row0 + row) * p.num_heads + h) * kHeadDim;
          const bool row_out = row_valid && BCA_IN_BOUNDS(p.status, row0 + row >= 0 &&
                                                                        row0 + row < p.total_q &&
                                                                        h < p.num_heads);
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t r0[16], r1[16];
            tmem_ld16(o_addr + c * 16, r0);
            if (use1) {
              tmem_ld16(o_addr + 128 + c * 16, r1);
            } else {
#pragma unroll
              for (int x = 0; x < 16; ++x) r1[x] = 0;
            }
            uint32_t w[8];
#pragma unroll
            for (int x = 0; x < 8; ++x)
              w[x] = pack_bf16x2(
                  __uint_as_float(r0[2 * x]) * c0 + __uint_as_float(r1[2 * x]) * c1,
                  __uint_as_float(r0[2 * x + 1]) * c0 + __uint_as_float(r1[2 * x + 1]) * c1);
            if (row_out) {
              uint4* dst = reinterpret_cast<uint4*>(orow + c * 16);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
          if (row_out) {
            p.lse[static_cast<size_t>(h) * p.total_q + row0 + row] =
                (m_fin + log2f(l_fin)) * 0.69314718055994530942f;
          }
        }
      }
    } else {
      if (ok && n_tiles > 0) ok = warp_wait(&sm.o_final[qi], 0, abort_flag);
      if (!ok) {
        if (lane == 0) give_up();
      } else if (kSeg && n_tiles > 0) {
        // Balanced-tail piece: the row's unnormalised O (against m_ref) and its
        // (m_ref, l) go to the partial slot; a warp's stores of one column group
        // cover 32 consecutive rows, 512 contiguous bytes.
        tc_fence_after();
        float4* o_part = reinterpret_cast<float4*>(seg_slot) + qi * 32 * kBlockM + row;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(o_addr + c * 32, r);
          if (row_valid) {
#pragma unroll
            for (int x = 0; x < 8; ++x)
              o_part[(c * 8 + x) * kBlockM] =
                  make_float4(__uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                              __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
          }
        }
        if (row_valid)
          reinterpret_cast<float2*>(seg_slot + kSegSlotO)[qi * kBlockM + row] =
              make_float2(m_ref, l_run);
      } else if (n_tiles > 0) {
        tc_fence_after();
        const float inv_l = 1.f / l_run;
        // A whole tile goes out by TMA: the rows, in bf16, are staged in this tile's
        // Q buffer (idle: the commit behind o_final covers every MMA that read it)
        // in the 128-byte swizzled layout of the box, then one thread stores the two
        // 64-column halves.  (Rows written one per thread, 8 KB apart, cost the
        // launch ~2%.)  A ragged tile writes its valid rows directly.
        const bool staged = rows_valid[qi] == kBlockM;
        uint8_t* const stage = sm.q[qi];
        __nv_bfloat16* orow =
            p.out + (static_cast<size_t>(row0 + row) * p.num_heads + h) * kHeadDim;
        const bool row_out = row_valid && BCA_IN_BOUNDS(p.status, row0 + row >= 0 &&
                                                                      row0 + row < p.total_q &&
                                                                      h < p.num_heads);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(o_addr + c * 32, r);
          uint32_t w[16];
#pragma unroll
          for (int x = 0; x < 16; ++x)
            w[x] = pack_bf16x2(__uint_as_float(r[2 * x]) * inv_l,
                               __uint_as_float(r[2 * x + 1]) * inv_l);
          if (staged) {
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const int cc = 4 * c + x;   // 16-byte chunk of the row, 0..15
              *reinterpret_cast<uint4*>(stage + (cc >> 3) * kHalfBytes + row * 128 +
                                        (((cc & 7) ^ (row & 7)) * 16)) =
                  make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
            }
          } else if (row_out) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int x = 0; x < 4; ++x)
              dst[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
          }
        }
        if (staged) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(&sm.epi[qi]);
          if (wq == 0 && lane == 0) {
            if (mbar_wait(&sm.epi[qi], 0, abort_flag, kWaitLimitNs)) {
              if (BCA_IN_BOUNDS(p.status, row0 >= 0 && row0 + kBlockM <= p.total_q &&
                                              h < p.num_heads)) {
                tma_store_3d(&tm_o, stage, 0, h, row0);
                tma_store_3d(&tm_o, stage + kHalfBytes, 64, h, row0);
                bulk_commit_group();
                // only the reads of the staged tile must end before the CTA does;
                // its global writes complete before the grid does (0.3% prefill,
                // 0.4% decode against waiting for them here)
                bulk_wait_read_all();
              }
            } else {
              give_up();
            }
          }
        }
        if (row_out) {
          p.lse[static_cast<size_t>(h) * p.total_q + row0 + row] =
              (m_ref + log2f(l_run)) * 0.69314718055994530942f;
        }
      }
    }
  }

  // ---- teardown ------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Prefill: a 3-D grid of (head in group, tile pair, sequence x head group): the
// pairs of a group of heads, costliest first, then the next group, so that the
// CTAs in flight share the K/V of a few heads in L2.
// Decode: a 1-D list of equal-cost tile pairs, the pairs of one head next to
// each other (they stream the same K/V tiles); the pairs of a last, partly
// filled wave become single-tile items (kSplit: two CTAs per pair, each with its
// key range split between the two softmax warpgroups), or, with a workspace,
// balanced-tail pieces (kSeg: one CTA per piece, longer pieces first), launched
// as a second grid that may start as soon as every pair CTA has started.
template <bool kDecode, bool kSplit, bool kPagedAppend = false, bool kSeg = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_k2,
                    const __grid_constant__ CUtensorMap tm_v2,
                    const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  if constexpr (!kDecode && !kSplit) {
    // the key-split grid launched after this one may start once every CTA here has
    grid_launch_dependents();
    const int h = blockIdx.x + (blockIdx.z % p.head_groups) * gridDim.x;   // groups are full
    const int b = blockIdx.z / p.head_groups;
    const int m_base = 2 * (static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y));
    // The pairs of the split set (the cheapest of every head group) are done by the
    // key-split grid (never the pair that appends to the cache).
    const int64_t split_idx =
        blockIdx.x + static_cast<int64_t>(gridDim.x) * (blockIdx.z + static_cast<int64_t>(gridDim.z) * blockIdx.y);
    if (split_idx >= p.prefill_split_from && !pair_appends(p, b, m_base)) return;
    // Any other pair CTA ends only after the schedule prep has completed, even with
    // no rows to do: the key-split grid relies on it.  (One that finds another CTA
    // has given up ends at once; the split CTAs, which start later, then do too.)
    if (m_base * kBlockM >= p.cu_q[b + 1] - p.cu_q[b]) {
      grid_dependency_wait();
      return;
    }
    attn_item<false, false, kPagedAppend>(tm_q, tm_k, tm_v, tm_k2, tm_v2, tm_o, p, sm, h, b,
                                          m_base, 2);
  } else if constexpr (!kDecode) {
    // Prefill key split: CTA 2i + s does query tile s of the pair CTA at split index
    // prefill_split_from + i of the pair grid (head in group fastest, then sequence x
    // head group, then tile pair).
    const int64_t split_idx = p.prefill_split_from + blockIdx.x / 2;
    const int x = static_cast<int>(split_idx % p.prefill_x);
    const int64_t zy = split_idx / p.prefill_x;
    const int n_z = p.batch * p.head_groups;
    const int z = static_cast<int>(zy % n_z);
    const int y = static_cast<int>(zy / n_z);
    const int h = x + (z % p.head_groups) * p.prefill_x;
    const int b = z / p.head_groups;
    const int m_base = 2 * (p.prefill_y - 1 - y);
    if (!pair_appends(p, b, m_base))
      attn_item<false, true, false>(tm_q, tm_k, tm_v, tm_k2, tm_v2, tm_o, p, sm, h, b,
                                    m_base + static_cast<int>(blockIdx.x & 1), 2);
    // do not complete before the pair grid has (work queued after the call sees both)
    grid_dependency_wait();
  } else if constexpr (kSeg) {
    // the merge grid launched after this one may start once every piece has
    grid_launch_dependents();
    // CTA i < seg_ranges: the longer part of range i; after them, the shorter
    // parts, longest first (their ranges in seg_order)
    const int i = blockIdx.x;
    const int c = i < p.seg_ranges ? i : static_cast<int>(p.seg_order[i - p.seg_ranges]);
    const int long_part = seg_long_part(c, p.seg_total, p.seg_ranges, p.seg_nkv);
    const int part = i < p.seg_ranges ? long_part : 1 - long_part;
    int64_t v0, v1;
    seg_piece(c, part, p.seg_total, p.seg_ranges, p.seg_nkv, v0, v1);
    const int t = static_cast<int>(v0 / p.seg_nkv);   // tail pair
    const int kt0 = static_cast<int>(v0 - static_cast<int64_t>(t) * p.seg_nkv);
    const int kt1 = static_cast<int>(v1 - static_cast<int64_t>(t) * p.seg_nkv);
    const int item = p.decode_split_from + t;
    const int rest = item / p.decode_pairs_per_seq;
    if (v1 > v0 && BCA_IN_BOUNDS(p.status, c < p.seg_ranges && kt0 >= 0 && kt1 <= p.seg_nkv))
      attn_item<true, false, false, true>(
          tm_q, tm_k, tm_v, tm_k2, tm_v2, tm_o, p, sm, rest % p.num_heads, rest / p.num_heads,
          2 * (item % p.decode_pairs_per_seq), 2, kt0, kt1,
          p.seg_ws + static_cast<size_t>(2 * c + part) * kSegSlotFloats);
    // do not complete before the pair grid has (work queued after the call sees both)
    grid_dependency_wait();
  } else if constexpr (!kSplit) {
    grid_launch_dependents();
    const int L = blockIdx.x;
    const int rest = L / p.decode_pairs_per_seq;
    attn_item<true, false, false>(tm_q, tm_k, tm_v, tm_k2, tm_v2, tm_o, p, sm, rest % p.num_heads,
                           rest / p.num_heads, 2 * (L % p.decode_pairs_per_seq), 2);
  } else {
    const int item = p.decode_split_from + static_cast<int>(blockIdx.x) / 2;
    const int sub = blockIdx.x & 1;
    const int rest = item / p.decode_pairs_per_seq;
    attn_item<true, true, false>(tm_q, tm_k, tm_v, tm_k2, tm_v2, tm_o, p, sm, rest % p.num_heads,
                          rest / p.num_heads, 2 * (item % p.decode_pairs_per_seq) + sub, 2);
    // This grid may run beside the pair grid launched before it: do not
    // complete before that grid has, so work queued after both sees its output.
    grid_dependency_wait();
  }
}

// Merge of the balanced decode tail: CTA (t, i, quarter) combines, for query tile
// i of tail pair t and 32 of the 128 columns, the partial rows its pieces left in
// the workspace (in key order), each against its own reference max, online:
// m = max m_s, O = sum 2^(m_s - m) O_s, l = sum 2^(m_s - m) l_s; out = O / l,
// lse = (m + log2 l) ln 2.  One thread per row; a warp's loads of one column
// group are 32 consecutive rows, 512 contiguous bytes, and the next piece's
// loads are in flight while the current one is added.
constexpr int kMergeThreads = kBlockM;

__global__ void __launch_bounds__(kMergeThreads)
    seg_merge_kernel(const __grid_constant__ FwdParams p) {
  __shared__ int s_c0, s_n, s_part0;
  const int quarter = blockIdx.x & 3, qi = (blockIdx.x >> 2) & 1, t = blockIdx.x >> 3;
  const int row = threadIdx.x;
  const int item = p.decode_split_from + t;
  const int rest = item / p.decode_pairs_per_seq;
  const int h = rest % p.num_heads, b = rest / p.num_heads;
  const int m = 2 * (item % p.decode_pairs_per_seq) + qi;
  // (inputs only before the wait: nothing here is written by the pieces)
  const int q_seq0 = p.cu_q[b];
  const int q_len = p.cu_q[b + 1] - q_seq0;
  if (q_seq0 < 0 || q_len < 0 || q_seq0 > p.total_q - q_len) return;   // reported by the pieces
  const int rows_valid = min(kBlockM, q_len - m * kBlockM);
  if (rows_valid <= 0) return;
  const int n_pre = p.cu_prefix[b + 1] - p.cu_prefix[b];
  const int n_all = (n_pre + kBlockN - 1) / kBlockN + (q_len + kBlockN - 1) / kBlockN;
  if (n_all > p.seg_nkv) {
    // more keys than max_prefix allowed for: they were planned for no piece
    if (row == 0 && quarter == 0) report_status(p.status, BCA_ERR_SEQLENS);
    return;
  }
  if (threadIdx.x == 0) {
    // the ranges holding this pair's key tiles [0, n_all): c0 (its part 1 when it
    // starts in the previous pair) and the ranges after it that start before n_all
    const int64_t lo = static_cast<int64_t>(t) * p.seg_nkv, hi = lo + n_all;
    int c = static_cast<int>(lo * p.seg_ranges / p.seg_total);
    while (c > 0 && seg_start(c, p.seg_total, p.seg_ranges) > lo) --c;
    while (c + 1 < p.seg_ranges && seg_start(c + 1, p.seg_total, p.seg_ranges) <= lo) ++c;
    int n = 1;
    while (c + n < p.seg_ranges && seg_start(c + n, p.seg_total, p.seg_ranges) < hi) ++n;
    s_c0 = c;
    s_n = n;
    s_part0 = seg_start(c, p.seg_total, p.seg_ranges) < lo ? 1 : 0;
  }
  // the pieces (and, through their own waits, the pair grid) have completed after this
  grid_dependency_wait();
  __syncthreads();
  if (p.status != nullptr && *reinterpret_cast<volatile int32_t*>(p.status) == BCA_ERR_TIMEOUT)
    return;
  if (row >= rows_valid) return;
  const int c0 = s_c0, n = s_n;
  // piece i: slot 2 (c0 + i) + part (part 1 only for the first, when it continues a range)
  auto slot_of = [&](int i) {
    return p.seg_ws + static_cast<size_t>(2 * (c0 + i) + (i == 0 ? s_part0 : 0)) * kSegSlotFloats;
  };
  const size_t o_off = static_cast<size_t>(qi * 32 + quarter * 8) * kBlockM + row;   // float4 units
  const size_t ml_off = static_cast<size_t>(qi * kBlockM + row);                       // float2 units
  float4 o[8];
  float2 ml;
  {
    const float* s0 = slot_of(0);
    ml = __ldcg(reinterpret_cast<const float2*>(s0 + kSegSlotO) + ml_off);
#pragma unroll
    for (int g = 0; g < 8; ++g) o[g] = __ldcg(reinterpret_cast<const float4*>(s0) + o_off + g * kBlockM);
  }
  float acc[32];
#pragma unroll
  for (int x = 0; x < 32; ++x) acc[x] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  bool failed = false;
  for (int i = 0; i < n; ++i) {
    float4 o_next[8];
    float2 ml_next = ml;
    if (i + 1 < n) {
      const float* sn = slot_of(i + 1);
      ml_next = __ldcg(reinterpret_cast<const float2*>(sn + kSegSlotO) + ml_off);
#pragma unroll
      for (int g = 0; g < 8; ++g)
        o_next[g] = __ldcg(reinterpret_cast<const float4*>(sn) + o_off + g * kBlockM);
    }
    failed = failed || ml.y < 0.f;   // the pair failed validation (reported by its pieces)
    const float m_new = fmaxf(m_run, ml.x);
    const float a_old = ex2_approx(m_run - m_new), a = ex2_approx(ml.x - m_new);
    l_run = l_run * a_old + ml.y * a;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      acc[4 * g] = acc[4 * g] * a_old + o[g].x * a;
      acc[4 * g + 1] = acc[4 * g + 1] * a_old + o[g].y * a;
      acc[4 * g + 2] = acc[4 * g + 2] * a_old + o[g].z * a;
      acc[4 * g + 3] = acc[4 * g + 3] * a_old + o[g].w * a;
    }
    m_run = m_new;
    if (i + 1 < n) {
#pragma unroll
      for (int g = 0; g < 8; ++g) o[g] = o_next[g];
      ml = ml_next;
    }
  }
  if (failed) return;
  const float inv_l = 1.f / l_run;
  const int r = q_seq0 + m * kBlockM + row;
  if (!BCA_IN_BOUNDS(p.status, r >= 0 && r < p.total_q && h < p.num_heads)) return;
  uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(r) * p.num_heads + h) * kHeadDim +
                                        quarter * 32);
#pragma unroll
  for (int x = 0; x < 4; ++x)
    dst[x] = make_uint4(pack_bf16x2(acc[8 * x] * inv_l, acc[8 * x + 1] * inv_l),
                        pack_bf16x2(acc[8 * x + 2] * inv_l, acc[8 * x + 3] * inv_l),
                        pack_bf16x2(acc[8 * x + 4] * inv_l, acc[8 * x + 5] * inv_l),
                        pack_bf16x2(acc[8 * x + 6] * inv_l, acc[8 * x + 7] * inv_l));
  if (quarter == 0)
    p.lse[static_cast<size_t>(h) * p.total_q + r] = (m_run + log2f(l_run)) * 0.69314718055994530942f;
}

// ---- host side ---------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Packed [tokens, H, 128] bf16: dims (d, head, token); box (64, 1, 128).
bool encode_packed(CUtensorMap* m, const void* base, int num_heads, int64_t tokens) {
  auto fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(num_heads),
                        static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim * 2),
                           static_cast<cuuint64_t>(num_heads) * kHeadDim * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kBlockN)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One layer of the cache, [H][capacity][128] bf16: dims (d, token, head); box (64, 128, 1).
bool encode_cache(CUtensorMap* m, const void* base, int num_heads, int64_t capacity) {
  auto fn = get_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(capacity),
                        static_cast<cuuint64_t>(num_heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim * 2),
                           static_cast<cuuint64_t>(capacity) * kHeadDim * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBlockN), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sms() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 1;
  }
  return sms;
}

// Balanced decode tail.  The pairs of a last, partly filled wave (all pairs when
// there are fewer than SMs) are laid end to end, nkv key tiles each, and cut into
// `ranges` equal ranges, one per SM: at least kMinSegTiles key tiles per range and
// fewer pairs than ranges (so a range crosses at most one pair boundary, and a
// piece lies inside one pair).  Only when a range plus kSegOverheadTiles is shorter
// than what the wave costs otherwise: 0.6 of a pair's key tiles as key-split
// single tiles (a wave at most half full), else a whole pair.  The overhead, in
// key-tile iterations of a pair (set-up and partial rows of up to two pieces per
// SM, and the merge), is measured: on the two-reference edit decode (56 pairs of
// 98 tiles, 36 per range) the balanced tail saved 13 us over the key-split one,
// on the text-to-image decode (56 pairs of 34 tiles, 12.5 per range) it lost 5 us.
constexpr int kMinSegTiles = 8;
constexpr int kSegOverheadTiles = 16;

struct TailPlan {
  int64_t split_from;   // first pair of the tail
  int64_t pairs;
  int ranges;
  int nkv;
  int64_t total;
  int n_short;          // ranges that cross a pair boundary
  uint16_t order[kMaxSegRanges];
};

bool plan_decode_tail(int64_t items, int nkv, TailPlan* tp) {
  const int sms = device_sms();
  if (items <= 0 || nkv <= 0) return false;
  const int64_t pairs = items % sms;
  if (pairs == 0) return false;
  const int64_t total = pairs * nkv;
  const int ranges = static_cast<int>(std::min<int64_t>(std::min(sms, kMaxSegRanges),
                                                        total / kMinSegTiles));
  if (ranges <= pairs) return false;
  const double per_range = static_cast<double>(total) / ranges;
  const double otherwise = 2 * pairs <= sms ? 0.6 * nkv : static_cast<double>(nkv);
  if (per_range + kSegOverheadTiles >= otherwise) return false;
  tp->split_from = items - pairs;
  tp->pairs = pairs;
  tp->ranges = ranges;
  tp->nkv = nkv;
  tp->total = total;
  // ranges with two parts, by ascending length of the longer one: their shorter
  // parts then launch longest first, after every longer part (an SM whose longer
  // part was short frees first; the hardware need not give it that range's other
  // part, and a per-CTA timeline showed it mostly does not, at little cost)
  int64_t longer[kMaxSegRanges];
  int n = 0;
  for (int c = 0; c < ranges; ++c) {
    int64_t a0, a1, b0, b1;
    seg_piece(c, 0, total, ranges, nkv, a0, a1);
    seg_piece(c, 1, total, ranges, nkv, b0, b1);
    if (b1 > b0) {
      longer[c] = std::max(a1 - a0, b1 - b0);
      tp->order[n++] = static_cast<uint16_t>(c);
    }
  }
  std::stable_sort(tp->order, tp->order + n,
                   [&](uint16_t x, uint16_t y) { return longer[x] < longer[y]; });
  tp->n_short = n;
  return true;
}

}  // namespace

size_t decode_tail_workspace_bytes(int batch, int num_heads, int max_seqlen_q, int max_prefix) {
  if (batch <= 0 || num_heads <= 0 || max_seqlen_q <= 0 || max_prefix < 0) return 0;
  const int tiles = (max_seqlen_q + kBlockM - 1) / kBlockM;
  const int64_t items = static_cast<int64_t>(num_heads) * ((tiles + 1) / 2) * batch;
  const int nkv = (max_prefix + kBlockN - 1) / kBlockN + tiles;
  TailPlan tp;
  if (!plan_decode_tail(items, nkv, &tp)) return 0;
  return static_cast<size_t>(2 * tp.ranges) * kSegSlotBytes;
}

int launch_attention(const AttnLaunch& a, bool decode, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tk2, tv2, to;
  bool ok = encode_packed(&tq, a.q, a.num_heads, a.total_q) &&
            encode_packed(&to, a.out, a.num_heads, a.total_q);
  if (!decode) {
    ok = ok && encode_packed(&tk, a.k, a.num_heads, a.total_k) &&
         encode_packed(&tv, a.v, a.num_heads, a.total_k);
    if (a.cache_k != nullptr) {   // cache append: the store maps over one cache layer
      const int64_t map_cap = a.capacity > 0 ? a.capacity : 1;
      ok = ok && encode_cache(&tk2, a.cache_k, a.num_heads, map_cap) &&
           encode_cache(&tv2, a.cache_v, a.num_heads, map_cap);
    } else {
      tk2 = tk;
      tv2 = tv;
    }
  } else {
    const int64_t map_cap = a.capacity > 0 ? a.capacity : 1;
    ok = ok && encode_cache(&tk, a.k, a.num_heads, map_cap) &&
         encode_cache(&tv, a.v, a.num_heads, map_cap) &&
         encode_packed(&tk2, a.k2, a.num_heads, a.total_q) &&
         encode_packed(&tv2, a.v2, a.num_heads, a.total_q);
  }
  if (!ok) return BCA_ERR_CUDA;

  FwdParams p{};
  p.num_heads = a.num_heads;
  p.total_q = a.total_q;
  p.total_k = a.total_k;
  p.tiles_per_seq = a.tiles_per_seq;
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  p.capacity = a.capacity;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.row_end = a.row_end;
  p.tiles = a.tiles;
  p.cu_prefix = a.cu_prefix;
  p.page_table = a.page_table;
  p.max_pages = a.max_pages;
  p.batch = a.batch;
  p.cache_k = static_cast<__nv_bfloat16*>(a.cache_k);
  p.cache_v = static_cast<__nv_bfloat16*>(a.cache_v);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.status = a.status;

  if (!decode) {
    const int mode = a.cache_k != nullptr && a.page_table != nullptr ? 1 : 0;   // paged append
    using Kernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap,
                            const CUtensorMap, const CUtensorMap, const CUtensorMap,
                            const FwdParams);
    const Kernel kernels[2] = {attn_fwd_kernel<false, false, false>,
                               attn_fwd_kernel<false, false, true>};
    static bool attr_set[2] = {false, false};
    if (!attr_set[mode]) {
      if (cudaFuncSetAttribute(kernels[mode], cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmemBytes)) != cudaSuccess)
        return BCA_ERR_CUDA;
      attr_set[mode] = true;
    }
    // Groups of 8 heads (about 50 MB of K/V at 12.5k keys, well inside L2), else
    // of the largest divisor of the head count down to 4, else one group: every
    // group is full, so the kernel needs no bound check (which measured slower).
    int per_group = a.num_heads;
    for (int d = 8; d >= 4; --d) {
      if (a.num_heads > d && a.num_heads % d == 0) {
        per_group = d;
        break;
      }
    }
    int groups = a.num_heads / per_group;
    if (static_cast<int64_t>(a.batch) * groups > 65535) {
      per_group = a.num_heads;
      groups = 1;
    }
    p.head_groups = groups;
    // The pair CTAs of a last, partly filled wave become key-split single-tile
    // items, two CTAs each, in a second grid that may start as soon as every pair
    // CTA has started.  They are the pairs with the highest pair index (the cheapest:
    // row ends never decrease along a sequence) across all head groups, not the last
    // CTAs in launch order (the cheapest pairs of the last group): on the
    // text-to-image layer that is all 32 two-tile text pairs and 56 image pairs,
    // against 80 image pairs and 8 text pairs, whose 160 heavy split items did not
    // fit one wave of 152 SMs.  The pair grid keeps its head groups outermost, so
    // that the CTAs in flight share the K/V of a few heads in L2.
    // Only when at least two full waves of pair CTAs keep their pairs: before every
    // pair CTA has started, one of those must have ended, which it cannot do before
    // the schedule prep has completed; the split grid reads the prep's records
    // without waiting for it.
    // And only for grids of at most four waves: a split item does its keys ~40%
    // slower than a pair (two K/V streams, its own set-up), which the last wave's
    // idle SMs pay back in a short grid (text-to-image layer: 226 -> 213 us) but not
    // in a long one (two-reference edit, 10 waves: 1059 -> 1067 us).
    const int sms = device_sms();
    const int pairs = (a.tiles_per_seq + 1) / 2;
    const int64_t total = static_cast<int64_t>(per_group) * pairs * a.batch * groups;
    const int64_t tail = total % sms;
    const bool split = tail > 0 && total - tail >= 2 * static_cast<int64_t>(sms) &&
                       total <= 4 * static_cast<int64_t>(sms);
    p.prefill_split_from = split ? total - tail : total;
    p.prefill_x = per_group;
    p.prefill_y = pairs;
    // A programmatic dependent of the schedule prep that every caller launches just
    // before this grid on the same stream: its CTAs start while the prep runs and
    // wait for it only where they read its tile records.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(per_group, pairs, a.batch * groups);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernels[mode], tq, tk, tv, tk2, tv2, to, p) != cudaSuccess)
      return BCA_ERR_CUDA;
    if (split) {
      static bool split_attr = false;
      if (!split_attr) {
        if (cudaFuncSetAttribute(attn_fwd_kernel<false, true, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes)) != cudaSuccess)
          return BCA_ERR_CUDA;
        split_attr = true;
      }
      cfg.gridDim = dim3(static_cast<unsigned>(2 * tail), 1, 1);   // the pair grid's dependent
      if (cudaLaunchKernelEx(&cfg, attn_fwd_kernel<false, true, false>, tq, tk, tv, tk2, tv2, to,
                             p) != cudaSuccess)
        return BCA_ERR_CUDA;
    }
    const cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
  }
  // Decode: equal-cost pair items.  The pairs of a last, partly filled wave run
  // as a balanced tail when the caller gave a workspace for it (pieces, then their
  // merge); without one, when that wave would be at most half full, they become
  // key-split single-tile items (two CTAs each, about 0.6 of a pair's time).
  // Either runs as a second grid that may start as the pair grid drains.
  const int sms = device_sms();
  const int pps = (a.tiles_per_seq + 1) / 2;
  const int64_t items = static_cast<int64_t>(a.num_heads) * pps * a.batch;
  TailPlan tp;
  const int nkv = (a.max_prefix + kBlockN - 1) / kBlockN + a.tiles_per_seq;
  const bool balanced = a.tail_ws != nullptr && plan_decode_tail(items, nkv, &tp) &&
                        a.tail_ws_bytes >= static_cast<size_t>(2 * tp.ranges) * kSegSlotBytes;
  const int64_t tail = items % sms;
  const int64_t split_from =
      balanced ? tp.split_from : ((tail > 0 && 2 * tail <= sms) ? items - tail : items);
  const int64_t n_second = balanced ? tp.ranges + tp.n_short : 2 * (items - split_from);
  if (split_from > 0x7fffffff || n_second > 0x7fffffff) return BCA_ERR_UNSUPPORTED;
  p.decode_pairs_per_seq = pps;
  p.decode_split_from = static_cast<int>(split_from);
  if (balanced) {
    p.seg_ranges = tp.ranges;
    p.seg_nkv = tp.nkv;
    p.seg_total = tp.total;
    p.seg_ws = static_cast<float*>(a.tail_ws);
    for (int i = 0; i < tp.n_short; ++i) p.seg_order[i] = tp.order[i];
  }
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_fwd_kernel<true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(attn_fwd_kernel<true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(attn_fwd_kernel<true, false, false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess)
      return BCA_ERR_CUDA;
    attr_set = true;
  }
  if (split_from > 0) {
    const dim3 grid(static_cast<unsigned>(split_from), 1, 1);
    attn_fwd_kernel<true, false><<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, tk2, tv2, to, p);
    if (cudaGetLastError() != cudaSuccess) return BCA_ERR_CUDA;
  }
  if (n_second > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_second), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = split_from > 0 ? 1 : 0;
    const cudaError_t e =
        balanced ? cudaLaunchKernelEx(&cfg, attn_fwd_kernel<true, false, false, true>, tq, tk, tv,
                                      tk2, tv2, to, p)
                 : cudaLaunchKernelEx(&cfg, attn_fwd_kernel<true, true>, tq, tk, tv, tk2, tv2, to, p);
    if (e != cudaSuccess) return BCA_ERR_CUDA;
    if (balanced) {
      // the merge, a programmatic dependent of the pieces
      cfg.gridDim = dim3(static_cast<unsigned>(8 * tp.pairs), 1, 1);   // (pair, tile, quarter)
      cfg.blockDim = dim3(kMergeThreads, 1, 1);
      cfg.dynamicSmemBytes = 0;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, seg_merge_kernel, p) != cudaSuccess) return BCA_ERR_CUDA;
    }
  }
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? BCA_OK : BCA_ERR_CUDA;
}

}  // namespace bca

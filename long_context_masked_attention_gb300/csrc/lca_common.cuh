// lca_common.cuh — structures shared by the host planner and the kernels, and
// the one device mask predicate that every kernel (materializer, tile
// classifier, forward, backward) evaluates.
//
// The mask families are the ones the LongCA-bench review lists (三 技术架构,
// 掩码模式分类); the page names them without formulas, so each family is
// encoded here by the plainest reading (see the lca_mask_kind comments in
// lca_attn.h).  For every family except the block-sparse ones, the keys a
// query row attends form at most two intervals of the segment's key axis;
// the kernels turn those into 32-column bit masks only on partially masked
// tiles.
#pragma once
#include <cstdint>

namespace lca {

constexpr int kTile = 128;  // query and key tile edge
constexpr int kHeadDim = 128;

enum MaskKind : int {
  kFull = 0,
  kCausal = 1,
  kSliding = 2,
  kCausalSliding = 3,
  kDoc = 4,
  kCausalDoc = 5,
  kSharedQuestion = 6,
  kGlobalSliding = 7,
  kCausalBlockwise = 8,
  kPrefixLmCausal = 9,
  kPrefixLmDoc = 10,
  kBlockCausalDoc = 11,
  kBlockSparseUniform = 12,
  kBlockSparseVariable = 13,
  kFlashMask = 14,
};

enum TileClass : uint32_t { kTileEmpty = 0, kTileFull = 1, kTilePartial = 2 };
// Flags a PARTIAL tile's class byte may carry above its class (bits 0-1): no
// attended cell in query rows [0, 64) / [64, 128) of the tile.
constexpr uint32_t kHalf0Empty = 4, kHalf1Empty = 8;

// Status codes written to the device status word (mirror lca_status).
constexpr int kStatusTimeout = 5;
constexpr int kStatusDeviceArg = 6;

struct SegInfo {  // 32 bytes
  int q_off, q_len, k_off, k_len;
  int prefix;  // PREFIX_LM_DOC prefix of this segment
  int kg;      // key group index
  int nk;      // number of 128-key tiles = ceil(k_len / 128)
  int pad;
};

struct KeyGroup {  // 32 bytes
  int k_off, k_len;        // k_len = longest member's k_len
  int seg_begin, seg_end;  // members: kg_segs[seg_begin, seg_end)
  int kt_start;            // first dK/dV unit row of this group
  int pairs;               // sum of members' 128-row query tiles
  long long entry_off;     // offset of this group's dK/dV entries (per map head)
};

struct MaskCtx {
  int kind;
  int wl, wr, ng, prefix, block;
  int n_parts;       // number of part bounds (SHARED_QUESTION)
  const int* parts;  // device copy of the part bounds
  // block-sparse
  int q_block, kv_block;
  int n_qb, n_kb, words;  // words = ceil(n_kb / 32)
  int hm_count;           // heads_in_map (1 or Hq)
  const uint32_t* keep;   // [hm][n_qb][words] bitmap built from the CSR
  const int* qb_of;       // variable: query block of each global row [Tq]
  const int* kb_of;       // variable: key block of each global key [Tk]
  const int* kb_start;    // variable: key block bounds [n_kb + 1]
  const int* qb_start;    // variable: query block bounds [n_qb + 1]
  const int4* cols;       // FlashMask: {lts, lte, uts, ute} per global key [Tk]
  // uniform block map whose blocks and segment starts are multiples of 32:
  // every 32 rows x 32 keys of a tile (a warp's rows, a 32-column chunk)
  // then lie in one (query block, key block) pair
  int aligned;
  // variable block map: per (map head, query block, key-group key tile) one
  // word of four chunk bytes (see vchunk_bits); vkt = first key tile of each
  // key group in that numbering, vrk = key tiles over all groups
  const uint32_t* vchunk;
  const int* vkt;
  int vrk;
};

// Mask forms the attention kernels are compiled for: the interval families
// and generic block maps (mask words per row), FlashMask's column bounds,
// and aligned uniform block maps (one keep bit per warp and 32-key chunk).
enum MaskForm : int { kFormSpans = 0, kFormCols = 1, kFormBlocks = 2 };

__host__ __device__ __forceinline__ bool is_block_sparse(int kind) {
  return kind == kBlockSparseUniform || kind == kBlockSparseVariable;
}

// Largest s in [0, n) with start[s] <= x (start non-decreasing, start[0] = 0).
__device__ __forceinline__ int find_bucket(const int* __restrict__ start, int n, int x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (start[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ int floordiv_i(int a, int b) { return (a >= 0) ? a / b : -((-a + b - 1) / b); }

// Keys attended by one query row, as [a0, b0) U [a1, b1), segment-relative,
// clipped to [0, k_len).  Rows outside [0, q_len) attend nothing.
struct Span {
  int a0, b0, a1, b1;
};

__device__ __forceinline__ Span row_span(const MaskCtx& m, const SegInfo& sg, int i) {
  Span s{0, 0, 0, 0};
  if (i < 0 || i >= sg.q_len) return s;
  const int K = sg.k_len;
  const int ie = i + (sg.k_len - sg.q_len);  // bottom-right aligned query position
  switch (m.kind) {
    case kFull:
    case kDoc:
      s.b0 = K;
      break;
    case kCausal:
    case kCausalDoc:
      s.b0 = ie + 1;
      break;
    case kSliding:
      s.a0 = ie - m.wl;
      s.b0 = ie + m.wr + 1;
      break;
    case kCausalSliding:
      s.a0 = ie - m.wl;
      s.b0 = ie + 1;
      break;
    case kSharedQuestion: {
      if (ie < 0) break;
      int p = 0;  // part holding position ie: largest p with parts[p] <= ie
      for (int t = 1; t < m.n_parts; ++t) p = (m.parts[t] <= ie) ? t : p;
      if (p == 0) {
        s.b0 = ie + 1;
      } else {
        s.b0 = m.parts[1];
        s.a1 = m.parts[p];
        s.b1 = ie + 1;
      }
      break;
    }
    case kGlobalSliding:
      if (ie < m.ng) {
        s.b0 = K;
      } else {
        s.b0 = m.ng;
        s.a1 = ie - m.wl;
        s.b1 = ie + m.wr + 1;
      }
      break;
    case kCausalBlockwise: {
      if (ie < 0) break;
      const int blk = ie / m.block, last = (K - 1) / m.block;
      s.a0 = (blk == last) ? 0 : blk * m.block;
      s.b0 = ie + 1;
      break;
    }
    case kPrefixLmCausal:
      s.b0 = max(m.prefix, ie + 1);
      break;
    case kPrefixLmDoc:
      s.b0 = max(sg.prefix, ie + 1);
      break;
    case kBlockCausalDoc:
      s.b0 = (floordiv_i(ie, m.block) + 1) * m.block;
      break;
    default:
      break;
  }
  s.a0 = max(s.a0, 0);
  s.b0 = min(s.b0, K);
  s.a1 = max(s.a1, 0);
  s.b1 = min(s.b1, K);
  return s;
}

// Bits of [a, b) inside the 32 columns [j0, j0 + 32).
__device__ __forceinline__ uint32_t range_bits(int a, int b, int j0) {
  const int lo = max(a - j0, 0), hi = min(b - j0, 32);
  if (hi <= lo) return 0u;
  const uint32_t upper = (hi >= 32) ? 0xFFFFFFFFu : ((1u << hi) - 1u);
  const uint32_t lower = (1u << lo) - 1u;
  return upper & ~lower;
}

__device__ __forceinline__ uint32_t span_bits(const Span& s, int j0) {
  return range_bits(s.a0, s.b0, j0) | range_bits(s.a1, s.b1, j0);
}

__device__ __forceinline__ bool span_covers(const Span& s, int c0, int c1) {
  const bool e0 = s.a0 < s.b0, e1 = s.a1 < s.b1;
  if (e0 && s.a0 <= c0 && s.b0 >= c1) return true;
  if (e1 && s.a1 <= c0 && s.b1 >= c1) return true;
  if (e0 && e1 && s.a1 <= s.b0 && s.a0 <= s.b1) {
    const int lo = min(s.a0, s.a1), hi = max(s.b0, s.b1);
    if (lo <= c0 && hi >= c1) return true;
  }
  return false;
}

__device__ __forceinline__ bool span_hits(const Span& s, int c0, int c1) {
  return (s.a0 < s.b0 && s.a0 < c1 && s.b0 > c0) || (s.a1 < s.b1 && s.a1 < c1 && s.b1 > c0);
}

__device__ __forceinline__ int span_count(const Span& s) {
  const int n0 = max(0, s.b0 - s.a0), n1 = max(0, s.b1 - s.a1);
  const int lo = max(s.a0, s.a1), hi = min(s.b0, s.b1);
  const int both = (n0 > 0 && n1 > 0) ? max(0, hi - lo) : 0;
  return n0 + n1 - both;
}

// Work item w of a query-major list: `rows` cost-sorted rows, each run for
// `expand` heads.  Rows are taken in groups of `group`, and a group's rows
// run head by head, so that the items in flight at once cover a few heads
// (K/V tiles shared in L2 when every head has its own K/V) while the order
// stays longest first up to the cost spread inside a group.  group = 1 is
// the plain order: row by row, all heads of a row together.
__device__ __forceinline__ void item_of(int w, int rows, int expand, int group, int& row, int& head) {
  const int base = (w / (group * expand)) * group;
  const int n = min(group, rows - base);
  const int local = w - base * expand;
  head = local / n;
  row = base + local % n;
}

// Work item w of a query-major list with one mask map, taken segment by
// segment, head by head, and within a head the segment's rows from last to
// first (the longest first for causal rows): the items in flight then cover
// a few heads of one segment, whose K/V stays in L2 when every head has its
// own K/V.  qstart = row prefix over segments; row is the list row.
__device__ __forceinline__ void seg_major_item(int w, const int* qstart, int n_seg, int expand, int& row, int& head) {
  const int s = find_bucket(qstart, n_seg, w / expand);
  const int rows_s = qstart[s + 1] - qstart[s];
  const int local = w - qstart[s] * expand;
  head = local / rows_s;
  row = qstart[s] + rows_s - 1 - local % rows_s;
}

// ---------------------------------------------------------------- block-sparse
__device__ __forceinline__ int q_block_of(const MaskCtx& m, int gq) {
  return (m.kind == kBlockSparseUniform) ? gq / m.q_block : m.qb_of[gq];
}
__device__ __forceinline__ int k_block_of(const MaskCtx& m, int gk) {
  return (m.kind == kBlockSparseUniform) ? gk / m.kv_block : m.kb_of[gk];
}
__device__ __forceinline__ int k_block_start(const MaskCtx& m, int kb) {
  return (m.kind == kBlockSparseUniform) ? kb * m.kv_block : m.kb_start[kb];
}
__device__ __forceinline__ bool block_kept(const MaskCtx& m, int hm, int qb, int kb) {
  const uint32_t w = m.keep[(static_cast<size_t>(hm) * m.n_qb + qb) * m.words + (kb >> 5)];
  return (w >> (kb & 31)) & 1u;
}

// 32-column mask chunk for block-sparse maps, row i being in query block
// qb.  A chunk touches at most two key blocks because every key block but
// the last is at least 32 wide.
__device__ __forceinline__ uint32_t block_chunk_bits_q(const MaskCtx& m, const SegInfo& sg, int hm, int i, int j0,
                                                       int qb) {
  if (i < 0 || i >= sg.q_len || j0 >= sg.k_len) return 0u;
  const int jl = min(j0 + 31, sg.k_len - 1);
  const int gj0 = sg.k_off + j0;
  const int kA = k_block_of(m, gj0), kB = k_block_of(m, sg.k_off + jl);
  const bool keepA = block_kept(m, hm, qb, kA);
  uint32_t bits;
  if (kA == kB) {
    bits = keepA ? 0xFFFFFFFFu : 0u;
  } else {
    const bool keepB = block_kept(m, hm, qb, kB);
    const int split = k_block_start(m, kB) - gj0;  // 1..31
    const uint32_t low = (1u << split) - 1u;
    bits = (keepA ? low : 0u) | (keepB ? ~low : 0u);
  }
  return bits & range_bits(0, sg.k_len, j0);
}

__device__ __forceinline__ uint32_t block_chunk_bits(const MaskCtx& m, const SegInfo& sg, int hm, int i, int j0) {
  if (i < 0 || i >= sg.q_len || j0 >= sg.k_len) return 0u;
  return block_chunk_bits_q(m, sg, hm, i, j0, q_block_of(m, sg.q_off + i));
}

// ---------------------------------------------------------------- FlashMask
// Column-wise form: key column j masks the segment rows [lts, lte) U [uts, ute).
__device__ __forceinline__ bool col_masks_row(const int4& b, int i) {
  return (b.x <= i && i < b.y) || (b.z <= i && i < b.w);
}

__device__ __forceinline__ uint32_t flashmask_chunk_bits(const MaskCtx& m, const SegInfo& sg, int i, int j0) {
  if (i < 0 || i >= sg.q_len || j0 >= sg.k_len) return 0u;
  const int n = min(32, sg.k_len - j0);
  const int4* c = m.cols + sg.k_off + j0;
  uint32_t bits = 0u;
  for (int t = 0; t < n; ++t) bits |= col_masks_row(__ldg(c + t), i) ? 0u : (1u << t);
  return bits;
}

// FlashMask, key-major: bit t = row i0 + t of the segment attends key j
// (segment-relative), from that key's column bounds alone.
__device__ __forceinline__ uint32_t flashmask_key_bits(const MaskCtx& m, const SegInfo& sg, int j, int i0) {
  if (j < 0 || j >= sg.k_len) return 0u;
  const int4 b = __ldg(m.cols + sg.k_off + j);
  return range_bits(0, sg.q_len, i0) & ~(range_bits(b.x, b.y, i0) | range_bits(b.z, b.w, i0));
}

// Rows of [r0, r1) that column bounds b mask.
__device__ __forceinline__ int col_masked_rows(const int4& b, int r0, int r1) {
  const int n0 = max(0, min(b.y, r1) - max(b.x, r0));
  const int n1 = max(0, min(b.w, r1) - max(b.z, r0));
  const int both = max(0, min(min(b.y, b.w), r1) - max(max(b.x, b.z), r0));
  return n0 + n1 - both;
}

// The mask predicate: bit t of the result is set iff query row i of the
// segment attends key j0 + t (segment-relative), for query head map index hm.
// kCols selects the FlashMask column form at compile time: the attention
// kernels are instantiated twice so that the column loop never enlarges the
// code the interval and block families run (a branch on the kind, even
// never taken and not inlined, slowed the dK/dV producer measurably).
template <bool kCols>
__device__ __forceinline__ uint32_t mask_bits(const MaskCtx& m, const SegInfo& sg, int hm, int i, int j0) {
  if constexpr (kCols) {
    return flashmask_chunk_bits(m, sg, i, j0);
  } else {
    if (is_block_sparse(m.kind)) return block_chunk_bits(m, sg, hm, i, j0);
    return span_bits(row_span(m, sg, i), j0);
  }
}
// Variable block maps.  The chunk byte of 32 keys starting at j0 for query
// block qb: bit 7 = the chunk's first key block is kept, bit 6 = its second
// one (if it has one) is kept, bits 0-5 = the number of its keys in the first
// block (32 when it lies in one block and inside its key group), or 63 when
// the chunk crosses both a block bound and the group's last key (the mask
// word is then evaluated per row).
__device__ __forceinline__ uint32_t vchunk_byte(const MaskCtx& m, int hm, int qb, int g0, int k_end) {
  if (g0 >= k_end) return 0u;
  const int gl = min(g0 + 31, k_end - 1);
  const int kA = m.kb_of[g0], kB = m.kb_of[gl];
  const uint32_t keepA = block_kept(m, hm, qb, kA) ? 128u : 0u;
  if (kA == kB) return keepA | static_cast<uint32_t>(gl - g0 + 1);
  if (gl != g0 + 31) return 63u;
  const uint32_t keepB = block_kept(m, hm, qb, kB) ? 64u : 0u;
  return keepA | keepB | static_cast<uint32_t>(m.kb_start[kB] - g0);
}

// Mask word of row i for the chunk at j0 from the row's tile word vw.
__device__ __forceinline__ uint32_t vchunk_bits(const MaskCtx& m, const SegInfo& sg, int hm, int i, int j0, int qb,
                                                uint32_t vw) {
  if (i < 0 || i >= sg.q_len || j0 >= sg.k_len) return 0u;
  const uint32_t c8 = (vw >> (8 * ((j0 >> 5) & 3))) & 0xFFu;
  const uint32_t split = c8 & 63u;
  if (split == 63u) return block_chunk_bits_q(m, sg, hm, i, j0, qb);
  const uint32_t low = split >= 32u ? ~0u : (1u << split) - 1u;
  return (((c8 & 128u) ? low : 0u) | ((c8 & 64u) ? ~low : 0u)) & range_bits(0, sg.k_len, j0);
}

// What a row's mask words need that does not change from tile to tile,
// computed once per work item: the interval families' key span, or for a
// block map the row's query block (carried in a0).
__device__ __forceinline__ Span row_mask_ctx(const MaskCtx& m, const SegInfo& sg, int i) {
  if (is_block_sparse(m.kind)) {
    Span s{0, 0, 0, 0};
    if (i >= 0 && i < sg.q_len) s.a0 = q_block_of(m, sg.q_off + i);
    return s;
  }
  return row_span(m, sg, i);
}

// The row's tile word for key tile kt of its segment (variable block maps;
// 0 otherwise): one load per row and tile instead of the block lookups of
// every chunk.
__device__ __forceinline__ uint32_t row_tile_word(const MaskCtx& m, const SegInfo& sg, int hm, int i, int kt,
                                                  const Span& row) {
  if (m.kind != kBlockSparseVariable || i < 0 || i >= sg.q_len) return 0u;
  return m.vchunk[(static_cast<size_t>(hm) * m.n_qb + row.a0) * m.vrk + m.vkt[sg.kg] + kt];
}

// mask_bits from the row's context (row_mask_ctx) and tile word (row_tile_word).
template <bool kCols>
__device__ __forceinline__ uint32_t mask_bits_row(const MaskCtx& m, const SegInfo& sg, int hm, int i, int j0,
                                                  const Span& row, uint32_t vw) {
  if constexpr (kCols) {
    return flashmask_chunk_bits(m, sg, i, j0);
  } else {
    if (m.kind == kBlockSparseVariable) return vchunk_bits(m, sg, hm, i, j0, row.a0, vw);
    if (is_block_sparse(m.kind)) return block_chunk_bits_q(m, sg, hm, i, j0, row.a0);
    return span_bits(row, j0);
  }
}
// Any family, chosen at run time (planning and test kernels).
__device__ __forceinline__ uint32_t mask_bits_any(const MaskCtx& m, const SegInfo& sg, int hm, int i, int j0) {
  return (m.kind == kFlashMask) ? mask_bits<true>(m, sg, hm, i, j0) : mask_bits<false>(m, sg, hm, i, j0);
}

// Class byte from the attended-cell facts of a tile (see classify_tile_warp).
__device__ __forceinline__ uint32_t tile_class(bool any0, bool any1, bool all, bool inside) {
  if (!any0 && !any1) return kTileEmpty;
  if (all && inside) return kTileFull;
  return kTilePartial | (any0 ? 0u : kHalf0Empty) | (any1 ? 0u : kHalf1Empty);
}

// Class of a 128x128 tile of a block-sparse map, computed by one thread: the
// (query block, key block) pairs the tile overlaps are few (at most 5 x 5
// for blocks of 32 or more keys and rows), so a thread reads their keep bits
// itself and a warp classifies 32 tiles at once.
__device__ __forceinline__ uint32_t classify_block_tile(const MaskCtx& m, const SegInfo& sg, int hm, int r0, int c0) {
  const int r1 = min(r0 + kTile, sg.q_len), c1 = min(c0 + kTile, sg.k_len);
  if (r1 <= r0 || c1 <= c0) return kTileEmpty;
  const bool inside = (r0 + kTile <= sg.q_len) && (c0 + kTile <= sg.k_len);
  const int rm = min(r0 + kTile / 2, r1);  // first row of the second half (r1 if it has none)
  const int qbA = q_block_of(m, sg.q_off + r0), qbB = q_block_of(m, sg.q_off + r1 - 1);
  const int kbA = k_block_of(m, sg.k_off + c0), kbB = k_block_of(m, sg.k_off + c1 - 1);
  const int qbM0 = q_block_of(m, sg.q_off + rm - 1);                    // last block of half 0
  const int qbM1 = (rm < r1) ? q_block_of(m, sg.q_off + rm) : qbB + 1;  // first block of half 1
  bool any0 = false, any1 = false, all = true;
  for (int qb = qbA; qb <= qbB; ++qb) {
    for (int kb = kbA; kb <= kbB; ++kb) {
      const bool kept = block_kept(m, hm, qb, kb);
      any0 |= kept && qb <= qbM0;
      any1 |= kept && qb >= qbM1;
      all &= kept;
    }
  }
  return tile_class(any0, any1, all, inside);
}

// Class of the 128x128 tile with rows [r0, r0+128) and keys [c0, c0+128) of
// one segment: EMPTY if no valid cell is attended, FULL if the tile lies
// inside the segment and every cell is attended, PARTIAL otherwise.  A
// PARTIAL tile also carries kHalf0Empty / kHalf1Empty when no cell of its
// rows [r0, r0+64) / [r0+64, r0+128) inside the segment is attended (the
// dK/dV kernel skips such 64-row steps).  All 32 lanes of the warp must call
// it; every lane gets the result.  (Block-sparse maps: every lane evaluates
// classify_block_tile, the per-thread form the planner uses.)
__device__ __forceinline__ uint32_t classify_tile_warp(const MaskCtx& m, const SegInfo& sg, int hm, int r0, int c0) {
  const int lane = threadIdx.x & 31;
  if (is_block_sparse(m.kind)) return classify_block_tile(m, sg, hm, r0, c0);
  const int r1 = min(r0 + kTile, sg.q_len), c1 = min(c0 + kTile, sg.k_len);
  if (r1 <= r0 || c1 <= c0) return kTileEmpty;
  const bool inside = (r0 + kTile <= sg.q_len) && (c0 + kTile <= sg.k_len);
  const int rm = min(r0 + kTile / 2, r1);  // first row of the second half (r1 if it has none)
  bool any0 = false, any1 = false, all = true;
  if (m.kind == kFlashMask) {
    for (int c = c0 + lane; c < c1; c += 32) {
      const int4 b = __ldg(m.cols + sg.k_off + c);
      const int masked0 = col_masked_rows(b, r0, rm), masked1 = col_masked_rows(b, rm, r1);
      any0 |= masked0 < rm - r0;
      any1 |= masked1 < r1 - rm;
      all &= masked0 == 0 && masked1 == 0;
    }
  } else {
    for (int r = r0 + lane; r < r1; r += 32) {
      const Span s = row_span(m, sg, r);
      const bool hit = span_hits(s, c0, c1);
      if (r < rm) any0 |= hit; else any1 |= hit;
      all &= span_covers(s, c0, c1);
    }
  }
  any0 = __any_sync(0xFFFFFFFFu, any0);
  any1 = __any_sync(0xFFFFFFFFu, any1);
  all = __all_sync(0xFFFFFFFFu, all);
  return tile_class(any0, any1, all, inside);
}

}  // namespace lca

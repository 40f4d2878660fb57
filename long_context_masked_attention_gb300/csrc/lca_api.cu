// lca_api.cu — the C ABI declared in include/lca_attn.h: argument
// validation (always before anything is launched), the workspace layout, the
// host part of the plan (per-segment tile prefixes, key groups), the TMA
// tensor maps, and the launch sequences of the forward and backward passes.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "../../include/lca_attn.h"
#include "lca_internal.h"

namespace lca {

static std::atomic<unsigned long long> g_launches{0};
void note_launches(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n), std::memory_order_relaxed); }

namespace {

thread_local char g_err_detail[256] = "";

lca_status cuda_fail(const char* what, cudaError_t e) {
  snprintf(g_err_detail, sizeof(g_err_detail), "%s: %s", what, cudaGetErrorString(e));
  return LCA_ERR_CUDA;
}

// Profiling ring (lca_set_kernel_events).
struct EventRing {
  void* const* events = nullptr;
  int32_t* phases = nullptr;
  int n_pairs = 0;
  int cursor = 0;
};
EventRing g_ring;

// Per-CTA profile buffer (lca_set_cta_profile): kernel slot k at
// k * kProfCtas records of 8 u64, or null when profiling is off.
unsigned long long* g_prof = nullptr;

// The profile records of kernel slot `k` for the launch about to be made on
// `st` (cleared first, so that CTAs beyond the grid read as zero), or null.
unsigned long long* prof_slot(int k, cudaStream_t st) {
  if (!g_prof) return nullptr;
  unsigned long long* p = g_prof + static_cast<size_t>(k) * kProfCtas * 8;
  if (cudaMemsetAsync(p, 0, sizeof(unsigned long long) * kProfCtas * 8, st) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return p;
}

// Records the opening event of a phase; returns the pair index or -1.
int phase_begin(int phase, cudaStream_t st) {
  if (!g_ring.events || g_ring.n_pairs == 0) return -1;
  const int p = g_ring.cursor;
  g_ring.cursor = (g_ring.cursor + 1) % g_ring.n_pairs;
  if (g_ring.phases) g_ring.phases[p] = phase;
  // a failed record must not leak into the call's own error checks
  if (cudaEventRecord(static_cast<cudaEvent_t>(g_ring.events[2 * p]), st) != cudaSuccess) (void)cudaGetLastError();
  return p;
}
void phase_end(int p, cudaStream_t st) {
  if (p < 0) return;
  if (cudaEventRecord(static_cast<cudaEvent_t>(g_ring.events[2 * p + 1]), st) != cudaSuccess)
    (void)cudaGetLastError();
}

constexpr size_t kAlign = 256;
constexpr size_t kMaxPartialSlots = 512;  // 64 MiB of f32 dK/dV partial sums at most
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------ host plan
struct HostPlan {
  int Tq = 0, Tk = 0, Hq = 0, Hkv = 0, G = 1, n_seg = 0;
  float scale = 0.f;
  int kind = 0;
  int hm_count = 1;
  std::vector<SegInfo> segs;
  std::vector<KeyGroup> kgs;
  std::vector<int> kg_segs, q256_start, q128_start, kt_start;
  std::vector<long long> fwd_off, dq_off;
  int R256 = 0, R128 = 0, RK = 0;
  long long fwd_per_hm = 0, dq_per_hm = 0, dkv_per_hm = 0;
  int max_q_len = 0;
  bool fwd_pair = false;  // forward items pair two query heads (see validate)
  std::vector<std::pair<int, int>> q_gaps, k_gaps;  // [start, len)
  // mask parameters
  MaskCtx mask{};
  std::vector<int> parts, qb_bounds, kb_bounds;
  const int* blk_row_ptr = nullptr;
  const int* blk_col_idx = nullptr;
  long long blk_nnz = 0;
};

struct Layout {
  size_t status = 0, counters = 0, hist = 0, acc = 0;
  size_t blob = 0, blob_bytes = 0;
  // blob-relative offsets
  size_t b_segs = 0, b_q256 = 0, b_q128 = 0, b_fwdoff = 0, b_dqoff = 0, b_kgs = 0, b_kgsegs = 0, b_kt = 0,
         b_parts = 0, b_qbb = 0, b_kbb = 0;
  size_t keep = 0, keep_bytes = 0, qb_of = 0, kb_of = 0, vchunk = 0;
  size_t tcls = 0;
  size_t f_cnt = 0, f_key = 0, f_order = 0, f_ent = 0;
  size_t D = 0, lse2 = 0, q_cnt = 0, q_key = 0, q_order = 0, q_ent = 0, k_ucost = 0, k_key = 0, k_order = 0,
         k_lcnt = 0, k_lsteps = 0, k_ent = 0;
  size_t k_usteps = 0, k_nchunk = 0, k_istart = 0, k_sstart = 0, k_nwork = 0, k_part = 0, k_runfirst = 0, k_runof = 0,
         k_runat = 0;
  int k_max_slots = 0;
  size_t total = 0;
};

lca_status validate(const lca_shape* sh, const lca_mask_desc* md, HostPlan& P) {
  if (!sh || !md) return LCA_ERR_INVALID_ARG;
  if (sh->d != kHeadDim) return LCA_ERR_UNSUPPORTED;
  if (sh->Tq < 0 || sh->Tk < 0 || sh->Hq <= 0 || sh->Hkv <= 0 || sh->n_seg < 0) return LCA_ERR_INVALID_ARG;
  if (sh->Hq % sh->Hkv != 0) return LCA_ERR_INVALID_ARG;
  if (sh->n_seg > 0 && !sh->segs) return LCA_ERR_INVALID_ARG;
  if (!(std::isfinite(sh->scale)) || sh->scale < 0.f) return LCA_ERR_INVALID_ARG;
  if (static_cast<long long>(sh->Hq) * kHeadDim > (1LL << 30)) return LCA_ERR_UNSUPPORTED;
  if (md->kind < LCA_MASK_FULL || md->kind > LCA_MASK_FLASHMASK) return LCA_ERR_INVALID_ARG;
  P.Tq = sh->Tq;
  P.Tk = sh->Tk;
  P.Hq = sh->Hq;
  P.Hkv = sh->Hkv;
  P.G = sh->Hq / sh->Hkv;
  P.n_seg = sh->n_seg;
  P.scale = sh->scale > 0.f ? sh->scale : 1.0f / std::sqrt(static_cast<float>(sh->d));
  P.kind = md->kind;

  // segments
  P.segs.resize(P.n_seg);
  std::vector<std::pair<long long, long long>> qr;
  for (int s = 0; s < P.n_seg; ++s) {
    const lca_segment& g = sh->segs[s];
    if (g.q_off < 0 || g.q_len < 0 || g.k_off < 0 || g.k_len < 0) return LCA_ERR_INVALID_ARG;
    if (static_cast<long long>(g.q_off) + g.q_len > P.Tq) return LCA_ERR_INVALID_ARG;
    if (static_cast<long long>(g.k_off) + g.k_len > P.Tk) return LCA_ERR_INVALID_ARG;
    SegInfo& si = P.segs[s];
    si.q_off = g.q_off;
    si.q_len = g.q_len;
    si.k_off = g.k_off;
    si.k_len = g.k_len;
    si.prefix = 0;
    si.kg = -1;
    si.nk = static_cast<int>(cdiv(g.k_len, kTile));
    si.pad = 0;
    if (g.q_len > 0) qr.push_back({g.q_off, g.q_off + g.q_len});
    P.max_q_len = std::max(P.max_q_len, g.q_len);
  }
  std::sort(qr.begin(), qr.end());
  long long cur = 0;
  for (auto& r : qr) {
    if (r.first < cur) return LCA_ERR_INVALID_ARG;  // overlapping query ranges
    if (r.first > cur) P.q_gaps.push_back({static_cast<int>(cur), static_cast<int>(r.first - cur)});
    cur = r.second;
  }
  if (cur < P.Tq) P.q_gaps.push_back({static_cast<int>(cur), static_cast<int>(P.Tq - cur)});

  // key groups: segments sharing k_off; ranges of different groups must not overlap
  std::map<int, std::vector<int>> by_off;
  for (int s = 0; s < P.n_seg; ++s)
    if (P.segs[s].k_len > 0) by_off[P.segs[s].k_off].push_back(s);
  long long kcur = 0;
  int kt_acc = 0;
  long long dkv_acc = 0;
  P.kt_start.push_back(0);
  for (auto& kv : by_off) {
    KeyGroup kg{};
    kg.k_off = kv.first;
    kg.k_len = 0;
    kg.seg_begin = static_cast<int>(P.kg_segs.size());
    int pairs = 0;
    for (int s : kv.second) {
      kg.k_len = std::max(kg.k_len, P.segs[s].k_len);
      P.segs[s].kg = static_cast<int>(P.kgs.size());
      P.kg_segs.push_back(s);
      pairs += static_cast<int>(cdiv(P.segs[s].q_len, kTile));
    }
    kg.seg_end = static_cast<int>(P.kg_segs.size());
    if (kg.k_off < kcur) return LCA_ERR_INVALID_ARG;  // key ranges of two groups overlap
    if (kg.k_off > kcur) P.k_gaps.push_back({static_cast<int>(kcur), static_cast<int>(kg.k_off - kcur)});
    kcur = static_cast<long long>(kg.k_off) + kg.k_len;
    kg.kt_start = kt_acc;
    kg.pairs = pairs;
    kg.entry_off = dkv_acc;
    const int nk = static_cast<int>(cdiv(kg.k_len, kTile));
    kt_acc += nk;
    dkv_acc += static_cast<long long>(nk) * pairs;
    P.kgs.push_back(kg);
    P.kt_start.push_back(kt_acc);
  }
  if (kcur < P.Tk) P.k_gaps.push_back({static_cast<int>(kcur), static_cast<int>(P.Tk - kcur)});
  P.RK = kt_acc;
  P.dkv_per_hm = dkv_acc;

  // query-side prefixes
  P.q256_start.assign(P.n_seg + 1, 0);
  P.q128_start.assign(P.n_seg + 1, 0);
  P.fwd_off.assign(P.n_seg, 0);
  P.dq_off.assign(P.n_seg, 0);
  long long f = 0, q = 0;
  for (int s = 0; s < P.n_seg; ++s) {
    const long long n256 = cdiv(P.segs[s].q_len, 2 * kTile), n128 = cdiv(P.segs[s].q_len, kTile);
    P.q256_start[s + 1] = P.q256_start[s] + static_cast<int>(n256);
    P.q128_start[s + 1] = P.q128_start[s] + static_cast<int>(n128);
    P.fwd_off[s] = f;
    P.dq_off[s] = q;
    f += n256 * P.segs[s].nk;
    q += n128 * P.segs[s].nk;
  }
  P.R256 = P.q256_start[P.n_seg];
  P.R128 = P.q128_start[P.n_seg];
  P.fwd_per_hm = f;
  P.dq_per_hm = q;

  // mask parameters
  MaskCtx& m = P.mask;
  m.kind = md->kind;
  m.wl = md->window_left;
  m.wr = md->window_right;
  m.ng = md->num_global;
  m.prefix = md->prefix_len;
  m.block = md->block;
  m.hm_count = 1;
  switch (md->kind) {
    case LCA_MASK_SLIDING:
    case LCA_MASK_CAUSAL_SLIDING:
      if (m.wl < 0 || m.wr < 0) return LCA_ERR_INVALID_ARG;
      break;
    case LCA_MASK_GLOBAL_SLIDING:
      if (m.wl < 0 || m.wr < 0 || m.ng < 0) return LCA_ERR_INVALID_ARG;
      break;
    case LCA_MASK_PREFIX_LM_CAUSAL:
      if (m.prefix < 0) return LCA_ERR_INVALID_ARG;
      break;
    case LCA_MASK_PREFIX_LM_DOC:
      if (P.n_seg > 0 && !md->seg_prefix) return LCA_ERR_INVALID_ARG;
      for (int s = 0; s < P.n_seg; ++s) {
        if (md->seg_prefix[s] < 0) return LCA_ERR_INVALID_ARG;
        P.segs[s].prefix = md->seg_prefix[s];
      }
      break;
    case LCA_MASK_CAUSAL_BLOCKWISE:
    case LCA_MASK_BLOCK_CAUSAL_DOC:
      if (m.block < 1) return LCA_ERR_INVALID_ARG;
      break;
    case LCA_MASK_FLASHMASK:
      if (P.Tk > 0 && (!md->col_bounds || (reinterpret_cast<uintptr_t>(md->col_bounds) & 15u) != 0))
        return LCA_ERR_INVALID_ARG;
      m.cols = reinterpret_cast<const int4*>(md->col_bounds);
      break;
    case LCA_MASK_SHARED_QUESTION: {
      const int n = md->n_part_bounds;
      if (!md->part_bounds || n < 2 || n > 64 || md->part_bounds[0] != 0) return LCA_ERR_INVALID_ARG;
      for (int t = 1; t < n; ++t)
        if (md->part_bounds[t] <= md->part_bounds[t - 1]) return LCA_ERR_INVALID_ARG;
      for (int s = 0; s < P.n_seg; ++s)
        if (md->part_bounds[n - 1] < P.segs[s].k_len) return LCA_ERR_INVALID_ARG;
      P.parts.assign(md->part_bounds, md->part_bounds + n);
      m.n_parts = n;
      break;
    }
    case LCA_MASK_BLOCK_SPARSE_UNIFORM:
    case LCA_MASK_BLOCK_SPARSE_VARIABLE: {
      if (md->heads_in_map != 1 && md->heads_in_map != P.Hq) return LCA_ERR_INVALID_ARG;
      if (md->blk_nnz < 0 || !md->blk_row_ptr || (md->blk_nnz > 0 && !md->blk_col_idx)) return LCA_ERR_INVALID_ARG;
      m.hm_count = md->heads_in_map;
      if (md->kind == LCA_MASK_BLOCK_SPARSE_UNIFORM) {
        if (md->q_block < 1 || md->kv_block < 32) return LCA_ERR_INVALID_ARG;
        m.q_block = md->q_block;
        m.kv_block = md->kv_block;
        m.n_qb = static_cast<int>(std::max<long long>(1, cdiv(P.Tq, md->q_block)));
        m.n_kb = static_cast<int>(std::max<long long>(1, cdiv(P.Tk, md->kv_block)));
        m.aligned = (md->q_block % 32 == 0 && md->kv_block % 32 == 0) ? 1 : 0;
        for (int s = 0; s < P.n_seg && m.aligned; ++s)
          if (P.segs[s].q_off % 32 != 0 || P.segs[s].k_off % 32 != 0) m.aligned = 0;
      } else {
        if (!md->qb_bounds || !md->kb_bounds || md->n_qb < 1 || md->n_kb < 1) return LCA_ERR_INVALID_ARG;
        if (md->qb_bounds[0] != 0 || md->kb_bounds[0] != 0) return LCA_ERR_INVALID_ARG;
        for (int t = 1; t <= md->n_qb; ++t)
          if (md->qb_bounds[t] <= md->qb_bounds[t - 1]) return LCA_ERR_INVALID_ARG;
        for (int t = 1; t <= md->n_kb; ++t) {
          if (md->kb_bounds[t] <= md->kb_bounds[t - 1]) return LCA_ERR_INVALID_ARG;
          if (t < md->n_kb && md->kb_bounds[t] - md->kb_bounds[t - 1] < 32) return LCA_ERR_UNSUPPORTED;
        }
        if (md->qb_bounds[md->n_qb] < P.Tq || md->kb_bounds[md->n_kb] < P.Tk) return LCA_ERR_INVALID_ARG;
        m.n_qb = md->n_qb;
        m.n_kb = md->n_kb;
        P.qb_bounds.assign(md->qb_bounds, md->qb_bounds + md->n_qb + 1);
        P.kb_bounds.assign(md->kb_bounds, md->kb_bounds + md->n_kb + 1);
      }
      m.words = (m.n_kb + 31) / 32;
      P.blk_row_ptr = md->blk_row_ptr;
      P.blk_col_idx = md->blk_col_idx;
      P.blk_nnz = md->blk_nnz;
      P.hm_count = m.hm_count;
      break;
    }
    default:
      break;
  }
  // Forward items of 128 rows of two query heads (which read the same KV
  // head and the same mask map) instead of 256 rows of one head, for the
  // families whose rows see few key tiles or tile ranges that shift row by
  // row: the two sub-tiles then share one key-tile list and never wait on
  // each other (measured: 8K windowed and document masks faster in the
  // forward; FULL, CAUSAL and PREFIX_LM_CAUSAL keep 256-row items).
  switch (P.kind) {
    case LCA_MASK_SLIDING:
    case LCA_MASK_CAUSAL_SLIDING:
    case LCA_MASK_GLOBAL_SLIDING:
    case LCA_MASK_DOC:
    case LCA_MASK_CAUSAL_DOC:
    case LCA_MASK_SHARED_QUESTION:
    case LCA_MASK_CAUSAL_BLOCKWISE:
    case LCA_MASK_PREFIX_LM_DOC:
    case LCA_MASK_BLOCK_CAUSAL_DOC:
      P.fwd_pair = P.hm_count == 1 && P.G % 2 == 0;
      break;
    default:
      P.fwd_pair = false;
  }
  return LCA_OK;
}

// Whether the call's K and V (bf16) exceed what L2 keeps for them: then the
// query-major items in flight should cover a few heads of one segment
// (seg_major_item), not every head of every segment as the cost order does.
bool kv_beyond_l2(const HostPlan& P) {
  return static_cast<long long>(P.Tk) * P.Hkv * kHeadDim * 2 * 2 > kKvL2Bytes;
}

Layout make_layout(const HostPlan& P, bool fwd, bool bwd) {
  Layout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.status = take(16);
  L.counters = take(16);
  L.hist = take(3 * kCostBuckets * sizeof(uint32_t));
  L.acc = take(sizeof(unsigned long long) * std::max(1, P.Hq));
  // blob
  size_t b = 0;
  auto btake = [&](size_t bytes) {
    const size_t at = b;
    b = (b + bytes + 15) / 16 * 16;
    return at;
  };
  L.b_segs = btake(sizeof(SegInfo) * P.segs.size());
  L.b_q256 = btake(sizeof(int) * P.q256_start.size());
  L.b_q128 = btake(sizeof(int) * P.q128_start.size());
  L.b_fwdoff = btake(sizeof(long long) * P.fwd_off.size());
  L.b_dqoff = btake(sizeof(long long) * P.dq_off.size());
  L.b_kgs = btake(sizeof(KeyGroup) * P.kgs.size());
  L.b_kgsegs = btake(sizeof(int) * P.kg_segs.size());
  L.b_kt = btake(sizeof(int) * P.kt_start.size());
  L.b_parts = btake(sizeof(int) * P.parts.size());
  L.b_qbb = btake(sizeof(int) * P.qb_bounds.size());
  L.b_kbb = btake(sizeof(int) * P.kb_bounds.size());
  L.blob_bytes = std::max<size_t>(b, 16);
  L.blob = take(L.blob_bytes);
  if (is_block_sparse(P.kind)) {
    L.keep_bytes = sizeof(uint32_t) * static_cast<size_t>(P.mask.hm_count) * P.mask.n_qb * P.mask.words;
    L.keep = take(L.keep_bytes);
    if (P.kind == kBlockSparseVariable) {
      L.qb_of = take(sizeof(int) * std::max(1, P.Tq));
      L.kb_of = take(sizeof(int) * std::max(1, P.Tk));
      L.vchunk =
          take(sizeof(uint32_t) * std::max<size_t>(1, static_cast<size_t>(P.mask.hm_count) * P.mask.n_qb * P.RK));
    }
  }
  const size_t H = static_cast<size_t>(P.hm_count);
  L.tcls = take(std::max<size_t>(1, H * P.dq_per_hm));
  if (fwd) {
    const size_t f_rows = P.fwd_pair ? P.R128 : P.R256;
    const size_t f_ents = static_cast<size_t>(P.fwd_pair ? P.dq_per_hm : P.fwd_per_hm);
    L.f_cnt = take(sizeof(int) * std::max<size_t>(1, H * f_rows));
    L.f_key = take(sizeof(int) * std::max<size_t>(1, H * f_rows));
    L.f_order = take(sizeof(int) * std::max<size_t>(1, H * f_rows));
    L.f_ent = take(sizeof(uint32_t) * std::max<size_t>(1, H * f_ents));
  }
  if (bwd) {
    const size_t hkv_m = (P.hm_count == 1) ? 1 : static_cast<size_t>(P.Hkv);
    L.D = take(sizeof(float) * std::max<size_t>(1, static_cast<size_t>(P.Hq) * P.Tq));
    L.lse2 = take(sizeof(float) * std::max<size_t>(1, static_cast<size_t>(P.Hq) * P.Tq));
    L.q_cnt = take(sizeof(int) * std::max<size_t>(1, H * P.R128));
    L.q_key = take(sizeof(int) * std::max<size_t>(1, H * P.R128));
    L.q_order = take(sizeof(int) * std::max<size_t>(1, H * P.R128));
    L.q_ent = take(sizeof(uint32_t) * std::max<size_t>(1, H * P.dq_per_hm));
    L.k_ucost = take(sizeof(int) * std::max<size_t>(1, hkv_m * P.RK));
    L.k_key = take(sizeof(int) * std::max<size_t>(1, hkv_m * P.RK));
    L.k_order = take(sizeof(int) * std::max<size_t>(1, hkv_m * P.RK));
    L.k_lcnt = take(sizeof(int) * std::max<size_t>(1, H * P.RK));
    L.k_lsteps = take(sizeof(int) * std::max<size_t>(1, H * P.RK));
    L.k_ent = take(sizeof(int2) * std::max<size_t>(1, H * P.dkv_per_hm));
    const size_t n_units = std::max<size_t>(1, hkv_m * P.RK);
    L.k_usteps = take(sizeof(int) * n_units);
    L.k_nchunk = take(sizeof(int) * n_units);
    L.k_istart = take(sizeof(int) * (n_units + 1));
    L.k_sstart = take(sizeof(int) * n_units);
    L.k_nwork = take(2 * sizeof(int));
    L.k_runfirst = take(sizeof(int) * n_units);
    L.k_runof = take(sizeof(int) * n_units);
    L.k_runat = take(sizeof(int) * n_units);
    // partial-sum slots for chunks of split dK/dV units: [slot][dV, dK][128][128] f32
    L.k_max_slots = static_cast<int>(std::min<size_t>(kMaxPartialSlots, 2 * n_units * (P.Hkv / hkv_m)));
    L.k_part = take(sizeof(float) * 2 * kTile * kHeadDim * static_cast<size_t>(L.k_max_slots));
  }
  L.total = o;
  return L;
}

std::vector<uint8_t> make_blob(const HostPlan& P, const Layout& L) {
  std::vector<uint8_t> blob(L.blob_bytes, 0);
  auto put = [&](size_t off, const void* src, size_t bytes) {
    if (bytes) std::memcpy(blob.data() + off, src, bytes);
  };
  put(L.b_segs, P.segs.data(), sizeof(SegInfo) * P.segs.size());
  put(L.b_q256, P.q256_start.data(), sizeof(int) * P.q256_start.size());
  put(L.b_q128, P.q128_start.data(), sizeof(int) * P.q128_start.size());
  put(L.b_fwdoff, P.fwd_off.data(), sizeof(long long) * P.fwd_off.size());
  put(L.b_dqoff, P.dq_off.data(), sizeof(long long) * P.dq_off.size());
  put(L.b_kgs, P.kgs.data(), sizeof(KeyGroup) * P.kgs.size());
  put(L.b_kgsegs, P.kg_segs.data(), sizeof(int) * P.kg_segs.size());
  put(L.b_kt, P.kt_start.data(), sizeof(int) * P.kt_start.size());
  put(L.b_parts, P.parts.data(), sizeof(int) * P.parts.size());
  put(L.b_qbb, P.qb_bounds.data(), sizeof(int) * P.qb_bounds.size());
  put(L.b_kbb, P.kb_bounds.data(), sizeof(int) * P.kb_bounds.size());
  return blob;
}

PlanView make_view(const HostPlan& P, const Layout& L, uint8_t* ws) {
  PlanView v{};
  uint8_t* blob = ws + L.blob;
  v.mask = P.mask;
  v.mask.parts = reinterpret_cast<const int*>(blob + L.b_parts);
  if (is_block_sparse(P.kind)) {
    v.mask.keep = reinterpret_cast<const uint32_t*>(ws + L.keep);
    if (P.kind == kBlockSparseVariable) {
      v.mask.qb_of = reinterpret_cast<const int*>(ws + L.qb_of);
      v.mask.kb_of = reinterpret_cast<const int*>(ws + L.kb_of);
      v.mask.kb_start = reinterpret_cast<const int*>(blob + L.b_kbb);
      v.mask.qb_start = reinterpret_cast<const int*>(blob + L.b_qbb);
      v.mask.vchunk = reinterpret_cast<const uint32_t*>(ws + L.vchunk);
      v.mask.vkt = reinterpret_cast<const int*>(blob + L.b_kt);
      v.mask.vrk = P.RK;
    }
  }
  v.segs = reinterpret_cast<const SegInfo*>(blob + L.b_segs);
  v.n_seg = P.n_seg;
  v.q256_start = reinterpret_cast<const int*>(blob + L.b_q256);
  v.q128_start = reinterpret_cast<const int*>(blob + L.b_q128);
  v.fwd_off = reinterpret_cast<const long long*>(blob + L.b_fwdoff);
  v.dq_off = reinterpret_cast<const long long*>(blob + L.b_dqoff);
  v.kgs = reinterpret_cast<const KeyGroup*>(blob + L.b_kgs);
  v.n_kg = static_cast<int>(P.kgs.size());
  v.kg_segs = reinterpret_cast<const int*>(blob + L.b_kgsegs);
  v.kt_start = reinterpret_cast<const int*>(blob + L.b_kt);
  v.hm_count = P.hm_count;
  v.R256 = P.R256;
  v.R128 = P.R128;
  v.RK = P.RK;
  v.fwd_per_hm = P.fwd_per_hm;
  v.dq_per_hm = P.dq_per_hm;
  v.dkv_per_hm = P.dkv_per_hm;
  v.Tq = P.Tq;
  v.Tk = P.Tk;
  v.Hq = P.Hq;
  v.Hkv = P.Hkv;
  v.G = P.G;
  return v;
}

// ------------------------------------------------------------------ CUDA helpers
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [rows][heads * 128] bf16, 64-column x box_rows boxes, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int rows, int heads, int box_rows) {
  auto fn = encode_fn();
  if (!fn) {
    snprintf(g_err_detail, sizeof(g_err_detail), "cuTensorMapEncodeTiled entry point unavailable");
    return false;
  }
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads) * kHeadDim, static_cast<cuuint64_t>(std::max(rows, 1))};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads) * kHeadDim * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    snprintf(g_err_detail, sizeof(g_err_detail), "cuTensorMapEncodeTiled(rows=%d, heads=%d, box_rows=%d): CUresult %d",
             rows, heads, box_rows, static_cast<int>(r));
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    cuda_fail("cudaDeviceGetAttribute(multiProcessorCount)", e);
    return 0;
  }
  return n;
}

// The backward's dK/dV work runs on a library-owned stream of the highest
// priority, forked from and joined back to the caller's stream by events, so
// that the dQ pass (which does not read dK/dV) runs beside it: its lists are
// built while dK/dV's are, and its persistent CTAs take the SMs that dK/dV
// CTAs leave at the end of their work.  With dK/dV's stream at the higher
// priority, dK/dV's CTAs are placed first when both kernels are ready, so the
// shorter dQ pass fills the tail of the longer one.  One stream per device,
// created on first use; calls that overlap on several caller streams share
// it (their dK/dV parts run one after another).
cudaStream_t side_stream(lca_status& err) {
  static std::mutex mu;
  static cudaStream_t streams[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    err = LCA_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!streams[dev]) {
    int lo = 0, hi = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&streams[dev], cudaStreamNonBlocking, hi);
    if (e != cudaSuccess) {
      err = cuda_fail("cudaStreamCreateWithPriority", e);
      streams[dev] = nullptr;
      return nullptr;
    }
  }
  err = LCA_OK;
  return streams[dev];
}

unsigned long long wait_limit_ns() {
  static unsigned long long v = 0;
  if (!v) {
    const char* e = std::getenv("LCA_WAIT_LIMIT_MS");
    const long long ms = e ? std::atoll(e) : 2000;
    v = static_cast<unsigned long long>(std::max(1LL, ms)) * 1000000ull;
  }
  return v;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Inputs are read through TMA tensor maps and must be device (or managed)
// memory.  Outputs are written with plain stores only, so they may also be
// page-locked host memory that CUDA maps into the device's address space:
// on a GB300 the kernels then store their results straight into the Grace
// host's memory over NVLink-C2C.  Device memory must belong to the device
// that is current for the call (the one the kernels run on): a pointer into
// another GPU's memory would make the kernels fault or read across the link.
// `device_input` says whether `p` is memory the kernels may read;
// `output_address` returns the address the kernels use for an output
// buffer, or nullptr for memory they must not write (another device's,
// pageable host memory, an unknown pointer), which the call refuses before
// launching.
int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return dev;
}

bool device_input(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  if (at.type == cudaMemoryTypeManaged) return true;
  return at.type == cudaMemoryTypeDevice && at.device == current_device();
}

void* output_address(void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (at.type == cudaMemoryTypeManaged) return p;
  if (at.type == cudaMemoryTypeDevice) return at.device == current_device() ? p : nullptr;
  // mapped host memory: the address valid on the current device (null when not mapped for it)
  if (at.type == cudaMemoryTypeHost) return at.devicePointer;
  return nullptr;
}


#define LCA_CUDA(x)                                  \
  do {                                               \
    const cudaError_t e_ = (x);                      \
    if (e_ != cudaSuccess) return cuda_fail(#x, e_); \
  } while (0)

// Common preamble of every entry point that launches: validate, lay out,
// check the workspace, clear the control block, upload the plan and build
// the block maps.
struct Call {
  HostPlan P;
  Layout L;
  PlanView V;
  uint8_t* ws = nullptr;
  cudaStream_t st = nullptr;
};

lca_status prepare(Call& c, const lca_shape* sh, const lca_mask_desc* md, void* ws, size_t ws_bytes, void* stream,
                   bool fwd, bool bwd) {
  lca_status r = validate(sh, md, c.P);
  if (r != LCA_OK) return r;
  c.L = make_layout(c.P, fwd, bwd);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < c.L.total) return LCA_ERR_WORKSPACE;
  if (!device_input(ws)) return LCA_ERR_WORKSPACE;  // counters and lists: device memory only
  c.ws = static_cast<uint8_t*>(ws);
  c.st = static_cast<cudaStream_t>(stream);
  c.V = make_view(c.P, c.L, c.ws);
  return LCA_OK;
}

lca_status upload(Call& c) {
  LCA_CUDA(cudaMemsetAsync(c.ws, 0, c.L.blob, c.st));  // status, counters, histograms, accumulators
  const std::vector<uint8_t> blob = make_blob(c.P, c.L);
  LCA_CUDA(cudaMemcpyAsync(c.ws + c.L.blob, blob.data(), blob.size(), cudaMemcpyHostToDevice, c.st));
  if (is_block_sparse(c.P.kind)) {
    launch_build_block_maps(c.V, reinterpret_cast<const int*>(c.ws + c.L.blob + c.L.b_qbb),
                            reinterpret_cast<const int*>(c.ws + c.L.blob + c.L.b_kbb),
                            reinterpret_cast<uint32_t*>(c.ws + c.L.keep), reinterpret_cast<int*>(c.ws + c.L.qb_of),
                            reinterpret_cast<int*>(c.ws + c.L.kb_of), c.P.blk_row_ptr, c.P.blk_col_idx, c.P.blk_nnz,
                            c.L.keep_bytes, reinterpret_cast<int*>(c.ws + c.L.status), c.st);
    if (c.P.kind == kBlockSparseVariable)
      launch_build_vchunk(c.V, reinterpret_cast<uint32_t*>(c.ws + c.L.vchunk), c.st);
  }
  LCA_CUDA(cudaGetLastError());
  return LCA_OK;
}

// Dropout parameters: threshold t = floor(256 p + 1/2) capped at 255 (t = 0
// turns dropout off), keep probability (256 - t) / 256.
struct Drop {
  int t = 0;
  uint64_t seed = 0;
  float keep = 1.f, inv = 1.f;
};

lca_status parse_dropout(const lca_dropout* d, Drop& out) {
  out = Drop{};
  if (!d) return LCA_OK;
  const double p = d->p;
  if (!(p >= 0.0 && p < 1.0)) return LCA_ERR_INVALID_ARG;  // also rejects NaN
  out.t = std::min(255, static_cast<int>(std::floor(256.0 * p + 0.5)));
  out.seed = d->seed;
  out.keep = static_cast<float>((256 - out.t) / 256.0);
  out.inv = static_cast<float>(256.0 / (256 - out.t));
  return LCA_OK;
}

AttnArgs base_args(const Call& c, const Drop& dr) {
  AttnArgs a{};
  a.pv = c.V;
  a.status = reinterpret_cast<int*>(c.ws + c.L.status);
  a.wait_limit_ns = wait_limit_ns();
  a.scale = c.P.scale;
  a.scale_log2 = c.P.scale * 1.4426950408889634f;
  a.drop_t = dr.t;
  a.drop_inv = dr.inv;
  a.drop_keys = philox_round_keys(dr.seed);
  a.row_group = 1;
  return a;
}

lca_status attn_fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, const lca_shape* shape,
                         const lca_mask_desc* mask, const lca_dropout* dropout, void* workspace,
                         size_t workspace_bytes, void* stream);
lca_status attn_bwd_impl(const void* dout, const void* q, const void* k, const void* v, const void* o,
                         const float* lse, void* dq, void* dk, void* dv, const lca_shape* shape,
                         const lca_mask_desc* mask, const lca_dropout* dropout, void* workspace,
                         size_t workspace_bytes, void* stream);

}  // namespace
}  // namespace lca

using namespace lca;

extern "C" {

const char* lca_status_string(lca_status s) {
  switch (s) {
    case LCA_OK: return "ok";
    case LCA_ERR_INVALID_ARG: return "invalid argument";
    case LCA_ERR_UNSUPPORTED: return "unsupported configuration";
    case LCA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case LCA_ERR_CUDA: return "CUDA call failed";
    case LCA_ERR_TIMEOUT: return "device pipeline wait timed out";
    case LCA_ERR_DEVICE_ARG: return "descriptor data out of range on the device";
  }
  return "unknown status";
}

int32_t lca_version(void) { return 104; }

lca_status lca_set_kernel_events(void* const* events, int32_t n_events, int32_t* phases) {
  if (events && (n_events < 2 || (n_events & 1))) return LCA_ERR_INVALID_ARG;
  for (int32_t i = 0; events && i < n_events; ++i)
    if (!events[i]) return LCA_ERR_INVALID_ARG;  // every handle must be a created event
  g_ring.events = events;
  g_ring.phases = phases;
  g_ring.n_pairs = events ? n_events / 2 : 0;
  g_ring.cursor = 0;
  return LCA_OK;
}

lca_status lca_set_cta_profile(void* buf, size_t bytes) {
  if (!buf) {
    g_prof = nullptr;
    return LCA_OK;
  }
  if (bytes < LCA_CTA_PROFILE_BYTES || (reinterpret_cast<uintptr_t>(buf) & 7u) != 0 || !device_input(buf))
    return LCA_ERR_INVALID_ARG;
  g_prof = static_cast<unsigned long long*>(buf);
  return LCA_OK;
}

const char* lca_last_error_detail(void) { return g_err_detail; }

uint64_t lca_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

lca_status lca_workspace_size(const lca_shape* shape, const lca_mask_desc* mask, int for_bwd, size_t* bytes) {
  if (!bytes) return LCA_ERR_INVALID_ARG;
  HostPlan P;
  const lca_status r = validate(shape, mask, P);
  if (r != LCA_OK) return r;
  *bytes = make_layout(P, true, for_bwd != 0).total;
  return LCA_OK;
}

lca_status lca_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const lca_shape* shape,
                        const lca_mask_desc* mask, void* workspace, size_t workspace_bytes, void* stream) {
  return attn_fwd_impl(q, k, v, o, lse, shape, mask, nullptr, workspace, workspace_bytes, stream);
}

lca_status lca_attn_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                                const lca_shape* shape, const lca_mask_desc* mask, const lca_dropout* dropout,
                                void* workspace, size_t workspace_bytes, void* stream) {
  return attn_fwd_impl(q, k, v, o, lse, shape, mask, dropout, workspace, workspace_bytes, stream);
}

lca_status lca_attn_bwd(const void* dout, const void* q, const void* k, const void* v, const void* o,
                        const float* lse, void* dq, void* dk, void* dv, const lca_shape* shape,
                        const lca_mask_desc* mask, void* workspace, size_t workspace_bytes, void* stream) {
  return attn_bwd_impl(dout, q, k, v, o, lse, dq, dk, dv, shape, mask, nullptr, workspace, workspace_bytes, stream);
}

lca_status lca_attn_bwd_dropout(const void* dout, const void* q, const void* k, const void* v, const void* o,
                                const float* lse, void* dq, void* dk, void* dv, const lca_shape* shape,
                                const lca_mask_desc* mask, const lca_dropout* dropout, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return attn_bwd_impl(dout, q, k, v, o, lse, dq, dk, dv, shape, mask, dropout, workspace, workspace_bytes, stream);
}
}  // extern "C"

namespace lca {
namespace {

lca_status attn_fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, const lca_shape* shape,
                         const lca_mask_desc* mask, const lca_dropout* dropout, void* workspace,
                         size_t workspace_bytes, void* stream) {
  Drop dr;
  lca_status r = parse_dropout(dropout, dr);
  if (r != LCA_OK) return r;
  Call c;
  r = prepare(c, shape, mask, workspace, workspace_bytes, stream, true, false);
  if (r != LCA_OK) return r;
  const HostPlan& P = c.P;
  if ((P.Tq > 0 && (!q || !o || !lse)) || (P.Tk > 0 && (!k || !v))) return LCA_ERR_INVALID_ARG;
  if (P.Tq > 0) {
    if (!device_input(q)) return LCA_ERR_INVALID_ARG;
    o = output_address(o);
    lse = static_cast<float*>(output_address(lse));
    if (!o || !lse) return LCA_ERR_INVALID_ARG;
  }
  if (P.Tk > 0 && (!device_input(k) || !device_input(v))) return LCA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return LCA_ERR_INVALID_ARG;
  const long long n_rows = static_cast<long long>(P.hm_count) * (P.fwd_pair ? P.R128 : P.R256);
  CUtensorMap tq, tk, tv;
  if (n_rows > 0) {
    if (!make_map(&tq, q, P.Tq, P.Hq, kTile) || !make_map(&tk, k, P.Tk, P.Hkv, kTile) ||
        !make_map(&tv, v, P.Tk, P.Hkv, kTile))
      return LCA_ERR_CUDA;
  }
  const int sms = num_sms();
  if (sms <= 0) return LCA_ERR_CUDA;
  r = upload(c);
  if (r != LCA_OK) return r;
  if (n_rows > 0) {
    WorkList wl{};
    wl.cnt = reinterpret_cast<int*>(c.ws + c.L.f_cnt);
    wl.key = reinterpret_cast<int*>(c.ws + c.L.f_key);
    wl.order = reinterpret_cast<int*>(c.ws + c.L.f_order);
    wl.entries = c.ws + c.L.f_ent;
    wl.hist = reinterpret_cast<uint32_t*>(c.ws + c.L.hist);
    wl.counter = reinterpret_cast<int*>(c.ws + c.L.counters);
    wl.n_sorted = static_cast<int>(n_rows);
    wl.expand = P.Hq / P.hm_count / (P.fwd_pair ? 2 : 1);  // heads (or head pairs) per list row
    int ph = phase_begin(0, c.st);
    uint8_t* tcls = c.ws + c.L.tcls;
    launch_classify(c.V, tcls, c.st);
    launch_plan_fwd(c.V, tcls, wl, P.fwd_pair, c.st);
    launch_sort(wl, c.st);
    phase_end(ph, c.st);
    AttnArgs a = base_args(c, dr);
    a.cnt = wl.cnt;
    a.order = wl.order;
    a.entries = wl.entries;
    a.counter = wl.counter;
    a.expand = wl.expand;
    a.n_work = static_cast<int>(n_rows * wl.expand);
    // K/V larger than L2 and segments of 8K rows or more on average: segment
    // by segment, head by head (shorter segments keep the cost order, whose
    // balance is worth more there: 2K and document batches were 10-13 %
    // slower; with K/V that fits in L2 the cost order is as local and
    // balances better)
    a.row_group = (wl.expand > 1 && kv_beyond_l2(P) && P.Tq >= 8192LL * std::max(1, P.n_seg)) ? -1 : 1;
    a.fwd_pair = P.fwd_pair ? 1 : 0;
    a.o = o;
    a.out_v8 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
    a.lse = lse;
    a.prof = prof_slot(0, c.st);
    ph = phase_begin(1, c.st);
    launch_fwd(tq, tk, tv, a, sms, c.st);
    phase_end(ph, c.st);
  }
  const size_t row_bytes = static_cast<size_t>(P.Hq) * kHeadDim * 2;
  for (auto& gp : P.q_gaps) {
    launch_zero16(static_cast<uint8_t*>(o) + gp.first * row_bytes, gp.second * row_bytes, c.st);
    launch_fill_lse(lse, P.Tq, P.Hq, gp.first, gp.second, c.st);
  }
  LCA_CUDA(cudaGetLastError());
  return LCA_OK;
}

}  // namespace
}  // namespace lca

extern "C" {

lca_status lca_attn_merge(const void* const* o_parts, const float* const* lse_parts, int32_t n_parts, void* o,
                          float* lse, int32_t Tq, int32_t Hq, int32_t d, void* stream) {
  if (d != kHeadDim) return LCA_ERR_UNSUPPORTED;
  if (n_parts < 1 || n_parts > LCA_MERGE_MAX_PARTS || Tq < 0 || Hq <= 0 || !o_parts || !lse_parts)
    return LCA_ERR_INVALID_ARG;
  if (static_cast<long long>(Tq) * Hq * 16 / 256 >= 0x7FFFFFFFLL) return LCA_ERR_UNSUPPORTED;  // grid size
  if (Tq == 0) return LCA_OK;
  if (!o || !aligned16(o) || !lse || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return LCA_ERR_INVALID_ARG;
  MergeArgs m{};
  for (int p = 0; p < n_parts; ++p) {
    if (!o_parts[p] || !aligned16(o_parts[p]) || !lse_parts[p] || (reinterpret_cast<uintptr_t>(lse_parts[p]) & 3u) != 0)
      return LCA_ERR_INVALID_ARG;
    m.o[p] = o_parts[p];
    m.lse[p] = lse_parts[p];
  }
  m.n = n_parts;
  m.out = o;
  m.lse_out = lse;
  m.Tq = Tq;
  m.Hq = Hq;
  launch_merge(m, static_cast<cudaStream_t>(stream));
  LCA_CUDA(cudaGetLastError());
  return LCA_OK;
}

}  // extern "C"

namespace lca {
namespace {

lca_status attn_bwd_impl(const void* dout, const void* q, const void* k, const void* v, const void* o,
                         const float* lse, void* dq, void* dk, void* dv, const lca_shape* shape,
                         const lca_mask_desc* mask, const lca_dropout* dropout, void* workspace,
                         size_t workspace_bytes, void* stream) {
  Drop dr;
  lca_status r = parse_dropout(dropout, dr);
  if (r != LCA_OK) return r;
  Call c;
  r = prepare(c, shape, mask, workspace, workspace_bytes, stream, true, true);
  if (r != LCA_OK) return r;
  const HostPlan& P = c.P;
  if ((P.Tq > 0 && (!dout || !q || !o || !lse || !dq)) || (P.Tk > 0 && (!k || !v || !dk || !dv)))
    return LCA_ERR_INVALID_ARG;
  if (P.Tq > 0) {
    if (!device_input(dout) || !device_input(q) || !device_input(o) || !device_input(lse)) return LCA_ERR_INVALID_ARG;
    dq = output_address(dq);
    if (!dq) return LCA_ERR_INVALID_ARG;
  }
  if (P.Tk > 0) {
    if (!device_input(k) || !device_input(v)) return LCA_ERR_INVALID_ARG;
    dk = output_address(dk);
    dv = output_address(dv);
    if (!dk || !dv) return LCA_ERR_INVALID_ARG;
  }
  if (!aligned16(dout) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return LCA_ERR_INVALID_ARG;
  const long long q_rows = static_cast<long long>(P.hm_count) * P.R128;
  const int hkv_m = (P.hm_count == 1) ? 1 : P.Hkv;
  const long long k_units = static_cast<long long>(hkv_m) * P.RK;
  CUtensorMap tq, tk, tv, tdo, tq64, tdo64;
  if (q_rows > 0 || k_units > 0) {
    if (P.Tq > 0 && (!make_map(&tq, q, P.Tq, P.Hq, kTile) || !make_map(&tdo, dout, P.Tq, P.Hq, kTile) ||
                     !make_map(&tq64, q, P.Tq, P.Hq, 64) || !make_map(&tdo64, dout, P.Tq, P.Hq, 64)))
      return LCA_ERR_CUDA;
    if (P.Tk > 0 && (!make_map(&tk, k, P.Tk, P.Hkv, kTile) || !make_map(&tv, v, P.Tk, P.Hkv, kTile)))
      return LCA_ERR_CUDA;
  }
  const int sms = num_sms();
  if (sms <= 0) return LCA_ERR_CUDA;
  r = upload(c);
  if (r != LCA_OK) return r;
  float* D = reinterpret_cast<float*>(c.ws + c.L.D);
  float* lse2 = reinterpret_cast<float*>(c.ws + c.L.lse2);
  uint32_t* hist = reinterpret_cast<uint32_t*>(c.ws + c.L.hist);
  int* counters = reinterpret_cast<int*>(c.ws + c.L.counters);
  uint8_t* tcls = c.ws + c.L.tcls;
  int ph = phase_begin(3, c.st);  // the tile classes serve both lists
  launch_classify(c.V, tcls, c.st);
  phase_end(ph, c.st);
  // dK/dV on the side stream when both passes have work (see side_stream):
  // its lists are built while the D prepass streams O and dO on the caller's
  // stream, and its kernel starts once both are done
  cudaStream_t sk = c.st;
  cudaEvent_t ev_fork = nullptr, ev_pre = nullptr, ev_planned = nullptr, ev_join = nullptr;
  // with a profiling hook on (phase events or the CTA profile) the passes run
  // one after another, so that each phase's events and each kernel's CTA
  // records cover that kernel alone
  const bool profiling = (g_ring.events != nullptr && g_ring.n_pairs > 0) || g_prof != nullptr;
  const bool fork = k_units > 0 && q_rows > 0 && !profiling;
  if (fork) {
    sk = side_stream(r);
    if (r != LCA_OK) return r;
    LCA_CUDA(cudaEventCreateWithFlags(&ev_fork, cudaEventDisableTiming));
    LCA_CUDA(cudaEventCreateWithFlags(&ev_pre, cudaEventDisableTiming));
    LCA_CUDA(cudaEventCreateWithFlags(&ev_planned, cudaEventDisableTiming));
    LCA_CUDA(cudaEventCreateWithFlags(&ev_join, cudaEventDisableTiming));
    LCA_CUDA(cudaEventRecord(ev_fork, c.st));
    LCA_CUDA(cudaStreamWaitEvent(sk, ev_fork, 0));
  }
  ph = phase_begin(2, c.st);
  launch_d_prepass(o, dout, lse, D, lse2, P.Tq, P.Hq, dr.keep, c.st);
  phase_end(ph, c.st);
  if (fork) LCA_CUDA(cudaEventRecord(ev_pre, c.st));
  if (k_units > 0) {
    WorkList wl{};
    wl.cnt = reinterpret_cast<int*>(c.ws + c.L.k_ucost);
    wl.key = reinterpret_cast<int*>(c.ws + c.L.k_key);
    wl.order = reinterpret_cast<int*>(c.ws + c.L.k_order);
    wl.entries = c.ws + c.L.k_ent;
    wl.hist = hist + kCostBuckets;
    wl.counter = counters + 1;
    wl.n_sorted = static_cast<int>(k_units);
    wl.expand = P.Hkv / hkv_m;
    int* list_cnt = reinterpret_cast<int*>(c.ws + c.L.k_lcnt);
    int* list_steps = reinterpret_cast<int*>(c.ws + c.L.k_lsteps);
    int* usteps = reinterpret_cast<int*>(c.ws + c.L.k_usteps);
    DkvSplit sp{};
    sp.nchunk = reinterpret_cast<int*>(c.ws + c.L.k_nchunk);
    sp.item_start = reinterpret_cast<int*>(c.ws + c.L.k_istart);
    sp.split_start = reinterpret_cast<int*>(c.ws + c.L.k_sstart);
    sp.n_work = reinterpret_cast<int*>(c.ws + c.L.k_nwork);
    sp.max_slots = c.L.k_max_slots;
    sp.run_first = reinterpret_cast<int*>(c.ws + c.L.k_runfirst);
    sp.run_of = reinterpret_cast<int*>(c.ws + c.L.k_runof);
    sp.run_at = reinterpret_cast<int*>(c.ws + c.L.k_runat);
    ph = phase_begin(3, sk);
    launch_plan_dkv(c.V, tcls, wl, list_cnt, list_steps, usteps, sk);
    launch_sort(wl, sk);
    // One mask map and enough work items to balance without cuts (MHA, or at
    // least eight items per SM): whole units, key group by key group and
    // head by head, so that the items in flight read one head's Q and dO
    const bool dkv_seg_major = P.hm_count == 1 && wl.expand > 1 &&
                               (P.Hq == P.Hkv || k_units * wl.expand >= 8LL * sms);
    launch_split_dkv(wl, usteps, sp, sms, dkv_seg_major, sk);
    phase_end(ph, sk);
    if (fork) LCA_CUDA(cudaEventRecord(ev_planned, sk));
    AttnArgs a = base_args(c, dr);
    a.cnt = wl.cnt;
    a.order = wl.order;
    a.entries = wl.entries;
    a.list_cnt = list_cnt;
    a.list_steps = list_steps;
    a.counter = wl.counter;
    a.expand = wl.expand;
    a.n_work = static_cast<int>(k_units * wl.expand + sp.max_slots);  // bound for the grid; the device holds the count
    a.item_start = sp.item_start;
    a.split_start = sp.split_start;
    a.nchunk = sp.nchunk;
    a.usteps = usteps;
    a.n_work_dev = sp.n_work;
    a.run_first = sp.run_first;
    a.run_of = sp.run_of;
    a.run_at = sp.run_at;
    a.dkv_seg_major = dkv_seg_major ? 1 : 0;
    a.partials = reinterpret_cast<float*>(c.ws + c.L.k_part);
    a.n_units = static_cast<int>(k_units);
    a.nD = D;
    a.nlse2 = lse2;
    a.dk = dk;
    a.dv = dv;
    a.out_v8 = ((reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 31u) == 0;
    a.prof = prof_slot(1, sk);
    if (fork) LCA_CUDA(cudaStreamWaitEvent(sk, ev_pre, 0));  // -D and -LSE*log2(e)
    ph = phase_begin(4, sk);
    launch_bwd_dkv(tq64, tk, tv, tdo64, a, sms, sk);
    launch_dkv_reduce(a, sk);
    phase_end(ph, sk);
    if (fork) LCA_CUDA(cudaEventRecord(ev_join, sk));
  }
  if (q_rows > 0) {
    WorkList wl{};
    wl.cnt = reinterpret_cast<int*>(c.ws + c.L.q_cnt);
    wl.key = reinterpret_cast<int*>(c.ws + c.L.q_key);
    wl.order = reinterpret_cast<int*>(c.ws + c.L.q_order);
    wl.entries = c.ws + c.L.q_ent;
    wl.hist = hist + 2 * kCostBuckets;
    wl.counter = counters + 2;
    wl.n_sorted = static_cast<int>(q_rows);
    wl.expand = P.Hq / P.hm_count;
    ph = phase_begin(5, c.st);
    launch_plan_dq(c.V, tcls, wl, c.st);
    launch_sort(wl, c.st);
    phase_end(ph, c.st);
    AttnArgs a = base_args(c, dr);
    a.cnt = wl.cnt;
    a.order = wl.order;
    a.entries = wl.entries;
    a.counter = wl.counter;
    a.expand = wl.expand;
    a.n_work = static_cast<int>(q_rows * wl.expand);
    a.row_group = (wl.expand > 1 && kv_beyond_l2(P)) ? -1 : 1;  // K/V larger than L2: segment by segment, head by head
    a.nD = D;
    a.nlse2 = lse2;
    a.dq = dq;
    a.out_v8 = (reinterpret_cast<uintptr_t>(dq) & 31u) == 0;
    a.prof = prof_slot(2, c.st);
    // the dQ kernel is queued once dK/dV's lists are built, so both kernels
    // become ready together and the higher-priority dK/dV CTAs go first
    if (fork) LCA_CUDA(cudaStreamWaitEvent(c.st, ev_planned, 0));
    ph = phase_begin(6, c.st);
    launch_bwd_dq(tq, tk, tv, tdo, a, sms, c.st);
    phase_end(ph, c.st);
  }
  if (fork) {
    LCA_CUDA(cudaStreamWaitEvent(c.st, ev_join, 0));
    // released by CUDA once recorded work completes
    cudaEventDestroy(ev_fork);
    cudaEventDestroy(ev_pre);
    cudaEventDestroy(ev_planned);
    cudaEventDestroy(ev_join);
  }
  const size_t qrow = static_cast<size_t>(P.Hq) * kHeadDim * 2, krow = static_cast<size_t>(P.Hkv) * kHeadDim * 2;
  for (auto& gp : P.q_gaps) launch_zero16(static_cast<uint8_t*>(dq) + gp.first * qrow, gp.second * qrow, c.st);
  for (auto& gp : P.k_gaps) {
    launch_zero16(static_cast<uint8_t*>(dk) + gp.first * krow, gp.second * krow, c.st);
    launch_zero16(static_cast<uint8_t*>(dv) + gp.first * krow, gp.second * krow, c.st);
  }
  LCA_CUDA(cudaGetLastError());
  return LCA_OK;
}

}  // namespace
}  // namespace lca

extern "C" {

lca_status lca_mask_materialize(const lca_shape* shape, const lca_mask_desc* mask, int32_t head, int32_t seg,
                                uint8_t* out, void* workspace, size_t workspace_bytes, void* stream) {
  Call c;
  lca_status r = prepare(c, shape, mask, workspace, workspace_bytes, stream, true, false);
  if (r != LCA_OK) return r;
  if (head < 0 || head >= c.P.Hq || seg < 0 || seg >= c.P.n_seg || !out) return LCA_ERR_INVALID_ARG;
  r = upload(c);
  if (r != LCA_OK) return r;
  const long long cells = static_cast<long long>(c.P.segs[seg].q_len) * c.P.segs[seg].k_len;
  if (cells > 0) launch_materialize_seg(c.V, seg, c.P.hm_count == 1 ? 0 : head, cells, out, c.st);
  LCA_CUDA(cudaGetLastError());
  return LCA_OK;
}

lca_status lca_mask_tile_classes(const lca_shape* shape, const lca_mask_desc* mask, int32_t head, int32_t seg,
                                 uint8_t* out, void* workspace, size_t workspace_bytes, void* stream) {
  Call c;
  lca_status r = prepare(c, shape, mask, workspace, workspace_bytes, stream, true, false);
  if (r != LCA_OK) return r;
  if (head < 0 || head >= c.P.Hq || seg < 0 || seg >= c.P.n_seg || !out) return LCA_ERR_INVALID_ARG;
  r = upload(c);
  if (r != LCA_OK) return r;
  const SegInfo& sg = c.P.segs[seg];
  const long long tiles = cdiv(sg.q_len, kTile) * sg.nk;
  launch_tile_classes_seg(c.V, seg, c.P.hm_count == 1 ? 0 : head, static_cast<int>(tiles), out, c.st);
  LCA_CUDA(cudaGetLastError());
  return LCA_OK;
}

lca_status lca_mask_nnz(const lca_shape* shape, const lca_mask_desc* mask, uint64_t* nnz, void* workspace,
                        size_t workspace_bytes, void* stream) {
  Call c;
  lca_status r = prepare(c, shape, mask, workspace, workspace_bytes, stream, true, false);
  if (r != LCA_OK) return r;
  if (!nnz) return LCA_ERR_INVALID_ARG;
  r = upload(c);
  if (r != LCA_OK) return r;
  launch_nnz(c.V, c.P.max_q_len, reinterpret_cast<unsigned long long*>(c.ws + c.L.acc),
             reinterpret_cast<unsigned long long*>(nnz), c.st);
  LCA_CUDA(cudaGetLastError());
  return LCA_OK;
}

lca_status lca_read_status(const void* workspace, int32_t out[2], void* stream) {
  if (!workspace || !out) return LCA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LCA_CUDA(cudaMemcpyAsync(out, workspace, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  LCA_CUDA(cudaStreamSynchronize(st));
  return LCA_OK;
}

lca_status lca_probe_wait_timeout(void* workspace, size_t workspace_bytes, int32_t limit_ms, void* stream) {
  if (!workspace || workspace_bytes < 16 || limit_ms <= 0) return LCA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LCA_CUDA(cudaMemsetAsync(workspace, 0, 16, st));
  launch_probe_timeout(static_cast<int*>(workspace), static_cast<unsigned long long>(limit_ms) * 1000000ull, st);
  LCA_CUDA(cudaGetLastError());
  return LCA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ static workspace
// The workspace of lca_attn_fwd_static_workspace: a file-scope device array.
// Host code must not use the symbol itself (on the host it is only a
// stand-in); it uses the device address looked up once per device.
static __device__ __align__(256) unsigned char g_static_workspace[LCA_STATIC_WORKSPACE_BYTES];

namespace {
constexpr int kMaxDevices = 64;
void* g_static_ws_ptr[kMaxDevices] = {};
std::mutex g_static_ws_mu;
}  // namespace

extern "C" lca_status lca_attn_fwd_static_workspace(const void* q, const void* k, const void* v, void* o, float* lse,
                                                    const lca_shape* shape, const lca_mask_desc* mask, void* stream) {
  size_t need = 0;
  const lca_status r = lca_workspace_size(shape, mask, 0, &need);
  if (r != LCA_OK) return r;
  if (need > LCA_STATIC_WORKSPACE_BYTES) {
    snprintf(g_err_detail, sizeof(g_err_detail), "forward needs %zu workspace bytes; the static workspace holds %u",
             need, LCA_STATIC_WORKSPACE_BYTES);
    return LCA_ERR_WORKSPACE;
  }
  int dev = -1;
  LCA_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return LCA_ERR_UNSUPPORTED;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_ws_mu);
    if (!g_static_ws_ptr[dev]) {
      void* p = nullptr;
      LCA_CUDA(cudaGetSymbolAddress(&p, g_static_workspace));  // with device `dev` current
      g_static_ws_ptr[dev] = p;
    }
    ws = g_static_ws_ptr[dev];
  }
  return lca_attn_fwd(q, k, v, o, lse, shape, mask, ws, LCA_STATIC_WORKSPACE_BYTES, stream);
}

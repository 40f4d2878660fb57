// lca_internal.h — what the host side (lca_api.cu) and the kernel files share:
// the device view of a call's plan and the kernel launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "lca_common.cuh"
#include "lca_dropout.cuh"

namespace lca {

constexpr int kCostBuckets = 4096;  // histogram buckets of the cost sort
constexpr int kProfCtas = 1024;     // CTA records per kernel in a profile buffer

// Cost of a FULL and a PARTIAL tile unit in the longest-first schedules
// (forward: 128-row sub-tile x key tile; dQ: 128x128 tile; dK/dV: 64-row
// query step), in units of a quarter of a full unit; how they were measured
// is described with the planner in lca_plan.cu.
struct CostWeights {
  int full, partial;
};
constexpr CostWeights kCostFwd{4, 10}, kCostDq{4, 5}, kCostDkv{4, 6};
// A dK/dV chunk is at least this many 64-row steps long (a chunk pays a K/V
// load and an epilogue, worth about ten steps).
constexpr int kMinChunkSteps = 64;
// When a call's K/V exceed this many bytes (less than the 126 MB L2, which
// also holds Q tiles and outputs), dQ items (and forward items when the
// segments average 8K rows or more) go segment by segment and head by head
// (seg_major_item), so the items in flight share K/V in L2 instead of
// streaming every head's K/V from HBM (8K causal MHA: forward and backward
// 10 % faster; 48K causal GQA forward 8 %).
constexpr long long kKvL2Bytes = 96LL << 20;

// Counts kernel launches made by this library (see lca_launch_count).
void note_launches(int n);

// Device-side view of one call's plan; every pointer lies in the workspace.
struct PlanView {
  MaskCtx mask;
  const SegInfo* segs;
  int n_seg;
  const int* q256_start;     // [n_seg + 1] prefix of 256-row query blocks
  const int* q128_start;     // [n_seg + 1] prefix of 128-row query tiles
  const long long* fwd_off;  // [n_seg] forward entry offset of each segment (per map head)
  const long long* dq_off;   // [n_seg] dQ entry offset of each segment (per map head)
  const KeyGroup* kgs;
  int n_kg;
  const int* kg_segs;   // segment ids grouped by key group
  const int* kt_start;  // [n_kg + 1] prefix of key tiles
  int hm_count;         // mask map heads H' (1 or Hq)
  int R256, R128, RK;   // rows per map head: 256-row blocks, 128-row tiles, key tiles
  long long fwd_per_hm, dq_per_hm, dkv_per_hm;
  int Tq, Tk, Hq, Hkv, G;
};

// Work lists produced by the planner for one kernel.
struct WorkList {
  int* cnt;           // entries per list row (dK/dV: weighted step cost per unit)
  int* key;           // cost bucket per row or unit (the sort key)
  int* order;         // rows (or units) sorted by descending cost
  void* entries;      // uint32 (query-major) or int2 (key-major) entries
  uint32_t* hist;     // [kCostBuckets]
  int* counter;       // persistent-scheduler work counter
  int n_sorted;       // number of sortable rows/units
  int expand;         // work items per sorted row (heads sharing one list)
};

// ------------------------------------------------------------ planning (lca_plan.cu)
void launch_build_block_maps(const PlanView& pv, const int* qb_bounds, const int* kb_bounds, uint32_t* keep,
                             int* qb_of, int* kb_of, const int* row_ptr, const int* col_idx, long long blk_nnz,
                             size_t keep_bytes, int* status, cudaStream_t st);
// Variable block maps: the chunk words of every (map head, query block,
// key-group key tile), [hm][n_qb][RK] (see vchunk_byte).
void launch_build_vchunk(const PlanView& pv, uint32_t* out, cudaStream_t st);
// Class of every 128x128 tile, [map head][segment at dq_off][query tile][key tile] bytes.
void launch_classify(const PlanView& pv, uint8_t* tcls, cudaStream_t st);
// Forward lists: one row per 256 query rows (two 128-row sub-tiles), or with
// `pair` one row per 128 query rows whose class serves both sub-tiles (two
// query heads of one KV head and one mask map).
void launch_plan_fwd(const PlanView& pv, const uint8_t* tcls, const WorkList& wl, bool pair, cudaStream_t st);
void launch_plan_dq(const PlanView& pv, const uint8_t* tcls, const WorkList& wl, cudaStream_t st);
void launch_plan_dkv(const PlanView& pv, const uint8_t* tcls, const WorkList& wl, int* list_cnt, int* list_steps,
                     int* usteps, cudaStream_t st);
// Chunk counts, item and partial-slot prefixes over the cost-sorted units.
// Chunk counts per unit; runs of sorted units (same cost bucket and chunk
// count) with their item and partial-slot prefixes.
struct DkvSplit {
  int* nchunk;       // per unit: chunks of each of its items (1 = whole)
  int* item_start;   // per claim position: first work item (n_runs + 1 entries)
  int* split_start;  // per run: first partial slot
  int* n_work;       // [0] work items, [1] runs
  int* run_first;    // per run: first sorted unit
  int* run_of;       // per sorted unit: its run
  int* run_at;       // per claim position: its run (runs by descending item cost)
  int max_slots;
};
// whole: no cuts (every unit one work item per KV head).
void launch_split_dkv(const WorkList& wl, const int* usteps, const DkvSplit& sp, int num_sms, bool whole,
                      cudaStream_t st);
void launch_sort(const WorkList& wl, cudaStream_t st);
void launch_materialize_seg(const PlanView& pv, int seg, int hm, long long cells, uint8_t* out, cudaStream_t st);
void launch_tile_classes_seg(const PlanView& pv, int seg, int hm, int tiles, uint8_t* out, cudaStream_t st);
void launch_nnz(const PlanView& pv, int max_q_len, unsigned long long* acc, unsigned long long* nnz, cudaStream_t st);
struct MergeArgs {
  const void* o[16];
  const float* lse[16];
  int n;
  void* out;
  float* lse_out;
  int Tq, Hq;
};
void launch_merge(const MergeArgs& m, cudaStream_t st);
// nD = -dmul * rowsum(dO * O) (dmul is the keep probability under dropout, 1
// otherwise) and nlse2 = -LSE * log2(e) (-inf for rows with no key).
void launch_d_prepass(const void* o, const void* dout, const float* lse, float* nD, float* nlse2, int Tq, int Hq,
                      float dmul, cudaStream_t st);
void launch_fill_lse(float* lse, int Tq, int Hq, int row0, int nrows, cudaStream_t st);
void launch_zero16(void* p, size_t bytes, cudaStream_t st);  // bytes a multiple of 16, p 16-byte aligned
void launch_probe_timeout(int* status, unsigned long long limit_ns, cudaStream_t st);

// ------------------------------------------------------------ attention kernels
struct AttnArgs {
  PlanView pv;
  const int* cnt;
  const int* order;
  const void* entries;
  const int* list_cnt;    // dK/dV: entries per (map head, key tile) list
  const int* list_steps;  // dK/dV: 64-row query steps per list
  int* counter;
  int n_work;
  int expand;
  int row_group;  // forward, dQ: sorted rows per group of the item order (see item_of); -1: seg_major_item
  int fwd_pair;   // forward: items are 128 rows of two query heads (1) or 256 rows of one (0)
  // dK/dV: whole units taken key group by key group, head by head, key tile
  // by key tile (MHA: the items in flight share a head's Q and dO in L2)
  int dkv_seg_major;
  // dK/dV: units far longer than a share of the per-SM load, and the last
  // units of the cost order, are cut into chunks of 64-row steps; a chunk
  // writes f32 partial dV, dK that a reduction sums.
  const int* item_start;   // [n_runs + 1] first work item of each claim position
  const int* split_start;  // [n_runs] first partial slot of each run
  const int* nchunk;       // [unit] chunks of each of the unit's items (1 = whole)
  const int* usteps;       // [unit] 64-row steps of each of the unit's items
  const int* n_work_dev;   // [0] work items, [1] runs, written on the device by the split pass
  const int* run_first;    // [n_runs] first sorted unit of each run
  const int* run_of;       // [n_units] run of each sorted unit
  const int* run_at;       // [n_runs] run at each claim position
  float* partials;         // [slot][dV, dK][128 rows][128] f32
  int n_units;
  int* status;
  unsigned long long wait_limit_ns;
  // per-CTA profile records (kProfCtas x 8 u64), or null when profiling is off
  unsigned long long* prof;
  float scale;       // softmax scale
  float scale_log2;  // scale * log2(e)
  // dropout on P: threshold t (0 = off; keep probability (256 - t) / 256),
  // the Philox round keys, and 1 / keep probability (1 without dropout)
  int drop_t;
  float drop_inv;
  PhiloxKeys drop_keys;
  // tensors
  void* o;
  int out_v8;  // the kernel's bf16 outputs are 32-byte aligned: rows are written in 32-byte stores
  float* lse;
  const float* nD;     // -D (times the keep probability under dropout), [Hq][Tq]
  const float* nlse2;  // -LSE * log2(e), [Hq][Tq]
  void* dq;
  void* dk;
  void* dv;
};

void launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a,
                int num_sms, cudaStream_t st);
void launch_bwd_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                   const AttnArgs& a, int num_sms, cudaStream_t st);
void launch_bwd_dkv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                    const AttnArgs& a, int num_sms, cudaStream_t st);
// Sums the partial dV, dK of split units into the bf16 outputs.
void launch_dkv_reduce(const AttnArgs& a, cudaStream_t st);

}  // namespace lca

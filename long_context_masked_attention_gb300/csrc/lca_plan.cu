// lca_plan.cu — the mask compiler and the cost-sorted work lists, plus the
// small HBM-bound kernels around the attention kernels.
//
//  * Block maps: the block-sparse CSR (LongCA-bench review, 动态掩码: uniform
//    and variable block masks) becomes a dense keep bitmap so every kernel can
//    test a (query block, key block) pair with one load.
//  * Mask compiler: every (128-row query tile, 128-key tile) pair of every
//    segment is classified EMPTY / FULL / PARTIAL and the non-empty ones are
//    written as per-row work lists: query-major for the forward and dQ passes,
//    key-major for the dK/dV pass.
//  * Cost sort: the list rows are ordered by descending cost (longest first)
//    so the persistent kernels, which claim rows through an atomic counter,
//    balance ragged documents and shards across the SMs (FlashAttention-2's
//    work partitioning; the disaggregation page's compute balancing).
//  * D prepass: D_i = sum_k dO_ik O_ik, the row statistic of the backward
//    (FlashAttention-2 核心优化, 反向传播), together with LSE in base 2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "lca_internal.h"
#include "sm103.cuh"

namespace lca {

// ---------------------------------------------------------------- block maps
__global__ void build_keep_kernel(MaskCtx m, const int* __restrict__ row_ptr, const int* __restrict__ col_idx,
                                  long long blk_nnz, uint32_t* keep, int* status) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int rows = m.hm_count * m.n_qb;
  if (warp >= rows) return;
  const long long b = row_ptr[warp], e = row_ptr[warp + 1];
  if (b < 0 || e < b || e > blk_nnz) {
    if (lane == 0) raise_status(status, kStatusDeviceArg, 100);
    return;
  }
  uint32_t* row = keep + static_cast<size_t>(warp) * m.words;
  for (long long t = b + lane; t < e; t += 32) {
    const int kb = col_idx[t];
    if (kb < 0 || kb >= m.n_kb) {
      raise_status(status, kStatusDeviceArg, 101);
      continue;
    }
    atomicOr(row + (kb >> 5), 1u << (kb & 31));
  }
}

__global__ void block_index_kernel(const int* __restrict__ bounds, int n_blocks, int T, int* map) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= n_blocks) return;
  const int lo = bounds[b], hi = min(bounds[b + 1], T);
  for (int t = lo; t < hi; ++t) map[t] = b;
}

void launch_build_block_maps(const PlanView& pv, const int* qb_bounds, const int* kb_bounds, uint32_t* keep,
                             int* qb_of, int* kb_of, const int* row_ptr, const int* col_idx, long long blk_nnz,
                             size_t keep_bytes, int* status, cudaStream_t st) {
  cudaMemsetAsync(keep, 0, keep_bytes, st);
  const int rows = pv.mask.hm_count * pv.mask.n_qb;
  note_launches(pv.mask.kind == kBlockSparseVariable ? 3 : 1);
  build_keep_kernel<<<(rows + 7) / 8, 256, 0, st>>>(pv.mask, row_ptr, col_idx, blk_nnz, keep, status);
  if (pv.mask.kind == kBlockSparseVariable) {
    block_index_kernel<<<(pv.mask.n_qb + 127) / 128, 128, 0, st>>>(qb_bounds, pv.mask.n_qb, pv.Tq, qb_of);
    block_index_kernel<<<(pv.mask.n_kb + 127) / 128, 128, 0, st>>>(kb_bounds, pv.mask.n_kb, pv.Tk, kb_of);
  }
}

// ---------------------------------------------------------------- variable-map chunk words
__global__ void build_vchunk_kernel(PlanView pv, uint32_t* __restrict__ out, long long total) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long w = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; w < total; w += stride) {
    const int rk = static_cast<int>(w % pv.RK);
    const long long r = w / pv.RK;
    const int qb = static_cast<int>(r % pv.mask.n_qb), hm = static_cast<int>(r / pv.mask.n_qb);
    const int kg = find_bucket(pv.kt_start, pv.n_kg, rk);
    const KeyGroup grp = pv.kgs[kg];
    const int g0 = grp.k_off + (rk - pv.kt_start[kg]) * kTile, k_end = grp.k_off + grp.k_len;
    uint32_t word = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) word |= vchunk_byte(pv.mask, hm, qb, g0 + 32 * c, k_end) << (8 * c);
    out[w] = word;
  }
}

void launch_build_vchunk(const PlanView& pv, uint32_t* out, cudaStream_t st) {
  const long long total = static_cast<long long>(pv.hm_count) * pv.mask.n_qb * pv.RK;
  if (total == 0) return;
  note_launches(1);
  const long long blocks = std::min<long long>((total + 255) / 256, 1 << 20);
  build_vchunk_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(pv, out, total);
}

// ---------------------------------------------------------------- tile classes
// Every 128x128 tile (query tile qt, key tile kt) of every segment and map
// head is classified once, one warp per tile, into a byte array laid out like
// the dQ lists: [map head][segment at dq_off[s]][qt][kt].  The three list
// builders below only compact this array.
__global__ void classify_tiles_kernel(PlanView pv, uint8_t* __restrict__ tcls, long long total) {
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < total; w += warps) {
    const int hm = static_cast<int>(w / pv.dq_per_hm);
    const long long t = w % pv.dq_per_hm;
    int lo = 0, hi = pv.n_seg;  // last segment whose offset is <= t (it holds t: empty ones share the next offset)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pv.dq_off[mid] <= t) lo = mid; else hi = mid;
    }
    const SegInfo sg = pv.segs[lo];
    const long long r = t - pv.dq_off[lo];
    const int qt = static_cast<int>(r / sg.nk), kt = static_cast<int>(r % sg.nk);
    const uint32_t c = classify_tile_warp(pv.mask, sg, hm, qt * kTile, kt * kTile);
    if (lane == 0) tcls[w] = static_cast<uint8_t>(c);
  }
}

// Block-sparse maps: one thread per tile (classify_block_tile).
__global__ void classify_block_tiles_kernel(PlanView pv, uint8_t* __restrict__ tcls, long long total) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long w = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; w < total; w += stride) {
    const int hm = static_cast<int>(w / pv.dq_per_hm);
    const long long t = w % pv.dq_per_hm;
    int lo = 0, hi = pv.n_seg;  // last segment whose offset is <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pv.dq_off[mid] <= t) lo = mid; else hi = mid;
    }
    const SegInfo sg = pv.segs[lo];
    const long long r = t - pv.dq_off[lo];
    const int qt = static_cast<int>(r / sg.nk), kt = static_cast<int>(r % sg.nk);
    tcls[w] = static_cast<uint8_t>(classify_block_tile(pv.mask, sg, hm, qt * kTile, kt * kTile));
  }
}

void launch_classify(const PlanView& pv, uint8_t* tcls, cudaStream_t st) {
  const long long total = static_cast<long long>(pv.hm_count) * pv.dq_per_hm;
  if (total == 0) return;
  note_launches(1);
  if (is_block_sparse(pv.mask.kind)) {
    const long long blocks = std::min<long long>((total + 255) / 256, 65536);
    classify_block_tiles_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(pv, tcls, total);
    return;
  }
  const long long blocks = std::min<long long>((total + 7) / 8, 16384);
  classify_tiles_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(pv, tcls, total);
}

// ---------------------------------------------------------------- cost model
// The schedulers hand out work longest first, by a cost that counts a
// kernel's tile units by class: cost = n_full * w_full + n_partial * w_partial
// (forward: 128-row sub-tile x key tile; dQ: 128-row query tile x key tile;
// dK/dV: 64-row query step).  A PARTIAL unit costs more than a FULL one
// because its mask is evaluated and applied element by element and, in the
// forward, because its softmax chain is on the critical path.  The weights
// are the ratios of the per-unit times fitted (least squares, time = a*full
// + b*partial + c*items) over every CTA's %globaltimer busy time and unit
// counts on the twelve 8K static masks (GQA 64:8): forward b/a = 2.6, dK/dV
// 1.5, dQ 1.2 (the weights, kCostFwd, kCostDq and kCostDkv, are in
// lca_internal.h, where the host sizes the dK/dV shares with them).

__device__ __forceinline__ int unit_cost(uint32_t cls, CostWeights w) {
  return cls == kTileFull ? w.full : (cls == kTilePartial ? w.partial : 0);
}

// Histogram bucket of a cost for the counting sort: exact below 1024, then
// coarser in three steps (4, 32 and 256 cost units per bucket, a relative
// resolution better than 0.7%), capped at the last bucket (cost 300032).
__device__ __forceinline__ int cost_bucket(long long c) {
  long long b;
  if (c < 1024) b = c;
  else if (c < 5120) b = 1024 + (c - 1024) / 4;
  else if (c < 37888) b = 2048 + (c - 5120) / 32;
  else b = 3072 + (c - 37888) / 256;
  return static_cast<int>(b < kCostBuckets - 1 ? b : kCostBuckets - 1);
}

// ---------------------------------------------------------------- query-major lists
// One warp per list row (map head, segment, query block of SUB*128 rows); the
// warp takes 32 key tiles at a time and places the non-empty ones with a ballot.
// Entry = key tile index | class of sub-tile 0 << 24 | class of sub-tile 1 << 26.
// SUB = 3: rows of 128 queries whose class serves both sub-tiles (the
// forward's paired heads).  cnt = entries of the row, key = its cost bucket.
template <int SUB>
__global__ void plan_q_rows_kernel(PlanView pv, const uint8_t* __restrict__ tcls, int* __restrict__ cnt,
                                   int* __restrict__ key, uint32_t* __restrict__ entries,
                                   uint32_t* __restrict__ hist, CostWeights w) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int R = (SUB == 2) ? pv.R256 : pv.R128;
  if (row >= pv.hm_count * R) return;
  const int hm = row / R, rr = row % R;
  const int* qstart = (SUB == 2) ? pv.q256_start : pv.q128_start;
  const int s = find_bucket(qstart, pv.n_seg, rr);
  const SegInfo sg = pv.segs[s];
  const int qb = rr - qstart[s];
  const int nq = (sg.q_len + kTile - 1) / kTile;
  const long long per_hm = (SUB == 2) ? pv.fwd_per_hm : pv.dq_per_hm;
  const long long off = (SUB == 2) ? pv.fwd_off[s] : pv.dq_off[s];
  uint32_t* out = entries + hm * per_hm + off + static_cast<long long>(qb) * sg.nk;
  const uint8_t* cls0 =
      tcls + hm * pv.dq_per_hm + pv.dq_off[s] + static_cast<long long>(qb * (SUB == 2 ? 2 : 1)) * sg.nk;
  const bool has1 = (SUB == 2) && (qb * SUB + 1 < nq);
  int n = 0, cost = 0;
  for (int k0 = 0; k0 < sg.nk; k0 += 32) {
    const int kt = k0 + lane;
    uint32_t c0 = 0, c1 = 0;
    if (kt < sg.nk) {
      c0 = cls0[kt] & 3u;  // the half-empty flags serve the 64-row dK/dV steps only
      if (has1) c1 = cls0[sg.nk + kt] & 3u;
      if (SUB == 3) c1 = c0;
    }
    const uint32_t keep = __ballot_sync(0xFFFFFFFFu, (c0 | c1) != 0);
    if ((c0 | c1) != 0) out[n + __popc(keep & ((1u << lane) - 1u))] = static_cast<uint32_t>(kt) | (c0 << 24) | (c1 << 26);
    n += __popc(keep);
    cost += __reduce_add_sync(0xFFFFFFFFu, unit_cost(c0, w) + unit_cost(c1, w));
  }
  if (lane == 0) {
    cnt[row] = n;
    const int b = cost_bucket(cost);
    key[row] = b;
    atomicAdd(hist + b, 1u);
  }
}

void launch_plan_fwd(const PlanView& pv, const uint8_t* tcls, const WorkList& wl, bool pair, cudaStream_t st) {
  const int rows = pv.hm_count * (pair ? pv.R128 : pv.R256);
  if (rows == 0) return;
  note_launches(1);
  if (pair)
    plan_q_rows_kernel<3><<<(rows + 7) / 8, 256, 0, st>>>(pv, tcls, wl.cnt, wl.key,
                                                          static_cast<uint32_t*>(wl.entries), wl.hist, kCostFwd);
  else
    plan_q_rows_kernel<2><<<(rows + 7) / 8, 256, 0, st>>>(pv, tcls, wl.cnt, wl.key,
                                                          static_cast<uint32_t*>(wl.entries), wl.hist, kCostFwd);
}

void launch_plan_dq(const PlanView& pv, const uint8_t* tcls, const WorkList& wl, cudaStream_t st) {
  const int rows = pv.hm_count * pv.R128;
  if (rows == 0) return;
  note_launches(1);
  plan_q_rows_kernel<1><<<(rows + 7) / 8, 256, 0, st>>>(pv, tcls, wl.cnt, wl.key,
                                                        static_cast<uint32_t*>(wl.entries), wl.hist, kCostDq);
}

// ---------------------------------------------------------------- key-major lists
// One warp per unit (map KV head gm, key group, key tile).  For a shared map
// (H' = 1) the unit has one list; for per-head maps it has one list per query
// head of the KV head.  Entry = {segment, query tile | class byte << 24}; the
// class byte keeps its half-empty flags, and a unit counts one step per
// 64-row half that lies inside the segment and is not flagged empty.
// ucost = the unit's weighted step cost (all G query heads), key = its bucket.
__global__ void plan_kv_units_kernel(PlanView pv, const uint8_t* __restrict__ tcls, int* __restrict__ ucost,
                                     int* __restrict__ key, int* __restrict__ list_cnt,
                                     int* __restrict__ list_steps, int* __restrict__ usteps,
                                     int2* __restrict__ entries, uint32_t* __restrict__ hist, int n_units,
                                     CostWeights w) {
  const int unit = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (unit >= n_units) return;
  const int gm = unit / pv.RK, rk = unit % pv.RK;
  const int kg = find_bucket(pv.kt_start, pv.n_kg, rk);
  const KeyGroup grp = pv.kgs[kg];
  const int kt = rk - pv.kt_start[kg];
  const int nlists = (pv.hm_count == 1) ? 1 : pv.G;
  int cost = 0, unit_steps = 0;  // weighted step cost and steps over the unit's lists
  for (int l = 0; l < nlists; ++l) {
    const int hm = (pv.hm_count == 1) ? 0 : gm * pv.G + l;
    int2* out = entries + hm * pv.dkv_per_hm + grp.entry_off + static_cast<long long>(kt) * grp.pairs;
    int n = 0, steps = 0;
    for (int si = grp.seg_begin; si < grp.seg_end; ++si) {
      const int s = pv.kg_segs[si];
      const SegInfo sg = pv.segs[s];
      if (kt * kTile >= sg.k_len) continue;
      const int nq = (sg.q_len + kTile - 1) / kTile;
      const uint8_t* col = tcls + hm * pv.dq_per_hm + pv.dq_off[s] + kt;
      for (int q0 = 0; q0 < nq; q0 += 32) {
        const int qt = q0 + lane;
        const uint32_t c = (qt < nq) ? col[static_cast<long long>(qt) * sg.nk] : 0u;
        const uint32_t keep = __ballot_sync(0xFFFFFFFFu, c != 0);
        int my_steps = 0;
        if (c != 0) {
          out[n + __popc(keep & ((1u << lane) - 1u))] = make_int2(s, qt | static_cast<int>(c << 24));
          my_steps = ((c & kHalf0Empty) ? 0 : 1) + ((qt * kTile + 64 < sg.q_len && !(c & kHalf1Empty)) ? 1 : 0);
        }
        n += __popc(keep);
        steps += __reduce_add_sync(0xFFFFFFFFu, my_steps);
        cost += __reduce_add_sync(0xFFFFFFFFu, my_steps * unit_cost(c & 3u, w));
      }
    }
    if (lane == 0) {
      list_cnt[hm * pv.RK + rk] = n;
      list_steps[hm * pv.RK + rk] = steps;
    }
    unit_steps += steps;
  }
  if (lane == 0) {
    // one work item covers all G query heads of a KV head; a shared map is one list used G times
    const int mult = (pv.hm_count == 1) ? pv.G : 1;
    usteps[unit] = mult * unit_steps;
    ucost[unit] = mult * cost;
    const int b = cost_bucket(static_cast<long long>(mult) * cost);
    key[unit] = b;
    atomicAdd(hist + b, 1u);
  }
}

void launch_plan_dkv(const PlanView& pv, const uint8_t* tcls, const WorkList& wl, int* list_cnt, int* list_steps,
                     int* usteps, cudaStream_t st) {
  const int n_units = wl.n_sorted;
  if (n_units == 0) return;
  note_launches(1);
  plan_kv_units_kernel<<<(n_units + 7) / 8, 256, 0, st>>>(pv, tcls, wl.cnt, wl.key, list_cnt, list_steps, usteps,
                                                          static_cast<int2*>(wl.entries), wl.hist, n_units,
                                                          kCostDkv);
}

// ---------------------------------------------------------------- dK/dV split
// One block.  The persistent CTAs claim dK/dV work items in cost order, so a
// CTA that finishes early takes the next item; what is left unbalanced is
// the end.  Two cuts keep it short:
//  * a unit whose items cost more than 3/4 of the average per-SM load (and
//    are longer than two minimum chunks) is cut into chunks of about that
//    cost, so that a few very long key tiles (keys every query attends, as
//    with global tokens) do not set the kernel's length;
//  * the units holding the last num_sms (unit, KV head) items of the cost
//    order are cut in two, so that the last round of claims is made of
//    half-size items: with equal units (every key tile of a FULL or sliding
//    mask: 512 units on 152 SMs) whole units leave 56 SMs a fourth unit
//    while the other 96 idle.
// Chunks split a unit's steps evenly and write partial sums to their own
// slots; if the slots would run out, the tail cut covers fewer units, then
// long-unit chunks grow, until they fit.
//
// Work items are then numbered by runs: maximal stretches of the sorted
// units with the same cost bucket and chunk count.  Inside a run the items
// go chunk by chunk, then KV head by KV head, then unit by unit, so that the
// CTAs claiming consecutive items work on the same KV head's query rows at
// the same time (they share Q and dO tiles in L2).  The runs are claimed in
// descending order of their items' cost (a unit's cost over its chunk
// count), so that the halves of the tail cut do not go before whole units
// that are longer than they are (short key tiles at the end of a sliding
// window stay whole while the equal tiles before them are halved).
__device__ __forceinline__ long long block_sum_ll(long long v, long long* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  long long t = 0;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += red[w];
  return t;
}

// Exclusive block scan of one int per thread; returns the prefix and the block total.
__device__ __forceinline__ int block_scan_excl(int v, int* red, int& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();
  if (lane == 31) red[wid] = incl;
  __syncthreads();
  int before = 0;
  total = 0;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
    if (w < wid) before += red[w];
    total += red[w];
  }
  return before + incl - v;
}

// Chunks of the unit at sorted position i: the long-unit cut by `target`
// (cost units), and at least two for the `tail` last sorted units that cost
// at least `tail_min` (a cut adds a work item, whose K/V load and epilogue
// cost about ten steps, so units small next to the per-SM share stay whole).
__device__ __forceinline__ int unit_chunks(long long cost, long long target, int i, int n_units, int tail,
                                           long long tail_min) {
  long long c = (cost + target - 1) / target;
  if (i >= n_units - tail && cost >= tail_min) c = c < 2 ? 2 : c;
  return static_cast<int>(c > 1 ? c : 1);
}

__global__ void __launch_bounds__(1024) split_dkv_kernel(const int* __restrict__ order, const int* __restrict__ ucost,
                                                         const int* __restrict__ usteps, const int* __restrict__ key,
                                                         int n_units, int expand,
                                                         int num_sms, int max_slots, int* __restrict__ nchunk,
                                                         int* __restrict__ item_start,
                                                         int* __restrict__ split_start, int* __restrict__ n_work,
                                                         int* __restrict__ run_first, int* __restrict__ run_of,
                                                         int* __restrict__ run_at, int whole) {
  __shared__ long long red_ll[32];
  __shared__ int red[32];
  __shared__ int bucket_pos[kCostBuckets];
  long long local = 0;
  for (int u = threadIdx.x; u < n_units; u += blockDim.x) local += ucost[u];
  const long long total = block_sum_ll(local, red_ll) * expand;
  long long target = total * 3 / (4LL * max(1, num_sms));
  if (target < kMinChunkSteps * kCostDkv.full) target = kMinChunkSteps * kCostDkv.full;
  int tail = (num_sms + expand - 1) / expand;  // units holding the last num_sms items
  if (whole) {  // no cuts: every unit is one work item per KV head
    target = 1LL << 60;
    tail = 0;
  }
  const long long share = total / max(1, num_sms);
  const long long tail_min = max(static_cast<long long>(kMinChunkSteps) * kCostDkv.full, share / 4);
  for (int round = 0; round < 80; ++round) {  // shrink the cuts until the partial slots suffice
    long long slots = 0;
    for (int i = threadIdx.x; i < n_units; i += blockDim.x) {
      const int u = order[i];
      const int c = unit_chunks(ucost[u], target, i, n_units, tail, tail_min);
      if (c > 1) slots += static_cast<long long>(c) * expand;
    }
    if (block_sum_ll(slots, red_ll) <= max_slots) break;
    if (tail > 0) tail = tail / 2; else target *= 2;
  }
  for (int i = threadIdx.x; i < n_units; i += blockDim.x) {
    const int u = order[i];
    nchunk[u] = unit_chunks(ucost[u], target, i, n_units, tail, tail_min);
  }
  __syncthreads();
  // runs: maximal stretches of sorted units with the same cost bucket and chunk count;
  // run_of[i] = run of sorted unit i, run_first[r] = its first sorted unit
  int run_base = 0;
  for (int i0 = 0; i0 < n_units; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    int head = 0;
    if (i < n_units) {
      const int u = order[i];
      head = (i == 0) || key[u] != key[order[i - 1]] || nchunk[u] != nchunk[order[i - 1]];
    }
    int tot;
    const int pr = block_scan_excl(head, red, tot);
    if (i < n_units) {
      const int r = run_base + pr + head - 1;
      run_of[i] = r;
      if (head) run_first[r] = i;
    }
    run_base += tot;
  }
  const int n_runs = run_base;
  __syncthreads();
  // partial slots, in run order
  int slot_base = 0;
  for (int r0 = 0; r0 < n_runs; r0 += blockDim.x) {
    const int r = r0 + threadIdx.x;
    int si = 0;
    if (r < n_runs) {
      const int first = run_first[r];
      const int last = (r + 1 < n_runs) ? run_first[r + 1] : n_units;
      const int c = nchunk[order[first]];
      si = (c > 1) ? c * expand * (last - first) : 0;
    }
    int tot_s;
    const int ps = block_scan_excl(si, red, tot_s);
    if (r < n_runs) split_start[r] = slot_base + ps;
    slot_base += tot_s;
  }
  // claim order: runs by descending item cost (a counting sort on the cost
  // bucket; runs in one bucket take its positions in no particular order,
  // which changes no result: a run's partial slots follow its run index),
  // run_at[position] = run
  for (int b = threadIdx.x; b < kCostBuckets; b += blockDim.x) bucket_pos[b] = 0;
  __syncthreads();
  for (int r = threadIdx.x; r < n_runs; r += blockDim.x) {
    const int u = order[run_first[r]];
    atomicAdd(&bucket_pos[kCostBuckets - 1 - cost_bucket(ucost[u] / nchunk[u])], 1);
  }
  __syncthreads();
  {
    constexpr int kPer = kCostBuckets / 1024;  // buckets per thread
    int v[kPer], sum = 0;
    for (int j = 0; j < kPer; ++j) {
      v[j] = bucket_pos[threadIdx.x * kPer + j];
      sum += v[j];
    }
    int tot;
    int pre = block_scan_excl(sum, red, tot);
    for (int j = 0; j < kPer; ++j) {
      bucket_pos[threadIdx.x * kPer + j] = pre;
      pre += v[j];
    }
  }
  __syncthreads();
  for (int r = threadIdx.x; r < n_runs; r += blockDim.x) {
    const int u = order[run_first[r]];
    run_at[atomicAdd(&bucket_pos[kCostBuckets - 1 - cost_bucket(ucost[u] / nchunk[u])], 1)] = r;
  }
  __syncthreads();
  // first work item of each claim position
  int item_base = 0;
  for (int p0 = 0; p0 < n_runs; p0 += blockDim.x) {
    const int p = p0 + threadIdx.x;
    int ni = 0;
    if (p < n_runs) {
      const int r = run_at[p];
      const int first = run_first[r];
      const int last = (r + 1 < n_runs) ? run_first[r + 1] : n_units;
      ni = nchunk[order[first]] * expand * (last - first);
    }
    int tot_i;
    const int pi = block_scan_excl(ni, red, tot_i);
    if (p < n_runs) item_start[p] = item_base + pi;
    item_base += tot_i;
  }
  if (threadIdx.x == 0) {
    item_start[n_runs] = item_base;
    n_work[0] = item_base;
    n_work[1] = n_runs;
  }
}

void launch_split_dkv(const WorkList& wl, const int* usteps, const DkvSplit& sp, int num_sms, bool whole,
                      cudaStream_t st) {
  note_launches(1);
  split_dkv_kernel<<<1, 1024, 0, st>>>(wl.order, wl.cnt, usteps, wl.key, wl.n_sorted, wl.expand, num_sms,
                                       sp.max_slots, sp.nchunk, sp.item_start, sp.split_start, sp.n_work,
                                       sp.run_first, sp.run_of, sp.run_at, whole ? 1 : 0);
}

// ---------------------------------------------------------------- cost sort
// Counting sort by descending cost in one block of 1024 threads.  Rows with
// equal cost keep no particular order (the result does not depend on it).
__global__ void __launch_bounds__(1024) sort_kernel(const int* __restrict__ key, int n, const uint32_t* __restrict__ hist,
                                                    int* __restrict__ order, int* __restrict__ counter) {
  __shared__ uint32_t start[kCostBuckets];
  __shared__ uint32_t warp_sums[32];
  const int tid = threadIdx.x;
  constexpr int kPer = kCostBuckets / 1024;  // buckets per thread
  // position p = 0 is the most expensive bucket
  uint32_t local[kPer];
  uint32_t sum = 0;
#pragma unroll
  for (int t = 0; t < kPer; ++t) {
    local[t] = hist[kCostBuckets - 1 - (tid * kPer + t)];
    sum += local[t];
  }
  // exclusive scan of `sum` over the block
  uint32_t incl = sum;
  const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    uint32_t w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += v;
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  uint32_t run = incl - sum + (wid > 0 ? warp_sums[wid - 1] : 0u);
#pragma unroll
  for (int t = 0; t < kPer; ++t) {
    start[kCostBuckets - 1 - (tid * kPer + t)] = run;
    run += local[t];
  }
  __syncthreads();
  for (int r = tid; r < n; r += blockDim.x) {
    const int b = key[r];
    const uint32_t pos = atomicAdd(&start[b], 1u);
    order[pos] = r;
  }
  if (tid == 0) *counter = 0;
}

void launch_sort(const WorkList& wl, cudaStream_t st) {
  note_launches(1);
  sort_kernel<<<1, 1024, 0, st>>>(wl.key, wl.n_sorted, wl.hist, wl.order, wl.counter);
}

// ---------------------------------------------------------------- test hooks
__global__ void materialize_seg_kernel(PlanView pv, int seg, int hm, uint8_t* __restrict__ out) {
  const SegInfo sg = pv.segs[seg];
  const int nch = (sg.k_len + 31) / 32;
  const long long total = static_cast<long long>(sg.q_len) * nch;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(idx / nch);
    const int c = static_cast<int>(idx % nch);
    const uint32_t bits = mask_bits_any(pv.mask, sg, hm, i, c * 32);
    uint8_t* row = out + static_cast<long long>(i) * sg.k_len;
    for (int t = 0; t < 32; ++t) {
      const int j = c * 32 + t;
      if (j < sg.k_len) row[j] = static_cast<uint8_t>((bits >> t) & 1u);
    }
  }
}

__global__ void tile_classes_kernel(PlanView pv, int seg, int hm, uint8_t* __restrict__ out) {
  const SegInfo sg = pv.segs[seg];
  const int nq = (sg.q_len + kTile - 1) / kTile;
  const int tile = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (tile >= nq * sg.nk) return;
  const int qt = tile / sg.nk, kt = tile % sg.nk;
  const uint32_t c = classify_tile_warp(pv.mask, sg, hm, qt * kTile, kt * kTile);
  if ((threadIdx.x & 31) == 0) out[tile] = static_cast<uint8_t>(c);  // class and half-empty flags
}

// nnz: interval families and FlashMask — one thread per query row, grid.y = segment.
__global__ void nnz_rows_kernel(PlanView pv, unsigned long long* acc) {
  const int s = blockIdx.y;
  const SegInfo sg = pv.segs[s];
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  unsigned long long n = 0;
  if (i < sg.q_len) {
    if (pv.mask.kind == kFlashMask) {
      for (int j0 = 0; j0 < sg.k_len; j0 += 32) n += __popc(flashmask_chunk_bits(pv.mask, sg, i, j0));
    } else {
      n = static_cast<unsigned long long>(span_count(row_span(pv.mask, sg, i)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, o);
  if ((threadIdx.x & 31) == 0 && n) atomicAdd(acc, n);
}

// nnz: block-sparse — one thread per CSR row (map head, query block).
__global__ void nnz_blocks_kernel(PlanView pv, unsigned long long* acc) {
  const MaskCtx& m = pv.mask;
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= m.hm_count * m.n_qb) return;
  const int hm = r / m.n_qb, qb = r % m.n_qb;
  const long long qs = (m.kind == kBlockSparseUniform) ? static_cast<long long>(qb) * m.q_block : -1;
  unsigned long long n = 0;
  for (int s = 0; s < pv.n_seg; ++s) {
    const SegInfo sg = pv.segs[s];
    // rows of this query block inside the segment
    const long long q0 = (m.kind == kBlockSparseUniform) ? qs : m.qb_start[qb];
    const long long q1 = (m.kind == kBlockSparseUniform) ? qs + m.q_block : m.qb_start[qb + 1];
    const long long r_lo = max(q0, static_cast<long long>(sg.q_off));
    const long long r_hi = min(q1, static_cast<long long>(sg.q_off + sg.q_len));
    if (r_hi <= r_lo) continue;
    const long long rows = r_hi - r_lo;
    for (int kb = 0; kb < m.n_kb; ++kb) {
      if (!block_kept(m, hm, qb, kb)) continue;
      const int k0 = k_block_start(m, kb);
      const int k1 = (m.kind == kBlockSparseUniform) ? k0 + m.kv_block : m.kb_start[kb + 1];
      const int c_lo = max(k0, sg.k_off), c_hi = min(k1, sg.k_off + sg.k_len);
      if (c_hi > c_lo) n += static_cast<unsigned long long>(rows) * (c_hi - c_lo);
    }
  }
  if (n) atomicAdd(acc + hm, n);
}

__global__ void nnz_broadcast_kernel(const unsigned long long* acc, int hm_count, int Hq, unsigned long long* nnz) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < Hq) nnz[h] = acc[hm_count == 1 ? 0 : h];
}

void launch_nnz(const PlanView& pv, int max_q_len, unsigned long long* acc, unsigned long long* nnz, cudaStream_t st) {
  if (is_block_sparse(pv.mask.kind)) {
    const int rows = pv.mask.hm_count * pv.mask.n_qb;
    if (rows > 0) nnz_blocks_kernel<<<(rows + 127) / 128, 128, 0, st>>>(pv, acc);
  } else if (pv.n_seg > 0 && max_q_len > 0) {
    dim3 grid((max_q_len + 255) / 256, pv.n_seg);
    nnz_rows_kernel<<<grid, 256, 0, st>>>(pv, acc);
  }
  nnz_broadcast_kernel<<<(pv.Hq + 127) / 128, 128, 0, st>>>(acc, pv.hm_count, pv.Hq, nnz);
  note_launches(2);
}

void launch_materialize_seg(const PlanView& pv, int seg, int hm, long long cells, uint8_t* out, cudaStream_t st) {
  const long long chunks = (cells + 31) / 32 + 1;
  const int blocks = static_cast<int>(min(65535LL, (chunks + 255) / 256));
  note_launches(1);
  materialize_seg_kernel<<<max(blocks, 1), 256, 0, st>>>(pv, seg, hm, out);
}

void launch_tile_classes_seg(const PlanView& pv, int seg, int hm, int tiles, uint8_t* out, cudaStream_t st) {
  if (tiles == 0) return;
  note_launches(1);
  tile_classes_kernel<<<(tiles + 7) / 8, 256, 0, st>>>(pv, seg, hm, out);
}

// ---------------------------------------------------------------- D prepass
// One block per (head, 64 rows).  Each half-warp reads one 256-byte row of O
// and of dO (16 lanes x 16 bytes), so every load is a full sector.  Both
// statistics are written negated (-dmul * D, -LSE * log2 e), the form in which
// the backward kernels add them.
__global__ void __launch_bounds__(256) d_prepass_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                                                        const float* __restrict__ lse, float* __restrict__ nD,
                                                        float* __restrict__ nlse2, int Tq, int Hq, float dmul) {
  const int h = blockIdx.y;
  const int t0 = blockIdx.x * 64;
  const int hw = threadIdx.x >> 4;  // half-warp 0..15
  const int l16 = threadIdx.x & 15;
  float acc[4];
  uint4 a[4], b[4];
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int t = t0 + it * 16 + hw;
    if (t < Tq) {
      const size_t base = (static_cast<size_t>(t) * Hq + h) * 16 + l16;  // 16 uint4 per 128-element row
      a[it] = __ldg(o + base);
      b[it] = __ldg(dout + base);
    } else {
      a[it] = make_uint4(0, 0, 0, 0);
      b[it] = make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a[it]);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b[it]);
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 x = __bfloat1622float2(pa[u]);
      const float2 y = __bfloat1622float2(pb[u]);
      s = fmaf(x.x, y.x, s);
      s = fmaf(x.y, y.y, s);
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off, 16);
    acc[it] = s;
  }
  if (l16 == 0) {
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int t = t0 + it * 16 + hw;
      if (t < Tq) {
        const size_t idx = static_cast<size_t>(h) * Tq + t;
        nD[idx] = -(acc[it] * dmul);
        const float l = lse[idx];
        // negated log2-domain LSE; a row with no key (LSE -inf) gets -inf so that P = 0
        nlse2[idx] = (l == -INFINITY) ? -INFINITY : -(l * 1.4426950408889634f);
      }
    }
  }
}

void launch_d_prepass(const void* o, const void* dout, const float* lse, float* nD, float* nlse2, int Tq, int Hq,
                      float dmul, cudaStream_t st) {
  if (Tq == 0) return;
  dim3 grid((Tq + 63) / 64, Hq);
  note_launches(1);
  d_prepass_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4*>(o), static_cast<const uint4*>(dout), lse, nD, nlse2,
                                         Tq, Hq, dmul);
}

// ---------------------------------------------------------------- partial merge
// Half a warp per (row, head): 16 lanes x 8 bf16 = one 256-byte output row.
__global__ void __launch_bounds__(256) merge_kernel(const MergeArgs m) {
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long rh = gid >> 4;  // row * Hq + head
  const int sub = threadIdx.x & 15;
  if (rh >= static_cast<long long>(m.Tq) * m.Hq) return;
  const int row = static_cast<int>(rh / m.Hq), h = static_cast<int>(rh % m.Hq);
  const size_t li = static_cast<size_t>(h) * m.Tq + row;
  float lp[16];
  float mx = -INFINITY;
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    lp[p] = (p < m.n) ? m.lse[p][li] : -INFINITY;
    mx = fmaxf(mx, lp[p]);
  }
  uint4* out = static_cast<uint4*>(m.out) + rh * 16 + sub;
  if (mx == -INFINITY) {  // no part attends this row
    *out = make_uint4(0, 0, 0, 0);
    if (sub == 0) m.lse_out[li] = -INFINITY;
    return;
  }
  float w[16], sum = 0.f;
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    w[p] = (lp[p] == -INFINITY) ? 0.f : expf(lp[p] - mx);
    sum += w[p];
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    if (w[p] == 0.f) continue;
    const uint4 v = static_cast<const uint4*>(m.o[p])[rh * 16 + sub];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      acc[2 * c] += w[p] * __uint_as_float(u[c] << 16);
      acc[2 * c + 1] += w[p] * __uint_as_float(u[c] & 0xFFFF0000u);
    }
  }
  const float inv = 1.f / sum;
  *out = make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                    pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
  if (sub == 0) m.lse_out[li] = mx + logf(sum);
}

void launch_merge(const MergeArgs& m, cudaStream_t st) {
  const long long threads = static_cast<long long>(m.Tq) * m.Hq * 16;
  if (threads == 0) return;
  note_launches(1);
  merge_kernel<<<static_cast<int>((threads + 255) / 256), 256, 0, st>>>(m);
}

__global__ void fill_lse_kernel(float* lse, int Tq, int Hq, int row0, int nrows) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(nrows) * Hq) return;
  const int h = static_cast<int>(idx / nrows), r = static_cast<int>(idx % nrows);
  lse[static_cast<size_t>(h) * Tq + row0 + r] = -INFINITY;
}

void launch_fill_lse(float* lse, int Tq, int Hq, int row0, int nrows, cudaStream_t st) {
  const long long n = static_cast<long long>(nrows) * Hq;
  if (n == 0) return;
  note_launches(1);
  fill_lse_kernel<<<static_cast<int>((n + 255) / 256), 256, 0, st>>>(lse, Tq, Hq, row0, nrows);
}

// Zero `n16` 16-byte words from `p` with plain stores, so that the rows no
// segment covers read as 0 in an output that may live in device memory or in
// device-mapped page-locked host memory.
__global__ void zero16_kernel(uint4* __restrict__ p, long long n16) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

void launch_zero16(void* p, size_t bytes, cudaStream_t st) {
  const long long n16 = static_cast<long long>(bytes / 16);
  if (n16 == 0) return;
  note_launches(1);
  const long long blocks = std::min<long long>((n16 + 255) / 256, 4096);
  zero16_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(static_cast<uint4*>(p), n16);
}

// ---------------------------------------------------------------- timeout probe
__global__ void probe_timeout_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the bounded wait must give up and record
  // LCA_ERR_TIMEOUT.
  mbar_wait(&bar, 0, status, limit_ns, kStatusTimeout, 900);
  __syncthreads();
}

void launch_probe_timeout(int* status, unsigned long long limit_ns, cudaStream_t st) {
  note_launches(1);
  probe_timeout_kernel<<<1, 32, 0, st>>>(status, limit_ns);
}

}  // namespace lca

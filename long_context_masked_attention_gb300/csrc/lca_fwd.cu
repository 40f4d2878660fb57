// lca_fwd.cu — masked attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes, per query row i of a segment and query head h:
//   O_i = sum_j P_ij V_j,  P_ij = exp(tau q_i.k_j - LSE_i) over attended keys,
//   LSE_i = log sum_j exp(tau q_i.k_j)   (natural log, -inf for no key).
// How (FlashAttention review page, FlashAttention-1 核心优化 and
// FlashAttention-2 核心优化): tiles of Q, K, V are staged in shared memory,
// scores live only on chip, the softmax is computed online with a running
// max and sum, the output is rescaled lazily and normalised once, and one
// statistic (LSE) per row is written.  Work is split over query blocks
// (Q-split), and the elementwise mask is applied only on tiles the mask
// compiler classified PARTIAL.
//
// GB300 mapping.  One persistent CTA per SM, 10 warps:
//   warp 9       TMA producer: claims work items from the cost-sorted list
//                through an atomic counter, loads Q (two 128-row sub-tiles)
//                and streams K, V tiles through a 5-stage ring;
//   warp 8       MMA issuer: S_x = Q_x K^T and O_x += P_x V with tcgen05.mma;
//                TMEM holds S0, S1, O0, O1 (4 x 128 columns) and P_x (bf16)
//                overwrites the first 64 columns of S_x once the softmax has
//                read it, so O_x += P_x V reads its A operand from TMEM;
//   warps 0-7    two softmax warpgroups, one per 128-row sub-tile; thread r
//                owns TMEM lane r (row r): it reads the score row, applies
//                the mask, runs the online softmax in base 2, rescales O in
//                TMEM only when its running max grows by more than 2^8,
//                writes P back into TMEM, and at the end normalises O and
//                writes O and LSE.
// With dropout (a compile-time instantiation), each softmax thread draws the
// keep bytes of its row chunk by chunk (two Philox calls per 32 keys); P goes
// into TMEM with the dropped entries zeroed (a byte-permute mask over the
// packed bf16 pairs) while the row sum l keeps them, and the final
// normalisation multiplies by 1/kp.
// Per sub-tile the MMA thread issues O_x += P_x(t-1) V(t-1) and then
// S_x(t) = Q_x K(t)^T (tcgen05.mma executes in issue order, so S_x(t) does not
// overwrite P_x(t-1) before it is read); while one warpgroup computes
// exponentials the tensor core runs the other sub-tile's products.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lca_dropout.cuh"
#include "lca_internal.h"
#include "sm103.cuh"

namespace lca {
namespace {

constexpr int kThreads = 320;
constexpr int kStages = 5;
constexpr uint32_t kTileBytes = 32768;   // 128 rows x 128 bf16
constexpr uint32_t kChunkBytes = 16384;  // 128 rows x 64 bf16: one 128-byte-swizzled TMA box
constexpr int kOffQ = 0;                 // Q sub-tile x at x * kTileBytes
constexpr int kOffKV = 2 * kTileBytes;   // K/V ring
constexpr int kOffCtl = kOffKV + kStages * kTileBytes;
constexpr int kSmemBytes = kOffCtl + 1024 + 1024;  // control block + alignment slack

enum : int {
  B_QFULL = 0,
  B_QEMPTY = 1,
  B_KVFULL = 2,
  B_KVEMPTY = B_KVFULL + kStages,
  B_SFULL = B_KVEMPTY + kStages,
  B_PFULL = B_SFULL + 2,
  B_OFULL = B_PFULL + 2,
  B_ITFULL = B_OFULL + 2,
  B_ITEMPTY = B_ITFULL + 2,
  B_DRAIN = B_ITEMPTY + 2,
  B_COUNT = B_DRAIN + 1
};

// 64 bytes, broadcast from the producer to the other roles; the segment's
// descriptor and the first list entry travel with the item, so the softmax
// warps start an item without a global load
struct Item {
  int valid, e0, qb, head, hm, cnt;
  long long ebase;
  SegInfo sg;
};
static_assert(sizeof(Item) == 64, "two items fill the 128 bytes between the barriers and the TMEM slot");

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);  // S = Q K^T (both K-major)
constexpr uint32_t kIdescO = idesc_bf16_f32(128, 128, false, true);   // O += P V (P in TMEM, V N-major)
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// Loads and the MMA warp's uses follow the same order: K0, V0, K1, V1, ...
__device__ __forceinline__ uint32_t k_load_index(int t) { return static_cast<uint32_t>(2 * t); }
__device__ __forceinline__ uint32_t v_load_index(int t) { return static_cast<uint32_t>(2 * t + 1); }

__device__ __forceinline__ bool wait1(uint64_t* bar, uint32_t parity, const AttnArgs& a, int where) {
  return mbar_wait(bar, parity, a.status, a.wait_limit_ns, kStatusTimeout, where);
}
// Warp-uniform wait: every lane polls, the warp proceeds only if all succeed.
__device__ __forceinline__ bool waitw(uint64_t* bar, uint32_t parity, const AttnArgs& a, int where) {
  const bool ok = mbar_wait(bar, parity, a.status, a.wait_limit_ns, kStatusTimeout, where);
  return __all_sync(0xFFFFFFFFu, ok);
}

// ------------------------------------------------------------------ producer
// `counts` (shared memory) receives the CTA's work items and its full and
// partial (sub-tile, key tile) units, for the optional per-CTA profile.
__device__ __forceinline__ void producer(const AttnArgs& a, const CUtensorMap* tq, const CUtensorMap* tk,
                                         const CUtensorMap* tv, uint8_t* sQ, uint8_t* sKV, uint64_t* bar,
                                         Item* items, uint32_t* counts) {
  const PlanView& pv = a.pv;
  const uint32_t* entries = static_cast<const uint32_t*>(a.entries);
  uint32_t n_items = 0, n_full = 0, n_part = 0;
  uint32_t kv_iter = 0;
  uint32_t issued = 0;  // K/V loads issued (ring index of the next one)
  int q_issued = 0;     // Q loads issued
  int it = 0;
  for (;; ++it) {
    const int slot = it & 1;
    if (it >= 2 && !wait1(&bar[B_ITEMPTY + slot], ((it >> 1) - 1) & 1, a, 10)) goto abort;
    {
      const int w = atomicAdd(a.counter, 1);
      Item inf;
      inf.valid = 0;
      if (w < a.n_work) {
        // an item is 256 rows of one head, or (paired) 128 rows of two heads
        const int R = a.fwd_pair ? pv.R128 : pv.R256;
        const int* qstart = a.fwd_pair ? pv.q128_start : pv.q256_start;
        int row, head;
        if (a.row_group < 0) {
          seg_major_item(w, qstart, pv.n_seg, a.expand, row, head);
        } else {
          int sorted_row;
          item_of(w, a.n_work / a.expand, a.expand, a.row_group, sorted_row, head);
          row = a.order[sorted_row];
        }
        const int hm = row / R, rr = row % R;
        const int s = find_bucket(qstart, pv.n_seg, rr);
        inf.valid = 1;
        inf.sg = pv.segs[s];
        inf.qb = rr - qstart[s];
        inf.hm = hm;
        inf.head = (pv.hm_count == 1) ? (a.fwd_pair ? 2 * head : head) : hm;
        inf.cnt = a.cnt[row];
        inf.ebase = a.fwd_pair ? hm * pv.dq_per_hm + pv.dq_off[s] + static_cast<long long>(inf.qb) * pv.segs[s].nk
                               : hm * pv.fwd_per_hm + pv.fwd_off[s] + static_cast<long long>(inf.qb) * pv.segs[s].nk;
      }
      inf.e0 = (inf.valid && inf.cnt > 0) ? static_cast<int>(entries[inf.ebase]) : 0;
      items[slot] = inf;
      mbar_arrive(&bar[B_ITFULL + slot]);
      if (!inf.valid) {
        counts[0] = n_items;
        counts[1] = n_full;
        counts[2] = n_part;
        return;
      }
      ++n_items;

      const SegInfo sg = inf.sg;
      if (it >= 1 && !wait1(&bar[B_QEMPTY], (it - 1) & 1, a, 11)) goto abort;
      mbar_arrive_expect_tx(&bar[B_QFULL], 2 * kTileBytes);
      const int y0 = sg.q_off + inf.qb * (a.fwd_pair ? 1 : 2) * kTile;
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_2d(sQ + x * kTileBytes + c * kChunkBytes, tq, &bar[B_QFULL],
                      (inf.head + (a.fwd_pair ? x : 0)) * kHeadDim + c * 64, y0 + (a.fwd_pair ? 0 : x * kTile));
      q_issued = it + 1;

      const int g = inf.head / pv.G;
      const int n = inf.cnt;
      uint32_t e_next = static_cast<uint32_t>(inf.e0);
      for (int t = 0; t < n; ++t) {
        const uint32_t e = e_next;
        if (t + 1 < n) e_next = entries[inf.ebase + t + 1];
        const uint32_t c0 = (e >> 24) & 3u, c1 = (e >> 26) & 3u;
        n_full += (c0 == kTileFull) + (c1 == kTileFull);
        n_part += (c0 == kTilePartial) + (c1 == kTilePartial);
        const int yk = sg.k_off + static_cast<int>(e & 0xFFFFFFu) * kTile;
#pragma unroll
        for (int which = 0; which < 2; ++which) {  // K(t) then V(t)
          const uint32_t idx = kv_iter + 2 * t + which;
          const int stg = idx % kStages;
          if (idx >= kStages && !wait1(&bar[B_KVEMPTY + stg], ((idx / kStages) - 1) & 1, a, 12)) goto abort;
          mbar_arrive_expect_tx(&bar[B_KVFULL + stg], kTileBytes);
          const CUtensorMap* m = which ? tv : tk;
          tma_load_2d(sKV + stg * kTileBytes, m, &bar[B_KVFULL + stg], g * kHeadDim, yk);
          tma_load_2d(sKV + stg * kTileBytes + kChunkBytes, m, &bar[B_KVFULL + stg], g * kHeadDim + 64, yk);
          issued = idx + 1;
        }
      }
      kv_iter += 2 * n;
    }
  }
abort:
  // Let the copies already issued land before the CTA leaves.
  for (uint32_t d = 0; d < kStages && d < issued; ++d) {
    const uint32_t idx = issued - 1 - d;
    mbar_wait(&bar[B_KVFULL + idx % kStages], (idx / kStages) & 1, nullptr, 100000000ull, 0, 0);
  }
  if (q_issued >= 1) mbar_wait(&bar[B_QFULL], (q_issued - 1) & 1, nullptr, 100000000ull, 0, 0);
}

// ------------------------------------------------------------------ MMA issuer
__device__ __forceinline__ void mma_issuer(const AttnArgs& a, uint8_t* sQ, uint8_t* sKV, uint64_t* bar, Item* items,
                                           uint32_t tbase) {
  const uint32_t* entries = static_cast<const uint32_t*>(a.entries);
  // operand descriptors built once; every MMA below only adds a byte offset
  const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16, 1024);           // Q_x, K-major
  const uint64_t dK0 = sdesc_sw128(smem_u32(sKV), 16, 1024);          // K tile, K-major
  const uint64_t dV0 = sdesc_sw128(smem_u32(sKV), kChunkBytes, 1024); // V tile, N-major
  uint32_t kv_iter = 0;
  uint32_t p_iss[2] = {0, 0};
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!waitw(&bar[B_ITFULL + slot], (it >> 1) & 1, a, 20)) goto abort;
    {
      const Item inf = items[slot];
      if ((threadIdx.x & 31) == 0) mbar_arrive(&bar[B_ITEMPTY + slot]);
      if (!inf.valid) return;
      if (!waitw(&bar[B_QFULL], it & 1, a, 21)) goto abort;
      tc_fence_after();
      const int n = inf.cnt;
      bool first_pv[2] = {true, true};
      uint32_t e_cur = static_cast<uint32_t>(inf.e0), e_prev = 0u;
      for (int t = 0; t <= n; ++t) {
        const uint32_t e_nxt = (t + 1 < n) ? entries[inf.ebase + t + 1] : 0u;
        const uint32_t vidx = kv_iter + v_load_index(t - 1), kidx = kv_iter + k_load_index(t);
        const int vst = vidx % kStages, kst = kidx % kStages;
        bool v_ready = false, k_ready = false;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const uint32_t tS = tbase + 128 * x, tO = tbase + 256 + 128 * x;
          if (t >= 1 && ((e_prev >> (24 + 2 * x)) & 3u) != 0) {  // O_x += P_x(t-1) V(t-1), P_x from TMEM
            if (!v_ready) {
              if (!waitw(&bar[B_KVFULL + vst], (vidx / kStages) & 1, a, 24)) goto abort;
              v_ready = true;
            }
            if (!waitw(&bar[B_PFULL + x], p_iss[x] & 1, a, 25)) goto abort;
            tc_fence_after();
            const uint64_t dV = desc_add(dV0, vst * kTileBytes);
            const uint32_t acc0 = first_pv[x] ? 0u : 1u;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              umma_ts(tO, tS + 8 * ks, desc_add(dV, ks * 2048), kIdescO, ks > 0 ? 1u : acc0);
            first_pv[x] = false;
            umma_commit(&bar[B_OFULL + x]);
            ++p_iss[x];
          }
          if (t < n && ((e_cur >> (24 + 2 * x)) & 3u) != 0) {  // S_x(t) = Q_x K(t)^T, after PV_x(t-1)
            if (!k_ready) {
              if (!waitw(&bar[B_KVFULL + kst], (kidx / kStages) & 1, a, 22)) goto abort;
              k_ready = true;
            }
            tc_fence_after();
            const uint64_t dK = desc_add(dK0, kst * kTileBytes);
            const uint64_t dQx = desc_add(dQ0, x * kTileBytes);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t koff = (ks >> 2) * kChunkBytes + (ks & 3) * 32;
              umma_ss(tS, desc_add(dQx, koff), desc_add(dK, koff), kIdescS, ks > 0 ? 1u : 0u);
            }
            umma_commit(&bar[B_SFULL + x]);
          }
        }
        if (t >= 1) umma_commit(&bar[B_KVEMPTY + vst]);
        if (t < n) {
          umma_commit(&bar[B_KVEMPTY + kst]);
          if (t == n - 1) umma_commit(&bar[B_QEMPTY]);
        }
        e_prev = e_cur;
        e_cur = e_nxt;
      }
      if (n == 0) umma_commit(&bar[B_QEMPTY]);
      kv_iter += 2 * n;
    }
  }
abort:
  umma_commit(&bar[B_DRAIN]);
  mbar_wait(&bar[B_DRAIN], 0, nullptr, 100000000ull, 0, 0);
}

// ------------------------------------------------------------------ softmax warpgroup
// The softmax reads a 128-column S row from TMEM twice (once for the row
// maximum, once for the exponentials) in 32-column chunks, so that only two
// chunks are live in registers at a time.
//
// Score of column k of a chunk, -inf where the mask word clears it.
template <bool kMasked>
__device__ __forceinline__ float score(uint32_t raw, uint32_t bits, int k) {
  return (!kMasked || ((bits >> k) & 1u)) ? __uint_as_float(raw) : -INFINITY;
}

// Partial tiles run rolled copies of the two passes: their code is a
// fraction of the fully unrolled full-tile passes, so the instruction cache
// keeps both when tiles of the two kinds alternate (measured: windowed and
// block-sparse masks 7-13% faster in the forward, full tiles unchanged).
//
// Folds one 64-column half of the row (chunks 2cp, 2cp+1) into eight
// independent partial maxima (3-input max), so the row maximum is not one
// 128-long dependency chain.
template <bool kMasked>
__device__ __forceinline__ void row_max_half(float (&mp)[8], uint32_t tS, int cp, uint32_t m0, uint32_t m1) {
  uint32_t r0[32], r1[32];
  tmem_ld32(tS + 64 * cp, r0);
  tmem_ld32(tS + 64 * cp + 32, r1);
  tmem_ld_wait();
#pragma unroll
  for (int g = 0; g < 2; ++g) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      mp[j] = fmax3(mp[j], score<kMasked>(r0[16 * g + j], m0, 16 * g + j),
                    score<kMasked>(r0[16 * g + 8 + j], m0, 16 * g + 8 + j));
      mp[j] = fmax3(mp[j], score<kMasked>(r1[16 * g + j], m1, 16 * g + j),
                    score<kMasked>(r1[16 * g + 8 + j], m1, 16 * g + 8 + j));
    }
  }
}

// Row maximum of the 128 scores.
template <bool kMasked>
__device__ __forceinline__ float tile_row_max(uint32_t tS, const uint32_t (&mb)[4]) {
  float mp[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) mp[j] = -INFINITY;
  if constexpr (kMasked) {
#pragma unroll 1
    for (int cp = 0; cp < 2; ++cp) row_max_half<true>(mp, tS, cp, cp ? mb[2] : mb[0], cp ? mb[3] : mb[1]);
  } else {
#pragma unroll
    for (int cp = 0; cp < 2; ++cp) row_max_half<false>(mp, tS, cp, 0u, 0u);
  }
  return fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
}

// Chunk c (columns 32c..32c+31) of the exponential pass: waits for its TMEM
// load, starts the next chunk's load into the other buffer, and writes the 16
// bf16 pairs of P over columns 16c..16c+15 (which belong to chunks already
// read); the f32 values are added to the four packed partial sums.  With
// dropout the chunk draws the keep bytes of its 32 keys (key groups g0 + 2c,
// g0 + 2c + 1 of query row `row`); dropped entries are written as 0 but still
// counted in the sum.
template <bool kMasked, bool kDrop>
__device__ __forceinline__ void exp_chunk(uint32_t tS, int c, const uint32_t (&cur)[32], uint32_t (&nxt)[32],
                                          uint32_t bits, uint64_t sl2x2, uint64_t nb2, uint64_t (&acc)[4],
                                          const AttnArgs& a, const DropCtx& dc, uint32_t row, uint32_t head,
                                          uint32_t g0) {
  tmem_ld_wait();
  if (c + 1 < 4) tmem_ld32(tS + 32 * (c + 1), nxt);
  uint32_t pk[16];
  uint32_t ks[8];  // keep signs of the chunk's 32 keys, 4 per word
  if (kDrop) {
    const uint4 r0 = philox4x32_10(g0 + 2 * c, row, head, 0u, a.drop_keys);
    const uint4 r1 = philox4x32_10(g0 + 2 * c + 1, row, head, 0u, a.drop_keys);
    ks[0] = keep_signs(r0.x, dc);
    ks[1] = keep_signs(r0.y, dc);
    ks[2] = keep_signs(r0.z, dc);
    ks[3] = keep_signs(r0.w, dc);
    ks[4] = keep_signs(r1.x, dc);
    ks[5] = keep_signs(r1.y, dc);
    ks[6] = keep_signs(r1.z, dc);
    ks[7] = keep_signs(r1.w, dc);
  }
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint64_t sv = f2(score<kMasked>(cur[2 * k], bits, 2 * k), score<kMasked>(cur[2 * k + 1], bits, 2 * k + 1));
    const uint64_t xx = ffma2(sv, sl2x2, nb2);
    const uint64_t pp = f2(ex2_approx(f2lo(xx)), ex2_approx(f2hi(xx)));
    acc[k & 3] = fadd2(acc[k & 3], pp);
    pk[k] = pack_bf16x2(f2lo(pp), f2hi(pp));
    if (kDrop) pk[k] &= (k & 1) ? keep_halves<1>(ks[k >> 1]) : keep_halves<0>(ks[k >> 1]);
  }
  tmem_st16(tS + 16 * c, pk);
}

// P = 2^(s*scale*log2(e) - base) for the thread's row, written as bf16 pairs
// over the first 64 columns of S in TMEM; returns the row sum of P in f32.
template <bool kMasked, bool kDrop>
__device__ __forceinline__ float tile_exp(uint32_t tS, const uint32_t (&mb)[4], float sl2, float base,
                                          const AttnArgs& a, const DropCtx& dc, uint32_t row, uint32_t head,
                                          uint32_t g0) {
  const uint64_t sl2x2 = f2(sl2, sl2), nb2 = f2(-base, -base);
  uint64_t acc[4] = {0, 0, 0, 0};  // four independent packed partial sums
  uint32_t ra[32], rb[32];
  tmem_ld32(tS, ra);
  if constexpr (kMasked) {
#pragma unroll 1
    for (int c = 0; c < 4; c += 2) {
      exp_chunk<true, kDrop>(tS, c, ra, rb, c ? mb[2] : mb[0], sl2x2, nb2, acc, a, dc, row, head, g0);
      exp_chunk<true, kDrop>(tS, c + 1, rb, ra, c ? mb[3] : mb[1], sl2x2, nb2, acc, a, dc, row, head, g0);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 4; c += 2) {
      exp_chunk<false, kDrop>(tS, c, ra, rb, ~0u, sl2x2, nb2, acc, a, dc, row, head, g0);
      exp_chunk<false, kDrop>(tS, c + 1, rb, ra, ~0u, sl2x2, nb2, acc, a, dc, row, head, g0);
    }
  }
  const uint64_t t = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
  return f2lo(t) + f2hi(t);
}

// Aligned uniform block maps: a warp's 32 rows and a 32-column chunk lie in
// one (query block, key block) pair, so the chunk is kept or masked for the
// whole warp (bit c of keep4).  Masked chunks are neither loaded nor
// exponentiated (their P is written as 0); kept ones need no selects.
__device__ __forceinline__ float tile_row_max_blk(uint32_t tS, uint32_t keep4) {
  float mp[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) mp[j] = -INFINITY;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    if (!((keep4 >> c) & 1u)) continue;  // warp-uniform
    uint32_t r[32];
    tmem_ld32(tS + 32 * c, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 8; ++j)
      mp[j] = fmax3(mp[j], fmax3(__uint_as_float(r[j]), __uint_as_float(r[8 + j]), __uint_as_float(r[16 + j])),
                    __uint_as_float(r[24 + j]));
  }
  return fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
}

__device__ __forceinline__ float tile_exp_blk(uint32_t tS, uint32_t keep4, float sl2, float base) {
  const uint64_t sl2x2 = f2(sl2, sl2), nb2 = f2(-base, -base);
  uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t pk[16];
    if ((keep4 >> c) & 1u) {  // warp-uniform
      uint32_t r[32];
      tmem_ld32(tS + 32 * c, r);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const uint64_t xx = ffma2(f2(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1])), sl2x2, nb2);
        const uint64_t pp = f2(ex2_approx(f2lo(xx)), ex2_approx(f2hi(xx)));
        acc[k & 3] = fadd2(acc[k & 3], pp);
        pk[k] = pack_bf16x2(f2lo(pp), f2hi(pp));
      }
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) pk[k] = 0u;
    }
    // P of chunk c goes over columns 16c..16c+15, which belong to chunks
    // already read or not needed
    tmem_st16(tS + 16 * c, pk);
  }
  const uint64_t t = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
  return f2lo(t) + f2hi(t);
}

template <int kForm, bool kDrop>
__device__ __forceinline__ void softmax_wg(const AttnArgs& a, int x, uint64_t* bar, Item* items, uint32_t tbase) {
  constexpr bool kCols = kForm == kFormCols;
  const PlanView& pv = a.pv;
  const uint32_t* entries = static_cast<const uint32_t*>(a.entries);
  const int wq = (threadIdx.x >> 5) & 3;
  const int lane = threadIdx.x & 31;
  const int row = wq * 32 + lane;  // TMEM lane = row of the sub-tile
  const uint32_t tl = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tbase + tl + 128 * x;
  const uint32_t tO = tbase + tl + 256 + 128 * x;
  __nv_bfloat16* O = static_cast<__nv_bfloat16*>(a.o);
  const float sl2 = a.scale_log2;
  const DropCtx dc = make_drop_ctx(a.drop_t);
  uint32_t s_cons = 0, p_prod = 0;
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!waitw(&bar[B_ITFULL + slot], (it >> 1) & 1, a, 30 + x)) return;
    const Item inf = items[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_ITEMPTY + slot]);
    if (!inf.valid) return;
    const SegInfo sg = inf.sg;
    // row inside the segment and query head of this sub-tile
    const int i = a.fwd_pair ? inf.qb * kTile + row : inf.qb * 2 * kTile + x * kTile + row;
    const int head = inf.head + (a.fwd_pair ? x : 0);
    const bool valid = i < sg.q_len;
    const Span row_sp = row_mask_ctx(pv.mask, sg, i);  // the row's span or query block, for every tile
    float m_use = -INFINITY, l = 0.f;
    bool any = false;
    uint32_t e_next = static_cast<uint32_t>(inf.e0);
    for (int t = 0; t < inf.cnt; ++t) {
      const uint32_t e = e_next;  // the next entry's load overlaps this tile's work
      if (t + 1 < inf.cnt) e_next = entries[inf.ebase + t + 1];
      const uint32_t cls = (e >> (24 + 2 * x)) & 3u;
      if (cls == kTileEmpty) continue;
      const int kt = static_cast<int>(e & 0xFFFFFFu);
      // mask words of a partial tile, computed while S is still being produced
      uint32_t mb[4] = {~0u, ~0u, ~0u, ~0u};
      // aligned block maps: one keep bit per 32-key chunk for the warp's rows,
      // when the warp's rows and the tile's keys all lie inside the segment
      bool blk = false;
      uint32_t keep4 = 0;
      if constexpr (kForm == kFormBlocks) {
        const int i0 = i - lane;  // the warp's first row
        blk = cls == kTilePartial && i0 + 32 <= sg.q_len && kt * kTile + kTile <= sg.k_len;
        if (blk) {
          const int qb = q_block_of(pv.mask, sg.q_off + i0);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            keep4 |= block_kept(pv.mask, inf.hm, qb, k_block_of(pv.mask, sg.k_off + kt * kTile + 32 * c)) ? 1u << c : 0u;
        }
      }
      if (cls == kTilePartial && !blk) {
        const uint32_t vw = row_tile_word(pv.mask, sg, inf.hm, i, kt, row_sp);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          mb[c] = mask_bits_row<kCols>(pv.mask, sg, inf.hm, i, kt * kTile + 32 * c, row_sp, vw);
      }
      if (!waitw(&bar[B_SFULL + x], s_cons & 1, a, 32 + x)) return;
      ++s_cons;
      tc_fence_after();
      const float mx = blk ? tile_row_max_blk(tS, keep4)
                           : ((cls == kTilePartial) ? tile_row_max<true>(tS, mb) : tile_row_max<false>(tS, mb));
      const float m_new = fmaxf(m_use, mx * sl2);
      float factor = 1.f;
      bool need = false;
      if (!any) {
        m_use = m_new;
      } else if (m_new > m_use + kRescaleThreshold) {
        factor = ex2_approx(m_use - m_new);
        need = true;
        m_use = m_new;
      }
      // P = exp2(s*scale*log2e - m) as bf16 pairs, written over the first 64
      // columns of S_x in TMEM (the A operand of O_x += P_x V)
      const float base = (m_use == -INFINITY) ? 0.f : m_use;
      const uint32_t grow = static_cast<uint32_t>(sg.q_off + i), g0 = static_cast<uint32_t>(kt * 8);
      float sum;
      if (blk)
        sum = tile_exp_blk(tS, keep4, sl2, base);
      else
        sum = (cls == kTilePartial) ? tile_exp<true, kDrop>(tS, mb, sl2, base, a, dc, grow, head, g0)
                                    : tile_exp<false, kDrop>(tS, mb, sl2, base, a, dc, grow, head, g0);
      l = l * factor + sum;
      if (__any_sync(0xFFFFFFFFu, need)) {
        // the previous O_x += P_x V must have finished before O_x is rescaled
        if (!waitw(&bar[B_OFULL + x], (p_prod - 1) & 1, a, 34 + x)) return;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tO + 32 * c, r);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * factor);
          tmem_st32(tO + 32 * c, r);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_PFULL + x]);
      ++p_prod;
      any = true;
    }
    // epilogue: O = O / l (bf16), LSE = (m + log2 l) ln 2
    __nv_bfloat16* orow = O + (static_cast<size_t>(sg.q_off + (valid ? i : 0)) * pv.Hq + head) * kHeadDim;
    if (any) {
      if (!waitw(&bar[B_OFULL + x], (p_prod - 1) & 1, a, 36 + x)) return;
      tc_fence_after();
      float inv = (l > 0.f) ? 1.f / l : 0.f;
      if (kDrop) inv *= a.drop_inv;
      uint32_t r[2][32];
      tmem_ld32(tO, r[0]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c < 3) tmem_ld32(tO + 32 * (c + 1), r[(c + 1) & 1]);
        if (valid) {
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            w[k] = pack_bf16x2(__uint_as_float(r[c & 1][2 * k]) * inv, __uint_as_float(r[c & 1][2 * k + 1]) * inv);
          if (a.out_v8) {
            st_global_v8(orow + 32 * c, w);
            st_global_v8(orow + 32 * c + 16, w + 8);
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<uint4*>(orow + 32 * c + 8 * u) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
          }
        }
        if (c < 3) tmem_ld_wait();
      }
    } else if (valid) {
#pragma unroll
      for (int u = 0; u < 16; ++u) *reinterpret_cast<uint4*>(orow + 8 * u) = make_uint4(0, 0, 0, 0);
    }
    if (valid) {
      a.lse[static_cast<size_t>(head) * pv.Tq + sg.q_off + i] =
          (l > 0.f) ? (m_use + log2f(l)) * kLn2 : -INFINITY;
    }
    tc_fence_before();
  }
}

template <int kForm, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sKV = sm + kOffKV;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kOffCtl);
  Item* items = reinterpret_cast<Item*>(sm + kOffCtl + 512);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffCtl + 640);
  uint32_t* counts = reinterpret_cast<uint32_t*>(sm + kOffCtl + 768);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(&bar[b], 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar[B_PFULL + x], 4);  // one arrival per softmax warp
      mbar_init(&bar[B_ITEMPTY + x], 9);
    }
    counts[0] = counts[1] = counts[2] = 0;
    if (a.prof != nullptr) *reinterpret_cast<unsigned long long*>(counts + 4) = globaltimer_ns();
    fence_mbar_init();
  }
  if (warp == 9 && lane == 0) {
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 9) {
    if (lane == 0) producer(a, &tmQ, &tmK, &tmV, sQ, sKV, bar, items, counts);
  } else if (warp == 8) {
    mma_issuer(a, sQ, sKV, bar, items, tbase);
  } else {
    softmax_wg<kForm, kDrop>(a, warp >> 2, bar, items, tbase);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (a.prof != nullptr && threadIdx.x == 0) write_cta_record(a.prof, counts);
}

}  // namespace

void launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, int num_sms,
                cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(fwd_kernel<kFormSpans, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    cudaFuncSetAttribute(fwd_kernel<kFormCols, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    cudaFuncSetAttribute(fwd_kernel<kFormBlocks, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    cudaFuncSetAttribute(fwd_kernel<kFormSpans, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    cudaFuncSetAttribute(fwd_kernel<kFormCols, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    configured = true;
  }
  const int grid = max(1, min(num_sms, a.n_work));
  note_launches(1);
  const bool cols = a.pv.mask.kind == kFlashMask, drop = a.drop_t > 0;
  const bool blocks = a.pv.mask.kind == kBlockSparseUniform && a.pv.mask.aligned;
  if (cols && drop)
    fwd_kernel<kFormCols, true><<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, a);
  else if (cols)
    fwd_kernel<kFormCols, false><<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, a);
  else if (drop)  // dropout on a block map takes the per-row mask words
    fwd_kernel<kFormSpans, true><<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, a);
  else if (blocks)
    fwd_kernel<kFormBlocks, false><<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, a);
  else
    fwd_kernel<kFormSpans, false><<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, a);
}

}  // namespace lca

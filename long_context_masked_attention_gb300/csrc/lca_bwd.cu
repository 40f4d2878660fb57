// lca_bwd.cu — masked attention backward for sm_103a (tcgen05 + TMEM + TMA).
//
// The gradient of O = softmax(tau Q K^T) V (FlashAttention review page,
// FlashAttention-2 核心优化, 反向传播), with P recomputed from the stored
// row statistic LSE and D_i = dO_i . O_i from the prepass:
//   dP = dO V^T,  dS = P * (dP - D),  dV = P^T dO,  dK = tau dS^T Q,
//   dQ = tau dS K.
// The page splits the backward both ways because dQ_i = sum_j dS_ij K_j
// crosses key blocks.  Here that is two kernels, neither using atomics:
//  * dkv_kernel — one work item per (KV head, key tile of 128 keys): it keeps
//    K and V resident, walks every query head of the group and every 64-row
//    query step that attends the tile (key-major list), and accumulates dV
//    and dK in TMEM.  Per step: S^T = K Q^T and dP^T = V dO^T (TMEM),
//    P^T, dS^T computed by 8 warps (thread = key row) and written back to
//    TMEM as bf16, then dV += P^T dO and dK += dS^T Q.
//  * dq_kernel — one work item per (query head, 128-row query tile): per key
//    tile S = Q K^T, dP = dO V^T (TMEM), dS by 8 warps (thread = query row),
//    then dQ += dS K.
// Both are persistent (one CTA per SM), claim cost-sorted items through an
// atomic counter, and use one TMA producer warp and one MMA-issue warp.
// Dropout (a compile-time instantiation of both) regenerates the forward's
// keep bits Z from the same counters: with P~ = P * Z / kp and D scaled by kp
// in the prepass, the kernels form dS' = P * (Z * dP~ - kp D) = kp dS and
// P * Z, and the epilogues multiply dQ, dK, dV by 1 / kp.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lca_dropout.cuh"
#include "lca_internal.h"
#include "sm103.cuh"

namespace lca {
namespace {

constexpr int kThreads = 320;  // 8 compute warps + MMA warp + TMA warp
constexpr uint32_t kTile128 = 32768;  // 128 rows x 128 bf16
constexpr uint32_t kChunk128 = 16384; // 128 rows x 64 bf16
constexpr uint32_t kTile64 = 16384;   // 64 rows x 128 bf16
constexpr uint32_t kChunk64 = 8192;   // 64 rows x 64 bf16
constexpr uint32_t kIdesc128 = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdesc64 = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t kIdescMN = idesc_bf16_f32(128, 128, false, true);

__device__ __forceinline__ bool wait1(uint64_t* bar, uint32_t parity, const AttnArgs& a, int where) {
  return mbar_wait(bar, parity, a.status, a.wait_limit_ns, kStatusTimeout, where);
}
__device__ __forceinline__ bool waitw(uint64_t* bar, uint32_t parity, const AttnArgs& a, int where) {
  const bool ok = mbar_wait(bar, parity, a.status, a.wait_limit_ns, kStatusTimeout, where);
  return __all_sync(0xFFFFFFFFu, ok);
}

// 32 f32 values (TMEM words) times `mul` as 32 bf16 at p: two 32-byte stores
// when the output is 32-byte aligned (v8), else four 16-byte ones.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* p, const uint32_t (&r)[32], float mul, bool v8) {
  uint32_t w[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(__uint_as_float(r[2 * k]) * mul, __uint_as_float(r[2 * k + 1]) * mul);
  if (v8) {
    st_global_v8(p, w);
    st_global_v8(p + 16, w + 8);
  } else {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      *reinterpret_cast<uint4*>(p + 8 * u) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
  }
}

// ====================================================================== dQ
namespace dq {

// Shared memory: Q and dO tiles of the item, a 3-slot K ring and a 2-slot V
// ring.  TMEM: S [0,128), dP [128,256), dQ [256,384), dS as bf16 pairs in
// [384,448), read by the dQ product directly, and the item's dO rows as bf16
// pairs in [448,512): the compute warps copy them there from shared memory
// at the start of each item, and dP = dO V^T takes its A operand from TMEM,
// so each key tile's products read 32 KB less from shared memory.
constexpr int kKRing = 3, kVRing = 2;
constexpr int kOffQ = 0;
constexpr int kOffDO = kOffQ + kTile128;
constexpr int kOffK = kOffDO + kTile128;
constexpr int kOffV = kOffK + kKRing * kTile128;
constexpr int kOffCtl = kOffV + kVRing * kTile128;
constexpr int kSmemBytes = kOffCtl + 1024 + 1024;

enum : int {
  B_QFULL = 0, B_QEMPTY,
  B_KFULL, B_KEMPTY = B_KFULL + kKRing, B_VFULL = B_KEMPTY + kKRing, B_VEMPTY = B_VFULL + kVRing,
  B_SFULL = B_VEMPTY + kVRing, B_SEMPTY, B_DSFULL, B_DSEMPTY, B_DQFULL, B_DOFULL,
  B_ITFULL, B_ITEMPTY = B_ITFULL + 2, B_DRAIN = B_ITEMPTY + 2, B_COUNT
};

// 64 bytes; the segment's descriptor and the first list entry travel with
// the item, so the compute warps start an item without a global load
struct Item {
  int valid, e0, qt, head, hm, cnt;
  long long ebase;
  SegInfo sg;
};
static_assert(sizeof(Item) == 64, "two items fill the 128 bytes between the barriers and the TMEM slot");

// `counts` (shared memory) receives the CTA's work items and its full and
// partial key tiles, for the optional per-CTA profile.
__device__ __forceinline__ void producer(const AttnArgs& a, const CUtensorMap* tq, const CUtensorMap* tk,
                                         const CUtensorMap* tv, const CUtensorMap* tdo, uint8_t* sm, uint64_t* bar,
                                         Item* items, uint32_t* counts) {
  const PlanView& pv = a.pv;
  const uint32_t* entries = static_cast<const uint32_t*>(a.entries);
  uint32_t n_items = 0, n_full = 0, n_part = 0;
  uint32_t tiles = 0;  // key tiles loaded so far
  uint32_t k_issued = 0, v_issued = 0;
  int q_issued = 0;
  int it = 0;
  for (;; ++it) {
    const int slot = it & 1;
    if (it >= 2 && !wait1(&bar[B_ITEMPTY + slot], ((it >> 1) - 1) & 1, a, 110)) goto abort;
    {
      const int w = atomicAdd(a.counter, 1);
      Item inf;
      inf.valid = 0;
      if (w < a.n_work) {
        int row, head;
        if (a.row_group < 0) {
          seg_major_item(w, pv.q128_start, pv.n_seg, a.expand, row, head);
        } else {
          int sorted_row;
          item_of(w, a.n_work / a.expand, a.expand, a.row_group, sorted_row, head);
          row = a.order[sorted_row];
        }
        const int hm = row / pv.R128, rr = row % pv.R128;
        const int s = find_bucket(pv.q128_start, pv.n_seg, rr);
        inf.valid = 1;
        inf.sg = pv.segs[s];
        inf.qt = rr - pv.q128_start[s];
        inf.hm = hm;
        inf.head = (pv.hm_count == 1) ? head : hm;
        inf.cnt = a.cnt[row];
        inf.ebase = hm * pv.dq_per_hm + pv.dq_off[s] + static_cast<long long>(inf.qt) * inf.sg.nk;
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
      if (it >= 1 && !wait1(&bar[B_QEMPTY], (it - 1) & 1, a, 111)) goto abort;
      mbar_arrive_expect_tx(&bar[B_QFULL], 2 * kTile128);
      const int y0 = sg.q_off + inf.qt * kTile;
      for (int c = 0; c < 2; ++c) {
        tma_load_2d(sm + kOffQ + c * kChunk128, tq, &bar[B_QFULL], inf.head * kHeadDim + c * 64, y0);
        tma_load_2d(sm + kOffDO + c * kChunk128, tdo, &bar[B_QFULL], inf.head * kHeadDim + c * 64, y0);
      }
      q_issued = it + 1;
      const int g = inf.head / pv.G;
      uint32_t e_next = static_cast<uint32_t>(inf.e0);
      for (int t = 0; t < inf.cnt; ++t, ++tiles) {
        const uint32_t e = e_next;
        if (t + 1 < inf.cnt) e_next = entries[inf.ebase + t + 1];
        n_full += ((e >> 24) & 3u) == kTileFull;
        n_part += ((e >> 24) & 3u) == kTilePartial;
        const int kt = static_cast<int>(e & 0xFFFFFFu);
        const int yk = sg.k_off + kt * kTile;
        const int kr = tiles % kKRing, vr = tiles % kVRing;
        if (tiles >= kKRing && !wait1(&bar[B_KEMPTY + kr], ((tiles / kKRing) - 1) & 1, a, 112)) goto abort;
        mbar_arrive_expect_tx(&bar[B_KFULL + kr], kTile128);
        tma_load_2d(sm + kOffK + kr * kTile128, tk, &bar[B_KFULL + kr], g * kHeadDim, yk);
        tma_load_2d(sm + kOffK + kr * kTile128 + kChunk128, tk, &bar[B_KFULL + kr], g * kHeadDim + 64, yk);
        k_issued = tiles + 1;
        if (tiles >= kVRing && !wait1(&bar[B_VEMPTY + vr], ((tiles / kVRing) - 1) & 1, a, 113)) goto abort;
        mbar_arrive_expect_tx(&bar[B_VFULL + vr], kTile128);
        tma_load_2d(sm + kOffV + vr * kTile128, tv, &bar[B_VFULL + vr], g * kHeadDim, yk);
        tma_load_2d(sm + kOffV + vr * kTile128 + kChunk128, tv, &bar[B_VFULL + vr], g * kHeadDim + 64, yk);
        v_issued = tiles + 1;
      }
    }
  }
abort:
  for (uint32_t d = 0; d < kKRing && d < k_issued; ++d) {
    const uint32_t idx = k_issued - 1 - d;
    mbar_wait(&bar[B_KFULL + idx % kKRing], (idx / kKRing) & 1, nullptr, 100000000ull, 0, 0);
  }
  for (uint32_t d = 0; d < kVRing && d < v_issued; ++d) {
    const uint32_t idx = v_issued - 1 - d;
    mbar_wait(&bar[B_VFULL + idx % kVRing], (idx / kVRing) & 1, nullptr, 100000000ull, 0, 0);
  }
  if (q_issued >= 1) mbar_wait(&bar[B_QFULL], (q_issued - 1) & 1, nullptr, 100000000ull, 0, 0);
}

__device__ __forceinline__ void mma_issuer(const AttnArgs& a, uint8_t* sm, uint64_t* bar, Item* items,
                                           uint32_t tbase) {
  const uint32_t base = smem_u32(sm);
  // operand descriptors built once; every MMA below only adds a byte offset
  const uint64_t dQd = sdesc_sw128(base + kOffQ, 16, 1024);
  const uint64_t dKk = sdesc_sw128(base + kOffK, 16, 1024);         // K ring, K-major
  const uint64_t dKn = sdesc_sw128(base + kOffK, kChunk128, 1024);  // K ring, N-major
  const uint64_t dVk = sdesc_sw128(base + kOffV, 16, 1024);
  uint32_t tiles = 0;  // key tiles consumed (ring positions, dS phases)
  uint32_t sdp = 0;    // S/dP products issued (TMEM reuse count)
  uint32_t do_items = 0;  // items whose dO rows were copied into TMEM
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!waitw(&bar[B_ITFULL + slot], (it >> 1) & 1, a, 120)) goto abort;
    {
      const Item inf = items[slot];
      if ((threadIdx.x & 31) == 0) mbar_arrive(&bar[B_ITEMPTY + slot]);
      if (!inf.valid) return;
      if (!waitw(&bar[B_QFULL], it & 1, a, 121)) goto abort;
      tc_fence_after();
      const int n = inf.cnt;
      for (int t = 0; t <= n; ++t) {
        if (t < n) {  // S = Q K^T, dP = dO V^T for key tile t
          const uint32_t idx = tiles + t;
          const int kr = idx % kKRing, vr = idx % kVRing;
          if (sdp >= 1 && !waitw(&bar[B_SEMPTY], (sdp - 1) & 1, a, 122)) goto abort;
          if (!waitw(&bar[B_KFULL + kr], (idx / kKRing) & 1, a, 123)) goto abort;
          tc_fence_after();
          const uint64_t dK = desc_add(dKk, kr * kTile128);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * kChunk128 + (ks & 3) * 32;
            umma_ss(tbase + 0, desc_add(dQd, off), desc_add(dK, off), kIdesc128, ks > 0);
          }
          if (!waitw(&bar[B_VFULL + vr], (idx / kVRing) & 1, a, 124)) goto abort;
          if (t == 0 && !waitw(&bar[B_DOFULL], do_items & 1, a, 126)) goto abort;  // dO rows in TMEM
          tc_fence_after();
          const uint64_t dV = desc_add(dVk, vr * kTile128);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * kChunk128 + (ks & 3) * 32;
            umma_ts(tbase + 128, tbase + 448 + 8 * ks, desc_add(dV, off), kIdesc128, ks > 0);
          }
          umma_commit(&bar[B_SFULL]);
          ++sdp;
        }
        if (t >= 1) {  // dQ += dS K for key tile t-1, dS read from TMEM
          const uint32_t idx = tiles + t - 1;
          const int kr = idx % kKRing;
          if (!waitw(&bar[B_DSFULL], idx & 1, a, 125)) goto abort;
          tc_fence_after();
          const uint64_t dK = desc_add(dKn, kr * kTile128);
          const uint32_t tA = tbase + 384;
          const uint32_t acc0 = (t > 1) ? 1u : 0u;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            umma_ts(tbase + 256, tA + 8 * ks, desc_add(dK, ks * 2048), kIdescMN, ks > 0 ? 1u : acc0);
          }
          umma_commit(&bar[B_DSEMPTY]);
          umma_commit(&bar[B_KEMPTY + kr]);
          if (t == n) umma_commit(&bar[B_DQFULL]);
        }
        if (t < n) {  // the V and Q/dO releases of tile t wait until after the dQ group, so
                      // that only the S/dP commit sits between the two MMA groups
          umma_commit(&bar[B_VEMPTY + (tiles + t) % kVRing]);
          if (t == n - 1) umma_commit(&bar[B_QEMPTY]);
        }
      }
      if (n == 0) umma_commit(&bar[B_QEMPTY]);
      tiles += n;
      do_items += (n > 0);
    }
  }
abort:
  umma_commit(&bar[B_DRAIN]);
  mbar_wait(&bar[B_DRAIN], 0, nullptr, 100000000ull, 0, 0);
}

template <int kForm, bool kDrop>
__device__ __forceinline__ void compute(const AttnArgs& a, uint8_t* sm, uint64_t* bar, Item* items, uint32_t tbase) {
  constexpr bool kCols = kForm == kFormCols;
  const PlanView& pv = a.pv;
  const uint32_t* entries = static_cast<const uint32_t*>(a.entries);
  const DropCtx dc = make_drop_ctx(a.drop_t);
  const float out_scale = kDrop ? a.scale * a.drop_inv : a.scale;
  const uint64_t sl2x2 = f2(a.scale_log2, a.scale_log2);
  const int warp = threadIdx.x >> 5;
  const int wq = warp & 3, half = warp >> 2;
  const int lane = threadIdx.x & 31;
  const int row = wq * 32 + lane;
  const uint32_t tl = static_cast<uint32_t>(wq * 32) << 16;
  __nv_bfloat16* dQ = static_cast<__nv_bfloat16*>(a.dq);
  uint32_t tiles = 0, sdp = 0, items_done = 0;
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!waitw(&bar[B_ITFULL + slot], (it >> 1) & 1, a, 130)) return;
    const Item inf = items[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_ITEMPTY + slot]);
    if (!inf.valid) return;
    // the row's statistics are loaded while the dO rows are copied
    const SegInfo sg = inf.sg;
    const int i = inf.qt * kTile + row;
    const bool valid = i < sg.q_len;
    const size_t stat = static_cast<size_t>(inf.head) * pv.Tq + sg.q_off + i;
    const float nl2v = valid ? a.nlse2[stat] : -INFINITY;
    const float nDv = valid ? a.nD[stat] : 0.f;
    if (inf.cnt > 0) {
      // this item's dO rows into TMEM, the A operand of dP = dO V^T: thread
      // (row, half) copies the row's 64 columns of its half from the
      // 128-byte-swizzled tile (16-byte unit u of row r sits at u ^ (r % 8)).
      // The previous item's last dP has completed: its S/dP commit was
      // waited for before that item's last dS.
      if (!waitw(&bar[B_QFULL], it & 1, a, 135)) return;
      const uint8_t* src = sm + kOffDO + half * kChunk128 + row * 128;
      uint32_t r[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 w = *reinterpret_cast<const uint4*>(src + ((u ^ (row & 7)) << 4));
        r[4 * u] = w.x;
        r[4 * u + 1] = w.y;
        r[4 * u + 2] = w.z;
        r[4 * u + 3] = w.w;
      }
      tmem_st32(tbase + tl + 448 + 32 * half, r);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_DOFULL]);
    }
    const Span row_sp = row_mask_ctx(pv.mask, sg, i);  // the row's span or query block, for every tile
    const uint64_t nl2 = f2(nl2v, nl2v);  // -LSE2, twice
    const uint64_t nD2 = f2(nDv, nDv);
    uint32_t e_next = static_cast<uint32_t>(inf.e0);
    for (int t = 0; t < inf.cnt; ++t, ++tiles) {
      const uint32_t e = e_next;  // the next entry's load overlaps this tile's work
      if (t + 1 < inf.cnt) e_next = entries[inf.ebase + t + 1];
      const uint32_t cls = (e >> 24) & 3u;
      const int kt = static_cast<int>(e & 0xFFFFFFu);
      uint32_t kb[2] = {~0u, ~0u};  // dropout keep bits of this thread's 64 keys, drawn while S is computed
      if (kDrop) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
          kb[c] = keep32(dc, a.drop_keys, static_cast<uint32_t>(sg.q_off + i), static_cast<uint32_t>(inf.head),
                         static_cast<uint32_t>(kt * 8 + half * 4 + 2 * c));
      }
      if (!waitw(&bar[B_SFULL], sdp & 1, a, 131)) return;
      tc_fence_after();
      float s[64], dp[64];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld32(tbase + tl + half * 64 + 32 * c, r);
#pragma unroll
        for (int k = 0; k < 32; ++k) s[32 * c + k] = __uint_as_float(r[k]);
        tmem_ld32(tbase + tl + 128 + half * 64 + 32 * c, r);
#pragma unroll
        for (int k = 0; k < 32; ++k) dp[32 * c + k] = __uint_as_float(r[k]);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_SEMPTY]);
      ++sdp;
      // aligned block maps: one keep bit per 32-key chunk of the thread's
      // half for the warp's 32 rows, when they and the tile's keys all lie
      // inside the segment; a masked chunk's dS is written as zeros
      bool blk = false;
      uint32_t keep2 = 3u;
      if constexpr (kForm == kFormBlocks) {
        const int i0 = inf.qt * kTile + wq * 32;
        blk = cls == kTilePartial && i0 + 32 <= sg.q_len && kt * kTile + kTile <= sg.k_len;
        if (blk) {
          const int qb = q_block_of(pv.mask, sg.q_off + i0);
          keep2 = 0u;
#pragma unroll
          for (int c = 0; c < 2; ++c)
            keep2 |= block_kept(pv.mask, inf.hm, qb, k_block_of(pv.mask, sg.k_off + kt * kTile + half * 64 + 32 * c))
                         ? 1u << c
                         : 0u;
        }
      }
      if (cls == kTilePartial) {
        const uint32_t vw = blk ? 0u : row_tile_word(pv.mask, sg, inf.hm, i, kt, row_sp);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint32_t bits = blk ? (((keep2 >> c) & 1u) ? ~0u : 0u)
                                    : mask_bits_row<kCols>(pv.mask, sg, inf.hm, i, kt * kTile + half * 64 + 32 * c,
                                                           row_sp, vw);
          if (!__all_sync(0xFFFFFFFFu, bits == ~0u)) {  // the warp's 32 rows do not all keep the chunk
#pragma unroll
            for (int k = 0; k < 32; ++k) s[32 * c + k] = ((bits >> k) & 1u) ? s[32 * c + k] : -INFINITY;
          }
        }
      }
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int k = 16 * c; k < 16 * c + 16; ++k) {
          const uint64_t xx = ffma2(f2(s[2 * k], s[2 * k + 1]), sl2x2, nl2);
          const uint64_t pp = f2(ex2_approx(f2lo(xx)), ex2_approx(f2hi(xx)));
          uint64_t dd;
          if (kDrop) {  // dS' = P (Z dP~ - kp D)
            const float z0 = ((kb[k >> 4] >> ((2 * k) & 31)) & 1u) ? dp[2 * k] : 0.f;
            const float z1 = ((kb[k >> 4] >> ((2 * k + 1) & 31)) & 1u) ? dp[2 * k + 1] : 0.f;
            dd = fadd2(f2(z0, z1), nD2);
          } else {
            dd = fadd2(f2(dp[2 * k], dp[2 * k + 1]), nD2);
          }
          const uint64_t ds = fmul2(pp, dd);
          pk[k] = pack_bf16x2(f2lo(ds), f2hi(ds));
        }
      }
      // dS (bf16) into TMEM, this thread's 64 key columns = 32 packed columns,
      // once the previous tile's dQ product has read the buffer
      if (tiles >= 1 && !waitw(&bar[B_DSEMPTY], (tiles - 1) & 1, a, 132)) return;
      tc_fence_after();
      tmem_st32(tbase + tl + 384 + 32 * half, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_DSFULL]);
    }
    __nv_bfloat16* qrow = dQ + (static_cast<size_t>(sg.q_off + (valid ? i : 0)) * pv.Hq + inf.head) * kHeadDim +
                          half * 64;
    if (inf.cnt > 0) {
      if (!waitw(&bar[B_DQFULL], items_done & 1, a, 133)) return;
      ++items_done;
      tc_fence_after();
      // the TMEM read of the second 32 columns overlaps the stores of the first
      uint32_t r[2][32];
      tmem_ld32(tbase + tl + 256 + half * 64, r[0]);
      tmem_ld_wait();
      tmem_ld32(tbase + tl + 256 + half * 64 + 32, r[1]);
      if (valid) store_bf16x32(qrow, r[0], out_scale, a.out_v8);
      tmem_ld_wait();
      if (valid) store_bf16x32(qrow + 32, r[1], out_scale, a.out_v8);
    } else if (valid) {
#pragma unroll
      for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(qrow + 8 * u) = make_uint4(0, 0, 0, 0);
    }
    tc_fence_before();
  }
}

template <int kForm, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kOffCtl);
  Item* items = reinterpret_cast<Item*>(sm + kOffCtl + 512);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffCtl + 640);
  uint32_t* counts = reinterpret_cast<uint32_t*>(sm + kOffCtl + 768);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(&bar[b], 1);
    mbar_init(&bar[B_SEMPTY], 8);  // one arrival per compute warp
    mbar_init(&bar[B_DSFULL], 8);
    mbar_init(&bar[B_DOFULL], 8);
    mbar_init(&bar[B_ITEMPTY], 9);
    mbar_init(&bar[B_ITEMPTY + 1], 9);
    counts[0] = counts[1] = counts[2] = 0;
    if (a.prof != nullptr) *reinterpret_cast<unsigned long long*>(counts + 4) = globaltimer_ns();
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  if (warp == 9) {
    if (lane == 0) producer(a, &tmQ, &tmK, &tmV, &tmDO, sm, bar, items, counts);
  } else if (warp == 8) {
    mma_issuer(a, sm, bar, items, tbase);
  } else {
    compute<kForm, kDrop>(a, sm, bar, items, tbase);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (a.prof != nullptr && threadIdx.x == 0) write_cta_record(a.prof, counts);
}

}  // namespace dq

// ====================================================================== dK / dV
namespace dkv {

constexpr int kRing = 4;                        // Q/dO (and staged statistics) ring depth
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTile128;
constexpr int kOffQ = kOffV + kTile128;          // ring of 64-row Q tiles
constexpr int kOffDO = kOffQ + kRing * kTile64;  // ring of 64-row dO tiles
constexpr int kOffStat = kOffDO + kRing * kTile64;  // kRing buffers of: -LSE*log2e[64], -D[64], meta
constexpr int kStatBytes = 64 * 4 * 2 + 64;
constexpr int kOffCtl = kOffStat + kRing * kStatBytes;
constexpr int kSmemBytes = kOffCtl + 1024 + 1024;

enum : int {
  B_KVFULL = 0, B_KVEMPTY,
  B_QFULL, B_QEMPTY = B_QFULL + kRing, B_MFULL = B_QEMPTY + kRing, B_MEMPTY = B_MFULL + kRing,
  B_SFULL = B_MEMPTY + kRing, B_PFULL = B_SFULL + 2, B_ACCFULL = B_PFULL + 2,
  B_ITFULL, B_ITEMPTY = B_ITFULL + 2, B_DRAIN = B_ITEMPTY + 2, B_COUNT
};

struct Item {
  int valid, kg, kt, g, unit_hm, nsteps;  // unit_hm: first map head of the unit's lists
  int rk;
  int begin;  // first of the unit's steps this item runs (chunks of split units)
  int slot;   // partial-sum slot of a chunk, -1 when the item writes dK/dV itself
};

// Per-step data the producer warp stages for the compute warps (ring slot b):
// the 64 query rows' -LSE*log2(e) and -D, and the step's class, first rows,
// query head, map head and segment.  The compute warps read only shared
// memory; on a partial tile they evaluate the mask themselves.
struct StepMeta {  // 64 bytes
  int cls;
  int row0;  // global query row of the step's first row
  int r0;    // the same row, relative to the segment
  int head;  // query head
  int hm;    // mask map head
  int pad0, pad1, pad2;
  SegInfo sg;
};
__device__ __forceinline__ float* stat_nlse2(uint8_t* sm, int b) {
  return reinterpret_cast<float*>(sm + kOffStat + b * kStatBytes);
}
__device__ __forceinline__ float* stat_nD(uint8_t* sm, int b) { return stat_nlse2(sm, b) + 64; }
__device__ __forceinline__ StepMeta* stat_meta(uint8_t* sm, int b) {
  return reinterpret_cast<StepMeta*>(stat_nlse2(sm, b) + 128);
}

// The whole producer warp runs this loop; lane 0 issues the TMA copies and
// the barrier arrivals, all lanes fetch list entries (32 at a time, so one
// memory latency covers 32 entries) and stage the per-step statistics with
// cp.async, whose completion the step's barrier tracks.
//
// Steps of an item: for each query head of the KV head, each entry of its
// list, each 64-row half of the 128-row query tile that lies inside the
// segment and holds an attended cell.
//
// `counts` (shared memory) receives the CTA's work items and its full and
// partial 64-row steps, for the optional per-CTA profile.
template <bool kCols>
__device__ __forceinline__ void producer(const AttnArgs& a, const CUtensorMap* tq, const CUtensorMap* tk,
                                         const CUtensorMap* tv, const CUtensorMap* tdo, uint8_t* sm, uint64_t* bar,
                                         Item* items, uint32_t* counts) {
  const PlanView& pv = a.pv;
  const int2* entries = static_cast<const int2*>(a.entries);
  const int lane = threadIdx.x & 31;
  uint32_t n_items = 0, n_full = 0, n_part = 0;
  uint32_t steps = 0;
  int kv_issued = 0;
  int it = 0;
  const int n_work = a.n_work_dev[0];
  const int n_runs = a.n_work_dev[1];
  for (;; ++it) {
    const int slot = it & 1;
    if (it >= 2 && !waitw(&bar[B_ITEMPTY + slot], ((it >> 1) - 1) & 1, a, 210)) goto abort;
    {
      int w = 0;
      if (lane == 0) w = atomicAdd(a.counter, 1);
      w = __shfl_sync(0xFFFFFFFFu, w, 0);
      Item inf;
      inf.valid = 0;
      if (w < n_work && a.dkv_seg_major) {
        // whole units, key group by key group, head by head, key tile by key tile
        const int kg = find_bucket(pv.kt_start, pv.n_kg, w / a.expand);
        const int nk = pv.kt_start[kg + 1] - pv.kt_start[kg];
        const int local = w - pv.kt_start[kg] * a.expand;
        const int kt = local % nk;
        const int unit = pv.kt_start[kg] + kt;  // one mask map: unit = key tile row
        inf.valid = 1;
        inf.kg = kg;
        inf.kt = kt;
        inf.rk = unit;
        inf.g = local / nk;
        inf.unit_hm = 0;
        inf.begin = 0;
        inf.nsteps = a.usteps[unit];
        inf.slot = -1;
      } else if (w < n_work) {
        // sorted unit i holding item w; its items are chunk-major, then KV head, so the
        // cost order (longest first) holds across heads and chunks
        int lo = 0, hi = n_runs;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (a.item_start[mid] <= w) lo = mid; else hi = mid;
        }
        // claim position `lo` holds item w; inside its run items go chunk, KV head, unit
        const int run = a.run_at[lo];
        const int first = a.run_first[run];
        const int n_r = ((run + 1 < n_runs) ? a.run_first[run + 1] : a.n_units) - first;
        const int local = w - a.item_start[lo];
        const int per_chunk = n_r * a.expand;
        const int c = local / per_chunk;
        const int rem = local % per_chunk;
        const int e = rem / n_r;
        const int unit = a.order[first + rem % n_r];
        const int P = a.nchunk[unit];
        const int gm = unit / pv.RK, rk = unit % pv.RK;
        const int kg = find_bucket(pv.kt_start, pv.n_kg, rk);
        inf.valid = 1;
        inf.kg = kg;
        inf.kt = rk - pv.kt_start[kg];
        inf.rk = rk;
        inf.g = (pv.hm_count == 1) ? e : gm;
        inf.unit_hm = 0;
        const long long S = a.usteps[unit];
        inf.begin = static_cast<int>(S * c / P);
        inf.nsteps = static_cast<int>(S * (c + 1) / P) - inf.begin;
        inf.slot = (P > 1) ? a.split_start[run] + local : -1;
      }
      if (lane == 0) {
        items[slot] = inf;
        mbar_arrive(&bar[B_ITFULL + slot]);
      }
      if (!inf.valid) {
        if (lane == 0) {
          counts[0] = n_items;
          counts[1] = n_full;
          counts[2] = n_part;
        }
        return;
      }
      ++n_items;
      const KeyGroup grp = pv.kgs[inf.kg];
      const int yk = grp.k_off + inf.kt * kTile;
      if (it >= 1 && !waitw(&bar[B_KVEMPTY], (it - 1) & 1, a, 211)) goto abort;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar[B_KVFULL], 2 * kTile128);
        for (int c = 0; c < 2; ++c) {
          tma_load_2d(sm + kOffK + c * kChunk128, tk, &bar[B_KVFULL], inf.g * kHeadDim + c * 64, yk);
          tma_load_2d(sm + kOffV + c * kChunk128, tv, &bar[B_KVFULL], inf.g * kHeadDim + c * 64, yk);
        }
      }
      kv_issued = it + 1;
      int us = 0;  // steps of the unit walked so far (loads issued only for [begin, begin + nsteps))
      const int us_end = inf.begin + inf.nsteps;
      for (int l = 0; l < pv.G && us < us_end; ++l) {
        const int h = inf.g * pv.G + l;
        const int hm = (pv.hm_count == 1) ? 0 : h;
        // a chunk starting further on skips whole query-head lists, then whole
        // batches of 32 entries, by their step counts
        const int list_steps = a.list_steps[hm * pv.RK + inf.rk];
        if (us + list_steps <= inf.begin) {
          us += list_steps;
          continue;
        }
        const int n_in_list = a.list_cnt[hm * pv.RK + inf.rk];
        const long long ebase = hm * pv.dkv_per_hm + grp.entry_off + static_cast<long long>(inf.kt) * grp.pairs;
        for (int e0 = 0; e0 < n_in_list && us < us_end; e0 += 32) {
          // lane-parallel fetch of up to 32 entries and their segments
          int2 en = make_int2(0, 0);
          SegInfo sgl{};
          int my_steps = 0;
          if (e0 + lane < n_in_list) {
            en = entries[ebase + e0 + lane];
            sgl = pv.segs[en.x];
            const int qt = en.y & 0xFFFFFF;
            const uint32_t sk = static_cast<uint32_t>(en.y >> 26) & 3u;
            my_steps = ((sk & 1u) ? 0 : 1) + ((qt * kTile + 64 < sgl.q_len && !(sk & 2u)) ? 1 : 0);
          }
          const int batch_steps = __reduce_add_sync(0xFFFFFFFFu, my_steps);
          if (us + batch_steps <= inf.begin) {
            us += batch_steps;
            continue;
          }
          const int batch = min(32, n_in_list - e0);
          for (int t = 0; t < batch && us < us_end; ++t) {
            SegInfo sg;
            sg.q_off = __shfl_sync(0xFFFFFFFFu, sgl.q_off, t);
            sg.q_len = __shfl_sync(0xFFFFFFFFu, sgl.q_len, t);
            sg.k_off = __shfl_sync(0xFFFFFFFFu, sgl.k_off, t);
            sg.k_len = __shfl_sync(0xFFFFFFFFu, sgl.k_len, t);
            sg.prefix = __shfl_sync(0xFFFFFFFFu, sgl.prefix, t);
            sg.kg = 0;
            sg.nk = 0;
            sg.pad = 0;
            const int ey = __shfl_sync(0xFFFFFFFFu, en.y, t);
            const int qt = ey & 0xFFFFFF;
            const uint32_t cls = static_cast<uint32_t>(ey >> 24) & 3u;
            const uint32_t skip = static_cast<uint32_t>(ey >> 26) & 3u;  // bit h: half h attends nothing
            for (int half = 0; half < 2; ++half) {
              const int r0 = qt * kTile + 64 * half;
              if (r0 >= sg.q_len || ((skip >> half) & 1u)) continue;
              if (us < inf.begin || us >= us_end) {  // outside this chunk
                ++us;
                continue;
              }
              ++us;
              n_full += cls == kTileFull;
              n_part += cls == kTilePartial;
              const int b = steps % kRing;
              const uint32_t reuse = steps / kRing;  // how many times ring slot b was filled before
              if (reuse >= 1 && !waitw(&bar[B_MEMPTY + b], (reuse - 1) & 1, a, 213)) goto abort;
              float* sl = stat_nlse2(sm, b);
              float* sd = stat_nD(sm, b);
              const size_t row0 = static_cast<size_t>(h) * pv.Tq + sg.q_off;
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                // rows past the segment end read nothing and get 0 (their tile is partial, so masked)
                const int qi = lane + 32 * u;
                const int i = r0 + qi;
                const uint32_t nb = (i < sg.q_len) ? 4u : 0u;
                const size_t src = row0 + ((i < sg.q_len) ? i : 0);
                cp_async_4(sl + qi, a.nlse2 + src, nb);
                cp_async_4(sd + qi, a.nD + src, nb);
              }
              cp_async_mbar_arrive_noinc(&bar[B_MFULL + b]);
              if (lane == 0) {
                StepMeta* meta = stat_meta(sm, b);
                meta->cls = static_cast<int>(cls);
                meta->row0 = sg.q_off + r0;
                meta->r0 = r0;
                meta->head = h;
                meta->hm = hm;
                meta->sg = sg;
              }
              __syncwarp();
              if (lane == 0) mbar_arrive(&bar[B_MFULL + b]);
              if (reuse >= 1 && !waitw(&bar[B_QEMPTY + b], (reuse - 1) & 1, a, 212)) goto abort;
              if (lane == 0) {
                mbar_arrive_expect_tx(&bar[B_QFULL + b], 2 * kTile64);
                const int y = sg.q_off + r0;
                for (int c = 0; c < 2; ++c) {
                  tma_load_2d(sm + kOffQ + b * kTile64 + c * kChunk64, tq, &bar[B_QFULL + b], h * kHeadDim + c * 64,
                              y);
                  tma_load_2d(sm + kOffDO + b * kTile64 + c * kChunk64, tdo, &bar[B_QFULL + b],
                              h * kHeadDim + c * 64, y);
                }
              }
              ++steps;
            }
          }
        }
      }
    }
  }
abort:
  if (lane == 0) {
    for (uint32_t d = 0; d < kRing && d < steps; ++d) {
      const uint32_t idx = steps - 1 - d;
      mbar_wait(&bar[B_QFULL + idx % kRing], (idx / kRing) & 1, nullptr, 100000000ull, 0, 0);
    }
    if (kv_issued >= 1) mbar_wait(&bar[B_KVFULL], (kv_issued - 1) & 1, nullptr, 100000000ull, 0, 0);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void mma_issuer(const AttnArgs& a, uint8_t* sm, uint64_t* bar, Item* items,
                                           uint32_t tbase) {
  const uint32_t base = smem_u32(sm);
  // operand descriptors built once; every MMA below only adds a byte offset
  const uint64_t dKk = sdesc_sw128(base + kOffK, 16, 1024);
  const uint64_t dVk = sdesc_sw128(base + kOffV, 16, 1024);
  const uint64_t dQk = sdesc_sw128(base + kOffQ, 16, 1024);         // Q ring, K-major (B of S^T)
  const uint64_t dOk = sdesc_sw128(base + kOffDO, 16, 1024);        // dO ring, K-major (B of dP^T)
  const uint64_t dQn = sdesc_sw128(base + kOffQ, kChunk64, 1024);   // Q ring, N-major (B of dK)
  const uint64_t dOn = sdesc_sw128(base + kOffDO, kChunk64, 1024);  // dO ring, N-major (B of dV)
  uint32_t steps = 0;  // global step counter (rings and TMEM double buffers)
  int acc_items = 0;
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!waitw(&bar[B_ITFULL + slot], (it >> 1) & 1, a, 220)) goto abort;
    {
      const Item inf = items[slot];
      if ((threadIdx.x & 31) == 0) mbar_arrive(&bar[B_ITEMPTY + slot]);
      if (!inf.valid) return;
      if (!waitw(&bar[B_KVFULL], it & 1, a, 221)) goto abort;
      tc_fence_after();
      const int n = inf.nsteps;
      for (int p = 0; p <= n; ++p) {
        if (p < n) {  // S^T = K Q^T, dP^T = V dO^T into TMEM buffer b, from ring slot r
          // Buffer b last held P^T / dS^T of step idx-2, whose dV/dK products were
          // issued earlier from this thread; MMAs run in issue order, so no wait.
          const uint32_t idx = steps + p;
          const int b = idx & 1, r = idx % kRing;
          if (!waitw(&bar[B_QFULL + r], (idx / kRing) & 1, a, 223)) goto abort;
          tc_fence_after();
          const uint64_t dQ = desc_add(dQk, r * kTile64), dO = desc_add(dOk, r * kTile64);
          const uint32_t tS = tbase + 64 * b, tP = tbase + 128 + 64 * b;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t ao = (ks >> 2) * kChunk128 + (ks & 3) * 32;
            const uint32_t bo = (ks >> 2) * kChunk64 + (ks & 3) * 32;
            umma_ss(tS, desc_add(dKk, ao), desc_add(dQ, bo), kIdesc64, ks > 0);
          }
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t ao = (ks >> 2) * kChunk128 + (ks & 3) * 32;
            const uint32_t bo = (ks >> 2) * kChunk64 + (ks & 3) * 32;
            umma_ss(tP, desc_add(dVk, ao), desc_add(dO, bo), kIdesc64, ks > 0);
          }
          umma_commit(&bar[B_SFULL + b]);
          if (p == n - 1) umma_commit(&bar[B_KVEMPTY]);
        }
        if (p >= 1) {  // dV += P^T dO, dK += dS^T Q for step p-1, P^T and dS^T read from TMEM
          const uint32_t idx = steps + p - 1;
          const int b = idx & 1, r = idx % kRing;
          if (!waitw(&bar[B_PFULL + b], (idx >> 1) & 1, a, 224)) goto abort;
          tc_fence_after();
          const uint64_t dQ = desc_add(dQn, r * kTile64), dO = desc_add(dOn, r * kTile64);
          const uint32_t acc = (p > 1) ? 1u : 0u;
          // queries 16ks..16ks+15 sit in columns 32*(ks/2) + 8*(ks%2) of the buffer (bf16 pairs)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_ts(tbase + 256, tbase + 64 * b + 32 * (ks >> 1) + 8 * (ks & 1), desc_add(dO, ks * 2048), kIdescMN,
                    (ks > 0) ? 1u : acc);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_ts(tbase + 384, tbase + 128 + 64 * b + 32 * (ks >> 1) + 8 * (ks & 1), desc_add(dQ, ks * 2048),
                    kIdescMN, (ks > 0) ? 1u : acc);
          umma_commit(&bar[B_QEMPTY + r]);
          if (p == n) umma_commit(&bar[B_ACCFULL]);
        }
      }
      if (n == 0) umma_commit(&bar[B_KVEMPTY]);
      steps += n;
      acc_items += (n > 0);
    }
  }
abort:
  umma_commit(&bar[B_DRAIN]);
  mbar_wait(&bar[B_DRAIN], 0, nullptr, 100000000ull, 0, 0);
}

template <int kForm, bool kDrop>
__device__ __forceinline__ void compute(const AttnArgs& a, uint8_t* sm, uint64_t* bar, Item* items, uint32_t tbase) {
  constexpr bool kCols = kForm == kFormCols;
  const PlanView& pv = a.pv;
  const DropCtx dc = make_drop_ctx(a.drop_t);
  const float dv_scale = kDrop ? a.drop_inv : 1.f, dk_scale = kDrop ? a.scale * a.drop_inv : a.scale;
  const int warp = threadIdx.x >> 5;
  const int wq = warp & 3, half = warp >> 2;  // half: which 32 of the 64 query columns
  const int lane = threadIdx.x & 31;
  const int j = wq * 32 + lane;  // key row inside the tile = TMEM lane
  const uint32_t tl = static_cast<uint32_t>(wq * 32) << 16;
  const float sl2 = a.scale_log2;
  const uint64_t sl2x2 = f2(sl2, sl2);
  __nv_bfloat16* dK = static_cast<__nv_bfloat16*>(a.dk);
  __nv_bfloat16* dV = static_cast<__nv_bfloat16*>(a.dv);
  uint32_t steps = 0, acc_items = 0;
  for (int it = 0;; ++it) {
    const int slot = it & 1;
    if (!waitw(&bar[B_ITFULL + slot], (it >> 1) & 1, a, 230)) return;
    const Item inf = items[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[B_ITEMPTY + slot]);
    if (!inf.valid) return;
    const KeyGroup grp = pv.kgs[inf.kg];
    for (int p = 0; p < inf.nsteps; ++p, ++steps) {
      const int b = steps & 1, r = steps % kRing;
      if (!waitw(&bar[B_MFULL + r], (steps / kRing) & 1, a, 234)) return;
      const float* s_nlse2 = stat_nlse2(sm, r);
      const float* s_nD = stat_nD(sm, r);
      const StepMeta* meta_s = stat_meta(sm, r);
      const int cls = meta_s->cls;
      // mask bits of a partial tile, bit k = query 32*half + k for this
      // thread's key: FlashMask reads them off the key's column bounds; the
      // other families evaluate one query row per lane over the warp's 32
      // keys and transpose the 32 x 32 bits across the warp
      // (aligned block maps: the warp's 32 keys and 32 queries lie in one
      // block pair when both are inside the segment; a masked pair writes
      // zero P^T and dS^T without reading S^T, dP^T)
      uint32_t mb = ~0u;
      bool skip = false;
      if (cls == kTilePartial) {
        const SegInfo sg = meta_s->sg;
        const int i0 = meta_s->r0 + 32 * half;
        const int j0 = inf.kt * kTile + wq * 32;
        if constexpr (kCols) {
          mb = flashmask_key_bits(pv.mask, sg, inf.kt * kTile + j, i0);
        } else if (kForm == kFormBlocks && i0 + 32 <= sg.q_len && j0 + 32 <= sg.k_len) {
          skip = !block_kept(pv.mask, meta_s->hm, q_block_of(pv.mask, sg.q_off + i0), k_block_of(pv.mask, sg.k_off + j0));
        } else {
          mb = warp_transpose_bits(mask_bits<false>(pv.mask, sg, meta_s->hm, i0 + lane, j0), lane);
        }
      }
      uint32_t kb = ~0u;  // dropout keep bits: bit k = query 32*half + k for this thread's key
      if (kDrop) {
        // lane l draws query row 32*half + l over the warp's 32 keys, then the
        // warp transposes the 32 x 32 bits so that each lane holds its key's
        const uint32_t rowbits = keep32(dc, a.drop_keys, static_cast<uint32_t>(meta_s->row0 + 32 * half + lane),
                                        static_cast<uint32_t>(meta_s->head), static_cast<uint32_t>(inf.kt * 8 + wq * 2));
        kb = warp_transpose_bits(rowbits, lane);
      }
      if (!waitw(&bar[B_SFULL + b], (steps >> 1) & 1, a, 231)) return;
      tc_fence_after();
      uint32_t pp[16], pd[16];
      if (kForm == kFormBlocks && skip) {  // warp-uniform
#pragma unroll
        for (int k = 0; k < 16; ++k) pp[k] = pd[k] = 0u;
      } else {
        float sv[32], dp[32];
        {
          uint32_t r[32];
          tmem_ld32(tbase + tl + 64 * b + 32 * half, r);
#pragma unroll
          for (int k = 0; k < 32; ++k) sv[k] = __uint_as_float(r[k]);
          tmem_ld32(tbase + tl + 128 + 64 * b + 32 * half, r);
#pragma unroll
          for (int k = 0; k < 32; ++k) dp[k] = __uint_as_float(r[k]);
        }
        tmem_ld_wait();
        if (cls == kTilePartial && !__all_sync(0xFFFFFFFFu, mb == ~0u)) {
#pragma unroll
          for (int k = 0; k < 32; ++k) sv[k] = ((mb >> k) & 1u) ? sv[k] : -INFINITY;
        }
        // the staged statistics of this thread's 32 queries as packed pairs
        const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(s_nlse2 + 32 * half);
        const uint64_t* nd2 = reinterpret_cast<const uint64_t*>(s_nD + 32 * half);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint64_t xx = ffma2(f2(sv[2 * k], sv[2 * k + 1]), sl2x2, nl2[k]);
          const float p0 = ex2_approx(f2lo(xx)), p1 = ex2_approx(f2hi(xx));
          if (kDrop) {  // P~ = P Z for dV; dS' = P Z dP~ - P kp D for dK
            const float pz0 = ((kb >> (2 * k)) & 1u) ? p0 : 0.f, pz1 = ((kb >> (2 * k + 1)) & 1u) ? p1 : 0.f;
            pp[k] = pack_bf16x2(pz0, pz1);
            const uint64_t pnd = fmul2(f2(p0, p1), nd2[k]);
            pd[k] = pack_bf16x2(fmaf(pz0, dp[2 * k], f2lo(pnd)), fmaf(pz1, dp[2 * k + 1], f2hi(pnd)));
          } else {
            pp[k] = pack_bf16x2(p0, p1);
            const uint64_t ds = fmul2(f2(p0, p1), fadd2(f2(dp[2 * k], dp[2 * k + 1]), nd2[k]));
            pd[k] = pack_bf16x2(f2lo(ds), f2hi(ds));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_MEMPTY + r]);  // done with this step's staged data
      // P^T and dS^T (bf16 pairs) go over the first 16 of the 32 S^T / dP^T
      // columns this thread just read; the dV/dK products take them from there.
      tmem_st16(tbase + tl + 64 * b + 32 * half, pp);
      tmem_st16(tbase + tl + 128 + 64 * b + 32 * half, pd);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[B_PFULL + b]);
    }
    // epilogue: rows of the key group only
    const int jg = inf.kt * kTile + j;
    const bool valid = jg < grp.k_len;
    const size_t orow = (static_cast<size_t>(grp.k_off + (valid ? jg : 0)) * pv.Hkv + inf.g) * kHeadDim + half * 64;
    if (inf.nsteps > 0 && inf.slot >= 0) {  // chunk of a split unit: f32 partial sums, all 128 rows
      if (!waitw(&bar[B_ACCFULL], acc_items & 1, a, 233)) return;
      ++acc_items;
      tc_fence_after();
      float* pdv = a.partials + static_cast<size_t>(inf.slot) * (2 * kTile * kHeadDim) + j * kHeadDim + half * 64;
      float* pdk = pdv + kTile * kHeadDim;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld32(tbase + tl + 256 + half * 64 + 32 * c, r);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 4; ++u) st_global_v8(pdv + 32 * c + 8 * u, r + 8 * u);
        tmem_ld32(tbase + tl + 384 + half * 64 + 32 * c, r);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 4; ++u) st_global_v8(pdk + 32 * c + 8 * u, r + 8 * u);
      }
    } else if (inf.nsteps > 0) {
      if (!waitw(&bar[B_ACCFULL], acc_items & 1, a, 233)) return;
      ++acc_items;
      tc_fence_after();
      // each TMEM read of 32 columns overlaps the stores of the previous ones
      uint32_t r[2][32];
      tmem_ld32(tbase + tl + 256 + half * 64, r[0]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // dV columns 0-31, 32-63, then dK
        if (c < 3) tmem_ld32(tbase + tl + 256 + 128 * ((c + 1) >> 1) + half * 64 + 32 * ((c + 1) & 1), r[(c + 1) & 1]);
        if (valid) store_bf16x32((c < 2 ? dV : dK) + orow + 32 * (c & 1), r[c & 1], c < 2 ? dv_scale : dk_scale, a.out_v8);
        if (c < 3) tmem_ld_wait();
      }
    } else if (valid) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        *reinterpret_cast<uint4*>(dV + orow + 8 * u) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(dK + orow + 8 * u) = make_uint4(0, 0, 0, 0);
      }
    }
    tc_fence_before();
  }
}

template <int kForm, bool kDrop>
__global__ void __launch_bounds__(kThreads, 1)
    dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kOffCtl);
  Item* items = reinterpret_cast<Item*>(sm + kOffCtl + 512);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffCtl + 640);
  uint32_t* counts = reinterpret_cast<uint32_t*>(sm + kOffCtl + 768);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(&bar[b], 1);
    for (int b = 0; b < 2; ++b) mbar_init(&bar[B_PFULL + b], 8);  // one arrival per compute warp
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&bar[B_MEMPTY + r], 8);
      mbar_init(&bar[B_MFULL + r], 33);  // 32 cp.async completions + the producer's own arrive
    }
    mbar_init(&bar[B_ITEMPTY], 9);
    mbar_init(&bar[B_ITEMPTY + 1], 9);
    counts[0] = counts[1] = counts[2] = 0;
    if (a.prof != nullptr) *reinterpret_cast<unsigned long long*>(counts + 4) = globaltimer_ns();
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  if (warp == 9) {
    producer<kForm == kFormCols>(a, &tmQ, &tmK, &tmV, &tmDO, sm, bar, items, counts);
  } else if (warp == 8) {
    mma_issuer(a, sm, bar, items, tbase);
  } else {
    compute<kForm, kDrop>(a, sm, bar, items, tbase);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (a.prof != nullptr && threadIdx.x == 0) write_cta_record(a.prof, counts);
}

// One block per (sorted unit, KV head of the unit); blocks of units that were
// not split return at once.
__global__ void __launch_bounds__(256) reduce_kernel(const AttnArgs a) {
  const int i = blockIdx.x / a.expand, gi = blockIdx.x % a.expand;
  const int unit = a.order[i];
  const int P = a.nchunk[unit];
  if (P <= 1) return;
  const int r = a.run_of[i];
  const int first = a.run_first[r];
  const int n_runs = a.n_work_dev[1];
  const int n_r = ((r + 1 < n_runs) ? a.run_first[r + 1] : a.n_units) - first;
  const PlanView& pv = a.pv;
  const int gm = unit / pv.RK, rk = unit % pv.RK;
  const int kg = find_bucket(pv.kt_start, pv.n_kg, rk);
  const KeyGroup grp = pv.kgs[kg];
  const int kt = rk - pv.kt_start[kg];
  const int g = (pv.hm_count == 1) ? gi : gm;
  __nv_bfloat16* dK = static_cast<__nv_bfloat16*>(a.dk);
  __nv_bfloat16* dV = static_cast<__nv_bfloat16*>(a.dv);
  for (int idx = threadIdx.x; idx < kTile * (kHeadDim / 4); idx += blockDim.x) {
    const int j = idx / (kHeadDim / 4), d4 = 4 * (idx % (kHeadDim / 4));
    const int jg = kt * kTile + j;
    if (jg >= grp.k_len) continue;
    float4 sv = make_float4(0.f, 0.f, 0.f, 0.f), sk = sv;
    for (int c = 0; c < P; ++c) {
      const float* base = a.partials + static_cast<size_t>(a.split_start[r] + (c * a.expand + gi) * n_r + (i - first)) *
                                           (2 * kTile * kHeadDim);
      const float4 v = *reinterpret_cast<const float4*>(base + j * kHeadDim + d4);
      const float4 k = *reinterpret_cast<const float4*>(base + kTile * kHeadDim + j * kHeadDim + d4);
      sv.x += v.x; sv.y += v.y; sv.z += v.z; sv.w += v.w;
      sk.x += k.x; sk.y += k.y; sk.z += k.z; sk.w += k.w;
    }
    const size_t row = (static_cast<size_t>(grp.k_off + jg) * pv.Hkv + g) * kHeadDim + d4;
    const float vs = a.drop_inv, ks = a.scale * a.drop_inv;  // drop_inv = 1 without dropout
    *reinterpret_cast<uint2*>(dV + row) =
        make_uint2(pack_bf16x2(sv.x * vs, sv.y * vs), pack_bf16x2(sv.z * vs, sv.w * vs));
    *reinterpret_cast<uint2*>(dK + row) =
        make_uint2(pack_bf16x2(sk.x * ks, sk.y * ks), pack_bf16x2(sk.z * ks, sk.w * ks));
  }
}

}  // namespace dkv
}  // namespace

void launch_bwd_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                   const AttnArgs& a, int num_sms, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(dq::dq_kernel<kFormSpans, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, dq::kSmemBytes);
    cudaFuncSetAttribute(dq::dq_kernel<kFormCols, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, dq::kSmemBytes);
    cudaFuncSetAttribute(dq::dq_kernel<kFormBlocks, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, dq::kSmemBytes);
    cudaFuncSetAttribute(dq::dq_kernel<kFormSpans, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, dq::kSmemBytes);
    cudaFuncSetAttribute(dq::dq_kernel<kFormCols, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, dq::kSmemBytes);
    configured = true;
  }
  const int grid = max(1, min(num_sms, a.n_work));
  note_launches(1);
  const bool cols = a.pv.mask.kind == kFlashMask, drop = a.drop_t > 0;
  const bool blocks = a.pv.mask.kind == kBlockSparseUniform && a.pv.mask.aligned;
  if (cols && drop)
    dq::dq_kernel<kFormCols, true><<<grid, kThreads, dq::kSmemBytes, st>>>(tq, tk, tv, tdo, a);
  else if (cols)
    dq::dq_kernel<kFormCols, false><<<grid, kThreads, dq::kSmemBytes, st>>>(tq, tk, tv, tdo, a);
  else if (drop)  // dropout on a block map takes the per-row mask words
    dq::dq_kernel<kFormSpans, true><<<grid, kThreads, dq::kSmemBytes, st>>>(tq, tk, tv, tdo, a);
  else if (blocks)
    dq::dq_kernel<kFormBlocks, false><<<grid, kThreads, dq::kSmemBytes, st>>>(tq, tk, tv, tdo, a);
  else
    dq::dq_kernel<kFormSpans, false><<<grid, kThreads, dq::kSmemBytes, st>>>(tq, tk, tv, tdo, a);
}

void launch_bwd_dkv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                    const AttnArgs& a, int num_sms, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(dkv::dkv_kernel<kFormSpans, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv::kSmemBytes);
    cudaFuncSetAttribute(dkv::dkv_kernel<kFormCols, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv::kSmemBytes);
    cudaFuncSetAttribute(dkv::dkv_kernel<kFormBlocks, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv::kSmemBytes);
    cudaFuncSetAttribute(dkv::dkv_kernel<kFormSpans, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv::kSmemBytes);
    cudaFuncSetAttribute(dkv::dkv_kernel<kFormCols, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv::kSmemBytes);
    configured = true;
  }
  // the item count is known on the device only (split pass); surplus CTAs find no work and exit
  const int grid = max(1, min(num_sms, a.n_work));
  note_launches(1);
  const bool cols = a.pv.mask.kind == kFlashMask, drop = a.drop_t > 0;
  const bool blocks = a.pv.mask.kind == kBlockSparseUniform && a.pv.mask.aligned;
  if (cols && drop)
    dkv::dkv_kernel<kFormCols, true><<<grid, kThreads, dkv::kSmemBytes, st>>>(tq, tk, tv, tdo, a);
  else if (cols)
    dkv::dkv_kernel<kFormCols, false><<<grid, kThreads, dkv::kSmemBytes, st>>>(tq, tk, tv, tdo, a);
  else if (drop)  // dropout on a block map takes the per-row mask words
    dkv::dkv_kernel<kFormSpans, true><<<grid, kThreads, dkv::kSmemBytes, st>>>(tq, tk, tv, tdo, a);
  else if (blocks)
    dkv::dkv_kernel<kFormBlocks, false><<<grid, kThreads, dkv::kSmemBytes, st>>>(tq, tk, tv, tdo, a);
  else
    dkv::dkv_kernel<kFormSpans, false><<<grid, kThreads, dkv::kSmemBytes, st>>>(tq, tk, tv, tdo, a);
}

void launch_dkv_reduce(const AttnArgs& a, cudaStream_t st) {
  const long long blocks = static_cast<long long>(a.n_units) * a.expand;
  if (blocks == 0) return;
  note_launches(1);
  dkv::reduce_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(a);
}

}  // namespace lca

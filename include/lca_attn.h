/* lca_attn.h — C ABI of the GB300 (sm_103a) masked core-attention library.
 *
 * What it computes.  Core attention softmax(Q K^T * scale) V, forward and
 * backward, as defined on the FlashAttention review page
 * ("长上下文能力：FlashAttention vs. RingAttention", FlashAttention-1
 * 问题和瓶颈), computed IO-aware (FlashAttention-1 核心优化: tiling, online
 * softmax, fusion; FlashAttention-2 核心优化: deferred rescaling, one stored
 * row statistic, sequence-parallel work split), under the mask families of
 * the LongCA-bench review ("Long-Context Attention Benchmark", 三 技术架构,
 * 掩码模式分类), over packed batches of token-level shards of arbitrary
 * length ("Efficient Long-context Language Model Training by Core Attention
 * Disaggregation", 方法详解: stateless, composable core attention).
 *
 * Conventions shared by every entry point.
 *  - Tensors are token-major packed, row-major, bf16 unless stated:
 *      Q, O, dO, dQ : [Tq][Hq][d]        K, V, dK, dV : [Tk][Hkv][d]
 *      LSE          : [Hq][Tq] float32, natural log; -inf for a row with no key
 *    d must be 128.  Query head h reads KV head h / (Hq / Hkv).
 *  - Work is described by segments: query rows [q_off, q_off+q_len) attend
 *    keys [k_off, k_off+k_len).  A plain batch is B equal segments, a
 *    document-packed sequence one segment per document, a shard batch one
 *    segment per shard with k_off = its document's start and k_len = the
 *    shard's end within the document.  Causal families align the diagonal
 *    bottom-right (query i sits at key position i + k_len - q_len).
 *    Segments' query ranges must not overlap.  Segments with the same k_off
 *    form a key group; different key groups' key ranges must not overlap.
 *    Query rows outside every segment get O = 0, LSE = -inf, dQ = 0; keys
 *    outside every segment get dK = dV = 0.
 *  - The caller owns every buffer.  Pointers documented "device" are CUDA
 *    device pointers; "host" pointers are read during the call only.  The
 *    calls allocate no device memory: they take a caller-provided workspace
 *    of at least lca_workspace_size() bytes, 256-byte aligned.  (The one
 *    static array of lca_attn_fwd_static_workspace is reserved by CUDA when
 *    it loads this library's device code on a device; see there.)
 *  - Every device pointer must belong to the device that is current when the
 *    call is made (or be managed memory); the stream must belong to that
 *    device too.  A pointer to another device's memory is refused with
 *    LCA_ERR_INVALID_ARG before anything is launched.
 *  - The outputs of lca_attn_fwd (o, lse) and lca_attn_bwd (dq, dk, dv) may
 *    also be page-locked host memory that CUDA maps for the device
 *    (cudaMallocHost, cudaHostAlloc, or cudaHostRegister with mapping): the
 *    kernels store the results into it directly, which on a GB300 goes over
 *    NVLink-C2C to the Grace host's memory and needs no copy afterwards.
 *    Inputs and the workspace must be device (or managed) memory.  The
 *    library asks CUDA what each pointer is before launching: a pointer of
 *    another kind (pageable host memory, an unknown address) makes the call
 *    return LCA_ERR_INVALID_ARG (LCA_ERR_WORKSPACE for the workspace).
 *  - Calls are asynchronous on `stream` and never synchronise, except
 *    lca_read_status.  Argument errors are returned before anything is
 *    launched.  Faults detected on the device (a bounded wait that ran out,
 *    a block index out of range) are recorded in a status word inside the
 *    workspace and read with lca_read_status.
 */
#ifndef LCA_ATTN_H
#define LCA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LCA_API __attribute__((visibility("default")))
#else
#define LCA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LCA_OK = 0,
  LCA_ERR_INVALID_ARG = 1, /* malformed shape, segments or mask descriptor   */
  LCA_ERR_UNSUPPORTED = 2, /* well-formed but outside what the kernels cover */
  LCA_ERR_WORKSPACE = 3,   /* workspace null, misaligned or too small        */
  LCA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed              */
  LCA_ERR_TIMEOUT = 5,     /* device: a bounded pipeline wait ran out        */
  LCA_ERR_DEVICE_ARG = 6   /* device: descriptor data out of range           */
} lca_status;

/* Mask families (LongCA-bench review, 三 技术架构, 掩码模式分类).  i and j are
 * positions inside a segment, ie = i + k_len - q_len.  Readings of the
 * unnamed details are stated per family. */
typedef enum {
  LCA_MASK_FULL = 0,             /* every key                                          */
  LCA_MASK_CAUSAL = 1,           /* j <= ie                                            */
  LCA_MASK_SLIDING = 2,          /* ie - window_left <= j <= ie + window_right          */
  LCA_MASK_CAUSAL_SLIDING = 3,   /* ie - window_left <= j <= ie                         */
  LCA_MASK_DOC = 4,              /* FULL inside each segment (segment = document)      */
  LCA_MASK_CAUSAL_DOC = 5,       /* CAUSAL inside each segment                         */
  LCA_MASK_SHARED_QUESTION = 6,  /* j <= ie and (part(j) == 0 or part(j) == part(ie));
                                    part 0 = question, parts from part_bounds          */
  LCA_MASK_GLOBAL_SLIDING = 7,   /* ie < num_global or j < num_global or
                                    ie - window_left <= j <= ie + window_right          */
  LCA_MASK_CAUSAL_BLOCKWISE = 8, /* j <= ie and (j/block == ie/block or
                                    ie/block == (k_len-1)/block)                       */
  LCA_MASK_PREFIX_LM_CAUSAL = 9, /* j < prefix_len or j <= ie                          */
  LCA_MASK_PREFIX_LM_DOC = 10,   /* j < seg_prefix[segment] or j <= ie                 */
  LCA_MASK_BLOCK_CAUSAL_DOC = 11,/* floor(j/block) <= floor(ie/block)                  */
  LCA_MASK_BLOCK_SPARSE_UNIFORM = 12,  /* keep[h][qb][kb], blocks q_block x kv_block  */
  LCA_MASK_BLOCK_SPARSE_VARIABLE = 13, /* keep[h][qb][kb], blocks from qb/kb_bounds   */
  LCA_MASK_FLASHMASK = 14  /* column-wise (FlashMask, named by the LongCA-bench review as
                              covering every family): key j (global position) is masked
                              for segment rows [lts_j, lte_j) U [uts_j, ute_j)            */
} lca_mask_kind;

typedef struct {
  int32_t q_off, q_len, k_off, k_len;
} lca_segment;

typedef struct {
  int32_t kind; /* lca_mask_kind */
  int32_t window_left, window_right; /* inclusive distances, >= 0 */
  int32_t num_global;                /* GLOBAL_SLIDING, >= 0 */
  int32_t prefix_len;                /* PREFIX_LM_CAUSAL, >= 0 */
  const int32_t* seg_prefix;         /* host [n_seg]: PREFIX_LM_DOC prefix per segment */
  int32_t block;                     /* CAUSAL_BLOCKWISE, BLOCK_CAUSAL_DOC, >= 1 */
  const int32_t* part_bounds;        /* host [n_part_bounds]: SHARED_QUESTION, strictly
                                        increasing key positions, part_bounds[0] == 0,
                                        last >= every segment's k_len, at most 64 */
  int32_t n_part_bounds;
  /* Block-sparse maps.  Block indices are over GLOBAL packed token positions
   * (query row q_off+i, key k_off+j); the mask is also limited to the segment. */
  int32_t q_block, kv_block;  /* UNIFORM: block sizes; kv_block >= 32            */
  const int32_t* qb_bounds;   /* VARIABLE host [n_qb+1]: 0 = b0 < b1 < ... , b_last >= Tq */
  const int32_t* kb_bounds;   /* VARIABLE host [n_kb+1]: every block but the last >= 32 */
  int32_t n_qb, n_kb;         /* VARIABLE: block counts (UNIFORM: ignored)         */
  int32_t heads_in_map;       /* 1 (one map for all heads) or Hq                   */
  const int32_t* blk_row_ptr; /* device [heads_in_map*n_qb+1]: CSR row starts      */
  const int32_t* blk_col_idx; /* device [blk_nnz]: kept kv block indices           */
  int64_t blk_nnz;
  /* FLASHMASK: device int32 [Tk][4] = {lts, lte, uts, ute} per global key
   * position, rows relative to the query segment reading that key; 16-byte
   * aligned.  One map for all heads. */
  const int32_t* col_bounds;
} lca_mask_desc;

typedef struct {
  int32_t Tq, Tk, Hq, Hkv, d;
  int32_t n_seg;
  const lca_segment* segs; /* host [n_seg] */
  float scale;             /* softmax scale; 0 selects 1/sqrt(d) */
} lca_shape;

/* Bytes of workspace that lca_attn_fwd (for_bwd = 0) or lca_attn_bwd
 * (for_bwd = 1) needs for this shape and mask; the same value serves
 * lca_mask_materialize and lca_mask_nnz.  Host only; no CUDA call. */
LCA_API lca_status lca_workspace_size(const lca_shape* shape, const lca_mask_desc* mask, int for_bwd, size_t* bytes);

/* Forward (FlashAttention-2 核心优化: Q-split work, deferred rescale, one LSE
 * per row).  q, k, v: device bf16 inputs; o: bf16 [Tq][Hq][d] output;
 * lse: float [Hq][Tq] output (outputs in device or mapped host memory).
 * q, k, v and o must be 16-byte aligned and lse 4-byte aligned
 * (LCA_ERR_INVALID_ARG otherwise); an o that is 32-byte aligned is written
 * with 32-byte stores, any other with 16-byte ones (same values). */
LCA_API lca_status lca_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const lca_shape* shape,
                        const lca_mask_desc* mask, void* workspace, size_t workspace_bytes, void* stream);

/* Backward (FlashAttention-2 核心优化, 反向传播: dK/dV per key tile, dQ in a
 * separate query-tile pass, D = rowsum(dO * O) prepass).  dout, q, k, v, o:
 * device bf16; lse: device float from lca_attn_fwd; dq, dk, dv: bf16 outputs
 * in device or mapped host memory (written, not accumulated).  Every bf16
 * pointer must be 16-byte aligned (LCA_ERR_INVALID_ARG otherwise); dq, and
 * dk with dv, are written with 32-byte stores when 32-byte aligned.
 * The dK/dV pass runs on a stream the library owns (one per device, highest
 * priority), forked from `stream` and joined back to it with events, so that
 * the dQ pass runs beside it; all of the call's work still comes after the
 * work queued on `stream` before the call and before the work queued after
 * it.  While a profiling hook is on (lca_set_kernel_events or
 * lca_set_cta_profile) the passes run one after another on `stream`. */
LCA_API lca_status lca_attn_bwd(const void* dout, const void* q, const void* k, const void* v, const void* o,
                        const float* lse, void* dq, void* dk, void* dv, const lca_shape* shape,
                        const lca_mask_desc* mask, void* workspace, size_t workspace_bytes, void* stream);

/* Attention dropout ("长上下文能力：FlashAttention vs. RingAttention",
 * FlashAttention-1 核心优化, 算子融合: dropout fused with the matmuls, the
 * mask and the softmax).  Inverted dropout on the probabilities:
 *     O = (P * Z / kp) V,  LSE that of P (unchanged by dropout),
 * with t = floor(256 p + 1/2) (at most 255) and kp = (256 - t) / 256.  Z_ij
 * for query head h, query row i (global packed index) and key j (counted
 * from the first key of row i's segment) is 1 iff byte j % 4 of word
 * (j % 16) / 4 of Philox4x32-10(counter = (j / 16, i, h, 0), key = (seed
 * low 32 bits, seed high 32 bits)) is >= t; the same Z is regenerated by the
 * backward, so a forward and a backward called with equal lca_dropout values
 * are consistent.  p must satisfy 0 <= p < 1 (LCA_ERR_INVALID_ARG
 * otherwise); t = 0 computes exactly what lca_attn_fwd / lca_attn_bwd do. */
typedef struct {
  float p;       /* drop probability */
  uint64_t seed; /* Philox key */
} lca_dropout;

/* lca_attn_fwd with dropout; dropout NULL means none. */
LCA_API lca_status lca_attn_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                                const lca_shape* shape, const lca_mask_desc* mask, const lca_dropout* dropout,
                                void* workspace, size_t workspace_bytes, void* stream);
/* lca_attn_bwd with dropout: o and lse must come from lca_attn_fwd_dropout
 * with the same shape, mask and dropout values; dropout NULL means none. */
LCA_API lca_status lca_attn_bwd_dropout(const void* dout, const void* q, const void* k, const void* v,
                                const void* o, const float* lse, void* dq, void* dk, void* dv,
                                const lca_shape* shape, const lca_mask_desc* mask, const lca_dropout* dropout,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Merge of partial forward results ("长上下文能力：FlashAttention vs.
 * RingAttention", Blockwise Parallel Transformer and RingAttention sections:
 * attention over a union of disjoint key blocks is assembled from each
 * block's output and softmax normaliser).  Part p holds o_parts[p] (device
 * bf16 [Tq][Hq][d]) and lse_parts[p] (device float [Hq][Tq], natural log) for
 * the same queries over a key set disjoint from every other part's, e.g. one
 * lca_attn_fwd call per key chunk.  Writes
 *     lse[h][i] = log sum_p exp(lse_p[h][i])
 *     o[i][h]   = sum_p exp(lse_p[h][i] - lse[h][i]) * o_p[i][h]   (bf16)
 * and o = 0, lse = -inf for rows no part attends (every lse_p = -inf).
 * A causal mask split into key chunks is a FULL call for the chunks below the
 * diagonal plus a CAUSAL call whose segments pair each query chunk with its
 * own, equally long key chunk.
 * o_parts, lse_parts: HOST arrays of n_parts device pointers,
 * 1 <= n_parts <= LCA_MERGE_MAX_PARTS; o may alias o_parts[0] and lse
 * lse_parts[0].  d must be 128; o pointers 16-byte aligned, lse pointers
 * 4-byte aligned.  Asynchronous on `stream`; needs no workspace. */
#define LCA_MERGE_MAX_PARTS 16
LCA_API lca_status lca_attn_merge(const void* const* o_parts, const float* const* lse_parts, int32_t n_parts, void* o,
                                  float* lse, int32_t Tq, int32_t Hq, int32_t d, void* stream);

/* Core-attention disaggregation planner ("Efficient Long-context Language
 * Model Training by Core Attention Disaggregation": core attention is cut
 * into token-level tasks that attention servers rebatch to balance compute).
 * Host only; no CUDA call.  Cuts documents of lengths doc_len[0..n_docs) into
 * query shards and assigns them to n_servers so that the causal attention
 * work per server -- the cells (b(b+1) - a(a+1))/2 of each of its shards
 * [a, b) -- is balanced:
 *   1. each document is cut into equal pieces no longer than max_shard
 *      (0 = no limit; else max_shard >= 2 * min_shard);
 *   2. pieces go to the least-loaded server, most expensive first;
 *   3. while the most loaded server exceeds the mean by more than
 *      `tolerance` (relative), its most expensive piece at least 2*min_shard
 *      long is cut where its cells halve, and step 2 is redone.
 * Shard [a, b) of a document whose keys start at position s is the segment
 * {q_off: its place in the server's packed query buffer, q_len: b - a,
 *  k_off: s, k_len: b} of a CAUSAL call: it attends keys [s, s + b).
 * Shards come out ordered by server, then document, then start.  Up to
 * max_shards entries are written to `shards` (host) and the count to
 * n_shards; server_cells (host, n_servers entries, may be NULL) receives each
 * server's cells per head.  LCA_ERR_WORKSPACE if max_shards is too small
 * (n_shards then holds the count needed). */
typedef struct {
  int32_t doc;    /* document index                        */
  int32_t start;  /* first query token, document-relative  */
  int32_t len;    /* query tokens                          */
  int32_t server; /* attention server it is assigned to    */
} lca_cad_shard;
LCA_API lca_status lca_cad_plan(const int32_t* doc_len, int32_t n_docs, int32_t n_servers, int32_t min_shard,
                                int32_t max_shard, double tolerance, lca_cad_shard* shards, int32_t max_shards,
                                int32_t* n_shards, int64_t* server_cells);

/* Test hook: writes the mask of one segment and query head, evaluated by the
 * same device predicate the attention kernels apply, as bytes (1 = attend)
 * into `out` (device, q_len*k_len, row-major). */
LCA_API lca_status lca_mask_materialize(const lca_shape* shape, const lca_mask_desc* mask, int32_t head, int32_t seg,
                                uint8_t* out, void* workspace, size_t workspace_bytes, void* stream);

/* Test hook: the tile classes of one segment and query head for 128 x 128
 * tiles, one byte per tile written to `out` (device, nq*nk bytes, row-major,
 * nq = ceil(q_len/128), nk = ceil(k_len/128)).  Bits 0-1: 0 empty, 1 full,
 * 2 partial.  A partial tile also sets bit 2 when its query rows [0, 64)
 * attend no key of the tile, bit 3 when its rows [64, 128) (those inside the
 * segment) attend none; the backward key-gradient pass skips those halves. */
LCA_API lca_status lca_mask_tile_classes(const lca_shape* shape, const lca_mask_desc* mask, int32_t head, int32_t seg,
                                 uint8_t* out, void* workspace, size_t workspace_bytes, void* stream);

/* Number of attended (query, key) cells per query head, summed over
 * segments, written to `nnz` (device, uint64 [Hq]).  Used for the effective
 * FLOP count 4*d*nnz (forward) and 10*d*nnz (backward). */
LCA_API lca_status lca_mask_nnz(const lca_shape* shape, const lca_mask_desc* mask, uint64_t* nnz, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Forward pass with a library-owned workspace, for callers that cannot
 * allocate device memory: processes whose device-memory pool was carved out
 * up front and may not grow, or code running where an allocation is not
 * allowed (inside an allocator's own callback, for example).  The pages have
 * no counterpart: this is a deployment convenience of this library.
 * Arguments and results are those of lca_attn_fwd; the caller still passes
 * (and owns) q, k, v, o and lse.
 * Scratch: one static device array of LCA_STATIC_WORKSPACE_BYTES (16 MiB),
 * which every GPU that loads this library holds until the process exits.  A
 * shape whose forward workspace (lca_workspace_size with for_bwd = 0) is
 * larger is rejected with LCA_ERR_WORKSPACE before anything is launched, and
 * lca_last_error_detail says how much it needed.
 * The array is reserved on a device when CUDA loads this library's device
 * code there: with CUDA's default lazy loading that happens at the latest
 * during the first call of this function on the device, which can then fail
 * with LCA_ERR_CUDA if the device is already full.  Make that first call at
 * set-up time, before the rest of device memory is handed out (a small shape
 * will do); it also looks up the array's device address with that device
 * current, so it must come before any stream capture.
 * Every call on a device shares the one array and clears what must start at
 * zero; calls that overlap on the GPU (two streams, or two host threads)
 * race on it, so the caller must serialise them.
 * No device memory is allocated: no cudaMalloc, cudaFree or allocating
 * library routine is called. */
#define LCA_STATIC_WORKSPACE_BYTES (16u << 20)
LCA_API lca_status lca_attn_fwd_static_workspace(const void* q, const void* k, const void* v, void* o, float* lse,
                                                 const lca_shape* shape, const lca_mask_desc* mask, void* stream);

/* Synchronises `stream`, then copies the device status word of the last
 * call that used this workspace: out[0] = lca_status code (0 = none),
 * out[1] = where it was raised.  Each fwd/bwd call clears it first. */
LCA_API lca_status lca_read_status(const void* workspace, int32_t out[2], void* stream);

/* Test hook: launches one block that waits on a barrier nothing arrives at,
 * with a wait limit of `limit_ms`; it must record LCA_ERR_TIMEOUT in the
 * workspace status word and exit. */
LCA_API lca_status lca_probe_wait_timeout(void* workspace, size_t workspace_bytes, int32_t limit_ms, void* stream);

/* Profiling hook.  With a non-null ring of CUDA events (cudaEvent_t handles
 * passed as void*, n_events even), every later fwd/bwd call records one
 * event pair around each of its phases, on its own stream, taking the next
 * pair of the ring (the cursor restarts at each call of this function):
 *   lca_attn_fwd: 0 = mask compiler + cost sort, 1 = forward kernel
 *   lca_attn_bwd: 2 = D prepass, 3 = dK/dV lists + sort, 4 = dK/dV kernel,
 *                 5 = dQ lists + sort, 6 = dQ kernel
 * The phase of each recorded pair is written to `phases` (host, n_events/2
 * entries, may be null).  Pass null to stop.  Process-wide, not thread-safe. */
LCA_API lca_status lca_set_kernel_events(void* const* events, int32_t n_events, int32_t* phases);

/* Profiling hook: per-CTA work and time of the attention kernels, the
 * evidence for how evenly the cost-sorted persistent scheduler spreads work
 * over the SMs.  With a non-null device buffer `buf` of at least
 * LCA_CTA_PROFILE_BYTES (8-byte aligned), every later forward and backward
 * call writes one record per CTA of each attention kernel it launches:
 * kernel slot k (0 forward, 1 dK/dV, 2 dQ) starts at byte k * 1024 * 64, and
 * CTA b's record at 64 * b within it, eight uint64 values:
 *   start and end of the CTA (%globaltimer, ns), work items it ran, full and
 *   partial tile units it ran (forward: 128-row query sub-tile x key tile;
 *   dK/dV: 64-row query step; dQ: 128-row query tile x key tile), the grid
 *   size, the SM it ran on, 0.
 * A call clears its kernel's slot on its stream before the launch, so
 * records of CTAs beyond the grid are zero.  Pass null to stop.
 * LCA_ERR_INVALID_ARG for a short, misaligned or non-device buffer.
 * Process-wide, not thread-safe. */
#define LCA_CTA_PROFILE_BYTES (3u * 1024u * 64u)
LCA_API lca_status lca_set_cta_profile(void* buf, size_t bytes);

/* Text of the last CUDA failure seen by this library in the calling thread
 * (the failing call and the runtime's message), or "" if none. */
LCA_API const char* lca_last_error_detail(void);

/* Number of kernels this library has launched since it was loaded. */
LCA_API uint64_t lca_launch_count(void);

LCA_API const char* lca_status_string(lca_status status);
/* Library revision, 100 + n; n grows whenever an entry point's behaviour
 * changes (102: lca_mask_tile_classes reports the empty-half flags; 103:
 * outputs may be mapped host memory, and every pointer's kind is checked;
 * 104: device pointers of another device than the current one are refused). */
LCA_API int32_t lca_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LCA_ATTN_H */

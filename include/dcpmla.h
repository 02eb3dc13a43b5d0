/*
 * dcpmla.h -- C ABI of libdcpmla.so, the GB300 (sm_103a) hot path of decode context
 * parallelism (DCP) for MLA and DeepSeek-style sparse attention (DSA) decode.
 *
 * DCP shards the KV tokens of every sequence across D shards; each decode row attends
 * to every shard's local KV and the shard results are merged with log-sum-exp weights
 * (LMDeploy PR #4952 "support decode context parallelism for PyTorch MLA", Summary).
 * On one GPU the shards are partitions of one paged KV pool in that GPU's HBM.
 *
 * Conventions shared by every entry point
 *   - Pointers marked (device) are CUDA device pointers; (host) are host pointers.
 *     The caller allocates, owns and frees every buffer.  The library never allocates,
 *     frees or synchronises; inputs are never written.
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream).  A return
 *     of DCP_OK means the work was queued; kernel-side findings go to err_flag.
 *   - Host-side argument checks run before any launch; a failed check returns a
 *     negative dcp_status and launches nothing.  A failed launch returns DCP_ERR_CUDA.
 *   - No kernel traps, asserts or waits without bound.
 *
 * Token row layout of the paged KV pool (a page is page_size consecutive token rows):
 *   DCP_KV_BF16          : 576 bf16 (latent 0..511, RoPE 512..575)              1152 B
 *   DCP_KV_FP8_E4M3_S128 : 512 e4m3 latent | 4 fp32 scales (one per 128 latent
 *                          values, value = e4m3 * scale) | 64 bf16 RoPE          656 B
 * Keys are the whole 576-value row; values are its first 512 values (MLA latent).
 *
 * Owner rule (DCP interleave): global slot t of a sequence lives on shard
 *   (t / I) % D at local slot (t / (I*D))*I + t % I,
 * with I = 1 (token-interleaved, "slot mod D") or I = page_size (page-interleaved,
 * "page mod D").  A shard keeps its slots of a sequence in increasing global order.
 */
#ifndef DCPMLA_H
#define DCPMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t (struct CUstream_st*); declared here so that this
 * header does not need the CUDA headers. */
typedef struct CUstream_st* dcp_stream_t;

typedef enum {
  DCP_OK = 0,
  DCP_ERR_INVALID_ARG = -1,  /* null pointer, bad size, misaligned pointer */
  DCP_ERR_UNSUPPORTED = -2,  /* valid but not implemented (e.g. head count) */
  DCP_ERR_CUDA = -3,         /* a CUDA call or launch failed */
  DCP_ERR_WORKSPACE = -4     /* workspace missing or smaller than required */
} dcp_status;

typedef enum {
  DCP_KV_BF16 = 0,
  DCP_KV_FP8_E4M3_S128 = 1
} dcp_kv_dtype;

/* Bits a kernel ORs into *err_flag (only when err_flag != NULL and checked != 0). */
#define DCP_ERRBIT_SLOT_RANGE 1   /* a slot id past the block table row, or negative local id */
#define DCP_ERRBIT_PAGE_RANGE 2   /* a block-table entry outside [0, num_pages) */
#define DCP_ERRBIT_TIMEOUT 4      /* a kernel-internal wait gave up (reported whenever
                                     err_flag != NULL); the outputs are then invalid */

#define DCP_MAX_SHARDS 64
#define DCP_MAX_TOPK 16384

/* Human-readable text for a dcp_status value (static storage). */
const char* dcp_status_string(int status);

/* ABI version of this header (bumped on any incompatible change). */
#define DCP_ABI_VERSION 2
int dcp_abi_version(void);

/*
 * dcp_remap_topk -- per-shard slot remap of DSA top-k indices.
 * Passage: SGLang PR #42536 "Fix DCP for RoPE sparse attention on Blackwell",
 *   Modifications, "Index remap": take the global top-k slots, keep the ones the shard
 *   owns, convert them to local slot ids, move them to the front of the row and return
 *   the count per row.
 *
 * global_idx (device) [rows][k] int32: global slot ids; any negative entry is padding.
 * dcp        number of shards D, 1..DCP_MAX_SHARDS.
 * interleave I >= 1 of the owner rule (1 or the page size).
 * shard      -1: produce every shard; 0..D-1: produce only that shard.
 * local_idx  (device) [n_out][rows][k] int32, n_out = D (shard = -1) or 1: for shard s
 *            the local ids of the owned slots in their original order, then -1.
 * count      (device) [n_out][rows] int32: number of owned slots of each row.
 * Exact integer work; results are bit-identical to the definition.
 * Errors: DCP_ERR_INVALID_ARG for null pointers, rows < 0, k < 1 or > DCP_MAX_TOPK,
 *   dcp out of range, interleave < 1, shard outside [-1, D).  rows = 0 is a no-op.
 */
int dcp_remap_topk(const int32_t* global_idx, int64_t rows, int32_t k, int32_t dcp,
                   int32_t interleave, int32_t shard, int32_t* local_idx, int32_t* count,
                   dcp_stream_t stream);

/*
 * dcp_local_lengths -- local KV length of each row on one shard for dense decode.
 * Passage: LMDeploy PR #4952, Summary (KV tokens are sharded across ranks; decode
 *   attends to the local KV); a row of visible global length L holds, on shard s, the
 *   slots t < L with owner s.
 * global_len (device) [rows] int32 >= 0; local_len (device) [n_out][rows] int32 with
 * n_out = D (shard = -1) or 1.  Errors as dcp_remap_topk.
 */
int dcp_local_lengths(const int32_t* global_len, int64_t rows, int32_t dcp,
                      int32_t interleave, int32_t shard, int32_t* local_len,
                      dcp_stream_t stream);

/*
 * dcp_kv_cache_write -- store new token rows in the paged pool of their owner shard.
 * Passage: LMDeploy PR #4952, files: "Interleaved DCP KV-cache writes" (each new token is
 *   written to the shard the owner rule assigns it, at that shard's local slot); SGLang
 *   PR #36990, review of quantize_k_cache_separate (an FP8 cache quantises the latent
 *   ("nope") part and keeps the RoPE part separately).
 *
 * kv         (device) [n][576] bf16 token rows (latent 0..511, RoPE 512..575), 16-B aligned.
 * seq, pos   (device) [n] int32: sequence index and global position of each row; a negative
 *            position is padding (skipped).
 * dcp, interleave  the owner rule (see above); shard -1 writes every row, 0..D-1 only the
 *            rows that shard owns.
 * kv_pool    (device) [num_pages][page_size][token bytes], written in place, 16-B aligned.
 * block_table (device) [dcp][num_seqs][bt_stride] int32, as for the fused decode: entry j of
 *            (shard, sequence) is the page holding local slots j*64 .. j*64+63.
 * FP8 rows: per block of 128 latent values scale = amax / 448 (fp32), codes = value / scale
 *   (fp32) rounded to the nearest E4M3 value, ties to even, saturating at 448; an all-zero
 *   block stores scale 0 and zero codes; RoPE is stored as given.  BF16 rows are copied.
 *   The bytes written are identical to that definition (exact integer result).
 * Rows whose sequence or block-table entry is out of range are skipped; with checked != 0
 *   they set DCP_ERRBIT_SLOT_RANGE / DCP_ERRBIT_PAGE_RANGE in *err_flag.  Rows of one call
 *   must not share a destination slot (the stored row is then unspecified).
 * Errors: DCP_ERR_INVALID_ARG for null or misaligned pointers, n < 0, num_pages < 1,
 *   num_seqs < 1, bt_stride < 1, a bad owner rule or shard; DCP_ERR_UNSUPPORTED for another
 *   page size or kv_dtype.  n = 0 is a no-op.
 */
int dcp_kv_cache_write(const void* kv, int64_t n, const int32_t* seq, const int32_t* pos,
                       int32_t dcp, int32_t interleave, int32_t shard, void* kv_pool,
                       int64_t num_pages, int32_t kv_dtype, int32_t page_size,
                       const int32_t* block_table, int32_t num_seqs, int32_t bt_stride,
                       int32_t checked, int32_t* err_flag, dcp_stream_t stream);

/*
 * dcp_topk_local -- DSA top-k producer under DCP, step 1: each shard's candidate list.
 * Passages: LMDeploy PR #4952 "support decode context parallelism for PyTorch MLA",
 *   Summary (for decode, DSA merges local candidates into the global top-k) and its file
 *   list (the DCP top-k kernel packs the distributed candidates and merges them); SGLang
 *   PR #36990, item 2 (with the index cache split across ranks, every indexer layer merges
 *   the ranks' local top-k candidates).
 *
 * scores     (device) [n_in][rows][score_stride] fp32: the indexer score of local slot l of
 *            each row on each shard, l < local_len (later entries are not read); n_in = D
 *            for shard = -1 (block o is shard o), else 1.
 * local_len  (device) [n_in][rows] int32: local slots of the row on that shard (clamped to
 *            [0, score_stride]); dcp_local_lengths gives them from the visible lengths.
 * k          candidates per list, 1..DCP_MAX_TOPK.
 * dcp, interleave, shard  the owner rule; local slot l of shard s is the l-th slot, in
 *            increasing global order, that the rule gives s, i.e. global slot
 *            (l / I)*I*D + s*I + l % I.
 * cand_score (device) [n_in][rows][k] fp32 and cand_idx (device) [n_in][rows][k] int32: the
 *            selected slots as GLOBAL slot ids in increasing order with their scores (the
 *            input values), then (-inf, -1).
 * Selection: a slot is a candidate unless its score is NaN or -inf; candidates rank by
 *   score, higher first (-0 equals +0), equal scores by the smaller global slot id, and the
 *   first min(k, candidates) are selected.  Comparisons only: bit-identical to that rule.
 * Errors: DCP_ERR_INVALID_ARG for null or misaligned (4-B) pointers, rows < 0,
 *   score_stride < 1, k outside [1, DCP_MAX_TOPK], a bad owner rule or shard, or global
 *   slot ids past INT32_MAX.  rows = 0 is a no-op.
 */
int dcp_topk_local(const float* scores, int64_t rows, int32_t score_stride,
                   const int32_t* local_len, int32_t k, int32_t dcp, int32_t interleave,
                   int32_t shard, float* cand_score, int32_t* cand_idx, dcp_stream_t stream);

/*
 * dcp_topk_merge -- DSA top-k producer under DCP, step 2: the global top-k of a row from
 * the D shards' candidate lists (passages as dcp_topk_local).
 *
 * cand_score, cand_idx (device) [dcp][rows][k_in]: every shard's list as dcp_topk_local
 *            writes it (on several GPUs, gathered from the D ranks); an id < 0 is padding.
 * topk       (device) [rows][k] int32: the selected global slot ids in increasing order,
 *            then -1 -- the input layout of dcp_remap_topk and of the fused decode.
 * count      (device, may be NULL) [rows] int32: number of selected slots.
 * Selection as dcp_topk_local over the D*k_in candidates of the row.  Since every global
 *   top-k slot is among its own shard's best k, for k <= k_in the result is the top-k of
 *   the unsharded scores.  Ids must be distinct within a row (else which of the tied
 *   entries are kept is unspecified; at most k are written).
 * Errors: DCP_ERR_INVALID_ARG for null or misaligned pointers, dcp outside
 *   [1, DCP_MAX_SHARDS], rows < 0, k_in < 1, k outside [1, DCP_MAX_TOPK], dcp*k_in past
 *   INT32_MAX.  rows = 0 is a no-op.
 */
int dcp_topk_merge(const float* cand_score, const int32_t* cand_idx, int32_t dcp, int64_t rows,
                   int32_t k_in, int32_t k, int32_t* topk, int32_t* count, dcp_stream_t stream);

/*
 * Arguments of the decode entry points.  Field meaning differs between the per-shard
 * call (mla_decode_partial_lse) and the fused call (mla_decode_dcp_fused) where noted.
 */
typedef struct {
  /* queries */
  const void* q;               /* (device) [rows][heads][576] bf16, 16-B aligned */
  int64_t rows;                /* decode rows (query tokens), >= 0 */
  int32_t heads;               /* query heads per row: a multiple of 16, 16..128 */
  float sm_scale;              /* softmax scale applied to q.k before exp */
  /* paged KV pool shared by all shards */
  const void* kv_pool;         /* (device) [num_pages][page_size][token bytes], 16-B aligned */
  int64_t num_pages;
  int32_t kv_dtype;            /* dcp_kv_dtype */
  int32_t page_size;           /* tokens per page: 64 */
  /* block tables: partial call: [num_shards][num_seqs][bt_stride] starting at the
   * first shard of the call; fused call: [dcp][num_seqs][bt_stride].  Entry j of a
   * (shard, sequence) row is the physical page holding local slots
   * j*page_size .. j*page_size+page_size-1. */
  const int32_t* block_table;  /* (device) */
  int32_t num_seqs;
  int32_t bt_stride;           /* entries per (shard, sequence) row */
  const int32_t* row_seq;      /* (device) [rows] sequence index of each row */
  /* token selection: sparse when idx != NULL, dense otherwise */
  const int32_t* idx;          /* (device) partial: [num_shards][rows][k] local ids as
                                  produced by dcp_remap_topk (valid ids first);
                                  fused: [rows][k] global ids, negatives = padding */
  const int32_t* count;        /* (device) partial sparse: [num_shards][rows] valid ids;
                                  fused: unused (NULL) */
  int32_t k;                   /* top-k row length, 1..DCP_MAX_TOPK (sparse) */
  const int32_t* kv_len;       /* (device) dense: partial: [num_shards][rows] local
                                  lengths (dcp_local_lengths); fused: [rows] visible
                                  global lengths */
  int32_t max_kv_len;          /* dense: an upper bound of kv_len (sizes the split-KV
                                  grid and the workspace); sparse: ignored */
  /* outputs */
  void* out;                   /* (device) partial: [num_shards][rows][heads][512] fp32;
                                  fused: [rows][heads][512] bf16; 16-B aligned */
  float* lse;                  /* (device) partial: [num_shards][rows][heads];
                                  fused: [rows][heads]; natural log; -inf = no KV */
  /* scratch */
  void* workspace;             /* (device) >= mla_decode_workspace_size() bytes, 256-B
                                  aligned; its contents need not persist between calls
                                  and need no initialisation (the tensor-core kernel
                                  writes everything it reads; the CUDA-core kernel clears
                                  its tickets with an asynchronous memset on the stream).
                                  Calls that share a workspace must not overlap on the
                                  GPU. */
  size_t workspace_bytes;
  int32_t num_splits;          /* split-KV factor per row: 0 = library choice */
  /* diagnostics */
  int32_t checked;             /* != 0: bounds-check every slot and page id */
  int32_t* err_flag;           /* (device, optional) DCP_ERRBIT_* ORed in when checked */
  /* kernel choice: DCP_PATH_AUTO or DCP_PATH_CUDA_CORES; the workspace size query must
   * see the same value as the call */
  int32_t kernel_path;
} dcp_mla_decode_args;

/* Values of dcp_mla_decode_args.kernel_path.  AUTO: the tensor-core kernel for 48..128
 * heads, the CUDA-core kernel otherwise.  CUDA_CORES: the CUDA-core kernel for every head
 * count (same results within the tolerances; slower; for comparing the two kernels). */
#define DCP_PATH_AUTO 0
#define DCP_PATH_CUDA_CORES 1

/*
 * mla_decode_partial_lse -- MLA decode attention over one or more shards' local KV,
 * returning the shard output and its log-sum-exp.
 * Passage: SGLang PR #42536, Modifications, "Backend": sparse attention is called with
 *   return_lse=True and rows that have no local KV are fixed up; LMDeploy PR #4952,
 *   Summary: attend to local KV (dense or sparse MLA, BF16 KV and sparse-MLA FP8 KV).
 * For each shard s of the call, row r, head h over the shard's slot set S (sparse: the
 * first count[s][r] local ids of idx[s][r]; dense: local slots 0..kv_len[s][r]-1):
 *   logit_t = sm_scale * q[r][h] . key_t (576 values),  lse = ln sum_t exp(logit_t),
 *   out[s][r][h] = sum_t exp(logit_t - lse) * key_t[0:512];
 * an empty S gives out = 0 and lse = -inf (the fix-up).  Arithmetic: BF16 or exact
 * E4M3->BF16 operands, FP32 accumulation; FP8 scales applied in FP32.
 * num_shards: shards in this call (1..DCP_MAX_SHARDS); arrays are strided by shard.
 * Errors: DCP_ERR_INVALID_ARG (null/misaligned pointers, bad sizes),
 *   DCP_ERR_UNSUPPORTED (heads, page size, dtype), DCP_ERR_WORKSPACE, DCP_ERR_CUDA.
 */
int mla_decode_partial_lse(const dcp_mla_decode_args* args, int32_t num_shards,
                           dcp_stream_t stream);

/*
 * dcp_lse_merge -- merge shard partials with LSE weights.
 * Passage: LMDeploy PR #4952, Summary ("merge outputs using LSE weights") and its
 *   review discussion (merge arithmetic in FP32, merged result stored in BF16);
 *   SGLang PR #36990 "DCP for DSA models with the flashmla_kv backend", review of the
 *   LSE combine, and SGLang PR #42536, Modifications, "Fixes in shared code": when every
 *   shard is empty the result is a zero output and a -inf LSE, not 0/0.
 *   m = max_s lse_s;  m = -inf -> out = 0, lse = -inf;
 *   else w_s = exp(lse_s - m), W = sum_s w_s, out = sum_s w_s out_s / W, lse = m + ln W.
 * part_out (device) [dcp][rows][heads][dv] fp32; part_lse (device) [dcp][rows][heads];
 * out (device) [rows][heads][dv] bf16; lse (device) [rows][heads] fp32.
 * dv: a multiple of 4 (512 for MLA).  Pointers 16-B aligned.
 */
int dcp_lse_merge(const float* part_out, const float* part_lse, int32_t dcp, int64_t rows,
                  int32_t heads, int32_t dv, void* out, float* lse, dcp_stream_t stream);

/*
 * mla_decode_dcp_fused -- the whole DCP decode of a row in one launch: for every
 * global slot of the row, read the key row from its owner shard's pages, attend, and
 * merge across shards on chip; the result equals unsharded attention.
 * Passage: SGLang PR #42536, Follow-ups #1: a fused merge kernel in place of the three
 *   per-layer merge kernels (pack, exchange, LSE combine) is the biggest remaining
 *   latency item; this is its single-GPU form (all shards of a row in one launch).
 * args: fused meanings (global idx or global kv_len, [dcp] block tables, bf16 out).
 * Rows whose work is divided between CTAs are merged without waiting: on the CUDA-core
 * path by the last CTA to finish (an atomic ticket in the workspace), on the tensor-core
 * path by a small merge kernel queued on the same stream after the decode.  Errors as
 * mla_decode_partial_lse.
 */
int mla_decode_dcp_fused(const dcp_mla_decode_args* args, int32_t dcp, int32_t interleave,
                         dcp_stream_t stream);

/*
 * mla_decode_dcp_fused_noalloc -- mla_decode_dcp_fused for callers that cannot
 * allocate device memory.  This entry point has no counterpart on the pages; it exists
 * for integration.  Some callers are handed only their inputs and outputs by a host
 * runtime that owns all device memory (a plugin or custom op inside another inference
 * engine, a serving loop that reserves its memory once at start-up, a step recorded
 * into a CUDA graph), and a cudaMalloc there is refused, breaks the capture or stalls
 * the device, so they cannot supply the split-KV workspace.
 * Same arguments and results as mla_decode_dcp_fused; args->workspace and
 * args->workspace_bytes are ignored.  The scratch is a static device array of
 * DCP_NOALLOC_SCRATCH_BYTES inside the library, held by every GPU that loads it until
 * the process exits.  The call allocates and frees nothing.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.
 *   - It runs the CUDA-core split-KV kernel for every head count (args->kernel_path is
 *     ignored): the tensor-core kernel's scratch (about 0.5 MB per pair of SMs) does not
 *     fit the array.  For 128 heads it is many times slower than mla_decode_dcp_fused.
 *   - With num_splits = 0 the library lowers its split count until the scratch
 *     (rows * splits * heads * 2 KB plus small tables) fits the array.  A call whose
 *     requested num_splits needs more returns DCP_ERR_WORKSPACE and launches nothing;
 *     lower num_splits or the rows per call.
 *   - All calls share the array and it keeps the last call's contents; each call clears
 *     the tickets it needs with an asynchronous memset on its stream.  Calls that overlap
 *     on the GPU (different streams or host threads) race on the array.
 */
#define DCP_NOALLOC_SCRATCH_BYTES (16u << 20)
int mla_decode_dcp_fused_noalloc(const dcp_mla_decode_args* args, int32_t dcp,
                                 int32_t interleave, dcp_stream_t stream);

/*
 * mla_prefill_chunk_dcp -- attention of a prefill chunk's query rows under DCP, as partials
 * merged with LSE weights.
 * Passage: LMDeploy PR #4952, Summary (prefill gathers the cached-prefix KV in bounded
 *   chunks; partial attention results merge with LSE weights).
 *
 * Row r attends to its sequence's cached prefix, global slots [0, kv_len[r]), and to the
 * chunk slots idx[r][0..k) it sees (global ids, -1 padded; the chunk tokens' KV already in
 * the pool).  Steps, on `stream`: each shard's local prefix length; one dense partial per
 * shard over its prefix slots; each shard's chunk slots (the remap); one sparse partial per
 * shard over them; the LSE merge of the 2*dcp partials into out / lse.
 * args: as mla_decode_dcp_fused, with kv_len = the rows' prefix lengths (device, [rows]
 *   int32), max_kv_len >= every one of them, idx / k = the chunk slots, block_table
 *   [dcp][num_seqs][bt_stride]; out [rows][heads][512] bf16, lse [rows][heads] fp32;
 *   workspace of mla_prefill_chunk_workspace_size bytes, 256-B aligned.
 * Errors: as mla_decode_dcp_fused; DCP_ERR_INVALID_ARG without idx or kv_len;
 *   DCP_ERR_UNSUPPORTED for dcp > DCP_MAX_SHARDS / 2 (the merge takes 2*dcp partials).
 */
size_t mla_prefill_chunk_workspace_size(const dcp_mla_decode_args* args, int32_t dcp,
                                        int32_t interleave);
int mla_prefill_chunk_dcp(const dcp_mla_decode_args* args, int32_t dcp, int32_t interleave,
                          dcp_stream_t stream);

/*
 * mla_decode_workspace_size -- bytes of workspace a decode call with these arguments
 * needs (0 when none).  fused = 0 for mla_decode_partial_lse (num_shards_or_dcp =
 * num_shards), 1 for mla_decode_dcp_fused (num_shards_or_dcp = dcp).  Returns
 * (size_t)-1 for invalid arguments.
 */
size_t mla_decode_workspace_size(const dcp_mla_decode_args* args, int32_t num_shards_or_dcp,
                                 int32_t fused);

#ifdef __cplusplus
}
#endif

#endif /* DCPMLA_H */

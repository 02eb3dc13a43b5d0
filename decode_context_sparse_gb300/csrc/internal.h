// Internal launchers of libdcpmla (host side; not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dcpmla.h"
#include "common.cuh"

namespace dcp {

// Device-side view of one decode call (partial or fused).
struct DecodeParams {
  const void* q;          // [rows][heads][576] bf16
  int64_t rows;
  int heads;
  float scale_log2;       // sm_scale * log2(e): logits are kept in base-2 units
  const uint8_t* pool;
  int64_t num_pages;
  int page_size;
  const int32_t* bt;      // partial: [shards][seqs][stride]; fused: [D][seqs][stride]
  int num_seqs;
  int bt_stride;
  const int32_t* row_seq;
  const int32_t* idx;     // sparse ids (local for partial, global for fused) or NULL
  const int32_t* count;   // partial sparse counts
  int k;
  const int32_t* kv_len;  // dense lengths (local for partial, global for fused)
  int D, I;               // fused: owner rule
  OwnerRule rule;         // the same as fast divisions
  int64_t num_units;      // partial: shards * rows; fused: rows
  int shards;             // partial: shards of the call (units per row); fused: 1
  FastDiv shards_div;     // division by shards
  int num_splits;
  void* out;              // partial: fp32 [units][H][512]; fused: bf16 [rows][H][512]
  float* lse;
  float* ws_o;            // split partials [units][splits][H][512]
  float* ws_lse;          // [units][splits][H]
  unsigned* ws_cnt;       // tickets [units][head groups]
  int32_t* err;           // optional error word
  // tensor-core path
  int use_tc;             // 1: decode_tc_kernel, 0: decode_simt_kernel
  int pairs;              // CTA pairs of the persistent grid
  float* tc_o;            // split-unit partials [pairs][2][128][512]
  float* tc_l;            // their LSEs [pairs][2][2][128]
  int64_t* tc_desc;       // [T, pairs owning tiles] + per (pair, slot) (unit, first tile, end tile)
  int32_t* err_timeout;   // error word for bounded-wait timeouts (whenever given)
  int tma_out;            // partial: finished units' rows go out by tiled stores (set at launch)
};

// Per-device facts (csrc/device.cu): the SM count of the current device, and raising a
// kernel's dynamic shared-memory limit once per (device, kernel).
int device_sm_count();
cudaError_t raise_smem_limit(const void* kernel, size_t bytes);

cudaError_t launch_remap_topk(const int32_t* gidx, int64_t rows, int k, int D, int I, int shard,
                              int32_t* local_idx, int32_t* count, cudaStream_t st);
cudaError_t launch_local_lengths(const int32_t* glen, int64_t rows, int D, int I, int shard,
                                 int32_t* llen, cudaStream_t st);
cudaError_t launch_kv_write(const void* kv, int64_t n, const int32_t* seq, const int32_t* pos,
                            int D, int I, int shard, void* pool, int64_t num_pages, int kv_dtype,
                            const int32_t* bt, int num_seqs, int bt_stride, int32_t* err,
                            cudaStream_t st);
// DSA top-k producer: per-shard candidate lists and their merge (csrc/topk.cu).
constexpr int kTkStageMax = 16384;  // list entries staged in shared memory (longer: L2)
struct TopkParams {
  const float* score;     // candidates: [n_in][rows][stride]; merge: [D][rows][stride]
  const int32_t* ids;     // merge: [D][rows][stride] global slot ids
  const int32_t* len;     // candidates: [n_in][rows] local lengths
  int64_t rows;
  int stride;             // candidates: score row stride; merge: entries per shard list
  int D, I, shard;        // candidates: owner rule and shard (-1: list block o is shard o)
  int k;
  int vec;                // lists 16-B aligned with a multiple of 4 entries per row / list
  int stage, kp;          // set by the launchers: staged entries, sort size (merge)
  FastDiv div;            // set by the launchers: candidates: by I; merge: by stride
  float* cand_score;      // candidates: [n_in][rows][k]
  int32_t* cand_idx;
  int32_t* topk;          // merge: [rows][k]
  int32_t* count;         // merge: [rows] or NULL
};
cudaError_t launch_topk_local(TopkParams p, int n_in, cudaStream_t st);
cudaError_t launch_topk_merge(TopkParams p, cudaStream_t st);
cudaError_t launch_lse_merge(const float* part_out, const float* part_lse, int D, int64_t rows,
                             int heads, int dv, void* out, float* lse, cudaStream_t st);

// SIMT decode (any head count that is a multiple of 16).
constexpr int kSimtHeadGroup = 16;
size_t simt_workspace_bytes(int64_t units, int heads, int splits);
int simt_auto_splits(int64_t units, int heads, int64_t max_tokens);
void simt_bind_workspace(DecodeParams& p, void* ws);
cudaError_t launch_decode_simt(const DecodeParams& p, int kv_dtype, bool fused, bool sparse,
                               cudaStream_t st);

// Tensor-core decode (48..128 heads, page size 64).
size_t tc_workspace_bytes(int64_t units, int pairs);
size_t tc_desc_bytes(int pairs);
void tc_bind_workspace(DecodeParams& p, void* ws);
int tc_pairs_for(int64_t units, int64_t tiles_bound);
int tc_tile_slots(int kv_dtype);
cudaError_t launch_decode_tc(const DecodeParams& p, int kv_dtype, bool fused, bool sparse,
                             cudaStream_t st);

// Host-side checks shared by the decode entry points; fills p (workspace not bound).
int prepare_decode(const dcp_mla_decode_args* a, int32_t n, bool fused, int32_t dcp,
                   int32_t interleave, DecodeParams& p, bool& sparse);

}  // namespace dcp

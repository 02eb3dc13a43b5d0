// extern "C" entry points of libdcpmla: host-side argument checks, path choice and
// launches on the caller's stream.  No allocation, no synchronisation.
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

using namespace dcp;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int status_of(cudaError_t e) { return e == cudaSuccess ? DCP_OK : DCP_ERR_CUDA; }

bool valid_rule(int32_t dcp, int32_t interleave) {
  return dcp >= 1 && dcp <= DCP_MAX_SHARDS && interleave >= 1 && interleave <= (1 << 16);
}

}  // namespace

namespace dcp {

// Common checks of a decode call; fills the device params (no workspace binding).
int prepare_decode(const dcp_mla_decode_args* a, int32_t n, bool fused, int32_t dcp,
                   int32_t interleave, DecodeParams& p, bool& sparse) {
  if (a == nullptr) return DCP_ERR_INVALID_ARG;
  if (a->rows < 0 || n < 1 || n > DCP_MAX_SHARDS) return DCP_ERR_INVALID_ARG;
  if (fused && !valid_rule(dcp, interleave)) return DCP_ERR_INVALID_ARG;
  if (!a->q || !a->kv_pool || !a->block_table || !a->row_seq || !a->out || !a->lse)
    return DCP_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->kv_pool, 16) || !aligned(a->out, 16) ||
      !aligned(a->lse, 4))
    return DCP_ERR_INVALID_ARG;
  if (a->num_pages < 1 || a->num_seqs < 1 || a->bt_stride < 1) return DCP_ERR_INVALID_ARG;
  if (a->kv_dtype != DCP_KV_BF16 && a->kv_dtype != DCP_KV_FP8_E4M3_S128)
    return DCP_ERR_UNSUPPORTED;
  if (a->heads < kSimtHeadGroup || a->heads > 128 || a->heads % kSimtHeadGroup != 0)
    return DCP_ERR_UNSUPPORTED;
  if (a->page_size != 64) return DCP_ERR_UNSUPPORTED;
  if (!(a->sm_scale == a->sm_scale)) return DCP_ERR_INVALID_ARG;  // NaN
  sparse = a->idx != nullptr;
  if (sparse) {
    if (a->k < 1 || a->k > DCP_MAX_TOPK) return DCP_ERR_INVALID_ARG;
    if (!fused && a->count == nullptr) return DCP_ERR_INVALID_ARG;
  } else {
    if (a->kv_len == nullptr || a->max_kv_len < 0) return DCP_ERR_INVALID_ARG;
  }
  if (a->num_splits < 0) return DCP_ERR_INVALID_ARG;
  if (a->kernel_path != DCP_PATH_AUTO && a->kernel_path != DCP_PATH_CUDA_CORES)
    return DCP_ERR_INVALID_ARG;
  const int64_t units = fused ? a->rows : a->rows * n;
  const int64_t max_tokens = sparse ? a->k : a->max_kv_len;
  int splits = a->num_splits > 0 ? a->num_splits : simt_auto_splits(units, a->heads, max_tokens);
  if (splits > 64) splits = 64;

  p.q = a->q;
  p.rows = a->rows;
  p.heads = a->heads;
  p.scale_log2 = a->sm_scale * kLog2e;
  p.pool = static_cast<const uint8_t*>(a->kv_pool);
  p.num_pages = a->num_pages;
  p.page_size = a->page_size;
  p.bt = a->block_table;
  p.num_seqs = a->num_seqs;
  p.bt_stride = a->bt_stride;
  p.row_seq = a->row_seq;
  p.idx = a->idx;
  p.count = a->count;
  p.k = a->k;
  p.kv_len = a->kv_len;
  p.D = fused ? dcp : 1;
  p.I = fused ? interleave : 1;
  p.rule = make_owner_rule(p.D, p.I);
  p.num_units = units;
  p.shards = fused ? 1 : n;
  p.shards_div = make_fastdiv(p.shards);
  p.num_splits = splits;
  p.out = a->out;
  p.lse = a->lse;
  p.ws_o = nullptr;
  p.ws_lse = nullptr;
  p.ws_cnt = nullptr;
  p.err = a->checked ? a->err_flag : nullptr;
  // tensor-core path for 48..128 heads (rows of up to 128 heads, padded)
  // (the tensor-core path addresses pool rows with 32-bit gather coordinates)
  p.use_tc = (a->kernel_path == DCP_PATH_AUTO && a->heads > 32 &&
              a->num_pages <= (int64_t)(INT32_MAX / 64)) ? 1 : 0;
  p.pairs = 0;
  p.tc_o = p.tc_l = nullptr;
  p.tc_desc = nullptr;
  p.err_timeout = a->err_flag;  // timeouts are reported whenever err_flag is given
  if (p.use_tc) {
    const int tn = tc_tile_slots(a->kv_dtype);
    p.pairs = tc_pairs_for(units, units * ((max_tokens + tn - 1) / tn));
  }
  return DCP_OK;
}

}  // namespace dcp

namespace {

// Binds the caller's workspace.  The tensor-core decode writes every split descriptor it
// later reads; the CUDA-core path's split tickets are cleared with an asynchronous memset
// on the call's stream.  Either way a workspace may be shared by calls of different shapes.
int bind_workspace(const dcp_mla_decode_args* a, DecodeParams& p, cudaStream_t st) {
  if (p.use_tc) {
    const size_t need = tc_workspace_bytes(p.num_units, p.pairs);
    if (a->workspace == nullptr || a->workspace_bytes < need || !aligned(a->workspace, 256))
      return DCP_ERR_WORKSPACE;
    tc_bind_workspace(p, a->workspace);
    return DCP_OK;
  }
  const size_t need = simt_workspace_bytes(p.num_units, p.heads, p.num_splits);
  if (need == 0) return DCP_OK;
  if (a->workspace == nullptr || a->workspace_bytes < need || !aligned(a->workspace, 256))
    return DCP_ERR_WORKSPACE;
  simt_bind_workspace(p, a->workspace);
  const size_t nbytes = (size_t)p.num_units * (p.heads / kSimtHeadGroup) * sizeof(unsigned);
  return status_of(cudaMemsetAsync(p.ws_cnt, 0, nbytes, st));
}

}  // namespace

extern "C" {

const char* dcp_status_string(int status) {
  switch (status) {
    case DCP_OK: return "DCP_OK";
    case DCP_ERR_INVALID_ARG: return "DCP_ERR_INVALID_ARG: invalid argument";
    case DCP_ERR_UNSUPPORTED: return "DCP_ERR_UNSUPPORTED: unsupported configuration";
    case DCP_ERR_CUDA: return "DCP_ERR_CUDA: a CUDA call or launch failed";
    case DCP_ERR_WORKSPACE: return "DCP_ERR_WORKSPACE: workspace missing, misaligned or too small";
    default: return "unknown dcp_status";
  }
}

int dcp_abi_version(void) { return DCP_ABI_VERSION; }

int dcp_remap_topk(const int32_t* global_idx, int64_t rows, int32_t k, int32_t dcp,
                   int32_t interleave, int32_t shard, int32_t* local_idx, int32_t* count,
                   dcp_stream_t stream) {
  if (!global_idx || !local_idx || !count) return DCP_ERR_INVALID_ARG;
  if (rows < 0 || rows > INT32_MAX || k < 1 || k > DCP_MAX_TOPK) return DCP_ERR_INVALID_ARG;
  if (!valid_rule(dcp, interleave) || shard < -1 || shard >= dcp) return DCP_ERR_INVALID_ARG;
  return status_of(launch_remap_topk(global_idx, rows, k, dcp, interleave, shard, local_idx, count,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int dcp_local_lengths(const int32_t* global_len, int64_t rows, int32_t dcp, int32_t interleave,
                      int32_t shard, int32_t* local_len, dcp_stream_t stream) {
  if (!global_len || !local_len || rows < 0) return DCP_ERR_INVALID_ARG;
  if (!valid_rule(dcp, interleave) || shard < -1 || shard >= dcp) return DCP_ERR_INVALID_ARG;
  return status_of(launch_local_lengths(global_len, rows, dcp, interleave, shard, local_len,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int dcp_kv_cache_write(const void* kv, int64_t n, const int32_t* seq, const int32_t* pos,
                       int32_t dcp, int32_t interleave, int32_t shard, void* kv_pool,
                       int64_t num_pages, int32_t kv_dtype, int32_t page_size,
                       const int32_t* block_table, int32_t num_seqs, int32_t bt_stride,
                       int32_t checked, int32_t* err_flag, dcp_stream_t stream) {
  if (!kv || !seq || !pos || !kv_pool || !block_table) return DCP_ERR_INVALID_ARG;
  if (n < 0 || num_pages < 1 || num_seqs < 1 || bt_stride < 1) return DCP_ERR_INVALID_ARG;
  if (!valid_rule(dcp, interleave) || shard < -1 || shard >= dcp) return DCP_ERR_INVALID_ARG;
  if (!aligned(kv, 16) || !aligned(kv_pool, 16)) return DCP_ERR_INVALID_ARG;
  if (kv_dtype != DCP_KV_BF16 && kv_dtype != DCP_KV_FP8_E4M3_S128) return DCP_ERR_UNSUPPORTED;
  if (page_size != 64) return DCP_ERR_UNSUPPORTED;
  if (n == 0) return DCP_OK;
  return status_of(launch_kv_write(kv, n, seq, pos, dcp, interleave, shard, kv_pool, num_pages,
                                   kv_dtype, block_table, num_seqs, bt_stride,
                                   checked ? err_flag : nullptr,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

int dcp_topk_local(const float* scores, int64_t rows, int32_t score_stride,
                   const int32_t* local_len, int32_t k, int32_t dcp, int32_t interleave,
                   int32_t shard, float* cand_score, int32_t* cand_idx, dcp_stream_t stream) {
  if (!scores || !local_len || !cand_score || !cand_idx) return DCP_ERR_INVALID_ARG;
  if (rows < 0 || score_stride < 1 || k < 1 || k > DCP_MAX_TOPK) return DCP_ERR_INVALID_ARG;
  if (!valid_rule(dcp, interleave) || shard < -1 || shard >= dcp) return DCP_ERR_INVALID_ARG;
  if (!aligned(scores, 4) || !aligned(cand_score, 4) || !aligned(local_len, 4) ||
      !aligned(cand_idx, 4))
    return DCP_ERR_INVALID_ARG;
  const int64_t n_in = shard < 0 ? dcp : 1;
  if (rows * n_in > INT32_MAX) return DCP_ERR_INVALID_ARG;
  // the global slot of the last local slot of a row must be an int32
  const int64_t span = ((int64_t)(score_stride - 1) / interleave + 1) * interleave * dcp;
  if (span - 1 > INT32_MAX) return DCP_ERR_INVALID_ARG;
  TopkParams p{};
  p.score = scores;
  p.len = local_len;
  p.rows = rows;
  p.stride = score_stride;
  p.D = dcp;
  p.I = interleave;
  p.shard = shard;
  p.k = k;
  p.cand_score = cand_score;
  p.cand_idx = cand_idx;
  p.vec = aligned(scores, 16) && score_stride % 4 == 0;
  return status_of(launch_topk_local(p, (int)n_in, reinterpret_cast<cudaStream_t>(stream)));
}

int dcp_topk_merge(const float* cand_score, const int32_t* cand_idx, int32_t dcp, int64_t rows,
                   int32_t k_in, int32_t k, int32_t* topk, int32_t* count, dcp_stream_t stream) {
  if (!cand_score || !cand_idx || !topk) return DCP_ERR_INVALID_ARG;
  if (dcp < 1 || dcp > DCP_MAX_SHARDS || rows < 0 || rows > INT32_MAX) return DCP_ERR_INVALID_ARG;
  if (k_in < 1 || k < 1 || k > DCP_MAX_TOPK || (int64_t)dcp * k_in > INT32_MAX)
    return DCP_ERR_INVALID_ARG;
  if (!aligned(cand_score, 4) || !aligned(cand_idx, 4) || !aligned(topk, 4) ||
      !aligned(count, 4))
    return DCP_ERR_INVALID_ARG;
  TopkParams p{};
  p.score = cand_score;
  p.ids = cand_idx;
  p.rows = rows;
  p.stride = k_in;
  p.D = dcp;
  p.k = k;
  p.topk = topk;
  p.count = count;
  p.vec = aligned(cand_score, 16) && aligned(cand_idx, 16) && k_in % 4 == 0;
  return status_of(launch_topk_merge(p, reinterpret_cast<cudaStream_t>(stream)));
}

int dcp_lse_merge(const float* part_out, const float* part_lse, int32_t dcp, int64_t rows,
                  int32_t heads, int32_t dv, void* out, float* lse, dcp_stream_t stream) {
  if (!part_out || !part_lse || !out || !lse) return DCP_ERR_INVALID_ARG;
  if (dcp < 1 || dcp > DCP_MAX_SHARDS || rows < 0 || heads < 1 || dv < 4 || dv % 4 != 0)
    return DCP_ERR_INVALID_ARG;
  if (!aligned(part_out, 16) || !aligned(out, 8) || !aligned(part_lse, 4) || !aligned(lse, 4))
    return DCP_ERR_INVALID_ARG;
  return status_of(launch_lse_merge(part_out, part_lse, dcp, rows, heads, dv, out, lse,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Workspace of mla_prefill_chunk_dcp: local prefix lengths, remapped chunk slots and their
// counts, the 2*dcp partial outputs and LSEs, and the partial decode calls' own workspace.
struct PrefillWs {
  size_t ll, loc, cnt, po, pl, dws, total;
};

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

// The two partial decode calls of a prefill chunk (the caller fills pointers later).
void prefill_calls(const dcp_mla_decode_args* a, int32_t dcp, int32_t interleave,
                   dcp_mla_decode_args& dense, dcp_mla_decode_args& sparse) {
  dense = *a;
  dense.idx = nullptr;
  dense.count = nullptr;
  // a shard holds at most interleave * ceil(L / (interleave * dcp)) of L slots
  const int64_t id = (int64_t)interleave * dcp;
  dense.max_kv_len = (int32_t)(interleave * ((a->max_kv_len + id - 1) / id));
  dense.num_splits = a->num_splits;
  sparse = *a;
  sparse.kv_len = nullptr;
  sparse.max_kv_len = 0;
}

bool prefill_layout(const dcp_mla_decode_args* a, int32_t dcp, int32_t interleave, PrefillWs& w) {
  const size_t R = (size_t)a->rows, H = (size_t)a->heads, D = (size_t)dcp, K = (size_t)a->k;
  w.ll = 0;
  w.loc = w.ll + a256(D * R * 4);
  w.cnt = w.loc + a256(D * R * K * 4);
  w.po = w.cnt + a256(D * R * 4);
  w.pl = w.po + a256(2 * D * R * H * kDv * 4);
  w.dws = w.pl + a256(2 * D * R * H * 4);
  dcp_mla_decode_args dense, sparse;
  prefill_calls(a, dcp, interleave, dense, sparse);
  // the partial calls' workspace sizes depend on shapes only: stand-in pointers suffice
  int32_t* fake = reinterpret_cast<int32_t*>((uintptr_t)256);
  dense.kv_len = fake;
  sparse.idx = fake;
  sparse.count = fake;
  const size_t n1 = mla_decode_workspace_size(&dense, dcp, 0);
  const size_t n2 = mla_decode_workspace_size(&sparse, dcp, 0);
  if (n1 == (size_t)-1 || n2 == (size_t)-1) return false;
  w.total = w.dws + a256(n1 > n2 ? n1 : n2);
  return true;
}

int prefill_check(const dcp_mla_decode_args* a, int32_t dcp, int32_t interleave) {
  if (a == nullptr) return DCP_ERR_INVALID_ARG;
  if (!valid_rule(dcp, interleave)) return DCP_ERR_INVALID_ARG;
  if (2 * dcp > DCP_MAX_SHARDS) return DCP_ERR_UNSUPPORTED;  // the merge takes 2*dcp partials
  if (a->idx == nullptr || a->kv_len == nullptr || a->max_kv_len < 0) return DCP_ERR_INVALID_ARG;
  if (a->k < 1 || a->k > DCP_MAX_TOPK || a->rows < 0) return DCP_ERR_INVALID_ARG;
  return DCP_OK;
}

}  // namespace

extern "C" {

size_t mla_prefill_chunk_workspace_size(const dcp_mla_decode_args* args, int32_t dcp,
                                        int32_t interleave) {
  if (prefill_check(args, dcp, interleave) != DCP_OK) return (size_t)-1;
  PrefillWs w;
  if (!prefill_layout(args, dcp, interleave, w)) return (size_t)-1;
  return w.total;
}

int mla_prefill_chunk_dcp(const dcp_mla_decode_args* args, int32_t dcp, int32_t interleave,
                          dcp_stream_t stream) {
  int rc = prefill_check(args, dcp, interleave);
  if (rc != DCP_OK) return rc;
  PrefillWs w;
  if (!prefill_layout(args, dcp, interleave, w)) return DCP_ERR_INVALID_ARG;
  if (args->workspace == nullptr || args->workspace_bytes < w.total || !aligned(args->workspace, 256))
    return DCP_ERR_WORKSPACE;
  if (!args->out || !args->lse || !aligned(args->out, 8) || !aligned(args->lse, 4))
    return DCP_ERR_INVALID_ARG;
  if (args->rows == 0) return DCP_OK;
  uint8_t* ws = static_cast<uint8_t*>(args->workspace);
  int32_t* ll = reinterpret_cast<int32_t*>(ws + w.ll);
  int32_t* loc = reinterpret_cast<int32_t*>(ws + w.loc);
  int32_t* cnt = reinterpret_cast<int32_t*>(ws + w.cnt);
  float* po = reinterpret_cast<float*>(ws + w.po);
  float* pl = reinterpret_cast<float*>(ws + w.pl);
  const size_t dws_bytes = w.total - w.dws;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t R = args->rows, H = args->heads;
  dcp_mla_decode_args dense, sparse;
  prefill_calls(args, dcp, interleave, dense, sparse);
  // 1-2. the cached prefix: each shard's local length, one dense partial per shard
  if ((rc = status_of(launch_local_lengths(args->kv_len, R, dcp, interleave, -1, ll, st))) != DCP_OK)
    return rc;
  dense.kv_len = ll;
  dense.out = po;
  dense.lse = pl;
  dense.workspace = ws + w.dws;
  dense.workspace_bytes = dws_bytes;
  if ((rc = mla_decode_partial_lse(&dense, dcp, stream)) != DCP_OK) return rc;
  // 3-4. the chunk: each shard's slots of it, one sparse partial per shard
  if ((rc = status_of(launch_remap_topk(args->idx, R, args->k, dcp, interleave, -1, loc, cnt, st))) !=
      DCP_OK)
    return rc;
  sparse.idx = loc;
  sparse.count = cnt;
  sparse.out = po + (int64_t)dcp * R * H * kDv;
  sparse.lse = pl + (int64_t)dcp * R * H;
  sparse.workspace = ws + w.dws;
  sparse.workspace_bytes = dws_bytes;
  if ((rc = mla_decode_partial_lse(&sparse, dcp, stream)) != DCP_OK) return rc;
  // 5. the LSE merge of the 2*dcp partials
  return status_of(launch_lse_merge(po, pl, 2 * dcp, R, (int)H, kDv, args->out, args->lse, st));
}

size_t mla_decode_workspace_size(const dcp_mla_decode_args* args, int32_t num_shards_or_dcp,
                                 int32_t fused) {
  DecodeParams p;
  bool sparse;
  const int32_t d = num_shards_or_dcp;
  if (prepare_decode(args, fused ? 1 : d, fused != 0, d, 1, p, sparse) != DCP_OK)
    return (size_t)-1;
  if (p.use_tc) return tc_workspace_bytes(p.num_units, p.pairs);
  return simt_workspace_bytes(p.num_units, p.heads, p.num_splits);
}

int mla_decode_partial_lse(const dcp_mla_decode_args* args, int32_t num_shards,
                           dcp_stream_t stream) {
  DecodeParams p;
  bool sparse;
  int rc = prepare_decode(args, num_shards, false, 1, 1, p, sparse);
  if (rc != DCP_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = bind_workspace(args, p, st)) != DCP_OK) return rc;
  if (p.num_units == 0) return DCP_OK;
  return status_of(p.use_tc ? launch_decode_tc(p, args->kv_dtype, false, sparse, st)
                            : launch_decode_simt(p, args->kv_dtype, false, sparse, st));
}

int mla_decode_dcp_fused(const dcp_mla_decode_args* args, int32_t dcp, int32_t interleave,
                         dcp_stream_t stream) {
  DecodeParams p;
  bool sparse;
  int rc = prepare_decode(args, 1, true, dcp, interleave, p, sparse);
  if (rc != DCP_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = bind_workspace(args, p, st)) != DCP_OK) return rc;
  if (p.num_units == 0) return DCP_OK;
  return status_of(p.use_tc ? launch_decode_tc(p, args->kv_dtype, true, sparse, st)
                            : launch_decode_simt(p, args->kv_dtype, true, sparse, st));
}

}  // extern "C"

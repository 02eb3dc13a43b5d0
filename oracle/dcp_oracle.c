/*
 * dcp_oracle.c -- TEST INFRASTRUCTURE ONLY (the oracle).
 *
 * A plain, slow, double-precision CPU statement of what the decode-context-parallel
 * (DCP) MLA decode path computes.  Only the test-suite, the smoke check and the
 * bench's CPU-baseline leg call it; the product library never links, loads or runs it,
 * and it shares no code, header or table with the CUDA path.
 *
 * What it follows (sources are three public pages on DCP for MLA / DSA decode):
 *   - LMDeploy PR #4952 "support decode context parallelism for PyTorch MLA", Summary:
 *     KV tokens are sharded across ranks; decode attends to the local KV and the shard
 *     outputs are merged with LSE weights.
 *   - SGLang PR #42536 "Fix DCP for RoPE sparse attention on Blackwell", Modifications
 *     (Index remap; Backend; Fixes in shared code): global top-k slots are filtered to
 *     the ones a rank owns, turned into local slot ids, moved to the front of the row with
 *     a per-row count; attention returns (output, LSE); rows without local KV are fixed
 *     up; the LSE combine returns zero when every shard is empty.
 *   - SGLang PR #36990 "DCP for DSA models with the flashmla_kv backend", review of the
 *     LSE combine: with every shard at LSE = -inf the weights are all zero; return a zero
 *     output and a -inf global LSE instead of 0/0.
 * Readings where the pages are silent (all stated again in the design notes):
 *   owner(t) = (t div I) mod D, local(t) = (t div (I*D))*I + (t mod I), with I = 1 for the
 *   token-interleaved rule ("slot mod D") and I = page size for the page-interleaved rule
 *   ("page mod D"); LSE is a natural log of sum(exp(sm_scale * q.k)); the value row is
 *   the first 512 dims of the 576-dim latent key row; FP8 latent values are
 *   e4m3(code) * scale[block of 128]; the RoPE tail of an FP8 row is BF16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_DQK 576
#define ORC_DV 512
#define ORC_KV_BF16 0
#define ORC_KV_FP8 1

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* E4M3 (OCP 8-bit float, "fn" variant): 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN;
 * there is no infinity. */
double orc_e4m3_decode(int code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

static double bf16_to_double(const uint8_t* p) {
  uint16_t h;
  memcpy(&h, p, 2);
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Owner shard of global slot t and its local slot id on that shard. */
int orc_owner(int64_t t, int dcp, int interleave) {
  return (int)((t / interleave) % dcp);
}
int64_t orc_local(int64_t t, int dcp, int interleave) {
  return (t / ((int64_t)interleave * dcp)) * interleave + (t % interleave);
}

/* Brute-force count of the slots 0..len-1 that shard s owns. */
int64_t orc_count_owned(int64_t len, int dcp, int interleave, int s) {
  int64_t n = 0;
  for (int64_t t = 0; t < len; ++t) n += (orc_owner(t, dcp, interleave) == s);
  return n;
}

/* Remap (SGLang PR #42536, Modifications, "Index remap"): for each row and each shard,
 * keep the owned slots (t >= 0) in their original order, write their local ids to the
 * front of the shard's row, fill the rest with -1 and return the count.
 * local_idx is [n_out][rows][k], count is [n_out][rows]; n_out = dcp when shard < 0,
 * else 1 (only that shard). */
int orc_remap(const int32_t* gidx, int64_t rows, int32_t k, int32_t dcp, int32_t interleave,
              int32_t shard, int32_t* local_idx, int32_t* count) {
  if (!gidx || !local_idx || !count || rows < 0 || k < 0 || dcp < 1 || interleave < 1) return -1;
  int s0 = shard < 0 ? 0 : shard, s1 = shard < 0 ? dcp : shard + 1;
  for (int s = s0; s < s1; ++s) {
    int o = s - s0;
    for (int64_t r = 0; r < rows; ++r) {
      int32_t* dst = local_idx + ((int64_t)o * rows + r) * k;
      int32_t n = 0;
      for (int32_t j = 0; j < k; ++j) {
        int32_t t = gidx[r * k + j];
        if (t < 0) continue;
        if (orc_owner(t, dcp, interleave) == s) dst[n++] = (int32_t)orc_local(t, dcp, interleave);
      }
      for (int32_t j = n; j < k; ++j) dst[j] = -1;
      count[(int64_t)o * rows + r] = n;
    }
  }
  return 0;
}

typedef struct {
  const uint8_t* q;            /* [rows][heads][576] bf16 */
  int64_t rows;
  int32_t heads;
  double sm_scale;
  const uint8_t* pool;         /* [num_pages][page_size][token_bytes] */
  int64_t num_pages;
  int32_t kv_dtype;            /* 0 = BF16 rows of 1152 B, 1 = FP8 rows of 656 B */
  int32_t page_size;
  const int32_t* block_table;  /* [dcp][num_seqs][bt_stride] physical page ids */
  int32_t num_seqs;
  int32_t bt_stride;
  const int32_t* row_seq;      /* [rows] sequence of each decode row */
  const int32_t* row_len;      /* [rows] visible global length (dense) */
  const int32_t* topk;         /* [rows][k] global slots, -1 = pad; NULL = dense */
  int32_t k;
  int32_t dcp;
  int32_t interleave;
  int32_t shard;               /* < 0: all owned slots (unsharded); s: shard s only */
  double* out;                 /* [rows][heads][512] */
  double* lse;                 /* [rows][heads] */
} orc_attn_args;

/* Decode one latent key row (576 values) of global slot t of sequence b.
 * Returns 0, or -2 when the block table or pool would be indexed out of range. */
static int fetch_row(const orc_attn_args* a, int b, int64_t t, double* kv) {
  int s = orc_owner(t, a->dcp, a->interleave);
  int64_t l = orc_local(t, a->dcp, a->interleave);
  int64_t pj = l / a->page_size;
  if (pj >= a->bt_stride) return -2;
  int32_t page = a->block_table[((int64_t)s * a->num_seqs + b) * a->bt_stride + pj];
  if (page < 0 || page >= a->num_pages) return -2;
  int64_t tb = a->kv_dtype == ORC_KV_BF16 ? 1152 : 656;
  const uint8_t* row = a->pool + ((int64_t)page * a->page_size + l % a->page_size) * tb;
  if (a->kv_dtype == ORC_KV_BF16) {
    for (int d = 0; d < ORC_DQK; ++d) kv[d] = bf16_to_double(row + 2 * d);
  } else {
    for (int blk = 0; blk < 4; ++blk) {
      float sc;
      memcpy(&sc, row + 512 + 4 * blk, 4);
      for (int i = 0; i < 128; ++i)
        kv[blk * 128 + i] = orc_e4m3_decode(row[blk * 128 + i]) * (double)sc;
    }
    for (int i = 0; i < 64; ++i) kv[512 + i] = bf16_to_double(row + 528 + 2 * i);
  }
  return 0;
}

/* Attention with LSE over the valid slots of each row (sparse: the row's top-k slots;
 * dense: 0..row_len-1), restricted to one shard's slots when shard >= 0:
 *   s_t = sm_scale * q.k_t (576 dims), lse = ln sum_t exp(s_t),
 *   o = sum_t exp(s_t - lse) * k_t[0:512];  an empty set gives o = 0, lse = -inf.
 * (LMDeploy PR #4952, Summary; SGLang PR #42536, Modifications, "Backend".) */
int orc_attention(const orc_attn_args* a) {
  if (!a || !a->q || !a->pool || !a->block_table || !a->row_seq || !a->out || !a->lse) return -1;
  if (!a->topk && !a->row_len) return -1;
  int err = 0;
  int H = a->heads;
  for (int64_t r = 0; r < a->rows; ++r) {
    int b = a->row_seq[r];
    if (b < 0 || b >= a->num_seqs) return -2;
    /* the row's slot set, in its given order */
    int64_t cap = a->topk ? a->k : (a->row_len[r] > 0 ? a->row_len[r] : 0);
    int64_t* slots = (int64_t*)malloc(sizeof(int64_t) * (cap > 0 ? cap : 1));
    int64_t n = 0;
    for (int64_t j = 0; j < cap; ++j) {
      int64_t t = a->topk ? a->topk[r * a->k + j] : j;
      if (t < 0) continue;
      if (a->shard >= 0 && orc_owner(t, a->dcp, a->interleave) != a->shard) continue;
      slots[n++] = t;
    }
    double* K = (double*)malloc(sizeof(double) * ORC_DQK * (n > 0 ? n : 1));
#pragma omp parallel for schedule(static) reduction(| : err)
    for (int64_t i = 0; i < n; ++i) err |= -fetch_row(a, b, slots[i], K + i * ORC_DQK);
    if (err) {
      free(K);
      free(slots);
      return -2;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < H; ++h) {
      const uint8_t* qh = a->q + ((r * H + h) * (int64_t)ORC_DQK) * 2;
      double q[ORC_DQK];
      for (int d = 0; d < ORC_DQK; ++d) q[d] = bf16_to_double(qh + 2 * d);
      double* o = a->out + (r * H + h) * (int64_t)ORC_DV;
      for (int d = 0; d < ORC_DV; ++d) o[d] = 0.0;
      if (n == 0) {
        a->lse[r * H + h] = -INFINITY;
        continue;
      }
      double* sc = (double*)malloc(sizeof(double) * n);
      double m = -INFINITY;
      for (int64_t i = 0; i < n; ++i) {
        const double* kt = K + i * ORC_DQK;
        double dot = 0.0;
        for (int d = 0; d < ORC_DQK; ++d) dot += q[d] * kt[d];
        sc[i] = a->sm_scale * dot;
        if (sc[i] > m) m = sc[i];
      }
      double sum = 0.0;
      for (int64_t i = 0; i < n; ++i) sum += exp(sc[i] - m);
      double lse = m + log(sum);
      for (int64_t i = 0; i < n; ++i) {
        double w = exp(sc[i] - lse);
        const double* kt = K + i * ORC_DQK;
        for (int d = 0; d < ORC_DV; ++d) o[d] += w * kt[d];
      }
      a->lse[r * H + h] = lse;
      free(sc);
    }
    free(K);
    free(slots);
  }
  return 0;
}

/* LSE merge of shard partials (LMDeploy PR #4952, Summary: "merge outputs using LSE
 * weights"; the all-empty case from SGLang PR #36990's review of the LSE combine and
 * SGLang PR #42536, Fixes in shared code):
 *   m = max_s lse_s; if m = -inf: out = 0, lse = -inf;
 *   else w_s = exp(lse_s - m), W = sum w_s, out = sum w_s o_s / W, lse = m + ln W.
 * part_out [dcp][rows][heads][dv], part_lse [dcp][rows][heads]. */
int orc_merge(const double* part_out, const double* part_lse, int32_t dcp, int64_t rows,
              int32_t heads, int32_t dv, double* out, double* lse) {
  if (!part_out || !part_lse || !out || !lse || dcp < 1 || rows < 0 || heads < 1 || dv < 1)
    return -1;
  int64_t RH = rows * heads;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < RH; ++i) {
    double m = -INFINITY;
    for (int s = 0; s < dcp; ++s)
      if (part_lse[s * RH + i] > m) m = part_lse[s * RH + i];
    double* o = out + i * dv;
    for (int d = 0; d < dv; ++d) o[d] = 0.0;
    if (m == -INFINITY) {
      lse[i] = -INFINITY;
      continue;
    }
    double W = 0.0;
    for (int s = 0; s < dcp; ++s) W += exp(part_lse[s * RH + i] - m);
    for (int s = 0; s < dcp; ++s) {
      double w = exp(part_lse[s * RH + i] - m) / W;
      const double* os = part_out + (s * RH + i) * dv;
      if (w == 0.0) continue;
      for (int d = 0; d < dv; ++d) o[d] += w * os[d];
    }
    lse[i] = m + log(W);
  }
  return 0;
}

/* ---- KV-cache write (interleaved DCP) -----------------------------------------------
 * A new token's latent row (576 bf16: 512 latent, 64 RoPE) at global position t of
 * sequence b is stored on shard s = owner(t) at that shard's local slot l = local(t):
 * page block_table[s][b][l / page_size], row l mod page_size (LMDeploy PR #4952, files:
 * "Interleaved DCP KV-cache writes").  FP8 pools quantise the latent part and keep the RoPE
 * part in bf16 (SGLang PR #36990, review of quantize_k_cache_separate: the "nope" and "pe"
 * parts are quantised separately).  Per block of 128 latent values: scale = amax / 448 in
 * fp32 (0 for an all-zero block, whose codes are 0), code = the E4M3 value nearest to
 * value / scale computed in fp32, ties to the even code, saturating at 448.  The code
 * decision is taken in fp32, the precision the writer computes in. */

/* Nearest E4M3 code of y (round to nearest, ties to even, saturate to +-448), by search
 * over the 127 non-negative finite codes. */
int orc_e4m3_encode(float y) {
  if (y != y) return 0x7F;
  const int sign = signbit(y) ? 1 : 0;
  double a = fabs((double)y);
  if (a > 448.0) a = 448.0;
  int best = 0;
  double bestd = INFINITY;
  for (int c = 0; c < 127; ++c) {
    const double d = fabs(orc_e4m3_decode(c) - a);
    if (d < bestd || (d == bestd && (c & 1) == 0)) {
      best = c;
      bestd = d;
    }
  }
  return best | (sign << 7);
}

static float bf16_bits_to_float(const uint8_t* p) {
  uint16_t h;
  memcpy(&h, p, 2);
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Writes n token rows kv[n][576] (bf16 bytes) of sequences seq[i] at global positions
 * pos[i] into the pool; shard >= 0 writes only the rows that shard owns.  Rows whose
 * position or sequence is negative / out of range, or whose block-table entry is missing or
 * out of range, are skipped and counted in *skipped.  Returns the number of rows written. */
int64_t orc_kv_write(const uint8_t* kv, int64_t n, const int32_t* seq, const int32_t* pos,
                     int32_t dcp, int32_t interleave, int32_t shard, uint8_t* pool,
                     int64_t num_pages, int32_t kv_dtype, int32_t page_size,
                     const int32_t* block_table, int32_t num_seqs, int32_t bt_stride,
                     int64_t* skipped) {
  const int tb = kv_dtype == ORC_KV_BF16 ? 1152 : 656;
  int64_t written = 0, skip = 0;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t t = pos[i];
    const int b = seq[i];
    if (t < 0 || b < 0 || b >= num_seqs) {
      ++skip;
      continue;
    }
    const int s = orc_owner(t, dcp, interleave);
    if (shard >= 0 && s != shard) continue;
    const int64_t l = orc_local(t, dcp, interleave);
    const int64_t pj = l / page_size;
    if (pj >= bt_stride) {
      ++skip;
      continue;
    }
    const int32_t page = block_table[((int64_t)s * num_seqs + b) * bt_stride + pj];
    if (page < 0 || page >= num_pages) {
      ++skip;
      continue;
    }
    uint8_t* dst = pool + ((int64_t)page * page_size + l % page_size) * tb;
    const uint8_t* src = kv + i * (int64_t)(ORC_DQK * 2);
    if (kv_dtype == ORC_KV_BF16) {
      memcpy(dst, src, 1152);
    } else {
      for (int blk = 0; blk < 4; ++blk) {
        float amax = 0.0f;
        for (int j = 0; j < 128; ++j) {
          const float v = fabsf(bf16_bits_to_float(src + 2 * (blk * 128 + j)));
          if (v > amax) amax = v;
        }
        const float scale = amax / 448.0f;
        for (int j = 0; j < 128; ++j) {
          const float v = bf16_bits_to_float(src + 2 * (blk * 128 + j));
          dst[blk * 128 + j] = (uint8_t)(scale > 0.0f ? orc_e4m3_encode(v / scale) : 0);
        }
        memcpy(dst + 512 + 4 * blk, &scale, 4);
      }
      memcpy(dst + 528, src + 1024, 128);
    }
    ++written;
  }
  if (skipped) *skipped = skip;
  return written;
}

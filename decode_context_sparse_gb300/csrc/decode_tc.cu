// Tensor-core (tcgen05 / TMEM) MLA decode attention with LSE for 48..128 heads, BF16 or
// FP8-E4M3 (per-128 scale) latent KV: the per-shard partial form and the fused
// all-shards form.  What it computes is the same as the CUDA-core path
// (LMDeploy PR #4952 "support decode context parallelism for PyTorch MLA", Summary;
// SGLang PR #42536 "Fix DCP for RoPE sparse attention on Blackwell", Modifications,
// "Backend"; Follow-ups #1).
//
// Why two CTAs per row.  With 128 heads the output accumulator O[128 heads x 512] fp32
// alone fills the 512 TMEM columns of an SM.  A cluster of two CTAs therefore shares
// each row: CTA c owns latent dims [256c, 256c+256) and RoPE dims [512+32c, 512+32c+32)
// of every key, computes the partial logits q.k over its 288 dims and the output columns
// of its 256 value dims.  The two partial logit tiles are exchanged through distributed
// shared memory (one bulk copy per warp, completing on the peer's mbarrier) and both CTAs
// run the same softmax.
//
// Per CTA (640 threads), tiles of 32 key slots:
//   warps 1-3   loaders (tiles round-robin; as many as staging slots, at most three; the
//               others idle):
//               slot id -> owner shard / local slot -> page
//               (a three-stage software pipeline over the dependent loads), then 4-row TMA
//               gathers of this CTA's latent half and of the row tail into a staging ring;
//   warp 0      TMEM owner and MMA issuer: S = Q K^T (latent part of Q in TMEM, RoPE part
//               of Q in shared memory) and O += P V (P in shared memory), each issued as
//               soon as its inputs are ready;
//   warps 4-7   converters: staging -> SWIZZLE_128B FP16 K tile (FP8: E4M3 code times the
//               power-of-two part of its block scale, exact), zero rows for padding,
//               per-slot scale factors;
//   warps 12-15 softmax stage A: thread h owns head h (TMEM lane h): reads its logits of
//               a tile, scales them, hands this CTA's partial to stage B through a local
//               box in shared memory and copies the box to the peer CTA's inbox; loads Q;
//   warps 8-11, 16-19  softmax stage B, two warps per group of 32 heads, each on half of
//               a tile's columns: adds the two partials, online softmax in base 2 with a
//               lazily raised reference max (the output is rescaled only when the max
//               grows by more than 2^8), writes P as FP16 into shared memory, and at the
//               end of a row normalises O and writes it out (or a partial of a split row).
// TMEM columns: O [0,256) | Q latent [256,384) | two logit buffers from 384.  P lives in
// shared memory, so a logit buffer is free again as soon as stage A has read it.
//
// Numerics.  The MMAs take FP16 operands and accumulate in fp32.  Q is multiplied per head by
// the power of two that puts its largest magnitude in [2^14, 2^15) and the head's logits by
// the inverse (both exact); BF16 keys are converted to FP16 (exact below 65504).  FP8: each
// CTA's 256 latent dims are two 128-blocks with scales s = m 2^E (E = floor(log2 s), at most
// 7; m in [1, 2)).  The K tile holds code * 2^E, exact in FP16, so the logit needs two
// accumulators, acc_lo and acc_hi, and is m_lo acc_lo + m_hi acc_hi in fp32.  The RoPE part
// rides in acc_lo: its keys are stored as k_rope / m_lo split into an FP16 high part and an
// FP16 remainder.  For P V the multipliers are folded into P: O[:, lo] += (P m_lo) V_lo,
// O[:, hi] += (P m_hi) V_hi, each P m rounded once to FP16 (relative error 2^-11).  A block
// whose scale is 0 or below 2^-24 counts as zero.
//
// Work: a persistent grid of pairs; the concatenated sequence of 32-slot tiles of all
// units (rows, or (shard, row) pairs) is cut into equal contiguous ranges, one per pair.
// A unit cut by a range edge leaves fp32 partials and a descriptor in the workspace;
// tc_split_merge_kernel, launched after this kernel on the same stream, merges them.  Every
// wait is bounded; a wait that expires sets an abort flag, the CTA winds down and
// DCP_ERRBIT_TIMEOUT is reported.
#include <cuda.h>
#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace dcp {
using namespace tc;

constexpr int kTN = 32;  // key slots per tile

template <int KVT>
struct TcCfg;
// Staged bytes per slot: this CTA's latent half, and the row tail (FP8: the four block
// scales and all 64 RoPE dims, 144 B; BF16: this CTA's 32 RoPE dims, 64 B).  A 4-row tail
// gather lands on a 128-B aligned stride.
template <>
struct TcCfg<DCP_KV_FP8_E4M3_S128> {
  static constexpr int NACC = 2, NS = 2, NK = 4, NP = 2, NSB = 1;
  static constexpr int LAT_TOK = 256, TAIL_TOK = 144, TAIL_GSTRIDE = 640;
};
template <>
struct TcCfg<DCP_KV_BF16> {
  static constexpr int NACC = 1, NS = 2, NK = 4, NP = 2, NSB = 1;
  static constexpr int LAT_TOK = 512, TAIL_TOK = 64, TAIL_GSTRIDE = 256;
};

constexpr int kTcThreads = 640;
constexpr int kMinTilesPerPair = 16;
constexpr int kColO = 0, kColQ = 256, kColS = 384;
constexpr uint32_t kTmemCols = 512;

template <int KVT>
struct TcLay {
  using C = TcCfg<KVT>;
  static constexpr int TN = kTN;
  static constexpr int BS = TN * 128;        // bytes between 64-dim column blocks of a K tile
  static constexpr int KT_BYTES = 5 * BS;    // 4 latent blocks + 1 RoPE block
  static constexpr int STG_TAIL = TN * C::LAT_TOK;
  static constexpr int STG_BYTES = STG_TAIL + (TN / 4) * C::TAIL_GSTRIDE;
  static constexpr int GROUP_TX = 4 * (C::LAT_TOK + C::TAIL_TOK);  // bytes of one 4-row group
  static constexpr int QR_BYTES = 128 * 128;  // RoPE part of Q: 128 rows of one SW128 row
  // exchange rows: TN floats padded to TN + 4 (rows 16-B aligned; a warp's 16-B accesses to
  // one column of 32 rows spread over all banks).  Measured faster than an XOR-swizzled
  // unpadded layout (when the partials still went over as per-thread remote stores).
  static constexpr int XSTRIDE = TN + 4;
  static constexpr int X_BYTES = 128 * XSTRIDE * 4;
  // per K tile: logit scale lo | logit scale hi (fp32, x sl2) | P scales s_lo, s_hi as bf16
  // (the slot mask is kept in TcShared::kt_mask)
  static constexpr int META_BYTES = 4 * TN * 4;
  static constexpr int SBUF = C::NACC * TN;
  static constexpr int OFF_KT = 0;
  static constexpr int OFF_STG = OFF_KT + C::NK * KT_BYTES;
  static constexpr int OFF_QR = OFF_STG + C::NS * STG_BYTES;
  static constexpr int P_BYTES = 128 * 128;   // P of a tile: 128 rows of one SW128 row
  static constexpr int OFF_P = OFF_QR + QR_BYTES;
  static constexpr int OFF_X = OFF_P + C::NP * P_BYTES;
  static constexpr int OFF_SELF = OFF_X + 2 * X_BYTES;
  static constexpr int SELF_BYTES = C::NSB * X_BYTES;  // local boxes: same padded rows
  static constexpr int OFF_META = OFF_SELF + SELF_BYTES;
  static constexpr int OFF_END = OFF_META + C::NK * META_BYTES;
  // at least 120 KB so that one CTA (and one TMEM owner) sits on an SM
  static constexpr int SMEM = (OFF_END + 1024 > 122880 ? OFF_END + 1024 : 122880);
  static_assert(OFF_STG % 1024 == 0 && STG_BYTES % 1024 == 0 && OFF_QR % 1024 == 0,
                "SW128 tiles and TMA destinations need 1024-B / 128-B alignment");
  static_assert(kColS + 2 * SBUF <= (int)kTmemCols, "TMEM columns");
};

struct TcShared {
  uint64_t stg_full[4], stg_empty[4], kt_full[8], kt_empty[8];
  uint64_t s_full[2], p_full[2], pv_done[2], q_ready, in_full[2], out_free[2], drain;
  uint64_t self_full[2], self_free[2];  // stage A -> stage B hand-over of this CTA's partial
  uint64_t s_free[2];                   // stage A has read a logit buffer out of TMEM
  uint64_t bx_full[4][2], bl_full[4];   // stage B pairs: partial row maxima / row sums posted
  uint64_t ep_done[4];                  // stage B pairs: a tiled-store epilogue's staging free
  float bx[2][2][128];                  // [half][tile parity][head] partial row max of a tile
  float bl[2][128];                     // [half][head] partial row sum of a unit
  uint32_t stg_mask[4];
  uint32_t kt_mask[8];        // valid-slot mask of each K tile
  uint32_t stg_issued[4];     // gathers issued per staging slot (for the teardown wait)
  uint32_t tmem_base;
  int abort_flag;
  int64_t T, t0;
  int Peff;  // pairs that own tiles: min(pairs, T), so no pair's range is empty
  int64_t unit0;  // order index of the pair's first unit
  int tile0, ntiles;
  int64_t scan_base;
};
// dynamic + static shared memory within the 227 KB a CTA may opt into
static_assert(TcLay<DCP_KV_FP8_E4M3_S128>::SMEM + sizeof(TcShared) <= 232448, "shared memory");
static_assert(TcLay<DCP_KV_BF16>::SMEM + sizeof(TcShared) <= 232448, "shared memory");

// A unit: a row (fused) or a (shard, row) pair (partial), whose id u indexes the caller's
// [shards][rows] arrays.  The kernel visits the partial form's units row by row, the shards
// of one row one after another (order index v = row * shards + shard), so that consecutive
// units share the row's queries and the Q load is skipped between them.
struct UnitInfo {
  int64_t u, r;
  int shard, b, n, ntile;
};

template <bool FUSED>
__device__ __forceinline__ int64_t unit_row(const DecodeParams& p, int64_t v) {
  return FUSED ? v : fdiv((int)v, p.shards_div);
}

template <bool FUSED, bool SPARSE>
__device__ __forceinline__ UnitInfo get_unit(const DecodeParams& p, int64_t v) {
  UnitInfo x;
  x.r = unit_row<FUSED>(p, v);
  x.shard = FUSED ? 0 : (int)(v - x.r * p.shards);
  x.u = FUSED ? v : (int64_t)x.shard * p.rows + x.r;
  x.b = __ldg(p.row_seq + x.r);
  if (SPARSE)
    x.n = FUSED ? p.k : min(max(__ldg(p.count + x.u), 0), p.k);
  else
    x.n = max(0, __ldg(p.kv_len + x.u));
  if (x.b < 0 || x.b >= p.num_seqs) x.n = 0;
  x.ntile = (x.n + kTN - 1) / kTN;
  return x;
}

// Walk over this pair's tiles, unit by unit in visiting order (empty units contribute no
// tiles); v is the order index, info.u the unit's id.
template <bool FUSED, bool SPARSE>
struct Walk {
  int64_t v;
  int lt, left;
  UnitInfo info;
  __device__ void init(const DecodeParams& p, int64_t v0, int tile0, int ntiles) {
    v = v0;
    lt = tile0;
    left = ntiles;
    if (left > 0) info = get_unit<FUSED, SPARSE>(p, v);
  }
  __device__ bool first() const { return lt == 0; }
  __device__ bool last() const { return lt == info.ntile - 1; }
  __device__ void next(const DecodeParams& p) {
    if (--left <= 0) return;
    if (++lt == info.ntile) {
      do {
        ++v;
        info = get_unit<FUSED, SPARSE>(p, v);
      } while (info.ntile == 0);
      lt = 0;
    }
  }
};

// Block-wide exclusive prefix of v (384 threads); returns the prefix, *total the sum.
// (warp_sum: 16 int64 of shared memory, free during set-up)
__device__ __forceinline__ int64_t block_scan_excl(int64_t v, int64_t* warp_sum, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sum[warp] = x;
  __syncthreads();
  int64_t base = 0, tot = 0;
  for (int w = 0; w < kTcThreads / 32; ++w) {
    if (w < warp) base += warp_sum[w];
    tot += warp_sum[w];
  }
  __syncthreads();
  *total = tot;
  return base + x - v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&t);
}

// FP8 block scale s = m * 2^E with E = floor(log2 s) clamped to at most 7 (so that codes *
// 2^E, |code| <= 448, stay finite in FP16) and m = s / 2^E, in [1, 2) unless E was clamped.
// A block whose scale is 0, or below 2^-24 (its values below 448 * 2^-24 in magnitude),
// counts as zero: multiplier 0, m 0.
__device__ __forceinline__ int fp8_block_exp(float s) {
  const int e = (int)((__float_as_uint(s) >> 23) & 0xFF) - 127;
  return e > 7 ? 7 : e;
}
__device__ __forceinline__ float fp8_block_m(float s) {
  const int e = fp8_block_exp(s);
  if (!(s > 0.f) || e < -24) return 0.f;
  return s * __uint_as_float((uint32_t)(127 - e) << 23);  // s * 2^-e, exact
}
// f16x2 holding 2^E twice (the codes' multiplier), or 0.
__device__ __forceinline__ uint32_t fp8_block_mul(float s) {
  const int e = fp8_block_exp(s);
  if (!(s > 0.f) || e < -24) return 0u;
  // 2^e as FP16: normal for e >= -14 (biased exponent e + 15), subnormal below
  const uint32_t h = e >= -14 ? (uint32_t)(e + 15) << 10 : (uint32_t)1 << (e + 24);
  return h | (h << 16);
}

// Q of one (row, head) for a CTA of a pair, as FP16: the CTA's 256 latent dims into TMEM
// (two per column, at taddr), its 32 RoPE dims into row h of the SW128 A-operand tile qr.
// The values are multiplied by 2^(14 - e), e the exponent of their largest magnitude (exact;
// keeps them in FP16's range); returns 2^(e - 14), the factor that undoes it on the logits.
// qs_prev is that factor of this head's previous row (0: none), whose e serves as a hint.
// Without a hint: two passes over the 36 16-B pieces (the largest magnitude, then the
// conversion).  With one (for the whole warp), one pass converts with it and finds the
// largest magnitude on the way; any e from the true one - 8 to the true one + 1 gives the
// same FP16 values up to the rounding of values 2^-20 below the largest, and none
// overflows, so only a hint outside that range makes the warp convert again with the true
// exponent.  Twelve or eight loads in flight.  Not inlined: it runs once per row, and the
// warps that call it keep their registers for the per-tile work.
constexpr int kNoQHint = -1000;

__device__ __forceinline__ uint32_t q_piece_mx(const uint4& v, uint32_t mx) {
  const uint32_t w[4] = {v.x & 0x7fff7fffu, v.y & 0x7fff7fffu, v.z & 0x7fff7fffu,
                         v.w & 0x7fff7fffu};
#pragma unroll
  for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0xffffu, w[k] >> 16));
  return mx;
}

// The conversion pass with exponent e; returns the largest |bf16| bit pattern it loaded.
__device__ __forceinline__ uint32_t tc_q_convert(const uint4* __restrict__ src, bool valid,
                                                 int crank, uint32_t taddr, unsigned char* qr,
                                                 int hrow, int e) {
  const bool noscale = e > 127 - 14;
  const float up = noscale ? 1.0f : __uint_as_float((uint32_t)(127 + 14 - e) << 23);
  uint32_t mx = 0;
#pragma unroll 1
  for (int c = 0; c < 8; c += 2) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      v[i] = valid ? __ldg(src + crank * 32 + c * 4 + i) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 u = v[4 * cc + i];
        mx = q_piece_mx(u, mx);
        w[4 * i] = bf16x2_to_f16x2_mul(u.x, up);
        w[4 * i + 1] = bf16x2_to_f16x2_mul(u.y, up);
        w[4 * i + 2] = bf16x2_to_f16x2_mul(u.z, up);
        w[4 * i + 3] = bf16x2_to_f16x2_mul(u.w, up);
      }
      tmem_st16(taddr + 16 * (c + cc), w);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 v = valid ? __ldg(src + 64 + crank * 4 + i) : make_uint4(0u, 0u, 0u, 0u);
    mx = q_piece_mx(v, mx);
    v = make_uint4(bf16x2_to_f16x2_mul(v.x, up), bf16x2_to_f16x2_mul(v.y, up),
                   bf16x2_to_f16x2_mul(v.z, up), bf16x2_to_f16x2_mul(v.w, up));
    *reinterpret_cast<uint4*>(qr + ((i ^ (hrow & 7)) << 4)) = v;
  }
  tmem_st_wait();
  return mx;
}

__device__ __noinline__ float tc_load_q(const uint4* __restrict__ src, bool valid, int crank,
                                        uint32_t taddr, unsigned char* qr, int hrow,
                                        float qs_prev) {
  const int e_hint =
      qs_prev == 0.0f ? kNoQHint : (int)((__float_as_uint(qs_prev) >> 23) & 255u) - 127 + 14;
  int e;
  if (__all_sync(0xffffffffu, e_hint != kNoQHint)) {
    e = e_hint;
    const uint32_t mx = tc_q_convert(src, valid, crank, taddr, qr, hrow, e);
    const int et = (int)(mx >> 7) - 127;
    const bool redo = valid && mx != 0 && (et > e + 1 || et < e - 8);
    if (__any_sync(0xffffffffu, redo)) {
      if (mx != 0) e = et;
      tc_q_convert(src, valid, crank, taddr, qr, hrow, e);
    }
  } else {
    uint32_t mx = 0;  // largest |bf16| bit pattern over the CTA's 288 dims
    if (valid) {
#pragma unroll 12
      for (int i = 0; i < 36; ++i)
        mx = q_piece_mx(__ldg(src + (i < 32 ? crank * 32 + i : 64 + crank * 4 + (i - 32))), mx);
    }
    e = mx == 0 ? 127 : (int)(mx >> 7) - 127;  // (an all-zero head: no scaling)
    tc_q_convert(src, valid, crank, taddr, qr, hrow, e);
  }
  return e > 127 - 14 ? 1.0f : __uint_as_float((uint32_t)(127 - 14 + e) << 23);
}

template <int KVT, bool FUSED, bool SPARSE>
__global__ void __launch_bounds__(kTcThreads, 1)
decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tm_lat,
                 const __grid_constant__ CUtensorMap tm_tail,
                 const __grid_constant__ CUtensorMap tm_out) {
  using C = TcCfg<KVT>;
  using L = TcLay<KVT>;
  constexpr int TN = kTN, NS = C::NS, NK = C::NK;
  constexpr bool FP8 = KVT == DCP_KV_FP8_E4M3_S128;
  extern __shared__ unsigned char smem_raw[];
  // 1024-B aligned base, derived from the shared array itself (keeps the address space)
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ TcShared sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_rank();
  const uint32_t peer = crank ^ 1u;
  const int pair = blockIdx.x >> 1;
  const int P = p.pairs;
  const int64_t U = p.num_units;
  const int H = p.heads;
  volatile int* abort_flag = &sh.abort_flag;

  // ---------------------------------------------------------------- set-up
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sh.stg_full[i], 1);  // the loader's expect-tx arrival; bytes from the gathers
      mbar_init(&sh.stg_empty[i], 4);
      sh.stg_issued[i] = 0;
    }
    for (int i = 0; i < NK; ++i) {
      mbar_init(&sh.kt_full[i], 4);
      mbar_init(&sh.kt_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.p_full[i], 8);
      mbar_init(&sh.in_full[i], 1);
      mbar_init(&sh.out_free[i], 8);  // one arrival per stage-B warp of the peer
      mbar_init(&sh.s_free[i], 4);
    }
    mbar_init(&sh.pv_done[0], 1);
    mbar_init(&sh.pv_done[1], 1);
    mbar_init(&sh.q_ready, 4);
    mbar_init(&sh.drain, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.self_full[i], 4);
      mbar_init(&sh.self_free[i], 8);
    }
    for (int g = 0; g < 4; ++g) {
      mbar_init(&sh.bx_full[g][0], 2);
      mbar_init(&sh.bx_full[g][1], 2);
      mbar_init(&sh.bl_full[g], 2);
      mbar_init(&sh.ep_done[g], 2);
    }
    sh.abort_flag = 0;
    fence_mbar_init();
    // the exchange inboxes expect one tile of partial logits each
    mbar_arrive_expect_tx(&sh.in_full[0], L::X_BYTES);
    mbar_arrive_expect_tx(&sh.in_full[1], L::X_BYTES);
  }

  // this pair's contiguous range of the tile sequence
  int64_t* scan_tmp = reinterpret_cast<int64_t*>(smem + L::OFF_META);  // metadata is unused yet
  if (FUSED && SPARSE) {
    const int64_t tu = (p.k + TN - 1) / TN;
    const int64_t T = U * tu;
    const int Pe = (int)(T < P ? (T > 0 ? T : 1) : P);
    const int64_t t0 = pair < Pe ? pair * T / Pe : T, t1 = pair < Pe ? (pair + 1) * T / Pe : T;
    if (tid == 0) {
      sh.Peff = Pe;
      sh.T = T;
      sh.t0 = t0;
      sh.ntiles = (int)(t1 - t0);
      sh.unit0 = t0 < T ? t0 / tu : 0;
      sh.tile0 = t0 < T ? (int)(t0 % tu) : 0;
    }
  } else {
    int64_t part = 0;
    for (int64_t v = tid; v < U; v += kTcThreads) part += get_unit<FUSED, SPARSE>(p, v).ntile;
    int64_t T;
    block_scan_excl(part, scan_tmp, &T);
    const int Pe = (int)(T < P ? (T > 0 ? T : 1) : P);
    const int64_t t0 = pair < Pe ? pair * T / Pe : T, t1 = pair < Pe ? (pair + 1) * T / Pe : T;
    if (tid == 0) {
      sh.Peff = Pe;
      sh.T = T;
      sh.t0 = t0;
      sh.ntiles = (int)(t1 - t0);
      sh.unit0 = 0;
      sh.tile0 = 0;
      sh.scan_base = 0;
    }
    __syncthreads();
    if (t1 > t0) {
      for (int64_t c0 = 0; c0 < U; c0 += kTcThreads) {
        const int64_t v = c0 + tid;  // order index
        const int nt = v < U ? get_unit<FUSED, SPARSE>(p, v).ntile : 0;
        int64_t chunk_total;
        const int64_t excl = block_scan_excl(nt, scan_tmp, &chunk_total) + sh.scan_base;
        if (nt > 0 && t0 >= excl && t0 < excl + nt) {
          sh.unit0 = v;
          sh.tile0 = (int)(t0 - excl);
        }
        __syncthreads();
        if (tid == 0) sh.scan_base += chunk_total;
        __syncthreads();
        if (sh.scan_base > t0) break;
      }
    }
  }
  // this pair's split descriptors start empty in every call (a descriptor is filled below
  // only when the pair's range cuts a unit), so the workspace needs no clearing between calls
  if (crank == 0 && tid == 0) {
    p.tc_desc[2 + (int64_t)pair * 6 + 2] = 0;
    p.tc_desc[2 + (int64_t)pair * 6 + 5] = 0;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // peers' barriers are initialised before any remote arrive or copy
  tc_fence_after();
  const uint32_t tbase = sh.tmem_base;
  const int ntiles = sh.ntiles;
  if (blockIdx.x == 0 && tid == 0) {  // the tile sequence, for the split-merge kernel
    p.tc_desc[0] = sh.T;
    p.tc_desc[1] = sh.Peff;
  }
  const int64_t t0 = sh.t0;

  // Loader warps take tiles round-robin; a staging slot's empty barrier is waited on by
  // parity, which tells phases apart only while the barrier is at most one phase behind:
  // with NS >= NLD every loader's previous wait (tile j - NLD) has already seen tile
  // j - NLD - NS >= j - 2 NS released.
  constexpr int NLD = NS < 3 ? NS : 3;
  static_assert(NS >= NLD, "staging slots must not be fewer than loader warps");
  if (warp >= 1 && warp <= NLD) {
    // ============================================================ loaders
    // Warp 1+li takes tiles j = li, li+NLD, ...; lane t handles slot t of a tile.  Stage I
    // loads the tile's slot ids (two tiles of this warp ahead), stage T maps them to owner
    // shard / local slot and loads the block-table entry (one tile ahead), stage C turns
    // pages into pool rows and issues one latent and one tail gather per 4 slots.
    const int li = warp - 1;
    if (li == 0 && lane == 0) {
      prefetch_tensormap(&tm_lat);
      prefetch_tensormap(&tm_tail);
    }
    // gather column offsets (elements of the map: bytes for FP8, bf16 for BF16)
    const int xa = (int)crank * 256;
    const int xb = FP8 ? 512 : 512 + 32 * (int)crank;
    Walk<FUSED, SPARSE> wi;
    wi.init(p, sh.unit0, sh.tile0, ntiles);
    for (int k = 0; k < li && k + 1 < ntiles; ++k) wi.next(p);
    int t_v = -1;                   // stage T: slot id (global, local, or position)
    bool t_has = false;             // stage T: the position holds a slot of the unit
    UnitInfo t_x = wi.info;
    int c_page = -1, c_l = -1;      // stage C: page and local slot (c_l < 0: no slot)
    for (int n = 0;; ++n) {
      const int jc = li + NLD * (n - 2), jt = jc + NLD, ji = jt + NLD;
      if (jc >= ntiles) break;
      if (jc >= 0) {
        const int slot = jc % NS;
        if (!mbar_wait(&sh.stg_empty[slot], ((jc / NS) & 1) ^ 1, abort_flag)) break;
        int row = -1;
        if (c_l >= 0) {
          if (c_page >= 0 && c_page < p.num_pages)
            row = c_page * 64 + (c_l & 63);  // < 2^31: the host checks num_pages * 64
          else
            set_err(p.err, DCP_ERRBIT_PAGE_RANGE);
        }
        const unsigned mask = __ballot_sync(0xffffffffu, row >= 0);
        // empty positions of a 4-slot group re-read a valid row of the group (their data
        // is replaced by zeros in the converter); groups without any row are not fetched
        const unsigned quad = (mask >> (lane & ~3)) & 0xFu;
        const int sub = __shfl_sync(0xffffffffu, row, (lane & ~3) + (quad ? __ffs(quad) - 1 : 0));
        const int rowfix = row >= 0 ? row : sub;
        const int g = lane & 7;
        const int y0 = __shfl_sync(0xffffffffu, rowfix, 4 * g);
        const int y1 = __shfl_sync(0xffffffffu, rowfix, 4 * g + 1);
        const int y2 = __shfl_sync(0xffffffffu, rowfix, 4 * g + 2);
        const int y3 = __shfl_sync(0xffffffffu, rowfix, 4 * g + 3);
        const bool gnz = ((mask >> (4 * g)) & 0xFu) != 0;
        const unsigned gmask = __ballot_sync(0xffffffffu, lane < 8 && gnz);
        unsigned char* stg = smem + L::OFF_STG + slot * L::STG_BYTES;
        if (lane == 0) {
          sh.stg_mask[slot] = mask;
          sh.stg_issued[slot] += 1;
          mbar_arrive_expect_tx(&sh.stg_full[slot], __popc(gmask) * L::GROUP_TX);
        }
        __syncwarp();
        if (lane < 8 && gnz) {
          tma_gather4(stg + g * 4 * C::LAT_TOK, &tm_lat, xa, y0, y1, y2, y3, &sh.stg_full[slot]);
          tma_gather4(stg + L::STG_TAIL + g * C::TAIL_GSTRIDE, &tm_tail, xb, y0, y1, y2, y3,
                      &sh.stg_full[slot]);
        }
      }
      // stage T for tile jt
      int n_page = -1, n_l = -1;
      if (jt >= 0 && jt < ntiles && t_has && t_v < 0 && !FUSED)
        set_err(p.err, DCP_ERRBIT_SLOT_RANGE);  // a negative local id among the valid ones
      if (jt >= 0 && jt < ntiles && t_has && t_v >= 0) {
        int l;
        const int32_t* table;
        if (FUSED) {
          int s;
          owner_local(t_v, p.rule, s, l);
          table = p.bt + ((int64_t)s * p.num_seqs + t_x.b) * p.bt_stride;
        } else {
          l = t_v;
          table = p.bt + ((int64_t)t_x.shard * p.num_seqs + t_x.b) * p.bt_stride;
        }
        const int pj = l >> 6;
        if (pj < p.bt_stride) {
          n_page = __ldg(table + pj);  // consumed in stage C, one tile of this warp later
          n_l = l;
        } else {
          set_err(p.err, DCP_ERRBIT_SLOT_RANGE);
        }
      }
      // stage I for tile ji
      int n_v = -1;
      bool n_has = false;
      const UnitInfo n_x = wi.info;
      if (ji < ntiles) {
        const int pos = wi.lt * TN + lane;
        if (pos < wi.info.n) {
          n_has = true;
          if (SPARSE) {
            const int64_t base = (FUSED ? wi.info.r : wi.info.u) * (int64_t)p.k;
            n_v = __ldg(p.idx + base + pos);  // consumed in stage T
          } else {
            n_v = pos;
          }
        }
      }
      if (ji < ntiles)
        for (int k = 0; k < NLD; ++k) wi.next(p);
      c_page = n_page;
      c_l = n_l;
      t_v = n_v;
      t_has = n_has;
      t_x = n_x;
    }
  } else if (warp >= 1 && warp <= 3) {
    // a loader warp this configuration does not use
  } else if (warp == 0) {
    // ============================================================ MMA issuer
    // Issues Q.K^T(jq) and P.V(jp) in whatever order their inputs become ready (P.V first:
    // it frees a K slot and a P buffer), polling the barriers without blocking on either.
    //   QK(jq): Q of its unit in TMEM (q_ready; the pair's first tile always loads Q), K tile
    //           jq converted (kt_full), logit buffer jq&1 read by stage A(jq-2) (s_free);
    //   PV(jp): P(jp) in shared memory (p_full).
    constexpr uint32_t idesc_qk = idesc_f16(128, TN, 0, 0);
    constexpr uint32_t idesc_pv = FP8 ? idesc_f16(128, 128, 0, 1) : idesc_f16(128, 256, 0, 1);
    const uint32_t qb = tbase + kColQ;
    const uint64_t qrd = smem_desc(smem_u32(smem + L::OFF_QR), 16, 1024);
    const uint32_t leader = elect_one();
    Walk<FUSED, SPARSE> wq, wp;
    wq.init(p, sh.unit0, sh.tile0, ntiles);
    wp = wq;
    int jq = 0, jp = 0, q_phase = 0;
    uint64_t t_last = globaltimer();
    int idle = 0;
    while (jp < ntiles) {
      bool progressed = false;
      if (jp < jq && mbar_test(&sh.p_full[jp & 1], (jp >> 1) & 1)) {
        tc_fence_after();
        const uint32_t kt = smem_u32(smem + L::OFF_KT + (jp % NK) * L::KT_BYTES);
        const uint64_t pd = smem_desc(smem_u32(smem + L::OFF_P + (jp % C::NP) * L::P_BYTES), 16, 1024);
        // a unit's (or this pair's) first tile overwrites O
        const uint32_t acc0 = (wp.first() || jp == 0) ? 0u : 1u;
        if (FP8) {  // P row: [p*s_lo for slots 0-31 | p*s_hi for slots 0-31]
          mma_ss_if(leader, tbase + kColO, pd, smem_desc(kt, L::BS, 1024), idesc_pv, acc0);
          mma_ss_if(leader, tbase + kColO + 128, pd + (64 >> 4),
                    smem_desc(kt + 2 * L::BS, L::BS, 1024), idesc_pv, acc0);
          mma_ss_if(leader, tbase + kColO, pd + (32 >> 4), smem_desc(kt + 2048, L::BS, 1024),
                    idesc_pv, 1);
          mma_ss_if(leader, tbase + kColO + 128, pd + (96 >> 4),
                    smem_desc(kt + 2 * L::BS + 2048, L::BS, 1024), idesc_pv, 1);
        } else {
          mma_ss_if(leader, tbase + kColO, pd, smem_desc(kt, L::BS, 1024), idesc_pv, acc0);
          mma_ss_if(leader, tbase + kColO, pd + (32 >> 4), smem_desc(kt + 2048, L::BS, 1024),
                    idesc_pv, 1);
        }
        mma_commit_if(leader, &sh.kt_empty[jp % NK]);
        mma_commit_if(leader, &sh.pv_done[jp & 1]);
        wp.next(p);
        ++jp;
        progressed = true;
      }
      if (jq < ntiles) {
        const bool unit_first = jq == 0 || wq.first();
        if ((!unit_first || mbar_test(&sh.q_ready, q_phase & 1)) &&
            mbar_test(&sh.kt_full[jq % NK], (jq / NK) & 1) &&
            (jq < 2 || mbar_test(&sh.s_free[jq & 1], ((jq - 2) >> 1) & 1))) {
          if (unit_first) ++q_phase;
          tc_fence_after();
          const uint32_t kt = smem_u32(smem + L::OFF_KT + (jq % NK) * L::KT_BYTES);
          const uint32_t sb = tbase + kColS + (jq & 1) * L::SBUF;
          const uint64_t kd = smem_desc(kt, 16, 1024);
          // start-address field (address >> 4) of K-step ks of the latent blocks / RoPE block
#define KOFF(ks) ((uint64_t)((((ks) >> 2) * L::BS + ((ks) & 3) * 32) >> 4))
#define ROFF(i) ((uint64_t)((4 * L::BS + (i) * 32) >> 4))
          if (FP8) {
            // the two latent-block chains interleaved (consecutive MMAs write different
            // accumulators), then the RoPE high parts and remainders into the lo chain
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int ks = (i >> 1) + 8 * (i & 1);
              mma_ts_if(leader, sb + (i & 1) * TN, qb + 8 * ks, kd + KOFF(ks), idesc_qk,
                        (ks & 7) != 0);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
              mma_ss_if(leader, sb, qrd + (uint64_t)(((i & 1) * 32) >> 4), kd + ROFF(i), idesc_qk, 1);
          } else {
#pragma unroll
            for (int ks = 0; ks < 16; ++ks)
              mma_ts_if(leader, sb, qb + 8 * ks, kd + KOFF(ks), idesc_qk, ks > 0);
#pragma unroll
            for (int i = 0; i < 2; ++i)
              mma_ss_if(leader, sb, qrd + (uint64_t)((i * 32) >> 4), kd + ROFF(i), idesc_qk, 1);
          }
#undef KOFF
#undef ROFF
          mma_commit_if(leader, &sh.s_full[jq & 1]);
          ++jq;
          wq.next(p);
          progressed = true;
        }
      }
      if (progressed) {
        idle = 0;
        t_last = globaltimer();
      } else {
        if (*abort_flag) break;
        if (++idle >= 32) {
          idle = 0;
          if (globaltimer() - t_last > kWaitLimitNs) {
            *abort_flag = 1;
            break;
          }
        }
        __nanosleep(32);
      }
    }
    mma_commit_elect(&sh.drain);
    volatile int no_abort = 0;
    mbar_wait(&sh.drain, 0, &no_abort);  // no MMA in flight before TMEM is released
  } else if (warp >= 4 && warp < 8) {
    // ============================================================ converters
    // Latent part: thread -> slot t = 8*(warp-4) + 2*(lane>>3) + ((lane>>2)&1), 16-B chunks
    // ch = (lane&3) + 4*(it ^ ((lane>>2)&1)): each 8-lane phase of a 16-B access reads 8
    // distinct bank groups of the staging rows and writes 8 distinct swizzled chunks.
    // The K tile holds FP16 values.  FP8: a block's codes times 2^E, E the power-of-two part
    // of the block's scale (exact in FP16), the rest m = scale / 2^E in [1, 2) kept for the
    // logit and P; BF16: the values themselves.
    const int ct = tid - 128;
    const int l8 = lane & 7, hb = l8 >> 2;
    const int t = 8 * (ct >> 5) + 2 * (lane >> 3) + hb;
    const float sl2 = p.scale_log2;
    for (int j = 0; j < ntiles; ++j) {
      const int slot = j % NS, ks = j % NK;
      if (!mbar_wait(&sh.stg_full[slot], (j / NS) & 1, abort_flag)) break;
      if (!mbar_wait(&sh.kt_empty[ks], ((j / NK) & 1) ^ 1, abort_flag)) break;
      const uint32_t mask = sh.stg_mask[slot];
      const unsigned char* stg = smem + L::OFF_STG + slot * L::STG_BYTES;
      unsigned char* kt = smem + L::OFF_KT + ks * L::KT_BYTES;
      unsigned char* meta = smem + L::OFF_META + ks * L::META_BYTES;
      const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
      const bool live = (mask >> t) & 1;
      if (FP8) {
        // this slot's two block scales -> f16x2 multipliers 2^E (0 for a negligible block)
        float2 sc = make_float2(0.f, 0.f);
        if (live) {
          const float* sp = reinterpret_cast<const float*>(
              stg + L::STG_TAIL + (t >> 2) * C::TAIL_GSTRIDE + (t & 3) * C::TAIL_TOK);
          sc = make_float2(sp[2 * crank], sp[2 * crank + 1]);
        }
        const uint32_t mul2[2] = {fp8_block_mul(sc.x), fp8_block_mul(sc.y)};
        uint4 v[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {  // 16 codes per chunk
          const int ch = (l8 & 3) + 4 * (it ^ hb);
          v[it] = live ? *reinterpret_cast<const uint4*>(stg + t * C::LAT_TOK + ch * 16) : zero;
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int ch = (l8 & 3) + 4 * (it ^ hb);
          const uint32_t mul = mul2[ch >> 3];
          const uint32_t in[4] = {v[it].x, v[it].y, v[it].z, v[it].w};
          uint32_t o[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            o[2 * e] = e4m3x2_to_f16x2_mul((uint16_t)(in[e] & 0xffffu), mul);
            o[2 * e + 1] = e4m3x2_to_f16x2_mul((uint16_t)(in[e] >> 16), mul);
          }
          unsigned char* base = kt + (ch >> 2) * L::BS + t * 128;
          const int c16 = (ch & 3) * 2;
          *reinterpret_cast<uint4*>(base + ((c16 ^ (t & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(base + (((c16 + 1) ^ (t & 7)) << 4)) =
              make_uint4(o[4], o[5], o[6], o[7]);
        }
        {  // RoPE: thread -> (slot rt, 8 of this CTA's 32 dims); block multipliers
          const int rt = ct >> 2, c4 = ct & 3;
          const unsigned char* tail = stg + L::STG_TAIL + (rt >> 2) * C::TAIL_GSTRIDE + (rt & 3) * C::TAIL_TOK;
          uint32_t hw[4] = {0u, 0u, 0u, 0u}, lw[4] = {0u, 0u, 0u, 0u};
          float mlo = 0.f, mhi = 0.f, mf = 1.f;
          if ((mask >> rt) & 1) {
            const float4 sc4 = *reinterpret_cast<const float4*>(tail);
            mlo = fp8_block_m(crank == 0 ? sc4.x : sc4.z);
            mhi = fp8_block_m(crank == 0 ? sc4.y : sc4.w);
            // the RoPE part rides in the lo accumulator, which is scaled by m_lo later;
            // m_lo is 0 only for a block whose values are all zero (its codes count as 0)
            mf = mlo > 0.f ? mlo : 1.f;
            const float inv = 1.0f / mf;
            const uint4 r = *reinterpret_cast<const uint4*>(tail + 16 + 64 * crank + 16 * c4);
            const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float y0 = __uint_as_float(rw[e] << 16) * inv;
              const float y1 = __uint_as_float(rw[e] & 0xffff0000u) * inv;
              const uint32_t h2 = pack_f16x2(y0, y1);
              const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&h2));
              hw[e] = h2;
              lw[e] = pack_f16x2(y0 - hf.x, y1 - hf.y);
            }
          }
          unsigned char* rb = kt + 4 * L::BS + rt * 128;
          *reinterpret_cast<uint4*>(rb + ((c4 ^ (rt & 7)) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(rb + (((4 + c4) ^ (rt & 7)) << 4)) =
              make_uint4(lw[0], lw[1], lw[2], lw[3]);
          if (c4 == 0) {
            float* mfp = reinterpret_cast<float*>(meta);
            mfp[rt] = mf * sl2;        // logit multiplier of the lo accumulator
            mfp[TN + rt] = mhi * sl2;  // of the hi accumulator
            mfp[2 * TN + rt] = mlo;    // P multipliers of the lo / hi block values
            mfp[3 * TN + rt] = mhi;
          }
        }
      } else {
        uint4 v[8];
#pragma unroll
        for (int it = 0; it < 8; ++it) {  // 8 bf16 per chunk
          const int ch = (l8 & 3) + 4 * (it ^ hb);
          v[it] = live ? *reinterpret_cast<const uint4*>(stg + t * C::LAT_TOK + ch * 16) : zero;
        }
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int ch = (l8 & 3) + 4 * (it ^ hb);
          const uint4 w = make_uint4(bf16x2_to_f16x2_mul(v[it].x, 1.f), bf16x2_to_f16x2_mul(v[it].y, 1.f),
                                     bf16x2_to_f16x2_mul(v[it].z, 1.f), bf16x2_to_f16x2_mul(v[it].w, 1.f));
          *reinterpret_cast<uint4*>(kt + (ch >> 3) * L::BS + t * 128 + (((ch & 7) ^ (t & 7)) << 4)) = w;
        }
        {
          const int rt = ct >> 2, c4 = ct & 3;
          uint4 r = (mask >> rt) & 1
                        ? *reinterpret_cast<const uint4*>(stg + L::STG_TAIL + rt * C::TAIL_TOK + c4 * 16)
                        : zero;
          r = make_uint4(bf16x2_to_f16x2_mul(r.x, 1.f), bf16x2_to_f16x2_mul(r.y, 1.f),
                         bf16x2_to_f16x2_mul(r.z, 1.f), bf16x2_to_f16x2_mul(r.w, 1.f));
          *reinterpret_cast<uint4*>(kt + 4 * L::BS + rt * 128 + ((c4 ^ (rt & 7)) << 4)) = r;
        }
      }
      if (ct == 0) sh.kt_mask[ks] = mask;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {  // one arrival per warp (arrivals of 128 threads serialise)
        mbar_arrive(&sh.kt_full[ks]);
        mbar_arrive(&sh.stg_empty[slot]);
      }
    }
  } else if (warp >= 12 && warp < 16) {
    // ============================================================ softmax stage A
    const int h = tid - 384;  // head = TMEM lane
    const uint32_t trow = tbase + ((uint32_t)((warp & 3) * 32) << 16);
    float* xin = reinterpret_cast<float*>(smem + L::OFF_X);
    float* xself = reinterpret_cast<float*>(smem + L::OFF_SELF);
    float qs = 0.0f;  // 2^(e - 14) of this head's Q in the current row (see tc_load_q)
    auto load_q = [&](int64_t r) {
      const uint4* src = reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(p.q) + (r * H + h) * kDqk);
      unsigned char* qr = smem + L::OFF_QR + (h >> 3) * 1024 + (h & 7) * 128;
      qs = tc_load_q(src, h < H, (int)crank, trow + kColQ, qr, h, qs);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.q_ready);
    };
    // this thread's lines of row r of Q into L2 (its CTA's latent half and the RoPE dims of
    // both CTAs), a few tiles before the row is needed
    auto prefetch_q = [&](int64_t r) {
      if (h >= H || r >= p.rows) return;
      const char* qn = reinterpret_cast<const char*>(p.q) + (r * H + h) * (kDqk * 2);
#pragma unroll
      for (int l = 0; l < 4; ++l) prefetch_l2(qn + crank * 512 + 128 * l);
      prefetch_l2(qn + 1024);
    };

    Walk<FUSED, SPARSE> wa;
    wa.init(p, sh.unit0, sh.tile0, ntiles);
    // the pair's first unit, even when it starts mid-unit
    if (ntiles > 0) load_q(wa.info.r);
    for (int j = 0; j < ntiles; ++j) {
      const int buf = j & 1;
      // the next row's Q into L2 four tiles before this unit's end (the rows of the
      // partial form's units follow one another too)
      if (wa.lt == max(0, wa.info.ntile - 4)) prefetch_q(wa.info.r + 1);
      if (!mbar_wait(&sh.s_full[buf], (j >> 1) & 1, abort_flag)) break;
      if (!mbar_wait(&sh.kt_full[j % NK], (j / NK) & 1, abort_flag)) break;
      tc_fence_after();
      const unsigned char* meta = smem + L::OFF_META + (j % NK) * L::META_BYTES;
      const uint32_t sb = trow + kColS + buf * L::SBUF;
      const float qs_tile = qs;  // this tile's unit (the next unit's Q may load below)
      float s[TN];
      if (!FP8) {
        uint32_t a[TN];
        tmem_ld16(sb, a);
        tmem_ld16(sb + 16, a + 16);
        tmem_ld_wait();
        const float f = p.scale_log2 * qs_tile;
#pragma unroll
        for (int t = 0; t < TN; ++t) s[t] = __uint_as_float(a[t]) * f;
      } else {
        const float4* ma = reinterpret_cast<const float4*>(meta);
        const float4* mb = ma + TN / 4;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t lo[16], hi[16];
          tmem_ld16(sb + 16 * hf, lo);
          tmem_ld16(sb + TN + 16 * hf, hi);
          tmem_ld_wait();
#pragma unroll
          for (int t4 = 0; t4 < 4; ++t4) {
            const float4 a = ma[4 * hf + t4], b = mb[4 * hf + t4];
            const int t = 16 * hf + 4 * t4;
            s[t] = fmaf(__uint_as_float(lo[4 * t4]), a.x, __uint_as_float(hi[4 * t4]) * b.x) * qs_tile;
            s[t + 1] = fmaf(__uint_as_float(lo[4 * t4 + 1]), a.y, __uint_as_float(hi[4 * t4 + 1]) * b.y) * qs_tile;
            s[t + 2] = fmaf(__uint_as_float(lo[4 * t4 + 2]), a.z, __uint_as_float(hi[4 * t4 + 2]) * b.z) * qs_tile;
            s[t + 3] = fmaf(__uint_as_float(lo[4 * t4 + 3]), a.w, __uint_as_float(hi[4 * t4 + 3]) * b.w) * qs_tile;
          }
        }
      }
      // logit buffer j&1 may take S(j+2) now
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.s_free[buf]);
      // this CTA's partial into the local box: read by stage B (free once B(j-1) read it)
      // and copied to the peer's inbox (the warp's 32 rows in one bulk copy, free once the
      // copy of tile j-1 has read them)
      const int x = buf;
      const int xs = j % C::NSB;  // local box of this tile
      if (!mbar_wait(&sh.self_free[xs], ((j / C::NSB) & 1) ^ 1, abort_flag)) break;
      if (lane == 0) bulk_wait_read<C::NSB - 1>();  // the copy of tile j - NSB has read it
      __syncwarp();
      float* srow = xself + (xs * 128 + h) * L::XSTRIDE;
#pragma unroll
      for (int c = 0; c < TN / 4; ++c)
        *reinterpret_cast<float4*>(srow + 4 * c) =
            make_float4(s[4 * c], s[4 * c + 1], s[4 * c + 2], s[4 * c + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.self_full[xs]);
      if (!mbar_wait(&sh.out_free[x], ((j >> 1) & 1) ^ 1, abort_flag, true)) break;
      if (lane == 0) {
        const int r0 = (warp & 3) * 32;
        bulk_s2peer(xin + (x * 128 + r0) * L::XSTRIDE, xself + (xs * 128 + r0) * L::XSTRIDE,
                    32 * L::XSTRIDE * 4, peer, &sh.in_full[x]);
        bulk_commit();
      }
      // the next unit's queries go in once this tile's Q.K^T is done and its partial is on
      // its way (the next unit's first Q.K^T waits for them; stage B of this tile does not);
      // the next shard's unit of the same row keeps them
      if (wa.last() && j + 1 < ntiles) {
        Walk<FUSED, SPARSE> wn = wa;
        wn.next(p);
        if (wn.info.r != wa.info.r) {
          load_q(wn.info.r);
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.q_ready);
        }
      }
      wa.next(p);
    }
    if (lane == 0) bulk_wait0();  // no copy to the peer in flight when the CTA winds down
    __syncwarp();
  } else if (warp >= 8) {
    // ============================================================ softmax stage B / epilogue
    // Warps 8-11 and 16-19: warp 8+g and warp 16+g share heads 32g .. 32g+31 (TMEM lanes of
    // sub-partition g); half 0 takes columns 0-15 of every tile and O columns 0-127, half 1
    // columns 16-31 and O columns 128-255.  The two exchange their partial row maxima every
    // tile and their partial row sums at the end of a unit (bounded mbarrier waits).
    constexpr int TH = TN / 2;
    const int half = warp >= 16 ? 1 : 0;
    const int grp = warp & 3;
    const int h = grp * 32 + lane;  // head = TMEM lane
    const int cb = half * TH;       // first column of this half
    const uint32_t trow = tbase + ((uint32_t)(grp * 32) << 16);
    const float* xin = reinterpret_cast<const float*>(smem + L::OFF_X);
    const float* xself = reinterpret_cast<const float*>(smem + L::OFF_SELF);

    // units without any slot: zero output, -inf LSE
    if (!(FUSED && SPARSE) && half == 0) {
      for (int64_t v = pair; v < U; v += P) {
        const UnitInfo x = get_unit<FUSED, SPARSE>(p, v);
        if (x.ntile != 0 || h >= H) continue;
        const int64_t u = x.u;
        const int64_t oi = (u * H + h) * kDv + crank * 256;
        if (FUSED) {
          uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + oi);
          for (int i = 0; i < 32; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
        } else {
          float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + oi);
          for (int i = 0; i < 64; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (crank == 0) p.lse[u * H + h] = -INFINITY;
      }
    }

    Walk<FUSED, SPARSE> w;
    w.init(p, sh.unit0, sh.tile0, ntiles);
    float m_ref = -INFINITY, lsum = 0.f;  // lsum: this half's share of the row sum
    int64_t U0 = t0 - sh.tile0;   // global index of the current unit's first tile
    bool from_start = sh.tile0 == 0;
    int slot_idx = 0;             // workspace slot of a split unit: 0 first unit, 1 last
    int nunit = 0;                // units finished (parity of the row-sum exchange)
    int nep = 0;                  // tiled-store epilogues done (phase of ep_done)
    bool ok = true;

    // Finish the current unit: normalise and write this half's O columns (or a split
    // partial) and the LSE.
    auto finish_unit = [&](int jl, bool complete) {
      sh.bl[half][h] = lsum;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.bl_full[grp]);
      if (!(ok = mbar_wait(&sh.bl_full[grp], nunit & 1, abort_flag))) return;
      ++nunit;
      const float ltot = lsum + sh.bl[half ^ 1][h];
      volatile int no_abort = 0;
      mbar_wait(&sh.pv_done[jl & 1], (jl >> 1) & 1, ok ? abort_flag : &no_abort);
      tc_fence_after();
      const float fix = ltot > 0.f ? 1.0f / ltot : 0.f;
      const float lse_v = ltot > 0.f ? (m_ref + __log2f(ltot)) * kLn2 : -INFINITY;
      const int64_t u = w.info.u;
      float* wso = p.tc_o + (((int64_t)pair * 2 + slot_idx) * 128 + h) * kDv + crank * 256;
      // This half's 128 O columns in four rounds of 32.  A split partial goes straight to the
      // workspace.  A finished unit goes through shared memory so that the global stores are
      // row-contiguous: each lane puts its head's 32 values into its row of this half's chunks
      // of the two P buffers (both free: P.V of this unit's last tile is done, and each half
      // uses only the chunks it writes P into), then the warp stores 4 heads (fp32) or 8 heads
      // (bf16) per instruction, 128 or 64 contiguous bytes each.
      unsigned char* pst = smem + L::OFF_P;
      auto stage_addr = [&](int r, int k) -> unsigned char* {  // row r, float4 k of 8
        const int cc = (k & 3) < 2 ? 2 * half + (k & 3) : 4 + 2 * half + (k & 3) - 2;
        return pst + (k >> 2) * L::P_BYTES + (r >> 3) * 1024 + (r & 7) * 128 +
               ((cc ^ (r & 7)) << 4);
      };
#pragma unroll 1
      for (int rc = 0; rc < 4; ++rc) {
        const int c0 = half * 8 + 2 * rc;  // first 16-column chunk of pass rc
        uint32_t v[2][16];
        tmem_ld16(trow + kColO + 16 * c0, v[0]);
        tmem_ld16(trow + kColO + 16 * (c0 + 1), v[1]);
        tmem_ld_wait();
        float f[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i >> 4][i & 15]) * fix;
        if (!complete) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            __stcg(reinterpret_cast<float4*>(wso + 16 * c0) + i,
                   make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]));
          continue;
        }
        if (!FUSED && p.tma_out) {
          // this warp's 32 rows x 32 columns, as the output map's 128-B swizzled box, in its
          // rows of the P buffer of its half (free: see the barrier after the rounds), then
          // one tiled store by lane 0; the previous round's store must have read the box
          unsigned char* box = smem + L::OFF_P + half * L::P_BYTES + grp * 4096;
          if (rc > 0) {
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
          }
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4*>(box + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && grp * 32 < H) {
            tma_store_3d(&tm_out, box, (int)crank * 256 + 16 * c0, grp * 32, (int)u);
            bulk_commit();
          }
          continue;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<float4*>(stage_addr(h, k)) =
              make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
        __syncwarp();
        const int64_t col = crank * 256 + 16 * c0;  // first output column of the round
        if (FUSED) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = grp * 32 + 8 * i + (lane >> 2), q = lane & 3;
            const float4 a = *reinterpret_cast<const float4*>(stage_addr(r, 2 * q));
            const float4 b = *reinterpret_cast<const float4*>(stage_addr(r, 2 * q + 1));
            if (r < H)
              *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                        (u * H + r) * kDv + col + 8 * q) =
                  make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                             pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = grp * 32 + 4 * i + (lane >> 3), q = lane & 7;
            const float4 a = *reinterpret_cast<const float4*>(stage_addr(r, q));
            if (r < H)
              *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + (u * H + r) * kDv +
                                         col + 4 * q) = a;
          }
        }
        __syncwarp();  // the rows are read before the next round overwrites them
      }
      tc_fence_before();
      if (!FUSED && complete && p.tma_out) {
        // both halves' boxes read out (each half stages in the P buffer whose other columns
        // the other half may fill with the next tile's P) before either half goes on
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.ep_done[grp]);
        if (!(ok = mbar_wait(&sh.ep_done[grp], nep & 1, abort_flag))) return;
        ++nep;
      }
      if (complete) {
        if (half == 0 && crank == 0 && h < H) p.lse[u * H + h] = lse_v;
        return;
      }
      // split unit: publish this pair's partial and its descriptor; the split-merge kernel
      // that follows on the stream combines the parts of every split unit
      if (half == 0) __stcg(p.tc_l + (((int64_t)pair * 2 + slot_idx) * 2 + crank) * 128 + h, lse_v);
      if (half == 0 && crank == 0 && h == 0) {
        int64_t* d = p.tc_desc + 2 + ((int64_t)pair * 2 + slot_idx) * 3;
        d[0] = u;
        d[1] = U0;
        d[2] = U0 + w.info.ntile;
      }
    };

    int j = 0;
    for (; ok && j < ntiles; ++j) {
      const int x = j & 1;
      const unsigned char* meta = smem + L::OFF_META + (j % NK) * L::META_BYTES;
      // P(j) goes into shared-memory buffer j % NP once P.V(j-NP) has read it (waited below)
      unsigned char* prow = smem + L::OFF_P + (j % C::NP) * L::P_BYTES + (h >> 3) * 1024 + (h & 7) * 128;
      float s[TH];
      // A(j) hands over after it saw the K tile complete: the tile's metadata is valid
      const int xs = j % C::NSB;
      if (!(ok = mbar_wait(&sh.self_full[xs], (j / C::NSB) & 1, abort_flag))) break;
      const uint32_t mask = sh.kt_mask[j % NK] >> cb;
      const float* srow = xself + (xs * 128 + h) * L::XSTRIDE + cb;
#pragma unroll
      for (int c = 0; c < TH / 4; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(srow + 4 * c);
        s[4 * c] = v.x;
        s[4 * c + 1] = v.y;
        s[4 * c + 2] = v.z;
        s[4 * c + 3] = v.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.self_free[xs]);
      if (!(ok = mbar_wait(&sh.in_full[x], (j >> 1) & 1, abort_flag, true))) break;
      const float* xrow = xin + (x * 128 + h) * L::XSTRIDE + cb;
#pragma unroll
      for (int c = 0; c < TH / 4; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(xrow + 4 * c);
        s[4 * c] += v.x;
        s[4 * c + 1] += v.y;
        s[4 * c + 2] += v.z;
        s[4 * c + 3] += v.w;
      }
      // inbox x is re-armed for the peer's next tile now (its phase is complete); each warp
      // hands its rows back to the peer at the end of this stage
      if (warp == 8 && lane == 0) mbar_arrive_expect_tx(&sh.in_full[x], L::X_BYTES);
      // online softmax (base 2) with a lazily raised reference
      if ((mask & 0xffffu) != 0xffffu) {
#pragma unroll
        for (int t = 0; t < TH; ++t)
          if (!((mask >> t) & 1)) s[t] = -INFINITY;
      }
      float mh;
      {
        float r[TH / 2];
#pragma unroll
        for (int t = 0; t < TH / 2; ++t) r[t] = fmaxf(s[t], s[t + TH / 2]);
#pragma unroll
        for (int w2 = TH / 4; w2 >= 1; w2 >>= 1)
#pragma unroll
          for (int t = 0; t < w2; ++t) r[t] = fmaxf(r[t], r[t + w2]);
        mh = r[0];
      }
      // the row max of the whole tile: the two halves post theirs and read the other's; every
      // inbox value of this warp has been loaded and used (the max depends on all of them),
      // so the rows go back to the peer at the same time (a relaxed arrive suffices)
      sh.bx[half][x][h] = mh;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster_relaxed(&sh.out_free[x], peer);
        mbar_arrive(&sh.bx_full[grp][x]);
      }
      if (!(ok = mbar_wait(&sh.bx_full[grp][x], (j >> 1) & 1, abort_flag))) break;
      const float mt = fmaxf(mh, sh.bx[half ^ 1][x][h]);
      // per head: raise the reference when the tile max exceeds it by more than 2^8; the
      // TMEM read-modify-write of O is warp-collective, so a warp rescales when any of its
      // heads needs it (alpha = 1 for the others); each half rescales its own O columns
      float alpha = 1.0f;
      const bool raise = mt > m_ref + 8.0f;
      if (raise && m_ref != -INFINITY) alpha = fast_exp2(m_ref - mt);
      const bool rescale = __any_sync(0xffffffffu, alpha != 1.0f);
      if (rescale) {
        if (!(ok = mbar_wait(&sh.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        for (int c = half * 8; c < half * 8 + 8; ++c) {
          uint32_t v[16];
          tmem_ld16(trow + kColO + 16 * c, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st16(trow + kColO + 16 * c, v);
        }
      }
      if (raise) {
        lsum *= alpha;
        m_ref = mt;
      }
      float pr[TH];
      {
        const float mr = m_ref == -INFINITY ? 0.f : m_ref;  // all -inf: every p is 0
#pragma unroll
        for (int t = 0; t < TH; ++t) pr[t] = fast_exp2(s[t] - mr);
        float r[TH / 2];
#pragma unroll
        for (int t = 0; t < TH / 2; ++t) r[t] = pr[t] + pr[t + TH / 2];
#pragma unroll
        for (int w2 = TH / 4; w2 >= 1; w2 >>= 1)
#pragma unroll
          for (int t = 0; t < w2; ++t) r[t] += r[t + w2];
        lsum += r[0];
      }
      if (j >= C::NP &&
          !(ok = mbar_wait(&sh.pv_done[(j - C::NP) & 1], ((j - C::NP) >> 1) & 1, abort_flag)))
        break;
      const int sw = h & 7;  // SW128: 16-B chunk c of row h sits at chunk c ^ (h & 7)
      if (!FP8) {  // P row: 32 fp16 in chunks 0-3; this half's 16 in chunks 2*half, 2*half+1
        uint32_t pw[TH / 2];
#pragma unroll
        for (int i = 0; i < TH / 2; ++i) pw[i] = pack_f16x2(pr[2 * i], pr[2 * i + 1]);
#pragma unroll
        for (int c = 0; c < 2; ++c)
          *reinterpret_cast<uint4*>(prow + (((2 * half + c) ^ sw) << 4)) =
              make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
      } else {  // P row: [p*m_lo slots 0-31 | p*m_hi slots 0-31] as fp16, chunks 0-3 | 4-7
        const float* ml = reinterpret_cast<const float*>(meta) + 2 * TN + cb;  // m_lo of the slots
        const float* mh = ml + TN;                                               // m_hi
        uint32_t plo[TH / 2], phi[TH / 2];
#pragma unroll
        for (int i = 0; i < TH / 4; ++i) {
          const float4 a = reinterpret_cast<const float4*>(ml)[i];
          const float4 b = reinterpret_cast<const float4*>(mh)[i];
          plo[2 * i] = pack_f16x2(pr[4 * i] * a.x, pr[4 * i + 1] * a.y);
          plo[2 * i + 1] = pack_f16x2(pr[4 * i + 2] * a.z, pr[4 * i + 3] * a.w);
          phi[2 * i] = pack_f16x2(pr[4 * i] * b.x, pr[4 * i + 1] * b.y);
          phi[2 * i + 1] = pack_f16x2(pr[4 * i + 2] * b.z, pr[4 * i + 3] * b.w);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          *reinterpret_cast<uint4*>(prow + (((2 * half + c) ^ sw) << 4)) =
              make_uint4(plo[4 * c], plo[4 * c + 1], plo[4 * c + 2], plo[4 * c + 3]);
          *reinterpret_cast<uint4*>(prow + (((4 + 2 * half + c) ^ sw) << 4)) =
              make_uint4(phi[4 * c], phi[4 * c + 1], phi[4 * c + 2], phi[4 * c + 3]);
        }
      }
      fence_proxy_async_smem();        // P is read by the tensor pipe
      if (rescale) tmem_st_wait();     // (the O rescale must land before P.V(j) accumulates)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.p_full[j & 1]);
      if (w.last()) {
        finish_unit(j, from_start);
        if (!ok) break;
        m_ref = -INFINITY;
        lsum = 0.f;
        from_start = true;
        slot_idx = 1;
        U0 = t0 + j + 1;
      }
      w.next(p);
    }
    // the range ended inside a unit (Walk.next does not move past the last tile):
    // publish that unit's partial
    if (ok && j == ntiles && ntiles > 0 && w.lt != w.info.ntile - 1) finish_unit(ntiles - 1, false);
    if (!FUSED && lane == 0) bulk_wait0();  // this warp's tiled stores complete
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && sh.abort_flag) {
    // an aborted CTA may still have gathers in flight into its staging ring: wait for the
    // last one issued into each slot (nothing is issued into a slot before the previous
    // gather there has landed, so only that one can be pending)
    volatile int no_abort = 0;
    for (int i = 0; i < NS; ++i)
      if (sh.stg_issued[i] > 0) mbar_wait(&sh.stg_full[i], (sh.stg_issued[i] - 1) & 1, &no_abort);
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  if (tid == 0 && sh.abort_flag && p.err_timeout) atomicOr(p.err_timeout, DCP_ERRBIT_TIMEOUT);
  cluster_sync();
}

// ------------------------------------------------------------------ host side
static size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t tc_desc_bytes(int pairs);

size_t tc_workspace_bytes(int64_t units, int pairs) {
  (void)units;
  return a256((size_t)pairs * 2 * 128 * kDv * sizeof(float)) +
         a256((size_t)pairs * 2 * 2 * 128 * sizeof(float)) + a256(tc_desc_bytes(pairs));
}

void tc_bind_workspace(DecodeParams& p, void* ws) {
  char* b = static_cast<char*>(ws);
  const size_t o = a256((size_t)p.pairs * 2 * 128 * kDv * sizeof(float));
  const size_t l = a256((size_t)p.pairs * 2 * 2 * 128 * sizeof(float));
  p.tc_o = reinterpret_cast<float*>(b);
  p.tc_l = reinterpret_cast<float*>(b + o);
  p.tc_desc = reinterpret_cast<int64_t*>(b + o + l);
}

// Tile-sequence header (T, pairs owning tiles) and one descriptor (unit, first tile, end
// tile) per (pair, slot), all written by every decode launch (an unused descriptor gets end
// tile 0), so nothing needs clearing between calls.
size_t tc_desc_bytes(int pairs) { return (2 + (size_t)pairs * 2 * 3) * sizeof(int64_t); }

// Merges the parts of units that several pairs' ranges cut.  One CTA per (descriptor,
// CTA half, 16-column chunk) and one thread per head: a descriptor is merged by its pair
// when that pair is the unit's first covering pair (exactly one per split unit).  Part q
// holds the unit in workspace slot 0 when its range starts inside the unit, else in slot 1.
template <bool FUSED>
__global__ void __launch_bounds__(128) tc_split_merge_kernel(const DecodeParams p) {
  const int64_t dix = blockIdx.x >> 5;
  const int half = (blockIdx.x >> 4) & 1, chunk = blockIdx.x & 15;
  const int h = threadIdx.x;
  const int64_t* d = p.tc_desc + 2 + dix * 3;
  const int64_t U1 = d[2];
  if (U1 == 0) return;  // no split unit published here
  const int64_t u = d[0], U0 = d[1];
  const int64_t T = p.tc_desc[0], Pe = p.tc_desc[1];
  const int64_t pf = min(Pe - 1, ((U0 + 1) * Pe - 1) / T);
  const int64_t pl = min(Pe - 1, (U1 * Pe - 1) / T);
  if ((dix >> 1) != pf) return;
  const int H = p.heads;
  float mx = -INFINITY;
  for (int64_t q = pf; q <= pl; ++q) {
    const int sq = (q * T / Pe) >= U0 ? 0 : 1;
    mx = fmaxf(mx, __ldcg(p.tc_l + ((q * 2 + sq) * 2 + half) * 128 + h));
  }
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  float W = 0.f;
  if (mx != -INFINITY) {
    for (int64_t q = pf; q <= pl; ++q) {
      const int sq = (q * T / Pe) >= U0 ? 0 : 1;
      const float lq = __ldcg(p.tc_l + ((q * 2 + sq) * 2 + half) * 128 + h);
      const float wq = fast_exp2((lq - mx) * kLog2e);
      W += wq;
      const float4* src = reinterpret_cast<const float4*>(
          p.tc_o + ((q * 2 + sq) * 128 + h) * kDv + half * 256 + 16 * chunk);
      float4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = __ldcg(src + i);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[4 * i] = fmaf(wq, v[i].x, acc[4 * i]);
        acc[4 * i + 1] = fmaf(wq, v[i].y, acc[4 * i + 1]);
        acc[4 * i + 2] = fmaf(wq, v[i].z, acc[4 * i + 2]);
        acc[4 * i + 3] = fmaf(wq, v[i].w, acc[4 * i + 3]);
      }
    }
  }
  if (h >= H) return;
  const float iw = W > 0.f ? 1.0f / W : 0.f;
  const int64_t oi = (u * H + h) * kDv + half * 256 + 16 * chunk;
  if (FUSED) {
    uint32_t b2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b2[i] = pack_bf16x2(acc[2 * i] * iw, acc[2 * i + 1] * iw);
    uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + oi);
    o[0] = make_uint4(b2[0], b2[1], b2[2], b2[3]);
    o[1] = make_uint4(b2[4], b2[5], b2[6], b2[7]);
  } else {
    float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + oi);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = make_float4(acc[4 * i] * iw, acc[4 * i + 1] * iw, acc[4 * i + 2] * iw, acc[4 * i + 3] * iw);
  }
  if (half == 0 && chunk == 0)
    p.lse[u * H + h] = mx == -INFINITY ? -INFINITY : mx + __log2f(W) * kLn2;
}

int tc_pairs_for(int64_t units, int64_t tiles_bound) {
  const int sms = device_sm_count();
  // at least kMinTilesPerPair tiles per pair: a pair's set-up and pipeline fill cost about as
  // much as a dozen tiles, and a row cut between pairs adds a split merge (on 16 rows of 16
  // tiles, 76 pairs of ~3 tiles take 44 us a call, 16 pairs of one row each 31 us)
  int64_t pairs = sms / 2;
  const int64_t want = (tiles_bound + kMinTilesPerPair - 1) / kMinTilesPerPair;
  if (want < pairs) pairs = want > 0 ? want : 1;
  (void)units;
  return (int)pairs;
}

int tc_tile_slots(int kv_dtype) {
  (void)kv_dtype;
  return kTN;
}

// The pool as a 2-D tensor [num_pages * 64 rows][row elements] for the 4-row gathers:
// FP8 rows as 656 bytes (latent box 256 B, tail box 144 B from byte 512), BF16 rows as 576
// bf16 (latent box 256 elements, RoPE box 32 elements).  No L2 promotion: rows are 656 /
// 1152 B apart, so promoting a box to 256-B lines would fetch bytes no box asks for.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

static cudaError_t make_pool_maps(const DecodeParams& p, int kv_dtype, CUtensorMap* lat,
                                  CUtensorMap* tail) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const bool bf = kv_dtype == DCP_KV_BF16;
  const CUtensorMapDataType dt = bf ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const cuuint64_t dims[2] = {bf ? 576ull : 656ull, (cuuint64_t)p.num_pages * 64};
  const cuuint64_t strides[1] = {bf ? 1152ull : 656ull};
  const cuuint32_t box_lat[2] = {256, 1};
  const cuuint32_t box_tail[2] = {bf ? 32u : 144u, 1};
  const cuuint32_t es[2] = {1, 1};
  void* base = const_cast<uint8_t*>(p.pool);
  if (enc(lat, dt, 2, base, dims, strides, box_lat, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (enc(tail, dt, 2, base, dims, strides, box_tail, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

// The partial form's output as a 3-D tensor [units][heads][512] fp32 with 32 x 32 boxes in the
// 128-B swizzle; only for a 16-B aligned output (else the kernel stores rows itself).
static bool make_out_map(const DecodeParams& p, CUtensorMap* out) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr || (reinterpret_cast<uintptr_t>(p.out) & 15) != 0 || p.num_units < 1)
    return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kDv, (cuuint64_t)p.heads, (cuuint64_t)p.num_units};
  const cuuint64_t strides[2] = {(cuuint64_t)kDv * 4, (cuuint64_t)p.heads * kDv * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.out, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KVT, bool FUSED, bool SPARSE>
static cudaError_t tc_launch_one(const DecodeParams& p0, cudaStream_t st) {
  auto kern = decode_tc_kernel<KVT, FUSED, SPARSE>;
  const int smem = TcLay<KVT>::SMEM;
  cudaError_t e = raise_smem_limit((const void*)kern, smem);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap lat, tail, outm;
  e = make_pool_maps(p0, KVT, &lat, &tail);
  if (e != cudaSuccess) return e;
  DecodeParams p = p0;
  memset(&outm, 0, sizeof(outm));
  p.tma_out = !FUSED && make_out_map(p, &outm) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.pairs, 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, p, lat, tail, outm);
  if (e != cudaSuccess || p.pairs < 2) return e;
  tc_split_merge_kernel<FUSED><<<p.pairs * 2 * 32, 128, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_tc(const DecodeParams& p, int kv_dtype, bool fused, bool sparse,
                             cudaStream_t st) {
  if (kv_dtype == DCP_KV_BF16) {
    if (fused) return sparse ? tc_launch_one<DCP_KV_BF16, true, true>(p, st)
                             : tc_launch_one<DCP_KV_BF16, true, false>(p, st);
    return sparse ? tc_launch_one<DCP_KV_BF16, false, true>(p, st)
                  : tc_launch_one<DCP_KV_BF16, false, false>(p, st);
  }
  if (fused) return sparse ? tc_launch_one<DCP_KV_FP8_E4M3_S128, true, true>(p, st)
                           : tc_launch_one<DCP_KV_FP8_E4M3_S128, true, false>(p, st);
  return sparse ? tc_launch_one<DCP_KV_FP8_E4M3_S128, false, true>(p, st)
                : tc_launch_one<DCP_KV_FP8_E4M3_S128, false, false>(p, st);
}

}  // namespace dcp

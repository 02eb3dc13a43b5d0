// DCP KV-cache write: new token rows into the paged pool of their owner shard, FP8 pools
// quantised per 128 latent values (LMDeploy PR #4952 "support decode context parallelism
// for PyTorch MLA", files: "Interleaved DCP KV-cache writes"; SGLang PR #36990 "DCP for
// DSA models with the flashmla_kv backend", review of quantize_k_cache_separate: the
// latent and RoPE parts are quantised separately).
//
// One warp per token row.  FP8: lane l holds latent values [16l, 16l+16); the 8 lanes of a
// 128-value block reduce its amax, scale = amax / 448 (IEEE fp32 division), every value is
// divided by the scale and rounded to nearest-even E4M3 with saturation at 448 by the
// hardware conversion; an all-zero block stores scale 0 and zero codes.  RoPE (64 bf16) is
// copied.  BF16: the 1152-byte row is copied.  HBM-bound: 1152 B read and 656 / 1152 B
// written per row.  A warp loads its next row (data, position, sequence) before it
// resolves and writes the current one, so two rows' loads are in flight per warp.
//
// The quotients.  With r = 1 / scale correctly rounded, q0 = v * r lies within one ulp of
// v / scale; the residual e = q0 * scale - v is exact in one fused multiply-add, and
// q = q0 - e * r (one more fused multiply-add) is the correctly rounded quotient v / scale
// (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990: the correction step with a correctly rounded
// reciprocal).  The theorem needs normal operands: a block whose scale lies outside
// [2^-100, FLT_MAX] takes IEEE divisions instead.  So the codes are those of the IEEE
// quotients, with three floating-point operations per value and no branch.
#include "common.cuh"
#include "internal.h"

namespace dcp {

constexpr int kKvwThreads = 256;
constexpr int kKvwRowsPerCta = kKvwThreads / 32;

// Two fp32 -> two E4M3 codes (round to nearest even, saturating), lo in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Largest of two bf16 pairs, lane by lane; a NaN never wins over a number (max.bf16x2
// returns the non-NaN operand), as with a float comparison.
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// v / scale correctly rounded, from r = 1 / scale correctly rounded (Markstein correction).
// The residual is taken as q0 * scale - v and subtracted, so that v = -0 gives -0, as the
// IEEE quotient does (the sign of a zero decides its E4M3 code).
__device__ __forceinline__ float quotient_rn(float v, float scale, float r) {
  const float q0 = v * r;
  const float e = fmaf(q0, scale, -v);
  return fmaf(-e, r, q0);
}

// This warp's share of one token row: 16 B loads at the offsets the writer uses.
template <int KVT>
__device__ __forceinline__ void load_row(const uint4* __restrict__ kv, int64_t i, int lane,
                                         uint4& d0, uint4& d1, uint4& d2) {
  const uint4* src = kv + i * (kDqk * 2 / 16);  // 72 chunks of 16 B
  d2 = make_uint4(0u, 0u, 0u, 0u);
  if (KVT == DCP_KV_BF16) {
    d0 = __ldg(src + lane);
    d1 = __ldg(src + 32 + lane);
  } else {
    d0 = __ldg(src + 2 * lane);
    d1 = __ldg(src + 2 * lane + 1);
  }
  if (lane < 8) d2 = __ldg(src + 64 + lane);  // RoPE (BF16: the row's last 128 B)
}

// Resolve where token t of sequence b goes and write it there (FP8: quantised).
template <int KVT>
__device__ __forceinline__ void write_row(const uint4& d0, const uint4& d1, const uint4& d2,
                                          int t, int b, int lane, const OwnerRule& rule,
                                          int shard, uint8_t* pool, int64_t num_pages,
                                          const int32_t* __restrict__ bt, int num_seqs,
                                          int bt_stride, int32_t* err) {
  if (t < 0) return;  // padding
  if (b < 0 || b >= num_seqs) {
    if (lane == 0) set_err(err, DCP_ERRBIT_SLOT_RANGE);
    return;
  }
  int s, l;
  owner_local(t, rule, s, l);
  if (shard >= 0 && s != shard) return;
  const int pj = l >> 6;  // page size 64
  if (pj >= bt_stride) {
    if (lane == 0) set_err(err, DCP_ERRBIT_SLOT_RANGE);
    return;
  }
  const int page = __ldg(bt + ((int64_t)s * num_seqs + b) * bt_stride + pj);
  if (page < 0 || page >= num_pages) {
    if (lane == 0) set_err(err, DCP_ERRBIT_PAGE_RANGE);
    return;
  }
  if (KVT == DCP_KV_BF16) {
    uint4* dst = reinterpret_cast<uint4*>(pool + ((int64_t)page * 64 + (l & 63)) * kTokBytesBF16);
    dst[lane] = d0;
    dst[32 + lane] = d1;
    if (lane < 8) dst[64 + lane] = d2;
    return;
  }
  const uint32_t w[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
  uint8_t* row = pool + ((int64_t)page * 64 + (l & 63)) * kTokBytesFP8;
  // the block's largest magnitude: packed bf16 maxima of the magnitudes
  uint32_t mx = 0u;
#pragma unroll
  for (int e = 0; e < 8; ++e) mx = bf16x2_max(mx, w[e] & 0x7fff7fffu);
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) mx = bf16x2_max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float amax = fmaxf(bf16_lo(mx), bf16_hi(mx));
  const float scale = amax / 448.0f;
  float qv[16];
  if (scale >= 0x1p-100f && scale <= 3.40282347e38f) {
    const float r = 1.0f / scale;  // correctly rounded
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      qv[2 * e] = quotient_rn(bf16_lo(w[e]), scale, r);
      qv[2 * e + 1] = quotient_rn(bf16_hi(w[e]), scale, r);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      qv[2 * e] = scale > 0.f ? bf16_lo(w[e]) / scale : 0.f;
      qv[2 * e + 1] = scale > 0.f ? bf16_hi(w[e]) / scale : 0.f;
    }
  }
  uint32_t q[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    q[e] = f32x2_to_e4m3x2(qv[4 * e], qv[4 * e + 1]) |
           (f32x2_to_e4m3x2(qv[4 * e + 2], qv[4 * e + 3]) << 16);
  *reinterpret_cast<uint4*>(row + 16 * lane) = make_uint4(q[0], q[1], q[2], q[3]);
  if ((lane & 7) == 0) *reinterpret_cast<float*>(row + 512 + 4 * (lane >> 3)) = scale;
  if (lane < 8) *reinterpret_cast<uint4*>(row + 528 + 16 * lane) = d2;
}

// A warp's rows are i0, i0 + stride, ...; the next row's data, position and sequence are
// loaded before the current row is resolved and written, so two rows' loads are in flight.
template <int KVT>
__global__ void __launch_bounds__(kKvwThreads)
kv_write_kernel(const uint4* __restrict__ kv, int64_t n, const int32_t* __restrict__ seq,
                const int32_t* __restrict__ pos, const OwnerRule rule, int shard, uint8_t* pool,
                int64_t num_pages, const int32_t* __restrict__ bt, int num_seqs, int bt_stride,
                int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kKvwRowsPerCta;
  const int64_t i0 = (int64_t)blockIdx.x * kKvwRowsPerCta + (threadIdx.x >> 5);
  if (i0 >= n) return;
  uint4 d0, d1, d2;
  load_row<KVT>(kv, i0, lane, d0, d1, d2);
  int t = __ldg(pos + i0), b = __ldg(seq + i0);
  for (int64_t i = i0; i < n; i += stride) {
    const int64_t j = i + stride;
    uint4 e0 = d0, e1 = d1, e2 = d2;
    int tn = -1, bn = -1;
    if (j < n) {
      load_row<KVT>(kv, j, lane, e0, e1, e2);
      tn = __ldg(pos + j);
      bn = __ldg(seq + j);
    }
    write_row<KVT>(d0, d1, d2, t, b, lane, rule, shard, pool, num_pages, bt, num_seqs,
                   bt_stride, err);
    d0 = e0;
    d1 = e1;
    d2 = e2;
    t = tn;
    b = bn;
  }
}

cudaError_t launch_kv_write(const void* kv, int64_t n, const int32_t* seq, const int32_t* pos,
                            int D, int I, int shard, void* pool, int64_t num_pages, int kv_dtype,
                            const int32_t* bt, int num_seqs, int bt_stride, int32_t* err,
                            cudaStream_t st) {
  const int sms = device_sm_count();
  const int64_t need = (n + kKvwRowsPerCta - 1) / kKvwRowsPerCta;
  const int grid = (int)(need < (int64_t)sms * 16 ? need : (int64_t)sms * 16);
  const uint4* k4 = static_cast<const uint4*>(kv);
  uint8_t* p8 = static_cast<uint8_t*>(pool);
  const OwnerRule rule = make_owner_rule(D, I);
  if (kv_dtype == DCP_KV_BF16)
    kv_write_kernel<DCP_KV_BF16><<<grid, kKvwThreads, 0, st>>>(k4, n, seq, pos, rule, shard, p8,
                                                               num_pages, bt, num_seqs, bt_stride, err);
  else
    kv_write_kernel<DCP_KV_FP8_E4M3_S128><<<grid, kKvwThreads, 0, st>>>(
        k4, n, seq, pos, rule, shard, p8, num_pages, bt, num_seqs, bt_stride, err);
  return cudaGetLastError();
}

}  // namespace dcp

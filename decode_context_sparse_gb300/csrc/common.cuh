// Shared device helpers of the DCP MLA decode library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dcpmla.h"

namespace dcp {

constexpr int kDqk = 576;      // latent 512 + RoPE 64
constexpr int kDv = 512;       // value = first 512 latent dims
constexpr int kTokBytesBF16 = 1152;
constexpr int kTokBytesFP8 = 656;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Exact n / d for 0 <= n < 2^31 and 1 <= d < 2^31 without a division instruction:
// (n * m) >> s with s = 32 + ceil(log2 d) and m = ceil(2^s / d).  The error term
// n (m - 2^s / d) / 2^s is below 2^31 / 2^s <= 1 / (2d), so it never carries the quotient
// past the next integer; n * m < 2^64.
struct FastDiv {
  uint64_t m;
  int s, d;
};
__host__ inline FastDiv make_fastdiv(int d) {
  int l = 0;
  while ((1ll << l) < (long long)d) ++l;
  FastDiv f;
  f.d = d;
  f.s = 32 + l;
  f.m = ((1ull << f.s) + (uint64_t)d - 1ull) / (uint64_t)d;
  return f;
}
__device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
  return (int)(((uint64_t)(uint32_t)n * f.m) >> f.s);
}

// Owner rule of D shards with interleave I: global slot t lives on shard (t / I) mod D at
// local slot (t / (I D)) I + t mod I.  Both from two divisions: q1 = t / I, q2 = t / (I D)
// = q1 / D, so the shard is q1 - D q2 and t mod I = t - I q1.
struct OwnerRule {
  FastDiv I, ID;
  int D;
};
__host__ inline OwnerRule make_owner_rule(int D, int I) {
  OwnerRule r;
  r.I = make_fastdiv(I);
  r.ID = make_fastdiv(I * D);
  r.D = D;
  return r;
}
__device__ __forceinline__ int owner_of(int t, const OwnerRule& r) {
  return fdiv(t, r.I) - r.D * fdiv(t, r.ID);
}
__device__ __forceinline__ void owner_local(int t, const OwnerRule& r, int& s, int& l) {
  const int q1 = fdiv(t, r.I), q2 = fdiv(t, r.ID);
  s = q1 - r.D * q2;
  l = q2 * r.I.d + (t - q1 * r.I.d);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two E4M3 codes (low 16 bits of w) -> two floats, exact.  The hardware conversion goes
// to f16x2, which holds every E4M3 value exactly.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t w) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(w));
  __half2 hh = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hh);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void set_err(int32_t* err, int bit) {
  if (err) atomicOr(err, bit);
}

}  // namespace dcp

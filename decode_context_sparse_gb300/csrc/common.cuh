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

// Owner rule: global slot t -> (shard, local slot).  I = interleave, D = shards.
__device__ __forceinline__ int owner_of(int t, int D, int I) { return (t / I) % D; }
__device__ __forceinline__ int local_of(int t, int D, int I) {
  return (t / (I * D)) * I + (t % I);
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

// LSE merge of DCP shard partials (HBM-bound streaming kernel).
//
// LMDeploy PR #4952 "support decode context parallelism for PyTorch MLA", Summary: merge
// outputs using LSE weights; its review discussion fixes the precision (FP32 arithmetic,
// BF16 storage of the merged output).  All-empty rows (every shard at LSE = -inf) give a
// zero output and -inf LSE (SGLang PR #36990 review of the LSE combine; SGLang PR #42536,
// Fixes in shared code).
//
// One warp per (row, head): lanes stream the dv-wide partial rows of every shard with
// 16-byte non-allocating loads, the weights are computed once per warp, and the merged row
// is written as BF16 with 8-byte stores.  The partials are read exactly once.
#include "common.cuh"
#include "internal.h"

namespace dcp {

constexpr int kMergeWarps = 8;

// Read-once partials: streaming (evict-first) load.
__device__ __forceinline__ float4 ld_stream(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}

// CHUNKS: float4 chunks per lane (dv = 128 * CHUNKS) or 0 for any dv;
// DT: shard count known at compile time (all loads of a row issued together) or 0.
template <int CHUNKS, int DT>
__global__ void __launch_bounds__(kMergeWarps * 32)
lse_merge_kernel(const float* __restrict__ part_out, const float* __restrict__ part_lse, int D,
                 int64_t RH, int dv, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  if (DT > 0) D = DT;
  __shared__ float wsm[kMergeWarps][DCP_MAX_SHARDS];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i = blockIdx.x * (int64_t)kMergeWarps + warp;
  if (i >= RH) return;
  // lane s holds shard s and shard s + 32
  const float l0 = lane < D ? __ldg(part_lse + (int64_t)lane * RH + i) : -INFINITY;
  const float l1 = lane + 32 < D ? __ldg(part_lse + (int64_t)(lane + 32) * RH + i) : -INFINITY;
  const float m = warp_max(fmaxf(l0, l1));
  __nv_bfloat16* o = out + i * dv;
  const int nchunk = dv / 4;
  if (m == -INFINITY) {  // every shard empty: zero output, -inf LSE
    for (int c = lane; c < nchunk; c += 32)
      *reinterpret_cast<uint2*>(o + 4 * c) = make_uint2(0u, 0u);
    if (lane == 0) lse[i] = -INFINITY;
    return;
  }
  const float w0 = fast_exp2((l0 - m) * kLog2e), w1 = fast_exp2((l1 - m) * kLog2e);
  const float W = warp_sum(w0 + w1);
  const float invW = 1.0f / W;
  wsm[warp][lane] = w0 * invW;
  wsm[warp][lane + 32] = w1 * invW;
  __syncwarp();
  constexpr int NC = CHUNKS > 0 ? CHUNKS : 1;
  const int nfull = CHUNKS > 0 ? 1 : (nchunk + 32 * NC - 1) / (32 * NC);
  for (int rep = 0; rep < nfull; ++rep) {
    float4 acc[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (DT > 0 && CHUNKS > 0) {
      // all shards' loads in flight at once
      float4 v[DT > 0 ? DT : 1][NC];
#pragma unroll
      for (int s = 0; s < (DT > 0 ? DT : 1); ++s) {
        const float* src = part_out + ((int64_t)s * RH + i) * dv;
        const bool live = wsm[warp][s] != 0.0f;  // empty shard contributes nothing
#pragma unroll
        for (int j = 0; j < NC; ++j)
          v[s][j] = live ? ld_stream(src + 4 * (j * 32 + lane)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int s = 0; s < (DT > 0 ? DT : 1); ++s) {
        const float ws = wsm[warp][s];
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          acc[j].x = fmaf(ws, v[s][j].x, acc[j].x);
          acc[j].y = fmaf(ws, v[s][j].y, acc[j].y);
          acc[j].z = fmaf(ws, v[s][j].z, acc[j].z);
          acc[j].w = fmaf(ws, v[s][j].w, acc[j].w);
        }
      }
    } else {
      for (int s = 0; s < D; ++s) {
        const float ws = wsm[warp][s];
        if (ws == 0.0f) continue;  // empty shard contributes nothing
        const float* src = part_out + ((int64_t)s * RH + i) * dv;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          const int c = (rep * NC + j) * 32 + lane;
          if (CHUNKS == 0 && c >= nchunk) continue;
          const float4 v = ld_stream(src + 4 * c);
          acc[j].x = fmaf(ws, v.x, acc[j].x);
          acc[j].y = fmaf(ws, v.y, acc[j].y);
          acc[j].z = fmaf(ws, v.z, acc[j].z);
          acc[j].w = fmaf(ws, v.w, acc[j].w);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int c = (rep * NC + j) * 32 + lane;
      if (CHUNKS == 0 && c >= nchunk) continue;
      __nv_bfloat162 a = __floats2bfloat162_rn(acc[j].x, acc[j].y);
      __nv_bfloat162 b = __floats2bfloat162_rn(acc[j].z, acc[j].w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&a);
      u.y = *reinterpret_cast<uint32_t*>(&b);
      *reinterpret_cast<uint2*>(o + 4 * c) = u;
    }
  }
  if (lane == 0) lse[i] = m + __log2f(W) * kLn2;
}

cudaError_t launch_lse_merge(const float* part_out, const float* part_lse, int D, int64_t rows,
                             int heads, int dv, void* out, float* lse, cudaStream_t st) {
  const int64_t RH = rows * heads;
  if (RH == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((RH + kMergeWarps - 1) / kMergeWarps);
  auto* o = reinterpret_cast<__nv_bfloat16*>(out);
  const dim3 blk(kMergeWarps * 32);
  if (dv == 512 && D == 2)
    lse_merge_kernel<4, 2><<<grid, blk, 0, st>>>(part_out, part_lse, D, RH, dv, o, lse);
  else if (dv == 512 && D == 4)
    lse_merge_kernel<4, 4><<<grid, blk, 0, st>>>(part_out, part_lse, D, RH, dv, o, lse);
  else if (dv == 512 && D == 8)
    lse_merge_kernel<4, 8><<<grid, blk, 0, st>>>(part_out, part_lse, D, RH, dv, o, lse);
  else if (dv == 512)
    lse_merge_kernel<4, 0><<<grid, blk, 0, st>>>(part_out, part_lse, D, RH, dv, o, lse);
  else
    lse_merge_kernel<0, 0><<<grid, blk, 0, st>>>(part_out, part_lse, D, RH, dv, o, lse);
  return cudaGetLastError();
}

}  // namespace dcp

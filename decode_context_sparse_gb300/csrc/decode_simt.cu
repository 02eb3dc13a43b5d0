// SIMT (CUDA-core) MLA decode attention with LSE over paged latent KV: the partial
// (one or more shards, local slot ids) and the fused (all shards, global slot ids)
// forms.  Any head count that is a multiple of 16; BF16 or FP8-E4M3/per-128-scale KV.
//
// What it computes (LMDeploy PR #4952 "support decode context parallelism for PyTorch
// MLA", Summary; SGLang PR #42536 "Fix DCP for RoPE sparse attention on Blackwell",
// Modifications, "Backend" and Follow-ups #1):
//   logit_t = sm_scale * q.key_t,  lse = ln sum exp(logit_t),  out = softmax . key[:512];
//   a row with no KV gives out = 0, lse = -inf.
//
// Layout of the work: CTA = (unit, split, group of 16 heads); 8 warps, warp w owns heads
// 2w and 2w+1 of the group.  Tiles of 32 slots are gathered into shared memory as fp32
// (BF16 widened, FP8 decoded exactly with the hardware E4M3->F16 conversion and scaled
// in fp32); lane j scores slot j of the tile for both heads, the online softmax runs in
// base 2 with warp reductions, and lane l accumulates value dims 4l..4l+3 (+128 i).
// Splits of a row are merged by the last CTA to finish, found with an atomic ticket.
#include "common.cuh"
#include "internal.h"

namespace dcp {

constexpr int kSimtThreads = 256;
constexpr int kTile = 32;
constexpr int kKStride = 580;  // fp32 row stride of the K tile: float4 reads conflict-free
constexpr int kHG = kSimtHeadGroup;

// Resolve position `pos` of unit (row r, shard s) to a pool row; NULL when it is padding
// or out of range (reported through err when given).
template <bool FUSED, bool SPARSE>
__device__ __forceinline__ const uint8_t* resolve_slot(const DecodeParams& p, int pos, int n,
                                                       const int32_t* idx_row, const int32_t* bt_s,
                                                       int b, int tok_bytes) {
  if (pos >= n) return nullptr;
  int l;
  const int32_t* table = bt_s;
  if (FUSED) {
    const int t = SPARSE ? __ldg(idx_row + pos) : pos;
    if (t < 0) return nullptr;
    int s;
    owner_local(t, p.rule, s, l);
    table = p.bt + (int64_t)s * p.num_seqs * p.bt_stride;
  } else {
    l = SPARSE ? __ldg(idx_row + pos) : pos;
    if (l < 0) {
      set_err(p.err, DCP_ERRBIT_SLOT_RANGE);
      return nullptr;
    }
  }
  const int pj = l / p.page_size;
  if (pj >= p.bt_stride) {
    set_err(p.err, DCP_ERRBIT_SLOT_RANGE);
    return nullptr;
  }
  const int page = __ldg(table + (int64_t)b * p.bt_stride + pj);
  if (page < 0 || page >= p.num_pages) {
    set_err(p.err, DCP_ERRBIT_PAGE_RANGE);
    return nullptr;
  }
  return p.pool + ((int64_t)page * p.page_size + (l - pj * p.page_size)) * tok_bytes;
}

template <int KVT, bool FUSED, bool SPARSE>
__global__ void __launch_bounds__(kSimtThreads)
decode_simt_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) float smem[];
  float* sQ = smem;                         // [16][576] q * scale_log2
  float* sK = sQ + kHG * kDqk;              // [32][580]
  __shared__ const uint8_t* sRow[kTile];
  __shared__ int sLast;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t unit = blockIdx.x;
  const int split = blockIdx.y, hg = blockIdx.z;
  const int H = p.heads;
  constexpr int tok_bytes = KVT == DCP_KV_BF16 ? kTokBytesBF16 : kTokBytesFP8;

  const int64_t r = FUSED ? unit : unit % p.rows;
  const int64_t shard = FUSED ? 0 : unit / p.rows;
  int b = __ldg(p.row_seq + r);
  bool row_ok = b >= 0 && b < p.num_seqs;
  if (!row_ok) set_err(p.err, DCP_ERRBIT_SLOT_RANGE);
  const int32_t* bt_s = p.bt + shard * p.num_seqs * p.bt_stride;
  const int32_t* idx_row = nullptr;
  int n;
  if (SPARSE) {
    idx_row = p.idx + unit * (int64_t)p.k;
    n = FUSED ? p.k : min(__ldg(p.count + unit), p.k);
  } else {
    n = max(0, __ldg(p.kv_len + unit));
  }
  if (!row_ok) n = 0;
  // contiguous chunk of positions for this split (multiple of the tile)
  int chunk = (n + p.num_splits - 1) / p.num_splits;
  chunk = (chunk + kTile - 1) / kTile * kTile;
  const int beg = min(n, split * chunk), end = min(n, beg + chunk);

  // Q of this head group, pre-scaled to base-2 logits
  const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(p.q) +
                            (r * H + (int64_t)hg * kHG) * kDqk;
  for (int i = tid; i < kHG * kDqk / 2; i += kSimtThreads) {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(qg) + i);
    sQ[2 * i] = bf16_lo(w) * p.scale_log2;
    sQ[2 * i + 1] = bf16_hi(w) * p.scale_log2;
  }

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float4 acc[2][4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[h][c] = make_float4(0.f, 0.f, 0.f, 0.f);

  for (int pos0 = beg; pos0 < end; pos0 += kTile) {
    __syncthreads();  // previous tile consumed (and sQ written on the first pass)
    if (tid < kTile)
      sRow[tid] = resolve_slot<FUSED, SPARSE>(p, pos0 + tid, end, idx_row, bt_s, b, tok_bytes);
    __syncthreads();
    {  // gather: 8 threads per slot
      const int j = tid >> 3, part = tid & 7;
      const uint8_t* src = sRow[j];
      float* dst = sK + j * kKStride;
      if (src == nullptr) {
        for (int d = part * 4; d < kKStride; d += 32)
          *reinterpret_cast<float4*>(dst + d) = make_float4(0.f, 0.f, 0.f, 0.f);
      } else if (KVT == DCP_KV_BF16) {
        uint4 v[9];
#pragma unroll
        for (int c = 0; c < 9; ++c) v[c] = __ldg(reinterpret_cast<const uint4*>(src) + part + 8 * c);
#pragma unroll
        for (int c = 0; c < 9; ++c) {
          const int d = (part + 8 * c) * 8;
          *reinterpret_cast<float4*>(dst + d) =
              make_float4(bf16_lo(v[c].x), bf16_hi(v[c].x), bf16_lo(v[c].y), bf16_hi(v[c].y));
          *reinterpret_cast<float4*>(dst + d + 4) =
              make_float4(bf16_lo(v[c].z), bf16_hi(v[c].z), bf16_lo(v[c].w), bf16_hi(v[c].w));
        }
      } else {
        uint4 v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = __ldg(reinterpret_cast<const uint4*>(src) + part + 8 * c);
        const float4 sc = __ldg(reinterpret_cast<const float4*>(src + 512));
        const uint4 rp = __ldg(reinterpret_cast<const uint4*>(src + 528) + part);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int ch = part + 8 * c;        // 16 codes: dims 16ch .. 16ch+15
          const int blk = ch >> 3;            // 128-value scale block
          const float s = blk == 0 ? sc.x : blk == 1 ? sc.y : blk == 2 ? sc.z : sc.w;
          const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 lo = e4m3x2_to_float2((uint16_t)(w[e] & 0xffffu));
            const float2 hi = e4m3x2_to_float2((uint16_t)(w[e] >> 16));
            *reinterpret_cast<float4*>(dst + ch * 16 + e * 4) =
                make_float4(lo.x * s, lo.y * s, hi.x * s, hi.y * s);
          }
        }
        const int d = 512 + part * 8;
        *reinterpret_cast<float4*>(dst + d) =
            make_float4(bf16_lo(rp.x), bf16_hi(rp.x), bf16_lo(rp.y), bf16_hi(rp.y));
        *reinterpret_cast<float4*>(dst + d + 4) =
            make_float4(bf16_lo(rp.z), bf16_hi(rp.z), bf16_lo(rp.w), bf16_hi(rp.w));
      }
    }
    __syncthreads();

    // scores: lane j = slot j of the tile, two heads per warp
    const bool valid = sRow[lane] != nullptr;
    float s0 = 0.f, s1 = 0.f;
    {
      const float* kr = sK + lane * kKStride;
      const float* q0 = sQ + (2 * warp) * kDqk;
      const float* q1 = q0 + kDqk;
#pragma unroll 4
      for (int d = 0; d < kDqk; d += 4) {
        const float4 kv = *reinterpret_cast<const float4*>(kr + d);
        const float4 a = *reinterpret_cast<const float4*>(q0 + d);
        const float4 c = *reinterpret_cast<const float4*>(q1 + d);
        s0 = fmaf(a.x, kv.x, s0); s0 = fmaf(a.y, kv.y, s0);
        s0 = fmaf(a.z, kv.z, s0); s0 = fmaf(a.w, kv.w, s0);
        s1 = fmaf(c.x, kv.x, s1); s1 = fmaf(c.y, kv.y, s1);
        s1 = fmaf(c.z, kv.z, s1); s1 = fmaf(c.w, kv.w, s1);
      }
    }
    float pr[2];
    const float sv[2] = {valid ? s0 : -INFINITY, valid ? s1 : -INFINITY};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mt = warp_max(sv[h]);
      const float mn = fmaxf(m[h], mt);
      if (mn == -INFINITY) {  // nothing valid yet
        pr[h] = 0.f;
        continue;
      }
      const float alpha = fast_exp2(m[h] - mn);
      pr[h] = fast_exp2(sv[h] - mn);
      l[h] = l[h] * alpha + warp_sum(pr[h]);
      m[h] = mn;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc[h][c].x *= alpha; acc[h][c].y *= alpha; acc[h][c].z *= alpha; acc[h][c].w *= alpha;
      }
    }
    // values: lane owns dims 4*lane + 128*c
#pragma unroll 4
    for (int j = 0; j < kTile; ++j) {
      const float p0 = __shfl_sync(0xffffffffu, pr[0], j);
      const float p1 = __shfl_sync(0xffffffffu, pr[1], j);
      const float* vr = sK + j * kKStride + 4 * lane;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(vr + 128 * c);
        acc[0][c].x = fmaf(p0, v.x, acc[0][c].x); acc[0][c].y = fmaf(p0, v.y, acc[0][c].y);
        acc[0][c].z = fmaf(p0, v.z, acc[0][c].z); acc[0][c].w = fmaf(p0, v.w, acc[0][c].w);
        acc[1][c].x = fmaf(p1, v.x, acc[1][c].x); acc[1][c].y = fmaf(p1, v.y, acc[1][c].y);
        acc[1][c].z = fmaf(p1, v.z, acc[1][c].z); acc[1][c].w = fmaf(p1, v.w, acc[1][c].w);
      }
    }
  }

  // normalise this split's result
  float lse_h[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float inv = l[h] > 0.f ? 1.0f / l[h] : 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      acc[h][c].x *= inv; acc[h][c].y *= inv; acc[h][c].z *= inv; acc[h][c].w *= inv;
    }
    lse_h[h] = l[h] > 0.f ? (m[h] + __log2f(l[h])) * kLn2 : -INFINITY;
  }
  const int h0 = hg * kHG + 2 * warp;  // first of this warp's two heads

  if (p.num_splits == 1) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t oi = (unit * H + h0 + h) * kDv;
      if (FUSED) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + oi;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          __nv_bfloat162 a = __floats2bfloat162_rn(acc[h][c].x, acc[h][c].y);
          __nv_bfloat162 bb = __floats2bfloat162_rn(acc[h][c].z, acc[h][c].w);
          *reinterpret_cast<uint2*>(o + 4 * lane + 128 * c) =
              make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&bb));
        }
      } else {
        float* o = reinterpret_cast<float*>(p.out) + oi;
#pragma unroll
        for (int c = 0; c < 4; ++c) *reinterpret_cast<float4*>(o + 4 * lane + 128 * c) = acc[h][c];
      }
      if (lane == 0) p.lse[unit * H + h0 + h] = lse_h[h];
    }
    return;
  }

  // split-KV: publish this split, the last CTA of the (unit, head group) merges
  const int S = p.num_splits;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t wi = ((unit * S + split) * H + h0 + h);
    float* o = p.ws_o + wi * kDv;
#pragma unroll
    for (int c = 0; c < 4; ++c) __stcg(reinterpret_cast<float4*>(o + 4 * lane + 128 * c), acc[h][c]);
    if (lane == 0) __stcg(p.ws_lse + wi, lse_h[h]);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int nhg = H / kHG;
    const unsigned prev = atomicAdd(p.ws_cnt + unit * nhg + hg, 1u);
    sLast = prev == (unsigned)(S - 1);
  }
  __syncthreads();
  if (!sLast) return;
  __threadfence();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float mx = -INFINITY;
    for (int s = 0; s < S; ++s) mx = fmaxf(mx, __ldcg(p.ws_lse + (unit * S + s) * H + h0 + h));
    float4 o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    float W = 0.f;
    if (mx != -INFINITY) {
      for (int s = 0; s < S; ++s) {
        const int64_t wi = (unit * S + s) * H + h0 + h;
        const float w = fast_exp2((__ldcg(p.ws_lse + wi) - mx) * kLog2e);
        if (w == 0.f) continue;
        W += w;
        const float* src = p.ws_o + wi * kDv;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src + 4 * lane + 128 * c));
          o[c].x = fmaf(w, v.x, o[c].x); o[c].y = fmaf(w, v.y, o[c].y);
          o[c].z = fmaf(w, v.z, o[c].z); o[c].w = fmaf(w, v.w, o[c].w);
        }
      }
      const float inv = 1.0f / W;
#pragma unroll
      for (int c = 0; c < 4; ++c) { o[c].x *= inv; o[c].y *= inv; o[c].z *= inv; o[c].w *= inv; }
    }
    const float lse_out = mx == -INFINITY ? -INFINITY : mx + __log2f(W) * kLn2;
    const int64_t oi = (unit * H + h0 + h) * kDv;
    if (FUSED) {
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + oi;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        __nv_bfloat162 a = __floats2bfloat162_rn(o[c].x, o[c].y);
        __nv_bfloat162 bb = __floats2bfloat162_rn(o[c].z, o[c].w);
        *reinterpret_cast<uint2*>(dst + 4 * lane + 128 * c) =
            make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&bb));
      }
    } else {
      float* dst = reinterpret_cast<float*>(p.out) + oi;
#pragma unroll
      for (int c = 0; c < 4; ++c) *reinterpret_cast<float4*>(dst + 4 * lane + 128 * c) = o[c];
    }
    if (lane == 0) p.lse[unit * H + h0 + h] = lse_out;
  }
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t simt_workspace_bytes(int64_t units, int heads, int splits) {
  if (splits <= 1) return 0;
  const size_t o = align256((size_t)units * splits * heads * kDv * sizeof(float));
  const size_t l = align256((size_t)units * splits * heads * sizeof(float));
  const size_t c = align256((size_t)units * (heads / kHG) * sizeof(unsigned));
  return o + l + c;
}

void simt_bind_workspace(DecodeParams& p, void* ws) {
  if (p.num_splits <= 1 || ws == nullptr) {
    p.ws_o = nullptr; p.ws_lse = nullptr; p.ws_cnt = nullptr;
    return;
  }
  char* base = static_cast<char*>(ws);
  const size_t o = align256((size_t)p.num_units * p.num_splits * p.heads * kDv * sizeof(float));
  const size_t l = align256((size_t)p.num_units * p.num_splits * p.heads * sizeof(float));
  p.ws_o = reinterpret_cast<float*>(base);
  p.ws_lse = reinterpret_cast<float*>(base + o);
  p.ws_cnt = reinterpret_cast<unsigned*>(base + o + l);
}

int simt_auto_splits(int64_t units, int heads, int64_t max_tokens) {
  const int64_t ctas = units * (heads / kHG);
  const int64_t target = 152 * 4;
  int64_t s = (target + ctas - 1) / ctas;
  const int64_t by_len = (max_tokens + kTile - 1) / kTile;  // at least one tile per split
  s = s < by_len ? s : by_len;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return (int)s;
}

template <int KVT, bool FUSED, bool SPARSE>
static cudaError_t launch_one(const DecodeParams& p, cudaStream_t st) {
  const size_t smem = (size_t)(kHG * kDqk + kTile * kKStride) * sizeof(float);
  cudaError_t e = raise_smem_limit((const void*)decode_simt_kernel<KVT, FUSED, SPARSE>, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)p.num_units, (unsigned)p.num_splits, (unsigned)(p.heads / kHG));
  decode_simt_kernel<KVT, FUSED, SPARSE><<<grid, kSimtThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_simt(const DecodeParams& p, int kv_dtype, bool fused, bool sparse,
                               cudaStream_t st) {
  if (p.num_units == 0) return cudaSuccess;
  if (kv_dtype == DCP_KV_BF16) {
    if (fused) return sparse ? launch_one<DCP_KV_BF16, true, true>(p, st)
                             : launch_one<DCP_KV_BF16, true, false>(p, st);
    return sparse ? launch_one<DCP_KV_BF16, false, true>(p, st)
                  : launch_one<DCP_KV_BF16, false, false>(p, st);
  }
  if (fused) return sparse ? launch_one<DCP_KV_FP8_E4M3_S128, true, true>(p, st)
                           : launch_one<DCP_KV_FP8_E4M3_S128, true, false>(p, st);
  return sparse ? launch_one<DCP_KV_FP8_E4M3_S128, false, true>(p, st)
                : launch_one<DCP_KV_FP8_E4M3_S128, false, false>(p, st);
}

}  // namespace dcp

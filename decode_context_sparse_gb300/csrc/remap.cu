// Slot remap of DSA top-k indices per DCP shard, and dense local lengths.
//
// Remap (SGLang PR #42536 "Fix DCP for RoPE sparse attention on Blackwell",
// Modifications, "Index remap"): keep the owned global slots, convert them to local ids,
// compact them to the front of the row in their original order, return the count.
//
// One CTA of 8 warps per row; warp w owns a contiguous segment of the row.  Pass 1
// counts each warp's owned ids per shard.  An exclusive scan over the 8 warps gives each
// warp its write base per shard.  Pass 2 re-reads the segment (L1/L2 hits) and writes
// every owned id at base + running count + rank among the lanes with the same owner, so
// the order is the input order.  The lanes with the same owner are found with one ballot
// per shard when the row is remapped for at most 16 shards (a ballot is one instruction),
// else with match.any (one instruction for any number of shards, but far slower).  The
// tail of every shard row is filled with -1.  Integer work only: bit-exact by construction.
#include "common.cuh"
#include "internal.h"

namespace dcp {

constexpr int kRemapWarps = 8;
constexpr int kRemapBallotShards = 16;
constexpr int kRemapBatch = 8;  // ids per lane loaded together

// The lanes of this warp whose key equals this lane's (key -1: none of interest); n_out
// shard keys 0 .. n_out-1.
template <bool BALLOT>
__device__ __forceinline__ unsigned same_key_lanes(int key, int n_out) {
  if (!BALLOT) return __match_any_sync(0xffffffffu, key);
  unsigned m = 0u;
#pragma unroll 4
  for (int s = 0; s < n_out; ++s) {
    const unsigned b = __ballot_sync(0xffffffffu, key == s);
    if (key == s) m = b;
  }
  return m;
}

template <bool BALLOT>
__global__ void __launch_bounds__(kRemapWarps * 32)
remap_topk_kernel(const int32_t* __restrict__ gidx, int k, const OwnerRule rule, int shard,
                  int32_t* __restrict__ local_idx, int32_t* __restrict__ count, int64_t rows) {
  const int D = rule.D;
  __shared__ int cnt[kRemapWarps][DCP_MAX_SHARDS];
  __shared__ int base[kRemapWarps][DCP_MAX_SHARDS];
  __shared__ int total[DCP_MAX_SHARDS];
  const int64_t row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s0 = shard < 0 ? 0 : shard;
  const int n_out = shard < 0 ? D : 1;
  for (int i = threadIdx.x; i < kRemapWarps * DCP_MAX_SHARDS; i += blockDim.x)
    (&cnt[0][0])[i] = 0;
  __syncthreads();

  const int seg = (k + kRemapWarps - 1) / kRemapWarps;
  const int p0 = warp * seg, p1 = min(k, p0 + seg);
  const int32_t* g = gidx + row * (int64_t)k;
  const unsigned lt = (1u << lane) - 1u;

  // The warp's segment in batches of kRemapBatch ids per lane, every load of a batch in
  // flight before any is used; a segment of one batch (k <= 2048) stays in registers for
  // pass 2, longer ones are re-read there (L1/L2 hits).
  auto load_batch = [&](int c0, int32_t (&t)[kRemapBatch]) {
#pragma unroll
    for (int u = 0; u < kRemapBatch; ++u) {
      const int pos = c0 + 32 * u + lane;
      t[u] = pos < p1 ? __ldg(g + pos) : -1;
    }
  };
  const bool one_batch = p1 - p0 <= 32 * kRemapBatch;
  int32_t t[kRemapBatch];

  // pass 1: per-warp per-shard counts
  for (int c0 = p0; c0 < p1; c0 += 32 * kRemapBatch) {
    load_batch(c0, t);
#pragma unroll
    for (int u = 0; u < kRemapBatch; ++u) {
      int key = -1;
      if (t[u] >= 0) {
        const int s = owner_of(t[u], rule);
        if (s - s0 >= 0 && s - s0 < n_out) key = s - s0;
      }
      const unsigned m = same_key_lanes<BALLOT>(key, n_out);
      if (key >= 0 && (m & lt) == 0) cnt[warp][key] += __popc(m);
      __syncwarp();
    }
  }
  __syncthreads();
  if (threadIdx.x < n_out) {
    int run = 0;
    for (int w = 0; w < kRemapWarps; ++w) {
      base[w][threadIdx.x] = run;
      run += cnt[w][threadIdx.x];
    }
    total[threadIdx.x] = run;
    count[(int64_t)threadIdx.x * rows + row] = run;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kRemapWarps * DCP_MAX_SHARDS; i += blockDim.x)
    (&cnt[0][0])[i] = 0;
  __syncthreads();

  // pass 2: write owned ids in input order
  for (int c0 = p0; c0 < p1; c0 += 32 * kRemapBatch) {
    if (!one_batch) load_batch(c0, t);
#pragma unroll
    for (int u = 0; u < kRemapBatch; ++u) {
      int key = -1, loc = 0;
      if (t[u] >= 0) {
        int s, l;
        owner_local(t[u], rule, s, l);
        if (s - s0 >= 0 && s - s0 < n_out) {
          key = s - s0;
          loc = l;
        }
      }
      const unsigned m = same_key_lanes<BALLOT>(key, n_out);
      if (key >= 0) {
        const int dst = base[warp][key] + cnt[warp][key] + __popc(m & lt);
        local_idx[((int64_t)key * rows + row) * k + dst] = loc;
      }
      __syncwarp();
      if (key >= 0 && (m & lt) == 0) cnt[warp][key] += __popc(m);
      __syncwarp();
    }
  }
  // tail fill
  for (int o = 0; o < n_out; ++o) {
    int32_t* dst = local_idx + ((int64_t)o * rows + row) * k;
    for (int pos = total[o] + threadIdx.x; pos < k; pos += blockDim.x) dst[pos] = -1;
  }
}

__global__ void local_lengths_kernel(const int32_t* __restrict__ glen, int64_t rows, int D, int I,
                                     int shard, int32_t* __restrict__ llen) {
  const int n_out = shard < 0 ? D : 1;
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= rows * n_out) return;
  const int o = (int)(i / rows);
  const int64_t r = i - (int64_t)o * rows;
  const int s = (shard < 0 ? 0 : shard) + o;
  const int L = max(0, glen[r]);
  const int ID = I * D;
  const int rem = L % ID - s * I;
  llen[i] = (L / ID) * I + min(max(rem, 0), I);
}

cudaError_t launch_remap_topk(const int32_t* gidx, int64_t rows, int k, int D, int I, int shard,
                              int32_t* local_idx, int32_t* count, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int n_out = shard < 0 ? D : 1;
  if (n_out <= kRemapBallotShards)
    remap_topk_kernel<true><<<(unsigned)rows, kRemapWarps * 32, 0, st>>>(
        gidx, k, make_owner_rule(D, I), shard, local_idx, count, rows);
  else
    remap_topk_kernel<false><<<(unsigned)rows, kRemapWarps * 32, 0, st>>>(
        gidx, k, make_owner_rule(D, I), shard, local_idx, count, rows);
  return cudaGetLastError();
}

cudaError_t launch_local_lengths(const int32_t* glen, int64_t rows, int D, int I, int shard,
                                 int32_t* llen, cudaStream_t st) {
  const int64_t n = rows * (shard < 0 ? D : 1);
  if (n == 0) return cudaSuccess;
  local_lengths_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(glen, rows, D, I, shard, llen);
  return cudaGetLastError();
}

}  // namespace dcp

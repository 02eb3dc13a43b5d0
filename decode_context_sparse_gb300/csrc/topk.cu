// DSA top-k producer under DCP: each shard's candidate list, and the merge of the D lists
// into a row's global top-k (LMDeploy PR #4952 "support decode context parallelism for
// PyTorch MLA", Summary: DSA merges the local candidates into the global top-k; SGLang
// PR #36990, item 2: with a split index cache every indexer layer merges the ranks'
// local top-k candidates).
//
// One CTA per list -- a (shard, row) for the candidates, a row for the merge -- selects the
// k best of its n entries by radix selection on a 64-bit key.  The high word is an
// order-preserving image of the fp32 score (NaN, -inf and padding ids map to 0 and are never
// selected; -0 maps like +0); the low word is the complement of the global slot id, so a
// larger key ranks first and the keys of one list are distinct.  Digits of 11, 11 and 10
// bits of each word are resolved from the top: a digit's histogram (shared-memory atomics)
// locates the bin of the k-th largest key among those still in play, and the search stops
// as soon as that bin is taken whole (two digits for continuous scores).  The high words of
// a list of up to kTkStageMax entries are staged in shared memory while the first digit's
// histogram is built from the global loads; longer lists re-read global memory (L2) for
// each further digit.  The selection is written in increasing slot order: a candidate list
// by a stable compaction (local slot order is global slot order on a shard), the merge by a
// bitonic sort of the selected ids in shared memory.
// Comparisons and integer work only: the result is bit-identical to the definition.
#include <limits.h>

#include "common.cuh"
#include "internal.h"

namespace dcp {

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkBins = 2048;

// Order-preserving image of an fp32 score; 0 for the entries that are never selected.
__device__ __forceinline__ uint32_t score_key(float s) {
  const uint32_t u = __float_as_uint(s);
  if (s != s || u == 0xff800000u) return 0u;   // NaN, -inf
  if (u == 0x80000000u) return 0x80000000u;     // -0 ranks as +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Entry i of one list.
template <bool MERGE>
struct TkList {
  const float* sc;     // candidates: the list's scores; merge: shard 0's list of the row
  const int32_t* id;   // merge: shard 0's ids of the row
  int64_t dstride;     // merge: elements between two shards' lists
  int kin;             // merge: entries per shard list
  int D, I, s;         // candidates: owner rule and shard

  __device__ __forceinline__ int64_t off(int i) const {
    if (!MERGE) return i;
    const int d = i / kin;
    return d * dstride + (i - d * kin);
  }
  __device__ __forceinline__ float score(int i) const { return __ldg(sc + off(i)); }
  __device__ __forceinline__ int gid(int i) const {
    if (MERGE) return __ldg(id + off(i));
    return (i / I) * I * D + s * I + i % I;  // local slot i of shard s (< 2^31, host-checked)
  }
  __device__ __forceinline__ uint32_t key(int i) const {
    if (MERGE && gid(i) < 0) return 0u;
    return score_key(score(i));
  }
};

// Exclusive block-wide prefix of v over threads in index order; *total the sum.
// ws: kTkWarps words of shared memory, free on entry and on return.
__device__ __forceinline__ uint32_t tk_scan(uint32_t v, uint32_t* ws, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kTkWarps; ++w) {
    const uint32_t t = ws[w];
    if (w < warp) before += t;
    tot += t;
  }
  __syncthreads();
  *total = tot;
  return before + x - v;
}

struct TkShared {
  uint32_t ws[2][kTkWarps];
  uint32_t bin, above;
};

// The bin (of nb) holding the krem-th largest in-play key, counting from the top bin, and
// the number of in-play keys in the bins above it.
__device__ __forceinline__ void tk_find_bin(const uint32_t* hist, int nb, uint32_t krem,
                                            TkShared& sh) {
  const int bpt = nb / kTkThreads;  // bins per thread, taken from the top
  const int top = nb - 1 - threadIdx.x * bpt;
  uint32_t mine = 0;
  for (int j = 0; j < bpt; ++j) mine += hist[top - j];
  uint32_t tot;
  uint32_t cum = tk_scan(mine, sh.ws[0], &tot);
  for (int j = 0; j < bpt; ++j) {
    const uint32_t h = hist[top - j];
    if (cum < krem && cum + h >= krem) {
      sh.bin = (uint32_t)(top - j);
      sh.above = cum;
    }
    cum += h;
  }
  __syncthreads();
}

template <bool MERGE>
__global__ void __launch_bounds__(kTkThreads) topk_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint32_t tk_smem[];
  uint32_t* hist = tk_smem;
  uint32_t* keys = tk_smem + kTkBins;                          // p.stage entries
  int32_t* sorted = reinterpret_cast<int32_t*>(keys + p.stage);  // merge: p.kp entries
  __shared__ TkShared sh;
  const int tid = threadIdx.x;
  const int64_t li = blockIdx.x;

  TkList<MERGE> src;
  int n;
  if (MERGE) {
    src.sc = p.score + li * (int64_t)p.stride;
    src.id = p.ids + li * (int64_t)p.stride;
    src.dstride = p.rows * (int64_t)p.stride;
    src.kin = p.stride;
    n = p.D * p.stride;
  } else {
    const int o = (int)(li / p.rows);
    src.sc = p.score + li * (int64_t)p.stride;
    src.D = p.D;
    src.I = p.I;
    src.s = p.shard < 0 ? o : p.shard;
    n = min(max(__ldg(p.len + li), 0), p.stride);
  }
  const bool staged = n <= p.stage;

  // pass 0: stage the high words, count the valid entries, histogram of the first digit
  for (int i = tid; i < kTkBins; i += kTkThreads) hist[i] = 0u;
  __syncthreads();
  uint32_t nv = 0;
  for (int i0 = 0; i0 < n; i0 += 4 * kTkThreads) {
    uint32_t h[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kTkThreads + tid;
      h[u] = i < n ? src.key(i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kTkThreads + tid;
      if (staged && i < n) keys[i] = h[u];
      if (h[u]) {
        ++nv;
        atomicAdd(&hist[h[u] >> 21], 1u);
      }
    }
  }
  __syncthreads();
  uint32_t nvalid;
  tk_scan(nv, sh.ws[0], &nvalid);

  // radix search for the k-th largest key T; the selection is then key >= T
  uint32_t t_hi = 1u, t_lo = 0u;  // fewer valid entries than k: all of them
  if (nvalid > (uint32_t)p.k) {
    uint32_t krem = (uint32_t)p.k, pre_hi = 0, msk_hi = 0, pre_lo = 0, msk_lo = 0;
    for (int dg = 0; dg < 6; ++dg) {
      const bool lo = dg >= 3;
      const int shift = dg % 3 == 0 ? 21 : dg % 3 == 1 ? 10 : 0;
      const int nb = dg % 3 == 2 ? 1024 : 2048;
      if (dg > 0) {
        for (int i = tid; i < kTkBins; i += kTkThreads) hist[i] = 0u;
        __syncthreads();
        for (int i = tid; i < n; i += kTkThreads) {
          const uint32_t h = staged ? keys[i] : src.key(i);
          if (h == 0u) continue;
          if (!lo) {
            if ((h & msk_hi) == pre_hi) atomicAdd(&hist[(h >> shift) & (nb - 1)], 1u);
          } else if (h == pre_hi) {
            const uint32_t l = ~(uint32_t)src.gid(i);
            if ((l & msk_lo) == pre_lo) atomicAdd(&hist[(l >> shift) & (nb - 1)], 1u);
          }
        }
        __syncthreads();
      }
      tk_find_bin(hist, nb, krem, sh);
      const uint32_t b = sh.bin;
      krem -= sh.above;
      const uint32_t hb = hist[b];
      if (!lo) {
        pre_hi |= b << shift;
        msk_hi |= (uint32_t)(nb - 1) << shift;
      } else {
        pre_lo |= b << shift;
        msk_lo |= (uint32_t)(nb - 1) << shift;
      }
      __syncthreads();  // every thread has read the bin before the histogram is cleared
      if (hb == krem) break;  // the bin is taken whole (always by the last digit: keys differ)
    }
    t_hi = pre_hi;
    t_lo = pre_lo;
  }

  // stable compaction of the selected entries in index order, at most k
  uint32_t base = 0;
  int rnd = 0;
  for (int i0 = 0; i0 < n; i0 += 4 * kTkThreads, ++rnd) {
    bool sel[4];
    uint32_t c = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + 4 * tid + u;
      bool s = false;
      if (i < n) {
        const uint32_t h = staged ? keys[i] : src.key(i);
        s = h != 0u && (h > t_hi || (h == t_hi && (t_lo == 0u || ~(uint32_t)src.gid(i) >= t_lo)));
      }
      sel[u] = s;
      c += s;
    }
    // exclusive prefix over threads (one barrier per round: warp totals double-buffered)
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    uint32_t* ws = sh.ws[rnd & 1];
    if (lane == 31) ws[warp] = x;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kTkWarps; ++w) {
      const uint32_t t = ws[w];
      if (w < warp) before += t;
      tot += t;
    }
    uint32_t pos = base + before + x - c;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (sel[u] && pos < (uint32_t)p.k) {
        const int i = i0 + 4 * tid + u;
        if (MERGE) {
          sorted[pos] = src.gid(i);
        } else {
          p.cand_score[li * p.k + pos] = src.score(i);
          p.cand_idx[li * p.k + pos] = src.gid(i);
        }
      }
      pos += sel[u];
    }
    base += tot;
  }
  const int cnt = (int)min(base, (uint32_t)p.k);

  if (!MERGE) {
    for (int j = cnt + tid; j < p.k; j += kTkThreads) {
      p.cand_score[li * p.k + j] = -INFINITY;
      p.cand_idx[li * p.k + j] = -1;
    }
    return;
  }
  // merge: the selected ids in increasing order (bitonic sort over p.kp >= k entries)
  __syncthreads();
  for (int j = cnt + tid; j < p.kp; j += kTkThreads) sorted[j] = INT_MAX;
  __syncthreads();
  for (int size = 2; size <= p.kp; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = tid; t < p.kp / 2; t += kTkThreads) {
        const int i = 2 * t - (t & (stride - 1));
        const int j = i + stride;
        const int a = sorted[i], b = sorted[j];
        if ((a > b) == ((i & size) == 0)) {
          sorted[i] = b;
          sorted[j] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int j = tid; j < p.k; j += kTkThreads) p.topk[li * p.k + j] = j < cnt ? sorted[j] : -1;
  if (tid == 0 && p.count) p.count[li] = cnt;
}

namespace {
size_t tk_smem_bytes(int stage, int kp) { return (size_t)(kTkBins + stage + kp) * 4; }

template <bool MERGE>
cudaError_t tk_launch(const TopkParams& p, int64_t lists, cudaStream_t st) {
  const size_t smem = tk_smem_bytes(p.stage, MERGE ? p.kp : 0);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel<MERGE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_kernel<MERGE><<<(unsigned)lists, kTkThreads, smem, st>>>(p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_topk_local(TopkParams p, int n_in, cudaStream_t st) {
  if (p.rows == 0) return cudaSuccess;
  p.stage = p.stride < kTkStageMax ? p.stride : kTkStageMax;
  p.kp = 0;
  return tk_launch<false>(p, p.rows * n_in, st);
}

cudaError_t launch_topk_merge(TopkParams p, cudaStream_t st) {
  if (p.rows == 0) return cudaSuccess;
  const int64_t n = (int64_t)p.D * p.stride;
  p.stage = n < kTkStageMax ? (int)n : kTkStageMax;
  int kp = 1;
  while (kp < p.k) kp <<= 1;
  p.kp = kp;
  return tk_launch<true>(p, p.rows, st);
}

}  // namespace dcp

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
// larger key ranks first and the keys of one list are distinct.  The first digit (the
// top 11 bits) is resolved by a histogram (shared-memory atomics) built while a list of up
// to kTkStageMax entries is staged in shared memory (aligned candidate lists: every 16-B
// piece of the row copied asynchronously at once, then turned into keys in place; otherwise
// through registers); the bin that holds the k-th largest key then usually holds a few
// hundred staged entries, whose 16-bit indices become the candidates, and the remaining
// digits (9 bits each) look at the candidates only, each digit's bin found by one warp.  The
// search stops as soon as a digit's bin is taken whole.  Lists longer than the staging, or
// with more candidates than the buffer holds, resolve the further digits (11, 10, then the
// low word) over every entry, re-reading global memory (L2) when not staged.  The
// selection is written in increasing slot order: a candidate list by a stable compaction
// (local slot order is global slot order on a shard), the merge by merging the shards'
// ascending runs (a bitonic sort when some run is out of order).
// Comparisons and integer work only: the result is bit-identical to the definition.
#include <limits.h>

#include "common.cuh"
#include "internal.h"

namespace dcp {

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkBins = 2048;
// candidates (the staged entries in the first digit's bin): their histogram takes the first
// kTkCandBins words of the first digit's, their 16-bit staging indices the rest (3072; a
// merge of lists that are each a shard's best entries puts ~13% of them in the first bin)
constexpr int kTkCandBins = 512;
constexpr int kTkCandCap = (kTkBins - kTkCandBins) * 2;
constexpr int kTkRound = 4 * kTkThreads;  // entries per round: four consecutive per thread
constexpr int kTkLoadRounds = 4;          // rounds whose loads are issued together
constexpr int kTkBlockRounds = kTkStageMax / kTkRound;  // rounds per compaction block
static_assert(kTkStageMax % kTkRound == 0, "staging holds whole rounds");
static_assert(kTkStageMax / kTkRound <= 8 && kTkStageMax <= 65536,
              "a thread's staged entries fit one 32-bit mask; staging indices fit 16 bits");

// Order-preserving image of an fp32 score; 0 for the entries that are never selected.
// Adding +0 turns -0 into +0 (so that it ranks as +0) and leaves every other value as it is.
// The image of -inf is 0x007fffff and that of +inf 0xff800000; NaNs map outside that range.
__device__ __forceinline__ uint32_t score_key(float s) {
  const uint32_t u = __float_as_uint(__fadd_rn(s, 0.0f));
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return k - 0x00800000u <= 0xff800000u - 0x00800000u ? k : 0u;
}

// The fp32 score of a key (inverse of score_key for keys other than 0).
__device__ __forceinline__ float key_score(uint32_t h) {
  return __uint_as_float((h & 0x80000000u) ? (h ^ 0x80000000u) : ~h);
}

// Entry i of one list.
template <bool MERGE>
struct TkList {
  const float* sc;     // candidates: the list's scores; merge: shard 0's list of the row
  const int32_t* id;   // merge: shard 0's ids of the row
  int64_t dstride;     // merge: elements between two shards' lists
  int kin;             // merge: entries per shard list
  int n;               // entries
  int D, I, s;         // candidates: owner rule and shard
  bool vec;            // four consecutive entries from one 16-B aligned load
  FastDiv div;         // candidates: division by I; merge: by kin

  __device__ __forceinline__ int64_t off(int i) const {
    if (!MERGE) return i;
    const int d = fdiv(i, div);
    return d * dstride + (i - d * kin);
  }
  __device__ __forceinline__ float score(int i) const { return __ldg(sc + off(i)); }
  __device__ __forceinline__ int gid(int i) const {
    if (MERGE) return __ldg(id + off(i));
    if (I == 1) return i * D + s;
    const int q = fdiv(i, div);
    return q * I * D + s * I + (i - q * I);  // local slot i of shard s (< 2^31, host-checked)
  }
  __device__ __forceinline__ uint32_t key(int i) const {
    if (MERGE && gid(i) < 0) return 0u;
    return score_key(score(i));
  }
  // scores (and merge: ids) of entries i .. i+3 (i a multiple of 4); past the end: -inf
  __device__ __forceinline__ void raw4(int i, float4& v, int4& t) const {
    if (vec && i + 3 < n) {
      const int64_t o = off(i);  // a multiple of 4 entries, all four in one list
      v = __ldg(reinterpret_cast<const float4*>(sc + o));
      if (MERGE) t = __ldg(reinterpret_cast<const int4*>(id + o));
      return;
    }
    v.x = i < n ? score(i) : -INFINITY;
    v.y = i + 1 < n ? score(i + 1) : -INFINITY;
    v.z = i + 2 < n ? score(i + 2) : -INFINITY;
    v.w = i + 3 < n ? score(i + 3) : -INFINITY;
    if (MERGE) {
      t.x = i < n ? gid(i) : -1;
      t.y = i + 1 < n ? gid(i + 1) : -1;
      t.z = i + 2 < n ? gid(i + 2) : -1;
      t.w = i + 3 < n ? gid(i + 3) : -1;
    }
  }
  __device__ __forceinline__ uint4 keys_of(const float4& v, const int4& t) const {
    uint4 k = make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
    if (MERGE) {
      k.x = t.x < 0 ? 0u : k.x;
      k.y = t.y < 0 ? 0u : k.y;
      k.z = t.z < 0 ? 0u : k.z;
      k.w = t.w < 0 ? 0u : k.w;
    }
    return k;
  }
  // keys of entries i .. i+3 (i a multiple of 4); 0 past the end
  __device__ __forceinline__ uint4 key4(int i) const {
    if (vec && i + 3 < n) {
      const int64_t o = off(i);  // a multiple of 4 entries, all four in one list
      const float4 v = __ldg(reinterpret_cast<const float4*>(sc + o));
      uint4 k = make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
      if (MERGE) {
        const int4 t = __ldg(reinterpret_cast<const int4*>(id + o));
        k.x = t.x < 0 ? 0u : k.x;
        k.y = t.y < 0 ? 0u : k.y;
        k.z = t.z < 0 ? 0u : k.z;
        k.w = t.w < 0 ? 0u : k.w;
      }
      return k;
    }
    return make_uint4(i < n ? key(i) : 0u, i + 1 < n ? key(i + 1) : 0u,
                      i + 2 < n ? key(i + 2) : 0u, i + 3 < n ? key(i + 3) : 0u);
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
  // every warp scans the warp totals itself
  const uint32_t wt = lane < kTkWarps ? ws[lane] : 0u;
  uint32_t wx = wt;
#pragma unroll
  for (int o = 1; o < kTkWarps; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, wx, o);
    if (lane >= o) wx += y;
  }
  const uint32_t before = __shfl_sync(0xffffffffu, wx - wt, warp);
  *total = __shfl_sync(0xffffffffu, wx, kTkWarps - 1);
  __syncthreads();
  return before + x - v;
}

struct TkShared {
  uint32_t ws[kTkWarps];
  uint32_t cw[kTkBlockRounds][kTkWarps];   // selected entries per (round, warp) of a block
  uint32_t off[kTkBlockRounds][kTkWarps];  // their output offsets
  uint32_t bin, above, binh, base;  // a digit's bin, the keys in play above it, its count
  int maxid;                         // merge: the largest selected id
  int run[DCP_MAX_SHARDS + 1];  // merge: first selected entry of each shard's list
};

// The bin (of BPT * kTkThreads) holding the krem-th largest in-play key, counting from the
// top bin, the number of in-play keys in the bins above it and in the bin (sh.bin,
// sh.above, sh.binh).  Returns the histogram's total.
template <int BPT>
__device__ __forceinline__ uint32_t tk_find_bin(const uint32_t* hist, uint32_t krem, TkShared& sh) {
  const int top = kTkThreads * BPT - 1 - threadIdx.x * BPT;  // bins top, top - 1, ...
  uint32_t h[BPT], mine = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    h[j] = hist[top - j];
    mine += h[j];
  }
  uint32_t tot;
  uint32_t cum = tk_scan(mine, sh.ws, &tot);
  // (a bin is always found: krem never exceeds the keys in play)
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    if (cum < krem && cum + h[j] >= krem) {
      sh.bin = (uint32_t)(top - j);
      sh.above = cum;
      sh.binh = h[j];
    }
    cum += h[j];
  }
  __syncthreads();
  return tot;
}

// The same search by one warp over NB bins (NB / 32 a multiple of 4, at most 64 bins a
// lane), for the histograms that the whole block built: lane l sums the l-th group of
// NB / 32 bins from the top (16-B reads in a lane-rotated order, so that the lanes of a
// quarter warp hit distinct banks), a scan of the sums finds the group holding the krem-th
// key, and a second scan over that group's bins (one or two a lane) the bin.  Every lane
// returns the bin, *above and *binh; krem above the total gives bin 0 with nothing in it.
template <int NB>
__device__ __forceinline__ uint32_t tk_find_bin_warp(const uint32_t* hist, uint32_t krem,
                                                     uint32_t* above, uint32_t* binh) {
  constexpr int BPL = NB / 32;
  static_assert(BPL % 4 == 0 && BPL <= 64, "whole 16-B pieces, at most two bins a lane after");
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const uint4* g = reinterpret_cast<const uint4*>(hist + NB - BPL * (lane + 1));
  uint32_t s = 0;
#pragma unroll
  for (int q = 0; q < BPL / 4; ++q) {
    const uint4 v = g[(q + lane) % (BPL / 4)];
    s += (v.x + v.y) + (v.z + v.w);
  }
  uint32_t x = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kAll, x, o);
    if (lane >= o) x += y;
  }
  const uint32_t hit = __ballot_sync(kAll, x >= krem);
  if (hit == 0u) {
    *above = __shfl_sync(kAll, x, 31);
    *binh = 0u;
    return 0u;
  }
  const int L = __ffs(hit) - 1;
  const uint32_t cum = __shfl_sync(kAll, x - s, L);  // keys in the groups above group L
  const int topL = NB - 1 - BPL * L;                  // group L's top bin
  constexpr int PER = BPL >= 32 ? BPL / 32 : 1;       // bins a lane takes in group L
  uint32_t h0 = 0u, h1 = 0u;
  if (PER == 2) {
    h0 = hist[topL - 2 * lane];
    h1 = hist[topL - 2 * lane - 1];
  } else if (lane < BPL) {
    h0 = hist[topL - lane];
  }
  const uint32_t ps = h0 + h1;
  uint32_t xx = ps;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kAll, xx, o);
    if (lane >= o) xx += y;
  }
  const int J = __ffs(__ballot_sync(kAll, cum + xx >= krem)) - 1;  // (there is one)
  const uint32_t before = cum + __shfl_sync(kAll, xx - ps, J);
  const uint32_t a0 = __shfl_sync(kAll, h0, J), a1 = __shfl_sync(kAll, h1, J);
  const bool first = PER == 1 || before + a0 >= krem;
  *above = first ? before : before + a0;
  *binh = first ? a0 : a1;
  return (uint32_t)(PER == 2 ? topL - 2 * J - (first ? 0 : 1) : topL - J);
}

// tk_find_bin_warp by warp 0, its result in sh.bin, sh.above, sh.binh for every thread.
template <int NB>
__device__ __forceinline__ void tk_find_bin_w0(const uint32_t* hist, uint32_t krem, TkShared& sh) {
  if (threadIdx.x < 32) {
    uint32_t ab, bh;
    const uint32_t b = tk_find_bin_warp<NB>(hist, krem, &ab, &bh);
    if (threadIdx.x == 0) {
      sh.bin = b;
      sh.above = ab;
      sh.binh = bh;
    }
  }
  __syncthreads();
}

// A 16-B asynchronous copy from global to shared memory (both 16-B aligned), and the wait
// for every such copy of the calling thread.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The first digit's bin (kTkBins = 128 bins per warp): warp w sums bins [128 w, 128 w + 128)
// (one 16-B read a lane), then warp 0 finds the group holding the krem-th key counting from
// the top and the bin within it (a 16-B read a lane again).  Results in sh as tk_find_bin.
__device__ __forceinline__ void tk_find_bin_first(const uint32_t* hist, uint32_t krem, TkShared& sh) {
  static_assert(kTkBins == 128 * kTkWarps, "a group of 128 bins per warp");
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  {
    const uint4 v = reinterpret_cast<const uint4*>(hist + 128 * warp)[lane];
    const uint32_t g = __reduce_add_sync(kAll, (v.x + v.y) + (v.z + v.w));
    if (lane == 0) sh.ws[warp] = g;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t s = lane < kTkWarps ? sh.ws[kTkWarps - 1 - lane] : 0u;  // groups from the top
    uint32_t x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kAll, x, o);
      if (lane >= o) x += y;
    }
    const uint32_t hit = __ballot_sync(kAll, lane < kTkWarps && x >= krem);
    uint32_t bin = 0u, above = __shfl_sync(kAll, x, 31), binh = 0u;
    if (hit != 0u) {
      const int gl = __ffs(hit) - 1;
      const int grp = kTkWarps - 1 - gl;
      const uint32_t cum = __shfl_sync(kAll, x - s, gl);
      // lane j: the group's bins 4 (31 - j) .. 4 (31 - j) + 3, from the top
      const uint4 q = reinterpret_cast<const uint4*>(hist + 128 * grp)[31 - lane];
      const uint32_t ps = (q.x + q.y) + (q.z + q.w);
      uint32_t xx = ps;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kAll, xx, o);
        if (lane >= o) xx += y;
      }
      const int J = __ffs(__ballot_sync(kAll, cum + xx >= krem)) - 1;  // (there is one)
      uint32_t before = cum + __shfl_sync(kAll, xx - ps, J);
      const uint32_t a[4] = {__shfl_sync(kAll, q.w, J), __shfl_sync(kAll, q.z, J),
                             __shfl_sync(kAll, q.y, J), __shfl_sync(kAll, q.x, J)};
      const int base = 128 * grp + 4 * (31 - J) + 3;
      bool found = false;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (!found && before + a[e] >= krem) {
          found = true;
          bin = (uint32_t)(base - e);
          above = before;
          binh = a[e];
        }
        if (!found) before += a[e];
      }
    }
    if (lane == 0) {
      sh.bin = bin;
      sh.above = above;
      sh.binh = binh;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t h, uint32_t msk, uint32_t pre,
                                         int shift, int nb) {
  // (msk covers the first digit and pre's first digit is a bin >= 1: h == 0 never counts)
  if ((h & msk) == pre) atomicAdd(&hist[(h >> shift) & (nb - 1)], 1u);
}

template <bool MERGE>
// (three CTAs per SM: 72 KB of shared memory each, at most 42 registers a thread)
__global__ void __launch_bounds__(kTkThreads, 3) topk_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint32_t tk_smem[];
  uint32_t* hist = tk_smem;
  uint32_t* keys = tk_smem + kTkBins;                          // p.stage entries
  // merge: two run buffers of p.kp entries; for kp <= kTkBins the histogram's words and the
  // staging, both free once the selection is compacted, else words past the staging
  const bool runs_inside = p.kp <= kTkBins;
  int32_t* sorted = reinterpret_cast<int32_t*>(runs_inside ? hist : keys + p.stage);
  int32_t* sorted2 = runs_inside ? reinterpret_cast<int32_t*>(keys) : sorted + p.kp;
  __shared__ TkShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t li = blockIdx.x;

  // aligned candidate lists whose whole row stride fits the staging: every 16-B piece of
  // the row is copied into the staging at once (asynchronous copies, no registers held),
  // before the list's length is known; the pieces are turned into keys in place below, each
  // by the thread that copied it
  const bool async = !MERGE && p.vec && p.stride <= p.stage;
  if (async) {
    const float* row = p.score + li * (int64_t)p.stride;
#pragma unroll
    for (int c = 0; c < kTkBlockRounds; ++c) {
      const int i = c * kTkRound + 4 * tid;
      if (i < p.stride) cp_async16(keys + i, row + i);
    }
  }

  TkList<MERGE> src;
  src.vec = p.vec != 0;
  src.div = p.div;
  if (MERGE) {
    src.sc = p.score + li * (int64_t)p.stride;
    src.id = p.ids + li * (int64_t)p.stride;
    src.dstride = p.rows * (int64_t)p.stride;
    src.kin = p.stride;
    src.n = p.D * p.stride;
  } else {
    const int o = (int)(li / p.rows);
    src.sc = p.score + li * (int64_t)p.stride;
    src.D = p.D;
    src.I = p.I;
    src.s = p.shard < 0 ? o : p.shard;
    src.n = min(max(__ldg(p.len + li), 0), p.stride);
  }
  const int n = src.n;
  const bool staged = n <= p.stage;
  const int rounds = (n + kTkRound - 1) / kTkRound;
  // keys of this thread's four entries of round c
  auto get4 = [&](int c) -> uint4 {
    const int i = c * kTkRound + 4 * tid;
    return staged ? *reinterpret_cast<const uint4*>(keys + i) : src.key4(i);
  };

  // A merge first selects by score alone (the ids not read): the result is the same unless
  // an entry with a padding id (< 0) is selected, which the id pass after the compaction
  // sees; the merge then selects again with the ids.  (A padding entry below the threshold
  // cannot move it; in a tie at the threshold the padding ids rank last.)
  for (int attempt = 0;; ++attempt) {
    const bool exact = !MERGE || attempt > 0;
    const bool masync = MERGE && !exact && staged && src.vec;
    if (masync) {  // the scores, every piece at once (n is a multiple of 4)
#pragma unroll 1
      for (int c = 0; c < kTkBlockRounds; ++c) {
        const int i = c * kTkRound + 4 * tid;
        if (i < n) cp_async16(keys + i, src.sc + src.off(i));
      }
    }

    // pass 0: stage the keys and build the histogram of the first digit.  Every entry counts,
    // the invalid ones (key 0, and the entries past the end) in bin 0, which holds no valid key.
    for (int i = tid; i < kTkBins; i += kTkThreads) hist[i] = 0u;
    __syncthreads();
    if (async || masync) {
      cp_async_wait_all();
#pragma unroll
      for (int c = 0; c < kTkBlockRounds; ++c) {
        if (c < rounds) {
          const int i = c * kTkRound + 4 * tid;
          float4 v = *reinterpret_cast<const float4*>(keys + i);
          if (i + 3 >= n) {  // the ragged end: entries past the list count as -inf
            v.x = i < n ? v.x : -INFINITY;
            v.y = i + 1 < n ? v.y : -INFINITY;
            v.z = i + 2 < n ? v.z : -INFINITY;
            v.w = i + 3 < n ? v.w : -INFINITY;
          }
          const int4 t = make_int4(0, 0, 0, 0);  // (a merge's first selection: ids not read)
          const uint4 k4 = src.keys_of(v, t);
          *reinterpret_cast<uint4*>(keys + i) = k4;
          atomicAdd(&hist[k4.x >> 21], 1u);
          atomicAdd(&hist[k4.y >> 21], 1u);
          atomicAdd(&hist[k4.z >> 21], 1u);
          atomicAdd(&hist[k4.w >> 21], 1u);
        }
      }
    }
    for (int c0 = 0; c0 < (async || masync ? 0 : rounds); c0 += kTkLoadRounds) {
      // every load of kTkLoadRounds rounds in flight before any is used
      float4 v[kTkLoadRounds];
      int4 t[kTkLoadRounds];
#pragma unroll
      for (int u = 0; u < kTkLoadRounds; ++u) {
        if (c0 + u < rounds) {
          src.raw4((c0 + u) * kTkRound + 4 * tid, v[u], t[u]);
        } else {
          v[u] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          t[u] = make_int4(-1, -1, -1, -1);
        }
      }
#pragma unroll
      for (int u = 0; u < kTkLoadRounds; ++u) {
        if (c0 + u < rounds) {
          const uint4 k4 = src.keys_of(v[u], t[u]);
          if (staged)  // the staging is a whole number of rounds
            *reinterpret_cast<uint4*>(keys + (c0 + u) * kTkRound + 4 * tid) = k4;
          atomicAdd(&hist[k4.x >> 21], 1u);
          atomicAdd(&hist[k4.y >> 21], 1u);
          atomicAdd(&hist[k4.z >> 21], 1u);
          atomicAdd(&hist[k4.w >> 21], 1u);
        }
      }
    }
    __syncthreads();
    // the first digit's bin; the valid entries are those outside bin 0
    tk_find_bin_first(hist, (uint32_t)p.k, sh);
    const uint32_t nvalid = (uint32_t)(rounds * kTkRound) - hist[0];
    // more valid entries than k: a radix search for the k-th largest key T, the selection
    // being key >= T; else every valid entry (key >= 1)
    const bool search = nvalid > (uint32_t)p.k;
    const uint32_t b0 = search ? sh.bin : 0u;
    uint32_t krem = search ? (uint32_t)p.k - sh.above : 0u;
    bool done = !search || sh.binh == krem;  // (a bin taken whole ends the search)
    uint32_t pre_hi = search ? b0 << 21 : 1u, msk_hi = 0xffe00000u, pre_lo = 0, msk_lo = 0;

    // staged lists: one pass over this thread's run of 32 entries [32 tid, 32 tid + 32) (read
    // in a rotated chunk order, so that the threads of a warp hit distinct banks) sorts them
    // into those above the first digit's bin (selected whatever T is) and those in it (the
    // candidates); bit b of a mask is entry 32 tid + b
    const int e0 = 32 * tid, lim = rounds * kTkRound;
    uint32_t amask = 0u, cmask = 0u;
    if (staged) {
      // above the bin: key > thr_a (no key when b0 is the top bin); in or above it: key >= thr_c.
      // Chunk j's bits go to positions 4j..4j+3 and the masks are rotated into entry order
      // at the end (chunk j holds entries 4 ((j + tid) mod 8) ..).
      const uint32_t thr_a = (uint32_t)((((uint64_t)b0 + 1u) << 21) - 1u);
      const uint32_t thr_c = b0 << 21;
      uint32_t ar = 0u, cr = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = e0 + 4 * ((j + tid) & 7);
        if (i < lim) {  // (entries past the staged rounds are past the end)
          const uint4 k4 = *reinterpret_cast<const uint4*>(keys + i);
          const uint32_t k[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (k[e] > thr_a) ar |= 1u << (4 * j + e);
            if (k[e] >= thr_c) cr |= 1u << (4 * j + e);
          }
        }
      }
      const int rot = 4 * (tid & 7);
      amask = __funnelshift_l(ar, ar, rot);
      cmask = search ? __funnelshift_l(cr, cr, rot) & ~amask : 0u;  // (bin 0: the invalid entries)
    }
    bool wide = !staged;  // the further digits run over every entry
    if (!done && staged) {
      // the candidates' 16-bit staging indices go to the histogram's upper words
      uint32_t nc;
      uint32_t o = tk_scan((uint32_t)__popc(cmask), sh.ws, &nc);  // (after every read of hist)
      if (nc <= (uint32_t)kTkCandCap) {
        uint16_t* cand = reinterpret_cast<uint16_t*>(hist + kTkCandBins);
        for (uint32_t m = cmask; m != 0u; m &= m - 1u) cand[o++] = (uint16_t)(e0 + __ffs(m) - 1);
        // digits of 9 bits (the last of each word narrower) over the candidates only
        for (int dg = 0; dg < 7 && !done; ++dg) {
          const bool lo = dg >= 3;
          const int shift = dg == 0 ? 12 : dg == 1 ? 3 : dg == 2 ? 0 : dg == 3 ? 23 : dg == 4 ? 14 : dg == 5 ? 5 : 0;
          const uint32_t wm = dg == 2 ? 7u : dg == 6 ? 31u : 511u;
          for (int i = tid; i < kTkCandBins; i += kTkThreads) hist[i] = 0u;
          __syncthreads();  // (also orders the candidate writes before their reads)
          for (int j = tid; j < (int)nc; j += kTkThreads) {
            const int i = cand[j];
            const uint32_t h = keys[i];
            if (!lo) {
              if ((h & msk_hi) == pre_hi) atomicAdd(&hist[(h >> shift) & wm], 1u);
            } else if (h == pre_hi) {
              const uint32_t l = ~(uint32_t)src.gid(i);
              if ((l & msk_lo) == pre_lo) atomicAdd(&hist[(l >> shift) & wm], 1u);
            }
          }
          __syncthreads();
          tk_find_bin_w0<kTkCandBins>(hist, krem, sh);
          krem -= sh.above;
          if (!lo) {
            pre_hi |= sh.bin << shift;
            msk_hi |= wm << shift;
          } else {
            pre_lo |= sh.bin << shift;
            msk_lo |= wm << shift;
          }
          done = sh.binh == krem;  // (always by the last digit: keys differ)
          // (the next digit's clear follows its reads of sh and of the histogram: warp 0 read
          // the histogram before the barrier above, and sh is next written after two more)
        }
      } else {
        wide = true;
      }
    }
    if (search) {
      // the further digits over every entry: lists past the staging, or too many candidates
      for (int dg = 1; dg < 6 && wide && !done; ++dg) {
        const bool lo = dg >= 3;
        const int shift = dg % 3 == 1 ? 10 : dg % 3 == 2 ? 0 : 21;
        const int nb = dg % 3 == 2 ? 1024 : 2048;
        for (int i = tid; i < kTkBins; i += kTkThreads) hist[i] = 0u;
        __syncthreads();
        if (staged && !lo) {
          // a high-word digit over the staged keys: compile-time shifts, one 16-B load per
          // four keys, an atomic only for the keys still in play
          for (int c = 0; c < rounds; ++c) {
            const uint4 k4 = *reinterpret_cast<const uint4*>(keys + c * kTkRound + 4 * tid);
            const uint32_t h[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if ((h[e] & msk_hi) == pre_hi)
                atomicAdd(&hist[dg == 1 ? (h[e] >> 10) & 2047u : h[e] & 1023u], 1u);
          }
        } else {
          for (int c = 0; c < rounds; ++c) {
            const uint4 k4 = get4(c);
            const uint32_t h[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (!lo) {
                hist_add(hist, h[e], msk_hi, pre_hi, shift, nb);
              } else if (h[e] == pre_hi) {
                const uint32_t l = ~(uint32_t)src.gid(c * kTkRound + 4 * tid + e);
                if ((l & msk_lo) == pre_lo) atomicAdd(&hist[(l >> shift) & (nb - 1)], 1u);
              }
            }
          }
        }
        __syncthreads();
        if (nb == 2048)
          tk_find_bin<2048 / kTkThreads>(hist, krem, sh);
        else
          tk_find_bin<1024 / kTkThreads>(hist, krem, sh);
        krem -= sh.above;
        if (!lo) {
          pre_hi |= sh.bin << shift;
          msk_hi |= (uint32_t)(nb - 1) << shift;
        } else {
          pre_lo |= sh.bin << shift;
          msk_lo |= (uint32_t)(nb - 1) << shift;
        }
        done = sh.binh == krem;
        __syncthreads();  // every thread has read the bin before the histogram is cleared
      }
    }
    const uint32_t t_hi = pre_hi, t_lo = pre_lo;

    auto selected = [&](uint32_t h, int i) -> bool {
      return h != 0u && (h > t_hi || (h == t_hi && (t_lo == 0u || ~(uint32_t)src.gid(i) >= t_lo)));
    };
    const bool no_ties = t_lo == 0u;  // then the selection is key >= t_hi (t_hi >= 1)
    // write selected entry i (with key h) at output position pos (< k)
    auto emit = [&](int i, uint32_t h, uint32_t pos) {
      if (MERGE) {
        sorted[pos] = i;  // the entry; its id is loaded below, all at once
      } else {
        // the score from its key (exact; a zero is re-read, the key merges -0 and +0)
        p.cand_score[li * p.k + pos] = h == 0x80000000u ? src.score(i) : key_score(h);
        p.cand_idx[li * p.k + pos] = src.gid(i);
      }
    };
    if (staged) {
      // the candidates that reach T join the entries above the first digit's bin; then a
      // stable compaction: one block scan of the counts, each thread's entries in order
      for (uint32_t m = cmask; m != 0u; m &= m - 1u) {
        const int b = __ffs(m) - 1;
        if (selected(keys[e0 + b], e0 + b)) amask |= 1u << b;
      }
      uint32_t smask = amask;
      uint32_t total;
      uint32_t pos = tk_scan((uint32_t)__popc(smask), sh.ws, &total);
      // candidate lists with k <= kTkBins: the selected entries' indices go to the histogram's
      // words first, and are written out with consecutive threads on consecutive positions
      const bool via_smem = !MERGE && p.k <= kTkBins;
      int32_t* sel = reinterpret_cast<int32_t*>(hist);
      while (smask != 0u && pos < (uint32_t)p.k) {
        const int e = __ffs(smask) - 1;
        smask &= smask - 1u;
        const int i = e0 + e;
        if (via_smem)
          sel[pos++] = i;
        else
          emit(i, keys[i], pos++);
      }
      if (tid == 0) sh.base = total;
      __syncthreads();
      if (via_smem) {
        const int ns = (int)min(total, (uint32_t)p.k);
        for (int j = tid; j < ns; j += kTkThreads) {
          const int i = sel[j];
          emit(i, keys[i], (uint32_t)j);
        }
      }
    } else {
      // lists past the staging: the keys come from L2, in rounds; a block of kTkBlockRounds
      // rounds at a time: count per (round, warp), one scan, then each warp writes its entries
      // at positions found with ballots
      auto sel4 = [&](const uint4& k4, int i) -> uint32_t {  // bit e: entry i + e is selected
        if (no_ties)
          return (uint32_t)(k4.x >= t_hi) | (uint32_t)(k4.y >= t_hi) << 1 |
                 (uint32_t)(k4.z >= t_hi) << 2 | (uint32_t)(k4.w >= t_hi) << 3;
        return (uint32_t)selected(k4.x, i) | (uint32_t)selected(k4.y, i + 1) << 1 |
               (uint32_t)selected(k4.z, i + 2) << 2 | (uint32_t)selected(k4.w, i + 3) << 3;
      };
      if (tid == 0) sh.base = 0u;
      for (int c0 = 0; c0 < rounds; c0 += kTkBlockRounds) {
        const int nr = min(kTkBlockRounds, rounds - c0);
        uint32_t selmask = 0;  // 4 bits per round of the block
        for (int cr = 0; cr < nr; ++cr) {
          const int c = c0 + cr;
          const uint32_t m4 = sel4(get4(c), c * kTkRound + 4 * tid);
          selmask |= m4 << (4 * cr);
          const uint32_t wsum = __reduce_add_sync(0xffffffffu, (uint32_t)__popc(m4));
          if (lane == 0) sh.cw[cr][warp] = wsum;
        }
        __syncthreads();
        if (warp == 0) {  // exclusive scan of the block's (round, warp) counts in index order
          const int per = kTkBlockRounds * kTkWarps / 32;
          uint32_t v[kTkBlockRounds * kTkWarps / 32], run = 0;
#pragma unroll
          for (int j = 0; j < per; ++j) {
            const int q = lane * per + j;
            v[j] = q / kTkWarps < nr ? sh.cw[q / kTkWarps][q % kTkWarps] : 0u;
            run += v[j];
          }
          uint32_t x = run;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
          }
          uint32_t pos = sh.base + x - run;
#pragma unroll
          for (int j = 0; j < per; ++j) {
            const int q = lane * per + j;
            sh.off[q / kTkWarps][q % kTkWarps] = pos;
            pos += v[j];
          }
          const uint32_t total = __shfl_sync(0xffffffffu, x, 31);
          __syncwarp();
          if (lane == 0) sh.base += total;
        }
        __syncthreads();
        const uint32_t lt = (1u << lane) - 1u;
        for (int cr = 0; cr < nr; ++cr) {
          const int c = c0 + cr;
          const uint32_t m4 = (selmask >> (4 * cr)) & 15u;
          // entries of lower lanes come first, then this lane's in order
          uint32_t pos = sh.off[cr][warp];
#pragma unroll
          for (int e = 0; e < 4; ++e) pos += __popc(__ballot_sync(0xffffffffu, (m4 >> e) & 1u) & lt);
          if (m4 == 0u) continue;
          const int i = c * kTkRound + 4 * tid;
          const uint4 k4 = get4(c);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (((m4 >> e) & 1u) && pos < (uint32_t)p.k)
              emit(i + e, e == 0 ? k4.x : e == 1 ? k4.y : e == 2 ? k4.z : k4.w, pos);
            pos += (m4 >> e) & 1u;
          }
        }
        __syncthreads();  // the offsets are read before the next block rewrites them
      }
    }
    const int cnt = (int)min(sh.base, (uint32_t)p.k);

    if constexpr (!MERGE) {
      for (int j = cnt + tid; j < p.k; j += kTkThreads) {
        p.cand_score[li * p.k + j] = -INFINITY;
        p.cand_idx[li * p.k + j] = -1;
      }
    } else {
      // sorted[0, cnt) holds the selected entries in index order: shard d's list is the run
      // of entries in [d * kin, (d + 1) * kin).  First the run boundaries, then the ids.
      if (tid <= p.D) {
        const int target = tid * p.stride;
        int lo = 0, hi = cnt;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (sorted[mid] < target) lo = mid + 1; else hi = mid;
        }
        sh.run[tid] = lo;
      }
      if (tid == 0) sh.maxid = -1;
      __syncthreads();
      int mx = -1;
      bool pad = false;
      for (int j0 = tid; j0 < cnt; j0 += 4 * kTkThreads) {  // four id loads in flight
        int id[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u * kTkThreads;
          id[u] = j < cnt ? src.gid(sorted[j]) : -1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u * kTkThreads;
          if (j < cnt) {
            sorted[j] = id[u];
            pad |= id[u] < 0;
          }
          mx = max(mx, id[u]);
        }
      }
      if (__syncthreads_or(pad && !exact)) continue;  // a padding entry was selected
      mx = __reduce_max_sync(0xffffffffu, mx);
      if (lane == 0 && mx >= 0) atomicMax(&sh.maxid, mx);
      __syncthreads();
      int32_t* out = p.topk + li * p.k;
      // ids below 32 x the staging's words: a bitmap of the selected ids over the staging (free
      // now) gives their increasing order directly -- each thread counts the set bits of its
      // words, one scan, and writes its ids in order.  Not taken when an id repeats (another
      // shard's list held it too): then the runs are merged as below.
      const int nw = (sh.maxid >> 5) + 1;
      if (runs_inside && sh.maxid >= 0 && nw <= p.stage) {
        uint32_t* bm = keys;
        for (int w = tid; w < nw; w += kTkThreads) bm[w] = 0u;
        __syncthreads();
        bool dup = false;
        for (int j = tid; j < cnt; j += kTkThreads) {
          const int id = sorted[j];
          const uint32_t bit = 1u << (id & 31);
          dup |= (atomicOr(&bm[id >> 5], bit) & bit) != 0u;
        }
        if (!__syncthreads_or(dup)) {
          const int W = (nw + kTkThreads - 1) / kTkThreads;
          const int w0 = min(tid * W, nw), w1 = min(w0 + W, nw);
          uint32_t c = 0;
          for (int w = w0; w < w1; ++w) c += __popc(bm[w]);
          uint32_t total;
          uint32_t pos = tk_scan(c, sh.ws, &total);
          for (int w = w0; w < w1; ++w) {
            uint32_t b = bm[w];
            while (b != 0u) {
              out[pos++] = 32 * w + __ffs(b) - 1;
              b &= b - 1u;
            }
          }
          for (int j = cnt + tid; j < p.k; j += kTkThreads) out[j] = -1;
          if (tid == 0 && p.count) p.count[li] = cnt;
          return;
        }
      }
      // runs in increasing id order (as dcp_topk_local writes its lists): merged pairwise
      bool unsorted = false;  // a pair inside a run out of order (pairs across runs may descend)
      for (int j = tid; j + 1 < cnt; j += kTkThreads) {
        int lo = 0, hi = p.D;  // the run of entry j + 1: the last d with run[d] <= j + 1
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (sh.run[mid] <= j + 1) lo = mid; else hi = mid - 1;
        }
        unsorted |= sh.run[lo] != j + 1 && sorted[j] >= sorted[j + 1];
      }
      if (!__syncthreads_or(unsorted)) {
        // merge the runs pairwise, ceil(log2 D) levels between sorted[] and a second buffer,
        // the last level into the output: each thread takes a slice of the output, finds
        // where its pair's two runs stand at the slice start (a merge-path binary search) and
        // merges sequentially from there
        int32_t* src_b = sorted;
        int32_t* dst_b = sorted2;
        int nr = p.D;
        const int E = (cnt + kTkThreads - 1) / kTkThreads;
        if (nr == 1) {
          for (int j = tid; j < cnt; j += kTkThreads) out[j] = src_b[j];
        }
        while (nr > 1) {
          const bool last = nr <= 2;
          const int np = (nr + 1) / 2;  // pairs; the last may hold one run
          const int o0 = tid * E, o1 = min(cnt, o0 + E);
          if (o0 < o1) {
            int q = 0, hi = np - 1;  // the pair holding output o0: last q with run[2q] <= o0
            while (q < hi) {
              const int mid = (q + hi + 1) >> 1;
              if (sh.run[2 * mid] <= o0) q = mid; else hi = mid - 1;
            }
            int ps = sh.run[2 * q], pm = sh.run[min(2 * q + 1, nr)], pe = sh.run[min(2 * q + 2, nr)];
            const int d = o0 - ps;
            int lo = max(0, d - (pe - pm)), up = min(d, pm - ps);
            while (lo < up) {
              const int mid = (lo + up) >> 1;
              if (src_b[ps + mid] < src_b[pm + d - mid - 1]) lo = mid + 1; else up = mid;
            }
            int ia = ps + lo, ib = pm + d - lo;
            for (int o = o0; o < o1; ++o) {
              while (o == pe && q + 1 < np) {  // the slice runs on into the next (non-empty) pair
                ++q;
                ps = sh.run[2 * q];
                pm = sh.run[min(2 * q + 1, nr)];
                pe = sh.run[min(2 * q + 2, nr)];
                ia = ps;
                ib = pm;
              }
              const int v = (ib >= pe || (ia < pm && src_b[ia] < src_b[ib])) ? src_b[ia++] : src_b[ib++];
              if (last) out[o] = v; else dst_b[o] = v;
            }
          }
          __syncthreads();
          if (tid == 0) {  // the merged runs' boundaries
            for (int r = 0; r < np; ++r) sh.run[r] = sh.run[2 * r];
            sh.run[np] = cnt;
          }
          __syncthreads();
          int32_t* t = src_b;
          src_b = dst_b;
          dst_b = t;
          nr = np;
        }
        for (int j = cnt + tid; j < p.k; j += kTkThreads) out[j] = -1;
      } else {
        // any order: bitonic sort over p.kp >= k entries
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
        for (int j = tid; j < p.k; j += kTkThreads) out[j] = j < cnt ? sorted[j] : -1;
      }
      if (tid == 0 && p.count) p.count[li] = cnt;
    }
    return;
  }
}

namespace {
size_t tk_smem_bytes(int stage, int kp) { return (size_t)(kTkBins + stage + kp) * 4; }

template <bool MERGE>
cudaError_t tk_launch(const TopkParams& p, int64_t lists, cudaStream_t st) {
  // merge: two run buffers, past the staging when they do not fit inside (see the kernel)
  const size_t smem = tk_smem_bytes(p.stage, MERGE && p.kp > kTkBins ? 2 * p.kp : 0);
  cudaError_t e = raise_smem_limit((const void*)topk_kernel<MERGE>, smem);
  if (e != cudaSuccess) return e;
  topk_kernel<MERGE><<<(unsigned)lists, kTkThreads, smem, st>>>(p);
  return cudaGetLastError();
}
}  // namespace

// entries staged per list: the longest list, at most kTkStageMax, in whole rounds
int tk_stage(int64_t n_max) {
  const int64_t s = n_max < kTkStageMax ? n_max : kTkStageMax;
  return (int)((s + kTkRound - 1) / kTkRound * kTkRound);
}

cudaError_t launch_topk_local(TopkParams p, int n_in, cudaStream_t st) {
  if (p.rows == 0) return cudaSuccess;
  p.stage = tk_stage(p.stride);
  p.kp = 0;
  p.div = make_fastdiv(p.I);
  return tk_launch<false>(p, p.rows * n_in, st);
}

cudaError_t launch_topk_merge(TopkParams p, cudaStream_t st) {
  if (p.rows == 0) return cudaSuccess;
  p.stage = tk_stage((int64_t)p.D * p.stride);
  p.div = make_fastdiv(p.stride);
  int kp = 1;
  while (kp < p.k) kp <<= 1;
  p.kp = kp;
  return tk_launch<true>(p, p.rows, st);
}

}  // namespace dcp

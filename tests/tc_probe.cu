// Test-only probe of the tcgen05 building blocks used by the tensor-core decode kernel:
// one CTA of 128 threads computes D[128 x N] = A[128 x K] * B with
//   mode 0: A in TMEM, B K-major (B given as [N][K] row-major)   -- the Q.K^T form
//   mode 1: A in TMEM, B MN-major (B given as [K][N] row-major)  -- the P.V form
//   mode 2: A in shared memory K-major, B K-major
//   mode 3: A in shared memory K-major, B MN-major                -- the P.V form, P in smem
// and a conversion probe for the exact E4M3 -> bf16 (x 2^-112) path, a wait that nothing
// satisfies, for the bounded mbarrier wait's time limit, and the TMEM layout of an M = 64
// MMA's result.
// Shapes accepted by tc_probe: K in {64, 128} (modes 0, 2) or {16, 32, 64, 128} (modes 1, 3),
// N a multiple of 16 in [16, 256] (modes 0, 2) or of 64 in [64, 256] (modes 1, 3).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../decode_context_sparse_gb300/csrc/tc_ptx.cuh"

using namespace dcp::tc;

constexpr int kSmemB = 65536, kSmemA = 32768;

__global__ void __launch_bounds__(128) tc_probe_kernel(const uint16_t* __restrict__ A,
                                                       const uint16_t* __restrict__ B,
                                                       float* __restrict__ D, int K, int N,
                                                       int mode, int* err) {
  extern __shared__ unsigned char sm_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* sB = sm;
  unsigned char* sA = sm + kSmemB;
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  const bool b_mn = mode == 1 || mode == 3, a_smem = mode == 2 || mode == 3;
  if (b_mn) {  // [N/64 groups][K rows][128 B], swizzled
    for (int i = tid; i < K * (N / 8); i += 128) {
      const int k = i / (N / 8), c8 = i % (N / 8), blk = c8 / 8, c = c8 % 8;
      const uint4 v = *reinterpret_cast<const uint4*>(B + (size_t)k * N + c8 * 8);
      *reinterpret_cast<uint4*>(sB + blk * (K * 128) + k * 128 + ((c ^ (k & 7)) * 16)) = v;
    }
  } else {  // [K/64 groups][N rows][128 B], swizzled
    for (int i = tid; i < N * (K / 8); i += 128) {
      const int n = i / (K / 8), c8 = i % (K / 8), blk = c8 / 8, c = c8 % 8;
      const uint4 v = *reinterpret_cast<const uint4*>(B + (size_t)n * K + c8 * 8);
      *reinterpret_cast<uint4*>(sB + blk * (N * 128) + n * 128 + ((c ^ (n & 7)) * 16)) = v;
    }
  }
  if (a_smem) {  // A: [K/64 groups][128 rows][128 B], swizzled (K < 64: part of each row)
    for (int i = tid; i < 128 * (K / 8); i += 128) {
      const int m = i / (K / 8), c8 = i % (K / 8), blk = c8 / 8, c = c8 % 8;
      const uint4 v = *reinterpret_cast<const uint4*>(A + (size_t)m * K + c8 * 8);
      *reinterpret_cast<uint4*>(sA + blk * (128 * 128) + m * 128 + ((c ^ (m & 7)) * 16)) = v;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  if (!a_smem) {  // row tid of A into TMEM columns [0, K/2)
    const uint32_t* arow = reinterpret_cast<const uint32_t*>(A + (size_t)tid * K);
    for (int c = 0; c < K / 2; c += 8) {
      uint32_t r[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) r[i] = arow[c + i];
      tmem_st8(tbase + lane_off + c, r);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint32_t d_tmem = tbase + 256;
    const uint32_t idesc = idesc_bf16(128, N, 0, b_mn ? 1 : 0);
    for (int ks = 0; ks < K / 16; ++ks) {
      uint64_t bdesc;
      if (b_mn)
        bdesc = smem_desc(smem_u32(sB) + ks * 2048, K * 128, 1024);
      else
        bdesc = smem_desc(smem_u32(sB) + (ks / 4) * (N * 128) + (ks % 4) * 32, 16, 1024);
      if (a_smem) {
        const uint64_t adesc = smem_desc(smem_u32(sA) + (ks / 4) * (128 * 128) + (ks % 4) * 32, 16, 1024);
        mma_ss(d_tmem, adesc, bdesc, idesc, ks > 0);
      } else {
        mma_ts(d_tmem, tbase + ks * 8, bdesc, idesc, ks > 0);
      }
    }
    mma_commit(&bar);
  }
  __syncwarp();
  const bool ok = mbar_wait(&bar, 0, &abort_flag);
  tc_fence_after();
  if (!ok) {
    if (tid == 0) atomicOr(err, 1);
  } else {
    for (int c = 0; c < N; c += 16) {
      uint32_t r[16];
      tmem_ld16(tbase + lane_off + 256 + c, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) D[(size_t)tid * N + c + i] = __uint_as_float(r[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

__global__ void e4m3_probe_kernel(const uint16_t* codes, uint32_t* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = e4m3x2_to_bf16x2_scaled(codes[i]);
}

__global__ void e4m3x4_probe_kernel(const uint32_t* words, uint2* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = e4m3x4_to_bf16x4(words[i]);
}

extern "C" int e4m3x4_probe(const void* words, void* out, int n) {
  e4m3x4_probe_kernel<<<(n + 255) / 256, 256>>>(static_cast<const uint32_t*>(words),
                                                 static_cast<uint2*>(out), n);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

extern "C" int tc_probe(const void* A, const void* B, float* D, int K, int N, int mode, int* err) {
  const bool kmaj = mode == 0 || mode == 2;
  if (mode < 0 || mode > 3) return -1;
  if (kmaj && !(K == 64 || K == 128)) return -1;
  if (!kmaj && !(K == 16 || K == 32 || K == 64 || K == 128)) return -1;
  if (kmaj && (N < 16 || N > 256 || N % 16)) return -1;
  if (!kmaj && (N < 64 || N > 256 || N % 64)) return -1;
  const int smem = kSmemB + kSmemA + 1024;
  if (cudaFuncSetAttribute(tc_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -3;
  tc_probe_kernel<<<1, 128, smem>>>(static_cast<const uint16_t*>(A),
                                    static_cast<const uint16_t*>(B), D, K, N, mode, err);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

extern "C" int e4m3_probe(const void* codes, void* out, int n) {
  e4m3_probe_kernel<<<(n + 255) / 256, 256>>>(static_cast<const uint16_t*>(codes),
                                               static_cast<uint32_t*>(out), n);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

// Two threads wait on an mbarrier nothing arrives on, with the bounded wait the kernels use:
// the first gives up after the time limit and sets the abort flag, the second sees the flag
// and gives up too; the kernel then finishes (no trap, no endless loop).
// out[0] = waits that returned false, out[1] = the abort flag, out[2] = elapsed ms.
__global__ void wait_timeout_kernel(int* out) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t t0 = globaltimer();
  __shared__ int gave_up;
  if (threadIdx.x == 0) gave_up = 0;
  __syncthreads();
  if ((threadIdx.x & 31) == 0 && !mbar_wait(&bar, 0, &abort_flag)) atomicAdd(&gave_up, 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    out[0] = gave_up;
    out[1] = abort_flag;
    out[2] = (int)((globaltimer() - t0) / 1000000ull);
  }
}

extern "C" int wait_timeout_probe(int* out) {
  wait_timeout_kernel<<<1, 64>>>(out);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}


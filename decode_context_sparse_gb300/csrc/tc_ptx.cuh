// Inline-PTX wrappers for the sm_100-family (sm_103a) tensor-core path: mbarriers,
// tensor memory (TMEM) allocation / loads / stores, tcgen05.mma with A in TMEM or in
// shared memory, shared-memory matrix descriptors, bulk async copies, clusters.
//
// Layout facts used throughout (PTX ISA, tcgen05 "matrix descriptors" and data paths):
//  * SWIZZLE_128B atoms are 8 rows x 128 B (1024 B, 1024-B aligned); 16-B chunk c of row r
//    is stored at chunk position c ^ (r & 7).
//  * K-major operand (rows = M or N, 64 bf16 of K per 128-B row): SBO = byte stride between
//    8-row groups, LBO unused; one MMA k-step (16 bf16 = 32 B) advances the start address by
//    32 B inside the atom.
//  * MN-major operand (rows = K, 64 bf16 of M/N per 128-B row): LBO = byte stride between
//    64-element groups along M/N, SBO = byte stride between 8-row groups along K.
//  * An M = 128 accumulator occupies TMEM lanes 0..127 (row i -> lane i), one fp32 per
//    column; an A operand in TMEM holds row i in lane i with two bf16 per column (even k in
//    the low half).  Warp w of a warpgroup may only touch lanes 32*(w%4) .. 32*(w%4)+31.
#pragma once

#include <stdint.h>

namespace dcp {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(tx)
               : "memory");
}
// Arrive on the barrier at the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint64_t* bar, uint32_t rank) {
  asm volatile(
      "{\n .reg .b32 ra;\n mapa.shared::cluster.u32 ra, %0, %1;\n"
      " mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n}" ::"r"(smem_u32(bar)),
      "r"(rank)
      : "memory");
}
// Relaxed remote arrive: no ordering of this thread's earlier memory operations.  Used to
// hand back buffers whose contents this thread has already read (and consumed).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint64_t* bar, uint32_t rank) {
  asm volatile(
      "{\n .reg .b32 ra;\n mapa.shared::cluster.u32 ra, %0, %1;\n"
      " mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [ra];\n}" ::"r"(smem_u32(bar)),
      "r"(rank)
      : "memory");
}
// try_wait with a suspend-time hint: a thread whose phase is not complete sleeps until it
// completes or the hint (ns) runs out, instead of returning at once to spin.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Non-blocking test of a phase (never suspends): for issuers that poll several barriers.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait.  Gives up after `limit_ns` of wall time or as soon as *abort is set;
// returns false in both cases (the caller then winds down).
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag, bool cluster_scope = false) {
  if (cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      return false;
    }
  }
}

// Bring the 128-B line holding addr into L2 (no register result, nothing to wait for).
__device__ __forceinline__ void prefetch_l2(const void* addr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(addr));
}

// ------------------------------------------------------------------ proxies / fences
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------ TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32x32b shape: lane i of the warp reads/writes TMEM lane (lane field of taddr) + i, N
// consecutive 32-bit columns starting at the column field of taddr.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// ------------------------------------------------------------------ MMA
// Instruction descriptor, kind::f16: BF16 A and B, FP32 accumulator, M x N, A/B K-major
// (0) or MN-major (1).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::f16: FP16 A and B, FP32 accumulator (A/B type fields 0).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

constexpr uint32_t kLayoutSW128 = 2;
// Shared-memory matrix descriptor (sm_100 format, version bit 46).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout = kLayoutSW128) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= (uint64_t)layout << 61;
  return d;
}

// D(tmem) (+)= A(smem desc) * B(smem desc)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem desc)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Warp-collective forms: every lane of a converged warp executes them with the same
// (warp-uniform) operands and one elected lane issues the instruction.
__device__ __forceinline__ void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// One elected lane of the (converged) warp: 1 in that lane, 0 elsewhere.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n selp.u32 %0, 1, 0, e;\n}"
      : "=r"(r));
  return r;
}
// Issued only where `leader` is non-zero; every lane passes the same operands.
__device__ __forceinline__ void mma_ts_if(uint32_t leader, uint32_t d_tmem, uint32_t a_tmem,
                                          uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 e, %5, 0;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
__device__ __forceinline__ void mma_ss_if(uint32_t leader, uint32_t d_tmem, uint64_t a_desc,
                                          uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 e, %5, 0;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
__device__ __forceinline__ void mma_commit_if(uint32_t leader, uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n setp.ne.b32 e, %1, 0;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(
          smem_u32(bar)),
      "r"(leader)
      : "memory");
}
__device__ __forceinline__ void mma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(
          smem_u32(bar))
      : "memory");
}
// Arrive once on `bar` when every previously issued tcgen05 op of this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ bulk copies
// Global -> own shared memory, completion counted in bytes on `bar`.  src, dst 16-B
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Four-row TMA gather (2-D tensor map with a one-row box): rows y0..y3 of the tensor, box
// columns [x, x + box width), land back to back at dst (128-B aligned); completion counted
// in bytes on `bar`.  x * element size must be a multiple of 16 B.
__device__ __forceinline__ void tma_gather4(void* dst, const void* tmap, int x, int y0, int y1,
                                            int y2, int y3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar))
      : "memory");
}
// Tiled store of a shared-memory box (1024-B aligned for a swizzled map) to the 3-D tensor
// `tmap` at element coordinates (x, y, z), as a bulk group of this thread; parts of the box
// outside the tensor are not written.  x * element size must be a multiple of 16 B.
__device__ __forceinline__ void tma_store_3d(const void* tmap, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::
                   "l"(tmap), "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Per-thread 16-B asynchronous copy global -> shared (L2 only), tracked by cp.async groups.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed (the arrival is
// counted in the barrier's initial count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ------------------------------------------------------------------ cluster
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Shared memory of this CTA -> the mirrored address in CTA `rank` of the cluster (bytes a
// multiple of 16, both ends 16-B aligned), completion counted in bytes on the barrier
// mirroring `bar` in that CTA.  The source may be reused after bulk_wait_read0().
__device__ __forceinline__ void bulk_s2peer(void* dst_mirror, const void* src, uint32_t bytes,
                                            uint32_t rank, uint64_t* bar) {
  asm volatile(
      "{\n .reg .b32 rd, rb;\n mapa.shared::cluster.u32 rd, %0, %3;\n"
      " mapa.shared::cluster.u32 rb, %4, %3;\n"
      " cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [rd], [%1], %2, [rb];\n}" ::
          "r"(smem_u32(dst_mirror)),
      "r"(smem_u32(src)), "r"(bytes), "r"(rank), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// At most N of this thread's bulk-copy groups may still be reading their sources.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ conversions
// Two E4M3 codes (lower code in the lower half) -> f16x2 of the same values, exactly (every
// E4M3 value is an FP16 value), each multiplied by the f16x2 `mul` (a power of two or 0;
// the product is exact while it stays in FP16's normal range).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_mul(uint16_t codes, uint32_t mul) {
  uint32_t h2, r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h2), "r"(mul));
  return r;
}
// Two floats -> f16x2 (a in the lower half), round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
// Two bf16 (a word: lower value in the lower half) times a power of two -> f16x2.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_mul(uint32_t w, float mul) {
  return pack_f16x2(__uint_as_float(w << 16) * mul, __uint_as_float(w & 0xffff0000u) * mul);
}

// Two E4M3 codes -> two bf16 holding value * 2^-112, exactly: the hardware E4M3 -> F16
// conversion is exact and every non-zero E4M3 value is a normal f16 with at most three
// mantissa bits, so shifting the f16 magnitude bits right by three re-reads them as a
// normal bf16 whose exponent bias is 112 larger (zero stays zero).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_scaled(uint16_t codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  return ((h2 >> 3) & 0x0FFF0FFFu) | (h2 & 0x80008000u);
}
// Four E4M3 codes (the bytes of x, lowest first) -> four bf16 of the same values, exactly,
// two per word (lower code in the lower half), with integer operations only.  Each code's
// four exponent and three mantissa bits are placed in the bf16 exponent field (low four
// bits) and the top of its mantissa, the sign bit on the sign: a bf16 of value * 2^-120 for
// every code (E4M3 subnormals, exponent 0, become bf16 subnormals with the same factor),
// which a power-of-two product then brings back exactly.  The byte permute replicates each
// code's sign over the byte above it (selector nibbles with bit 3 set), so one shift and one
// mask place both codes of a word half.
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t x) {
  uint32_t a, b;  // [code, sign x 8, code, sign x 8] for codes 0,1 and 2,3
  asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(a) : "r"(x));
  asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(b) : "r"(x));
  const uint32_t ia = (a << 4) & 0x87F087F0u;
  const uint32_t ib = (b << 4) & 0x87F087F0u;
  uint2 r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r.x) : "r"(ia), "r"(0x7B807B80u));  // * 2^120
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r.y) : "r"(ib), "r"(0x7B807B80u));
  return r;
}


}  // namespace tc
}  // namespace dcp

// Device helpers shared by the kernels: status reporting, bf16 bit handling, and
// inline-PTX wrappers for mbarriers, TMA (cp.async.bulk.tensor) and the 5th
// generation tensor cores (tcgen05: TMEM allocation, MMA, commit, loads).
//
// Every mbarrier wait here is bounded: after TW_WAIT_LIMIT_NS of polling it raises
// TW_ETIMEOUT in the caller's status word, sets a CTA-wide abort flag and returns
// false, so no kernel of this library can spin forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include "../../include/twell.h"

#define TW_DEV __device__ __forceinline__

#ifndef TW_WAIT_LIMIT_NS
#define TW_WAIT_LIMIT_NS 1000000000ull  // 1 s
#endif

namespace tw {

// ------------------------------------------------------------------ status
// Programmatic dependent launch: wait until the grids this one depends on have
// completed and their writes are visible; then let the next grid start its launch.
TW_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
TW_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
TW_DEV void pdl_enter() {
  pdl_wait();
  pdl_trigger();
}

TW_DEV void raise_status(int32_t* status, int code) {
  if (status != nullptr) atomicMax(status, code);
}

// ------------------------------------------------------------------ checked builds
// A build with -DTW_CHECK compares every index that a kernel computes from data it
// reads (neuron indices of the formats, token rows of the row gathers and scatters,
// record slots of the transposed Hybrid, counts that size a loop) with the size of
// the buffer it addresses. TW_CHECKED(cond, status) is then false when the index
// does not fit: TW_EBOUNDS is raised in *status (when non-null), the first few
// violations of each translation unit print their source line, and the caller skips
// the access. Without TW_CHECK it is the constant true and costs nothing.
#ifdef TW_CHECK
static __device__ unsigned int tw_check_prints;
TW_DEV bool check_bound(bool ok, int32_t* status, const char* file, int line) {
  if (!ok) {
    raise_status(status, TW_EBOUNDS);
    if (atomicAdd(&tw_check_prints, 1u) < 16u) printf("TW_CHECK: index out of bounds at %s:%d\n", file, line);
  }
  return ok;
}
#define TW_CHECKED(cond, status) (::tw::check_bound((cond), (status), __FILE__, __LINE__))
#else
#define TW_CHECKED(cond, status) (true)
#endif

// ------------------------------------------------------------------ bf16 bits
TW_DEV float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
TW_DEV float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }
TW_DEV float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
TW_DEV uint16_t f32_to_bf16(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
TW_DEV uint32_t pack_bf16x2(float lo, float hi) {
  return static_cast<uint32_t>(f32_to_bf16(lo)) | (static_cast<uint32_t>(f32_to_bf16(hi)) << 16);
}
// the same with one paired conversion (round to nearest even on both halves)
TW_DEV uint32_t pack_bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}
// fp16 (IEEE binary16) bits: the Hybrid's stored u and the dense route's backward
// operands, which need 11 significant bits where bf16 has 8
TW_DEV uint16_t f32_to_f16(float v) { return __half_as_ushort(__float2half_rn(v)); }
TW_DEV float f16_to_f32(uint16_t b) { return __half2float(__ushort_as_half(b)); }
TW_DEV uint32_t pack_f16x2_rn(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ------------------------------------------------------------------ packed fp32 pairs
// Two fp32 lanes in one 64-bit register, the operand form of Blackwell's packed
// `fma.rn.f32x2`, which the CUDA-core accumulations use (half the FMA instructions).
typedef unsigned long long f32x2;
TW_DEV f32x2 pair(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
TW_DEV float2 unpair(f32x2 v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return make_float2(lo, hi);
}
// acc += a * b on both lanes (round to nearest even, one rounding per lane)
TW_DEV void fma2(f32x2& acc, f32x2 a, f32x2 b) { asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b)); }
// a packed bf16 pair (low half = element 0) widened exactly to two fp32 lanes
TW_DEV f32x2 widen(uint32_t w) { return pair(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)); }
// A 16-byte read-only load through the non-coherent path (the gathers' row slices).
TW_DEV uint4 ldg16(const uint4* p) { return __ldg(p); }

// ------------------------------------------------------------------ smem / timers
TW_DEV uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
TW_DEV uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
TW_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
TW_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
TW_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
TW_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
TW_DEV bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete. Returns false when the CTA
// is aborting (flag set by any thread) or when this wait exceeded the time limit
// (then it sets the flag and raises TW_ETIMEOUT).
TW_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int32_t* status) {
  const uint32_t addr = smem_addr(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((n & 31u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > TW_WAIT_LIMIT_NS) {
        *abort_flag = 1;
        raise_status(status, TW_ETIMEOUT);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ TMA
TW_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2D tiled load of one box into shared memory; completion is signalled on `bar`
// as transaction bytes. c0 is the innermost coordinate (elements), c1 the row.
TW_DEV void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
      : "memory");
}
// The same load for a CTA of a pair: completion is signalled on the barrier at
// `bar_cluster` (a shared::cluster address, here the pair's rank-0 barrier).
TW_DEV void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar_cluster, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}


// Bounded wait used only while draining after an abort: ignores the abort flag.
TW_DEV bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_addr(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(addr, parity)) {
    if (global_timer_ns() - t0 > TW_WAIT_LIMIT_NS) return false;
  }
  return true;
}


// ------------------------------------------------------------------ tcgen05
// TMEM allocation: executed by one whole warp. The allocated base address is
// written to *smem_dst.
TW_DEV void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(smem_dst)),
               "r"(ncols)
               : "memory");
}
TW_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
TW_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
TW_DEV void tc_fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
TW_DEV void tc_fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulation, one thread issues.
TW_DEV void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on `bar` when every tcgen05 operation this thread issued so far is done.
TW_DEV void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}
TW_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ CTA pairs (cta_group::2)
// Two CTAs of a cluster share each MMA: the pair's accumulator tile is 256 rows, the
// first 128 in rank 0's TMEM and the next 128 in rank 1's, and each CTA holds its own
// A rows and half of the B tile in shared memory at the same offsets. Rank 0 issues
// the MMAs. Allocation, its permit and deallocation are done by one warp of each CTA.
TW_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of both CTAs; orders the shared-memory writes before it (barrier
// initialisation, the TMEM address) for the other CTA.
TW_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of the variable at `p` (this CTA's shared memory) in
// the cluster's CTA `rank`.
TW_DEV uint32_t peer_smem_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
TW_DEV void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
TW_DEV void tmem_alloc_pair(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(smem_dst)),
               "r"(ncols)
               : "memory");
}
TW_DEV void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
TW_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// The pair's MMA: D rows [0, 128) into rank 0's TMEM at d_tmem and rows [128, 256)
// into rank 1's; A and B descriptors address this CTA's shared memory, the other
// CTA's operand halves sit at the same offsets.
TW_DEV void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the barrier at `bar`'s offset in both CTAs of the pair when every
// tcgen05 operation this thread issued so far is done.
TW_DEV void tc_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// Each lane of the warp reads 32 consecutive fp32 columns of its own TMEM lane.
TW_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Shared-memory matrix descriptor for a 128-byte-swizzled bf16 operand tile
// (sm_100 family layout: start address >> 4 in bits 0-13, leading byte offset >> 4
// in bits 16-29, stride byte offset >> 4 in bits 32-45, descriptor version 1 in
// bits 46-47, swizzle mode 2 = 128B in bits 61-63).
//  K-major tiles: rows of 128 bytes (64 bf16 along K), 8-row groups 1024 bytes apart
//    (SBO = 1024); the leading offset is unused.
//  MN-major tiles: 64 contiguous MN elements (128 bytes) per K row, 8-row K groups
//    1024 bytes apart (SBO), 64-element MN chunks LBO bytes apart.
TW_DEV uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: A and B both bf16 (or, with f16,
// both fp16), fp32 D.
//  bits 4-5 D format (1 = f32), 7-9 A format and 10-12 B format (0 = f16, 1 = bf16),
//  bit 15 A major (1 = MN), bit 16 B major (1 = MN), bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn, bool f16 = false) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------ warp helpers
TW_DEV int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

}  // namespace tw

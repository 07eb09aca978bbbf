// CUDA-core kernels of the backward's column side (gist.science explainer, 2.B:
// "Sparse MatMul" and "Backpropagation"): the transposed Hybrid (per-neuron columns
// of the ELL entries) and the weight gradients accumulated over it,
//   dWg[j] = sum dg x_t,  dWu[j] = sum du x_t,  dWd[j] = sum h dy_t  (h = a u),
// plus the backward's launcher. The token side (dh, dg, du, dx) is in tw_token.cu.
//
// Every column entry costs gathers of token-row slices (x_t, dy_t) from the 129 MB
// L2; they are loaded straight into registers, several per warp in flight.
#include <algorithm>

#include "tw_common.cuh"
#include "tw_internal.h"

namespace tw {

namespace {

constexpr int kWgradUnroll = 8;

// ---------------------------------------------------------------- row arithmetic
// The accumulation is bound by instruction issue, so it uses Blackwell's packed
// fp32x2 FMA. Eight fp32 accumulators live as four packed pairs.
struct F8 {
  f32x2 v[4];
};
TW_DEV void f8_zero(F8& a) { a.v[0] = a.v[1] = a.v[2] = a.v[3] = 0ull; }
// y += h * w over 8 bf16 elements (h2 = {h, h})
TW_DEV void axpy8(F8& y, f32x2 h2, const uint4& w) {
  fma2(y.v[0], h2, widen(w.x));
  fma2(y.v[1], h2, widen(w.y));
  fma2(y.v[2], h2, widen(w.z));
  fma2(y.v[3], h2, widen(w.w));
}
// g += cg * x and u += cu * x sharing one conversion of x
TW_DEV void axpy8_two(F8& g, f32x2 cg2, F8& u, f32x2 cu2, const uint4& x) {
  const f32x2 x0 = widen(x.x), x1 = widen(x.y), x2 = widen(x.z),
              x3 = widen(x.w);
  fma2(g.v[0], cg2, x0);
  fma2(g.v[1], cg2, x1);
  fma2(g.v[2], cg2, x2);
  fma2(g.v[3], cg2, x3);
  fma2(u.v[0], cu2, x0);
  fma2(u.v[1], cu2, x1);
  fma2(u.v[2], cu2, x2);
  fma2(u.v[3], cu2, x3);
}
TW_DEV void stcs_f32x8(float* p, const F8& y) {
  const float2 a = unpair(y.v[0]), b = unpair(y.v[1]), c = unpair(y.v[2]), d = unpair(y.v[3]);
  __stcs(reinterpret_cast<float4*>(p), make_float4(a.x, a.y, b.x, b.y));
  __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(c.x, c.y, d.x, d.y));
}
// y added into p with fp32 vector reductions (the L2 does the adds; no round trip)
TW_DEV void red_f32x8(float* p, const F8& y) {
  const float2 a = unpair(y.v[0]), b = unpair(y.v[1]), c = unpair(y.v[2]), d = unpair(y.v[3]);
  atomicAdd(reinterpret_cast<float4*>(p), make_float4(a.x, a.y, b.x, b.y));
  atomicAdd(reinterpret_cast<float4*>(p) + 1, make_float4(c.x, c.y, d.x, d.y));
}
TW_DEV void out_f32x8(float* p, const F8& y, bool add) {
  if (add)
    red_f32x8(p, y);
  else
    stcs_f32x8(p, y);
}
constexpr int kCountHistMaxBins = 48 * 1024;  // 192 KB of shared memory
template <class K>
cudaError_t set_smem_bytes(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}
int grid_for(long items, int per_block, int blocks_per_sm) {
  const long blocks = (items + per_block - 1) / per_block;
  return static_cast<int>(
      std::max<long>(1, std::min<long>(blocks, static_cast<long>(device_sm_count()) * blocks_per_sm)));
}


}  // namespace

// ====================================================================== transposed Hybrid
// Exclusive scan of the per-neuron counts: col_ptr[0..I], col_cur = col_ptr. The CTA
// walks the counts in chunks of 16 x blockDim neurons; each thread takes 16
// consecutive counts (four 16-byte loads, issued together, when I is a multiple of
// 4), so a chunk costs one round trip to memory instead of one per count.
TW_DEV void scan_counts(const int32_t* __restrict__ col_cnt, int I, int32_t* __restrict__ col_ptr,
                        int32_t* __restrict__ col_cur) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const bool vec = I % 4 == 0;
  int carry = 0;
  for (int base = 0; base < I; base += 16 * blockDim.x) {
    const int j0 = base + 16 * tid;
    int v[16];
    if (vec && j0 + 16 <= I) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int4 c = __ldcg(reinterpret_cast<const int4*>(col_cnt + j0) + q);
        v[4 * q] = c.x;
        v[4 * q + 1] = c.y;
        v[4 * q + 2] = c.z;
        v[4 * q + 3] = c.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = j0 + i < I ? __ldcg(col_cnt + j0 + i) : 0;
    }
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) sum += v[i];
    const int incl = warp_inclusive_scan(sum);
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const int w = lane < (blockDim.x >> 5) ? warp_tot[lane] : 0;
      warp_tot[lane] = warp_inclusive_scan(w);
    }
    __syncthreads();
    int run = carry + (wid ? warp_tot[wid - 1] : 0) + incl - sum;
    carry += warp_tot[(blockDim.x >> 5) - 1];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int e = run;
      run += v[i];
      v[i] = e;
    }
    if (vec && j0 + 16 <= I) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int4 e = make_int4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        reinterpret_cast<int4*>(col_ptr + j0)[q] = e;
        reinterpret_cast<int4*>(col_cur + j0)[q] = e;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (j0 + i < I) col_ptr[j0 + i] = col_cur[j0 + i] = v[i];
    }
    __syncthreads();  // warp_tot is rewritten by the next chunk
  }
  if (tid == 0) col_ptr[I] = carry;
}

// Column counts of the transposed Hybrid, then their scan. Every CTA counts the
// entries of its tokens (four tokens a warp) into a shared-memory histogram of the I
// columns, then adds its nonzero bins to col_cnt (zero at launch): a neuron that is
// active in many tokens then takes one global atomic per CTA, not one per entry.
// With hist_bins == 0 (I too large for shared memory) entries go to col_cnt
// directly. The CTA that finishes last, as told by a ticket counter (zero at
// launch), scans the counts. The token pass then claims each entry's slot from
// col_cur and writes its record there.
__global__ void __launch_bounds__(1024) csc_count_scan_kernel(const SparseBwdArgs a, int32_t* ticket, int hist_bins) {
  pdl_enter();
  if (a.route != nullptr && *a.route == 1) return;  // the call took the dense route
  extern __shared__ int hist[];
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int j = threadIdx.x; j < hist_bins; j += blockDim.x) hist[j] = 0;
  __syncthreads();
  int* cnt = hist_bins > 0 ? hist : a.col_cnt;
  // a warp takes four tokens at a time: their lengths in one round trip, then their
  // neuron indices in another
  const int gwarp = blockIdx.x * wpb + (threadIdx.x >> 5), nwarps = gridDim.x * wpb;
  for (int t0 = 4 * gwarp; t0 < a.T; t0 += 4 * nwarps) {
    int len = 0;
    if (lane < 4 && t0 + lane < a.T) {
      const int t = t0 + lane;
      const int slot = a.backup_slot != nullptr ? a.backup_slot[t] : -1;
      int n = a.ell_nnz[t];
      if (!TW_CHECKED(n >= 0 && n <= a.R, a.status)) n = 0;
      len = slot >= 0 ? 0 : n;  // exactly the entries the token pass writes: none of a backup row's
    }
    int n[4], nmax = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      n[q] = __shfl_sync(0xFFFFFFFFu, len, q);
      nmax = max(nmax, n[q]);
    }
    for (int k = lane; k < nmax; k += 32) {
      int j[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) j[q] = k < n[q] ? a.ell_idx[static_cast<size_t>(t0 + q) * a.R + k] : -1;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (j[q] >= 0 && TW_CHECKED(j[q] < a.I, a.status)) atomicAdd(cnt + j[q], 1);
    }
  }
  __syncthreads();
  for (int j = threadIdx.x; j < hist_bins; j += blockDim.x) {
    const int c = hist[j];
    if (c != 0) atomicAdd(a.col_cnt + j, c);
  }
  __threadfence();  // this thread's counts are visible before the CTA takes its ticket
  __syncthreads();
  __shared__ int last;
  if (threadIdx.x == 0) last = atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  scan_counts(a.col_cnt, a.I, a.col_ptr, a.col_cur);
}

// ====================================================================== backward: dW
// One warp per (256-wide slice c of d, neuron j, side), slices outermost, so that
// while slice c is processed only x[:, slice c] and dy[:, slice c] (16 MB at
// T = 16384) are gathered: they stay in L2. The x side accumulates
//   dWg[j] += dg x_t,  dWu[j] += du x_t   (gated)
// and the dy side
//   dWd[j] += h dy_t,  h = a u (non-gated: a)
// (fp32; streaming stores, or reductions into dW when it already holds the dense
// backup rows' part); splitting the sides halves the registers a
// warp needs, so more warps and more row slices are in flight per SM. Lane l owns 8
// columns of the slice. The column's records are staged 32 at a time in the warp's
// shared memory with the coefficients already paired for the packed FMA
// ({dg, dg, du, du}, {h, h, row}); a chunk whose length is not a multiple of the
// unroll is padded with zero coefficients on the chunk's last row (an L1 hit), so
// the inner loop has no predication and keeps kWgradUnroll row slices in flight.
constexpr int kWgradChunk = 4;
// Chunks after the warps' first ones are handed out by kSchedCounters counters (each
// in its own 128-byte line, zero at launch): counter q serves chunks
// nwarps + q, nwarps + q + kSchedCounters, ... to the warps with index = q modulo
// kSchedCounters, so no single address takes every claim. Returns the first item of
// the warp's next chunk (round-robin without counters).
TW_DEV int next_chunk(int32_t* sched, int prev, int nwarps, int gwarp) {
  if (sched == nullptr) return prev + nwarps * kWgradChunk;
  const int q = gwarp % kSchedCounters;
  return (nwarps + q + kSchedCounters * atomicAdd(sched + q * kSchedStride, 1)) * kWgradChunk;
}

template <bool GATED>
__global__ void __launch_bounds__(256, 4) ell_weight_grad_kernel(const SparseBwdArgs a) {
  pdl_enter();
  if (a.route != nullptr && *a.route == 1) return;  // the call took the dense route
  constexpr int U = kWgradUnroll;
  static_assert(32 % U == 0, "the unroll must divide the staging chunk");
  __shared__ float4 stage[8][32];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  float4(&rec)[32] = stage[warp];  // {dg, du, h, row offset}: one 16-byte read a record
  // dW already holds the dense backup rows' part when there are backup rows
  const bool add = a.dW_base_rows != nullptr && *a.dW_base_rows > 0;
  const int items = (a.d / 256) * a.I * 2;
  // Items are claimed kWgradChunk at a time, in order (slices outermost): a warp's
  // first chunk by its index, the rest from the scheduling counter, so warps that
  // drew long columns take fewer chunks.
  const int nwarps = gridDim.x * wpb, gwarp = blockIdx.x * wpb + warp;
  int32_t* const sched = nwarps >= kSchedCounters ? a.sched_w : nullptr;  // every counter needs its warps
  int it = gwarp * kWgradChunk, it_end = it + kWgradChunk;
  for (; it < items; ++it) {
    if (it == it_end) {
      const int c0 =
          __shfl_sync(0xFFFFFFFFu, lane == 0 ? next_chunk(sched, it - kWgradChunk, nwarps, gwarp) : 0, 0);
      it = c0;
      it_end = c0 + kWgradChunk;
      if (it >= items) break;
    }
    const bool xside = (it & 1) == 0;
    const int cj = it >> 1;
    const int c = cj / a.I;
    const int j = cj - c * a.I;
    const uint4* src = reinterpret_cast<const uint4*>(xside ? a.x : a.dy) + c * 32 + lane;
    int lo = a.col_ptr[j], hi = a.col_ptr[j + 1];
    if (!TW_CHECKED(lo >= 0 && lo <= hi && hi <= a.csc_cap, a.status)) lo = hi = 0;
    const uint32_t rows16 = static_cast<uint32_t>(a.T) * static_cast<uint32_t>(a.d / 8);  // bound of a record's row
    F8 p, q2;
    f8_zero(p);
    f8_zero(q2);
    for (int e0 = lo; e0 < hi; e0 += 32) {
      const int m = min(32, hi - e0);
      uint4 r = lane < m ? a.csc[e0 + lane] : make_uint4(0u, 0u, 0u, 0u);
      if (!TW_CHECKED(r.x < rows16, a.status)) r = make_uint4(0u, 0u, 0u, 0u);
      const uint32_t last = __shfl_sync(0xFFFFFFFFu, r.x, m - 1);
      if (lane >= m) r.x = last;
      __syncwarp();  // the previous chunk's reads of the stage are done
      rec[lane] = make_float4(__uint_as_float(r.y), __uint_as_float(r.z), __uint_as_float(r.w), __uint_as_float(r.x));
      __syncwarp();
      if (xside) {
        for (int k = 0; k < m; k += U) {
          uint4 v[U];
          float cg[U], cu[U];
#pragma unroll
          for (int q = 0; q < U; ++q) {
            const float4 e = rec[k + q];
            cg[q] = e.x;
            cu[q] = e.y;
            v[q] = ldg16(src + __float_as_uint(e.w));
          }
#pragma unroll
          for (int q = 0; q < U; ++q) {
            if (GATED)
              axpy8_two(p, pair(cg[q], cg[q]), q2, pair(cu[q], cu[q]), v[q]);
            else
              axpy8(p, pair(cg[q], cg[q]), v[q]);
          }
        }
      } else {
        for (int k = 0; k < m; k += U) {
          uint4 v[U];
          float ch[U];
#pragma unroll
          for (int q = 0; q < U; ++q) {
            const float4 e = rec[k + q];
            ch[q] = e.z;
            v[q] = ldg16(src + __float_as_uint(e.w));
          }
#pragma unroll
          for (int q = 0; q < U; ++q) axpy8(p, pair(ch[q], ch[q]), v[q]);
        }
      }
    }
    const size_t o = static_cast<size_t>(j) * a.d + c * 256 + lane * 8;
    if (xside) {
      out_f32x8(a.dWg + o, p, add);
      if (GATED) out_f32x8(a.dWu + o, q2, add);
    } else {
      out_f32x8(a.dWd + o, p, add);
    }
  }
}

// ====================================================================== launchers
static cudaError_t token_side(const SparseBwdArgs& a, cudaStream_t s) {
  // column counts, the scheduling counters of both passes and the count pass's ticket
  cudaError_t e =
      launch_zero(a.col_cnt, sizeof(int32_t) * (a.I + 1), a.sched, a.sched ? sizeof(int32_t) * kSchedWords : 0, s);
  if (e != cudaSuccess) return e;
  int32_t* ticket = a.sched + kSchedTicket;
  // one CTA per SM; a shared-memory histogram of the columns when it fits
  const int bins = a.I <= kCountHistMaxBins ? a.I : 0;
  const size_t smem = sizeof(int) * static_cast<size_t>(bins);
  e = set_smem_bytes(csc_count_scan_kernel, smem);
  if (e != cudaSuccess) return e;
  e = launch(csc_count_scan_kernel, dim3(grid_for(a.T, 32, 1)), dim3(1024), smem, s, a, ticket, bins);
  trace_mark(s, "csc_count_scan");
  if (e != cudaSuccess) return e;
  return launch_token_bwd(a, s);  // dh, dg, du, the records of the transposed Hybrid, dx
}

cudaError_t launch_sparse_bwd_tokens(const SparseBwdArgs& a, cudaStream_t s) {
  if (a.sched == nullptr) return cudaErrorInvalidValue;  // holds the count pass's ticket
  return token_side(a, s);
}

cudaError_t launch_sparse_bwd_weights(const SparseBwdArgs& a, cudaStream_t s) {
  const long items = static_cast<long>(a.d / 256) * a.I * 2;
  const dim3 grid(grid_for(items, 8, 4));
  const cudaError_t e = a.Wu != nullptr ? launch(ell_weight_grad_kernel<true>, grid, dim3(256), 0, s, a)
                                        : launch(ell_weight_grad_kernel<false>, grid, dim3(256), 0, s, a);
  trace_mark(s, "ell_weight_grad");
  return e;
}

}  // namespace tw

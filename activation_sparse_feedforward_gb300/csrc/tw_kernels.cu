// CUDA-core kernels of the sparse FFN path:
//  * TwELL packing of a dense bf16 matrix (standalone packer),
//  * ordered row compaction (overflow list for TwELL, backup routing for Hybrid),
//  * row gathers feeding the dense tensor-core backup,
//  * the fused sparse up/down projection over TwELL (inference) and its Hybrid
//    variant that also writes the compact ELL (training forward),
//  * the sparse backward over the Hybrid ELL: per-token dh/du/dg/dx, the transposed
//    Hybrid (CSC by neuron) and the weight gradients accumulated over it.
//
// Weight rows are gathered with 128-bit read-only loads: one warp owns one token,
// lane l holds elements [256*q + 8*l, 256*q + 8*l + 8) of every d-vector, so each
// weight row is read as fully coalesced 512-byte warp transactions.
#include <algorithm>

#include "tw_common.cuh"
#include "tw_internal.h"

namespace tw {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// ---------------------------------------------------------------- timing trace
namespace {
constexpr int kTraceLabels = 16384;
struct TraceState {
  void* const* events = nullptr;
  int cap = 0;
  int n = 0;
  bool on = false;
  const char* labels[kTraceLabels];
};
TraceState g_trace;
}  // namespace

void trace_begin(void* const* events, int capacity) {
  g_trace.events = events;
  g_trace.cap = capacity;
  g_trace.n = 0;
  g_trace.on = events != nullptr && capacity > 0;
}
int trace_end() {
  g_trace.on = false;
  return g_trace.n;
}
const char* trace_label(int i) {
  if (i < 0 || i >= g_trace.n || i >= kTraceLabels) return nullptr;
  return g_trace.labels[i];
}
void trace_mark(cudaStream_t s, const char* label) {
  if (!g_trace.on || g_trace.n >= g_trace.cap) return;
  cudaEventRecord(static_cast<cudaEvent_t>(g_trace.events[g_trace.n]), s);
  if (g_trace.n < kTraceLabels) g_trace.labels[g_trace.n] = label;
  ++g_trace.n;
}
cudaError_t memset_async(void* p, int v, size_t bytes, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(p, v, bytes, s);
  trace_mark(s, "memset");
  return e;
}

static int warp_grid(long rows, int warps_per_block) {
  const long blocks = (rows + warps_per_block - 1) / warps_per_block;
  const long cap = static_cast<long>(device_sm_count()) * 32;
  return static_cast<int>(std::max<long>(1, std::min(blocks, cap)));
}

// ================================================================ dense -> TwELL
// One warp per row; lane l holds columns [VPL*l, VPL*l + VPL) of each tile
// (W = 32 * VPL). A warp prefix sum over the per-lane nonzero counts gives each
// nonzero its slot, so slots come out in ascending column order.
template <int VPL>
__global__ void __launch_bounds__(256) pack_dense_kernel(const uint16_t* __restrict__ A, int T, int I, int C, int nT,
                                                         uint16_t* __restrict__ cnt, uint16_t* __restrict__ val,
                                                         uint8_t* __restrict__ idx, int32_t* __restrict__ row_nnz,
                                                         uint8_t* __restrict__ ovf) {
  constexpr int W = 32 * VPL;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    const uint16_t* row = A + static_cast<size_t>(t) * I;
    int total = 0;
    bool any = false;
    for (int k = 0; k < nT; ++k) {
      uint16_t v[VPL];
      const int col = k * W + lane * VPL;
      if (VPL == 4) {
        const uint2 q = *reinterpret_cast<const uint2*>(row + col);
        v[0] = q.x & 0xFFFF; v[1] = q.x >> 16; v[2 % VPL] = q.y & 0xFFFF; v[3 % VPL] = q.y >> 16;
      } else {
        const uint32_t q = *reinterpret_cast<const uint32_t*>(row + col);
        v[0] = q & 0xFFFF; v[1 % VPL] = q >> 16;
      }
      int n = 0;
#pragma unroll
      for (int i = 0; i < VPL; ++i) n += (v[i] & 0x7FFF) != 0;
      const int incl = warp_inclusive_scan(n);
      const int tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
      int pos = incl - n;
      const size_t base = (static_cast<size_t>(t) * nT + k) * C;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        if (v[i] & 0x7FFF) {
          if (pos < C) {
            val[base + pos] = v[i];
            idx[base + pos] = static_cast<uint8_t>(lane * VPL + i);
          }
          ++pos;
        }
      }
      if (lane == 0) cnt[static_cast<size_t>(t) * nT + k] = static_cast<uint16_t>(tot);
      total += tot;
      any |= (tot > C);
    }
    if (lane == 0) {
      row_nnz[t] = total;
      ovf[t] = any ? 1 : 0;
    }
  }
}

cudaError_t launch_pack_dense(const uint16_t* A, int T, int I, int W, int C, const tw_twell& o, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int nT = I / W;
  const int grid = warp_grid(T, 8);
  if (W == 128)
    pack_dense_kernel<4><<<grid, 256, 0, s>>>(A, T, I, C, nT, o.cnt, o.val, o.idx, o.row_nnz, o.ovf);
  else
    pack_dense_kernel<2><<<grid, 256, 0, s>>>(A, T, I, C, nT, o.cnt, o.val, o.idx, o.row_nnz, o.ovf);
  trace_mark(s, "pack_dense");
  return cudaGetLastError();
}

// ================================================================ ordered compaction
// One CTA of 1024 threads walks the rows in chunks; a block-wide exclusive scan of
// the flags gives every flagged row its rank, so the list is in ascending order.
__global__ void __launch_bounds__(1024) compact_rows_kernel(const uint8_t* __restrict__ ovf,
                                                            const int32_t* __restrict__ row_nnz, int R, int T,
                                                            int32_t* __restrict__ list, int list_cap,
                                                            int32_t* __restrict__ count, int32_t* __restrict__ slot_of,
                                                            int32_t* __restrict__ ell_nnz, int cap_check,
                                                            int32_t* status) {
  __shared__ int warp_tot[32];
  __shared__ int carry_s;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  if (tid == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < T; base += blockDim.x) {
    const int t = base + tid;
    int f = 0, nnz = 0;
    if (t < T) {
      nnz = row_nnz ? row_nnz[t] : 0;
      f = (ovf[t] != 0 || (row_nnz != nullptr && nnz > R)) ? 1 : 0;
    }
    const int incl = warp_inclusive_scan(f);
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      int v = lane < nwarps ? warp_tot[lane] : 0;
      v = warp_inclusive_scan(v);
      warp_tot[lane] = v;
    }
    __syncthreads();
    const int carry = carry_s;
    const int pos = carry + (wid ? warp_tot[wid - 1] : 0) + incl - f;
    if (t < T) {
      if (f) {
        if (pos < list_cap) list[pos] = t;
        if (slot_of) slot_of[t] = pos < list_cap ? pos : -2;
      } else if (slot_of) {
        slot_of[t] = -1;
      }
      if (ell_nnz) ell_nnz[t] = f ? 0 : nnz;
    }
    __syncthreads();
    if (tid == 0) carry_s = carry + warp_tot[nwarps - 1];
    __syncthreads();
  }
  if (tid == 0) {
    *count = carry_s;
    if (carry_s > cap_check) raise_status(status, TW_ECAPACITY);
  }
}

cudaError_t launch_compact_rows(const uint8_t* ovf, const int32_t* row_nnz, int R, int T, int32_t* list,
                                int list_cap, int32_t* count, int32_t* slot_of, int32_t* ell_nnz, int cap_check,
                                int32_t* status, cudaStream_t s) {
  compact_rows_kernel<<<1, 1024, 0, s>>>(ovf, row_nnz, R, T, list, list_cap, count, slot_of, ell_nnz, cap_check,
                                         status);
  trace_mark(s, "compact_rows");
  return cudaGetLastError();
}

// ================================================================ row gather
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ src, int d,
                                                          const int32_t* __restrict__ rows,
                                                          const int32_t* __restrict__ n_dev, int cap, int rows_alloc,
                                                          uint16_t* __restrict__ out) {
  const int n = min(max(*n_dev, 0), cap);
  const int limit = min(rows_alloc, (n + 127) / 128 * 128);
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int vec = d / 8;
  for (int i = blockIdx.x * wpb + (threadIdx.x >> 5); i < limit; i += gridDim.x * wpb) {
    uint4* o = reinterpret_cast<uint4*>(out + static_cast<size_t>(i) * d);
    if (i < n) {
      const uint4* r = reinterpret_cast<const uint4*>(src + static_cast<size_t>(rows[i]) * d);
      for (int c = lane; c < vec; c += 32) o[c] = __ldg(r + c);
    } else {
      for (int c = lane; c < vec; c += 32) o[c] = make_uint4(0, 0, 0, 0);
    }
  }
}

cudaError_t launch_gather_rows(const uint16_t* src, int d, const int32_t* rows, const int32_t* n, int cap,
                               int rows_alloc, uint16_t* out, cudaStream_t s) {
  if (rows_alloc <= 0) return cudaSuccess;
  const int grid = warp_grid(rows_alloc, 8);
  gather_rows_kernel<<<std::min(grid, device_sm_count() * 4), 256, 0, s>>>(src, d, rows, n, cap, rows_alloc, out);
  trace_mark(s, "gather_rows");
  return cudaGetLastError();
}

// ================================================================ vector helpers
TW_DEV float dot8(const uint4& a, const uint4& b, float acc) {
  acc = fmaf(bf16_lo(a.x), bf16_lo(b.x), acc);
  acc = fmaf(bf16_hi(a.x), bf16_hi(b.x), acc);
  acc = fmaf(bf16_lo(a.y), bf16_lo(b.y), acc);
  acc = fmaf(bf16_hi(a.y), bf16_hi(b.y), acc);
  acc = fmaf(bf16_lo(a.z), bf16_lo(b.z), acc);
  acc = fmaf(bf16_hi(a.z), bf16_hi(b.z), acc);
  acc = fmaf(bf16_lo(a.w), bf16_lo(b.w), acc);
  acc = fmaf(bf16_hi(a.w), bf16_hi(b.w), acc);
  return acc;
}
TW_DEV void axpy8(float (&y)[8], float h, const uint4& w) {
  y[0] = fmaf(h, bf16_lo(w.x), y[0]);
  y[1] = fmaf(h, bf16_hi(w.x), y[1]);
  y[2] = fmaf(h, bf16_lo(w.y), y[2]);
  y[3] = fmaf(h, bf16_hi(w.y), y[3]);
  y[4] = fmaf(h, bf16_lo(w.z), y[4]);
  y[5] = fmaf(h, bf16_hi(w.z), y[5]);
  y[6] = fmaf(h, bf16_lo(w.w), y[6]);
  y[7] = fmaf(h, bf16_hi(w.w), y[7]);
}
TW_DEV uint4 pack8(const float (&y)[8]) {
  return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                    pack_bf16x2(y[6], y[7]));
}
TW_DEV uint4 ldg_nc(const uint4* p) { return __ldg(p); }

// ================================================================ fused sparse up/down
// One warp per token. The token's entries are enumerated tile by tile from the
// TwELL counts (ballot over tiles with nonzero count; the tile's slots are read
// by the first cnt lanes and broadcast one at a time), so they arrive in ascending
// neuron order. Per entry (j, a):
//   gated:     u = x_t . Wu[j] (warp reduction),  h = a * u
//   non-gated: h = a
//   y_t += h * Wd[j]                              (fp32 accumulators in registers)
// HYBRID additionally writes the entry (j, a, bf16(u)) to the row's ELL slots.
template <int NCH, bool GATED, bool HYBRID>
__global__ void __launch_bounds__(256) sparse_fwd_kernel(const SparseFwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int d = NCH * 256;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < a.T; t += gridDim.x * wpb) {
    if (HYBRID) {
      if (a.backup_slot[t] != -1) continue;
    } else {
      if (a.ovf[t]) continue;
    }
    uint4 xv[NCH];
    if (GATED) {
      const uint4* xr = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * d);
#pragma unroll
      for (int q = 0; q < NCH; ++q) xv[q] = ldg_nc(xr + q * 32 + lane);
    }
    float y[NCH][8];
#pragma unroll
    for (int q = 0; q < NCH; ++q)
#pragma unroll
      for (int i = 0; i < 8; ++i) y[q][i] = 0.f;
    int pos = 0;
    const uint16_t* cnt_row = a.cnt + static_cast<size_t>(t) * a.nT;
    for (int kb = 0; kb < a.nT; kb += 32) {
      const int k = kb + lane;
      const int c = (k < a.nT) ? min(static_cast<int>(cnt_row[k]), a.C) : 0;
      unsigned mask = __ballot_sync(0xFFFFFFFFu, c > 0);
      while (mask) {
        const int src = __ffs(mask) - 1;
        mask &= mask - 1;
        const int kk = kb + src;
        const int cc = __shfl_sync(0xFFFFFFFFu, c, src);
        const size_t sb = (static_cast<size_t>(t) * a.nT + kk) * a.C;
        int jv = 0;
        uint32_t av = 0;
        if (lane < cc) {
          jv = kk * a.W + a.idx[sb + lane];
          av = a.val[sb + lane];
        }
        for (int s = 0; s < cc; ++s) {
          const int j = __shfl_sync(0xFFFFFFFFu, jv, s);
          const uint32_t abits = __shfl_sync(0xFFFFFFFFu, av, s);
          const float af = bf16_to_f32(static_cast<uint16_t>(abits));
          const uint4* wd = reinterpret_cast<const uint4*>(a.Wd + static_cast<size_t>(j) * d);
          uint4 wdv[NCH];
#pragma unroll
          for (int q = 0; q < NCH; ++q) wdv[q] = ldg_nc(wd + q * 32 + lane);
          float h = af;
          if (GATED) {
            const uint4* wu = reinterpret_cast<const uint4*>(a.Wu + static_cast<size_t>(j) * d);
            uint4 wuv[NCH];
#pragma unroll
            for (int q = 0; q < NCH; ++q) wuv[q] = ldg_nc(wu + q * 32 + lane);
            float dot = 0.f;
#pragma unroll
            for (int q = 0; q < NCH; ++q) dot = dot8(xv[q], wuv[q], dot);
            dot = warp_sum(dot);
            h = af * dot;
            if (HYBRID && lane == 0) a.ell_u[static_cast<size_t>(t) * a.R + pos] = f32_to_bf16(dot);
          }
          if (HYBRID && lane == 0) {
            a.ell_idx[static_cast<size_t>(t) * a.R + pos] = static_cast<uint16_t>(j);
            a.ell_a[static_cast<size_t>(t) * a.R + pos] = static_cast<uint16_t>(abits);
          }
#pragma unroll
          for (int q = 0; q < NCH; ++q) axpy8(y[q], h, wdv[q]);
          ++pos;
        }
      }
    }
    uint4* yr = reinterpret_cast<uint4*>(a.y + static_cast<size_t>(t) * d);
#pragma unroll
    for (int q = 0; q < NCH; ++q) yr[q * 32 + lane] = pack8(y[q]);
  }
}

template <bool GATED, bool HYBRID>
static cudaError_t sparse_fwd_dispatch(const SparseFwdArgs& a, cudaStream_t s) {
  const int grid = warp_grid(a.T, 8);
  switch (a.d / 256) {
#define TW_CASE(n) \
  case n: sparse_fwd_kernel<n, GATED, HYBRID><<<grid, 256, 0, s>>>(a); break;
    TW_CASE(1) TW_CASE(2) TW_CASE(3) TW_CASE(4) TW_CASE(5) TW_CASE(6) TW_CASE(7) TW_CASE(8)
#undef TW_CASE
    default: return cudaErrorInvalidValue;
  }
  trace_mark(s, "sparse_fwd");
  return cudaGetLastError();
}

cudaError_t launch_sparse_fwd(const SparseFwdArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const bool gated = a.Wu != nullptr;
  const bool hybrid = a.backup_slot != nullptr;
  if (gated && hybrid) return sparse_fwd_dispatch<true, true>(a, s);
  if (gated) return sparse_fwd_dispatch<true, false>(a, s);
  if (hybrid) return sparse_fwd_dispatch<false, true>(a, s);
  return sparse_fwd_dispatch<false, false>(a, s);
}

// ================================================================ sparse backward
// One warp per ELL token. Per entry (j, a, u):
//   dh = dy_t . Wd[j];  du = dh * a;  dg = dh * u + l1  (non-gated: dg = dh + l1)
//   dx_t += dg * Wg[j] + du * Wu[j]
// dg and du are kept per entry for the weight gradients.
template <int NCH, bool GATED>
__global__ void __launch_bounds__(256) sparse_bwd_token_kernel(const SparseBwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int d = NCH * 256;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < a.T; t += gridDim.x * wpb) {
    if (a.backup_slot[t] != -1) continue;
    const int n = a.ell_nnz[t];
    uint4 dyv[NCH];
    const uint4* dyr = reinterpret_cast<const uint4*>(a.dy + static_cast<size_t>(t) * d);
#pragma unroll
    for (int q = 0; q < NCH; ++q) dyv[q] = ldg_nc(dyr + q * 32 + lane);
    float dx[NCH][8];
#pragma unroll
    for (int q = 0; q < NCH; ++q)
#pragma unroll
      for (int i = 0; i < 8; ++i) dx[q][i] = 0.f;
    const size_t rb = static_cast<size_t>(t) * a.R;
    for (int eb = 0; eb < n; eb += 32) {
      const int e = eb + lane;
      int jv = 0;
      uint32_t avb = 0, uvb = 0;
      if (e < n) {
        jv = a.ell_idx[rb + e];
        avb = a.ell_a[rb + e];
        if (GATED) uvb = a.ell_u[rb + e];
      }
      const int m = min(32, n - eb);
      for (int s = 0; s < m; ++s) {
        const int j = __shfl_sync(0xFFFFFFFFu, jv, s);
        const float af = bf16_to_f32(static_cast<uint16_t>(__shfl_sync(0xFFFFFFFFu, avb, s)));
        const float uf = GATED ? bf16_to_f32(static_cast<uint16_t>(__shfl_sync(0xFFFFFFFFu, uvb, s))) : 1.f;
        const size_t jr = static_cast<size_t>(j) * d;
        const uint4* wd = reinterpret_cast<const uint4*>(a.Wd + jr);
        const uint4* wg = reinterpret_cast<const uint4*>(a.Wg + jr);
        uint4 wdv[NCH], wgv[NCH], wuv[NCH];
#pragma unroll
        for (int q = 0; q < NCH; ++q) wdv[q] = ldg_nc(wd + q * 32 + lane);
#pragma unroll
        for (int q = 0; q < NCH; ++q) wgv[q] = ldg_nc(wg + q * 32 + lane);
        if (GATED) {
          const uint4* wu = reinterpret_cast<const uint4*>(a.Wu + jr);
#pragma unroll
          for (int q = 0; q < NCH; ++q) wuv[q] = ldg_nc(wu + q * 32 + lane);
        }
        float dh = 0.f;
#pragma unroll
        for (int q = 0; q < NCH; ++q) dh = dot8(dyv[q], wdv[q], dh);
        dh = warp_sum(dh);
        const float dg = (GATED ? dh * uf : dh) + a.l1;
        const float du = dh * af;
        if (lane == 0) {
          a.dg[rb + eb + s] = dg;
          if (GATED) a.du[rb + eb + s] = du;
        }
#pragma unroll
        for (int q = 0; q < NCH; ++q) {
          axpy8(dx[q], dg, wgv[q]);
          if (GATED) axpy8(dx[q], du, wuv[q]);
        }
      }
    }
    uint4* dxr = reinterpret_cast<uint4*>(a.dx + static_cast<size_t>(t) * d);
#pragma unroll
    for (int q = 0; q < NCH; ++q) dxr[q * 32 + lane] = pack8(dx[q]);
  }
}

// transposed Hybrid: count entries per neuron
__global__ void __launch_bounds__(256) csc_count_kernel(const int32_t* __restrict__ ell_nnz,
                                                        const uint16_t* __restrict__ ell_idx, int T, int R,
                                                        int32_t* __restrict__ col_cnt) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    const int n = ell_nnz[t];
    for (int s = lane; s < n; s += 32) atomicAdd(col_cnt + ell_idx[static_cast<size_t>(t) * R + s], 1);
  }
}

// exclusive scan of the per-neuron counts (one CTA): col_ptr[0..I], col_cur = col_ptr
__global__ void __launch_bounds__(1024) csc_scan_kernel(const int32_t* __restrict__ col_cnt, int I,
                                                        int32_t* __restrict__ col_ptr, int32_t* __restrict__ col_cur) {
  __shared__ int warp_tot[32];
  __shared__ int carry_s;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  if (tid == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < I; base += blockDim.x) {
    const int j = base + tid;
    const int v = j < I ? col_cnt[j] : 0;
    const int incl = warp_inclusive_scan(v);
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      int w = lane < nwarps ? warp_tot[lane] : 0;
      w = warp_inclusive_scan(w);
      warp_tot[lane] = w;
    }
    __syncthreads();
    const int carry = carry_s;
    const int ex = carry + (wid ? warp_tot[wid - 1] : 0) + incl - v;
    if (j < I) {
      col_ptr[j] = ex;
      col_cur[j] = ex;
    }
    __syncthreads();
    if (tid == 0) carry_s = carry + warp_tot[nwarps - 1];
    __syncthreads();
  }
  if (tid == 0) col_ptr[I] = carry_s;
}

__global__ void __launch_bounds__(256) csc_fill_kernel(const int32_t* __restrict__ ell_nnz,
                                                       const uint16_t* __restrict__ ell_idx, int T, int R,
                                                       int32_t* __restrict__ col_cur, int32_t* __restrict__ csc) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    const int n = ell_nnz[t];
    for (int s = lane; s < n; s += 32) {
      const size_t e = static_cast<size_t>(t) * R + s;
      const int p = atomicAdd(col_cur + ell_idx[e], 1);
      csc[p] = static_cast<int32_t>(e);
    }
  }
}

// ELL part of the weight gradients, one CTA per neuron j (d/8 threads, 8 columns
// each): dWg[j] = sum dg x_t, dWu[j] = sum du x_t, dWd[j] = sum (a u) dy_t over the
// transposed Hybrid's entries of column j. Overwrites the three rows.
template <bool GATED>
__global__ void __launch_bounds__(256) ell_weight_grad_kernel(const SparseBwdArgs a) {
  const int tid = threadIdx.x;
  const int d = a.d;
  for (int j = blockIdx.x; j < a.I; j += gridDim.x) {
    const int lo = a.col_ptr[j], hi = a.col_ptr[j + 1];
    float g[8], u[8], h[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = u[i] = h[i] = 0.f;
    int e = lo;
    for (; e + 2 <= hi; e += 2) {
      int ent[2];
      float cg[2], cu[2], ch[2];
      uint4 xv[2], dv[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) ent[r] = a.csc[e + r];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int t = ent[r] / a.R;
        cg[r] = a.dg[ent[r]];
        const float av = bf16_to_f32(a.ell_a[ent[r]]);
        if (GATED) {
          cu[r] = a.du[ent[r]];
          ch[r] = av * bf16_to_f32(a.ell_u[ent[r]]);
        } else {
          cu[r] = 0.f;
          ch[r] = av;
        }
        xv[r] = ldg_nc(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * d) + tid);
        dv[r] = ldg_nc(reinterpret_cast<const uint4*>(a.dy + static_cast<size_t>(t) * d) + tid);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        axpy8(g, cg[r], xv[r]);
        if (GATED) axpy8(u, cu[r], xv[r]);
        axpy8(h, ch[r], dv[r]);
      }
    }
    for (; e < hi; ++e) {
      const int en = a.csc[e];
      const int t = en / a.R;
      const float av = bf16_to_f32(a.ell_a[en]);
      const uint4 xv = ldg_nc(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * d) + tid);
      const uint4 dv = ldg_nc(reinterpret_cast<const uint4*>(a.dy + static_cast<size_t>(t) * d) + tid);
      axpy8(g, a.dg[en], xv);
      if (GATED) {
        axpy8(u, a.du[en], xv);
        axpy8(h, av * bf16_to_f32(a.ell_u[en]), dv);
      } else {
        axpy8(h, av, dv);
      }
    }
    const size_t o = static_cast<size_t>(j) * d + tid * 8;
    float4* pg = reinterpret_cast<float4*>(a.dWg + o);
    pg[0] = make_float4(g[0], g[1], g[2], g[3]);
    pg[1] = make_float4(g[4], g[5], g[6], g[7]);
    if (GATED) {
      float4* pu = reinterpret_cast<float4*>(a.dWu + o);
      pu[0] = make_float4(u[0], u[1], u[2], u[3]);
      pu[1] = make_float4(u[4], u[5], u[6], u[7]);
    }
    float4* ph = reinterpret_cast<float4*>(a.dWd + o);
    ph[0] = make_float4(h[0], h[1], h[2], h[3]);
    ph[1] = make_float4(h[4], h[5], h[6], h[7]);
  }
}

template <bool GATED>
static cudaError_t sparse_bwd_dispatch(const SparseBwdArgs& a, cudaStream_t s) {
  const int grid = warp_grid(a.T, 8);
  switch (a.d / 256) {
#define TW_CASE(n) \
  case n: sparse_bwd_token_kernel<n, GATED><<<grid, 256, 0, s>>>(a); break;
    TW_CASE(1) TW_CASE(2) TW_CASE(3) TW_CASE(4) TW_CASE(5) TW_CASE(6) TW_CASE(7) TW_CASE(8)
#undef TW_CASE
    default: return cudaErrorInvalidValue;
  }
  trace_mark(s, "sparse_bwd_token");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = memset_async(a.col_cnt, 0, sizeof(int32_t) * (a.I + 1), s);
  if (e != cudaSuccess) return e;
  csc_count_kernel<<<grid, 256, 0, s>>>(a.ell_nnz, a.ell_idx, a.T, a.R, a.col_cnt);
  trace_mark(s, "csc_count");
  csc_scan_kernel<<<1, 1024, 0, s>>>(a.col_cnt, a.I, a.col_ptr, a.col_cur);
  trace_mark(s, "csc_scan");
  csc_fill_kernel<<<grid, 256, 0, s>>>(a.ell_nnz, a.ell_idx, a.T, a.R, a.col_cur, a.csc);
  trace_mark(s, "csc_fill");
  const int gw = std::min(a.I, device_sm_count() * 8);
  ell_weight_grad_kernel<GATED><<<gw, a.d / 8, 0, s>>>(a);
  trace_mark(s, "ell_weight_grad");
  return cudaGetLastError();
}

cudaError_t launch_sparse_bwd(const SparseBwdArgs& a, cudaStream_t s) {
  if (a.Wu != nullptr) return sparse_bwd_dispatch<true>(a, s);
  return sparse_bwd_dispatch<false>(a, s);
}

}  // namespace tw

// Small CUDA-core kernels around the sparse path (the gathers themselves live in
// tw_sparse.cu) and the library's timing trace:
//  * TwELL packing of a dense bf16 matrix (standalone packer),
//  * ordered row compaction (overflow list for TwELL, backup routing for Hybrid),
//  * row gathers feeding the dense tensor-core backup.
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
// ---------------------------------------------------------------- zero fill
// Zeroes two byte ranges (16-byte aligned starts): 16-byte stores, then the tails
// byte by byte.
__global__ void __launch_bounds__(256) zero_kernel(uint8_t* __restrict__ p0, size_t b0, uint8_t* __restrict__ p1,
                                                  size_t b1) {
  pdl_enter();
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const size_t i0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t n0 = b0 / 16, n1 = b1 / 16;
  for (size_t i = i0; i < n0; i += stride) reinterpret_cast<uint4*>(p0)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (size_t i = i0; i < n1; i += stride) reinterpret_cast<uint4*>(p1)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (i0 < b0 % 16) p0[n0 * 16 + i0] = 0;
  if (i0 < b1 % 16) p1[n1 * 16 + i0] = 0;
}

cudaError_t launch_zero(void* p0, size_t b0, void* p1, size_t b1, cudaStream_t s) {
  if (p1 == nullptr) b1 = 0;
  if (b0 == 0 && b1 == 0) return cudaSuccess;
  const size_t most = std::max(std::max(b0, b1) / 16, static_cast<size_t>(16));
  const int grid = static_cast<int>(std::min<size_t>((most + 255) / 256, static_cast<size_t>(device_sm_count()) * 4));
  cudaError_t e = launch(zero_kernel, dim3(std::max(grid, 1)), dim3(256), 0, s, static_cast<uint8_t*>(p0), b0,
                         static_cast<uint8_t*>(p1), b1);
  trace_mark(s, "zero");
  return e;
}

// ---------------------------------------------------------------- bf16 -> fp16
// Up to four tensors converted element by element, round to nearest even (exact for
// magnitudes in fp16's normal range, 2^-14 to 65504; smaller ones become fp16
// subnormals, larger ones infinity). Only when *route == 1 (route may be null).
struct ToF16Args {
  const uint16_t* src[4];
  uint16_t* dst[4];
  size_t n8[4];  // elements / 8
  int count;
  const int32_t* route;
};
__global__ void __launch_bounds__(256) to_f16_kernel(const ToF16Args a) {
  pdl_enter();
  if (a.route != nullptr && *a.route != 1) return;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (int k = 0; k < a.count; ++k) {
    const uint4* s = reinterpret_cast<const uint4*>(a.src[k]);
    uint4* d = reinterpret_cast<uint4*>(a.dst[k]);
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < a.n8[k]; i += stride) {
      const uint4 v = s[i];
      d[i] = make_uint4(pack_f16x2_rn(bf16_lo(v.x), bf16_hi(v.x)), pack_f16x2_rn(bf16_lo(v.y), bf16_hi(v.y)),
                        pack_f16x2_rn(bf16_lo(v.z), bf16_hi(v.z)), pack_f16x2_rn(bf16_lo(v.w), bf16_hi(v.w)));
    }
  }
}

cudaError_t launch_to_f16(const uint16_t* const* src, uint16_t* const* dst, const size_t* n, int count,
                          const int32_t* route, cudaStream_t s) {
  if (count < 1 || count > 4) return cudaErrorInvalidValue;
  ToF16Args a{};
  size_t most = 0;
  for (int k = 0; k < count; ++k) {
    if (n[k] % 8 != 0) return cudaErrorInvalidValue;
    a.src[k] = src[k];
    a.dst[k] = dst[k];
    a.n8[k] = n[k] / 8;
    most = std::max(most, a.n8[k]);
  }
  a.count = count;
  a.route = route;
  if (most == 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<size_t>((most + 255) / 256, static_cast<size_t>(device_sm_count()) * 8));
  cudaError_t e = launch(to_f16_kernel, dim3(grid), dim3(256), 0, s, a);
  trace_mark(s, "to_f16");
  return e;
}

// ---------------------------------------------------------------- fp32 FMA probe
// CUDA-core throughput of the packed two-lane fp32 FMA (`fma.rn.f32x2`), the
// instruction of the sparse kernels' accumulations: every thread runs kProbeChains
// independent chains of `iters` dependent FMAs each, on values that stay finite
// (|m| < 1), and stores the sum so no chain is dead code.
constexpr int kProbeChains = 8;
__global__ void __launch_bounds__(256) fma_probe_kernel(float* __restrict__ out, int iters) {
  pdl_enter();
  const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
  const float seed = static_cast<float>(tid & 1023u) * 0x1p-12f;
  uint64_t acc[kProbeChains], mul, add;
  {
    const float m = 0.5f + seed * 0.25f, c = 0.25f - seed;
    asm("mov.b64 %0, {%1, %2};" : "=l"(mul) : "f"(m), "f"(m * 0.5f));
    asm("mov.b64 %0, {%1, %2};" : "=l"(add) : "f"(c), "f"(-c));
  }
#pragma unroll
  for (int c = 0; c < kProbeChains; ++c) {
    const float v = seed + static_cast<float>(c);
    asm("mov.b64 %0, {%1, %2};" : "=l"(acc[c]) : "f"(v), "f"(-v));
  }
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kProbeChains; ++c) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc[c]) : "l"(mul), "l"(add));
  }
  float sum = 0.f;
#pragma unroll
  for (int c = 0; c < kProbeChains; ++c) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc[c]));
    sum += lo + hi;
  }
  out[tid] = sum;
}

cudaError_t launch_fma_probe(float* out, int blocks, int iters, cudaStream_t s) {
  cudaError_t e = launch(fma_probe_kernel, dim3(blocks), dim3(256), 0, s, out, iters);
  trace_mark(s, "fma_probe");
  return e;
}
long fma_probe_flops(int blocks, int iters) {
  return static_cast<long>(blocks) * 256L * iters * kProbeChains * 2L * 2L;  // 2 lanes, 2 FLOP per FMA
}

// ---------------------------------------------------------------- L2 gather probe
// Row-slice gather rate from an L2-resident table, the access pattern of the sparse
// kernels: a CTA of d / 256 warps takes groups of eight row indices; warp c loads the
// 512-byte slice c of each of the eight rows (16 bytes a lane, all eight loads in
// flight together) and accumulates them with packed fp32 FMAs. Six CTAs per SM at
// d = 2048 (48 warps), like the token kernels. Each thread writes its sum.
__global__ void __launch_bounds__(256) l2_gather_probe_kernel(const uint16_t* __restrict__ table, int rows, int d,
                                                             const int32_t* __restrict__ idx, int n_groups,
                                                             float* __restrict__ out) {
  pdl_enter();
  const int lane = threadIdx.x & 31, c = threadIdx.x >> 5;
  const uint32_t row16 = static_cast<uint32_t>(d / 8);
  const uint4* base = reinterpret_cast<const uint4*>(table) + c * 32 + lane;
  f32x2 acc[4] = {0ull, 0ull, 0ull, 0ull};
  const f32x2 one = pair(1.f, 1.f);
  for (int g = blockIdx.x; g < n_groups; g += gridDim.x) {
    const int4 i0 = reinterpret_cast<const int4*>(idx)[2 * g];
    const int4 i1 = reinterpret_cast<const int4*>(idx)[2 * g + 1];
    const int r[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
    uint4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t rr = static_cast<uint32_t>(min(max(r[q], 0), rows - 1));
      v[q] = __ldg(base + rr * row16);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      fma2(acc[0], one, widen(v[q].x));
      fma2(acc[1], one, widen(v[q].y));
      fma2(acc[2], one, widen(v[q].z));
      fma2(acc[3], one, widen(v[q].w));
    }
  }
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = unpair(acc[i]);
    sum += p.x + p.y;
  }
  out[static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x] = sum;
}

cudaError_t launch_l2_gather_probe(const uint16_t* table, int rows, int d, const int32_t* idx, int n_idx, float* out,
                                   int blocks, cudaStream_t s) {
  cudaError_t e = launch(l2_gather_probe_kernel, dim3(blocks), dim3(d / 8), 0, s, table, rows, d, idx, n_idx / 8, out);
  trace_mark(s, "l2_gather_probe");
  return e;
}

int l2_gather_probe_blocks(int d) { return device_sm_count() * std::max(1, std::min(32, 48 / (d / 256))); }

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
  pdl_enter();
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
  cudaError_t e = (W == 128) ? launch(pack_dense_kernel<4>, dim3(grid), dim3(256), 0, s, A, T, I, C, nT, o.cnt, o.val,
                                      o.idx, o.row_nnz, o.ovf)
                             : launch(pack_dense_kernel<2>, dim3(grid), dim3(256), 0, s, A, T, I, C, nT, o.cnt, o.val,
                                      o.idx, o.row_nnz, o.ovf);
  trace_mark(s, "pack_dense");
  return e;
}

// ================================================================ ordered compaction
// One CTA of 1024 threads walks the rows in rounds of 4 x 1024: in a round, thread i
// owns rows base + 4 i .. base + 4 i + 3, so a warp's loads and stores cover 128
// consecutive rows (one 512-byte line run per int32 array, 128 bytes of flags). A
// block-wide exclusive scan of the threads' flagged counts, plus the rounds before,
// gives each flagged row its rank, so the list comes out in ascending row order. The
// next round's rows are loaded before the current round's scan.
namespace {
struct Rows4 {
  uint32_t flags;  // bit b: row base + 4 tid + b is flagged
  int z[4];        // their row_nnz (0 without it)
};
TW_DEV Rows4 load_rows4(const uint8_t* __restrict__ ovf, const int32_t* __restrict__ row_nnz, int R, int T, int t,
                        bool vec) {
  Rows4 r{0u, {0, 0, 0, 0}};
  uint32_t o4 = 0;
  if (vec && t + 3 < T) {
    o4 = *reinterpret_cast<const uint32_t*>(ovf + t);
    if (row_nnz != nullptr) {
      const int4 z = *reinterpret_cast<const int4*>(row_nnz + t);
      r.z[0] = z.x;
      r.z[1] = z.y;
      r.z[2] = z.z;
      r.z[3] = z.w;
    }
  } else {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      if (t + b < T) {
        o4 |= static_cast<uint32_t>(ovf[t + b] != 0) << (8 * b);
        if (row_nnz != nullptr) r.z[b] = row_nnz[t + b];
      }
    }
  }
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const bool f = ((o4 >> (8 * b)) & 0xFFu) != 0 || (row_nnz != nullptr && r.z[b] > R);
    r.flags |= (f && t + b < T ? 1u : 0u) << b;
  }
  return r;
}
}  // namespace

__global__ void __launch_bounds__(1024) compact_rows_kernel(const uint8_t* __restrict__ ovf,
                                                            const int32_t* __restrict__ row_nnz, int R, int T,
                                                            int32_t* __restrict__ list, int list_cap,
                                                            int32_t* __restrict__ count, int32_t* __restrict__ slot_of,
                                                            int32_t* __restrict__ ell_nnz, int cap_check,
                                                            int32_t* status, int32_t* zero_word, int route_mode,
                                                            float dense_above, int32_t* route_out) {
  pdl_enter();
  long long ell_sum = 0;  // row_nnz over the unflagged rows, and their number (the route decision)
  int ell_rows = 0;
  if (zero_word != nullptr && threadIdx.x == 0) *zero_word = 0;
  __shared__ int warp_tot[2][32];  // by round parity: a round's totals are read while the next round's are written
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int per_round = 4 * static_cast<int>(blockDim.x);
  const bool vec_in = reinterpret_cast<uintptr_t>(ovf) % 4 == 0 &&
                      (row_nnz == nullptr || reinterpret_cast<uintptr_t>(row_nnz) % 16 == 0);
  const bool vec_out = (slot_of == nullptr || reinterpret_cast<uintptr_t>(slot_of) % 16 == 0) &&
                       (ell_nnz == nullptr || reinterpret_cast<uintptr_t>(ell_nnz) % 16 == 0);
  int carry = 0;  // flagged rows in the rounds before
  Rows4 next = load_rows4(ovf, row_nnz, R, T, 4 * tid, vec_in);
  for (int base = 0, round = 0; base < T; base += per_round, ++round) {
    const Rows4 cur = next;
    if (base + per_round < T) next = load_rows4(ovf, row_nnz, R, T, base + per_round + 4 * tid, vec_in);
    const int c = __popc(cur.flags);
    const int incl = warp_inclusive_scan(c);
    int* wt = warp_tot[round & 1];
    if (lane == 31) wt[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const int v = lane < nwarps ? wt[lane] : 0;
      wt[lane] = warp_inclusive_scan(v);
    }
    __syncthreads();
    int pos = carry + (wid ? wt[wid - 1] : 0) + incl - c;
    carry += wt[nwarps - 1];
    const int t = base + 4 * tid;
    int sl[4], en[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const bool f = (cur.flags >> b) & 1u;
      if (f && pos < list_cap) list[pos] = t + b;
      sl[b] = f ? (pos < list_cap ? pos : -2) : -1;
      en[b] = f ? 0 : cur.z[b];
      pos += f ? 1 : 0;
      if (!f && t + b < T) {
        ell_sum += cur.z[b];
        ++ell_rows;
      }
    }
    if (vec_out && t + 3 < T) {
      if (slot_of) *reinterpret_cast<int4*>(slot_of + t) = make_int4(sl[0], sl[1], sl[2], sl[3]);
      if (ell_nnz) *reinterpret_cast<int4*>(ell_nnz + t) = make_int4(en[0], en[1], en[2], en[3]);
    } else {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (t + b < T) {
          if (slot_of) slot_of[t + b] = sl[b];
          if (ell_nnz) ell_nnz[t + b] = en[b];
        }
      }
    }
  }
  if (tid == 0) {
    *count = carry;
    if (carry > cap_check) raise_status(status, TW_ECAPACITY);
  }
  if (route_out != nullptr) {
    __shared__ long long sum_w[32];
    __shared__ int rows_w[32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ell_sum += __shfl_xor_sync(0xFFFFFFFFu, ell_sum, o);
      ell_rows += __shfl_xor_sync(0xFFFFFFFFu, ell_rows, o);
    }
    if (lane == 0) {
      sum_w[wid] = ell_sum;
      rows_w[wid] = ell_rows;
    }
    __syncthreads();
    if (tid == 0) {
      long long tot = 0;
      long long nr = 0;
      for (int w = 0; w < nwarps; ++w) {
        tot += sum_w[w];
        nr += rows_w[w];
      }
      // the sparse route's work per row, in ELL entries: an ELL row its entries, a
      // backup row 2 dense_above (its hi/lo GEMMs cost about twice the dense route's
      // per-row work, which dense_above entries price); dense when the mean is larger
      const double work = static_cast<double>(tot) + 2.0 * static_cast<double>(dense_above) * static_cast<double>(T - nr);
      const bool dense = route_mode == TW_ROUTE_DENSE ||
                         (route_mode == TW_ROUTE_AUTO && T > 0 &&
                          work > static_cast<double>(dense_above) * static_cast<double>(T));
      *route_out = dense ? 1 : 0;
    }
  }
}

cudaError_t launch_compact_rows(const uint8_t* ovf, const int32_t* row_nnz, int R, int T, int32_t* list,
                                int list_cap, int32_t* count, int32_t* slot_of, int32_t* ell_nnz, int cap_check,
                                int32_t* status, cudaStream_t s, int32_t* zero_word, int route_mode,
                                float dense_above, int32_t* route_out) {
  cudaError_t e = launch(compact_rows_kernel, dim3(1), dim3(1024), 0, s, ovf, row_nnz, R, T, list, list_cap, count,
                         slot_of, ell_nnz, cap_check, status, zero_word, route_mode, dense_above, route_out);
  trace_mark(s, "compact_rows");
  return e;
}

// ================================================================ row gather
// 16-byte pieces a lane moves per row of the row gather and scatter: rows of up to
// 2048 bf16 (d at most 2048) are 256 pieces, eight per lane.
constexpr int kRowVecs = 8;
struct GatherArgs {
  const uint16_t* src[2];
  uint16_t* out[2];
  int nsrc, d;
  int src_rows;  // rows of src (and src2): the bound of rows[i]
  const int32_t* rows;
  const int32_t* n_dev;
  int cap, rows_alloc;
  float* zero;
  int zero_row_f32;  // floats per accumulator row; rows [0, min(n, cap)) are zeroed
  int32_t* status;
  const int32_t* sparse_only;  // optional: nothing to do when *sparse_only == 1 (the dense route)
  const int32_t* zero_if_sparse;  // optional: the accumulator rows are zeroed only when this reads != 1
};
__global__ void __launch_bounds__(256) gather_rows_kernel(const GatherArgs g) {
  pdl_enter();
  if (g.sparse_only != nullptr && *g.sparse_only == 1) return;
  if (g.status != nullptr && blockIdx.x == 0 && threadIdx.x == 0 && *g.n_dev > g.cap)
    raise_status(g.status, TW_ECAPACITY);
  const int n = min(max(*g.n_dev, 0), g.cap);
  const int limit = min(g.rows_alloc, (n + 127) / 128 * 128);
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int vec = g.d / 8;
  // one warp per (row, matrix); a lane's (at most kRowVecs) 16-byte pieces of the
  // row are all loaded before any is stored, so their round trips overlap
  for (int w = blockIdx.x * wpb + (threadIdx.x >> 5); w < limit * g.nsrc; w += gridDim.x * wpb) {
    const int i = w / g.nsrc, which = w - i * g.nsrc;
    uint4* o = reinterpret_cast<uint4*>((which ? g.out[1] : g.out[0]) + static_cast<size_t>(i) * g.d);
    uint4 v[kRowVecs];
#pragma unroll
    for (int q = 0; q < kRowVecs; ++q) v[q] = make_uint4(0, 0, 0, 0);
    if (i < n && TW_CHECKED(g.rows[i] >= 0 && g.rows[i] < g.src_rows, g.status)) {
      const uint4* r =
          reinterpret_cast<const uint4*>((which ? g.src[1] : g.src[0]) + static_cast<size_t>(g.rows[i]) * g.d);
#pragma unroll
      for (int q = 0; q < kRowVecs; ++q)
        if (lane + 32 * q < vec) v[q] = __ldg(r + lane + 32 * q);
    }
#pragma unroll
    for (int q = 0; q < kRowVecs; ++q)
      if (lane + 32 * q < vec) o[lane + 32 * q] = v[q];
  }
  // the accumulator rows the split-K product adds into: 16-byte stores over the grid
  const bool zero = g.zero_if_sparse == nullptr || *g.zero_if_sparse != 1;
  const size_t z4 = zero ? static_cast<size_t>(n) * g.zero_row_f32 / 4 : 0;
  for (size_t k = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < z4;
       k += static_cast<size_t>(gridDim.x) * blockDim.x)
    reinterpret_cast<float4*>(g.zero)[k] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// out[row_map[i]][:] = bf16(acc[i][0 .. N)) for i < min(*n, cap) (acc rows of stride
// lda): the finished rows of a split-K product. One warp per row, 8 columns per lane
// per step.
__global__ void __launch_bounds__(256) scatter_rows_bf16_kernel(const float* __restrict__ acc, int N, int lda,
                                                                const int32_t* __restrict__ n_dev, int cap,
                                                                const int32_t* __restrict__ row_map,
                                                                uint16_t* __restrict__ out, int ldo, int out_rows,
                                                                const int32_t* sparse_only) {
  pdl_enter();
  if (sparse_only != nullptr && *sparse_only == 1) return;
  const int n = min(max(*n_dev, 0), cap);
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int i = blockIdx.x * wpb + (threadIdx.x >> 5); i < n; i += gridDim.x * wpb) {
    if (!TW_CHECKED(row_map[i] >= 0 && row_map[i] < out_rows, nullptr)) continue;
    const float4* src = reinterpret_cast<const float4*>(acc + static_cast<size_t>(i) * lda);
    uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(row_map[i]) * ldo);
    // all of the lane's (at most kRowVecs) pieces are loaded before any is stored
    float4 a[kRowVecs], b[kRowVecs];
#pragma unroll
    for (int q = 0; q < kRowVecs; ++q) {
      const int c = lane + 32 * q;
      if (c < N / 8) {
        a[q] = src[2 * c];
        b[q] = src[2 * c + 1];
      }
    }
#pragma unroll
    for (int q = 0; q < kRowVecs; ++q) {
      const int c = lane + 32 * q;
      if (c < N / 8)
        dst[c] = make_uint4(pack_bf16x2(a[q].x, a[q].y), pack_bf16x2(a[q].z, a[q].w), pack_bf16x2(b[q].x, b[q].y),
                            pack_bf16x2(b[q].z, b[q].w));
    }
  }
}

cudaError_t launch_scatter_rows_bf16(const float* acc, int N, const int32_t* n_dev, int cap, const int32_t* row_map,
                                     uint16_t* out, int ldo, int out_rows, cudaStream_t s, const int32_t* sparse_only,
                                     int ld_acc) {
  if (cap <= 0) return cudaSuccess;
  const int lda = ld_acc > 0 ? ld_acc : N;
  if (N % 8 != 0 || N > 8 * 32 * kRowVecs || lda < N || lda % 4 != 0) return cudaErrorInvalidValue;
  cudaError_t e = launch(scatter_rows_bf16_kernel, dim3(std::min(warp_grid(cap, 8), device_sm_count() * 2)), dim3(256),
                         0, s, acc, N, lda, n_dev, cap, row_map, out, ldo, out_rows, sparse_only);
  trace_mark(s, "scatter_rows");
  return e;
}

// ------------------------------------------------------------------ split-K backup: finishing kernels
// Both take eight columns of one row a thread-step over rows [0, round_up(n, 128))
// (below rows_alloc); rows past n get zeros in the bf16 outputs, as the direct forms'
// epilogues write them (the later GEMMs read whole 64-row K blocks of them).
namespace {
struct Row8 {
  float v[8];
};
TW_DEV Row8 load8(const float* p) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  return Row8{{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w}};
}
TW_DEV void store8(float* p, const Row8& r) {
  reinterpret_cast<float4*>(p)[0] = make_float4(r.v[0], r.v[1], r.v[2], r.v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(r.v[4], r.v[5], r.v[6], r.v[7]);
}
// the bf16 pair of eight values: hi = bf16(v), lo = bf16(v - hi)
TW_DEV void store_pair8(uint16_t* hi, uint16_t* lo, size_t off, const Row8& r) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float v0 = r.v[2 * q], v1 = r.v[2 * q + 1];
    h[q] = pack_bf16x2_rn(v0, v1);
    l[q] = pack_bf16x2_rn(v0 - bf16_lo(h[q]), v1 - bf16_hi(h[q]));
  }
  *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
}
int finish_grid(int rows_alloc, int I) {
  const long work = static_cast<long>(rows_alloc) * (I / 8);
  return static_cast<int>(std::max(1L, std::min<long>((work + 255) / 256, device_sm_count() * 4L)));
}
}  // namespace

// Forward: row i < n of acc holds g (columns [0, I)) and, gated, u ([I, 2 I)):
// a = ReLU(g) (strictly positive g), h = a u (non-gated: a) as the pair H + H_lo, and
// the saved fp32 a and u. A route word reading 1 (the dense route) skips H and H_lo.
// from_saved: acc is save_a, already ReLU(g), u is save_u's row; only H, H_lo.
__global__ void __launch_bounds__(256) backup_hidden_finish_kernel(const float* acc, int ld,
                                                                   const int32_t* __restrict__ n_dev, int cap, int I,
                                                                   bool gated, uint16_t* __restrict__ H,
                                                                   uint16_t* __restrict__ H_lo, int rows_alloc,
                                                                   float* save_a, float* save_u, const int32_t* route,
                                                                   bool from_saved) {
  pdl_enter();
  const bool want_h = route == nullptr || *route != 1;
  if (from_saved && !want_h) return;
  const int n = min(max(*n_dev, 0), cap);
  const int rows = min(rows_alloc, (n + 127) / 128 * 128);
  const int v8 = I / 8;
  const long total = static_cast<long>(rows) * v8;
  for (long k = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; k < total;
       k += static_cast<long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(k / v8);
    const int c = static_cast<int>(k - static_cast<long>(r) * v8) * 8;
    const size_t o = static_cast<size_t>(r) * I + c;
    Row8 h{};
    if (r < n) {
      const float* row = acc + static_cast<size_t>(r) * ld;
      Row8 a = load8(row + c);
      Row8 u{};
      if (gated) u = load8(from_saved ? save_u + o : row + I + c);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        a.v[e] = a.v[e] > 0.f ? a.v[e] : 0.f;
        h.v[e] = gated ? a.v[e] * u.v[e] : a.v[e];
      }
      if (!from_saved) {
        if (save_a != nullptr) store8(save_a + o, a);
        if (gated && save_u != nullptr) store8(save_u + o, u);
      }
    }
    if (want_h) store_pair8(H, H_lo, o, h);
  }
}

// Backward: row i < n of acc holds dh = dY Wd^T (columns [0, I)); with the saved fp32
// a and u, dg = (dh u + l1) where a > 0 (non-gated: dh + l1), du = dh a where a > 0,
// h = a u (non-gated: a), each as a bf16 pair.
__global__ void __launch_bounds__(256) backup_grad_finish_kernel(const float* __restrict__ acc, int ld,
                                                                 const int32_t* __restrict__ n_dev, int cap, int I,
                                                                 const float* __restrict__ a_sv,
                                                                 const float* __restrict__ u_sv, float l1,
                                                                 const BackupGradOut o, int rows_alloc,
                                                                 const int32_t* sparse_only) {
  pdl_enter();
  if (sparse_only != nullptr && *sparse_only == 1) return;
  const bool gated = u_sv != nullptr;
  const int n = min(max(*n_dev, 0), cap);
  const int rows = min(rows_alloc, (n + 127) / 128 * 128);
  const int v8 = I / 8;
  const long total = static_cast<long>(rows) * v8;
  for (long k = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; k < total;
       k += static_cast<long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(k / v8);
    const int c = static_cast<int>(k - static_cast<long>(r) * v8) * 8;
    const size_t off = static_cast<size_t>(r) * I + c;
    Row8 dg{}, du{}, h{};
    if (r < n) {
      const Row8 dh = load8(acc + static_cast<size_t>(r) * ld + c);
      const Row8 a = load8(a_sv + off);
      Row8 u{};
      if (gated) u = load8(u_sv + off);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const bool act = a.v[e] > 0.f;
        dg.v[e] = act ? (gated ? dh.v[e] * u.v[e] : dh.v[e]) + l1 : 0.f;
        du.v[e] = act ? dh.v[e] * a.v[e] : 0.f;
        h.v[e] = gated ? a.v[e] * u.v[e] : a.v[e];
      }
    }
    store_pair8(o.dG, o.dG_lo, off, dg);
    if (gated) store_pair8(o.dU, o.dU_lo, off, du);
    store_pair8(o.H, o.H_lo, off, h);
  }
}

cudaError_t launch_backup_hidden_finish(const float* acc, int ld, const int32_t* n_dev, int cap, int I, bool gated,
                                        uint16_t* H, uint16_t* H_lo, int rows_alloc, float* save_a, float* save_u,
                                        const int32_t* route, cudaStream_t s, bool from_saved) {
  if (cap <= 0 || rows_alloc <= 0) return cudaSuccess;
  if (I % 8 != 0 || ld % 4 != 0) return cudaErrorInvalidValue;
  cudaError_t e = launch(backup_hidden_finish_kernel, dim3(finish_grid(rows_alloc, I)), dim3(256), 0, s, acc, ld,
                         n_dev, cap, I, gated, H, H_lo, rows_alloc, save_a, save_u, route, from_saved);
  trace_mark(s, "backup_hidden_finish");
  return e;
}

cudaError_t launch_backup_grad_finish(const float* acc, int ld, const int32_t* n_dev, int cap, int I, const float* a,
                                      const float* u, float l1, const BackupGradOut& o, int rows_alloc,
                                      const int32_t* sparse_only, cudaStream_t s) {
  if (cap <= 0 || rows_alloc <= 0) return cudaSuccess;
  if (I % 8 != 0 || ld % 4 != 0) return cudaErrorInvalidValue;
  cudaError_t e = launch(backup_grad_finish_kernel, dim3(finish_grid(rows_alloc, I)), dim3(256), 0, s, acc, ld, n_dev,
                         cap, I, a, u, l1, o, rows_alloc, sparse_only);
  trace_mark(s, "backup_grad_finish");
  return e;
}

cudaError_t launch_gather_rows(const uint16_t* src, int d, int src_rows, const int32_t* rows, const int32_t* n, int cap,
                               int rows_alloc, uint16_t* out, cudaStream_t s, int32_t* status, const uint16_t* src2,
                               uint16_t* out2, float* zero, int zero_row_f32, const int32_t* sparse_only,
                               const int32_t* zero_if_sparse) {
  if (rows_alloc <= 0) return cudaSuccess;
  if (d % 8 != 0 || d > 8 * 32 * kRowVecs) return cudaErrorInvalidValue;
  if (zero_row_f32 % 4 != 0 || (zero != nullptr && reinterpret_cast<uintptr_t>(zero) % 16 != 0))
    return cudaErrorInvalidValue;
  GatherArgs g{};
  g.src[0] = src;
  g.out[0] = out;
  g.src[1] = src2;
  g.out[1] = out2;
  g.nsrc = (src2 != nullptr && out2 != nullptr) ? 2 : 1;
  g.d = d;
  g.src_rows = src_rows;
  g.rows = rows;
  g.n_dev = n;
  g.cap = cap;
  g.rows_alloc = rows_alloc;
  g.zero = zero;
  g.zero_row_f32 = zero != nullptr ? zero_row_f32 : 0;
  g.status = status;
  g.sparse_only = sparse_only;
  g.zero_if_sparse = zero_if_sparse;
  const long work = static_cast<long>(rows_alloc) * g.nsrc;
  const int grid = warp_grid(work, 8);
  cudaError_t e = launch(gather_rows_kernel, dim3(std::min(grid, device_sm_count() * 4)), dim3(256), 0, s, g);
  trace_mark(s, "gather_rows");
  return e;
}

}  // namespace tw

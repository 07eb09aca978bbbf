// CUDA-core kernels of the sparse part of the FFN (gist.science explainer, 2.B:
// "Fused Up/Down Projection" for inference, "Sparse MatMul" and "Backpropagation"
// for training), organised for GB300's memory system.
//
// Every stored entry (t, j) costs whole d-vector gathers of weight rows (Wu[j],
// Wd[j], Wg[j]) or token rows (x_t, dy_t). They are served from the 129 MB L2, which
// delivers ~20 TB/s of random-row gathers only when every SM keeps ~30 rows (4 KB
// each) in flight all the time. Register-resident accumulators (x_t, y_t, dx_t) leave
// no room for that many rows in registers, so the row passes stream weight rows
// through a small per-warp shared-memory ring filled by bulk copies (cp.async.bulk)
// that lane 0 issues a few rows ahead:
//
//  forward   warp per token: enumerate the token's TwELL entries into a shared-memory
//            list (j, a); stream Wu[j] rows: u = x_t . Wu[j], h = a u (gated); then
//            stream Wd[j] rows: y_t = sum h Wd[j]                 (x_t, then y_t, in registers)
//  dh        warp per ELL token: stream Wd[j]: dh = dy_t . Wd[j];
//            dg = dh u + l1 (non-gated: dh + l1), du = dh a; counts the columns of
//            the transposed Hybrid                                 (dy_t in registers)
//  dx        warp per ELL token: stream Wg[j], Wu[j]: dx_t = sum dg Wg[j] + du Wu[j]
//  dW        warp per (256-wide slice of d, neuron j) over the transposed Hybrid:
//            dWg[j] = sum dg x_t, dWu[j] = sum du x_t, dWd[j] = sum a u dy_t;
//            slices outermost so the x / dy slices in use stay in L2, and the fp32
//            gradient rows are written with streaming stores that do not evict them.
//
// Lane l of a warp owns elements [256 q + 8 l, 256 q + 8 l + 8) of each 256-wide
// chunk q of a d-vector, so every shared-memory row read is conflict-free and every
// direct global read is a coalesced 512-byte transaction.
#include <algorithm>

#include "tw_common.cuh"
#include "tw_internal.h"

namespace tw {

namespace {

constexpr int kFwdRing = 2;   // row slots per warp
constexpr int kDhRing = 3;
constexpr int kDxRing = 3;
constexpr int kWgradUnroll = 8;

// ---------------------------------------------------------------- row arithmetic
// These loops are bound by instruction issue, so they use Blackwell's
// mixed-precision FMA (bf16 x bf16 + fp32: the product of two bf16 values is exact
// in fp32, one rounding per FMA, like converting first) for dot products, and its
// packed fp32x2 FMA for axpys. Eight fp32 accumulators live as four packed pairs.
typedef unsigned long long f32x2;
struct F8 {
  f32x2 v[4];
};
TW_DEV void f8_zero(F8& a) { a.v[0] = a.v[1] = a.v[2] = a.v[3] = 0ull; }
TW_DEV f32x2 f2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
TW_DEV float2 f2_split(f32x2 v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return make_float2(lo, hi);
}
TW_DEV f32x2 bf16x2_to_f32x2(uint32_t w) { return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)); }
TW_DEV void fma2(f32x2& acc, f32x2 a, f32x2 b) { asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b)); }
// y += h * w over 8 bf16 elements (h2 = {h, h})
TW_DEV void axpy8(F8& y, f32x2 h2, const uint4& w) {
  fma2(y.v[0], h2, bf16x2_to_f32x2(w.x));
  fma2(y.v[1], h2, bf16x2_to_f32x2(w.y));
  fma2(y.v[2], h2, bf16x2_to_f32x2(w.z));
  fma2(y.v[3], h2, bf16x2_to_f32x2(w.w));
}
// g += cg * x and u += cu * x sharing one conversion of x
TW_DEV void axpy8_two(F8& g, f32x2 cg2, F8& u, f32x2 cu2, const uint4& x) {
  const f32x2 x0 = bf16x2_to_f32x2(x.x), x1 = bf16x2_to_f32x2(x.y), x2 = bf16x2_to_f32x2(x.z),
              x3 = bf16x2_to_f32x2(x.w);
  fma2(g.v[0], cg2, x0);
  fma2(g.v[1], cg2, x1);
  fma2(g.v[2], cg2, x2);
  fma2(g.v[3], cg2, x3);
  fma2(u.v[0], cu2, x0);
  fma2(u.v[1], cu2, x1);
  fma2(u.v[2], cu2, x2);
  fma2(u.v[3], cu2, x3);
}
TW_DEV uint4 pack8(const F8& y) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = f2_split(y.v[i]);
    w[i] = pack_bf16x2(p.x, p.y);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
TW_DEV void stcs_f32x8(float* p, const F8& y) {
  const float2 a = f2_split(y.v[0]), b = f2_split(y.v[1]), c = f2_split(y.v[2]), d = f2_split(y.v[3]);
  __stcs(reinterpret_cast<float4*>(p), make_float4(a.x, a.y, b.x, b.y));
  __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(c.x, c.y, d.x, d.y));
}
// p[0..3] += x . w over 8 bf16 pairs (mixed-precision FMA, four partial sums)
TW_DEV void dot8(const uint4& x, const uint4& w, float (&p)[4]) {
  asm("{\n\t"
      ".reg .b16 x0, x1, x2, x3, x4, x5, x6, x7, w0, w1, w2, w3, w4, w5, w6, w7;\n\t"
      "mov.b32 {x0, x1}, %4;\n\t"
      "mov.b32 {x2, x3}, %5;\n\t"
      "mov.b32 {x4, x5}, %6;\n\t"
      "mov.b32 {x6, x7}, %7;\n\t"
      "mov.b32 {w0, w1}, %8;\n\t"
      "mov.b32 {w2, w3}, %9;\n\t"
      "mov.b32 {w4, w5}, %10;\n\t"
      "mov.b32 {w6, w7}, %11;\n\t"
      "fma.rn.f32.bf16 %0, x0, w0, %0;\n\t"
      "fma.rn.f32.bf16 %1, x1, w1, %1;\n\t"
      "fma.rn.f32.bf16 %2, x2, w2, %2;\n\t"
      "fma.rn.f32.bf16 %3, x3, w3, %3;\n\t"
      "fma.rn.f32.bf16 %0, x4, w4, %0;\n\t"
      "fma.rn.f32.bf16 %1, x5, w5, %1;\n\t"
      "fma.rn.f32.bf16 %2, x6, w6, %2;\n\t"
      "fma.rn.f32.bf16 %3, x7, w7, %3;\n\t"
      "}"
      : "+f"(p[0]), "+f"(p[1]), "+f"(p[2]), "+f"(p[3])
      : "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w), "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w));
}
TW_DEV uint4 ldg16(const uint4* p) { return __ldg(p); }
// dot product of a lane's NCH chunks with a row in shared memory
template <int NCH>
TW_DEV float dot_row(const uint4 (&xv)[NCH], const uint4* row, int lane) {
  float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int q = 0; q < NCH; ++q) dot8(xv[q], row[q * 32 + lane], p);
  return (p[0] + p[1]) + (p[2] + p[3]);
}

int grid_for(long items, int per_block, int blocks_per_sm) {
  const long blocks = (items + per_block - 1) / per_block;
  return static_cast<int>(
      std::max<long>(1, std::min<long>(blocks, static_cast<long>(device_sm_count()) * blocks_per_sm)));
}

__host__ __device__ constexpr uint32_t round_up_u(uint32_t v, uint32_t m) { return (v + m - 1) / m * m; }

// shared memory of one forward warp: ring | neuron list (u16) | h list (f32)
__host__ __device__ inline uint32_t fwd_warp_smem(int nch, int L) {
  return round_up_u(kFwdRing * nch * 512u + round_up_u(2u * L, 16u) + 4u * L, 128u);
}

}  // namespace

// ====================================================================== forward
// Rows served by the dense path (TwELL overflow, Hybrid backup) are skipped. The
// token's entries come from the TwELL counts tile by tile (ballot over tiles with a
// nonzero count; the first cnt lanes take the tile's slots), i.e. in ascending
// neuron order, into the warp's list; in training they also go to the Hybrid ELL.
// The warp's row stream is then Wu[j_0..j_n-1] (gated only) followed by
// Wd[j_0..j_n-1]. The list holds up to a.L = (I / W) * C entries, the most a
// non-overflow row has.
template <int NCH, bool GATED, bool HYBRID>
__global__ void __launch_bounds__(256) sparse_fwd_kernel(const SparseFwdArgs a, int32_t* status) {
  constexpr int S = kFwdRing;
  constexpr uint32_t ROWB = NCH * 512;
  constexpr int d = NCH * 256;
  extern __shared__ __align__(128) uint8_t fwd_smem[];
  __shared__ uint64_t bars[8 * S];
  __shared__ int abort_flag;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  uint8_t* wbase = fwd_smem + static_cast<size_t>(warp) * fwd_warp_smem(NCH, a.L);
  WarpRing<S> ring{wbase, bars + warp * S, ROWB};
  uint16_t* lj = reinterpret_cast<uint16_t*>(wbase + S * ROWB);
  float* lh = reinterpret_cast<float*>(wbase + S * ROWB + round_up_u(2u * a.L, 16u));
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  ring.init(lane);

  uint32_t g = 0;  // rows of this warp's stream consumed so far
  for (int t = blockIdx.x * wpb + warp; t < a.T; t += gridDim.x * wpb) {
    const bool skip = HYBRID ? (a.backup_slot[t] != -1) : (a.ovf[t] != 0);
    if (skip) continue;
    // ------------------------------------------------------------ entry list
    const size_t rb = static_cast<size_t>(t) * a.R;
    const uint16_t* cnt_row = a.cnt + static_cast<size_t>(t) * a.nT;
    int n = 0;
    for (int kb = 0; kb < a.nT; kb += 32) {
      const int k = kb + lane;
      const int c = (k < a.nT) ? min(static_cast<int>(cnt_row[k]), a.C) : 0;
      unsigned mask = __ballot_sync(0xFFFFFFFFu, c > 0);
      while (mask) {
        const int src = __ffs(mask) - 1;
        mask &= mask - 1;
        const int kk = kb + src;
        const int cc = __shfl_sync(0xFFFFFFFFu, c, src);
        if (lane < cc) {
          const size_t sb = (static_cast<size_t>(t) * a.nT + kk) * a.C + lane;
          const int j = kk * a.W + a.idx[sb];
          const uint16_t ab = a.val[sb];
          lj[n + lane] = static_cast<uint16_t>(j);
          lh[n + lane] = bf16_to_f32(ab);
          if (HYBRID) {
            a.ell_idx[rb + n + lane] = static_cast<uint16_t>(j);
            a.ell_a[rb + n + lane] = ab;
          }
        }
        n += cc;
      }
    }
    __syncwarp();
    const int total = GATED ? 2 * n : n;
    auto row_src = [&](int k) -> const uint16_t* {
      if (GATED && k < n) return a.Wu + static_cast<size_t>(lj[k]) * d;
      return a.Wd + static_cast<size_t>(lj[GATED ? k - n : k]) * d;
    };
    if (lane == 0)
      for (int k = 0; k < S && k < total; ++k) ring.issue(g + k, row_src(k));
    int k = 0;
    bool ok = true;
    // ------------------------------------------------------------ up: h = a (x_t . Wu[j])
    if (GATED) {
      uint4 xv[NCH];
      const uint4* xr = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * d);
#pragma unroll
      for (int q = 0; q < NCH; ++q) xv[q] = ldg16(xr + q * 32 + lane);
      for (; k < n; ++k) {
        if (!ring.wait(g + k, &abort_flag, status)) {
          ok = false;
          break;
        }
        const float u = warp_sum(dot_row<NCH>(xv, reinterpret_cast<const uint4*>(ring.slot(g + k)), lane));
        if (lane == 0) {
          lh[k] *= u;
          if (HYBRID) a.ell_u[rb + k] = f32_to_bf16(u);
        }
        __syncwarp();
        if (lane == 0 && k + S < total) {
          fence_proxy_async_smem();
          ring.issue(g + k + S, row_src(k + S));
        }
      }
    }
    // ------------------------------------------------------------ down: y_t = sum h Wd[j]
    if (ok) {
      F8 y[NCH];
#pragma unroll
      for (int q = 0; q < NCH; ++q) f8_zero(y[q]);
      for (; k < total; ++k) {
        if (!ring.wait(g + k, &abort_flag, status)) {
          ok = false;
          break;
        }
        const float h = lh[GATED ? k - n : k];
        const f32x2 h2 = f2(h, h);
        const uint4* row = reinterpret_cast<const uint4*>(ring.slot(g + k));
#pragma unroll
        for (int q = 0; q < NCH; ++q) axpy8(y[q], h2, row[q * 32 + lane]);
        __syncwarp();
        if (lane == 0 && k + S < total) {
          fence_proxy_async_smem();
          ring.issue(g + k + S, row_src(k + S));
        }
      }
      if (ok) {
        uint4* yr = reinterpret_cast<uint4*>(a.y + static_cast<size_t>(t) * d);
#pragma unroll
        for (int q = 0; q < NCH; ++q) yr[q * 32 + lane] = pack8(y[q]);
      }
    }
    if (!ok) {
      if (lane == 0) ring.drain(g + k, g + min(total, k + S));
      break;
    }
    g += total;
    __syncwarp();  // the list is rewritten by the next token
  }
}

// ====================================================================== backward: dh
// One warp per ELL token, dy_t in registers, the row stream is Wd[j_0..j_n-1].
// Lane l holds entry 32 b + l of the current batch b (neuron, a, u) and the neurons
// of batch b + 1, which is all the producer needs to issue rows up to 32 ahead.
//   dh = dy_t . Wd[j];  dg = dh u + l1 (non-gated: dh + l1);  du = dh a.
// Also counts the entries of every neuron column for the transposed Hybrid.
template <int NCH, bool GATED>
__global__ void __launch_bounds__(256) sparse_dh_kernel(const SparseBwdArgs a, int32_t* status) {
  constexpr int S = kDhRing;
  constexpr uint32_t ROWB = NCH * 512;
  constexpr int d = NCH * 256;
  extern __shared__ __align__(128) uint8_t dh_smem[];
  __shared__ uint64_t bars[8 * S];
  __shared__ int abort_flag;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  WarpRing<S> ring{dh_smem + static_cast<size_t>(warp) * S * ROWB, bars + warp * S, ROWB};
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  ring.init(lane);
  uint32_t g = 0;
  for (int t = blockIdx.x * wpb + warp; t < a.T; t += gridDim.x * wpb) {
    const int n = a.ell_nnz[t];
    if (n == 0) continue;
    const size_t rb = static_cast<size_t>(t) * a.R;
    auto load_j = [&](int e) { return e < n ? static_cast<int>(a.ell_idx[rb + e]) : 0; };
    int jcur = load_j(lane), jnxt = load_j(32 + lane);
    if (lane < n) atomicAdd(a.col_cnt + jcur, 1);
    if (32 + lane < n) atomicAdd(a.col_cnt + jnxt, 1);
    for (int k = 0; k < S && k < n; ++k) {
      const int j = __shfl_sync(0xFFFFFFFFu, k < 32 ? jcur : jnxt, k & 31);
      if (lane == 0) ring.issue(g + k, a.Wd + static_cast<size_t>(j) * d);
    }
    uint4 dyv[NCH];
    const uint4* dyr = reinterpret_cast<const uint4*>(a.dy + static_cast<size_t>(t) * d);
#pragma unroll
    for (int q = 0; q < NCH; ++q) dyv[q] = ldg16(dyr + q * 32 + lane);
    float acur = 0.f, ucur = 1.f, dg_keep = 0.f, du_keep = 0.f;
    bool ok = true;
    int k = 0;
    for (; k < n; ++k) {
      if ((k & 31) == 0) {  // new batch: coefficients of its entries, neurons of the one after
        if (k > 0) {
          jcur = jnxt;
          jnxt = load_j(k + 32 + lane);
          if (k + 32 + lane < n) atomicAdd(a.col_cnt + jnxt, 1);
        }
        acur = (k + lane < n) ? bf16_to_f32(a.ell_a[rb + k + lane]) : 0.f;
        ucur = (GATED && k + lane < n) ? bf16_to_f32(a.ell_u[rb + k + lane]) : 1.f;
      }
      if (!ring.wait(g + k, &abort_flag, status)) {
        ok = false;
        break;
      }
      const float dh = warp_sum(dot_row<NCH>(dyv, reinterpret_cast<const uint4*>(ring.slot(g + k)), lane));
      if (lane == (k & 31)) {
        dg_keep = (GATED ? dh * ucur : dh) + a.l1;
        du_keep = dh * acur;
      }
      __syncwarp();
      const int kn = k + S;
      if (kn < n) {
        const int j = __shfl_sync(0xFFFFFFFFu, (kn >> 5) == (k >> 5) ? jcur : jnxt, kn & 31);
        if (lane == 0) {
          fence_proxy_async_smem();
          ring.issue(g + kn, a.Wd + static_cast<size_t>(j) * d);
        }
      }
      if ((k & 31) == 31 || k == n - 1) {  // batch done: its lanes store their coefficients
        const int e = (k & ~31) + lane;
        if (e < n) {
          a.dg[rb + e] = dg_keep;
          if (GATED) a.du[rb + e] = du_keep;
        }
      }
    }
    if (!ok) {
      if (lane == 0) ring.drain(g + k, g + min(n, k + S));
      break;
    }
    g += n;
  }
}

// ====================================================================== backward: dx
// One warp per ELL token, dx_t accumulated in registers (fp32), the row stream is
// Wg[j_0], Wu[j_0], Wg[j_1], Wu[j_1], ... (non-gated: Wg only):
//   dx_t = sum over entries of dg Wg[j] + du Wu[j].
// Tokens without ELL entries get dx = 0 (backup rows are overwritten by the dense
// path afterwards).
template <int NCH, bool GATED>
__global__ void __launch_bounds__(256) sparse_dx_kernel(const SparseBwdArgs a, int32_t* status) {
  constexpr int S = kDxRing;
  constexpr int RPE = GATED ? 2 : 1;  // rows per entry
  constexpr uint32_t ROWB = NCH * 512;
  constexpr int d = NCH * 256;
  extern __shared__ __align__(128) uint8_t dx_smem[];
  __shared__ uint64_t bars[8 * S];
  __shared__ int abort_flag;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  WarpRing<S> ring{dx_smem + static_cast<size_t>(warp) * S * ROWB, bars + warp * S, ROWB};
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  ring.init(lane);
  uint32_t g = 0;
  for (int t = blockIdx.x * wpb + warp; t < a.T; t += gridDim.x * wpb) {
    const int n = a.ell_nnz[t];
    F8 acc[NCH];
#pragma unroll
    for (int q = 0; q < NCH; ++q) f8_zero(acc[q]);
    const size_t rb = static_cast<size_t>(t) * a.R;
    const int total = RPE * n;
    bool ok = true;
    int k = 0;
    if (n > 0) {
      auto load_j = [&](int e) { return e < n ? static_cast<int>(a.ell_idx[rb + e]) : 0; };
      int jcur = load_j(lane), jnxt = load_j(32 + lane);
      auto src_of = [&](int kk, int j) -> const uint16_t* {
        return ((GATED && (kk & 1)) ? a.Wu : a.Wg) + static_cast<size_t>(j) * d;
      };
      for (int kk = 0; kk < S && kk < total; ++kk) {
        const int e = kk / RPE;
        const int j = __shfl_sync(0xFFFFFFFFu, e < 32 ? jcur : jnxt, e & 31);
        if (lane == 0) ring.issue(g + kk, src_of(kk, j));
      }
      float gcur = 0.f, ucur = 0.f;
      for (; k < total; ++k) {
        const int e = k / RPE;
        if ((k % (32 * RPE)) == 0) {
          if (k > 0) {
            jcur = jnxt;
            jnxt = load_j(e + 32 + lane);
          }
          gcur = (e + lane < n) ? a.dg[rb + e + lane] : 0.f;
          ucur = (GATED && e + lane < n) ? a.du[rb + e + lane] : 0.f;
        }
        if (!ring.wait(g + k, &abort_flag, status)) {
          ok = false;
          break;
        }
        const float c = __shfl_sync(0xFFFFFFFFu, (GATED && (k & 1)) ? ucur : gcur, e & 31);
        const f32x2 c2 = f2(c, c);
        const uint4* row = reinterpret_cast<const uint4*>(ring.slot(g + k));
#pragma unroll
        for (int q = 0; q < NCH; ++q) axpy8(acc[q], c2, row[q * 32 + lane]);
        __syncwarp();
        const int kn = k + S;
        if (kn < total) {
          const int en = kn / RPE;
          const int j = __shfl_sync(0xFFFFFFFFu, (en >> 5) == (e >> 5) ? jcur : jnxt, en & 31);
          if (lane == 0) {
            fence_proxy_async_smem();
            ring.issue(g + kn, src_of(kn, j));
          }
        }
      }
    }
    if (!ok) {
      if (lane == 0) ring.drain(g + k, g + min(total, k + S));
      break;
    }
    uint4* dr = reinterpret_cast<uint4*>(a.dx + static_cast<size_t>(t) * d);
#pragma unroll
    for (int q = 0; q < NCH; ++q) dr[q * 32 + lane] = pack8(acc[q]);
    g += total;
  }
}

// ====================================================================== transposed Hybrid
// Exclusive scan of the per-neuron counts (one CTA, each thread a run of consecutive
// neurons): col_ptr[0..I], col_cur = col_ptr.
__global__ void __launch_bounds__(1024) csc_scan_kernel(const int32_t* __restrict__ col_cnt, int I,
                                                        int32_t* __restrict__ col_ptr, int32_t* __restrict__ col_cur) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int per = (I + blockDim.x - 1) / blockDim.x;
  const int lo = min(I, tid * per), hi = min(I, lo + per);
  int sum = 0;
  for (int j = lo; j < hi; ++j) sum += col_cnt[j];
  const int incl = warp_inclusive_scan(sum);
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int v = lane < (blockDim.x >> 5) ? warp_tot[lane] : 0;
    warp_tot[lane] = warp_inclusive_scan(v);
  }
  __syncthreads();
  int run = (wid ? warp_tot[wid - 1] : 0) + incl - sum;
  for (int j = lo; j < hi; ++j) {
    col_ptr[j] = run;
    col_cur[j] = run;
    run += col_cnt[j];
  }
  if (tid == blockDim.x - 1) col_ptr[I] = warp_tot[(blockDim.x >> 5) - 1];
}

// Scatters every ELL entry into its column of the transposed Hybrid as one
// 16-byte record {token row offset in 16-byte units, dg, du, h = a u (non-gated: a)},
// so the weight-gradient pass reads one coalesced record per entry and nothing else
// but the gathered rows.
template <bool GATED>
__global__ void __launch_bounds__(256) csc_fill_kernel(const SparseBwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const uint32_t row16 = static_cast<uint32_t>(a.d / 8);
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < a.T; t += gridDim.x * wpb) {
    const int n = a.ell_nnz[t];
    for (int s = lane; s < n; s += 32) {
      const size_t e = static_cast<size_t>(t) * a.R + s;
      const float av = bf16_to_f32(a.ell_a[e]);
      const float h = GATED ? av * bf16_to_f32(a.ell_u[e]) : av;
      const uint4 rec = make_uint4(static_cast<uint32_t>(t) * row16, __float_as_uint(a.dg[e]),
                                   GATED ? __float_as_uint(a.du[e]) : 0u, __float_as_uint(h));
      a.csc[atomicAdd(a.col_cur + a.ell_idx[e], 1)] = rec;
    }
  }
}

// ====================================================================== backward: dW
// One warp per (256-wide slice c of d, neuron j, side), slices outermost, so that
// while slice c is processed only x[:, slice c] and dy[:, slice c] (16 MB at
// T = 16384) are gathered: they stay in L2. The x side accumulates
//   dWg[j] += dg x_t,  dWu[j] += du x_t   (gated)
// and the dy side
//   dWd[j] += h dy_t,  h = a u (non-gated: a)
// (fp32, overwritten, streaming stores); splitting the sides halves the registers a
// warp needs, so more warps and more row slices are in flight per SM. Lane l owns 8
// columns of the slice. The column's records are staged 32 at a time in the warp's
// shared memory with the coefficients already paired for the packed FMA
// ({dg, dg, du, du}, {h, h, row}); a chunk whose length is not a multiple of the
// unroll is padded with zero coefficients on the chunk's last row (an L1 hit), so
// the inner loop has no predication and keeps kWgradUnroll row slices in flight.
template <bool GATED>
__global__ void __launch_bounds__(256, 3) ell_weight_grad_kernel(const SparseBwdArgs a) {
  constexpr int U = kWgradUnroll;
  static_assert(32 % U == 0, "the unroll must divide the staging chunk");
  __shared__ float4 stage[8][2][32];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wpb = blockDim.x >> 5;
  float4(&cgu)[32] = stage[warp][0];
  float4(&chr)[32] = stage[warp][1];
  const int items = (a.d / 256) * a.I * 2;
  for (int it = blockIdx.x * wpb + warp; it < items; it += gridDim.x * wpb) {
    const bool xside = (it & 1) == 0;
    const int cj = it >> 1;
    const int c = cj / a.I;
    const int j = cj - c * a.I;
    const uint4* src = reinterpret_cast<const uint4*>(xside ? a.x : a.dy) + c * 32 + lane;
    const int lo = a.col_ptr[j], hi = a.col_ptr[j + 1];
    F8 p, q2;
    f8_zero(p);
    f8_zero(q2);
    for (int e0 = lo; e0 < hi; e0 += 32) {
      const int m = min(32, hi - e0);
      uint4 r = lane < m ? a.csc[e0 + lane] : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t last = __shfl_sync(0xFFFFFFFFu, r.x, m - 1);
      if (lane >= m) r.x = last;
      __syncwarp();  // the previous chunk's reads of the stage are done
      const float cg = __uint_as_float(r.y), cu = __uint_as_float(r.z), ch = __uint_as_float(r.w);
      cgu[lane] = make_float4(cg, cg, cu, cu);
      chr[lane] = make_float4(ch, ch, __uint_as_float(r.x), 0.f);
      __syncwarp();
      if (xside) {
        for (int k = 0; k < m; k += U) {
          uint4 v[U];
#pragma unroll
          for (int q = 0; q < U; ++q) v[q] = ldg16(src + __float_as_uint(chr[k + q].z));
#pragma unroll
          for (int q = 0; q < U; ++q) {
            const float4 e = cgu[k + q];
            if (GATED)
              axpy8_two(p, f2(e.x, e.y), q2, f2(e.z, e.w), v[q]);
            else
              axpy8(p, f2(e.x, e.y), v[q]);
          }
        }
      } else {
        for (int k = 0; k < m; k += U) {
          uint4 v[U];
#pragma unroll
          for (int q = 0; q < U; ++q) v[q] = ldg16(src + __float_as_uint(chr[k + q].z));
#pragma unroll
          for (int q = 0; q < U; ++q) {
            const float2 hh = *reinterpret_cast<const float2*>(&chr[k + q]);
            axpy8(p, f2(hh.x, hh.y), v[q]);
          }
        }
      }
    }
    const size_t o = static_cast<size_t>(j) * a.d + c * 256 + lane * 8;
    if (xside) {
      stcs_f32x8(a.dWg + o, p);
      if (GATED) stcs_f32x8(a.dWu + o, q2);
    } else {
      stcs_f32x8(a.dWd + o, p);
    }
  }
}

// ====================================================================== launchers
#define TW_NCH_SWITCH(nch, CALL)           \
  switch (nch) {                           \
    case 1: CALL(1); break;                \
    case 2: CALL(2); break;                \
    case 3: CALL(3); break;                \
    case 4: CALL(4); break;                \
    case 5: CALL(5); break;                \
    case 6: CALL(6); break;                \
    case 7: CALL(7); break;                \
    case 8: CALL(8); break;                \
    default: return cudaErrorInvalidValue; \
  }

// largest per-warp entry list the forward supports
constexpr int kFwdListMax = 12288;

template <class K>
static cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

// warps per CTA for a kernel whose warps need `per_warp` bytes of shared memory:
// at most 8, and a CTA of at most 110 KB so that two fit on an SM
static int warps_for(size_t per_warp) {
  return static_cast<int>(std::max<size_t>(1, std::min<size_t>(8, (110u << 10) / per_warp)));
}

template <bool GATED, bool HYBRID>
static cudaError_t launch_fwd(const SparseFwdArgs& a, int32_t* status, cudaStream_t s) {
  const int nch = a.d / 256;
  const size_t per_warp = fwd_warp_smem(nch, a.L);
  const int wpb = warps_for(per_warp);
  const size_t smem = per_warp * wpb;
  const int grid = grid_for(a.T, wpb, 8);
#define TW_FWD(n)                                                                    \
  {                                                                                  \
    cudaError_t e = set_smem(sparse_fwd_kernel<n, GATED, HYBRID>, smem);             \
    if (e != cudaSuccess) return e;                                                  \
    sparse_fwd_kernel<n, GATED, HYBRID><<<grid, wpb * 32, smem, s>>>(a, status);     \
  }
  TW_NCH_SWITCH(nch, TW_FWD)
#undef TW_FWD
  trace_mark(s, "sparse_fwd");
  return cudaGetLastError();
}

cudaError_t launch_sparse_fwd(const SparseFwdArgs& a, int32_t* status, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (a.L < 1 || a.L > kFwdListMax) return cudaErrorInvalidValue;
  const bool gated = a.Wu != nullptr;
  const bool hybrid = a.backup_slot != nullptr;
  if (gated) return hybrid ? launch_fwd<true, true>(a, status, s) : launch_fwd<true, false>(a, status, s);
  return hybrid ? launch_fwd<false, true>(a, status, s) : launch_fwd<false, false>(a, status, s);
}

template <bool GATED>
static cudaError_t launch_bwd(const SparseBwdArgs& a, int32_t* status, cudaStream_t s) {
  cudaError_t e = memset_async(a.col_cnt, 0, sizeof(int32_t) * (a.I + 1), s);
  if (e != cudaSuccess) return e;
  const int nch = a.d / 256;
  const size_t rowb = static_cast<size_t>(nch) * 512;
  if (a.T > 0) {
    const int wpb = warps_for(kDhRing * rowb);
    const size_t smem = kDhRing * rowb * wpb;
    const int grid = grid_for(a.T, wpb, 8);
#define TW_DH(n)                                                         \
  {                                                                      \
    e = set_smem(sparse_dh_kernel<n, GATED>, smem);                      \
    if (e != cudaSuccess) return e;                                      \
    sparse_dh_kernel<n, GATED><<<grid, wpb * 32, smem, s>>>(a, status);  \
  }
    TW_NCH_SWITCH(nch, TW_DH)
#undef TW_DH
    trace_mark(s, "sparse_dh");
  }
  csc_scan_kernel<<<1, 1024, 0, s>>>(a.col_cnt, a.I, a.col_ptr, a.col_cur);
  trace_mark(s, "csc_scan");
  if (a.T > 0) {
    csc_fill_kernel<GATED><<<grid_for(a.T, 8, 8), 256, 0, s>>>(a);
    trace_mark(s, "csc_fill");
    const int wpb = warps_for(kDxRing * rowb);
    const size_t smem = kDxRing * rowb * wpb;
    const int grid = grid_for(a.T, wpb, 8);
#define TW_DX(n)                                                         \
  {                                                                      \
    e = set_smem(sparse_dx_kernel<n, GATED>, smem);                      \
    if (e != cudaSuccess) return e;                                      \
    sparse_dx_kernel<n, GATED><<<grid, wpb * 32, smem, s>>>(a, status);  \
  }
    TW_NCH_SWITCH(nch, TW_DX)
#undef TW_DX
    trace_mark(s, "sparse_dx");
  }
  const long items = static_cast<long>(nch) * a.I * 2;
  ell_weight_grad_kernel<GATED><<<grid_for(items, 8, 3), 256, 0, s>>>(a);
  trace_mark(s, "ell_weight_grad");
  return cudaGetLastError();
}

cudaError_t launch_sparse_bwd(const SparseBwdArgs& a, int32_t* status, cudaStream_t s) {
  if (a.Wu != nullptr) return launch_bwd<true>(a, status, s);
  return launch_bwd<false>(a, status, s);
}

}  // namespace tw

// Token-major CUDA-core kernels of the sparse FFN (gist.science explainer, 2.B:
// "Fused Up/Down Projection" for inference and the training forward, and the
// hidden-gradient / input-gradient half of "Backpropagation").
//
// One CTA per token (a persistent loop over tokens), one warp per 256-wide slice of
// d: lane l of warp c owns elements [256 c + 8 l, 256 c + 8 l + 8) of every d-vector.
// Weight-row slices (512 bytes per warp) are gathered straight into registers, eight
// entries at a time, so no row passes through shared memory. Each token runs two
// passes over its entries, in windows of kWin entries:
//
//   pass A (dot)   every warp forms its slice's partial dot products of eight rows
//                  with the token's vector slice; a shuffle reduce-scatter leaves
//                  entry e's warp sum on lanes 4e..4e+3; the CTA adds the slices'
//                  partials in shared memory;
//   pass B (axpy)  every warp accumulates its slice of sum_k c_k W[j_k] in fp32.
//
//  forward   list = the token's TwELL entries (j, a) in ascending neuron order,
//            pass A: u = x_t . Wu[j], h = a u (gated; non-gated h = a),
//            pass B: y_t = sum h Wd[j]; in training the list is also the Hybrid
//            ELL row (idx, bf16 a, fp16 u).
//  backward  list = the token's ELL row (j, a, u),
//            pass A: dh = dy_t . Wd[j]; dg = dh u + l1 (non-gated: dh + l1), du = dh a,
//            pass B: dx_t = sum dg Wg[j] + du Wu[j]; between the passes every entry's
//            record {token row, dg, du, h} goes to its neuron column of the
//            transposed Hybrid, at a slot claimed from that column's cursor.
#include <algorithm>

#include "tw_common.cuh"
#include "tw_internal.h"

namespace tw {

namespace {

constexpr int kGroup = 8;   // entries gathered together by a warp
constexpr int kWin = 256;   // entries per window (shared-memory partial sums)
// Resident CTAs per SM: 48 warps at d = 2048 (six CTAs of eight warps, 40 registers
// a thread). The passes stall on L2 latency between short bursts of arithmetic, so
// warps, not per-warp loads in flight, are what keeps the gathers streaming.
__host__ __device__ constexpr int ctas_per_sm(int nch) { return 48 / nch < 32 ? 48 / nch : 32; }

__host__ __device__ constexpr uint32_t rup(uint32_t v, uint32_t m) { return (v + m - 1) / m * m; }

// eight fp32 accumulators as four packed pairs
struct Acc8 {
  f32x2 v[4];
  TW_DEV void zero() { v[0] = v[1] = v[2] = v[3] = 0ull; }
  // this += c2 * w over 8 bf16 elements (c2 = {c, c})
  TW_DEV void axpy(f32x2 c2, const uint4& w) {
    fma2(v[0], c2, widen(w.x));
    fma2(v[1], c2, widen(w.y));
    fma2(v[2], c2, widen(w.z));
    fma2(v[3], c2, widen(w.w));
  }
  TW_DEV uint4 to_bf16() const {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = unpair(v[i]);
      o[i] = pack_bf16x2(p.x, p.y);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  }
};

// x . w over 8 bf16 pairs: Blackwell's mixed-precision FMA (bf16 x bf16 + fp32; the
// product is exact in fp32, one rounding per step), two chains
TW_DEV float dot8(const uint4& x, const uint4& w) {
  float s0 = 0.f, s1 = 0.f;
  asm("{\n\t"
      ".reg .b16 x0, x1, x2, x3, x4, x5, x6, x7, w0, w1, w2, w3, w4, w5, w6, w7;\n\t"
      "mov.b32 {x0, x1}, %2;\n\t"
      "mov.b32 {x2, x3}, %3;\n\t"
      "mov.b32 {x4, x5}, %4;\n\t"
      "mov.b32 {x6, x7}, %5;\n\t"
      "mov.b32 {w0, w1}, %6;\n\t"
      "mov.b32 {w2, w3}, %7;\n\t"
      "mov.b32 {w4, w5}, %8;\n\t"
      "mov.b32 {w6, w7}, %9;\n\t"
      "fma.rn.f32.bf16 %0, x0, w0, %0;\n\t"
      "fma.rn.f32.bf16 %1, x1, w1, %1;\n\t"
      "fma.rn.f32.bf16 %0, x2, w2, %0;\n\t"
      "fma.rn.f32.bf16 %1, x3, w3, %1;\n\t"
      "fma.rn.f32.bf16 %0, x4, w4, %0;\n\t"
      "fma.rn.f32.bf16 %1, x5, w5, %1;\n\t"
      "fma.rn.f32.bf16 %0, x6, w6, %0;\n\t"
      "fma.rn.f32.bf16 %1, x7, w7, %1;\n\t"
      "}"
      : "+f"(s0), "+f"(s1)
      : "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w), "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w));
  return s0 + s1;
}

// Warp reduce-scatter of eight per-lane values: on return every lane of the quad
// 4e..4e+3 holds the warp-wide sum of p[e].
TW_DEV float reduce8(float (&p)[8], int lane) {
  const bool b16 = lane & 16, b8 = lane & 8, b4 = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b16 ? p[i] : p[i + 4];
    const float keep = b16 ? p[i + 4] : p[i];
    p[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b8 ? p[i] : p[i + 2];
    const float keep = b8 ? p[i + 2] : p[i];
    p[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
  }
  const float send = b4 ? p[0] : p[1];
  float s = (b4 ? p[1] : p[0]) + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
  s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
  s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
  return s;
}


// Token scheduling: a CTA's first token is its index; after that it takes the next
// unclaimed token from a device counter (zero at launch), so CTAs that start late or
// run slower take fewer tokens. Without a counter the assignment is round-robin.
TW_DEV int next_token(int32_t* sched, int t) {
  return sched != nullptr ? static_cast<int>(gridDim.x) + atomicAdd(sched, 1) : t + static_cast<int>(gridDim.x);
}

// Lists are read from shared memory sixteen bytes at a time (one broadcast
// wavefront for the whole warp): eight neuron indices, or two coefficient pairs.
// jsel(jv, q) is index q of a 16-byte block of eight; hsel(hv, odd) is pair `odd` of
// a block of two.
TW_DEV uint4 lds16(const void* p) { return *reinterpret_cast<const uint4*>(p); }
TW_DEV uint32_t jsel(const uint4& jv, int q) {
  const uint32_t w = q < 2 ? jv.x : q < 4 ? jv.y : q < 6 ? jv.z : jv.w;
  return (q & 1) ? (w >> 16) : (w & 0xFFFFu);
}
TW_DEV f32x2 hsel(const uint4& hv, int odd) {
  return odd ? ((static_cast<uint64_t>(hv.w) << 32) | hv.z) : ((static_cast<uint64_t>(hv.y) << 32) | hv.x);
}

// Block-wide exclusive scan of one int per thread; *total gets the sum. One
// __syncthreads, plus a trailing one when `reuse` (scratch is rewritten before the
// caller's next barrier); scratch holds one int per warp.
TW_DEV int block_exclusive_scan(int v, int* scratch, int* total, bool reuse) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int incl = warp_inclusive_scan(v);
  if (lane == 31) scratch[wid] = incl;
  __syncthreads();
  int before = 0, all = 0;
  for (int w = 0; w < nw; ++w) {
    const int s = scratch[w];
    before += w < wid ? s : 0;
    all += s;
  }
  if (reuse) __syncthreads();
  *total = all;
  return before + incl - v;
}

// Pass A over the list window [w0, w0 + m): part[k - w0] = this warp's slice of
// vec . W[j_k] for every k of the window rounded up to kGroup (entries past the list
// end repeat its last neuron; their sums are never read).
// VEC reads the group's eight indices in one 16-byte load (faster in the forward,
// slower in the backward, by measurement).
template <bool VEC>
TW_DEV void pass_dot(const uint4* Wslice, uint32_t row16, const uint16_t* lj, int w0, int m, const uint4& vec,
                     float* part, int lane, int I, int32_t* status) {
  for (int k0 = 0; k0 < m; k0 += kGroup) {
    uint4 v[kGroup];
    if (VEC) {
      const uint4 jv = lds16(lj + w0 + k0);
#pragma unroll
      for (int q = 0; q < kGroup; ++q) {
        const uint32_t j = jsel(jv, q);
        v[q] = TW_CHECKED(j < static_cast<uint32_t>(I), status) ? ldg16(Wslice + j * row16) : make_uint4(0u, 0u, 0u, 0u);
      }
    } else {
#pragma unroll
      for (int q = 0; q < kGroup; ++q) {
        const uint32_t j = lj[w0 + k0 + q];
        v[q] = TW_CHECKED(j < static_cast<uint32_t>(I), status) ? ldg16(Wslice + j * row16) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float p[kGroup];
#pragma unroll
    for (int q = 0; q < kGroup; ++q) p[q] = dot8(vec, v[q]);
    const float s = reduce8(p, lane);
    if ((lane & 3) == 0) part[k0 + (lane >> 2)] = s;
  }
}

// shared memory of one token CTA: two buffers of (neuron list | coefficient pairs),
// partial sums, scan scratch. Lists hold cap entries plus a group of padding.
__host__ __device__ inline uint32_t token_smem_bytes(int nch, int cap, int ncoef) {
  const uint32_t lp = rup(static_cast<uint32_t>(cap) + kGroup, kGroup);
  return 2u * (rup(2u * lp, 16u) + ncoef * 8u * lp) + 4u * nch * kWin + 4u * 33u;
}

}  // namespace

// ====================================================================== forward
// Rows served by the dense path (TwELL overflow, Hybrid backup) are skipped. In
// TwELL mode the entry list is built by the CTA: thread k takes TwELL tile k, an
// exclusive scan of the tiles' counts places their slots, so the list is in ascending
// neuron order. In Hybrid mode it is the row's ELL (idx, a), which a warp-per-row
// conversion wrote before this kernel: building it here cost the kernel 27 us at the
// bench workload (a block scan and the TwELL reads per token), the conversion 15.
// Lists are double-buffered over tokens, so a token needs no closing barrier: a
// warp still in the down pass of token t reads the other buffer than token t + 1
// writes, and token t + 2 writes it only after barriers every warp passes.
template <int NCH, bool GATED, bool HYBRID>
__global__ void __launch_bounds__(NCH * 32, ctas_per_sm(NCH)) token_fwd_kernel(const SparseFwdArgs a) {
  pdl_enter();
  if (a.route != nullptr && *a.route == 1) return;  // the call took the dense route
  constexpr uint32_t row16 = NCH * 32;  // uint4 per d-row
  extern __shared__ __align__(16) uint8_t tsm[];
  const int lane = threadIdx.x & 31, c = threadIdx.x >> 5;
  const uint32_t lp = rup(static_cast<uint32_t>(a.L) + kGroup, kGroup);
  const uint32_t list_bytes = rup(2u * lp, 16u) + 8u * lp;
  float* part = reinterpret_cast<float*>(tsm + 2 * list_bytes);
  int* scratch = reinterpret_cast<int*>(part + NCH * kWin);
  const uint4* Wu4 = reinterpret_cast<const uint4*>(a.Wu) + c * 32 + lane;
  const uint4* Wd4 = reinterpret_cast<const uint4*>(a.Wd) + c * 32 + lane;
  const bool vec_slots = a.C % 16 == 0;  // a tile's slots load as 16-byte vectors
  int buf = 0;
  __shared__ int next_tok[2];  // the CTA's next token, double-buffered like the lists
  int nb = 0;

  for (int t = blockIdx.x; t < a.T; nb ^= 1) {
    // the next token is fetched now and read after this token's first barrier
    if (threadIdx.x == 0) next_tok[nb] = next_token(a.sched, t);
    const bool skip = HYBRID ? (a.backup_slot[t] != -1) : (a.ovf[t] != 0);
    if (skip) {
      __syncthreads();
      t = next_tok[nb];
      continue;
    }
    uint16_t* lj = reinterpret_cast<uint16_t*>(tsm + buf * list_bytes);
    f32x2* lh = reinterpret_cast<f32x2*>(tsm + buf * list_bytes + rup(2u * lp, 16u));
    buf ^= 1;
    const size_t rb = static_cast<size_t>(t) * a.R;
    // ------------------------------------------------------------ entry list
    int n = 0, last_pos = -1, last_j = 0;
    if (HYBRID) {
      // the row's ELL entries (written by the ELL conversion before this kernel), padded
      // to a whole group with its last neuron and zero coefficients
      n = a.ell_nnz[t];
      if (!TW_CHECKED(n >= 0 && n <= a.R && n <= a.L, a.status)) n = 0;
      for (int k = threadIdx.x; k < rup(n, kGroup); k += blockDim.x) {
        const int e = min(k, n - 1);
        const uint16_t j = a.ell_idx[rb + e];
        lj[k] = TW_CHECKED(j < a.I, a.status) ? j : 0;
        const float av = k < n ? bf16_to_f32(a.ell_a[rb + e]) : 0.f;
        lh[k] = pair(av, av);
      }
    }
    for (int kb = 0; !HYBRID && kb < a.nT; kb += blockDim.x) {
      const int k = kb + threadIdx.x;
      const int cnt = k < a.nT ? min(static_cast<int>(a.cnt[static_cast<size_t>(t) * a.nT + k]), a.C) : 0;
      const size_t sb = (static_cast<size_t>(t) * a.nT + k) * a.C;
      // the tile's first 16 slots, loaded before the scan so the load overlaps it
      uint4 iv = make_uint4(0u, 0u, 0u, 0u), v0 = iv, v1 = iv;
      if (vec_slots && cnt > 0) {
        iv = *reinterpret_cast<const uint4*>(a.idx + sb);
        v0 = *reinterpret_cast<const uint4*>(a.val + sb);
        v1 = *reinterpret_cast<const uint4*>(a.val + sb + 8);
      }
      int tot;
      const int off = n + block_exclusive_scan(cnt, scratch, &tot, kb + static_cast<int>(blockDim.x) < a.nT);
      auto put = [&](int i, int jj, uint16_t ab) {
        const int j = k * a.W + jj;
        if (!TW_CHECKED(off + i < a.L && jj < a.W, a.status)) return;
        const float av = bf16_to_f32(ab);
        lj[off + i] = static_cast<uint16_t>(j);
        lh[off + i] = pair(av, av);
        last_pos = off + i;
        last_j = j;
      };
      if (vec_slots) {
        const uint32_t iw[4] = {iv.x, iv.y, iv.z, iv.w};
        const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < cnt)
            put(i, static_cast<int>((iw[i >> 2] >> (8 * (i & 3))) & 0xFFu), static_cast<uint16_t>(vw[i >> 1] >> (16 * (i & 1))));
      }
      for (int i = vec_slots ? 16 : 0; i < cnt; ++i) put(i, a.idx[sb + i], a.val[sb + i]);
      n += tot;
    }
    if (!HYBRID && n > 0 && last_pos == n - 1) {  // the list's last writer pads it to a whole group (zero coefficients)
#pragma unroll
      for (int i = 0; i < kGroup; ++i) {
        lj[n + i] = static_cast<uint16_t>(last_j);
        lh[n + i] = 0ull;
      }
    }
    const uint4 xs = GATED ? ldg16(reinterpret_cast<const uint4*>(a.x) + static_cast<size_t>(t) * row16 + c * 32 + lane)
                           : make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    Acc8 y;
    y.zero();
    for (int w0 = 0; w0 < n; w0 += kWin) {
      const int m = min(kWin, n - w0);
      if (GATED) {
        // -------------------------------------------------------- up: h = a (x_t . Wu[j])
        pass_dot<true>(Wu4, row16, lj, w0, m, xs, part + c * kWin, lane, a.I, a.status);
        __syncthreads();
        for (int k = threadIdx.x; k < m; k += blockDim.x) {
          float u = 0.f;
#pragma unroll
          for (int w = 0; w < NCH; ++w) u += part[w * kWin + k];
          const float h = unpair(lh[w0 + k]).x * u;
          lh[w0 + k] = pair(h, h);
          if (HYBRID && TW_CHECKED(w0 + k < a.R, a.status)) a.ell_u[rb + w0 + k] = f32_to_f16(u);
        }
        __syncthreads();
      }
      // ---------------------------------------------------------- down: y_t += sum h Wd[j]
      for (int k0 = 0; k0 < m; k0 += kGroup) {
        const uint4 jv = lds16(lj + w0 + k0);
        uint4 v[kGroup];
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
          const uint32_t j = jsel(jv, q);
          v[q] = TW_CHECKED(j < static_cast<uint32_t>(a.I), a.status) ? ldg16(Wd4 + j * row16) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < kGroup; q += 2) {
          const uint4 hv = lds16(lh + w0 + k0 + q);
          y.axpy(hsel(hv, 0), v[q]);
          y.axpy(hsel(hv, 1), v[q + 1]);
        }
      }
    }
    reinterpret_cast<uint4*>(a.y)[static_cast<size_t>(t) * row16 + c * 32 + lane] = y.to_bf16();
    t = next_tok[nb];
  }
}

// ====================================================================== forward, warp-specialised
// The same forward with the entry lists built off the critical path: warp NCH of
// the CTA is a producer that enumerates the CTA's tokens' TwELL rows (lane k takes
// tile k; a warp scan of the tile counts places the slots, so the list is in
// ascending neuron order; in training the same writes produce the Hybrid ELL row)
// into a ring of kListRing list buffers, while warps 0 .. NCH - 1 run the passes of
// an earlier token. Buffers are handed over with mbarriers: "full" (one producer
// arrival, after the list and its header {token, n} are written) and "empty" (one
// arrival per consumer warp, after its down pass). Every wait is bounded; the
// consumers synchronise among themselves with a named barrier. A header with token
// -1 ends the stream.
constexpr int kListRing = 2;

__host__ __device__ inline uint32_t fwd_ws_list_bytes(int L) {
  const uint32_t lp = rup(static_cast<uint32_t>(L) + kGroup, kGroup);
  return rup(16u + 2u * lp, 16u) + 8u * lp;
}
__host__ __device__ inline uint32_t fwd_ws_smem_bytes(int nch, int L) {
  return kListRing * fwd_ws_list_bytes(L) + 4u * nch * kWin + 8u * 2u * kListRing + 16u;
}
__host__ __device__ constexpr int ws_ctas_per_sm(int nch) { return 45 / (nch + 1) < 32 ? 45 / (nch + 1) : 32; }

TW_DEV void consumers_sync(int nthreads) { asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory"); }
// Barrier 1 with an OR reduction: true on every consumer thread when v is true on any.
TW_DEV bool consumers_any(bool v, int nthreads) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(nthreads)
      : "memory");
  return r != 0;
}

template <int NCH, bool GATED, bool HYBRID>
__global__ void __launch_bounds__((NCH + 1) * 32, ws_ctas_per_sm(NCH))
    token_fwd_ws_kernel(const SparseFwdArgs a) {
  int32_t* status = a.status;
  constexpr uint32_t row16 = NCH * 32;
  constexpr int kConsumers = NCH * 32;
  extern __shared__ __align__(16) uint8_t tsm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lp = rup(static_cast<uint32_t>(a.L) + kGroup, kGroup);
  const uint32_t lbytes = fwd_ws_list_bytes(a.L);
  float* part = reinterpret_cast<float*>(tsm + kListRing * lbytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(part + NCH * kWin);
  uint64_t* empty = full + kListRing;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kListRing);
  auto header = [&](int b) { return reinterpret_cast<int*>(tsm + b * lbytes); };
  auto list_j = [&](int b) { return reinterpret_cast<uint16_t*>(tsm + b * lbytes + 16); };
  auto list_h = [&](int b) { return reinterpret_cast<f32x2*>(tsm + b * lbytes + rup(16u + 2u * lp, 16u)); };
  if (threadIdx.x == 0) {
    for (int b = 0; b < kListRing; ++b) {
      mbar_init(full + b, 1);
      mbar_init(empty + b, NCH);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_enter();
  if (a.route != nullptr && *a.route == 1) return;  // the call took the dense route (uniform over the CTA)

  if (warp == NCH) {
    // ------------------------------------------------------------ producer warp
    const bool vec_slots = a.C % 16 == 0;
    int k = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok;) {  // the first t past the range sends the end header
      const bool end = t >= a.T;
      const int t_next = end ? t : __shfl_sync(0xFFFFFFFFu, lane == 0 ? next_token(a.sched, t) : 0, 0);
      if (!end && (HYBRID ? (a.backup_slot[t] != -1) : (a.ovf[t] != 0))) {
        t = t_next;
        continue;
      }
      const int b = k % kListRing;
      const uint32_t use = static_cast<uint32_t>(k / kListRing);
      ++k;
      if (!mbar_wait(empty + b, (use & 1u) ^ 1u, abort_flag, status)) {
        ok = false;
        break;
      }
      uint16_t* lj = list_j(b);
      f32x2* lh = list_h(b);
      int n = 0;
      if (!end) {
        const size_t rb = static_cast<size_t>(t) * a.R;
        for (int kb = 0; kb < a.nT; kb += 32) {
          const int kt = kb + lane;
          const int cnt = kt < a.nT ? min(static_cast<int>(a.cnt[static_cast<size_t>(t) * a.nT + kt]), a.C) : 0;
          const size_t sb = (static_cast<size_t>(t) * a.nT + kt) * a.C;
          const int incl = warp_inclusive_scan(cnt);
          const int off = n + incl - cnt;
          auto put = [&](int i, int jj, uint16_t ab) {
            const int j = kt * a.W + jj;
            if (!TW_CHECKED(off + i < a.L && jj < a.W, status)) return;
            const float av = bf16_to_f32(ab);
            lj[off + i] = static_cast<uint16_t>(j);
            lh[off + i] = pair(av, av);
            if (HYBRID && TW_CHECKED(off + i < a.R, status)) {
              a.ell_idx[rb + off + i] = static_cast<uint16_t>(j);
              a.ell_a[rb + off + i] = ab;
            }
          };
          if (vec_slots && cnt > 0) {
            const uint4 iv = *reinterpret_cast<const uint4*>(a.idx + sb);
            const uint4 v0 = *reinterpret_cast<const uint4*>(a.val + sb);
            const uint4 v1 = *reinterpret_cast<const uint4*>(a.val + sb + 8);
            const uint32_t iw[4] = {iv.x, iv.y, iv.z, iv.w};
            const uint32_t vw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (i < cnt)
                put(i, static_cast<int>((iw[i >> 2] >> (8 * (i & 3))) & 0xFFu),
                    static_cast<uint16_t>(vw[i >> 1] >> (16 * (i & 1))));
          }
          for (int i = vec_slots ? 16 : 0; i < cnt; ++i) put(i, a.idx[sb + i], a.val[sb + i]);
          n += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        __syncwarp();
        if (n > 0 && lane < kGroup) {  // pad to a whole group: the last neuron, zero coefficient
          lj[n + lane] = lj[n - 1];
          lh[n + lane] = 0ull;
        }
      }
      if (lane == 0) {
        header(b)[0] = end ? -1 : t;
        header(b)[1] = n;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(full + b);  // release: the list and header are visible to the waiters
      if (end) break;
      t = t_next;
    }
    return;
  }

  // -------------------------------------------------------------- consumer warps
  const int c = warp;
  const uint4* Wu4 = reinterpret_cast<const uint4*>(a.Wu) + c * 32 + lane;
  const uint4* Wd4 = reinterpret_cast<const uint4*>(a.Wd) + c * 32 + lane;
  for (int k = 0;; ++k) {
    const int b = k % kListRing;
    const uint32_t use = static_cast<uint32_t>(k / kListRing);
    const bool failed = !mbar_wait(full + b, use & 1u, abort_flag, status);
    if (consumers_any(failed, kConsumers)) break;  // one decision for every consumer warp
    const int t = header(b)[0], n = header(b)[1];
    if (t < 0) break;
    const uint16_t* lj = list_j(b);
    f32x2* lh = list_h(b);
    const size_t rb = static_cast<size_t>(t) * a.R;
    const uint4 xs = GATED ? ldg16(reinterpret_cast<const uint4*>(a.x) + static_cast<size_t>(t) * row16 + c * 32 + lane)
                           : make_uint4(0u, 0u, 0u, 0u);
    Acc8 y;
    y.zero();
    for (int w0 = 0; w0 < n; w0 += kWin) {
      const int m = min(kWin, n - w0);
      if (GATED) {
        pass_dot<true>(Wu4, row16, lj, w0, m, xs, part + c * kWin, lane, a.I, status);
        consumers_sync(kConsumers);
        for (int kk = threadIdx.x; kk < m; kk += kConsumers) {
          float u = 0.f;
#pragma unroll
          for (int w = 0; w < NCH; ++w) u += part[w * kWin + kk];
          const float h = unpair(lh[w0 + kk]).x * u;
          lh[w0 + kk] = pair(h, h);
          if (HYBRID && TW_CHECKED(w0 + kk < a.R, status)) a.ell_u[rb + w0 + kk] = f32_to_f16(u);
        }
        consumers_sync(kConsumers);
      }
      for (int k0 = 0; k0 < m; k0 += kGroup) {
        uint4 v[kGroup];
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
          const uint32_t j = lj[w0 + k0 + q];
          v[q] = TW_CHECKED(j < static_cast<uint32_t>(a.I), status) ? ldg16(Wd4 + j * row16) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < kGroup; ++q) y.axpy(lh[w0 + k0 + q], v[q]);
      }
    }
    reinterpret_cast<uint4*>(a.y)[static_cast<size_t>(t) * row16 + c * 32 + lane] = y.to_bf16();
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + b);
  }
}

// ====================================================================== backward
// Tokens without ELL entries get dx = 0; rows in the dense backup (slot >= 0) are
// left to the dense path, which writes their dx. The window lists are
// double-buffered like the forward's.
template <int NCH, bool GATED>
__global__ void __launch_bounds__(NCH * 32, ctas_per_sm(NCH)) token_bwd_kernel(const SparseBwdArgs a) {
  pdl_enter();
  if (a.route != nullptr && *a.route == 1) return;  // the call took the dense route
  constexpr uint32_t row16 = NCH * 32;
  constexpr int kPerThread = (kWin + NCH * 32 - 1) / (NCH * 32);  // window entries per thread, at most
  static_assert(rup(kWin, kGroup) == kWin, "a window is whole groups");
  constexpr uint32_t lp = rup(kWin + kGroup, kGroup);
  constexpr uint32_t list_bytes = rup(2u * lp, 16u) + 2u * 8u * lp;
  extern __shared__ __align__(16) uint8_t tsm[];
  const int lane = threadIdx.x & 31, c = threadIdx.x >> 5;
  float* part = reinterpret_cast<float*>(tsm + 2 * list_bytes);
  const uint4* Wg4 = reinterpret_cast<const uint4*>(a.Wg) + c * 32 + lane;
  const uint4* Wu4 = reinterpret_cast<const uint4*>(a.Wu) + c * 32 + lane;
  const uint4* Wd4 = reinterpret_cast<const uint4*>(a.Wd) + c * 32 + lane;
  int buf = 0;
  __shared__ int next_tok[2];  // the CTA's next token (read after this token's first barrier)
  int nb = 0;

  for (int t = blockIdx.x; t < a.T; nb ^= 1) {
    if (threadIdx.x == 0) next_tok[nb] = next_token(a.sched, t);
    if (a.backup_slot != nullptr && a.backup_slot[t] >= 0) {  // the dense path writes this row's dx
      __syncthreads();
      t = next_tok[nb];
      continue;
    }
    int n = a.ell_nnz[t];
    if (!TW_CHECKED(n >= 0 && n <= a.R, a.status)) n = 0;
    const size_t rb = static_cast<size_t>(t) * a.R;
    const uint4 dys = n > 0 ? ldg16(reinterpret_cast<const uint4*>(a.dy) + static_cast<size_t>(t) * row16 + c * 32 + lane)
                            : make_uint4(0u, 0u, 0u, 0u);
    Acc8 dx;
    dx.zero();
    for (int w0 = 0; w0 < n; w0 += kWin) {
      const int m = min(kWin, n - w0);
      uint16_t* lj = reinterpret_cast<uint16_t*>(tsm + buf * list_bytes);
      f32x2* lg = reinterpret_cast<f32x2*>(tsm + buf * list_bytes + rup(2u * lp, 16u));  // a, then dg
      f32x2* lu = lg + lp;                                                                // u, then du
      buf ^= 1;
      // each thread takes entries threadIdx.x + i * blockDim.x. It claims the slot of
      // its first one in the transposed Hybrid here and fills it after pass A, which
      // hides the claim's round trip (further entries, when a window has more than
      // blockDim of them, claim theirs when they are filled)
      int slot0 = 0;
#pragma unroll
      for (int i = 0; i < kPerThread; ++i) {
        const int k = threadIdx.x + i * static_cast<int>(blockDim.x);
        if (k >= rup(m, kGroup)) break;
        const int e = min(k, m - 1);
        int j = a.ell_idx[rb + w0 + e];
        if (!TW_CHECKED(j < a.I, a.status)) j = 0;
        lj[k] = static_cast<uint16_t>(j);
        if (k < m) {
          if (i == 0) slot0 = atomicAdd(a.col_cur + j, 1);
          lg[k] = pair(bf16_to_f32(a.ell_a[rb + w0 + k]), 0.f);
          lu[k] = pair(GATED ? f16_to_f32(a.ell_u[rb + w0 + k]) : 1.f, 0.f);
        } else {
          lg[k] = 0ull;
          lu[k] = 0ull;
        }
      }
      __syncthreads();
      // ---------------------------------------------------------- dh = dy_t . Wd[j]
      pass_dot<false>(Wd4, row16, lj, 0, m, dys, part + c * kWin, lane, a.I, a.status);
      __syncthreads();
#pragma unroll
      for (int i = 0; i < kPerThread; ++i) {
        const int k = threadIdx.x + i * static_cast<int>(blockDim.x);
        if (k >= m) break;
        float dh = 0.f;
#pragma unroll
        for (int w = 0; w < NCH; ++w) dh += part[w * kWin + k];
        const float av = unpair(lg[k]).x, uv = unpair(lu[k]).x;
        const float dg = (GATED ? dh * uv : dh) + a.l1;
        const float du = dh * av;
        // the entry's record {token row offset in 16-byte units, dg, du, h = a u (or a)}
        const int sl = i == 0 ? slot0 : atomicAdd(a.col_cur + lj[k], 1);
        if (TW_CHECKED(sl >= 0 && sl < a.csc_cap, a.status))
          a.csc[sl] = make_uint4(static_cast<uint32_t>(t) * row16, __float_as_uint(dg),
                                    GATED ? __float_as_uint(du) : 0u, __float_as_uint(GATED ? av * uv : av));
        lg[k] = pair(dg, dg);
        lu[k] = pair(du, du);
      }
      __syncthreads();
      // ---------------------------------------------------------- dx_t += dg Wg[j] + du Wu[j]
      for (int k0 = 0; k0 < m; k0 += kGroup / 2) {
        uint4 v[kGroup];
#pragma unroll
        for (int q = 0; q < kGroup / 2; ++q) {
          const uint32_t r = static_cast<uint32_t>(lj[k0 + q]) * row16;
          v[2 * q] = ldg16(Wg4 + r);
          if (GATED) v[2 * q + 1] = ldg16(Wu4 + r);
        }
#pragma unroll
        for (int q = 0; q < kGroup / 2; ++q) {
          dx.axpy(lg[k0 + q], v[2 * q]);
          if (GATED) dx.axpy(lu[k0 + q], v[2 * q + 1]);
        }
      }
    }
    if (n == 0) __syncthreads();  // the windows' barriers publish next_tok otherwise
    reinterpret_cast<uint4*>(a.dx)[static_cast<size_t>(t) * row16 + c * 32 + lane] = dx.to_bf16();
    t = next_tok[nb];
  }
}

// ====================================================================== launchers
namespace {
template <class K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}
int token_grid(int T, int nch) {
  const int per_sm = ctas_per_sm(nch);
  return std::max(1, std::min(T, device_sm_count() * per_sm));
}
}  // namespace

#define TW_NCH_CASES(CALL) \
  case 1: CALL(1); break;  \
  case 2: CALL(2); break;  \
  case 3: CALL(3); break;  \
  case 4: CALL(4); break;  \
  case 5: CALL(5); break;  \
  case 6: CALL(6); break;  \
  case 7: CALL(7); break;  \
  case 8: CALL(8); break;  \
  default: return cudaErrorInvalidValue;

// Kernel choice, by measurement on GB300 at d 2048: the gated forward (training and
// inference) runs the single-role kernel; with its list reads vectorised it matches
// the warp-specialised kernel in training and is 4 % faster in inference. The
// warp-specialised kernel, which runs out of registers for vectorised reads, is
// 2.5 % faster for the non-gated forward.
template <bool GATED, bool HYBRID>
static cudaError_t token_fwd(const SparseFwdArgs& a, cudaStream_t s) {
  const int nch = a.d / 256;
  if (a.sched != nullptr && !a.sched_zeroed) {
    const cudaError_t z = launch_zero(a.sched, sizeof(int32_t), nullptr, 0, s);
    if (z != cudaSuccess) return z;
  }
  constexpr bool kSpecialised = !GATED;
  const size_t smem = kSpecialised ? fwd_ws_smem_bytes(nch, a.L) : token_smem_bytes(nch, a.L, 1);
  cudaError_t e = cudaSuccess;
#define TW_TF(n)                                                                                        \
  if constexpr (kSpecialised) {                                                                         \
    const int grid = std::max(1, std::min(a.T, device_sm_count() * ws_ctas_per_sm(n)));                \
    e = set_smem(token_fwd_ws_kernel<n, GATED, HYBRID>, smem);                                          \
    if (e != cudaSuccess) return e;                                                                     \
    e = launch(token_fwd_ws_kernel<n, GATED, HYBRID>, dim3(grid), dim3((n + 1) * 32), smem, s, a);     \
  } else {                                                                                              \
    e = set_smem(token_fwd_kernel<n, GATED, HYBRID>, smem);                                             \
    if (e != cudaSuccess) return e;                                                                     \
    e = launch(token_fwd_kernel<n, GATED, HYBRID>, dim3(token_grid(a.T, n)), dim3(n * 32), smem, s, a); \
  }
  switch (nch) { TW_NCH_CASES(TW_TF) }
#undef TW_TF
  trace_mark(s, "sparse_fwd");
  return e;
}

cudaError_t launch_token_fwd(const SparseFwdArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (a.L < 1 || a.L > kMaxList) return cudaErrorInvalidValue;
  const bool gated = a.Wu != nullptr;
  const bool hybrid = a.backup_slot != nullptr;
  if (gated) return hybrid ? token_fwd<true, true>(a, s) : token_fwd<true, false>(a, s);
  return hybrid ? token_fwd<false, true>(a, s) : token_fwd<false, false>(a, s);
}

template <bool GATED>
static cudaError_t token_bwd(const SparseBwdArgs& a, cudaStream_t s) {
  const int nch = a.d / 256;
  const size_t smem = token_smem_bytes(nch, kWin, 2);
  const int grid = token_grid(a.T, nch);
  cudaError_t e = cudaSuccess;
#define TW_TB(n)                                                                    \
  {                                                                                 \
    e = set_smem(token_bwd_kernel<n, GATED>, smem);                                 \
    if (e != cudaSuccess) return e;                                                 \
    e = launch(token_bwd_kernel<n, GATED>, dim3(grid), dim3(n * 32), smem, s, a); \
  }
  switch (nch) { TW_NCH_CASES(TW_TB) }
#undef TW_TB
  trace_mark(s, "sparse_bwd_token");
  return e;
}

cudaError_t launch_token_bwd(const SparseBwdArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  return a.Wu != nullptr ? token_bwd<true>(a, s) : token_bwd<false>(a, s);
}

}  // namespace tw

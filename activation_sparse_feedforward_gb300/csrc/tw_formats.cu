// Format conversions on a given matrix (gist.science explainer, 2.A "New Sparse
// Data Format: TwELL" and "Hybrid Format for Training"; wispaper blog, "1. TwELL:
// Tile-wise ELLPACK" and "2. The Hybrid Training Algorithm"):
//  * TwELL unpack: the stored slots scattered back into a dense bf16 matrix;
//  * Hybrid pack from a dense bf16 A (and U, gated form): per-row tile counts and
//    the TwELL overflow flag, the routing (the row compaction of tw_kernels.cu), then
//    every row written either as its ELL row or as its fp32 backup rows;
//  * Hybrid unpack: dense fp32 A (and U) from the ELL rows and the backup rows.
// The training forward builds the same Hybrid from the fused gate kernel's TwELL;
// these calls define the formats on a chosen matrix, so round trips and hand-placed
// edge cases can be checked against the pages' definitions.
//
// Every kernel gives one warp a row; lane l holds the eight columns
// [256 c + 8 l, 256 c + 8 l + 8) of the row's 256-column chunk c (I % 64 == 0, so a
// chunk's tail is whole 8-column pieces, and rows are 16-byte aligned).
#include <algorithm>

#include "tw_common.cuh"
#include "tw_internal.h"

namespace tw {

namespace {

// nonzero mask of eight bf16 values (bit i = element i; magnitude bits nonzero)
TW_DEV uint32_t nz_mask8(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m |= ((w[i] & 0x7FFFu) != 0u ? 1u : 0u) << (2 * i);
    m |= ((w[i] & 0x7FFF0000u) != 0u ? 1u : 0u) << (2 * i + 1);
  }
  return m;
}
TW_DEV uint16_t elem8(const uint4& v, int i) {
  const uint32_t w = i < 2 ? v.x : i < 4 ? v.y : i < 6 ? v.z : v.w;
  return static_cast<uint16_t>((i & 1) ? (w >> 16) : (w & 0xFFFFu));
}

int rows_grid(int T) {
  const long blocks = (static_cast<long>(T) + 7) / 8;  // eight warps a block
  return static_cast<int>(std::max<long>(1, std::min<long>(blocks, static_cast<long>(device_sm_count()) * 16)));
}

}  // namespace

// ------------------------------------------------------------------ TwELL unpack
// Row t of A = zeros, then slot s < min(cnt, C) of each tile k written at column
// k W + idx. On rows without overflow this is the packed matrix itself.
__global__ void __launch_bounds__(256) twell_unpack_kernel(const tw_twell tw, uint16_t* __restrict__ A) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int nT = tw.I / tw.W;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < tw.T; t += gridDim.x * 8) {
    uint4* row = reinterpret_cast<uint4*>(A + static_cast<size_t>(t) * tw.I);
    for (int c = lane; c < tw.I / 8; c += 32) row[c] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();  // the zeros land before any lane's slots
    for (int k = lane; k < nT; k += 32) {
      const size_t tk = static_cast<size_t>(t) * nT + k;
      const int n = min(static_cast<int>(tw.cnt[tk]), tw.C);
      for (int s = 0; s < n; ++s) {
        const int col = tw.idx[tk * tw.C + s];
        if (col < tw.W) A[static_cast<size_t>(t) * tw.I + k * tw.W + col] = tw.val[tk * tw.C + s];
      }
    }
  }
}

cudaError_t launch_twell_unpack(const tw_twell& tw, uint16_t* A, cudaStream_t s) {
  if (tw.T == 0) return cudaSuccess;
  cudaError_t e = launch(twell_unpack_kernel, dim3(rows_grid(tw.T)), dim3(256), 0, s, tw, A);
  trace_mark(s, "twell_unpack");
  return e;
}

// ------------------------------------------------------------------ Hybrid pack
// Per row: row_nnz (all nonzeros) and ovf = some W-column tile holds more than C.
// A tile is W / 8 consecutive lanes of a chunk (W in {64, 128}), so its count is a
// reduction over that lane group.
__global__ void __launch_bounds__(256) row_tile_counts_kernel(const uint16_t* __restrict__ A, int T, int I, int W,
                                                             int C, int32_t* __restrict__ row_nnz,
                                                             uint8_t* __restrict__ ovf) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int group = W / 8;  // lanes a tile spans
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < T; t += gridDim.x * 8) {
    const uint4* row = reinterpret_cast<const uint4*>(A + static_cast<size_t>(t) * I);
    int total = 0;
    bool over = false;
    for (int c0 = 0; c0 < I; c0 += 256) {
      const int col = c0 + 8 * lane;
      const int n = col < I ? __popc(nz_mask8(row[col / 8])) : 0;
      int tile = n;
      for (int o = 1; o < group; o <<= 1) tile += __shfl_xor_sync(0xFFFFFFFFu, tile, o);
      over |= col < I && tile > C;
      total += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xFFFFFFFFu, total, o);
    over = __any_sync(0xFFFFFFFFu, over);
    if (lane == 0) {
      row_nnz[t] = total;
      ovf[t] = over ? 1 : 0;
    }
  }
}

// Rows in the backup (slot in [0, cap)) get their full A and U rows as fp32; ELL rows
// get their nonzeros in ascending column order (global index, A and U values). Rows
// past the backup capacity (slot -2) are not written.
__global__ void __launch_bounds__(256) hybrid_fill_kernel(const uint16_t* __restrict__ A,
                                                         const uint16_t* __restrict__ U, const tw_hybrid h) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int I = h.I;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < h.T; t += gridDim.x * 8) {
    const uint4* arow = reinterpret_cast<const uint4*>(A + static_cast<size_t>(t) * I);
    const uint4* urow = U != nullptr ? reinterpret_cast<const uint4*>(U + static_cast<size_t>(t) * I) : nullptr;
    const int slot = h.backup_slot[t];
    if (slot >= 0) {
      float4* da = reinterpret_cast<float4*>(h.backup_a + static_cast<size_t>(slot) * I);
      float4* du = U != nullptr ? reinterpret_cast<float4*>(h.backup_u + static_cast<size_t>(slot) * I) : nullptr;
      for (int c = lane; c < I / 8; c += 32) {
        const uint4 v = arow[c];
        da[2 * c] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
        da[2 * c + 1] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
        if (du != nullptr) {
          const uint4 w = urow[c];
          du[2 * c] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
          du[2 * c + 1] = make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
        }
      }
      continue;
    }
    if (slot != -1) continue;  // past the backup capacity: the row is not stored
    const size_t rb = static_cast<size_t>(t) * h.R;
    int base = 0;  // entries placed by the chunks before
    for (int c0 = 0; c0 < I; c0 += 256) {
      const int col = c0 + 8 * lane;
      const uint4 v = col < I ? arow[col / 8] : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t m = nz_mask8(v);
      const int n = __popc(m);
      const int incl = warp_inclusive_scan(n);
      int off = base + incl - n;
      if (m != 0u) {
        const uint4 w = urow != nullptr ? urow[col / 8] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if ((m >> i) & 1u) {
            if (off < h.R) {  // an ELL row has at most R nonzeros; the bound keeps stores inside the row
              h.ell_idx[rb + off] = static_cast<uint16_t>(col + i);
              h.ell_a[rb + off] = elem8(v, i);
              if (urow != nullptr) h.ell_u[rb + off] = f32_to_f16(bf16_to_f32(elem8(w, i)));
            }
            ++off;
          }
        }
      }
      base += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
}

cudaError_t launch_hybrid_pack(const uint16_t* A, const uint16_t* U, int T, int I, int W, int C, const tw_hybrid& h,
                               uint8_t* ovf_ws, int32_t* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  cudaError_t e = launch(row_tile_counts_kernel, dim3(rows_grid(T)), dim3(256), 0, s, A, T, I, W, C, h.row_nnz,
                         ovf_ws);
  trace_mark(s, "row_tile_counts");
  if (e != cudaSuccess) return e;
  // backup <=> TwELL overflow or row_nnz > R; backup slots by ascending row; ell_nnz
  e = launch_compact_rows(ovf_ws, h.row_nnz, h.R, T, h.backup_tok, h.backup_cap, h.n_backup, h.backup_slot,
                          h.ell_nnz, h.backup_cap, status, s);
  if (e != cudaSuccess) return e;
  e = launch(hybrid_fill_kernel, dim3(rows_grid(T)), dim3(256), 0, s, A, U, h);
  trace_mark(s, "hybrid_fill");
  return e;
}

// ------------------------------------------------------------------ Hybrid unpack
// Row t of A (and U) in fp32: the backup row when the row has a slot below the
// capacity; else zeros with the ELL entries written at their columns (zeros for a
// row that did not fit in the backup).
__global__ void __launch_bounds__(256) hybrid_unpack_kernel(const tw_hybrid h, float* __restrict__ A,
                                                           float* __restrict__ U) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int I = h.I;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < h.T; t += gridDim.x * 8) {
    float4* arow = reinterpret_cast<float4*>(A + static_cast<size_t>(t) * I);
    float4* urow = U != nullptr ? reinterpret_cast<float4*>(U + static_cast<size_t>(t) * I) : nullptr;
    const int slot = h.backup_slot[t];
    if (slot >= 0) {
      const float4* sa = reinterpret_cast<const float4*>(h.backup_a + static_cast<size_t>(slot) * I);
      const float4* su = U != nullptr ? reinterpret_cast<const float4*>(h.backup_u + static_cast<size_t>(slot) * I) : nullptr;
      for (int c = lane; c < I / 4; c += 32) {
        arow[c] = sa[c];
        if (urow != nullptr) urow[c] = su[c];
      }
      continue;
    }
    for (int c = lane; c < I / 4; c += 32) {
      arow[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (urow != nullptr) urow[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncwarp();  // the zeros land before any lane's entries
    if (slot != -1) continue;
    const size_t rb = static_cast<size_t>(t) * h.R;
    const int n = min(h.ell_nnz[t], h.R);
    for (int s = lane; s < n; s += 32) {
      const int j = h.ell_idx[rb + s];
      if (j >= I) continue;  // not a column of this matrix: nothing to write
      A[static_cast<size_t>(t) * I + j] = bf16_to_f32(h.ell_a[rb + s]);
      if (U != nullptr) U[static_cast<size_t>(t) * I + j] = f16_to_f32(h.ell_u[rb + s]);
    }
  }
}

cudaError_t launch_hybrid_unpack(const tw_hybrid& h, float* A, float* U, cudaStream_t s) {
  if (h.T == 0) return cudaSuccess;
  cudaError_t e = launch(hybrid_unpack_kernel, dim3(rows_grid(h.T)), dim3(256), 0, s, h, A, U);
  trace_mark(s, "hybrid_unpack");
  return e;
}

// ------------------------------------------------------------------ dense route, non-gated
// H is fp16 (the down GEMM's operand). Row t without a backup slot: H[t] = its TwELL
// activations (zeros elsewhere), and its ELL row: the slots of tile k go to ELL offsets
// starting at the nonzeros of tiles 0 .. k - 1 (a warp scan over the tiles, 32 at a
// time). Backup rows: H[t] = fp16 of the saved fp32 a row; rows past the backup
// capacity: 0.
__global__ void __launch_bounds__(256) twell_to_dense_ell_kernel(const tw_twell tw, const int32_t* __restrict__ backup_slot,
                                                                const float* __restrict__ backup_a, int cap, int R,
                                                                uint16_t* __restrict__ H,
                                                                uint16_t* __restrict__ ell_idx,
                                                                uint16_t* __restrict__ ell_a, const int32_t* route,
                                                                int32_t* status) {
  pdl_enter();
  if (route != nullptr && *route != 1) return;  // the call took the sparse route
  const int lane = threadIdx.x & 31;
  const int nT = tw.I / tw.W;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < tw.T; t += gridDim.x * 8) {
    uint4* row = reinterpret_cast<uint4*>(H + static_cast<size_t>(t) * tw.I);
    const int slot = backup_slot[t];
    if (slot >= 0 && TW_CHECKED(slot < cap, status)) {
      const float4* src = reinterpret_cast<const float4*>(backup_a + static_cast<size_t>(slot) * tw.I);
      for (int c = lane; c < tw.I / 8; c += 32) {
        const float4 x0 = src[2 * c], x1 = src[2 * c + 1];
        row[c] = make_uint4(pack_f16x2_rn(x0.x, x0.y), pack_f16x2_rn(x0.z, x0.w), pack_f16x2_rn(x1.x, x1.y),
                            pack_f16x2_rn(x1.z, x1.w));
      }
      continue;
    }
    for (int c = lane; c < tw.I / 8; c += 32) row[c] = make_uint4(0u, 0u, 0u, 0u);
    if (slot != -1) continue;
    __syncwarp();  // the zeros land before any lane's slots
    const size_t rb = static_cast<size_t>(t) * R;
    int base = 0;
    for (int k0 = 0; k0 < nT; k0 += 32) {
      const int k = k0 + lane;
      const size_t tk = static_cast<size_t>(t) * nT + k;
      const int n = k < nT ? min(static_cast<int>(tw.cnt[tk]), tw.C) : 0;
      const int incl = warp_inclusive_scan(n);
      int off = base + incl - n;
      for (int s = 0; s < n; ++s, ++off) {
        const int li = tw.idx[tk * tw.C + s];
        if (!TW_CHECKED(li < tw.W && off < R, status)) continue;
        const int j = k * tw.W + li;
        const uint16_t v = tw.val[tk * tw.C + s];
        H[static_cast<size_t>(t) * tw.I + j] = f32_to_f16(bf16_to_f32(v));
        ell_idx[rb + off] = static_cast<uint16_t>(j);
        ell_a[rb + off] = v;
      }
      base += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
}

// The ELL rows' entries (idx, a) alone, for the sparse route's forward: a warp a row,
// lane l taking TwELL tiles 2 l and 2 l + 1 of each group of 64; a group's loads (the
// row's backup slot, the tiles' counts and their first sixteen slots as 16-byte
// vectors) are issued together before the warp scan that places the tiles' slots at
// their ELL offsets.
namespace {
struct TileSlots {
  int n;
  uint4 iv, v0, v1;
};
TW_DEV TileSlots load_tile(const tw_twell& tw, size_t tk, bool live, bool vec) {
  TileSlots r{0, make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
  if (live) {
    r.n = min(static_cast<int>(tw.cnt[tk]), tw.C);
    if (vec) {
      r.iv = *reinterpret_cast<const uint4*>(tw.idx + tk * tw.C);
      r.v0 = *reinterpret_cast<const uint4*>(tw.val + tk * tw.C);
      r.v1 = *reinterpret_cast<const uint4*>(tw.val + tk * tw.C + 8);
    }
  }
  return r;
}
TW_DEV void put_tile(const tw_twell& tw, const TileSlots& ts, size_t tk, int k, int off, int R, size_t rb,
                     uint16_t* ell_idx, uint16_t* ell_a, bool vec, int32_t* status) {
  if (vec) {
    const uint32_t iw[4] = {ts.iv.x, ts.iv.y, ts.iv.z, ts.iv.w};
    const uint32_t vw[8] = {ts.v0.x, ts.v0.y, ts.v0.z, ts.v0.w, ts.v1.x, ts.v1.y, ts.v1.z, ts.v1.w};
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      if (s >= ts.n) break;
      const int li = static_cast<int>((iw[s >> 2] >> (8 * (s & 3))) & 0xFFu);
      if (!TW_CHECKED(li < tw.W && off + s < R, status)) continue;
      ell_idx[rb + off + s] = static_cast<uint16_t>(k * tw.W + li);
      ell_a[rb + off + s] = static_cast<uint16_t>(vw[s >> 1] >> (16 * (s & 1)));
    }
  }
  for (int s = vec ? 16 : 0; s < ts.n; ++s) {
    const int li = tw.idx[tk * tw.C + s];
    if (!TW_CHECKED(li < tw.W && off + s < R, status)) continue;
    ell_idx[rb + off + s] = static_cast<uint16_t>(k * tw.W + li);
    ell_a[rb + off + s] = tw.val[tk * tw.C + s];
  }
}
}  // namespace

__global__ void __launch_bounds__(256) twell_to_ell_kernel(const tw_twell tw, const int32_t* __restrict__ backup_slot,
                                                          int R, uint16_t* __restrict__ ell_idx,
                                                          uint16_t* __restrict__ ell_a, const int32_t* route,
                                                          int32_t* status) {
  pdl_enter();
  if (route != nullptr && *route == 1) return;  // the call took the dense route
  const int lane = threadIdx.x & 31;
  const int nT = tw.I / tw.W;
  const bool vec = tw.C % 16 == 0;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < tw.T; t += gridDim.x * 8) {
    const size_t rb = static_cast<size_t>(t) * R;
    int base = 0;
    for (int k0 = 0; k0 < nT; k0 += 64) {
      const int ka = k0 + 2 * lane, kb = ka + 1;
      const size_t ta = static_cast<size_t>(t) * nT + ka;
      const int slot = backup_slot[t];
      const TileSlots sa = load_tile(tw, ta, ka < nT, vec);
      const TileSlots sb = load_tile(tw, ta + 1, kb < nT, vec);
      if (slot != -1) break;  // uniform over the warp: a backup row has no ELL entries
      const int pair_n = sa.n + sb.n;
      const int incl = warp_inclusive_scan(pair_n);
      const int off = base + incl - pair_n;
      put_tile(tw, sa, ta, ka, off, R, rb, ell_idx, ell_a, vec, status);
      put_tile(tw, sb, ta + 1, kb, off + sa.n, R, rb, ell_idx, ell_a, vec, status);
      base += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
}

cudaError_t launch_twell_to_ell(const tw_twell& tw, const int32_t* backup_slot, int R, uint16_t* ell_idx,
                                uint16_t* ell_a, const int32_t* route, int32_t* status, cudaStream_t s) {
  if (tw.T == 0) return cudaSuccess;
  cudaError_t e = launch(twell_to_ell_kernel, dim3(rows_grid(tw.T)), dim3(256), 0, s, tw, backup_slot, R, ell_idx,
                         ell_a, route, status);
  trace_mark(s, "twell_to_ell");
  return e;
}

cudaError_t launch_twell_to_dense_ell(const tw_twell& tw, const int32_t* backup_slot, const float* backup_a, int cap,
                                      int R, uint16_t* H, uint16_t* ell_idx, uint16_t* ell_a, const int32_t* route,
                                      int32_t* status, cudaStream_t s) {
  if (tw.T == 0) return cudaSuccess;
  cudaError_t e = launch(twell_to_dense_ell_kernel, dim3(rows_grid(tw.T)), dim3(256), 0, s, tw, backup_slot, backup_a,
                         cap, R, H, ell_idx, ell_a, route, status);
  trace_mark(s, "twell_to_dense_ell");
  return e;
}

}  // namespace tw

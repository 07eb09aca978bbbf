// Host launchers of the tcgen05 GEMM instances used by the library: the fused
// gate projection + TwELL pack, the dense backup forward and backward GEMMs, and a
// plain fp32-output GEMM that exposes the operand layouts for testing.
#include <algorithm>

#include <cudaTypedefs.h>

#include "tw_gemm.cuh"
#include "tw_internal.h"

namespace tw {

static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2D bf16 tensor map with 128-byte swizzle: dims {inner, outer}, rows row_bytes apart,
// box {box_inner, box_outer} (box_inner * 2 bytes must be <= 128). Out-of-range
// elements read as zero.
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                    uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_tiled_fn();
  if (fn == nullptr || inner == 0 || outer == 0) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// tensor maps for the operand forms: K-major [rows, K] (box 64 x box_rows) and
// MN-major [K, cols] (box 64 x 64)
static bool tmap_kmajor(CUtensorMap* m, const uint16_t* p, int rows, int K, int box_rows) {
  return make_tmap_bf16(m, p, K, rows, static_cast<uint64_t>(K) * 2, 64, box_rows);
}
static bool tmap_mnmajor(CUtensorMap* m, const uint16_t* p, int K, int cols) {
  return make_tmap_bf16(m, p, cols, K, static_cast<uint64_t>(cols) * 2, 64, 64);
}

template <int BN, bool A_MN, bool B_MN, bool DUAL, int STAGES, class Epi>
static cudaError_t run_gemm(const CUtensorMap& a0, const CUtensorMap& b0, const CUtensorMap& a1,
                            const CUtensorMap& b1, const GemmShape& sh, const typename Epi::Params& ep,
                            int max_rows, cudaStream_t s) {
  using Tr = GemmTraits<BN, A_MN, B_MN, DUAL, STAGES>;
  auto kern = gemm_tc_kernel<BN, A_MN, B_MN, DUAL, STAGES, Epi>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long tiles = static_cast<long>((max_rows + GEMM_BM - 1) / GEMM_BM) * (sh.N / BN);
  if (tiles <= 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<long>(tiles, device_sm_count()));
  kern<<<grid, GEMM_THREADS, Tr::SMEM_BYTES, s>>>(a0, b0, a1, b1, sh, ep);
  return cudaGetLastError();
}

static GemmShape shape_static(int M, int N, int K, int32_t* status) {
  GemmShape g{};
  g.M = M;
  g.m_dev = nullptr;
  g.m_cap = M;
  g.N = N;
  g.K = K;
  g.k_dev = nullptr;
  g.k_cap = K;
  g.segments = 1;
  g.status = status;
  return g;
}

// ------------------------------------------------------------------ gate + pack
cudaError_t gemm_gate_pack(const uint16_t* x, const uint16_t* Wg, int T, int d, int I, int W, int C,
                           const tw_twell& o, uint16_t* a_dense, int32_t* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  EpiTwellPack::Params ep{T, W, C, I / W, o.cnt, o.val, o.idx, o.row_nnz, o.ovf, a_dense, I};
  const GemmShape sh = shape_static(T, I, d, status);
  CUtensorMap ta, tb;
  if (I % 256 == 0) {
    if (!tmap_kmajor(&ta, x, T, d, 128) || !tmap_kmajor(&tb, Wg, I, d, 256)) return cudaErrorInvalidValue;
    return run_gemm<256, false, false, false, 4, EpiTwellPack>(ta, tb, ta, tb, sh, ep, T, s);
  }
  if (I % 128 == 0) {
    if (!tmap_kmajor(&ta, x, T, d, 128) || !tmap_kmajor(&tb, Wg, I, d, 128)) return cudaErrorInvalidValue;
    return run_gemm<128, false, false, false, 6, EpiTwellPack>(ta, tb, ta, tb, sh, ep, T, s);
  }
  if (!tmap_kmajor(&ta, x, T, d, 128) || !tmap_kmajor(&tb, Wg, I, d, 64)) return cudaErrorInvalidValue;
  return run_gemm<64, false, false, false, 8, EpiTwellPack>(ta, tb, ta, tb, sh, ep, T, s);
}

// ------------------------------------------------------------------ dense backup, forward
cudaError_t gemm_backup_hidden(const uint16_t* X, const uint16_t* Wg, const uint16_t* Wu, int rows_alloc,
                               const int32_t* n_dev, int cap, int d, int I, uint16_t* H, uint16_t* save_a,
                               uint16_t* save_u, int32_t* status, cudaStream_t s) {
  if (cap <= 0) return cudaSuccess;
  GemmShape sh = shape_static(0, I, d, status);
  sh.m_dev = n_dev;
  sh.m_cap = cap;
  CUtensorMap ta, tg, tu;
  if (!tmap_kmajor(&ta, X, rows_alloc, d, 128) || !tmap_kmajor(&tg, Wg, I, d, 64)) return cudaErrorInvalidValue;
  if (Wu != nullptr) {
    if (!tmap_kmajor(&tu, Wu, I, d, 64)) return cudaErrorInvalidValue;
    typename EpiBackupHidden<true>::Params ep{H, save_a, save_u, I, rows_alloc};
    return run_gemm<64, false, false, true, 6, EpiBackupHidden<true>>(ta, tg, ta, tu, sh, ep, cap, s);
  }
  typename EpiBackupHidden<false>::Params ep{H, save_a, nullptr, I, rows_alloc};
  return run_gemm<64, false, false, false, 8, EpiBackupHidden<false>>(ta, tg, ta, tg, sh, ep, cap, s);
}

cudaError_t gemm_rows_times_nmajor(const uint16_t* A0, const uint16_t* B0, const uint16_t* A1, const uint16_t* B1,
                                   int segments, int rows_alloc, const int32_t* n_dev, int cap, int K, int N,
                                   uint16_t* out, int ldo, const int32_t* row_map, int32_t* status, cudaStream_t s) {
  if (cap <= 0) return cudaSuccess;
  GemmShape sh = shape_static(0, N, K, status);
  sh.m_dev = n_dev;
  sh.m_cap = cap;
  sh.segments = segments;
  CUtensorMap ta0, tb0, ta1, tb1;
  if (!tmap_kmajor(&ta0, A0, rows_alloc, K, 128) || !tmap_mnmajor(&tb0, B0, K, N)) return cudaErrorInvalidValue;
  if (segments > 1) {
    if (!tmap_kmajor(&ta1, A1, rows_alloc, K, 128) || !tmap_mnmajor(&tb1, B1, K, N)) return cudaErrorInvalidValue;
  } else {
    ta1 = ta0;
    tb1 = tb0;
  }
  EpiScatterBf16::Params ep{out, ldo, row_map};
  return run_gemm<64, false, true, false, 8, EpiScatterBf16>(ta0, tb0, ta1, tb1, sh, ep, cap, s);
}

// ------------------------------------------------------------------ dense backup, backward
cudaError_t gemm_backup_grad(const uint16_t* dY, const uint16_t* Wd, int rows_alloc, const int32_t* n_dev, int cap,
                             int d, int I, const uint16_t* a, const uint16_t* u, float l1, uint16_t* dG,
                             uint16_t* dU, uint16_t* H, int32_t* status, cudaStream_t s) {
  if (cap <= 0) return cudaSuccess;
  GemmShape sh = shape_static(0, I, d, status);
  sh.m_dev = n_dev;
  sh.m_cap = cap;
  CUtensorMap ta, tb;
  if (!tmap_kmajor(&ta, dY, rows_alloc, d, 128) || !tmap_kmajor(&tb, Wd, I, d, 64)) return cudaErrorInvalidValue;
  if (u != nullptr) {
    typename EpiBackupGrad<true>::Params ep{a, u, dG, dU, H, l1, I, rows_alloc};
    return run_gemm<64, false, false, false, 8, EpiBackupGrad<true>>(ta, tb, ta, tb, sh, ep, cap, s);
  }
  typename EpiBackupGrad<false>::Params ep{a, nullptr, dG, nullptr, H, l1, I, rows_alloc};
  return run_gemm<64, false, false, false, 8, EpiBackupGrad<false>>(ta, tb, ta, tb, sh, ep, cap, s);
}

cudaError_t gemm_weight_grad_add(const uint16_t* P, const uint16_t* Q, int rows_alloc, const int32_t* n_dev,
                                 int cap, int I, int d, float* D, int32_t* status, cudaStream_t s) {
  if (cap <= 0) return cudaSuccess;
  GemmShape sh = shape_static(I, d, 0, status);
  sh.k_dev = n_dev;
  sh.k_cap = cap;
  CUtensorMap ta, tb;
  if (!tmap_mnmajor(&ta, P, rows_alloc, I) || !tmap_mnmajor(&tb, Q, rows_alloc, d)) return cudaErrorInvalidValue;
  EpiAddF32::Params ep{D, d};
  if (d % 256 == 0) return run_gemm<256, true, true, false, 4, EpiAddF32>(ta, tb, ta, tb, sh, ep, I, s);
  return run_gemm<64, true, true, false, 8, EpiAddF32>(ta, tb, ta, tb, sh, ep, I, s);
}

// ------------------------------------------------------------------ layout test GEMM
cudaError_t gemm_dense_test(const uint16_t* A, const uint16_t* B, int M, int N, int K, int a_mn, int b_mn, float* D,
                            int32_t* status, cudaStream_t s) {
  const GemmShape sh = shape_static(M, N, K, status);
  EpiStoreF32::Params ep{D, N};
  CUtensorMap ta, tb;
  const bool oka = a_mn ? tmap_mnmajor(&ta, A, K, M) : tmap_kmajor(&ta, A, M, K, 128);
  const bool okb = b_mn ? tmap_mnmajor(&tb, B, K, N) : tmap_kmajor(&tb, B, N, K, 64);
  if (!oka || !okb) return cudaErrorInvalidValue;
  if (!a_mn && !b_mn) return run_gemm<64, false, false, false, 8, EpiStoreF32>(ta, tb, ta, tb, sh, ep, M, s);
  if (!a_mn && b_mn) return run_gemm<64, false, true, false, 8, EpiStoreF32>(ta, tb, ta, tb, sh, ep, M, s);
  if (a_mn && !b_mn) return run_gemm<64, true, false, false, 8, EpiStoreF32>(ta, tb, ta, tb, sh, ep, M, s);
  return run_gemm<64, true, true, false, 8, EpiStoreF32>(ta, tb, ta, tb, sh, ep, M, s);
}

}  // namespace tw

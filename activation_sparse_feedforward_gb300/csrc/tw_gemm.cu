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

// 2D bf16 tensor map with 128-byte swizzle (64-byte with swizzle64): dims {inner,
// outer}, rows row_bytes apart, box {box_inner, box_outer} (box_inner * 2 bytes must
// be at most the swizzle span). Out-of-range elements read as zero; stores past the
// dims are clipped.
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                    uint32_t box_inner, uint32_t box_outer, bool swizzle64) {
  auto fn = encode_tiled_fn();
  if (fn == nullptr || inner == 0 || outer == 0) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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

// max_rows bounds the rows of D (the grid has at most one CTA per tile); a device-
// chosen split (sh.ksplit < 0) gets one CTA per SM.
//
// PAIR launches clusters of two CTAs (one 256-row unit per pair at a time), as many
// pairs as can be resident at once (at most one CTA per SM), without a K split.
template <int BN, bool A_MN, bool B_MN, bool DUAL, int STAGES, class Epi, int NA = 1, bool PAIR = false>
static cudaError_t run_gemm(const GemmMaps& maps, const GemmShape& sh, const typename Epi::Params& ep, int max_rows,
                            cudaStream_t s, const char* label) {
  using Tr = GemmTraits<BN, A_MN, B_MN, DUAL, STAGES, NA, false, PAIR>;
  auto kern = gemm_tc_kernel<BN, A_MN, B_MN, DUAL, STAGES, Epi, NA, PAIR>;
  constexpr int smem = Tr::SMEM_BYTES + Epi::kStageBytes * (epi_warps<BN, Epi>() / 4);
  static_assert(smem <= 232448, "GEMM shared memory above the 227 KiB opt-in limit");
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long tiles = static_cast<long>((max_rows + Tr::UNIT_ROWS - 1) / Tr::UNIT_ROWS) * (sh.N / BN);
  if (tiles <= 0) return cudaSuccess;
  if constexpr (PAIR) {
    if (sh.ksplit > 1 || sh.ksplit < 0) return cudaErrorInvalidValue;  // CTA pairs run whole tiles
    static int resident_pairs = -1;  // per instantiation: the query depends only on the kernel
    if (resident_pairs < 0) resident_pairs = max_active_clusters(kern, gemm_threads<BN, Epi>(), smem, 2);
    const int pairs = static_cast<int>(std::min<long>(tiles, std::min(resident_pairs, device_sm_count() / 2)));
    if (pairs < 1) return cudaErrorInvalidConfiguration;
    e = launch_clustered(kern, dim3(2 * pairs), dim3(gemm_threads<BN, Epi>()), smem, 2, s, maps, sh, ep);
  } else {
    const int grid = sh.ksplit < 0 ? device_sm_count() : static_cast<int>(std::min<long>(tiles, device_sm_count()));
    e = launch(kern, dim3(grid), dim3(gemm_threads<BN, Epi>()), smem, s, maps, sh, ep);
  }
  trace_mark(s, label);
  return e;
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
  g.problems = 1;
  g.status = status;
  g.withhold_kb = -1;
  g.route_dev = nullptr;
  g.route_want = 0;
  return g;
}

// unused map slots repeat the first ones so that every slot holds a valid map
static void fill_unused(GemmMaps& m, int used_a, int used_b) {
  for (int i = used_a; i < GEMM_MAX_SEGMENTS; ++i) m.a[i] = m.a[0];
  for (int i = used_b; i < GEMM_MAX_SEGMENTS; ++i) m.b[i] = m.b[0];
}

// ------------------------------------------------------------------ gate + pack
cudaError_t gemm_gate_pack(const uint16_t* x, const uint16_t* Wg, int T, int d, int I, int W, int C,
                           const tw_twell& o, uint16_t* a_dense, int32_t* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  EpiTwellPack::Params ep{T, W, C, I / W, o.cnt, o.val, o.idx, o.row_nnz, o.ovf, a_dense, I};
  GemmShape sh = shape_static(T, I, d, status);
  GemmMaps maps;
  const int bn = (I % 256 == 0) ? 256 : (I % 128 == 0) ? 128 : 64;
  sh.split_tail = (bn / 2) % W == 0;  // a half unit must hold whole TwELL tiles
  // 256-wide tiles run on CTA pairs, each CTA loading half of the B tile
  if (!tmap_kmajor(&maps.a[0], x, T, d, 128) || !tmap_kmajor(&maps.b[0], Wg, I, d, bn == 256 ? 128 : bn))
    return cudaErrorInvalidValue;
  fill_unused(maps, 1, 1);
  if (bn == 256) return run_gemm<256, false, false, false, 6, EpiTwellPack, 1, true>(maps, sh, ep, T, s, "gate_pack");
  if (bn == 128) return run_gemm<128, false, false, false, 6, EpiTwellPack>(maps, sh, ep, T, s, "gate_pack");
  return run_gemm<64, false, false, false, 8, EpiTwellPack>(maps, sh, ep, T, s, "gate_pack");
}

// ------------------------------------------------------------------ unfused gate
cudaError_t gemm_gate_relu_dense(const uint16_t* x, const uint16_t* Wg, int T, int d, int I, uint16_t* a,
                                 int32_t* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  EpiReluBf16::Params ep{a, I};
  GemmShape sh = shape_static(T, I, d, status);
  sh.split_tail = true;
  GemmMaps maps;
  const int bn = (I % 256 == 0) ? 256 : (I % 128 == 0) ? 128 : 64;
  // 256-wide tiles run on CTA pairs, each CTA loading half of the B tile
  if (!tmap_kmajor(&maps.a[0], x, T, d, 128) || !tmap_kmajor(&maps.b[0], Wg, I, d, bn == 256 ? 128 : bn))
    return cudaErrorInvalidValue;
  fill_unused(maps, 1, 1);
  if (bn == 256) return run_gemm<256, false, false, false, 6, EpiReluBf16, 1, true>(maps, sh, ep, T, s, "gate_dense");
  if (bn == 128) return run_gemm<128, false, false, false, 6, EpiReluBf16>(maps, sh, ep, T, s, "gate_dense");
  return run_gemm<64, false, false, false, 8, EpiReluBf16>(maps, sh, ep, T, s, "gate_dense");
}

// ------------------------------------------------------------------ dense backup, split-K forms
// For few backup rows the hidden and grad products would run a fraction of a round of
// tiles on the SMs (2 row tiles x 44 column tiles at 164 rows); instead each output
// tile's K loop is cut into units spread over every SM (the split chosen on the device
// from the actual row count by split_by_cost), whose partial sums are added into
// fp32 accumulators that the row gather zeroed; a finishing kernel then applies the
// epilogue's arithmetic (tw_kernels.cu).
template <int BN>
static cudaError_t rows_split_bn(const GemmMaps& maps, const GemmShape& sh, const EpiRedF32Grouped::Params& ep,
                                 int max_rows, cudaStream_t s, const char* label) {
  constexpr int kStageBytes = (128 + BN) * 64 * 2;
  constexpr int kStages = (192 * 1024) / kStageBytes < 8 ? (192 * 1024) / kStageBytes : 8;
  return run_gemm<BN, false, false, false, kStages, EpiRedF32Grouped>(maps, sh, ep, max_rows, s, label);
}

// acc[p][i][:] += X[i] . B_p^T for the n (device) rows i of X [rows_alloc, K] and
// problems p < n_b (B_p [N, K], K-major); acc rows have stride ld.
static cudaError_t rows_times_kmajor_split(const uint16_t* X, const uint16_t* const* B, int n_b, int rows_alloc,
                                           const int32_t* n_dev, int cap, int K, int N, float* const* acc, int ld,
                                           int32_t* status, cudaStream_t s, const int32_t* sparse_only,
                                           const char* label) {
  if (n_b < 1 || n_b > EpiRedF32Grouped::kMaxProblems || N % 64 != 0) return cudaErrorInvalidValue;
  GemmShape sh = shape_static(0, N, K, status);
  sh.m_dev = n_dev;
  sh.m_cap = cap;
  sh.problems = n_b;
  sh.ksplit = -2;
  sh.route_dev = sparse_only;
  sh.route_want = 0;
  const int bn = (N % 256 == 0) ? 256 : (N % 128 == 0) ? 128 : 64;
  GemmMaps maps;
  EpiRedF32Grouped::Params ep{};
  for (int p = 0; p < n_b; ++p) {
    if (!tmap_kmajor(&maps.a[p], X, rows_alloc, K, 128) || !tmap_kmajor(&maps.b[p], B[p], N, K, bn))
      return cudaErrorInvalidValue;
    ep.acc[p] = acc[p];
  }
  fill_unused(maps, n_b, n_b);
  ep.ld = ld;
  const int max_rows = (cap + GEMM_BM - 1) / GEMM_BM * GEMM_BM * n_b;
  if (bn == 256) return rows_split_bn<256>(maps, sh, ep, max_rows, s, label);
  if (bn == 128) return rows_split_bn<128>(maps, sh, ep, max_rows, s, label);
  return rows_split_bn<64>(maps, sh, ep, max_rows, s, label);
}

// save_a = ReLU(X Wg^T) and (when Wu) save_u = X Wu^T over the n (device) rows of X
// [rows_alloc, d]: one grouped launch of one or two problems on 256-wide tiles (128 or
// 64 when I requires), fp32 rows of stride I.
template <int BN>
static cudaError_t rows_store_bn(const GemmMaps& maps, const GemmShape& sh, const EpiStoreF32RowsGrouped::Params& ep,
                                 int max_rows, cudaStream_t s) {
  constexpr bool kPair = BN == 256;  // CTA pairs, each CTA loading half of the B tile
  constexpr int kStageBytes = (128 + (kPair ? BN / 2 : BN)) * 64 * 2;
  constexpr int kStages = (192 * 1024) / kStageBytes < 8 ? (192 * 1024) / kStageBytes : 8;
  return run_gemm<BN, false, false, false, kStages, EpiStoreF32RowsGrouped, 1, kPair>(maps, sh, ep, max_rows, s,
                                                                                      "backup_hidden");
}
static cudaError_t rows_store_a_u(const uint16_t* X, const uint16_t* Wg, const uint16_t* Wu, int rows_alloc,
                                  const int32_t* n_dev, int cap, int d, int I, float* save_a, float* save_u,
                                  int32_t* status, cudaStream_t s, const int32_t* route) {
  const int n_b = Wu != nullptr ? 2 : 1;
  GemmShape sh = shape_static(0, I, d, status);
  sh.m_dev = n_dev;
  sh.m_cap = cap;
  sh.problems = n_b;
  // the dense route's up GEMM saves u for these rows itself
  if (n_b == 2) sh.drop_last_problem_if = route;
  const int bn = (I % 256 == 0) ? 256 : (I % 128 == 0) ? 128 : 64;
  GemmMaps maps;
  const uint16_t* B[2] = {Wg, Wu};
  const int unit_rows = bn == 256 ? 2 * GEMM_BM : GEMM_BM;  // CTA pairs on 256-wide tiles
  EpiStoreF32RowsGrouped::Params ep{{save_a, save_u}, I, 1u, unit_rows};
  for (int p = 0; p < n_b; ++p)
    if (!tmap_kmajor(&maps.a[p], X, rows_alloc, d, 128) || !tmap_kmajor(&maps.b[p], B[p], I, d, bn == 256 ? 128 : bn))
      return cudaErrorInvalidValue;
  fill_unused(maps, n_b, n_b);
  const int max_rows = (cap + unit_rows - 1) / unit_rows * unit_rows * n_b;
  if (bn == 256) return rows_store_bn<256>(maps, sh, ep, max_rows, s);
  if (bn == 128) return rows_store_bn<128>(maps, sh, ep, max_rows, s);
  return rows_store_bn<64>(maps, sh, ep, max_rows, s);
}

// ------------------------------------------------------------------ dense backup, forward
// The form without saved rows (the inference forward's overflow rows): h formed in
// the epilogue from both accumulators. The gated form (two B operands, gate and up,
// into two accumulators) runs 64-wide column tiles; the non-gated form 128-wide tiles
// when I allows them, else 64-wide; as many stages as fit about 192 KB.
template <int BN, bool GATED>
static cudaError_t backup_hidden_bn(const uint16_t* X, const uint16_t* Wg, const uint16_t* Wu, int rows_alloc,
                                    const int32_t* n_dev, int cap, int d, int I, uint16_t* H, uint16_t* H_lo,
                                    float* save_a, float* save_u, int32_t* status, cudaStream_t s,
                                    const int32_t* route) {
  GemmShape sh = shape_static(0, I, d, status);
  sh.m_dev = n_dev;
  sh.m_cap = cap;
  GemmMaps maps;
  if (!tmap_kmajor(&maps.a[0], X, rows_alloc, d, 128) || !tmap_kmajor(&maps.b[0], Wg, I, d, BN))
    return cudaErrorInvalidValue;
  if (GATED && !tmap_kmajor(&maps.b[1], Wu, I, d, BN)) return cudaErrorInvalidValue;
  fill_unused(maps, 1, GATED ? 2 : 1);
  typename EpiBackupHidden<GATED>::Params ep{H, H_lo, save_a, GATED ? save_u : nullptr, I, rows_alloc, route};
  constexpr int kStageBytes = (128 + (GATED ? 2 : 1) * BN) * 64 * 2;
  constexpr int kStages = (192 * 1024) / kStageBytes < 8 ? (192 * 1024) / kStageBytes : 8;
  return run_gemm<BN, false, false, GATED, kStages, EpiBackupHidden<GATED>>(maps, sh, ep, cap, s, "backup_hidden");
}

cudaError_t gemm_backup_hidden(const uint16_t* X, const uint16_t* Wg, const uint16_t* Wu, int rows_alloc,
                               const int32_t* n_dev, int cap, int d, int I, uint16_t* H, uint16_t* H_lo,
                               float* save_a, float* save_u, int32_t* status, cudaStream_t s,
                               const int32_t* route, float* split_acc, int split_ld) {
  if (cap <= 0) return cudaSuccess;
  if (split_acc != nullptr) {
    const uint16_t* B[2] = {Wg, Wu};
    float* acc[2] = {split_acc, split_acc + I};
    const cudaError_t e = rows_times_kmajor_split(X, B, Wu != nullptr ? 2 : 1, rows_alloc, n_dev, cap, d, I, acc,
                                                  split_ld, status, s, nullptr, "backup_hidden");
    if (e != cudaSuccess) return e;
    return launch_backup_hidden_finish(split_acc, split_ld, n_dev, cap, I, Wu != nullptr, H, H_lo, rows_alloc, save_a,
                                       save_u, route, s, false);
  }
  if (save_a != nullptr && (Wu == nullptr || save_u != nullptr)) {
    // a large backup in training: a = ReLU(x Wg^T) and u = x Wu^T stored straight into
    // the saved fp32 rows by one grouped launch on full-width tiles, then h as its hi /
    // lo pair from them (only when the call takes the sparse route, whose down GEMM
    // reads it)
    const cudaError_t e = rows_store_a_u(X, Wg, Wu, rows_alloc, n_dev, cap, d, I, save_a, save_u, status, s, route);
    if (e != cudaSuccess) return e;
    return launch_backup_hidden_finish(save_a, I, n_dev, cap, I, Wu != nullptr, H, H_lo, rows_alloc, save_a, save_u,
                                       route, s, true);
  }
  if (Wu != nullptr)
    return backup_hidden_bn<64, true>(X, Wg, Wu, rows_alloc, n_dev, cap, d, I, H, H_lo, save_a, save_u, status, s,
                                      route);
  if (I % 128 == 0)
    return backup_hidden_bn<128, false>(X, Wg, Wu, rows_alloc, n_dev, cap, d, I, H, H_lo, save_a, save_u, status, s,
                                        route);
  return backup_hidden_bn<64, false>(X, Wg, Wu, rows_alloc, n_dev, cap, d, I, H, H_lo, save_a, save_u, status, s,
                                     route);
}

// Same product for few rows, spread over every SM: 256-wide column tiles, each tile's
// K loop (all segments; a pair of segments over the same B is one K step) cut into
// slices whose partial sums are added into the fp32
// accumulator acc [cap, N] (zeroed beforehand, by the row gather); launch_scatter_rows_bf16
// then writes the bf16 rows out.
cudaError_t gemm_rows_times_nmajor_splitk(const uint16_t* const* A, const uint16_t* const* B, int segments,
                                          int rows_alloc, const int32_t* n_dev, int cap, int K, int N, float* acc,
                                          int32_t* status, cudaStream_t s, const int32_t* sparse_only, int ld_acc) {
  if (cap <= 0) return cudaSuccess;
  if (segments < 1 || segments > GEMM_MAX_SEGMENTS || N % 256 != 0) return cudaErrorInvalidValue;
  GemmShape sh = shape_static(0, N, K, status);
  sh.m_dev = n_dev;
  sh.m_cap = cap;
  sh.segments = segments;
  sh.ksplit = -1;  // the row count is on the device: the kernel picks the split
  sh.route_dev = sparse_only;
  sh.route_want = 0;
  GemmMaps maps;
  for (int i = 0; i < segments; ++i)
    if (!tmap_kmajor(&maps.a[i], A[i], rows_alloc, K, 128) || !tmap_mnmajor(&maps.b[i], B[i], K, N))
      return cudaErrorInvalidValue;
  fill_unused(maps, segments, segments);
  EpiRedF32::Params ep{acc, ld_acc > 0 ? ld_acc : N};
  // segments that come in pairs over one B (the hi / lo halves of a split operand)
  // load that B tile once for both
  bool paired = segments % 2 == 0;
  for (int i = 0; paired && i < segments; i += 2) paired = B[i] == B[i + 1];
  // (the trace label names the segment count, which sets the product's FLOPs)
  const char* label = segments == 4 ? "backup_rows_gemm4" : "backup_rows_gemm";
  if (paired) return run_gemm<256, false, true, false, 3, EpiRedF32, 2>(maps, sh, ep, cap, s, label);
  return run_gemm<256, false, true, false, 4, EpiRedF32>(maps, sh, ep, cap, s, label);
}

// ------------------------------------------------------------------ dense backup, backward
// 128-wide column tiles when I allows them, else 64-wide; as many stages as fit
// about 192 KB.
template <int BN, bool GATED>
static cudaError_t backup_grad_bn(const uint16_t* dY, const uint16_t* Wd, int rows_alloc, const int32_t* n_dev,
                                  int cap, int d, int I, const float* a, const float* u, float l1,
                                  const BackupGradOut& o, int32_t* status, cudaStream_t s, const int32_t* sparse_only) {
  GemmShape sh = shape_static(0, I, d, status);
  sh.m_dev = n_dev;
  sh.m_cap = cap;
  sh.route_dev = sparse_only;
  sh.route_want = 0;
  GemmMaps maps;
  if (!tmap_kmajor(&maps.a[0], dY, rows_alloc, d, 128) || !tmap_kmajor(&maps.b[0], Wd, I, d, BN))
    return cudaErrorInvalidValue;
  fill_unused(maps, 1, 1);
  typename EpiBackupGrad<GATED>::Params ep{a,    u,  o.dG, o.dG_lo, GATED ? o.dU : nullptr, GATED ? o.dU_lo : nullptr,
                                           o.H,  o.H_lo, l1,  I,       rows_alloc};
  constexpr int kStageBytes = (128 + BN) * 64 * 2;
  constexpr int kStages = (192 * 1024) / kStageBytes < 8 ? (192 * 1024) / kStageBytes : 8;
  return run_gemm<BN, false, false, false, kStages, EpiBackupGrad<GATED>>(maps, sh, ep, cap, s, "backup_grad");
}

cudaError_t gemm_backup_grad(const uint16_t* dY, const uint16_t* Wd, int rows_alloc, const int32_t* n_dev, int cap,
                             int d, int I, const float* a, const float* u, float l1, const BackupGradOut& o,
                             int32_t* status, cudaStream_t s, const int32_t* sparse_only, float* split_acc,
                             int split_ld) {
  if (cap <= 0) return cudaSuccess;
  const bool gated = u != nullptr;
  if (split_acc != nullptr) {
    const uint16_t* B[1] = {Wd};
    float* acc[1] = {split_acc};
    const cudaError_t e =
        rows_times_kmajor_split(dY, B, 1, rows_alloc, n_dev, cap, d, I, acc, split_ld, status, s, sparse_only,
                                "backup_grad");
    if (e != cudaSuccess) return e;
    return launch_backup_grad_finish(split_acc, split_ld, n_dev, cap, I, a, u, l1, o, rows_alloc, sparse_only, s);
  }
  if (I % 128 == 0)
    return gated ? backup_grad_bn<128, true>(dY, Wd, rows_alloc, n_dev, cap, d, I, a, u, l1, o, status, s, sparse_only)
                 : backup_grad_bn<128, false>(dY, Wd, rows_alloc, n_dev, cap, d, I, a, u, l1, o, status, s, sparse_only);
  return gated ? backup_grad_bn<64, true>(dY, Wd, rows_alloc, n_dev, cap, d, I, a, u, l1, o, status, s, sparse_only)
               : backup_grad_bn<64, false>(dY, Wd, rows_alloc, n_dev, cap, d, I, a, u, l1, o, status, s, sparse_only);
}

cudaError_t gemm_weight_grads(const WeightGradProblem* probs, int n_probs, int rows_alloc, const int32_t* n_dev,
                              int cap, int I, int d, int32_t* status, cudaStream_t s, const int32_t* sparse_only) {
  if (cap <= 0 || n_probs <= 0) return cudaSuccess;
  if (n_probs > EpiStoreF32Grouped::kMaxProblems || d % 256 != 0) return cudaErrorInvalidValue;
  GemmShape sh = shape_static(I, d, 0, status);
  sh.k_dev = n_dev;
  sh.k_cap = cap;
  sh.segments = 2;  // P = P_hi + P_lo
  sh.problems = n_probs;
  sh.route_dev = sparse_only;
  sh.route_want = 0;
  GemmMaps maps;
  EpiStoreF32Grouped::Params ep{};
  for (int p = 0; p < n_probs; ++p) {
    if (!tmap_mnmajor(&maps.a[2 * p], probs[p].P_hi, rows_alloc, I) ||
        !tmap_mnmajor(&maps.a[2 * p + 1], probs[p].P_lo, rows_alloc, I) ||
        !tmap_mnmajor(&maps.b[2 * p], probs[p].Q, rows_alloc, d))
      return cudaErrorInvalidValue;
    maps.b[2 * p + 1] = maps.b[2 * p];
    ep.D[p] = probs[p].D;
  }
  fill_unused(maps, 2 * n_probs, 2 * n_probs);
  ep.ldd = d;
  // each problem takes whole 128-row tiles; rows I .. of its last tile are skipped
  ep.rows_per_problem = (I + GEMM_BM - 1) / GEMM_BM * GEMM_BM;
  // the hi and lo segments share Q: one Q tile a K step for both
  return run_gemm<256, true, true, false, 3, EpiStoreF32Grouped, 2>(maps, sh, ep, ep.rows_per_problem * n_probs, s,
                                                                     "backup_weight_grad");
}

// ------------------------------------------------------------------ dense route
static void set_route(GemmShape& sh, const int32_t* route) {
  sh.route_dev = route;
  sh.route_want = 1;
}

cudaError_t gemm_up_hybrid(const uint16_t* x, const uint16_t* Wu, int T, int d, int I, const tw_twell& tw, int R,
                           const int32_t* backup_slot, const float* backup_a, float* backup_u, int cap, uint16_t* H,
                           uint16_t* ell_idx, uint16_t* ell_a, uint16_t* ell_u, const int32_t* route,
                           int32_t* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  GemmShape sh = shape_static(T, I, d, status);
  set_route(sh, route);
  sh.split_tail = ((I % 256 == 0 ? 256 : I % 128 == 0 ? 128 : 64) / 2) % tw.W == 0;  // whole TwELL tiles a unit
  EpiUpHybrid::Params ep{T,      tw.W,        tw.C,     I / tw.W, R,   tw.cnt, tw.val,  tw.idx, backup_slot,
                         backup_a, backup_u, cap,      H,        I,   ell_idx, ell_a, ell_u,  status};
  GemmMaps maps;
  const int bn = (I % 256 == 0) ? 256 : (I % 128 == 0) ? 128 : 64;
  // 256-wide tiles run on CTA pairs, each CTA loading half of the B tile
  if (!tmap_kmajor(&maps.a[0], x, T, d, 128) || !tmap_kmajor(&maps.b[0], Wu, I, d, bn == 256 ? 128 : bn))
    return cudaErrorInvalidValue;
  fill_unused(maps, 1, 1);
  if (bn == 256) return run_gemm<256, false, false, false, 6, EpiUpHybrid, 1, true>(maps, sh, ep, T, s, "dense_up");
  if (bn == 128) return run_gemm<128, false, false, false, 6, EpiUpHybrid>(maps, sh, ep, T, s, "dense_up");
  return run_gemm<64, false, false, false, 8, EpiUpHybrid>(maps, sh, ep, T, s, "dense_up");
}

cudaError_t gemm_rows_nmajor_bf16(const uint16_t* const* A, const uint16_t* const* B, int segments, int M, int K,
                                  int N, uint16_t* out, int ld, const int32_t* route, int32_t* status,
                                  cudaStream_t s, bool f16, const char* label) {
  if (M == 0) return cudaSuccess;
  if (segments < 1 || segments > GEMM_MAX_SEGMENTS || N % 256 != 0) return cudaErrorInvalidValue;
  GemmShape sh = shape_static(M, N, K, status);
  sh.segments = segments;
  sh.split_tail = true;
  set_route(sh, route);
  GemmMaps maps;
  for (int i = 0; i < segments; ++i)
    if (!tmap_kmajor(&maps.a[i], A[i], M, K, 128) || !tmap_mnmajor(&maps.b[i], B[i], K, N))
      return cudaErrorInvalidValue;
  fill_unused(maps, segments, segments);
  EpiStoreBf16::Params ep{out, ld};
  // CTA pairs (each CTA loads 128 of the tile's 256 B columns)
  if (f16) return run_gemm<256, false, true, false, 6, F16Operands<EpiStoreBf16>, 1, true>(maps, sh, ep, M, s, label);
  return run_gemm<256, false, true, false, 6, EpiStoreBf16, 1, true>(maps, sh, ep, M, s, label);
}

template <int BN, bool GATED>
static cudaError_t dense_grad_bn(const uint16_t* dY, const uint16_t* Wd, int T, int d, int I, const tw_hybrid& h,
                                 float l1, uint16_t* dG, uint16_t* dU, uint16_t* H, const int32_t* route,
                                 int32_t* status, cudaStream_t s) {
  GemmShape sh = shape_static(T, I, d, status);
  set_route(sh, route);
  sh.split_tail = true;
  GemmMaps maps;
  // 256-wide tiles run on CTA pairs, each CTA loading half of the B tile
  constexpr bool kPair = BN == 256;
  constexpr int kBRows = kPair ? BN / 2 : BN;
  if (!tmap_kmajor(&maps.a[0], dY, T, d, 128) || !tmap_kmajor(&maps.b[0], Wd, I, d, kBRows)) return cudaErrorInvalidValue;
  fill_unused(maps, 1, 1);
  typename EpiDenseGrad<GATED>::Params ep{h.R,
                                          I,
                                          h.ell_nnz,
                                          h.backup_slot,
                                          h.ell_idx,
                                          h.ell_a,
                                          GATED ? h.ell_u : nullptr,
                                          h.backup_cap > 0 ? h.backup_a : nullptr,
                                          GATED && h.backup_cap > 0 ? h.backup_u : nullptr,
                                          h.backup_cap,
                                          l1,
                                          dG,
                                          GATED ? dU : nullptr,
                                          H,
                                          I,
                                          status};
  // the outputs as 32 x 32 fp16 boxes (the bits are copied as they are; rows past T are
  // clipped by the stores)
  const uint64_t row_bytes = static_cast<uint64_t>(I) * 2;
  if (!make_tmap_bf16(&ep.tm_dG, dG, I, T, row_bytes, 32, 32, true) ||
      !make_tmap_bf16(&ep.tm_H, H, I, T, row_bytes, 32, 32, true) ||
      !make_tmap_bf16(&ep.tm_dU, GATED ? dU : dG, I, T, row_bytes, 32, 32, true))
    return cudaErrorInvalidValue;
  constexpr int kStageBytes = (128 + kBRows) * 64 * 2;
  constexpr int kBudget = 232448 - 1280 - EpiDenseGrad<GATED>::kStageBytes * (epi_warps<BN, EpiDenseGrad<GATED>>() / 4);
  constexpr int kStages = kBudget / kStageBytes < 8 ? kBudget / kStageBytes : 8;
  return run_gemm<BN, false, false, false, kStages, EpiDenseGrad<GATED>, 1, kPair>(maps, sh, ep, T, s, "dense_grad");
}

cudaError_t gemm_dense_grad(const uint16_t* dY, const uint16_t* Wd, int T, int d, int I, const tw_hybrid& h,
                            bool gated, float l1, uint16_t* dG, uint16_t* dU, uint16_t* H, const int32_t* route,
                            int32_t* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (I % 256 == 0)
    return gated ? dense_grad_bn<256, true>(dY, Wd, T, d, I, h, l1, dG, dU, H, route, status, s)
                 : dense_grad_bn<256, false>(dY, Wd, T, d, I, h, l1, dG, dU, H, route, status, s);
  if (I % 128 == 0)
    return gated ? dense_grad_bn<128, true>(dY, Wd, T, d, I, h, l1, dG, dU, H, route, status, s)
                 : dense_grad_bn<128, false>(dY, Wd, T, d, I, h, l1, dG, dU, H, route, status, s);
  return gated ? dense_grad_bn<64, true>(dY, Wd, T, d, I, h, l1, dG, dU, H, route, status, s)
               : dense_grad_bn<64, false>(dY, Wd, T, d, I, h, l1, dG, dU, H, route, status, s);
}

cudaError_t gemm_dense_weight_grads(const DenseWeightGradProblem* probs, int n_probs, int T, int I, int d,
                                    const int32_t* add_if, const int32_t* route, int32_t* status, cudaStream_t s) {
  if (T == 0 || n_probs <= 0) return cudaSuccess;
  if (n_probs > EpiF32GroupedStoreOrAdd::kMaxProblems || d % 256 != 0) return cudaErrorInvalidValue;
  GemmShape sh = shape_static(I, d, T, status);
  sh.problems = n_probs;
  set_route(sh, route);
  GemmMaps maps;
  EpiF32GroupedStoreOrAdd::Params ep{};
  for (int p = 0; p < n_probs; ++p) {
    if (!tmap_mnmajor(&maps.a[p], probs[p].P, T, I) || !tmap_mnmajor(&maps.b[p], probs[p].Q, T, d))
      return cudaErrorInvalidValue;
    ep.D[p] = probs[p].D;
  }
  fill_unused(maps, n_probs, n_probs);
  ep.ldd = d;
  // CTA pairs: a problem's rows are whole 256-row units
  ep.rows_per_problem = (I + 2 * GEMM_BM - 1) / (2 * GEMM_BM) * (2 * GEMM_BM);
  ep.add_if = add_if;
  return run_gemm<256, true, true, false, 6, F16Operands<EpiF32GroupedStoreOrAdd>, 1, true>(
      maps, sh, ep, ep.rows_per_problem * n_probs, s, "dense_weight_grad");
}

// ------------------------------------------------------------------ layout test GEMM
cudaError_t gemm_dense_test(const uint16_t* A, const uint16_t* B, int M, int N, int K, int a_mn, int b_mn, float* D,
                            int32_t* status, cudaStream_t s, int withhold_kb, bool pair) {
  GemmShape sh = shape_static(M, N, K, status);
  sh.withhold_kb = withhold_kb;
  sh.split_tail = true;
  EpiStoreF32::Params ep{D, N};
  GemmMaps maps;
  const bool oka = a_mn ? tmap_mnmajor(&maps.a[0], A, K, M) : tmap_kmajor(&maps.a[0], A, M, K, 128);
  const bool okb = b_mn ? tmap_mnmajor(&maps.b[0], B, K, N) : tmap_kmajor(&maps.b[0], B, N, K, pair ? 128 : 64);
  if (!oka || !okb) return cudaErrorInvalidValue;
  fill_unused(maps, 1, 1);
  if (pair) {
    // 256 x 256 units on CTA pairs (N % 256 == 0)
    if (!a_mn && !b_mn) return run_gemm<256, false, false, false, 6, EpiStoreF32, 1, true>(maps, sh, ep, M, s, "dense_gemm");
    if (!a_mn && b_mn) return run_gemm<256, false, true, false, 6, EpiStoreF32, 1, true>(maps, sh, ep, M, s, "dense_gemm");
    if (a_mn && !b_mn) return run_gemm<256, true, false, false, 6, EpiStoreF32, 1, true>(maps, sh, ep, M, s, "dense_gemm");
    return run_gemm<256, true, true, false, 6, EpiStoreF32, 1, true>(maps, sh, ep, M, s, "dense_gemm");
  }
  if (!a_mn && !b_mn) return run_gemm<64, false, false, false, 8, EpiStoreF32>(maps, sh, ep, M, s, "dense_gemm");
  if (!a_mn && b_mn) return run_gemm<64, false, true, false, 8, EpiStoreF32>(maps, sh, ep, M, s, "dense_gemm");
  if (a_mn && !b_mn) return run_gemm<64, true, false, false, 8, EpiStoreF32>(maps, sh, ep, M, s, "dense_gemm");
  return run_gemm<64, true, true, false, 8, EpiStoreF32>(maps, sh, ep, M, s, "dense_gemm");
}

}  // namespace tw

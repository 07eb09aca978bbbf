// Host-side interfaces between the C-ABI layer (tw_api.cu) and the kernel
// launchers (tw_kernels.cu, tw_gemm.cu). Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/twell.h"

namespace tw {

int device_sm_count();

// Every host-side argument check of twell_ffn_fwd except the workspace size
// (tw_api.cu), shared with the fixed-scratch entry point.
tw_status check_twell_fwd_operands(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd,
                                   int T, int d, int I, int W, int C, int ovf_cap, const tw_twell* tw_out,
                                   uint16_t* y, int32_t* dev_status);

// Timing trace (tw_trace_begin): records the next caller event on `s` after a launch.
void trace_begin(void* const* events, int capacity);
int trace_end();
const char* trace_label(int i);
void trace_mark(cudaStream_t s, const char* label);

// Zeroes [p0, p0 + b0) and [p1, p1 + b1) (16-byte aligned starts, any sizes; p1 may
// be null) with one kernel, followed by a trace mark.
cudaError_t launch_zero(void* p0, size_t b0, void* p1, size_t b1, cudaStream_t s);
// bf16 -> fp16 conversion of up to four tensors of n[k] elements (multiples of 8),
// only when *route == 1 (route may be null): the dense route backward's operands.
cudaError_t launch_to_f16(const uint16_t* const* src, uint16_t* const* dst, const size_t* n, int count,
                          const int32_t* route, cudaStream_t s);
// fp32 FMA throughput probe (tw_kernels.cu): blocks x 256 threads, `iters` steps;
// out holds blocks * 256 floats
cudaError_t launch_fma_probe(float* out, int blocks, int iters, cudaStream_t s);
long fma_probe_flops(int blocks, int iters);
// L2 row-gather probe (tw_kernels.cu): `blocks` CTAs of d / 8 threads gather the
// rows idx[0 .. n_idx) of table [rows, d] (n_idx % 8 == 0); out holds blocks * d / 8
// floats. l2_gather_probe_blocks(d) is the grid the bench uses (the token kernels'
// residency).
cudaError_t launch_l2_gather_probe(const uint16_t* table, int rows, int d, const int32_t* idx, int n_idx, float* out,
                                   int blocks, cudaStream_t s);
int l2_gather_probe_blocks(int d);

// Every library kernel is launched with programmatic stream serialization: it may
// start (and run its prologue) while the kernel before it on the stream finishes,
// and it calls pdl_wait() (griddepcontrol.wait) before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// The same launch as clusters of `cluster` CTAs along x (gridDim.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_clustered(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster, cudaStream_t s,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = static_cast<unsigned>(cluster);
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// How many clusters of `cluster` CTAs of `kern` (block threads, smem bytes) can be
// resident at once on this device; 0 when the query fails.
template <typename... KArgs>
int max_active_clusters(void (*kern)(KArgs...), int block, size_t smem, int cluster) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
  return n;
}

// ---------------------------------------------------------------- tw_kernels.cu
// Dense bf16 [T, I] -> TwELL counts/slots/row_nnz/ovf (not the overflow list).
cudaError_t launch_pack_dense(const uint16_t* A, int T, int I, int W, int C, const tw_twell& o, cudaStream_t s);

// Ascending list of rows whose flag holds. flag(t) = ovf[t] != 0, or, when
// row_nnz != nullptr, ovf[t] != 0 || row_nnz[t] > R. Writes list[0..min(n, list_cap)),
// *count = n, slot_of[t] (rank, -1 when unflagged, -2 when past list_cap) and
// ell_nnz[t] (row_nnz when unflagged, else 0) when those pointers are non-null.
// Raises TW_ECAPACITY when n > cap_check.
// zero_word (optional) is set to 0 by the kernel, for a scheduling counter used later
// in the stream.
// Route decision (when route_out != nullptr): *route_out = 1 (dense) when route_mode
// is TW_ROUTE_DENSE, or TW_ROUTE_AUTO and the unflagged rows' mean row_nnz exceeds
// dense_above; else 0.
cudaError_t launch_compact_rows(const uint8_t* ovf, const int32_t* row_nnz, int R, int T, int32_t* list,
                                int list_cap, int32_t* count, int32_t* slot_of, int32_t* ell_nnz, int cap_check,
                                int32_t* status, cudaStream_t s, int32_t* zero_word = nullptr,
                                int route_mode = TW_ROUTE_SPARSE, float dense_above = 0.f, int32_t* route_out = nullptr);

// ---------------------------------------------------------------- tw_formats.cu
// TwELL slots scattered into a dense bf16 [T, I] matrix (zeros elsewhere).
cudaError_t launch_twell_unpack(const tw_twell& tw, uint16_t* A, cudaStream_t s);
// Hybrid of a dense bf16 A (and U) with tile width W and capacity C for the overflow
// test: every field of h; ovf_ws holds T bytes of per-row overflow flags.
cudaError_t launch_hybrid_pack(const uint16_t* A, const uint16_t* U, int T, int I, int W, int C, const tw_hybrid& h,
                               uint8_t* ovf_ws, int32_t* status, cudaStream_t s);
// Dense fp32 A [T, I] (and U when non-null) from a Hybrid.
cudaError_t launch_hybrid_unpack(const tw_hybrid& h, float* A, float* U, cudaStream_t s);
// Dense route, non-gated forward (only when *route == 1): H [T, I] fp16 = the TwELL's
// activations on rows without a backup slot, and those rows' ELL entries (idx, a)
// written at their ELL offsets; backup rows get fp16 of their saved fp32 a (backup_a
// [cap, I], written by the backup's GEMM before this launch), rows past the capacity 0.
cudaError_t launch_twell_to_dense_ell(const tw_twell& tw, const int32_t* backup_slot, const float* backup_a, int cap,
                                      int R, uint16_t* H, uint16_t* ell_idx, uint16_t* ell_a, const int32_t* route,
                                      int32_t* status, cudaStream_t s);
// The ELL entries (idx, a) of the rows without a backup slot from the TwELL, for the
// sparse route's forward (nothing when *route == 1; route may be null).
cudaError_t launch_twell_to_ell(const tw_twell& tw, const int32_t* backup_slot, int R, uint16_t* ell_idx,
                                uint16_t* ell_a, const int32_t* route, int32_t* status, cudaStream_t s);

// ---------------------------------------------------------------- tw_neurons.cu
cudaError_t launch_neuron_counts(const tw_hybrid& h, int32_t* counts, cudaStream_t s);
cudaError_t launch_reinit_rows(uint16_t* W, int I, int d, const int32_t* counts, uint64_t seed, float stdv,
                               int32_t* n_reinit, cudaStream_t s);

// out[i] = src[rows[i]] for i < min(*n, cap) (src holds src_rows rows, and so does
// src2); rows [n, round_up(n, 128)) (below
// rows_alloc) are zero-filled. Row length d bf16. With src2/out2 the same rows of a
// second matrix are gathered in the same launch; with `zero`, rows [0, min(*n, cap))
// of that fp32 accumulator (zero_row_f32 floats a row, a multiple of 4) are set to 0
// for the split-K product that adds into them next (with zero_if_sparse, only when
// that route word does not read 1: the accumulator serves only the sparse route).
// Raises TW_ECAPACITY into `status` (when non-null) if *n > cap.
cudaError_t launch_gather_rows(const uint16_t* src, int d, int src_rows, const int32_t* rows, const int32_t* n, int cap,
                               int rows_alloc, uint16_t* out, cudaStream_t s, int32_t* status = nullptr,
                               const uint16_t* src2 = nullptr, uint16_t* out2 = nullptr, float* zero = nullptr,
                               int zero_row_f32 = 0, const int32_t* sparse_only = nullptr,
                               const int32_t* zero_if_sparse = nullptr);

// Largest per-token entry list of the sparse forward, (I / W) * C: two lists of
// 10 bytes an entry live in one CTA's shared memory.
constexpr int kMaxList = 10240;

struct SparseFwdArgs {
  const uint16_t *x, *Wu, *Wd;
  int T, d, I, W, C, nT;
  const uint16_t* cnt;
  const uint16_t* val;
  const uint8_t* idx;
  const uint8_t* ovf;             // TwELL mode: skip rows with ovf
  const int32_t* backup_slot;     // Hybrid mode: skip rows with slot != -1
  const int32_t* ell_nnz;         // Hybrid mode, gated: the ELL rows' lengths (their idx and a
                                  // written by launch_twell_to_dense_ell beforehand)
  uint16_t* ell_idx;              // Hybrid mode outputs (R slots per row)
  uint16_t* ell_a;
  uint16_t* ell_u;
  int R;
  int L;                          // per-token entry list capacity: nT * C (<= kMaxList)
  uint16_t* y;
  int32_t* status;                // device status word (TW_ETIMEOUT from a bounded wait)
  // token scheduling counter (device int): CTAs take their first token by index and
  // the rest from this counter; nullptr = static round-robin. It must read 0 when the
  // kernel starts: the launcher zeroes it unless sched_zeroed says an earlier kernel
  // in the stream did.
  int32_t* sched;
  bool sched_zeroed;
  const int32_t* route;  // optional: the kernel does nothing when *route == 1 (the dense route)
};
// TwELL / Hybrid forward of the non-dense rows (tw_token.cu)
cudaError_t launch_token_fwd(const SparseFwdArgs& a, cudaStream_t s);

struct SparseBwdArgs {
  const uint16_t *dy, *x, *Wg, *Wu, *Wd;
  int T, d, I, R;
  float l1;
  const int32_t* ell_nnz;
  const int32_t* backup_slot;
  const uint16_t* ell_idx;
  const uint16_t* ell_a;
  const uint16_t* ell_u;
  uint16_t* dx;
  // transposed Hybrid (workspace)
  int32_t* col_cnt;   // [I + 1]
  int32_t* col_ptr;   // [I + 1]
  int32_t* col_cur;   // [I]
  uint4* csc;         // [csc_cap] column-ordered entry records
  long long csc_cap;  // T * R
  int32_t* status;    // device status word (TW_EBOUNDS in bounds-checked builds)
  float *dWg, *dWu, *dWd;
  // when non-null and *dW_base_rows > 0, dW already holds the dense backup rows'
  // part and the ELL part is added to it; otherwise dW is overwritten
  const int32_t* dW_base_rows;
  // scheduling counters (as SparseFwdArgs::sched): the token pass's at sched[0], the
  // weight pass's kSchedCounters at sched_w = sched + kSchedStride, each
  // kSchedStride ints apart, and the count pass's ticket at sched + kSchedTicket;
  // the kSchedWords ints are zeroed together with col_cnt
  int32_t* sched;
  int32_t* sched_w;
  const int32_t* route;  // optional: the kernels do nothing when *route == 1 (the dense route)
};
constexpr int kSchedCounters = 8;
constexpr int kSchedStride = 32;  // ints: one 128-byte line per counter
constexpr int kSchedTicket = (1 + kSchedCounters) * kSchedStride;
constexpr int kSchedWords = (2 + kSchedCounters) * kSchedStride;
// Token side of the ELL backward (tw_token.cu): dh, dg and du per entry, each
// entry's record of the transposed Hybrid written at a slot claimed from col_cur
// (set by the count pass), dx.
cudaError_t launch_token_bwd(const SparseBwdArgs& a, cudaStream_t s);
// ELL backward (tw_sparse.cu), token side: zeroes the counters, counts and scans the
// columns of the transposed Hybrid, then launch_token_bwd fills in its records.
cudaError_t launch_sparse_bwd_tokens(const SparseBwdArgs& a, cudaStream_t s);
// ELL backward, column side: weight gradients over the transposed Hybrid (see
// SparseBwdArgs::dW_base_rows for overwrite / accumulate).
cudaError_t launch_sparse_bwd_weights(const SparseBwdArgs& a, cudaStream_t s);

// ---------------------------------------------------------------- tw_gemm.cu
// 2D tensor map of 16-bit elements with the 128-byte swizzle (operand loads), or the
// 64-byte swizzle (swizzle64: the 32 x 32 output boxes of bulk stores).
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                    uint32_t box_inner, uint32_t box_outer, bool swizzle64 = false);

// gate projection + ReLU + TwELL pack
cudaError_t gemm_gate_pack(const uint16_t* x, const uint16_t* Wg, int T, int d, int I, int W, int C,
                           const tw_twell& o, uint16_t* a_dense, int32_t* status, cudaStream_t s);

// unfused gate: a = bf16(ReLU(x Wg^T)) written densely [T, I]
cudaError_t gemm_gate_relu_dense(const uint16_t* x, const uint16_t* Wg, int T, int d, int I, uint16_t* a,
                                 int32_t* status, cudaStream_t s);

// Backup capacities up to this many rows take the split-K forms of the dense backup's
// hidden and grad products (gemm_backup_hidden / gemm_backup_grad with split_acc):
// their fp32 accumulators hold (gated) 2 I or I floats a row, zeroed by the row gather.
constexpr int kBackupSplitRows = 512;

// dense backup forward: h(X Wg^T, X Wu^T) over n (device) rows of X [rows_alloc, d],
// written as the bf16 pair H + H_lo; optional saved fp32 a / u. With a route word
// that reads 1 (the dense route) only a and u are written. With split_acc (rows of
// stride split_ld holding g in columns [0, I) and, gated, u in [I, 2 I), rows
// [0, n) zeroed beforehand) the products run split-K and a finishing kernel follows;
// without it but with the saved rows, a and u are stored by a grouped launch on
// full-width tiles (u only when the route word does not read 1: the dense route's
// up GEMM saves it) and H / H_lo formed from them by the finishing kernel.
cudaError_t gemm_backup_hidden(const uint16_t* X, const uint16_t* Wg, const uint16_t* Wu, int rows_alloc,
                               const int32_t* n_dev, int cap, int d, int I, uint16_t* H, uint16_t* H_lo,
                               float* save_a, float* save_u, int32_t* status, cudaStream_t s,
                               const int32_t* route = nullptr, float* split_acc = nullptr, int split_ld = 0);

// The same product spread over every SM with split K: partial sums are added into
// the fp32 accumulator acc [cap, N], which must hold zeros (launch_gather_rows zeroes
// it alongside the row gather); launch_scatter_rows_bf16 writes the finished rows.
cudaError_t gemm_rows_times_nmajor_splitk(const uint16_t* const* A, const uint16_t* const* B, int segments,
                                          int rows_alloc, const int32_t* n_dev, int cap, int K, int N, float* acc,
                                          int32_t* status, cudaStream_t s, const int32_t* sparse_only = nullptr,
                                          int ld_acc = 0);
// sparse_only (optional, here and below): the launch does its work only when
// *sparse_only != 1, i.e. when the call took the sparse route (the dense route's
// backward folds the backup rows into its own GEMMs).
cudaError_t launch_scatter_rows_bf16(const float* acc, int N, const int32_t* n_dev, int cap, const int32_t* row_map,
                                     uint16_t* out, int ldo, int out_rows, cudaStream_t s,
                                     const int32_t* sparse_only = nullptr, int ld_acc = 0);

// dense backup backward part 1: dh = dY Wd^T and the epilogue producing dG, dU and H,
// each as a (hi, lo) bf16 pair [rows_alloc, I].
struct BackupGradOut {
  uint16_t *dG, *dG_lo, *dU, *dU_lo, *H, *H_lo;
};
// With split_acc (rows of stride split_ld, columns [0, I) zeroed beforehand on rows
// [0, n)) the product runs split-K and a finishing kernel follows.
cudaError_t gemm_backup_grad(const uint16_t* dY, const uint16_t* Wd, int rows_alloc, const int32_t* n_dev, int cap,
                             int d, int I, const float* a, const float* u, float l1, const BackupGradOut& o,
                             int32_t* status, cudaStream_t s, const int32_t* sparse_only = nullptr,
                             float* split_acc = nullptr, int split_ld = 0);
// The finishing kernels of the split-K forms (tw_kernels.cu): the arithmetic of the
// direct forms' epilogues (EpiBackupHidden, EpiBackupGrad) on the accumulated rows.
// from_saved: acc is save_a, whose rows already hold a = ReLU(g), and u comes from
// save_u; only H / H_lo are written (nothing when the route word reads 1).
cudaError_t launch_backup_hidden_finish(const float* acc, int ld, const int32_t* n_dev, int cap, int I, bool gated,
                                        uint16_t* H, uint16_t* H_lo, int rows_alloc, float* save_a, float* save_u,
                                        const int32_t* route, cudaStream_t s, bool from_saved);
cudaError_t launch_backup_grad_finish(const float* acc, int ld, const int32_t* n_dev, int cap, int I, const float* a,
                                      const float* u, float l1, const BackupGradOut& o, int rows_alloc,
                                      const int32_t* sparse_only, cudaStream_t s);
// The dense backup rows' weight gradients, D_p = (P_hi,p + P_lo,p)^T Q_p for up to
// three problems in one launch (P [rows, I] bf16 hi/lo pairs, Q [rows, d] bf16, K =
// the device row count), written (overwritten) as fp32 [I, d]; nothing is written
// when the row count is 0. Requires d % 256 == 0.
struct WeightGradProblem {
  const uint16_t* P_hi;
  const uint16_t* P_lo;
  const uint16_t* Q;
  float* D;
};
cudaError_t gemm_weight_grads(const WeightGradProblem* probs, int n_probs, int rows_alloc, const int32_t* n_dev,
                              int cap, int I, int d, int32_t* status, cudaStream_t s,
                              const int32_t* sparse_only = nullptr);

// withhold_kb >= 0: the test hook of GemmShape::withhold_kb (a bounded wait runs out)
// ---------------------------------------------------------------- dense route (tw_gemm.cu)
// Every launch below does its work only when *route == 1 (route may be null: always).
// Gated forward: u = x Wu^T over all T rows, with h = a u at the TwELL's active columns
// written densely into H [T, I] fp16 and the Hybrid's ELL rows (idx, a, fp16 u) of
// the rows without a backup slot; backup rows get H = fp16(a u) from their saved fp32
// a (backup_a [cap, I], written by the backup's GEMM before this launch) and their u
// saved into backup_u (unless null), rows past the capacity H = 0.
cudaError_t gemm_up_hybrid(const uint16_t* x, const uint16_t* Wu, int T, int d, int I, const tw_twell& tw, int R,
                           const int32_t* backup_slot, const float* backup_a, float* backup_u, int cap, uint16_t* H,
                           uint16_t* ell_idx, uint16_t* ell_a, uint16_t* ell_u, const int32_t* route,
                           int32_t* status, cudaStream_t s);
// out [M, N] bf16 (row stride ld) = sum over segments of A_s [M, K] (K-major) B_s [K, N]
// (N contiguous); operands bf16, or fp16 when f16.
cudaError_t gemm_rows_nmajor_bf16(const uint16_t* const* A, const uint16_t* const* B, int segments, int M, int K,
                                  int N, uint16_t* out, int ld, const int32_t* route, int32_t* status, cudaStream_t s,
                                  bool f16, const char* label);
// Backward: dh = dY Wd^T over all T rows; dG, dU (gated) and H [T, I] fp16 from the
// saved Hybrid's ELL rows and fp32 backup rows (zeros off the support and on rows
// past the backup capacity).
cudaError_t gemm_dense_grad(const uint16_t* dY, const uint16_t* Wd, int T, int d, int I, const tw_hybrid& h,
                            bool gated, float l1, uint16_t* dG, uint16_t* dU, uint16_t* H, const int32_t* route,
                            int32_t* status, cudaStream_t s);
// D_p = P_p^T Q_p (P [T, I] fp16, Q [T, d] fp16, K = T) for up to three problems,
// written as fp32 [I, d], or added when *add_if > 0 (the dense backup's part is there).
struct DenseWeightGradProblem {
  const uint16_t* P;
  const uint16_t* Q;
  float* D;
};
cudaError_t gemm_dense_weight_grads(const DenseWeightGradProblem* probs, int n_probs, int T, int I, int d,
                                    const int32_t* add_if, const int32_t* route, int32_t* status, cudaStream_t s);

// The layout-test GEMM (fp32 D = A B); pair runs it on CTA pairs (N % 256 == 0).
cudaError_t gemm_dense_test(const uint16_t* A, const uint16_t* B, int M, int N, int K, int a_mn, int b_mn, float* D,
                            int32_t* status, cudaStream_t s, int withhold_kb = -1, bool pair = false);

}  // namespace tw

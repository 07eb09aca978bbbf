/*
 * twell.h -- C ABI of the activation-sparse ReLU feedforward library (sm_103a).
 *
 * The operation (gist.science explainer "Sparser, Faster, Lighter Transformer
 * Language Models", section 2.B "Kernel Design"; Table 2 of the thelatestinai
 * listing for the two forms):
 *
 *   gated:      a = ReLU(x Wg^T),  u = x Wu^T,  h = a * u,  y = h Wd
 *   non-gated:  a = ReLU(x W1^T),                h = a,      y = h W2
 *
 * computed through the TwELL format (inference) and the Hybrid format (training),
 * with an L1 penalty l1 * sum(a) on the hidden activations in training
 * (explainer 2.C "Training Recipe").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers, row-major, densely packed. bf16 values
 *   are passed as their 16-bit patterns (uint16_t). x, y, dy, dx are [T, d].
 *   Every weight is [I, d]: row j of Wg (W1) and Wu is neuron j's input weight
 *   vector; row j of Wd (W2) is the vector neuron j adds to y. Wu == NULL selects
 *   the non-gated form.
 * - Shapes: T >= 0 tokens; d % 256 == 0 and 256 <= d <= 2048 (the sparse kernels
 *   give each warp of a token's CTA one 256-wide slice of d); W in {64, 128};
 *   I % W == 0, 64 <= I <= 65536; 1 <= C <= W; (I / W) * C <= 10240 (a token's
 *   entry list lives in shared memory); 1 <= R <= I; 0 <= backup_cap <= T.
 *   T == 0 is valid: the forwards and packers do nothing, and hybrid_ffn_bwd
 *   writes dW = 0 (sums over no tokens). Other shapes return TW_EUNSUPPORTED.
 * - Alignment: every pointer must be 16-byte aligned (TMA and 128-bit accesses).
 * - Ownership: the caller allocates and frees every buffer, including the
 *   workspace whose size the *_workspace_size() functions return. The library
 *   never allocates, frees or synchronises; it only enqueues kernels on `stream`,
 *   a cudaStream_t passed as void* (NULL = the legacy default stream).
 * - Workspaces need no initial contents: every call zeroes, on its stream, what it
 *   reads before writing (list counters, column counts, split-K accumulators, the
 *   counters from which the sparse kernels take their tokens).
 * - Determinism: TwELL and Hybrid contents, the ELL rows' y and dx, and every count
 *   are the same on every run. The weight gradients and the dense rows' y and dx
 *   (overflow / backup rows) are fp32 sums whose order depends on the order of
 *   atomic updates, so they can differ in the last bits from run to run.
 * - Errors found on the host (bad shape, NULL or misaligned pointer, workspace too
 *   small) are returned synchronously before anything is enqueued. Launch errors
 *   return TW_ECUDA. Conditions only the GPU can see (a capacity exceeded, a
 *   bounded wait that timed out) are written to *dev_status, a device int32 the
 *   caller zeroes beforehand and reads after synchronising: kernels only raise it
 *   (atomicMax of the tw_status code), never clear it.
 * - Calls on one stream are ordered; calls on different streams must not share a
 *   workspace or output.
 */
#ifndef TWELL_H
#define TWELL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TW_OK = 0,
  TW_EINVAL = 1,        /* bad shape / NULL pointer / bad parameter */
  TW_EALIGN = 2,        /* pointer not 16-byte aligned */
  TW_EUNSUPPORTED = 3,  /* shape outside what the kernels implement */
  TW_ECAPACITY = 4,     /* device: more overflow/backup rows than the buffers hold */
  TW_ETIMEOUT = 5,      /* device: a bounded pipeline wait gave up */
  TW_ECUDA = 6,         /* a CUDA runtime call or launch failed */
  TW_EWORKSPACE = 7,    /* workspace smaller than *_workspace_size() */
  TW_EBOUNDS = 8        /* device, bounds-checked builds only (-DTW_CHECK): an index
                           computed from the inputs or workspaces did not fit its
                           buffer; the access was skipped */
} tw_status;

/* TwELL (tile-wise ELLPACK) of a [T, I] activation matrix with tile width W and
 * capacity C (explainer 2.A "New Sparse Data Format: TwELL"; wispaper blog,
 * "1. TwELL: Tile-wise ELLPACK"). nT = I / W tiles per row.
 *   cnt[t*nT + k]           true (uncapped) number of nonzeros of row t in tile k
 *   val[(t*nT + k)*C + s]   bf16 value of the s-th nonzero (ascending column), s < min(cnt, C)
 *   idx[(t*nT + k)*C + s]   its column inside the tile, 0 <= idx < W
 *   row_nnz[t]              sum over k of cnt
 *   ovf[t]                  1 if some cnt > C (the row is served by the dense path)
 *   ovf_rows[0 .. *n_ovf)   the rows with ovf == 1, ascending (array holds T entries)
 * Slots s >= min(cnt, C) are left unspecified. A value is nonzero when its bf16
 * magnitude bits are nonzero (-0.0 is zero). All arrays are caller-allocated. */
typedef struct {
  int32_t T, I, W, C;
  uint16_t* cnt;
  uint16_t* val;
  uint8_t* idx;
  int32_t* row_nnz;
  uint8_t* ovf;
  int32_t* ovf_rows;
  int32_t* n_ovf;
} tw_twell;

/* Hybrid format saved by the training forward (explainer 2.A "Hybrid Format for
 * Training"; wispaper blog, "2. The Hybrid Training Algorithm"). Row t goes to the
 * dense backup when its TwELL overflowed or row_nnz[t] > R, else to the ELL.
 *   row_nnz[t]                      active neurons of row t
 *   ell_nnz[t]                      entries stored in the ELL (0 for backup rows)
 *   ell_idx[t*R + s]                global neuron index, ascending in s
 *   ell_a[t*R + s]                  bf16 a at that neuron (the TwELL's value)
 *   ell_u[t*R + s]                  u at that neuron as fp16 bits (IEEE binary16: 11
 *                                   significant bits where bf16 has 8, for the weight
 *                                   gradients' long sums; |u| must stay below 65504,
 *                                   which the backup rows' fp32 storage covers for the
 *                                   largest activations); unused when non-gated
 *   backup_slot[t]                  slot of row t in the backup, or -1
 *   backup_tok[b]                   token of backup slot b, ascending in b
 *   backup_a[b*I + j], backup_u[b*I + j]   full fp32 rows of a = ReLU(g) and u (the
 *                                   backup rows carry the largest activations, so
 *                                   they are kept at full precision)
 *   n_backup[0]                     number of backup rows (may exceed backup_cap:
 *                                   then only backup_cap rows are written and
 *                                   TW_ECAPACITY is raised in *dev_status)
 * ell_* slots s >= ell_nnz[t] are unspecified. */
typedef struct {
  int32_t T, I, R, backup_cap;
  int32_t* row_nnz;
  int32_t* ell_nnz;
  uint16_t* ell_idx;
  uint16_t* ell_a;
  uint16_t* ell_u;
  int32_t* backup_slot;
  int32_t* backup_tok;
  float* backup_a;
  float* backup_u;
  int32_t* n_backup;
  int32_t route;          /* how the ELL rows' projections run: TW_ROUTE_* below */
  float dense_above;      /* TW_ROUTE_AUTO: the dense route when the mean over all rows
                             of (ELL row: its nonzeros; backup row: 2 dense_above)
                             exceeds this */
  int32_t* route_taken;   /* device int32: the forward writes the route it took (0 sparse,
                             1 dense); the backward takes the same one. May be NULL only
                             with TW_ROUTE_SPARSE */
} tw_hybrid;

/* Routes of a Hybrid layer's projections. The backup rows' fp32 a and u always come
 * from a dense tensor-core GEMM.
 *  TW_ROUTE_SPARSE  the pages' method: CUDA-core gathers over the active neurons of
 *                   the ELL rows (explainer 2.B "Training Kernels",
 *                   "Backpropagation"); the backup rows' y, dx and dW from dense GEMMs
 *                   on split fp32 (hi + lo bf16) operands;
 *  TW_ROUTE_DENSE   every row's up / down projections and their backward as dense
 *                   tensor-core GEMMs over all neurons, with the TwELL / Hybrid masks
 *                   applied in the GEMM epilogues (the backup rows' h, dg, du from
 *                   their saved fp32 a and u): the forward's up GEMM on the bf16
 *                   inputs, its down GEMM and the backward's dx and dW on fp16
 *                   operands (h, dg, du rounded once to fp16; fp16 copies of Wd, Wg,
 *                   Wu, x, dy, whose magnitudes must stay below 65504); the saved
 *                   Hybrid is the same;
 *  TW_ROUTE_AUTO    decided on the device by each forward, after the gate kernel: dense
 *                   when the sparse route's work per row, in ELL entries, exceeds
 *                   dense_above on average, counting an ELL row's nonzeros and
 *                   2 dense_above for a backup row (whose split-operand GEMMs cost
 *                   about twice the dense route's work per row). A row's gathers cost
 *                   L2 traffic in proportion to its nonzeros, the dense GEMMs a fixed
 *                   amount, so above some activity the dense route is faster; the
 *                   tunx.ai page has the dense backup take the rows that activity
 *                   makes expensive, and this extends that choice to a whole call. */
#define TW_ROUTE_SPARSE 0
#define TW_ROUTE_DENSE 1
#define TW_ROUTE_AUTO 2

/* Human-readable name of a tw_status code. */
const char* tw_status_str(int status);

/* ABI version of this header (bumped on any incompatible change). */
int tw_abi_version(void);

/* Pack a dense bf16 [T, I] matrix A into TwELL (all fields of *out, including
 * row_nnz, ovf, ovf_rows and n_ovf). Bit-exact: the result depends only on A.
 * Defines the format of explainer 2.A; used standalone and as a test hook. */
tw_status twell_pack(const uint16_t* A, int T, int I, int W, int C,
                     const tw_twell* out, int32_t* dev_status, void* stream);

/* TwELL unpack (explainer 2.A "New Sparse Data Format: TwELL"; wispaper blog,
 * "1. TwELL: Tile-wise ELLPACK"): A [in->T, in->I] bf16 (device, caller-owned) is
 * overwritten with zeros and every stored slot s < min(cnt, C) of tile k of row t is
 * written at column k W + idx. On a row without overflow this gives back exactly the
 * packed row; on an overflow row only its first C nonzeros of each tile. Slot indices
 * >= W are skipped. Reads cnt, val and idx only. Enqueued on `stream`. */
tw_status twell_unpack(const tw_twell* in, uint16_t* A, void* stream);

/* Workspace bytes hybrid_pack needs (one byte a row). */
size_t hybrid_pack_workspace_size(int T);

/* Hybrid pack of a given dense bf16 activation matrix A [T, I] and, in the gated
 * form, the up-projection U [T, I] (NULL: non-gated, ell_u / backup_u unused)
 * (explainer 2.A "Hybrid Format for Training"; wispaper blog, "2. The Hybrid
 * Training Algorithm"). Fills every field of *out exactly as the training forward
 * does from its own a and u: row_nnz = nonzeros of row t (bf16 magnitude bits
 * nonzero); the row goes to the dense backup when some W-column tile of it holds
 * more than C nonzeros (its TwELL overflows) or row_nnz > out->R; backup slots are
 * given by ascending row (backup_tok, backup_slot, n_backup; more than
 * out->backup_cap backup rows raise TW_ECAPACITY in *dev_status, the extra rows get
 * slot -2 and are not stored); ELL rows store their nonzeros in ascending column
 * order (ell_idx, ell_a, ell_u as fp16 of U's values; ell_nnz = row_nnz, 0 for backup
 * rows); backup rows
 * store the full rows of A and U widened exactly to fp32. Shapes as twell_pack; ws
 * holds hybrid_pack_workspace_size(T) bytes. Enqueued on `stream`. */
tw_status hybrid_pack(const uint16_t* A, const uint16_t* U, int T, int I, int W, int C,
                      const tw_hybrid* out, void* ws, size_t ws_bytes, int32_t* dev_status,
                      void* stream);

/* Hybrid unpack (explainer 2.A "Hybrid Format for Training"): dense fp32 A [T, I]
 * and, when U != NULL (gated Hybrid), U [T, I] (device, caller-owned). A row with a
 * backup slot is its backup row; an ELL row is zeros with its ell_nnz entries written
 * at their columns (bf16 widened exactly); a row past the backup capacity (slot -2)
 * is zeros. Unpacking a hybrid_pack result gives A back on every row and U on the
 * support of ELL rows and on all of backup rows. I % 64 == 0, 64 <= I <= 65536.
 * Enqueued on `stream`. */
tw_status hybrid_unpack(const tw_hybrid* in, float* A, float* U, void* stream);

/* Gate projection with the TwELL pack fused into its epilogue (explainer 2.B
 * "Inference Kernels", "Gate Projection"): a = bf16(ReLU(x Wg^T)) with fp32
 * accumulation on the tensor cores, written straight into *out; the dense [T, I]
 * activation is never stored unless a_dense != NULL (a [T, I] bf16 buffer that
 * receives it, for verification only). Fills every field of *out. */
tw_status twell_gate_pack(const uint16_t* x, const uint16_t* Wg, int T, int d, int I,
                          int W, int C, const tw_twell* out, uint16_t* a_dense,
                          int32_t* dev_status, void* stream);

/* Workspace bytes twell_ffn_fwd needs for up to ovf_cap overflow rows. */
size_t twell_ffn_fwd_workspace_size(int T, int d, int I, int W, int C, int ovf_cap);

/* Inference forward through TwELL (explainer 2.B "Inference Kernels"): the fused
 * gate+pack kernel, then one kernel that, for every stored entry (t, j) of a
 * non-overflow row, takes the dot product u = x_t . Wu[j] and adds (a*u) * Wd[j]
 * to y_t (never materialising the dense hidden state), and the dense tensor-core
 * path for overflow rows (at most ovf_cap of them; more raise TW_ECAPACITY and
 * leave the extra rows of y unwritten). y is [T, d] bf16 (fp32 accumulation, one
 * rounding). *tw receives the TwELL of a as a by-product. */
tw_status twell_ffn_fwd(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu,
                        const uint16_t* Wd, int T, int d, int I, int W, int C,
                        int ovf_cap, const tw_twell* tw, void* ws, size_t ws_bytes,
                        uint16_t* y, int32_t* dev_status, void* stream);

/* twell_ffn_fwd for callers that cannot allocate device memory (the pages have no
 * counterpart of this call). Some callers own only their inputs and outputs: a
 * plugin that a host framework hands I/O pointers but no workspace, or a serving
 * loop where cudaMalloc is off limits because it can synchronise the device and
 * stall for milliseconds. This call computes exactly what twell_ffn_fwd computes,
 * with the same arguments minus the workspace: the overflow path's scratch comes
 * from one fixed 20 MiB array in device memory that the library defines.
 *  - Limit: returns TW_EWORKSPACE (before enqueuing anything) when
 *    twell_ffn_fwd_workspace_size(T, d, I, W, C, ovf_cap) exceeds 20 MiB; at
 *    d = 2048, I = 5632 that allows ovf_cap up to 512 overflow rows.
 *  - The array occupies 20 MiB on every GPU where the library's code is loaded,
 *    until the process exits.
 *  - The first call on each device looks up the array's device address (with that
 *    device current); make that first call before any stream capture. The address
 *    is kept for the life of the process, so every call on that device must run in
 *    the same context as the first one (the runtime's primary context), and the
 *    device must not be reset (cudaDeviceReset) between calls.
 *  - Arguments are checked as twell_ffn_fwd checks them (same error codes); only
 *    then is the size compared with the array.
 *  - All calls share the one array and it keeps the previous call's contents;
 *    nothing in it needs to start at zero. Calls whose GPU work overlaps (on
 *    unordered streams) race on it: order them on one stream.
 *  - Allocates and frees nothing. */
tw_status twell_ffn_fwd_fixed_scratch(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu,
                                      const uint16_t* Wd, int T, int d, int I, int W, int C,
                                      int ovf_cap, const tw_twell* tw, uint16_t* y,
                                      int32_t* dev_status, void* stream);

/* Workspace bytes hybrid_ffn_fwd needs for a Hybrid with the given route (any route
 * other than TW_ROUTE_SPARSE adds the dense route's [T, I] fp16 hidden matrix and an
 * fp16 copy of Wd). */
size_t hybrid_ffn_fwd_workspace_size(int T, int d, int I, int W, int C, int R, int backup_cap, int route);

/* Training forward (explainer 2.B "Training Kernels"): gate+pack into TwELL,
 * conversion of TwELL into the Hybrid *saved (sizes taken from saved->R and
 * saved->backup_cap), the backup rows' fp32 a and u on the tensor cores, u on the
 * support of ELL rows; y from the ELL rows on the CUDA cores and from the backup
 * rows on the tensor cores, or, when the call takes the dense route, from one
 * tensor-core GEMM over all rows. *saved holds what the backward needs. */
tw_status hybrid_ffn_fwd(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu,
                         const uint16_t* Wd, int T, int d, int I, int W, int C,
                         const tw_hybrid* saved, void* ws, size_t ws_bytes,
                         uint16_t* y, int32_t* dev_status, void* stream);

/* Workspace bytes hybrid_ffn_bwd needs (routes other than TW_ROUTE_SPARSE add the
 * dense route's [T, I] fp16 dG, dU and h and fp16 copies of Wg, Wu, x and dy). */
size_t hybrid_ffn_bwd_workspace_size(int T, int d, int I, int R, int backup_cap, int route);

/* Training backward over the saved Hybrid (explainer 2.B "Backpropagation"):
 * gradient of L = sum(dy * y) + l1 * sum(a):
 *   dh = dy Wd^T on the support;  du = dh * a;  dg = (dh * u + l1) on the support
 *   (non-gated: dg = dh + l1);  dx = dg Wg + du Wu  (bf16 [T, d]);
 *   dWg = dg^T x, dWu = du^T x, dWd = h^T dy  (fp32 [I, d], overwritten).
 * The sparse route runs the ELL part on the CUDA cores with the weight gradients
 * accumulated over the transposed Hybrid and the backup rows as tensor-core GEMMs;
 * the dense route (the one the forward took) runs all rows as tensor-core GEMMs.
 * dWu is ignored when
 * Wu == NULL. TW_EUNSUPPORTED when T * d / 8 exceeds 2^32 - 1 (token rows are
 * addressed by 32-bit offsets). */
tw_status hybrid_ffn_bwd(const uint16_t* dy, const uint16_t* x, const uint16_t* Wg,
                         const uint16_t* Wu, const uint16_t* Wd, int T, int d, int I,
                         const tw_hybrid* saved, float l1, uint16_t* dx, float* dWg,
                         float* dWu, float* dWd, void* ws, size_t ws_bytes,
                         int32_t* dev_status, void* stream);

/* The sparse part of the TwELL inference forward on an already packed TwELL (from
 * twell_pack or twell_gate_pack, including its overflow list): y for the rows
 * without overflow from the CUDA-core kernel, y for the overflow rows from the
 * dense tensor-core path. Together with tw_gate_relu_dense and twell_pack this is
 * the unfused pipeline (dense a through HBM, separate conversion, sparse matmuls)
 * that the pages argue against (explainer 1 "Problem Statement"; blog "1. TwELL");
 * twell_ffn_fwd is the fused form. Arguments as twell_ffn_fwd, with `packed` read
 * instead of written; TW_ECAPACITY when the packed TwELL lists more than ovf_cap
 * overflow rows. */
tw_status twell_ffn_sparse_fwd(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu,
                               const uint16_t* Wd, int T, int d, int I, int W, int C, int ovf_cap,
                               const tw_twell* packed, void* ws, size_t ws_bytes, uint16_t* y,
                               int32_t* dev_status, void* stream);

/* Dense gate activations a = bf16(ReLU(x Wg^T)) [T, I] (round to nearest even), the
 * first stage of the unfused pipeline. Shapes as twell_gate_pack (I % 64 == 0). */
tw_status tw_gate_relu_dense(const uint16_t* x, const uint16_t* Wg, int T, int d, int I,
                             uint16_t* a, int32_t* dev_status, void* stream);

/* Per-neuron activity counts of one Hybrid training forward (the statistic behind
 * the pages' dead-neuron analysis: thelatestinai listing, Figure 8, Table 5):
 * counts[j] += the number of tokens t with a_tj != 0, over the saved Hybrid's ELL
 * entries and its dense backup rows (fp32 a > 0). counts is [I] int32 on the
 * device, accumulated (zero it to start a window). Enqueues on `stream` after the
 * forward that filled `saved`. */
tw_status hybrid_neuron_counts(const tw_hybrid* saved, int32_t* counts, void* stream);

/* Dead-neuron re-initialisation of a weight matrix W [I, d] bf16 (the pages apply
 * it to the gate projection, Table 5 "Dead neuron reinit."): every row j with
 * counts[j] == 0 is overwritten with std * z, z = (sum of 12 uniforms) - 6
 * (Irwin-Hall: mean 0, variance 1, |z| <= 6). The uniforms are the top 24 bits of
 * SplitMix64 outputs number 12 (j d + k) + i (i < 12) of a generator seeded with
 * `seed`, so the values depend only on (seed, j, k). z is exact in float64; the value
 * is rounded once to float32, then to bf16 (nearest even). *n_reinit (device int32)
 * receives the number of rows rewritten. Rows with counts[j] != 0 are untouched.
 * Requires I >= 0, d > 0, std finite. */
tw_status tw_reinit_dead_rows(uint16_t* W, int I, int d, const int32_t* counts, uint64_t seed,
                              float std_dev, int32_t* n_reinit, void* stream);

/* Dense bf16 GEMM on the tensor cores, D[M, N] (fp32) = A B, the engine of the
 * dense backup path, exposed to check its operand layouts. a_mn == 0: A is [M, K]
 * (K contiguous); a_mn == 1: A is stored [K, M]. b_mn == 0: B is stored [N, K];
 * b_mn == 1: B is stored [K, N]. Requires M, N, K >= 1, N % 64 == 0, K % 64 == 0,
 * and M % 64 == 0 when a_mn == 1. */
tw_status tw_dense_gemm(const uint16_t* A, const uint16_t* B, int M, int N, int K,
                        int a_mn, int b_mn, float* D, int32_t* dev_status, void* stream);

/* tw_dense_gemm on CTA pairs: clusters of two CTAs, each 256 x 256 unit computed by
 * the two-SM form of the MMA (tcgen05.mma.cta_group::2) with each CTA holding its 128
 * rows of A and half of the B tile, as the library's 256-wide GEMMs run. Arguments
 * and layouts as tw_dense_gemm; requires N % 256 == 0 (TW_EINVAL otherwise). */
tw_status tw_dense_gemm_pair(const uint16_t* A, const uint16_t* B, int M, int N, int K,
                             int a_mn, int b_mn, float* D, int32_t* dev_status, void* stream);

/* L2 row-gather throughput probe for measurement tools (no counterpart on the pages):
 * the access pattern of the sparse kernels, with nothing else. `blocks` CTAs of d / 8
 * threads (one warp per 256-wide slice of d) take groups of eight indices from idx
 * [n_idx] (int32, device; values clamped to [0, rows)) and gather the eight rows'
 * slices of table [rows, d] bf16 (device) into registers, 16 bytes a lane, all eight
 * loads in flight together, summing them with packed fp32 FMAs; out [blocks * d / 8]
 * fp32 (device) receives each thread's sum. *bytes (host, may be NULL) = the row
 * bytes gathered (n_idx * d * 2); bytes / device time = the gather rate, from L2 when
 * the table fits in it. d as the FFN calls; n_idx a positive multiple of 8;
 * 1 <= blocks <= 2^20. Enqueued on `stream`. */
tw_status tw_l2_gather_probe(const uint16_t* table, int rows, int d, const int32_t* idx, int n_idx, float* out,
                             int blocks, double* bytes, void* stream);

/* The grid tw_l2_gather_probe is measured with: as many CTAs as the token kernels keep
 * resident (48 warps per SM at d = 2048) on every SM of the current device; 0 when d
 * is unsupported. */
int tw_l2_gather_probe_blocks(int d);

/* Test hook for the bounded waits (no counterpart on the pages): the GEMM of
 * tw_dense_gemm (a_mn = b_mn = 0; M <= 128, one 128-row tile; N in 64..256, a multiple
 * of 64; K a multiple of 64) with the TMA loads of K block `withhold_kb` (0 <=
 * withhold_kb < K / 64) never issued. The MMA issuer's wait for that pipeline stage
 * therefore runs out after the library's wait limit (1 s): the kernel raises
 * TW_ETIMEOUT in *dev_status, every role drains the copies and MMAs it issued, TMEM
 * is freed, and the kernel returns, leaving the context usable. D [M, N] fp32 is
 * left unspecified. Nothing faults, traps or spins without a limit. */
tw_status tw_wait_timeout_probe(const uint16_t* A, const uint16_t* B, int M, int N, int K, int withhold_kb,
                                float* D, int32_t* dev_status, void* stream);

/* The same test hook on a CTA pair (tw_dense_gemm_pair with a_mn = b_mn = 0; M <= 256,
 * one 256-row unit; N == 256; K a multiple of 64): both CTAs leave K block
 * `withhold_kb` unloaded, the MMA issuer's wait runs out, each CTA's waits end by the
 * abort flag or their own limit, and the two CTAs meet at the closing cluster barrier
 * before TMEM is freed. TW_ETIMEOUT in *dev_status; D left unspecified. */
tw_status tw_wait_timeout_probe_pair(const uint16_t* A, const uint16_t* B, int M, int N, int K, int withhold_kb,
                                     float* D, int32_t* dev_status, void* stream);

/* CUDA-core fp32 throughput probe for measurement tools (no counterpart on the
 * pages): `blocks` CTAs of 256 threads each run 8 independent chains of `iters`
 * packed two-lane FMAs (fma.rn.f32x2, the sparse kernels' accumulation
 * instruction) and write one float per thread to out [blocks * 256] (device,
 * caller-owned). *flops (host, may be NULL) receives the FLOPs the launch performs
 * (4 per packed FMA); FLOPs / device time = the fp32 FMA rate. Requires
 * 1 <= blocks <= 2^20, iters >= 1; enqueued on `stream`. */
tw_status tw_fma_probe(float* out, int blocks, int iters, double* flops, void* stream);

/* Kernel-level timing hook for measurement tools (no counterpart on the pages).
 * While a trace is active, every kernel or memset the library enqueues is followed
 * by cudaEventRecord(events[i], stream) with the next caller-created event, and its
 * label is kept; the time between consecutive events (the first measured from an
 * event the caller records just before the call) is that launch's device duration.
 * Recording stops silently when `capacity` events are used. Process-wide state, not
 * thread-safe: trace one host thread at a time. tw_trace_end() stops tracing and
 * returns the number of events recorded; tw_trace_label(i) names event i (a static
 * string; "memset" for cudaMemsetAsync calls), or NULL when i is out of range. */
tw_status tw_trace_begin(void* const* events, int capacity);
int tw_trace_end(void);
const char* tw_trace_label(int i);

#ifdef __cplusplus
}
#endif

#endif /* TWELL_H */

// extern "C" entry points declared in include/twell.h: host-side validation,
// workspace layout and the launch sequence of each operation. Everything is
// enqueued on the caller's stream; nothing is allocated, freed or synchronised.
#include <cmath>
#include <stdint.h>
#include <string.h>

#include <initializer_list>

#include "tw_internal.h"

namespace {

constexpr int kAbiVersion = 2;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Bump allocator over the caller's workspace (or a dry run with base == nullptr
// that only measures). Every block starts on a 256-byte boundary.
struct Carve {
  uint8_t* base;
  size_t off = 0;
  explicit Carve(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <class T>
  T* take(size_t n) {
    off = (off + 255) & ~static_cast<size_t>(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += n * sizeof(T);
    return p;
  }
};

tw_status from_cuda(cudaError_t e) { return e == cudaSuccess ? TW_OK : TW_ECUDA; }

#define TW_TRY(expr)                           \
  do {                                         \
    cudaError_t e_ = (expr);                   \
    if (e_ != cudaSuccess) return TW_ECUDA;    \
  } while (0)

tw_status check_tile_geometry(int T, int I, int W, int C) {
  if (T < 0) return TW_EINVAL;
  if (W != 64 && W != 128) return TW_EUNSUPPORTED;
  if (I < 64 || I > 65536 || I % W != 0) return TW_EUNSUPPORTED;
  if (C < 1 || C > W) return TW_EINVAL;
  if ((I / W) * C > tw::kMaxList) return TW_EUNSUPPORTED;  // per-token entry list of the sparse forward
  return TW_OK;
}

tw_status check_model_width(int d) {
  if (d < 256 || d > 2048 || d % 256 != 0) return TW_EUNSUPPORTED;
  return TW_OK;
}

tw_status check_twell(const tw_twell* o, int T, int I, int W, int C) {
  if (o == nullptr) return TW_EINVAL;
  if (o->T != T || o->I != I || o->W != W || o->C != C) return TW_EINVAL;
  if (T == 0) return TW_OK;
  const void* ptrs[] = {o->cnt, o->val, o->idx, o->row_nnz, o->ovf, o->ovf_rows, o->n_ovf};
  for (const void* p : ptrs) {
    if (p == nullptr) return TW_EINVAL;
    if (!aligned16(p)) return TW_EALIGN;
  }
  return TW_OK;
}

tw_status check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs) {
    if (p == nullptr) return TW_EINVAL;
    if (!aligned16(p)) return TW_EALIGN;
  }
  return TW_OK;
}

tw_status check_hybrid(const tw_hybrid* h, int T, int I, bool gated) {
  if (h == nullptr) return TW_EINVAL;
  if (h->T != T || h->I != I || h->R < 1 || h->R > I || h->backup_cap < 0 || h->backup_cap > T) return TW_EINVAL;
  if (h->route < TW_ROUTE_SPARSE || h->route > TW_ROUTE_AUTO) return TW_EINVAL;
  if (h->route != TW_ROUTE_SPARSE) {
    if (!(h->dense_above >= 0.f) || h->route_taken == nullptr) return TW_EINVAL;
    if (reinterpret_cast<uintptr_t>(h->route_taken) % 4 != 0) return TW_EALIGN;
  }
  tw_status st = check_ptrs({h->row_nnz, h->ell_nnz, h->ell_idx, h->ell_a, h->backup_slot, h->n_backup});
  if (st != TW_OK) return st;
  if (gated) {
    st = check_ptrs({h->ell_u});
    if (st != TW_OK) return st;
  }
  if (h->backup_cap > 0) {
    st = check_ptrs({h->backup_tok, h->backup_a});
    if (st != TW_OK) return st;
    if (gated) {
      st = check_ptrs({h->backup_u});
      if (st != TW_OK) return st;
    }
  }
  return TW_OK;
}

// ------------------------------------------------------------------ workspace layouts
struct FwdWs {
  uint16_t* X;
  uint16_t* H;
  uint16_t* H_lo;
  float* acc;      // split-K accumulator of the overflow rows' down projection [ra, d]
  int32_t* sched;  // token scheduling counter of the sparse forward
};
FwdWs carve_twell_fwd(Carve& c, int d, int I, int ovf_cap) {
  const int ra = round_up(ovf_cap, 128);
  FwdWs w{};
  w.X = c.take<uint16_t>(static_cast<size_t>(ra) * d);
  w.H = c.take<uint16_t>(static_cast<size_t>(ra) * I);
  w.H_lo = c.take<uint16_t>(static_cast<size_t>(ra) * I);
  w.acc = c.take<float>(static_cast<size_t>(ra) * d);
  w.sched = c.take<int32_t>(4);
  return w;
}

struct HybFwdWs {
  uint16_t* cnt;
  uint16_t* val;
  uint8_t* idx;
  uint8_t* ovf;
  int32_t* ovf_rows;
  int32_t* n_ovf;
  uint16_t* X;
  uint16_t* H;
  uint16_t* H_lo;
  float* acc;  // split-K accumulators [ra, acc_ld]: the down projection (columns [0, d)),
               // and for a small backup the hidden product's g and u ([d, d + 2 I))
  int acc_ld;
  bool split;      // backup_cap <= kBackupSplitRows: the hidden product runs split-K
  int32_t* sched;  // token scheduling counter of the sparse forward
  uint16_t* Hd;    // dense route: fp16 h of every row [T, I] (null for the sparse route)
  uint16_t* Wd16;  // dense route: fp16 copy of Wd [I, d] (the down GEMM's operand)
};
HybFwdWs carve_hybrid_fwd(Carve& c, int T, int d, int I, int W, int C, int backup_cap, int route) {
  const size_t nT = static_cast<size_t>(I / W);
  const int ra = round_up(backup_cap, 128);
  HybFwdWs w{};
  w.cnt = c.take<uint16_t>(static_cast<size_t>(T) * nT);
  w.val = c.take<uint16_t>(static_cast<size_t>(T) * nT * C);
  w.idx = c.take<uint8_t>(static_cast<size_t>(T) * nT * C);
  w.ovf = c.take<uint8_t>(static_cast<size_t>(T));
  w.ovf_rows = c.take<int32_t>(static_cast<size_t>(T));
  w.n_ovf = c.take<int32_t>(1);
  w.X = c.take<uint16_t>(static_cast<size_t>(ra) * d);
  w.H = c.take<uint16_t>(static_cast<size_t>(ra) * I);
  w.H_lo = c.take<uint16_t>(static_cast<size_t>(ra) * I);
  w.split = backup_cap <= tw::kBackupSplitRows;
  w.acc_ld = d + (w.split ? 2 * I : 0);
  w.acc = c.take<float>(static_cast<size_t>(ra) * w.acc_ld);
  w.sched = c.take<int32_t>(4);
  w.Hd = route != TW_ROUTE_SPARSE ? c.take<uint16_t>(static_cast<size_t>(T) * I) : nullptr;
  w.Wd16 = route != TW_ROUTE_SPARSE ? c.take<uint16_t>(static_cast<size_t>(I) * d) : nullptr;
  return w;
}

struct HybBwdWs {
  int32_t* col_cnt;
  int32_t* col_ptr;
  int32_t* col_cur;
  uint4* csc;
  uint16_t* dY;
  uint16_t* X;
  tw::BackupGradOut g;  // dG, dU, H as (hi, lo) bf16 pairs
  float* acc;           // split-K accumulators [ra, acc_ld]: dx of the backup rows (columns
                        // [0, d)), and for a small backup dh ([d, d + I))
  int acc_ld;
  bool split;           // backup_cap <= kBackupSplitRows: the grad product runs split-K
  int32_t* sched;       // token scheduling counter of the token pass
  uint16_t *dGd, *dUd, *Hd;  // dense route: fp16 dg, du, h of every row [T, I] (null for the sparse route)
  uint16_t *Wg16, *Wu16;     // dense route: fp16 copies of the weights [I, d] (the dx GEMM's operands)
  uint16_t *X16, *dY16;      // and of x and dy [T, d] (the weight-gradient GEMMs' operands)
};
HybBwdWs carve_hybrid_bwd(Carve& c, int T, int d, int I, int R, int backup_cap, int route) {
  const size_t TR = static_cast<size_t>(T) * R;
  const int ra = round_up(backup_cap, 128);
  const size_t rI = static_cast<size_t>(ra) * I;
  HybBwdWs w{};
  w.col_cnt = c.take<int32_t>(static_cast<size_t>(I) + 1);
  w.col_ptr = c.take<int32_t>(static_cast<size_t>(I) + 1);
  w.col_cur = c.take<int32_t>(static_cast<size_t>(I));
  w.csc = c.take<uint4>(TR);
  w.dY = c.take<uint16_t>(static_cast<size_t>(ra) * d);
  w.X = c.take<uint16_t>(static_cast<size_t>(ra) * d);
  w.g.dG = c.take<uint16_t>(rI);
  w.g.dG_lo = c.take<uint16_t>(rI);
  w.g.dU = c.take<uint16_t>(rI);
  w.g.dU_lo = c.take<uint16_t>(rI);
  w.g.H = c.take<uint16_t>(rI);
  w.g.H_lo = c.take<uint16_t>(rI);
  w.split = backup_cap <= tw::kBackupSplitRows;
  w.acc_ld = d + (w.split ? I : 0);
  w.acc = c.take<float>(static_cast<size_t>(ra) * w.acc_ld);
  w.sched = c.take<int32_t>(tw::kSchedWords);
  if (route != TW_ROUTE_SPARSE) {
    const size_t TI = static_cast<size_t>(T) * I;
    w.dGd = c.take<uint16_t>(TI);
    w.dUd = c.take<uint16_t>(TI);
    w.Hd = c.take<uint16_t>(TI);
    w.Wg16 = c.take<uint16_t>(static_cast<size_t>(I) * d);
    w.Wu16 = c.take<uint16_t>(static_cast<size_t>(I) * d);
    w.X16 = c.take<uint16_t>(static_cast<size_t>(T) * d);
    w.dY16 = c.take<uint16_t>(static_cast<size_t>(T) * d);
  } else {
    w.dGd = w.dUd = w.Hd = w.Wg16 = w.Wu16 = w.X16 = w.dY16 = nullptr;
  }
  return w;
}

}  // namespace

extern "C" {

const char* tw_status_str(int status) {
  switch (status) {
    case TW_OK: return "TW_OK";
    case TW_EINVAL: return "TW_EINVAL: invalid argument";
    case TW_EALIGN: return "TW_EALIGN: pointer not 16-byte aligned";
    case TW_EUNSUPPORTED: return "TW_EUNSUPPORTED: shape outside the implemented range";
    case TW_ECAPACITY: return "TW_ECAPACITY: more overflow/backup rows than the buffers hold";
    case TW_ETIMEOUT: return "TW_ETIMEOUT: a bounded pipeline wait gave up";
    case TW_ECUDA: return "TW_ECUDA: CUDA runtime error";
    case TW_EWORKSPACE: return "TW_EWORKSPACE: workspace too small";
    case TW_EBOUNDS: return "TW_EBOUNDS: an index read from the data fell outside its buffer (checked build)";
    default: return "unknown tw_status";
  }
}

int tw_abi_version(void) { return kAbiVersion; }

tw_status tw_trace_begin(void* const* events, int capacity) {
  if (events == nullptr || capacity < 1) return TW_EINVAL;
  tw::trace_begin(events, capacity);
  return TW_OK;
}

int tw_trace_end(void) { return tw::trace_end(); }

const char* tw_trace_label(int i) { return tw::trace_label(i); }

tw_status twell_pack(const uint16_t* A, int T, int I, int W, int C, const tw_twell* out, int32_t* dev_status,
                     void* stream) {
  tw_status st = check_tile_geometry(T, I, W, C);
  if (st != TW_OK) return st;
  st = check_twell(out, T, I, W, C);
  if (st != TW_OK) return st;
  if (T == 0) return TW_OK;
  st = check_ptrs({A, dev_status});
  if (st != TW_OK) return st;
  cudaStream_t s = as_stream(stream);
  TW_TRY(tw::launch_pack_dense(A, T, I, W, C, *out, s));
  TW_TRY(tw::launch_compact_rows(out->ovf, nullptr, 0, T, out->ovf_rows, T, out->n_ovf, nullptr, nullptr, T,
                                 dev_status, s));
  return TW_OK;
}

static tw_status gate_pack_impl(const uint16_t* x, const uint16_t* Wg, int T, int d, int I, int W, int C,
                                const tw_twell& o, uint16_t* a_dense, int cap_check, int32_t* dev_status,
                                cudaStream_t s, bool list_overflow = true) {
  TW_TRY(tw::launch_zero(o.row_nnz, sizeof(int32_t) * T, o.ovf, static_cast<size_t>(T), s));
  TW_TRY(tw::gemm_gate_pack(x, Wg, T, d, I, W, C, o, a_dense, dev_status, s));
  if (list_overflow)
    TW_TRY(tw::launch_compact_rows(o.ovf, nullptr, 0, T, o.ovf_rows, T, o.n_ovf, nullptr, nullptr, cap_check,
                                   dev_status, s));
  return TW_OK;
}

tw_status twell_gate_pack(const uint16_t* x, const uint16_t* Wg, int T, int d, int I, int W, int C,
                          const tw_twell* out, uint16_t* a_dense, int32_t* dev_status, void* stream) {
  tw_status st = check_tile_geometry(T, I, W, C);
  if (st != TW_OK) return st;
  st = check_model_width(d);
  if (st != TW_OK) return st;
  st = check_twell(out, T, I, W, C);
  if (st != TW_OK) return st;
  if (T == 0) return TW_OK;
  st = check_ptrs({x, Wg, dev_status});
  if (st != TW_OK) return st;
  if (a_dense != nullptr && !aligned16(a_dense)) return TW_EALIGN;
  return gate_pack_impl(x, Wg, T, d, I, W, C, *out, a_dense, T, dev_status, as_stream(stream));
}

size_t twell_ffn_fwd_workspace_size(int T, int d, int I, int W, int C, int ovf_cap) {
  (void)T;
  (void)W;
  (void)C;
  Carve c(nullptr);
  carve_twell_fwd(c, d, I, ovf_cap < 0 ? 0 : ovf_cap);
  return c.off + 256;
}

// The sparse part of the TwELL forward, given a packed TwELL with its overflow list:
// the token kernel on the non-overflow rows, the dense tensor-core path on the
// overflow rows (TW_ECAPACITY when more than ovf_cap rows overflowed).
static tw_status twell_sparse_impl(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd,
                                   int T, int d, int I, int W, int C, int ovf_cap, const tw_twell& o, void* ws,
                                   uint16_t* y, int32_t* dev_status, cudaStream_t s) {
  Carve c(reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~static_cast<uintptr_t>(255)));
  const FwdWs w = carve_twell_fwd(c, d, I, ovf_cap);
  const int ra = round_up(ovf_cap, 128);
  tw::SparseFwdArgs a{};
  a.x = x; a.Wu = Wu; a.Wd = Wd;
  a.T = T; a.d = d; a.I = I; a.W = W; a.C = C; a.nT = I / W; a.L = (I / W) * C;
  a.cnt = o.cnt; a.val = o.val; a.idx = o.idx; a.ovf = o.ovf;
  a.backup_slot = nullptr;
  a.y = y;
  a.status = dev_status;
  a.sched = w.sched;
  a.sched_zeroed = false;
  TW_TRY(tw::launch_token_fwd(a, s));
  if (ovf_cap > 0) {
    TW_TRY(tw::launch_gather_rows(x, d, T, o.ovf_rows, o.n_ovf, ovf_cap, ra, w.X, s, dev_status, nullptr, nullptr,
                                  w.acc, d));
    TW_TRY(tw::gemm_backup_hidden(w.X, Wg, Wu, ra, o.n_ovf, ovf_cap, d, I, w.H, w.H_lo, nullptr, nullptr,
                                  dev_status, s));
    // the down projection spread over every SM (split-K into an fp32 accumulator),
    // then the rows written out as bf16
    const uint16_t* A[2] = {w.H, w.H_lo};
    const uint16_t* B[2] = {Wd, Wd};
    TW_TRY(tw::gemm_rows_times_nmajor_splitk(A, B, 2, ra, o.n_ovf, ovf_cap, I, d, w.acc, dev_status, s));
    TW_TRY(tw::launch_scatter_rows_bf16(w.acc, d, o.n_ovf, ovf_cap, o.ovf_rows, y, d, T, s));
  }
  return TW_OK;
}

}  // extern "C"

namespace tw {
// Every argument check of twell_ffn_fwd except the workspace's.
tw_status check_twell_fwd_operands(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd,
                                   int T, int d, int I, int W, int C, int ovf_cap, const tw_twell* tw_out,
                                   uint16_t* y, int32_t* dev_status) {
  tw_status st = check_tile_geometry(T, I, W, C);
  if (st != TW_OK) return st;
  st = check_model_width(d);
  if (st != TW_OK) return st;
  if (ovf_cap < 0 || ovf_cap > T) return TW_EINVAL;
  st = check_twell(tw_out, T, I, W, C);
  if (st != TW_OK) return st;
  if (T == 0) return TW_OK;
  st = check_ptrs({x, Wg, Wd, y, dev_status});
  if (st != TW_OK) return st;
  if (Wu != nullptr && !aligned16(Wu)) return TW_EALIGN;
  return TW_OK;
}
}  // namespace tw

extern "C" {

static tw_status check_twell_fwd_args(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd,
                                      int T, int d, int I, int W, int C, int ovf_cap, const tw_twell* tw_out,
                                      void* ws, size_t ws_bytes, uint16_t* y, int32_t* dev_status) {
  tw_status st = tw::check_twell_fwd_operands(x, Wg, Wu, Wd, T, d, I, W, C, ovf_cap, tw_out, y, dev_status);
  if (st != TW_OK || T == 0) return st;
  if (ws_bytes < twell_ffn_fwd_workspace_size(T, d, I, W, C, ovf_cap)) return TW_EWORKSPACE;
  if (ovf_cap > 0 && ws == nullptr) return TW_EINVAL;
  return TW_OK;
}

tw_status twell_ffn_fwd(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, int T, int d,
                        int I, int W, int C, int ovf_cap, const tw_twell* tw_out, void* ws, size_t ws_bytes,
                        uint16_t* y, int32_t* dev_status, void* stream) {
  tw_status st = check_twell_fwd_args(x, Wg, Wu, Wd, T, d, I, W, C, ovf_cap, tw_out, ws, ws_bytes, y, dev_status);
  if (st != TW_OK || T == 0) return st;
  cudaStream_t s = as_stream(stream);
  st = gate_pack_impl(x, Wg, T, d, I, W, C, *tw_out, nullptr, ovf_cap, dev_status, s);
  if (st != TW_OK) return st;
  return twell_sparse_impl(x, Wg, Wu, Wd, T, d, I, W, C, ovf_cap, *tw_out, ws, y, dev_status, s);
}

tw_status twell_ffn_sparse_fwd(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, int T,
                               int d, int I, int W, int C, int ovf_cap, const tw_twell* packed, void* ws,
                               size_t ws_bytes, uint16_t* y, int32_t* dev_status, void* stream) {
  tw_status st = check_twell_fwd_args(x, Wg, Wu, Wd, T, d, I, W, C, ovf_cap, packed, ws, ws_bytes, y, dev_status);
  if (st != TW_OK || T == 0) return st;
  return twell_sparse_impl(x, Wg, Wu, Wd, T, d, I, W, C, ovf_cap, *packed, ws, y, dev_status, as_stream(stream));
}

tw_status tw_gate_relu_dense(const uint16_t* x, const uint16_t* Wg, int T, int d, int I, uint16_t* a,
                             int32_t* dev_status, void* stream) {
  if (T < 0 || I < 64 || I > 65536 || I % 64 != 0) return TW_EUNSUPPORTED;
  tw_status st = check_model_width(d);
  if (st != TW_OK) return st;
  if (T == 0) return TW_OK;
  st = check_ptrs({x, Wg, a, dev_status});
  if (st != TW_OK) return st;
  TW_TRY(tw::gemm_gate_relu_dense(x, Wg, T, d, I, a, dev_status, as_stream(stream)));
  return TW_OK;
}

size_t hybrid_ffn_fwd_workspace_size(int T, int d, int I, int W, int C, int R, int backup_cap, int route) {
  (void)R;
  if (T < 0 || W <= 0 || C <= 0) return 0;
  Carve c(nullptr);
  carve_hybrid_fwd(c, T, d, I, W, C, backup_cap < 0 ? 0 : backup_cap, route);
  return c.off + 256;
}

tw_status hybrid_ffn_fwd(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, int T, int d,
                         int I, int W, int C, const tw_hybrid* saved, void* ws, size_t ws_bytes, uint16_t* y,
                         int32_t* dev_status, void* stream) {
  tw_status st = check_tile_geometry(T, I, W, C);
  if (st != TW_OK) return st;
  st = check_model_width(d);
  if (st != TW_OK) return st;
  const bool gated = Wu != nullptr;
  st = check_hybrid(saved, T, I, gated);
  if (st != TW_OK) return st;
  if (T == 0) return TW_OK;
  st = check_ptrs({x, Wg, Wd, y, dev_status, ws});
  if (st != TW_OK) return st;
  if (gated && !aligned16(Wu)) return TW_EALIGN;
  const int R = saved->R, cap = saved->backup_cap;
  const int route = saved->route;
  if (ws_bytes < hybrid_ffn_fwd_workspace_size(T, d, I, W, C, R, cap, route)) return TW_EWORKSPACE;
  cudaStream_t s = as_stream(stream);
  Carve c(reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~static_cast<uintptr_t>(255)));
  const HybFwdWs w = carve_hybrid_fwd(c, T, d, I, W, C, cap, route);
  const int ra = round_up(cap, 128);
  tw_twell o{T, I, W, C, w.cnt, w.val, w.idx, saved->row_nnz, w.ovf, w.ovf_rows, w.n_ovf};
  // the route this call takes, decided on the device by the row compaction (it is
  // known on the host only for the fixed routes); kernels of the other route return
  const int32_t* taken = route == TW_ROUTE_SPARSE ? nullptr : saved->route_taken;

  // the backup list below covers the overflow rows, so the TwELL's own list is not built
  st = gate_pack_impl(x, Wg, T, d, I, W, C, o, nullptr, T, dev_status, s, false);
  if (st != TW_OK) return st;
  TW_TRY(tw::launch_compact_rows(o.ovf, saved->row_nnz, R, T, saved->backup_tok, cap, saved->n_backup,
                                 saved->backup_slot, saved->ell_nnz, cap, dev_status, s, w.sched, route,
                                 saved->dense_above, saved->route_taken));
  tw::SparseFwdArgs a{};
  a.x = x; a.Wu = Wu; a.Wd = Wd;
  a.T = T; a.d = d; a.I = I; a.W = W; a.C = C; a.nT = I / W; a.L = (I / W) * C;
  a.cnt = o.cnt; a.val = o.val; a.idx = o.idx; a.ovf = o.ovf;
  a.backup_slot = saved->backup_slot;
  a.ell_nnz = saved->ell_nnz;
  a.ell_idx = saved->ell_idx; a.ell_a = saved->ell_a; a.ell_u = saved->ell_u; a.R = R;
  a.y = y;
  a.status = dev_status;
  a.sched = w.sched;
  a.sched_zeroed = true;  // by compact_rows above
  a.route = taken;
  if (route != TW_ROUTE_DENSE) {
    // gated: the ELL rows' idx and a from the TwELL first (a warp a row), which the
    // token kernel then reads as its entry lists
    if (gated) TW_TRY(tw::launch_twell_to_ell(o, saved->backup_slot, R, saved->ell_idx, saved->ell_a, taken,
                                              dev_status, s));
    TW_TRY(tw::launch_token_fwd(a, s));
  }
  // the backup rows' fp32 a and u (saved for the backward) on the tensor cores; the
  // sparse route also takes the hi/lo bf16 pair of their h here and their y below
  if (cap > 0) {
    // the accumulator holds only the sparse route's y unless the hidden product runs
    // split-K into it too
    TW_TRY(tw::launch_gather_rows(x, d, T, saved->backup_tok, saved->n_backup, cap, ra, w.X, s, dev_status, nullptr,
                                  nullptr, w.acc, w.acc_ld, nullptr, w.split ? nullptr : taken));
    TW_TRY(tw::gemm_backup_hidden(w.X, Wg, Wu, ra, saved->n_backup, cap, d, I, w.H, w.H_lo, saved->backup_a,
                                  gated ? saved->backup_u : nullptr, dev_status, s, taken,
                                  w.split ? w.acc + d : nullptr, w.acc_ld));
  }
  if (route != TW_ROUTE_SPARSE) {
    // the dense route: h of every row on the tensor cores (the ELL rows from the TwELL,
    // writing the saved Hybrid's ELL; the backup rows from their fp32 a), then
    // y = h Wd over all rows on fp16 operands
    {
      const uint16_t* src[1] = {Wd};
      uint16_t* dst[1] = {w.Wd16};
      const size_t n[1] = {static_cast<size_t>(I) * d};
      TW_TRY(tw::launch_to_f16(src, dst, n, 1, taken, s));
    }
    if (gated)
      // u of the backup rows is saved here unless the split-K backup product saved it
      TW_TRY(tw::gemm_up_hybrid(x, Wu, T, d, I, o, R, saved->backup_slot, saved->backup_a,
                                w.split ? nullptr : saved->backup_u, cap, w.Hd, saved->ell_idx, saved->ell_a,
                                saved->ell_u, taken, dev_status, s));
    else
      TW_TRY(tw::launch_twell_to_dense_ell(o, saved->backup_slot, saved->backup_a, cap, R, w.Hd, saved->ell_idx,
                                           saved->ell_a, taken, dev_status, s));
    const uint16_t* A[1] = {w.Hd};
    const uint16_t* B[1] = {w.Wd16};
    TW_TRY(tw::gemm_rows_nmajor_bf16(A, B, 1, T, I, d, y, d, taken, dev_status, s, true, "dense_down"));
  }
  if (cap > 0 && route != TW_ROUTE_DENSE) {
    const uint16_t* A[2] = {w.H, w.H_lo};
    const uint16_t* B[2] = {Wd, Wd};
    TW_TRY(tw::gemm_rows_times_nmajor_splitk(A, B, 2, ra, saved->n_backup, cap, I, d, w.acc, dev_status, s, taken,
                                             w.acc_ld));
    TW_TRY(tw::launch_scatter_rows_bf16(w.acc, d, saved->n_backup, cap, saved->backup_tok, y, d, T, s, taken,
                                        w.acc_ld));
  }
  return TW_OK;
}

size_t hybrid_ffn_bwd_workspace_size(int T, int d, int I, int R, int backup_cap, int route) {
  if (T < 0 || R < 1) return 0;
  Carve c(nullptr);
  carve_hybrid_bwd(c, T, d, I, R, backup_cap < 0 ? 0 : backup_cap, route);
  return c.off + 256;
}

tw_status hybrid_ffn_bwd(const uint16_t* dy, const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu,
                         const uint16_t* Wd, int T, int d, int I, const tw_hybrid* saved, float l1, uint16_t* dx,
                         float* dWg, float* dWu, float* dWd, void* ws, size_t ws_bytes, int32_t* dev_status,
                         void* stream) {
  if (T < 0 || I < 64 || I > 65536 || I % 64 != 0) return TW_EUNSUPPORTED;
  tw_status st = check_model_width(d);
  if (st != TW_OK) return st;
  // token rows are addressed by 32-bit offsets in 16-byte units in the transposed Hybrid
  if (static_cast<uint64_t>(T) * static_cast<uint64_t>(d / 8) > 0xFFFFFFFFull) return TW_EUNSUPPORTED;
  const bool gated = Wu != nullptr;
  st = check_hybrid(saved, T, I, gated);
  if (st != TW_OK) return st;
  st = check_ptrs({Wg, Wd, dWg, dWd, dev_status, ws});
  if (st != TW_OK) return st;
  if (gated) {
    st = check_ptrs({Wu, dWu});
    if (st != TW_OK) return st;
  }
  if (T > 0) {
    st = check_ptrs({dy, x, dx});
    if (st != TW_OK) return st;
  }
  const int R = saved->R, cap = saved->backup_cap;
  const int route = saved->route;
  if (ws_bytes < hybrid_ffn_bwd_workspace_size(T, d, I, R, cap, route)) return TW_EWORKSPACE;
  cudaStream_t s = as_stream(stream);
  Carve c(reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~static_cast<uintptr_t>(255)));
  const HybBwdWs w = carve_hybrid_bwd(c, T, d, I, R, cap, route);
  const int ra = round_up(cap, 128);
  // the route the forward took (T == 0: no forward ran, the sparse path writes dW = 0)
  const bool dense_possible = route != TW_ROUTE_SPARSE && T > 0;
  const int32_t* taken = dense_possible ? saved->route_taken : nullptr;

  tw::SparseBwdArgs a{};
  a.dy = dy; a.x = x; a.Wg = Wg; a.Wu = Wu; a.Wd = Wd;
  a.T = T; a.d = d; a.I = I; a.R = R; a.l1 = l1;
  a.ell_nnz = saved->ell_nnz; a.backup_slot = saved->backup_slot;
  a.ell_idx = saved->ell_idx; a.ell_a = saved->ell_a; a.ell_u = saved->ell_u;
  a.dx = dx;
  a.col_cnt = w.col_cnt; a.col_ptr = w.col_ptr; a.col_cur = w.col_cur; a.csc = w.csc;
  a.csc_cap = static_cast<long long>(T) * R;
  a.status = dev_status;
  a.dWg = dWg; a.dWu = dWu; a.dWd = dWd;
  a.sched = w.sched;
  a.sched_w = w.sched + tw::kSchedStride;
  a.route = taken;
  const bool sparse_possible = route != TW_ROUTE_DENSE || T == 0;
  if (sparse_possible) TW_TRY(tw::launch_sparse_bwd_tokens(a, s));
  if (dense_possible) {
    // the dense route: dg, du, h of every row (fp16; the backup rows' from their saved
    // fp32 a and u) from dh = dY Wd^T on the tensor cores, then dx = dg Wg + du Wu over
    // all rows on fp16 operands
    const uint16_t* src[4] = {Wg, x, dy, Wu};
    uint16_t* dst[4] = {w.Wg16, w.X16, w.dY16, w.Wu16};
    const size_t n[4] = {static_cast<size_t>(I) * d, static_cast<size_t>(T) * d, static_cast<size_t>(T) * d,
                         static_cast<size_t>(I) * d};
    TW_TRY(tw::launch_to_f16(src, dst, n, gated ? 4 : 3, taken, s));
    TW_TRY(tw::gemm_dense_grad(dy, Wd, T, d, I, *saved, gated, l1, w.dGd, w.dUd, w.Hd, taken, dev_status, s));
    const uint16_t* A[2] = {w.dGd, w.dUd};
    const uint16_t* B[2] = {w.Wg16, w.Wu16};
    TW_TRY(tw::gemm_rows_nmajor_bf16(A, B, gated ? 2 : 1, T, I, d, dx, d, taken, dev_status, s, true, "dense_dx"));
  }
  const bool backup = cap > 0 && T > 0;
  if (backup && route != TW_ROUTE_DENSE) {
    // the sparse route's dense backup (the dense route's GEMMs above cover the backup
    // rows, so these launches do nothing when the call took that route)
    TW_TRY(tw::launch_gather_rows(dy, d, T, saved->backup_tok, saved->n_backup, cap, ra, w.dY, s, dev_status, x, w.X,
                                  w.acc, w.acc_ld, taken));
    const int32_t* nb = saved->n_backup;
    const tw::BackupGradOut& g = w.g;
    TW_TRY(tw::gemm_backup_grad(w.dY, Wd, ra, nb, cap, d, I, saved->backup_a, gated ? saved->backup_u : nullptr,
                                l1, g, dev_status, s, taken, w.split ? w.acc + d : nullptr, w.acc_ld));
    // dx = (dG + dG_lo) Wg + (dU + dU_lo) Wu, scattered back to the backup tokens
    const uint16_t* A[4] = {g.dG, g.dG_lo, g.dU, g.dU_lo};
    const uint16_t* B[4] = {Wg, Wg, Wu, Wu};
    TW_TRY(tw::gemm_rows_times_nmajor_splitk(A, B, gated ? 4 : 2, ra, nb, cap, I, d, w.acc, dev_status, s, taken,
                                             w.acc_ld));
    TW_TRY(tw::launch_scatter_rows_bf16(w.acc, d, nb, cap, saved->backup_tok, dx, d, T, s, taken, w.acc_ld));
    // the backup rows' weight gradients are written first (when there are any);
    // the ELL part is then added to them
    // all (two or three) in one launch
    const tw::WeightGradProblem probs[3] = {{g.dG, g.dG_lo, w.X, dWg},
                                            {g.H, g.H_lo, w.dY, dWd},
                                            {g.dU, g.dU_lo, w.X, dWu}};
    TW_TRY(tw::gemm_weight_grads(probs, gated ? 3 : 2, ra, nb, cap, I, d, dev_status, s, taken));
  }
  a.dW_base_rows = backup ? saved->n_backup : nullptr;
  if (sparse_possible) TW_TRY(tw::launch_sparse_bwd_weights(a, s));
  if (dense_possible) {
    // dense route weight gradients over all rows, the backup rows included: written
    const tw::DenseWeightGradProblem probs[3] = {{w.dGd, w.X16, dWg}, {w.Hd, w.dY16, dWd}, {w.dUd, w.X16, dWu}};
    TW_TRY(tw::gemm_dense_weight_grads(probs, gated ? 3 : 2, T, I, d, nullptr, taken, dev_status, s));
  }
  return TW_OK;
}

tw_status twell_unpack(const tw_twell* in, uint16_t* A, void* stream) {
  if (in == nullptr) return TW_EINVAL;
  tw_status st = check_tile_geometry(in->T, in->I, in->W, in->C);
  if (st != TW_OK) return st;
  st = check_twell(in, in->T, in->I, in->W, in->C);
  if (st != TW_OK || in->T == 0) return st;
  st = check_ptrs({A});
  if (st != TW_OK) return st;
  TW_TRY(tw::launch_twell_unpack(*in, A, as_stream(stream)));
  return TW_OK;
}

size_t hybrid_pack_workspace_size(int T) {
  if (T < 0) return 0;
  Carve c(nullptr);
  c.take<uint8_t>(static_cast<size_t>(T));
  return c.off + 256;
}

tw_status hybrid_pack(const uint16_t* A, const uint16_t* U, int T, int I, int W, int C, const tw_hybrid* out, void* ws,
                      size_t ws_bytes, int32_t* dev_status, void* stream) {
  tw_status st = check_tile_geometry(T, I, W, C);
  if (st != TW_OK) return st;
  const bool gated = U != nullptr;
  st = check_hybrid(out, T, I, gated);
  if (st != TW_OK) return st;
  if (T == 0) return TW_OK;
  st = check_ptrs({A, dev_status, ws});
  if (st != TW_OK) return st;
  if (gated && !aligned16(U)) return TW_EALIGN;
  if (ws_bytes < hybrid_pack_workspace_size(T)) return TW_EWORKSPACE;
  Carve c(reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~static_cast<uintptr_t>(255)));
  uint8_t* ovf = c.take<uint8_t>(static_cast<size_t>(T));
  TW_TRY(tw::launch_hybrid_pack(A, U, T, I, W, C, *out, ovf, dev_status, as_stream(stream)));
  return TW_OK;
}

tw_status hybrid_unpack(const tw_hybrid* in, float* A, float* U, void* stream) {
  if (in == nullptr) return TW_EINVAL;
  if (in->T < 0 || in->I < 64 || in->I > 65536 || in->I % 64 != 0) return TW_EUNSUPPORTED;
  tw_status st = check_hybrid(in, in->T, in->I, U != nullptr);
  if (st != TW_OK || in->T == 0) return st;
  st = check_ptrs({A});
  if (st != TW_OK) return st;
  if (U != nullptr && !aligned16(U)) return TW_EALIGN;
  TW_TRY(tw::launch_hybrid_unpack(*in, A, U, as_stream(stream)));
  return TW_OK;
}

tw_status hybrid_neuron_counts(const tw_hybrid* saved, int32_t* counts, void* stream) {
  if (saved == nullptr) return TW_EINVAL;
  if (saved->T < 0 || saved->I < 1 || saved->R < 1 || saved->backup_cap < 0 || saved->backup_cap > saved->T)
    return TW_EINVAL;
  if (saved->T == 0) return TW_OK;
  tw_status st = check_ptrs({counts, saved->ell_nnz, saved->ell_idx, saved->n_backup});
  if (st != TW_OK) return st;
  if (saved->backup_cap > 0) {
    st = check_ptrs({saved->backup_a});
    if (st != TW_OK) return st;
  }
  TW_TRY(tw::launch_neuron_counts(*saved, counts, as_stream(stream)));
  return TW_OK;
}

tw_status tw_reinit_dead_rows(uint16_t* W, int I, int d, const int32_t* counts, uint64_t seed, float std_dev,
                              int32_t* n_reinit, void* stream) {
  if (I < 0 || d < 1 || !std::isfinite(std_dev)) return TW_EINVAL;
  tw_status st = check_ptrs({n_reinit});
  if (st != TW_OK) return st;
  if (I > 0) {
    if (W == nullptr || counts == nullptr) return TW_EINVAL;
    if (reinterpret_cast<uintptr_t>(W) % 2 != 0 || reinterpret_cast<uintptr_t>(counts) % 4 != 0) return TW_EALIGN;
  }
  TW_TRY(tw::launch_reinit_rows(W, I, d, counts, seed, std_dev, n_reinit, as_stream(stream)));
  return TW_OK;
}

tw_status tw_fma_probe(float* out, int blocks, int iters, double* flops, void* stream) {
  if (blocks < 1 || iters < 1 || blocks > (1 << 20)) return TW_EINVAL;
  tw_status st = check_ptrs({out});
  if (st != TW_OK) return st;
  if (reinterpret_cast<uintptr_t>(out) % 4 != 0) return TW_EALIGN;
  if (flops != nullptr) *flops = static_cast<double>(tw::fma_probe_flops(blocks, iters));
  return from_cuda(tw::launch_fma_probe(out, blocks, iters, as_stream(stream)));
}

int tw_l2_gather_probe_blocks(int d) {
  if (d < 256 || d > 2048 || d % 256 != 0) return 0;
  return tw::l2_gather_probe_blocks(d);
}

tw_status tw_l2_gather_probe(const uint16_t* table, int rows, int d, const int32_t* idx, int n_idx, float* out,
                             int blocks, double* bytes, void* stream) {
  tw_status st = check_model_width(d);
  if (st != TW_OK) return st;
  if (rows < 1 || n_idx < 8 || n_idx % 8 != 0 || blocks < 1 || blocks > (1 << 20)) return TW_EINVAL;
  st = check_ptrs({table, idx, out});
  if (st != TW_OK) return st;
  if (bytes != nullptr) *bytes = static_cast<double>(n_idx) * d * 2.0;
  return from_cuda(tw::launch_l2_gather_probe(table, rows, d, idx, n_idx, out, blocks, as_stream(stream)));
}

tw_status tw_wait_timeout_probe(const uint16_t* A, const uint16_t* B, int M, int N, int K, int withhold_kb, float* D,
                                int32_t* dev_status, void* stream) {
  if (M < 1 || M > 128 || N < 64 || N > 256 || N % 64 != 0 || K < 64 || K % 64 != 0) return TW_EINVAL;
  if (withhold_kb < 0 || withhold_kb >= K / 64) return TW_EINVAL;
  tw_status st = check_ptrs({A, B, D, dev_status});
  if (st != TW_OK) return st;
  return from_cuda(tw::gemm_dense_test(A, B, M, N, K, 0, 0, D, dev_status, as_stream(stream), withhold_kb));
}

tw_status tw_dense_gemm(const uint16_t* A, const uint16_t* B, int M, int N, int K, int a_mn, int b_mn, float* D,
                        int32_t* dev_status, void* stream) {
  if (M < 1 || N < 1 || K < 1 || N % 64 != 0 || K % 64 != 0) return TW_EINVAL;
  if (a_mn && M % 64 != 0) return TW_EINVAL;
  tw_status st = check_ptrs({A, B, D, dev_status});
  if (st != TW_OK) return st;
  return from_cuda(tw::gemm_dense_test(A, B, M, N, K, a_mn, b_mn, D, dev_status, as_stream(stream)));
}

tw_status tw_dense_gemm_pair(const uint16_t* A, const uint16_t* B, int M, int N, int K, int a_mn, int b_mn, float* D,
                             int32_t* dev_status, void* stream) {
  if (M < 1 || N < 1 || K < 1 || N % 256 != 0 || K % 64 != 0) return TW_EINVAL;
  if (a_mn && M % 64 != 0) return TW_EINVAL;
  tw_status st = check_ptrs({A, B, D, dev_status});
  if (st != TW_OK) return st;
  return from_cuda(tw::gemm_dense_test(A, B, M, N, K, a_mn, b_mn, D, dev_status, as_stream(stream), -1, true));
}

tw_status tw_wait_timeout_probe_pair(const uint16_t* A, const uint16_t* B, int M, int N, int K, int withhold_kb,
                                     float* D, int32_t* dev_status, void* stream) {
  if (M < 1 || M > 256 || N != 256 || K < 64 || K % 64 != 0) return TW_EINVAL;
  if (withhold_kb < 0 || withhold_kb >= K / 64) return TW_EINVAL;
  tw_status st = check_ptrs({A, B, D, dev_status});
  if (st != TW_OK) return st;
  return from_cuda(tw::gemm_dense_test(A, B, M, N, K, 0, 0, D, dev_status, as_stream(stream), withhold_kb, true));
}

}  // extern "C"

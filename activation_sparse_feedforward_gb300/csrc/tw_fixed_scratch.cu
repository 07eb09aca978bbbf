// twell_ffn_fwd_fixed_scratch: the TwELL inference forward for callers that cannot
// allocate device memory.
//
// Some callers can only hand the library the buffers they already own: a plugin
// inside a host framework that passes its input and output pointers but no
// workspace, or a latency-critical serving loop where cudaMalloc is not allowed
// because it can synchronise the whole device and take milliseconds. This entry
// point gives them the same forward as twell_ffn_fwd with the scratch the dense
// overflow path needs (the gathered overflow rows and their hidden activations)
// taken from one fixed array in device memory that this file defines.
//
// The array is kFixedScratchBytes (20 MiB). Every GPU on which the library's code
// is loaded holds it until the process exits. Every call uses the same array, and
// the array keeps whatever the previous call left in it: nothing in it has to start
// at zero, because every byte the forward reads from its scratch is written earlier
// in the same call. Two calls whose work overlaps on the GPU (different streams,
// no ordering between them) race on the array.
//
// The array's device address is looked up once per device, in the context that is
// current on the first call (the CUDA runtime's primary context for that device),
// and kept for the life of the process. The call therefore assumes that every later
// call on that device runs in the same context, and that the device is not reset
// (cudaDeviceReset) in between: after a reset the kept address would point into a
// context that no longer exists.
#include <mutex>

#include "tw_internal.h"

namespace {

constexpr size_t kFixedScratchBytes = static_cast<size_t>(20) << 20;
constexpr int kMaxDevices = 64;

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

// The fixed scratch. In host code this name is only a host-side stand-in for the
// device array, never a device address: its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

extern "C" tw_status twell_ffn_fwd_fixed_scratch(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu,
                                                 const uint16_t* Wd, int T, int d, int I, int W, int C, int ovf_cap,
                                                 const tw_twell* tw_out, uint16_t* y, int32_t* dev_status,
                                                 void* stream) {
  // the arguments are checked as twell_ffn_fwd checks them, so a bad argument gets the
  // same error code from both entry points; then the size against the fixed array
  const tw_status st = tw::check_twell_fwd_operands(x, Wg, Wu, Wd, T, d, I, W, C, ovf_cap, tw_out, y, dev_status);
  if (st != TW_OK || T == 0) return st;
  if (twell_ffn_fwd_workspace_size(T, d, I, W, C, ovf_cap) > kFixedScratchBytes) return TW_EWORKSPACE;

  // one-time set-up per device, with that device current: look up the device
  // address of the fixed array
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TW_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return TW_EUNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_fixed_scratch) != cudaSuccess || p == nullptr) return TW_ECUDA;
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  return twell_ffn_fwd(x, Wg, Wu, Wd, T, d, I, W, C, ovf_cap, tw_out, scratch, kFixedScratchBytes, y, dev_status,
                       stream);
}

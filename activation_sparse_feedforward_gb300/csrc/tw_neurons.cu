// Per-neuron activity counts of a Hybrid training forward and the dead-neuron
// re-initialisation of the gate projection (thelatestinai listing, Table 5 "Dead
// neuron reinit." and Figure 8; wispaper blog "Critical Analysis & Conclusion").
//
//  counts   counts[j] += number of tokens whose activation a_tj is nonzero: one
//           atomic per ELL entry (warp per token), and for the dense backup rows one
//           column sum per neuron (thread per neuron, rows in order) and one atomic.
//  reinit   every row j of W with counts[j] == 0 is redrawn: element (j, k) is
//           std * z, z = sum of twelve uniforms minus 6 (Irwin-Hall), the uniforms
//           being the top 24 bits of SplitMix64 outputs 12 (j d + k) + i, i < 12, of a
//           generator seeded with `seed` (counter form: state = seed + (c + 1) gamma).
//           z is exact in float64; w = float32(float64(std) z) is rounded to bf16.
#include <algorithm>

#include "tw_common.cuh"
#include "tw_internal.h"

namespace tw {

namespace {

TW_DEV uint64_t splitmix64_at(uint64_t seed, uint64_t counter) {
  uint64_t z = seed + (counter + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

}  // namespace

__global__ void __launch_bounds__(256) neuron_counts_kernel(const int32_t* __restrict__ ell_nnz,
                                                            const uint16_t* __restrict__ ell_idx, int T, int R,
                                                            const float* __restrict__ backup_a,
                                                            const int32_t* __restrict__ n_backup, int cap, int I,
                                                            int token_blocks, int32_t* __restrict__ counts) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  if (static_cast<int>(blockIdx.x) < token_blocks) {
    for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += token_blocks * wpb) {
      int n = ell_nnz[t];
      if (!TW_CHECKED(n >= 0 && n <= R, nullptr)) n = 0;
      for (int e = lane; e < n; e += 32) {
        const int j = ell_idx[static_cast<size_t>(t) * R + e];
        if (TW_CHECKED(j < I, nullptr)) atomicAdd(counts + j, 1);
      }
    }
  } else if (backup_a != nullptr) {
    const int nb = min(max(*n_backup, 0), cap);
    const int nblk = gridDim.x - token_blocks;
    for (int j = (blockIdx.x - token_blocks) * blockDim.x + threadIdx.x; j < I; j += nblk * blockDim.x) {
      int c = 0;
      for (int s = 0; s < nb; ++s) c += backup_a[static_cast<size_t>(s) * I + j] > 0.f ? 1 : 0;
      if (c) atomicAdd(counts + j, c);
    }
  }
}

__global__ void __launch_bounds__(256) reinit_rows_kernel(uint16_t* __restrict__ W, int I, int d,
                                                          const int32_t* __restrict__ counts, uint64_t seed,
                                                          float stdv, int32_t* __restrict__ n_reinit) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int j = blockIdx.x * wpb + (threadIdx.x >> 5); j < I; j += gridDim.x * wpb) {
    if (counts[j] != 0) continue;
    if (lane == 0) atomicAdd(n_reinit, 1);
    for (int k = lane; k < d; k += 32) {
      const uint64_t base = (static_cast<uint64_t>(j) * static_cast<uint64_t>(d) + static_cast<uint64_t>(k)) * 12ull;
      long long total = 0;
#pragma unroll
      for (int i = 0; i < 12; ++i) total += static_cast<long long>(splitmix64_at(seed, base + i) >> 40);
      const double z = static_cast<double>(total) * (1.0 / 16777216.0) - 6.0;
      const float w = static_cast<float>(static_cast<double>(stdv) * z);
      W[static_cast<size_t>(j) * d + k] = f32_to_bf16(w);
    }
  }
}

cudaError_t launch_neuron_counts(const tw_hybrid& h, int32_t* counts, cudaStream_t s) {
  const int token_blocks = std::max(1, std::min((h.T + 7) / 8, device_sm_count() * 4));
  const int backup_blocks = h.backup_cap > 0 ? std::max(1, std::min((h.I + 255) / 256, device_sm_count())) : 0;
  if (h.T == 0) return cudaSuccess;
  cudaError_t e = launch(neuron_counts_kernel, dim3(token_blocks + backup_blocks), dim3(256), 0, s,
                         static_cast<const int32_t*>(h.ell_nnz), static_cast<const uint16_t*>(h.ell_idx), h.T, h.R,
                         static_cast<const float*>(h.backup_cap > 0 ? h.backup_a : nullptr),
                         static_cast<const int32_t*>(h.n_backup), h.backup_cap, h.I, token_blocks, counts);
  trace_mark(s, "neuron_counts");
  return e;
}

cudaError_t launch_reinit_rows(uint16_t* W, int I, int d, const int32_t* counts, uint64_t seed, float stdv,
                               int32_t* n_reinit, cudaStream_t s) {
  cudaError_t e = launch_zero(n_reinit, sizeof(int32_t), nullptr, 0, s);
  if (e != cudaSuccess || I == 0) return e;
  const int grid = std::max(1, std::min((I + 7) / 8, device_sm_count() * 4));
  e = launch(reinit_rows_kernel, dim3(grid), dim3(256), 0, s, W, I, d, counts, seed, stdv, n_reinit);
  trace_mark(s, "reinit_rows");
  return e;
}

}  // namespace tw

// Persistent tcgen05 GEMM for sm_103a:  D[M, N] = sum over segments of A_s B_s
// (bf16 operands, fp32 accumulation in TMEM), with a pluggable epilogue that reads
// the accumulator straight out of TMEM.
//
//  * Warp 0 (one lane) streams A and B tiles into a STAGES-deep shared-memory ring
//    with TMA (cp.async.bulk.tensor, 128-byte swizzle), signalling mbarriers.
//  * Warp 1 allocates TMEM; one lane issues tcgen05.mma (M = 128, N = BN, K = 16)
//    into one of two accumulator buffers and commits each ring slot back to the
//    producer when its MMAs retire.
//  * Warps 2-5 (128 threads, one accumulator row each) run the epilogue of tile i
//    while the MMAs of tile i + 1 fill the other TMEM buffer. An epilogue that does
//    much per element (kSplitColumns) gets eight warps on 256-wide tiles: two per
//    TMEM lane quarter, each taking one half of the tile's columns.
//
// A is [M, K] with K contiguous ("K-major") or stored [K, M] ("MN-major"); the same
// for B with N in place of M. DUAL issues a second MMA with a second B operand into
// its own accumulator (gate and up projections of the same rows in one pass).
// `segments == S` continues the K loop over S (A, B) pairs into the same
// accumulator: a second product (dx = dG Wg + dU Wu) or the low half of an operand
// split into two bf16 parts (x = hi + lo) to keep fp32-level precision.
// `problems == P` runs P products of the same shape in one launch, their row tiles
// one after the other (the backup rows' two or three weight gradients), so the
// tiles of all of them share the persistent grid. M and K may be read from device
// memory (counts produced by earlier kernels in the stream), so the launch does not
// need them on the host.
//
// PAIR runs the same roles on clusters of two CTAs with the two-SM MMA
// (tcgen05.mma.cta_group::2, M = 256): each CTA stages its own 128 rows of A and half
// of the B tile, rank 0's MMA thread issues for both, and each CTA's epilogue reads its
// own 128 accumulator rows. Per MMA a CTA's shared memory serves 128 + BN / 2 operand
// rows instead of 128 + BN; at BN = 256 the single-CTA form asks more of shared memory
// (operand reads plus TMA writes) than one SM delivers at the tensor rate.
#pragma once

#include <type_traits>

#include "tw_common.cuh"

namespace tw {

constexpr int GEMM_BM = 128;
constexpr int GEMM_BK = 64;
// per-warp transpose buffer of the fp32 row epilogues (`transposed_rows`): 32 rows of
// kEpiStageStride floats, for each of the four epilogue warps
constexpr int kEpiStageStride = 36;
constexpr int kEpiTransposeBytes = 4 * 32 * kEpiStageStride * 4;

struct GemmShape {
  int M;             // rows of D when m_dev == nullptr
  const int* m_dev;  // optional device row count, clamped to [0, m_cap]
  int m_cap;
  int N;             // multiple of BN
  int K;             // reduction length when k_dev == nullptr
  const int* k_dev;  // optional device K, clamped to [0, k_cap]; memory past K must read as zero
  int k_cap;
  int segments;      // (A, B) pairs summed into each output tile
  int problems;      // 1, or several products of the same shape in one launch: problem
                     // p reads maps a/b[p * segments + s]; its row tiles follow the
                     // previous problem's (the epilogue sees rows p * m_tiles * 128 + m)
  int ksplit;        // >= 1: each output tile's K loop is cut into ksplit work units
                     // (only for epilogues that accumulate, e.g. EpiRedF32); -1:
                     // chosen on the device from the actual tile count so that the
                     // units fill the grid once (grid / tiles slices per tile); -2:
                     // chosen on the device by split_by_cost (for tile counts near
                     // the SM count, where whole rounds of units matter)
  int32_t* status;
  int withhold_kb;   // test hook, -1 normally: in a CTA's first work unit, the TMA loads of
                     // this K block are never issued, so the MMA issuer's bounded wait for
                     // that stage runs out (TW_ETIMEOUT) and every role drains and returns
  const int* route_dev;  // optional: the launch does its work only when *route_dev == route_want
  int route_want;        // (the route a call took, decided on the device by an earlier kernel)
  const int* drop_last_problem_if;  // optional: when it reads 1, the launch runs one problem fewer
  bool split_tail;   // tiles of the last round, when they fill at most half the grid, run as
                     // two half-width units each (launches without a K split, BN >= 128)
};

constexpr int GEMM_MAX_SEGMENTS = 6;  // segments x problems

// Tensor maps of every operand: segment s of problem p reads a[p * segments + s] and
// b[p * segments + s]; the DUAL form reads b[0] and b[1] against a[0].
struct GemmMaps {
  CUtensorMap a[GEMM_MAX_SEGMENTS];
  CUtensorMap b[GEMM_MAX_SEGMENTS];
};

// An epilogue that reads global memory for its tile may define prefetch(BN); the
// epilogue warps call it before they wait for the tile's accumulator, so the reads
// overlap the K loop.
template <class E, class = void>
struct epi_prefetches : std::false_type {};
template <class E>
struct epi_prefetches<E, std::void_t<decltype(&E::prefetch)>> : std::true_type {};
// An epilogue with kOverlapLoads = true (single accumulator only) has each chunk's
// TMEM load issued before the previous chunk is written out, at the cost of a
// second 32-register buffer.
template <class E, class = void>
struct epi_overlaps_loads : std::false_type {};
template <class E>
struct epi_overlaps_loads<E, std::void_t<decltype(E::kOverlapLoads)>> : std::bool_constant<E::kOverlapLoads> {};

// An epilogue wrapped in F16Operands<> runs its GEMM on fp16 operands (A and B both
// fp16; the tensor maps copy the bits as they are): the dense route's backward, whose
// operands need 11 significant bits.
template <class E, class = void>
struct epi_f16_operands : std::false_type {};
template <class E>
struct epi_f16_operands<E, std::void_t<decltype(E::kF16Operands)>> : std::bool_constant<E::kF16Operands> {};

// An epilogue with kSplitColumns = true runs on eight warps when BN == 256 (each warp
// sees an epilogue object over its 128 columns); the others on four. kStageBytes is
// an epilogue's staging for four warps, so eight warps take twice as much.
template <class E, class = void>
struct epi_splits : std::false_type {};
template <class E>
struct epi_splits<E, std::void_t<decltype(E::kSplitColumns)>> : std::bool_constant<E::kSplitColumns> {};
template <int BN, class Epi>
__host__ __device__ constexpr int epi_warps() {
  return (epi_splits<Epi>::value && BN == 256) ? 8 : 4;
}
template <int BN, class Epi>
__host__ __device__ constexpr int gemm_threads() {
  return 64 + 32 * epi_warps<BN, Epi>();
}

// NA = 2 pairs the segments: segments 2i and 2i + 1 share one B operand (b[2i]), so
// a stage holds both A tiles and one B tile, and both products go into the same
// accumulator (the hi / lo halves of a split fp32 operand against one weight).
// PAIR runs the GEMM on CTA pairs (clusters of two, cta_group::2 MMAs): a unit is a
// 256-row tile, each CTA loads its 128 A rows and BN / 2 of the tile's B rows, and
// the pair's shared-memory operand traffic per FLOP is two thirds of a single CTA's
// at BN = 256, below what one SM's shared memory delivers at the MMA rate.
template <int BN, bool A_MN, bool B_MN, bool DUAL, int STAGES, int NA = 1, bool F16 = false, bool PAIR = false>
struct GemmTraits {
  static constexpr int NB = DUAL ? 2 : 1;
  static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // B rows (N) of a stage in one CTA
  static constexpr int B_BYTES = B_ROWS * GEMM_BK * 2;
  static constexpr int STAGE_BYTES = NA * A_BYTES + NB * B_BYTES;
  static constexpr int ACC_COLS = BN * NB;
  static constexpr int TMEM_COLS = 2 * ACC_COLS;
  static constexpr int UNIT_ROWS = PAIR ? 2 * GEMM_BM : GEMM_BM;
  static constexpr uint32_t IDESC = idesc_bf16_f32(UNIT_ROWS, BN, A_MN, B_MN, F16);
  static constexpr uint32_t IDESC_HALF = idesc_bf16_f32(UNIT_ROWS, BN / 2, A_MN, B_MN, F16);  // half-width units
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + BAR_BYTES;
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be 64, 128, 192 or 256");
  static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation must be a power of two");
  static_assert((2 * STAGES + 4) * 8 + 8 <= BAR_BYTES, "barrier area");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(NA == 1 || (NA == 2 && !DUAL), "paired A segments take one B operand");
  static_assert(!PAIR || (!DUAL && NA == 1 && BN >= 128), "CTA pairs: one B operand, one A tile, BN >= 128");
};

// The K split of a launch whose units are handed out to `grid` CTAs in rounds: the
// number of slices s (at most 16) that minimises rounds x (K blocks a unit + 2), the
// 2 standing for a unit's fixed cost (pipeline fill, the accumulator's drain and its
// fp32 reductions). Every thread computes the same value.
TW_DEV int split_by_cost(int tiles, int kb_total, int grid) {
  if (tiles <= 0 || kb_total <= 0) return 1;
  int best = 1;
  long best_cost = -1;
  for (int s = 1; s <= min(kb_total, 16); ++s) {
    const long chunk = (kb_total + s - 1) / s;
    const long rounds = (static_cast<long>(tiles) * s + grid - 1) / grid;
    const long cost = rounds * (chunk + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// A work unit: an output tile (or, with the tail split, a half of one: half 0 or 1, the
// columns [0, BN/2) or [BN/2, BN) of the tile; -1 = the whole tile) and the slice of
// its K loop. Units [0, full_units) are whole tiles cut into ksplit slices each; with
// the tail split, the units after them are the last tiles' halves (ksplit == 1).
struct UnitInfo {
  int tile, kb_lo, kb_hi, half;
};
TW_DEV UnitInfo unit_info(int unit, int ksplit, int kb_chunk, int kb_total, int full_units) {
  UnitInfo u;
  if (unit < full_units) {
    u.tile = unit / ksplit;
    u.kb_lo = (unit - u.tile * ksplit) * kb_chunk;
    u.kb_hi = min(kb_total, u.kb_lo + kb_chunk);
    u.half = -1;
  } else {
    const int h = unit - full_units;
    u.tile = full_units + h / 2;
    u.kb_lo = 0;
    u.kb_hi = kb_total;
    u.half = h & 1;
  }
  return u;
}

template <int BN, bool A_MN, bool B_MN, bool DUAL, int STAGES, class Epi, int NA = 1, bool PAIR = false>
__global__ void __launch_bounds__(gemm_threads<BN, Epi>(), 1)
    gemm_tc_kernel(const __grid_constant__ GemmMaps maps, const GemmShape shape,
                   const __grid_constant__ typename Epi::Params ep) {
  using Tr = GemmTraits<BN, A_MN, B_MN, DUAL, STAGES, NA, epi_f16_operands<Epi>::value, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* tiles = smem_raw + pad;
  uint64_t* full = reinterpret_cast<uint64_t*>(tiles + STAGES * Tr::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;   // [2] accumulator ready for the epilogue
  uint64_t* tempty = tfull + 2;       // [2] accumulator drained by the epilogue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pairs: rank 0 issues the MMAs and owns the "full" and "accumulator empty"
  // barriers both CTAs signal; each CTA's own "empty" and "accumulator full" barriers
  // get the MMA commits of rank 0 (multicast)
  const uint32_t rank = PAIR ? cluster_rank() : 0u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, (PAIR ? 2 : 1) * epi_warps<BN, Epi>());
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int sgi = 0; sgi < shape.segments * max(1, shape.problems); ++sgi) {
      tma_prefetch_desc(&maps.a[sgi]);
      tma_prefetch_desc(&maps.b[sgi]);
    }
    if (DUAL) tma_prefetch_desc(&maps.b[1]);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, Tr::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, Tr::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers and TMEM exist before either signals the other
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  pdl_enter();  // the setup above overlaps the previous kernel's tail

  int M = shape.M;
  if (shape.m_dev != nullptr) M = min(max(*shape.m_dev, 0), shape.m_cap);
  int K = shape.K;
  if (shape.k_dev != nullptr) K = min(max(*shape.k_dev, 0), shape.k_cap);
  if (shape.route_dev != nullptr && *shape.route_dev != shape.route_want) K = 0;  // not this call's route: no work
  const int m_tiles = (M + Tr::UNIT_ROWS - 1) / Tr::UNIT_ROWS;
  const int n_tiles = shape.N / BN;
  const int problems = max(1, shape.problems) -
                       ((shape.drop_last_problem_if != nullptr && *shape.drop_last_problem_if == 1) ? 1 : 0);
  const int num_tiles = (K > 0) ? problems * m_tiles * n_tiles : 0;
  const int kb_per_seg = (K + GEMM_BK - 1) / GEMM_BK;
  const int kb_total = kb_per_seg * (shape.segments / NA);  // one K step covers NA segments
  // work unit = (output tile, slice of its K loop); empty slices are skipped by
  // every role alike
  // units are handed out per CTA, or per pair
  const int grid = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int first_unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int ksplit = PAIR                ? 1
                     : shape.ksplit >= 0 ? max(1, shape.ksplit)
                     : shape.ksplit == -2 ? split_by_cost(num_tiles, kb_total, grid)
                                          : (num_tiles > 0 ? max(1, min(kb_total, grid / num_tiles)) : 1);
  const int kb_chunk = (kb_total + ksplit - 1) / ksplit;
  // the tail split: the last round's tiles as two half-width units each, when they fill
  // at most half the grid (so the last round takes half a tile's time)
  const int rem = num_tiles % grid;
  // (not on CTA pairs: half-width pair units, measured at T 8192, were slower than whole ones)
  const bool tail =
      !PAIR && shape.split_tail && !DUAL && BN >= 128 && ksplit == 1 && rem > 0 && 2 * rem <= grid;
  const int full_units = tail ? num_tiles - rem : num_tiles * ksplit;
  const int num_units = tail ? full_units + 2 * rem : num_tiles * ksplit;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      bool ok = true;
      for (int unit = first_unit; ok && unit < num_units; unit += grid) {
        const UnitInfo ui = unit_info(unit, ksplit, kb_chunk, kb_total, full_units);
        const int tile = ui.tile, kb_lo = ui.kb_lo, kb_hi = ui.kb_hi;
        if (kb_lo >= kb_hi) continue;
        const int row_tile = tile / n_tiles;
        const int prob = row_tile / m_tiles;
        // within the problem; a pair's rank 1 loads the unit's second 128 rows
        const int m0 = (row_tile - prob * m_tiles) * Tr::UNIT_ROWS + static_cast<int>(rank) * GEMM_BM;
        // a second half's B box starts at its own columns (the box's other half, past
        // the tile or past N, is loaded but not used); a pair's ranks load one half of
        // the B tile each
        const int n0 = (tile % n_tiles) * BN + (ui.half == 1 ? BN / 2 : 0) + static_cast<int>(rank) * Tr::B_ROWS;
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait(empty + stage, phase ^ 1u, abort_flag, shape.status)) {
            ok = false;
            break;
          }
          if (kb == shape.withhold_kb && unit == first_unit) {
            // test hook: this stage is never filled (its "full" barrier gets no arrival)
            ++issued;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          uint8_t* sA = tiles + stage * Tr::STAGE_BYTES;
          uint8_t* sB = sA + NA * Tr::A_BYTES;
          const int grp = kb / kb_per_seg;
          const int seg = grp * NA;
          const int k0 = (kb - grp * kb_per_seg) * GEMM_BK;
          const CUtensorMap* tb = &maps.b[prob * shape.segments + seg];
          // a pair's loads all complete on rank 0's barrier, which expects both CTAs' bytes
          if (rank == 0) mbar_arrive_expect_tx(full + stage, (PAIR ? 2 : 1) * Tr::STAGE_BYTES);
          const uint32_t fbar = PAIR ? peer_smem_addr(full + stage, 0) : 0u;
          auto load = [&](uint8_t* dst, const CUtensorMap* map, int c0, int c1) {
            if constexpr (PAIR)
              tma_load_2d_pair(dst, map, fbar, c0, c1);
            else
              tma_load_2d(dst, map, full + stage, c0, c1);
          };
#pragma unroll
          for (int na = 0; na < NA; ++na) {
            const CUtensorMap* ta = &maps.a[prob * shape.segments + seg + na];
            uint8_t* dA = sA + na * Tr::A_BYTES;
            if (!A_MN) {
              load(dA, ta, k0, m0);
            } else {
              load(dA, ta, m0, k0);
              load(dA + 8192, ta, m0 + 64, k0);
            }
          }
#pragma unroll
          for (int nb = 0; nb < Tr::NB; ++nb) {
            const CUtensorMap* tbb = (nb == 0) ? tb : &maps.b[1];
            uint8_t* dst = sB + nb * Tr::B_BYTES;
            if (!B_MN) {
              load(dst, tbb, k0, n0);
            } else {
#pragma unroll
              for (int c = 0; c < Tr::B_ROWS / 64; ++c) load(dst + c * 8192, tbb, n0 + c * 64, k0);
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && rank == 0) {
        // let the loads already issued land before the CTA can exit (a pair's rank 1
        // loads complete on rank 0's barriers, which rank 0 drains; rank 1 stays until
        // rank 0 reaches the closing cluster barrier)
        for (long i = 0; i < STAGES && i < issued; ++i) {
          const long q = issued - 1 - i;
          mbar_wait_drain(full + (q % STAGES), static_cast<uint32_t>((q / STAGES) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      bool issued_any = false;
      for (int unit = first_unit; ok && unit < num_units; unit += grid) {
        const UnitInfo ui = unit_info(unit, ksplit, kb_chunk, kb_total, full_units);
        const int kb_lo = ui.kb_lo, kb_hi = ui.kb_hi;
        if (kb_lo >= kb_hi) continue;
        const uint32_t idesc = ui.half < 0 ? Tr::IDESC : Tr::IDESC_HALF;
        const int buf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        ++local;
        if (!mbar_wait(tempty + buf, (use & 1u) ^ 1u, abort_flag, shape.status)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(buf * Tr::ACC_COLS);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait(full + stage, phase, abort_flag, shape.status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_base = smem_addr(tiles + stage * Tr::STAGE_BYTES);
          const uint32_t b_base = a_base + NA * Tr::A_BYTES;
#pragma unroll
          for (int k16 = 0; k16 < GEMM_BK / 16; ++k16) {
#pragma unroll
            for (int na = 0; na < NA; ++na) {
              const uint32_t ab = a_base + na * Tr::A_BYTES;
              const uint64_t ad = A_MN ? smem_desc_sw128(ab + k16 * 2048, 8192, 1024)
                                       : smem_desc_sw128(ab + k16 * 32, 16, 1024);
              const uint32_t acc = (kb > kb_lo || k16 > 0 || na > 0) ? 1u : 0u;
#pragma unroll
              for (int nb = 0; nb < Tr::NB; ++nb) {
                const uint32_t bb = b_base + nb * Tr::B_BYTES;
                const uint64_t bd = B_MN ? smem_desc_sw128(bb + k16 * 2048, 8192, 1024)
                                         : smem_desc_sw128(bb + k16 * 32, 16, 1024);
                if constexpr (PAIR)
                  tc_mma_bf16_pair(d0 + nb * BN, ad, bd, idesc, acc);
                else
                  tc_mma_bf16(d0 + nb * BN, ad, bd, idesc, acc);
              }
            }
          }
          issued_any = true;
          if constexpr (PAIR)
            tc_commit_pair(empty + stage);
          else
            tc_commit(empty + stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          tc_commit_pair(tfull + buf);
        else
          tc_commit(tfull + buf);
      }
      if (!ok && issued_any) {
        // wait for MMAs in flight before TMEM is released: the commit completes the
        // current phase of this ring slot's "empty" barrier (parity == phase)
        uint64_t* drain = empty + stage;
        if constexpr (PAIR)
          tc_commit_pair(drain);
        else
          tc_commit(drain);
        mbar_wait_drain(drain, phase);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    constexpr int kEW = epi_warps<BN, Epi>();
    constexpr int kCols = BN * 4 / kEW;  // the columns of the tile one epilogue warp takes
    const int ew = warp - 2;
    const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter + 32)
    const int half = ew >> 2;      // which kCols columns of the tile (0 with four warps)
    const int row = quarter * 32 + lane;
    int local = 0;
    for (int unit = first_unit; unit < num_units; unit += grid) {
      const UnitInfo ui = unit_info(unit, ksplit, kb_chunk, kb_total, full_units);
      if (ui.kb_lo >= ui.kb_hi) continue;
      const int tile = ui.tile;
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      ++local;
      const int m = (tile / n_tiles) * Tr::UNIT_ROWS + static_cast<int>(rank) * GEMM_BM + row;
      // this warp's columns: kCols at half * kCols of a whole tile; of a half unit, its
      // BN / 2 columns (with eight warps all of them for the first group's warps, none
      // for the second's), at the start of the accumulator
      int cols = kCols, col_off = half * kCols;
      if (ui.half >= 0) {
        cols = (kEW == 8) ? (half == 0 ? kCols : 0) : kCols / 2;
        col_off = 0;
      }
      const int n0 = (tile % n_tiles) * BN + (ui.half == 1 ? BN / 2 : 0) + col_off;
      Epi e(ep, m, M, n0);
      if constexpr (epi_prefetches<Epi>::value)
        if (cols > 0) e.prefetch(cols);  // while the tile's K loop runs
      int ok = 0;
      if (lane == 0) ok = mbar_wait(tfull + buf, use & 1u, abort_flag, shape.status) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      if constexpr (Epi::kStageBytes > 0)
        e.stage = reinterpret_cast<float*>(tiles + STAGES * Tr::STAGE_BYTES + Tr::BAR_BYTES) + ew * (Epi::kStageBytes / 16);
      const uint32_t tbase = tmem_base + static_cast<uint32_t>(buf * Tr::ACC_COLS + col_off) +
                             (static_cast<uint32_t>(quarter * 32) << 16);
      const int nch = cols / 32;
      if constexpr (!DUAL && epi_overlaps_loads<Epi>::value) {
        // the next chunk's TMEM load is in flight while this chunk is written out
        if (nch > 0) {
          uint32_t va[32], vb[32];
          tmem_ld32(tbase, va);
          tmem_wait_ld();
#pragma unroll 1
          for (int c = 0; c < nch; c += 2) {
            if (c + 1 < nch) tmem_ld32(tbase + (c + 1) * 32, vb);
            e.chunk(c, va, va);
            tmem_wait_ld();
            if (c + 1 < nch) {
              if (c + 2 < nch) tmem_ld32(tbase + (c + 2) * 32, va);
              e.chunk(c + 1, vb, vb);
              tmem_wait_ld();
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          uint32_t v0[32];
          uint32_t v1[32];
          tmem_ld32(tbase + c * 32, v0);
          if (DUAL) tmem_ld32(tbase + BN + c * 32, v1);
          tmem_wait_ld();
          e.chunk(c, v0, v1);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR)
          mbar_arrive_cluster(peer_smem_addr(tempty + buf, 0));  // rank 0's MMA issuer waits for both CTAs
        else
          mbar_arrive(tempty + buf);
      }
      e.finish();
    }
  }

  __syncthreads();
  // a pair's CTAs leave together: no signal or MMA write of one may reach the other
  // after it has released its TMEM or exited
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after_sync();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, Tr::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, Tr::TMEM_COLS);
  }
}

// ======================================================================= epilogues
// Bulk tensor stores from shared memory (TMA, async proxy). The issuing thread
// commits its stores as one bulk group and later waits for them: `_read` until the
// shared-memory sources have been read (the buffer may be rewritten), the plain form
// until the global writes are done.
TW_DEV void tma_store_2d(const CUtensorMap* map, const void* smem_src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(smem_src)), "r"(c0), "r"(c1)
               : "memory");
}
TW_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
TW_DEV void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
TW_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
TW_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Row-to-column transpose through shared memory for epilogues that write fp32 rows:
// each epilogue warp holds 32 accumulator rows (one per lane) x 32 columns. Each lane
// writes its row as eight 16-byte vectors; the warp then reads back four rows per
// step, eight lanes per row, so one 16-byte-per-lane instruction covers four whole
// 128-byte row segments instead of 16 bytes in each of 32 rows. The buffer is
// 32 x 36 floats per warp: with a row stride of 36 floats, every group of eight
// lanes touches all 32 banks once in both phases. `put(r, c4, x)` stores the four
// columns 4 c4 .. 4 c4 + 3 of output row r; rows at or past M are skipped. Every
// lane of the warp must call it.
template <class Put>
TW_DEV void transposed_rows(float* stage, const uint32_t (&v)[32], int m, int M, Put put) {
  const int lane = threadIdx.x & 31;
  float4* mine = reinterpret_cast<float4*>(stage + lane * kEpiStageStride);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    mine[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                          __uint_as_float(v[4 * i + 3]));
  __syncwarp();
  const int m0 = m - lane;  // the warp's first row
  const int sub = lane >> 3, c4 = lane & 7;
#pragma unroll
  for (int r0 = 0; r0 < 32; r0 += 4) {
    const int r = r0 + sub;
    if (m0 + r < M) put(m0 + r, c4, *reinterpret_cast<const float4*>(stage + r * kEpiStageStride + 4 * c4));
  }
  __syncwarp();
}

// The 16-bit counterpart for one 32-column output block: the lane's row arrives as 16
// packed words (two columns each); the warp then writes eight rows per step, four
// lanes x 16 bytes covering each row's 64-byte segment. Rows m0 + r with r < rows
// are written to dst + (m0 + r) * ld. In the staging buffer a row is 16 words and
// its four 16-byte chunks are XOR-swizzled by (row / 2) mod 4, so both the lanes'
// row writes and the quarter-warps' two-row reads touch every bank once: the
// epilogue's shared-memory traffic competes with the MMAs' operand reads. Every lane
// of the warp must call it.
TW_DEV void transposed_rows_bf16(float* stage, const uint32_t (&w)[16], int m0, int rows, uint16_t* dst, int ld) {
  const int lane = threadIdx.x & 31;
  uint32_t* st = reinterpret_cast<uint32_t*>(stage);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<uint4*>(st + lane * 16 + 4 * ((i ^ (lane >> 1)) & 3)) =
        make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  __syncwarp();
  const int sub = lane >> 2, c4 = lane & 3;
#pragma unroll
  for (int r0 = 0; r0 < 32; r0 += 8) {
    const int r = r0 + sub;
    if (r < rows)
      *reinterpret_cast<uint4*>(dst + static_cast<size_t>(m0 + r) * ld + 8 * c4) =
          *reinterpret_cast<const uint4*>(st + r * 16 + 4 * ((c4 ^ (r >> 1)) & 3));
  }
  __syncwarp();
}

// Each epilogue object lives in one thread for one tile: it owns accumulator row m
// (valid when m < M) and columns [n0, n0 + BN), delivered 32 columns at a time.

// D[m][n] = acc (fp32), row stride ldd.
struct EpiStoreF32 {
  static constexpr int kStageBytes = kEpiTransposeBytes;
  static constexpr bool kOverlapLoads = true;
  struct Params {
    float* D;
    int ldd;
  };
  const Params& p;
  int m, M, n0;
  float* stage = nullptr;  // this warp's transpose buffer
  TW_DEV EpiStoreF32(const Params& p_, int m_, int M_, int n0_) : p(p_), m(m_), M(M_), n0(n0_) {}
  TW_DEV void chunk(int c, const uint32_t (&v)[32], const uint32_t (&)[32]) {
    float* col = p.D + n0 + c * 32;
    transposed_rows(stage, v, m, M, [&](int r, int c4, float4 x) {
      reinterpret_cast<float4*>(col + static_cast<size_t>(r) * p.ldd)[c4] = x;
    });
  }
  TW_DEV void finish() {}
};

// EpiStoreF32 for a grouped launch: row m of the stacked tiles belongs to problem
// m / rows_per_problem and is row m % rows_per_problem of that problem's D.
struct EpiStoreF32Grouped {
  static constexpr int kStageBytes = kEpiTransposeBytes;
  static constexpr bool kOverlapLoads = true;
  static constexpr int kMaxProblems = 3;
  struct Params {
    float* D[kMaxProblems];
    int ldd;
    int rows_per_problem;  // the problem's row tiles x 128
  };
  const Params& p;
  int m, M, n0;
  float* stage = nullptr;  // this warp's transpose buffer
  TW_DEV EpiStoreF32Grouped(const Params& p_, int m_, int M_, int n0_) : p(p_), m(m_), M(M_), n0(n0_) {}
  TW_DEV void chunk(int c, const uint32_t (&v)[32], const uint32_t (&)[32]) {
    const int prob = m / p.rows_per_problem;  // the same for the warp's 32 rows
    float* col = p.D[prob] + n0 + c * 32;
    transposed_rows(stage, v, m - prob * p.rows_per_problem, M, [&](int r, int c4, float4 x) {
      reinterpret_cast<float4*>(col + static_cast<size_t>(r) * p.ldd)[c4] = x;
    });
  }
  TW_DEV void finish() {}
};

// D_p[m][n] = acc (fp32), or ReLU(acc) for the problems whose bit is set in relu, for a
// grouped launch over a device row count M (problem p's row tiles follow problem
// p - 1's, M rounded up to whole units of unit_rows each: 128, or 256 on CTA pairs);
// rows at or past M are skipped.
struct EpiStoreF32RowsGrouped {
  static constexpr int kStageBytes = kEpiTransposeBytes;
  static constexpr bool kOverlapLoads = true;
  static constexpr int kMaxProblems = 2;
  struct Params {
    float* D[kMaxProblems];
    int ldd;
    unsigned relu;
    int unit_rows;
  };
  const Params& p;
  int m, M, n0;
  float* stage = nullptr;  // this warp's transpose buffer
  TW_DEV EpiStoreF32RowsGrouped(const Params& p_, int m_, int M_, int n0_) : p(p_), m(m_), M(M_), n0(n0_) {}
  TW_DEV void chunk(int c, const uint32_t (&v)[32], const uint32_t (&)[32]) {
    const int rows_per_problem = (M + p.unit_rows - 1) / p.unit_rows * p.unit_rows;
    const int prob = m / rows_per_problem;  // the same for the warp's 32 rows
    if (prob >= kMaxProblems) return;       // uniform over the warp
    uint32_t w[32];
    const bool relu = (p.relu >> prob) & 1u;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float x = __uint_as_float(v[i]);
      w[i] = __float_as_uint(relu ? (x > 0.f ? x : 0.f) : x);
    }
    float* col = p.D[prob] + n0 + c * 32;
    transposed_rows(stage, w, m - prob * rows_per_problem, M, [&](int r, int c4, float4 x) {
      reinterpret_cast<float4*>(col + static_cast<size_t>(r) * p.ldd)[c4] = x;
    });
  }
  TW_DEV void finish() {}
};

// Any epilogue, with its GEMM run on fp16 operands.
template <class E>
struct F16Operands : E {
  static constexpr bool kF16Operands = true;
  using E::E;
};

// EpiStoreF32Grouped that adds instead of storing when *add_if (a device count, read
// once a thread) is positive: the dense route's weight gradients, added to the dense
// backup rows' part when there are backup rows, else written.
struct EpiF32GroupedStoreOrAdd {
  static constexpr int kStageBytes = kEpiTransposeBytes;
  static constexpr bool kOverlapLoads = true;
  static constexpr int kMaxProblems = 3;
  struct Params {
    float* D[kMaxProblems];
    int ldd;
    int rows_per_problem;  // the problem's rows rounded up to whole units (256 rows on CTA pairs)
    const int32_t* add_if;
  };
  const Params& p;
  int m, M, n0;
  bool add;
  float* stage = nullptr;
  TW_DEV EpiF32GroupedStoreOrAdd(const Params& p_, int m_, int M_, int n0_)
      : p(p_), m(m_), M(M_), n0(n0_), add(p_.add_if != nullptr && *p_.add_if > 0) {}
  TW_DEV void chunk(int c, const uint32_t (&v)[32], const uint32_t (&)[32]) {
    const int prob = m / p.rows_per_problem;
    float* col = p.D[prob] + n0 + c * 32;
    transposed_rows(stage, v, m - prob * p.rows_per_problem, M, [&](int r, int c4, float4 x) {
      float4* dst = reinterpret_cast<float4*>(col + static_cast<size_t>(r) * p.ldd) + c4;
      if (add)
        atomicAdd(dst, x);
      else
        *dst = x;
    });
  }
  TW_DEV void finish() {}
};

// D[m][n] = bf16(acc) (round to nearest even) for rows m < M, row stride ld: the dense
// route's y and dx (rows of the dense backup are written again by its row scatter).
struct EpiStoreBf16 {
  static constexpr int kStageBytes = kEpiTransposeBytes;
  static constexpr bool kOverlapLoads = true;
  struct Params {
    uint16_t* D;
    int ld;
  };
  const Params& p;
  int m, M, n0;
  float* stage = nullptr;
  TW_DEV EpiStoreBf16(const Params& p_, int m_, int M_, int n0_) : p(p_), m(m_), M(M_), n0(n0_) {}
  // Every lane of the warp calls it (the stores are warp-cooperative).
  TW_DEV void chunk(int c, const uint32_t (&v)[32], const uint32_t (&)[32]) {
    const int lane = threadIdx.x & 31;
    const int m0 = m - lane;
    const int rows = min(32, M - m0);
    if (rows <= 0) return;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    transposed_rows_bf16(stage, w, m0, rows, p.D + n0 + c * 32, p.ld);
  }
  TW_DEV void finish() {}
};

// Element q (0..7) of eight 16-bit values held in a uint4, and byte q (0..15) of a uint4.
TW_DEV uint32_t sel16(const uint4& v, int q) {
  const uint32_t w = q < 2 ? v.x : q < 4 ? v.y : q < 6 ? v.z : v.w;
  return (q & 1) ? (w >> 16) : (w & 0xFFFFu);
}
TW_DEV uint32_t sel8(const uint4& v, int q) {
  const uint32_t w = q < 4 ? v.x : q < 8 ? v.y : q < 12 ? v.z : v.w;
  return (w >> (8 * (q & 3))) & 0xFFu;
}

// Dense route, gated forward: the accumulator is u = x Wu^T for token row m over the
// columns [n0, n0 + BN). With the row's TwELL slots of a (the gate kernel's output;
// a row served here never overflowed, so its slots hold all its nonzeros) the
// epilogue forms h = a u at the active columns and writes
//   H[m][:]        fp16(h) at active columns, 0 elsewhere (the down GEMM's operand;
//                  fp16's 11 significant bits, because the backup rows' large
//                  activations put bf16's rounding of h above the parity bound),
//   the ELL row    global index, a and fp16(u) per nonzero, at the row's ELL offset
//                  (the nonzeros of the row's tiles before this CTA tile),
// the same ELL the sparse route's token kernel writes. Rows of the dense backup get
// no ELL entries and H = fp16(a u) from their saved fp32 a (the backup's own GEMM has
// run before this one) and this accumulator's u, which is also saved as their fp32 u,
// so the down GEMM covers them too; a row past the backup capacity gets H = 0.
// A TwELL tile's slots are read sixteen at a time (one 16-byte load of indices and
// two of values, all issued together; the first tile's before the accumulator is
// ready), not one dependent load per slot. The accumulator's 32 columns of a chunk go
// through the thread's part of the staging buffer (a row of kUpStride floats, an odd
// stride, so lanes reading the same column hit distinct banks), where active columns
// are looked up by index; H leaves through the per-warp transpose (in the same
// buffer, once every lane has read its row), whole 64-byte row segments per store.
struct EpiUpHybrid {
  static constexpr int kUpStride = 33;
  static constexpr int kStageBytes = 4 * 32 * kUpStride * 4;
  static constexpr bool kSplitColumns = true;  // eight epilogue warps on 256-wide tiles
  struct Params {
    int T, W, C, nT, R;
    const uint16_t* cnt;
    const uint16_t* val;
    const uint8_t* idx;
    const int32_t* backup_slot;
    const float* backup_a;  // [cap, I] fp32 (may be null when cap == 0)
    float* backup_u;        // [cap, I] fp32: written for the backup rows (this accumulator's u), or
                            // null when the backup's own GEMM saved u
    int cap;
    uint16_t* H;
    int ldh;  // row stride of H, backup_a and backup_u (= I)
    uint16_t* ell_idx;
    uint16_t* ell_a;
    uint16_t* ell_u;
    int32_t* status;
  };
  const Params& p;
  int m, M, n0;
  bool valid, ell_row;
  int bslot;    // backup slot of the row when it has one below the capacity, else -1
  int off;      // ELL slot of the next nonzero of this row
  int k_cur;    // TwELL tile of the slot cursor, its count, the cursor within it
  int n_cur;
  int s_cur;
  int g_cur;    // first slot of the group of sixteen held in iv / v0 / v1
  uint4 iv, v0, v1;
  float* stage = nullptr;
  TW_DEV EpiUpHybrid(const Params& p_, int m_, int M_, int n0_)
      : p(p_), m(m_), M(M_), n0(n0_), valid(m_ < M_), ell_row(false), bslot(-1), off(0), k_cur(-1), n_cur(0),
        s_cur(0), g_cur(-16) {}
  TW_DEV void load_group(int k, int g) {
    const size_t base = (static_cast<size_t>(m) * p.nT + k) * p.C + g;
    if (p.C % 16 == 0) {
      iv = *reinterpret_cast<const uint4*>(p.idx + base);
      v0 = *reinterpret_cast<const uint4*>(p.val + base);
      v1 = *reinterpret_cast<const uint4*>(p.val + base + 8);
    } else {
      uint32_t b[4] = {0u, 0u, 0u, 0u}, w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      for (int q = 0; q < 16 && g + q < p.C; ++q) {
        b[q >> 2] |= static_cast<uint32_t>(p.idx[base + q]) << (8 * (q & 3));
        w[q >> 1] |= static_cast<uint32_t>(p.val[base + q]) << (16 * (q & 1));
      }
      iv = make_uint4(b[0], b[1], b[2], b[3]);
      v0 = make_uint4(w[0], w[1], w[2], w[3]);
      v1 = make_uint4(w[4], w[5], w[6], w[7]);
    }
    g_cur = g;
  }
  TW_DEV void open_tile(int k) {
    k_cur = k;
    s_cur = 0;
    n_cur = min(static_cast<int>(p.cnt[static_cast<size_t>(m) * p.nT + k]), p.C);
    if (n_cur > 0) load_group(k, 0);
  }
  // before the accumulator is ready: the routing of the row, the ELL offset of its
  // first tile in [n0, n0 + BN) (a sum over the counts of the row's earlier tiles) and
  // that tile's first sixteen slots
  TW_DEV void prefetch(int bn) {
    if (!valid) return;
    const int slot = p.backup_slot[m];
    ell_row = slot == -1;
    if (slot >= 0 && TW_CHECKED(slot < p.cap, p.status)) bslot = slot;
    if (bslot >= 0) {  // the saved fp32 a of a backup row over the tile's columns, into L2
      const float* ra = p.backup_a + static_cast<size_t>(bslot) * p.ldh + n0;
      for (int i = 0; i < bn; i += 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(ra + i));
    }
    if (!ell_row) return;
    const int k0 = n0 / p.W;
    const uint16_t* cr = p.cnt + static_cast<size_t>(m) * p.nT;
    int o = 0;
    for (int k = 0; k < k0; ++k) o += min(static_cast<int>(cr[k]), p.C);
    off = o;
    open_tile(k0);
  }
  // Every lane of the warp calls it (H's stores are warp-cooperative).
  TW_DEV void chunk(int c, const uint32_t (&v)[32], const uint32_t (&)[32]) {
    const int lane = threadIdx.x & 31;
    const int m0 = m - lane;
    const int rows = min(32, M - m0);
    if (rows <= 0) return;  // uniform over the warp
    const int col0 = n0 + c * 32;
    uint32_t mask = 0u;
    float* mine = stage + lane * kUpStride;
    if (valid && ell_row) {
#pragma unroll
      for (int i = 0; i < 32; ++i) mine[i] = __uint_as_float(v[i]);
      const int k = col0 / p.W;
      const int local0 = col0 - k * p.W;
      if (k != k_cur) open_tile(k);
      const size_t rb = static_cast<size_t>(m) * p.R;
      // the tile's slots are in ascending column order: take those inside this chunk
      for (; s_cur < n_cur; ++s_cur) {
        if (s_cur - g_cur >= 16) load_group(k, s_cur);
        const int q = s_cur - g_cur;
        const int li = static_cast<int>(sel8(iv, q));
        if (li >= local0 + 32) break;
        const int i = li - local0;
        if (!TW_CHECKED(i >= 0 && i < 32, p.status)) continue;
        const uint16_t ab = static_cast<uint16_t>(q < 8 ? sel16(v0, q) : sel16(v1, q - 8));
        const float u = mine[i];
        mine[i] = bf16_to_f32(ab) * u;  // h, in place of u
        mask |= 1u << i;
        if (TW_CHECKED(off < p.R, p.status)) {
          p.ell_idx[rb + off] = static_cast<uint16_t>(col0 + i);
          p.ell_a[rb + off] = ab;
          p.ell_u[rb + off] = f32_to_f16(u);
        }
        ++off;
      }
    } else if (valid && bslot >= 0) {
      // a backup row: h = a u with its saved fp32 a (0 off the support)
      const float4* ra = reinterpret_cast<const float4*>(p.backup_a + static_cast<size_t>(bslot) * p.ldh + col0);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 x = ra[i];
        const float av[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) mine[4 * i + e] = av[e] > 0.f ? av[e] * __uint_as_float(v[4 * i + e]) : 0.f;
      }
      mask = 0xFFFFFFFFu;
    }
    uint32_t w[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float h0 = ((mask >> (2 * q)) & 1u) ? mine[2 * q] : 0.f;
      const float h1 = ((mask >> (2 * q + 1)) & 1u) ? mine[2 * q + 1] : 0.f;
      w[q] = pack_f16x2_rn(h0, h1);
    }
    // the backup rows' fp32 u is saved from here (the backup's own GEMM skips u on this
    // route): the lanes' rows go through the staging buffer, and each backup row leaves
    // as whole 128-byte segments at its slot
    const int my_slot = (valid && bslot >= 0 && p.backup_u != nullptr) ? bslot : -1;
    if (__any_sync(0xFFFFFFFFu, my_slot >= 0)) {
      __syncwarp();  // every lane has read its h from the staging row
#pragma unroll
      for (int i = 0; i < 32; ++i) mine[i] = __uint_as_float(v[i]);
      __syncwarp();
      const int sub = lane >> 3, c8 = lane & 7;
#pragma unroll
      for (int r0 = 0; r0 < 32; r0 += 4) {
        const int r = r0 + sub;
        const int sl = __shfl_sync(0xFFFFFFFFu, my_slot, r);
        if (sl >= 0 && r < rows) {
          const float* src = stage + r * kUpStride + 4 * c8;
          reinterpret_cast<float4*>(p.backup_u + static_cast<size_t>(sl) * p.ldh + col0)[c8] =
              make_float4(src[0], src[1], src[2], src[3]);
        }
      }
    }
    __syncwarp();  // every lane has read the staging rows: the transpose reuses the buffer
    transposed_rows_bf16(stage, w, m0, rows, p.H + col0, p.ldh);
  }
  TW_DEV void finish() {}
};

// Dense route, backward: the accumulator is dh = dY Wd^T for token row m over the
// columns [n0, n0 + BN). The row's saved ELL entries (global index ascending, a, u)
// give the support; on it
//   dg = dh u + l1 (non-gated: dh + l1),  du = dh a,  h = a u (non-gated: a),
// and the epilogue writes fp16 dG, dU (gated) and H over the tile's columns, 0 off
// the support, as the operands of the dx and weight-gradient GEMMs (run on fp16: a
// weight-gradient element sums thousands of these products at high activity, and
// bf16's 8 significant bits then leave errors above the parity bound where the sum
// cancels). Rows of the dense backup take their a and u from the saved fp32 backup
// rows (support a > 0), so the dense GEMMs cover them too and the backup's own
// backward GEMMs do not run; a row past the backup capacity gets zeros.
// The row's entries are read eight at a time (16-byte loads of indices, a and u,
// issued together; the tile's first eight before the accumulator is ready, after a
// binary search for the tile's first entry), not one dependent load per entry. A
// chunk's entries are placed in the thread's staging row, word i = a's bf16 bits |
// u's fp16 bits << 16 (stride kGradStride, odd), and read back by column; the three
// outputs leave through the per-warp transpose (in the same buffer, once every lane
// has read its row), whole 64-byte row segments per store.
template <bool GATED>
struct EpiDenseGrad {
  static constexpr int kGradStride = 33;
  // a warp's staging: its lanes' rows of ELL (a, u) words (32 x kGradStride words),
  // overlapped by the three 2 KB output blocks at the next 512-byte boundary
  static constexpr int kWarpStageBytes = 7168;
  static_assert(32 * kGradStride * 4 <= kWarpStageBytes && 511 + 3 * 2048 <= kWarpStageBytes, "grad staging");
  static constexpr int kStageBytes = 4 * kWarpStageBytes;
  static constexpr bool kSplitColumns = true;  // eight epilogue warps on 256-wide tiles
  struct Params {
    int R, I;
    const int32_t* ell_nnz;
    const int32_t* backup_slot;
    const uint16_t* ell_idx;
    const uint16_t* ell_a;
    const uint16_t* ell_u;
    const float* backup_a;  // [cap, I] fp32 (may be null when cap == 0)
    const float* backup_u;
    int cap;
    float l1;
    uint16_t *dG, *dU, *H;
    int ld;
    int32_t* status;
    // dG, dU, H [T, I] fp16 as tensor maps of 32 x 32 boxes with the 64-byte swizzle
    // (the staging layout): each warp's blocks leave by bulk tensor stores
    CUtensorMap tm_dG, tm_dU, tm_H;
  };
  const Params& p;
  int m, M, n0;
  bool valid, ell_row;
  int bslot;     // backup slot of the row when it has one below the capacity, else -1
  int cur, end;  // ELL entry cursor and end of the row
  int b_cur;     // first entry of the batch of eight held in bi / ba / bu
  uint4 bi, ba, bu;
  float* stage = nullptr;
  TW_DEV EpiDenseGrad(const Params& p_, int m_, int M_, int n0_)
      : p(p_), m(m_), M(M_), n0(n0_), valid(m_ < M_), ell_row(false), bslot(-1), cur(0), end(0), b_cur(-8) {}
  TW_DEV void load_batch(int e) {
    const size_t base = static_cast<size_t>(m) * p.R + e;
    if (p.R % 8 == 0) {
      bi = *reinterpret_cast<const uint4*>(p.ell_idx + base);
      ba = *reinterpret_cast<const uint4*>(p.ell_a + base);
      bu = GATED ? *reinterpret_cast<const uint4*>(p.ell_u + base) : make_uint4(0u, 0u, 0u, 0u);
    } else {
      uint32_t wi[4] = {0u, 0u, 0u, 0u}, wa[4] = {0u, 0u, 0u, 0u}, wu[4] = {0u, 0u, 0u, 0u};
      for (int q = 0; q < 8 && e + q < end; ++q) {
        wi[q >> 1] |= static_cast<uint32_t>(p.ell_idx[base + q]) << (16 * (q & 1));
        wa[q >> 1] |= static_cast<uint32_t>(p.ell_a[base + q]) << (16 * (q & 1));
        if (GATED) wu[q >> 1] |= static_cast<uint32_t>(p.ell_u[base + q]) << (16 * (q & 1));
      }
      bi = make_uint4(wi[0], wi[1], wi[2], wi[3]);
      ba = make_uint4(wa[0], wa[1], wa[2], wa[3]);
      bu = make_uint4(wu[0], wu[1], wu[2], wu[3]);
    }
    b_cur = e;
  }
  // before the accumulator is ready: the first ELL entry at or past column n0 (binary
  // search over the row's ascending indices) and the batch holding it
  TW_DEV void prefetch(int bn) {
    if (!valid) return;
    const int slot = p.backup_slot[m];
    ell_row = slot == -1;
    if (slot >= 0 && TW_CHECKED(slot < p.cap, p.status)) bslot = slot;
    if (bslot >= 0) {  // the saved fp32 a and u of a backup row over the tile's columns, into L2
      const size_t off = static_cast<size_t>(bslot) * p.I + n0;
      for (int i = 0; i < bn; i += 32) {
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.backup_a + off + i));
        if (GATED) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.backup_u + off + i));
      }
    }
    if (!ell_row) return;
    int n = p.ell_nnz[m];
    if (!TW_CHECKED(n >= 0 && n <= p.R, p.status)) n = 0;
    const uint16_t* ri = p.ell_idx + static_cast<size_t>(m) * p.R;
    int lo = 0, hi = n;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (static_cast<int>(ri[mid]) < n0)
        lo = mid + 1;
      else
        hi = mid;
    }
    cur = lo;
    end = n;
    if (cur < end) load_batch(p.R % 8 == 0 ? (cur & ~7) : cur);
  }
  // Every lane of the warp calls it (the stores are warp-cooperative).
  TW_DEV void chunk(int c, const uint32_t (&dh)[32], const uint32_t (&)[32]) {
    const int lane = threadIdx.x & 31;
    const int m0 = m - lane;
    const int rows = min(32, M - m0);
    if (rows <= 0) return;  // uniform over the warp
    const int col0 = n0 + c * 32;
    // the previous chunk's bulk stores have read their blocks, which the ELL words
    // below overwrite
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    uint32_t mask = 0u;
    uint32_t* mine = reinterpret_cast<uint32_t*>(stage) + lane * kGradStride;
    if (valid && ell_row) {
      for (; cur < end; ++cur) {
        if (cur - b_cur >= 8) load_batch(p.R % 8 == 0 ? (cur & ~7) : cur);
        const int q = cur - b_cur;
        const int j = static_cast<int>(sel16(bi, q));
        if (j >= col0 + 32) break;
        const int i = j - col0;
        if (!TW_CHECKED(i >= 0, p.status)) continue;
        mine[i] = sel16(ba, q) | (GATED ? sel16(bu, q) << 16 : 0u);
        mask |= 1u << i;
      }
    }
    // a backup row's a and u over the chunk: its saved fp32 rows
    float ba_[32], bu_[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) ba_[i] = bu_[i] = 0.f;
    const bool bk = valid && bslot >= 0;
    if (bk) {
      const float4* ra = reinterpret_cast<const float4*>(p.backup_a + static_cast<size_t>(bslot) * p.I + col0);
      const float4* ru = reinterpret_cast<const float4*>(p.backup_u + static_cast<size_t>(bslot) * p.I + col0);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 x = ra[i];
        ba_[4 * i] = x.x;
        ba_[4 * i + 1] = x.y;
        ba_[4 * i + 2] = x.z;
        ba_[4 * i + 3] = x.w;
        if (GATED) {
          const float4 y = ru[i];
          bu_[4 * i] = y.x;
          bu_[4 * i + 1] = y.y;
          bu_[4 * i + 2] = y.z;
          bu_[4 * i + 3] = y.w;
        }
      }
    }
    uint32_t wg[16], wu[16], wh[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      float g2[2], u2[2], h2[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = 2 * q + e;
        const uint32_t au = ((mask >> i) & 1u) ? mine[i] : 0u;
        const bool act = bk ? ba_[i] > 0.f : ((mask >> i) & 1u) != 0u;
        const float a = bk ? ba_[i] : bf16_to_f32(static_cast<uint16_t>(au & 0xFFFFu));
        const float u = GATED ? (bk ? bu_[i] : f16_to_f32(static_cast<uint16_t>(au >> 16))) : 1.f;
        const float d = __uint_as_float(dh[i]);
        g2[e] = act ? (GATED ? d * u : d) + p.l1 : 0.f;
        u2[e] = act ? d * a : 0.f;
        h2[e] = act ? (GATED ? a * u : a) : 0.f;
      }
      wg[q] = pack_f16x2_rn(g2[0], g2[1]);
      wu[q] = pack_f16x2_rn(u2[0], u2[1]);
      wh[q] = pack_f16x2_rn(h2[0], h2[1]);
    }
    __syncwarp();  // every lane has read its staging row: the blocks reuse the buffer
    // lane r writes row r of each block (64 bytes, 16-byte pieces at piece ^ ((r >> 1) & 3),
    // the tensor maps' 64-byte swizzle); rows past T are clipped by the stores
    const uint32_t base = smem_addr(stage);
    uint8_t* blk = reinterpret_cast<uint8_t*>(stage) + (((base + 511u) & ~511u) - base);
    auto put_block = [&](uint8_t* b, const uint32_t (&w)[16]) {
      uint32_t* st = reinterpret_cast<uint32_t*>(b);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4*>(st + lane * 16 + 4 * ((i ^ (lane >> 1)) & 3)) =
            make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    };
    put_block(blk, wg);
    put_block(blk + 2048, wh);
    if (GATED) put_block(blk + 4096, wu);
    fence_proxy_async_smem();  // the generic-proxy writes are visible to the bulk copies
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&p.tm_dG, blk, col0, m0);
      tma_store_2d(&p.tm_H, blk + 2048, col0, m0);
      if (GATED) tma_store_2d(&p.tm_dU, blk + 4096, col0, m0);
      bulk_commit();
    }
  }
  // the tile's stores are complete before the warp's staging is reused or the CTA exits
  TW_DEV void finish() {
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    __syncwarp();
  }
};

// a[m][n] = bf16(ReLU(acc)) (round to nearest even), row stride lda: the dense
// activation matrix of an unfused pipeline (pack in a separate pass).
struct EpiReluBf16 {
  static constexpr int kStageBytes = 0;
  struct Params {
    uint16_t* a;
    int lda;
  };
  const Params& p;
  int m, M, n0;
  TW_DEV EpiReluBf16(const Params& p_, int m_, int M_, int n0_) : p(p_), m(m_), M(M_), n0(n0_) {}
  TW_DEV void chunk(int c, const uint32_t (&v)[32], const uint32_t (&)[32]) {
    if (m >= M) return;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float g0 = __uint_as_float(v[2 * i]), g1 = __uint_as_float(v[2 * i + 1]);
      w[i] = pack_bf16x2(g0 > 0.f ? g0 : 0.f, g1 > 0.f ? g1 : 0.f);
    }
    uint4* dst = reinterpret_cast<uint4*>(p.a + static_cast<size_t>(m) * p.lda + n0 + c * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
  TW_DEV void finish() {}
};

// acc[m][n] += D with fp32 vector atomics: one K slice of a split-K product (acc is
// zeroed beforehand, and every slice of the tile adds its part).
struct EpiRedF32 {
  static constexpr int kStageBytes = kEpiTransposeBytes;
  static constexpr bool kOverlapLoads = true;
  struct Params {
    float* acc;
    int ld;
  };
  const Params& p;
  int m, M, n0;
  float* stage = nullptr;  // this warp's transpose buffer
  TW_DEV EpiRedF32(const Params& p_, int m_, int M_, int n0_) : p(p_), m(m_), M(M_), n0(n0_) {}
  TW_DEV void chunk(int c, const uint32_t (&v)[32], const uint32_t (&)[32]) {
    float* col = p.acc + n0 + c * 32;
    transposed_rows(stage, v, m, M, [&](int r, int c4, float4 x) {
      atomicAdd(reinterpret_cast<float4*>(col + static_cast<size_t>(r) * p.ld) + c4, x);
    });
  }
  TW_DEV void finish() {}
};

// EpiRedF32 for a grouped launch over a device row count M: problem p's row tiles
// follow problem p - 1's (M rounded up to whole 128-row tiles each), and its partial
// sums are added into acc[p] (row stride ld).
struct EpiRedF32Grouped {
  static constexpr int kStageBytes = kEpiTransposeBytes;
  static constexpr bool kOverlapLoads = true;
  static constexpr int kMaxProblems = 2;
  struct Params {
    float* acc[kMaxProblems];
    int ld;
  };
  const Params& p;
  int m, M, n0;
  float* stage = nullptr;  // this warp's transpose buffer
  TW_DEV EpiRedF32Grouped(const Params& p_, int m_, int M_, int n0_) : p(p_), m(m_), M(M_), n0(n0_) {}
  TW_DEV void chunk(int c, const uint32_t (&v)[32], const uint32_t (&)[32]) {
    const int rows_per_problem = (M + GEMM_BM - 1) / GEMM_BM * GEMM_BM;
    const int prob = m / rows_per_problem;  // the same for the warp's 32 rows
    if (prob >= kMaxProblems) return;       // uniform over the warp
    float* col = p.acc[prob] + n0 + c * 32;
    transposed_rows(stage, v, m - prob * rows_per_problem, M, [&](int r, int c4, float4 x) {
      atomicAdd(reinterpret_cast<float4*>(col + static_cast<size_t>(r) * p.ld) + c4, x);
    });
  }
  TW_DEV void finish() {}
};

// Gate projection epilogue: a = bf16(ReLU(acc)) packed into TwELL. The thread owns
// one token row; it walks its columns in ascending order, so every (row, tile)
// ELL is filled in ascending column order without atomics. Only nonzeros are
// stored (padding slots stay untouched); cnt is always written; row_nnz and ovf
// are combined across column tiles with one atomic per (row, CTA tile).
// Per 32-column chunk the thread converts its values two at a time, forms a bit mask
// of the nonzero bf16 results and visits only the set bits; the chunk's bf16 words
// sit in the thread's part of the staging buffer so a set bit's value is read by
// index (a register array indexed at run time would go to local memory). Most rows
// have one or two nonzeros in a chunk, so the loop is short and has no per-column
// branch.
struct EpiTwellPack {
  static constexpr int kWordsPerLane = 20;                      // a thread's chunk of bf16 words
  static constexpr int kStageBytes = 4 * 32 * kWordsPerLane * 4;
  static constexpr bool kSplitColumns = true;  // eight epilogue warps on 256-wide tiles (W <= 128)
  struct Params {
    int T, W, C, nT;
    uint16_t* cnt;
    uint16_t* val;
    uint8_t* idx;
    int32_t* row_nnz;
    uint8_t* ovf;
    uint16_t* a_dense;  // optional [T, I] bf16 copy of a (verification only)
    int lda;
  };
  const Params& p;
  int m, n0;
  bool valid;
  int c_tile;   // nonzeros seen so far in the current TwELL tile
  int total;    // nonzeros of this row in this CTA tile
  bool any_ovf;
  float* stage = nullptr;  // this warp's staging buffer
  TW_DEV EpiTwellPack(const Params& p_, int m_, int M_, int n0_)
      : p(p_), m(m_), n0(n0_), valid(m_ < M_), c_tile(0), total(0), any_ovf(false) {}
  TW_DEV void chunk(int c, const uint32_t (&v)[32], const uint32_t (&)[32]) {
    if (!valid) return;
    const int col0 = n0 + c * 32;
    const int k = col0 / p.W;
    const int local0 = col0 - k * p.W;
    if (!TW_CHECKED(k < p.nT && m < p.T, nullptr)) return;
    uint32_t w[16];
    uint32_t mask = 0u;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float g0 = __uint_as_float(v[2 * q]), g1 = __uint_as_float(v[2 * q + 1]);
      w[q] = pack_bf16x2_rn(g0 > 0.0f ? g0 : 0.0f, g1 > 0.0f ? g1 : 0.0f);
      mask |= ((w[q] & 0x7FFFu) != 0u ? 1u : 0u) << (2 * q);
      mask |= ((w[q] & 0x7FFF0000u) != 0u ? 1u : 0u) << (2 * q + 1);
    }
    if (p.a_dense != nullptr) {
      uint4* dst = reinterpret_cast<uint4*>(p.a_dense + static_cast<size_t>(m) * p.lda + col0);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
    const int before = c_tile;
    c_tile += __popc(mask);
    if (mask != 0u && before < p.C) {
      uint32_t* mine = reinterpret_cast<uint32_t*>(stage) + (threadIdx.x & 31) * kWordsPerLane;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        reinterpret_cast<uint4*>(mine)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      const size_t slot_base = (static_cast<size_t>(m) * p.nT + k) * p.C;
      for (int s = before; mask != 0u && s < p.C; ++s) {
        const int i = __ffs(mask) - 1;
        mask &= mask - 1u;
        const uint32_t word = mine[i >> 1];
        p.val[slot_base + s] = static_cast<uint16_t>((i & 1) ? (word >> 16) : (word & 0xFFFFu));
        p.idx[slot_base + s] = static_cast<uint8_t>(local0 + i);
      }
    }
    if (local0 + 32 == p.W) {  // last chunk of this TwELL tile
      p.cnt[static_cast<size_t>(m) * p.nT + k] = static_cast<uint16_t>(c_tile);
      total += c_tile;
      any_ovf |= (c_tile > p.C);
      c_tile = 0;
    }
  }
  TW_DEV void finish() {
    if (!valid) return;
    if (total) atomicAdd(p.row_nnz + m, total);
    if (any_ovf) p.ovf[m] = 1;
  }
};
static_assert(EpiTwellPack::kWordsPerLane * 4 * 32 * 4 <= EpiTwellPack::kStageBytes,
              "a warp's staging region holds 32 lanes of 20 words");

// Eight fp32 values as an exact-to-2^-16 pair of bf16 vectors: hi = bf16(v),
// lo = bf16(v - hi). A GEMM run over both halves (two K segments against the same
// other operand) keeps the precision of an fp32 operand.
TW_DEV void split8(const float (&v)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    l[i] = pack_bf16x2(v[2 * i] - bf16_lo(h[i]), v[2 * i + 1] - bf16_hi(h[i]));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Dense-backup forward epilogue on a (gate, up) accumulator pair:
//   a = ReLU(g), h = a * u (gated) or a (non-gated), all fp32.
// h is written as the bf16 pair (H, H_lo) that the down-projection GEMM runs over,
// so backup rows lose no more precision than the CUDA-core path, whose h never
// leaves fp32. Backup rows are the high-activity rows (hundreds of large terms per
// output), where a single bf16 rounding of h would dominate the error of y.
// Optionally saves a and u in fp32 (the Hybrid's dense backup) for the backward.
// Rows in [M, end of tile) are written as zeros so that later GEMMs whose K runs
// over these rows read zeros.
template <bool GATED>
struct EpiBackupHidden {
  static constexpr int kStageBytes = kEpiTransposeBytes;
  struct Params {
    uint16_t* H;
    uint16_t* H_lo;
    float* save_a;  // optional
    float* save_u;  // optional
    int ld;         // row stride of every buffer (= I)
    int rows_alloc; // rows H / H_lo hold
    // optional route word: when it reads 1 (the dense route, whose own GEMMs take the
    // backup rows' y) only the saved a and u are written, not H / H_lo
    const int32_t* route;
  };
  const Params& p;
  int m, M, n0;
  bool want_h;
  float* stage = nullptr;  // this warp's staging buffer
  TW_DEV EpiBackupHidden(const Params& p_, int m_, int M_, int n0_)
      : p(p_), m(m_), M(M_), n0(n0_), want_h(p_.route == nullptr || *p_.route != 1) {}
  // Every lane of the warp calls it (the stores are warp-cooperative).
  TW_DEV void chunk(int c, const uint32_t (&g)[32], const uint32_t (&u)[32]) {
    const int lane = threadIdx.x & 31;
    const int m0 = m - lane;                      // the warp's first row
    const int rows = min(32, p.rows_alloc - m0);  // rows of H / H_lo (zeros past M)
    if (rows <= 0) return;                        // uniform over the warp
    const bool live = m < M;
    const int col = n0 + c * 32;
    uint32_t av[32], uv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float gv = __uint_as_float(g[i]);
      av[i] = __float_as_uint((live && gv > 0.f) ? gv : 0.f);
      uv[i] = (GATED && live) ? u[i] : 0u;
    }
    // h = a u (or a), then its two bf16 halves
#pragma unroll
    for (int half = 0; half < 2 && want_h; ++half) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float h2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int k = 2 * i + e;
          float h = __uint_as_float(av[k]);
          if (GATED) h *= __uint_as_float(uv[k]);
          if (half) h = h - bf16_lo(pack_bf16x2_rn(h, 0.f));  // the low half: h - bf16(h)
          h2[e] = h;
        }
        w[i] = pack_bf16x2_rn(h2[0], h2[1]);
      }
      transposed_rows_bf16(stage, w, m0, rows, (half ? p.H_lo : p.H) + col, p.ld);
    }
    if (p.save_a != nullptr) {
      float* dst = p.save_a + col;
      transposed_rows(stage, av, m, M, [&](int r, int c4, float4 x) {
        reinterpret_cast<float4*>(dst + static_cast<size_t>(r) * p.ld)[c4] = x;
      });
    }
    if (GATED && p.save_u != nullptr) {
      float* dst = p.save_u + col;
      transposed_rows(stage, uv, m, M, [&](int r, int c4, float4 x) {
        reinterpret_cast<float4*>(dst + static_cast<size_t>(r) * p.ld)[c4] = x;
      });
    }
  }
  TW_DEV void finish() {}
};

// Dense-backup backward epilogue on dh = dY Wd^T with the saved fp32 a and u rows:
//   du = dh * a,  dg = (dh * u + l1) where a > 0 (non-gated: dh + l1), else 0,
//   h = a * u (non-gated: a),
// each written as a (hi, lo) bf16 pair for the dx and weight-gradient GEMMs. Rows in
// [M, end of tile) become zeros.
template <bool GATED>
struct EpiBackupGrad {
  static constexpr int kStageBytes = kEpiTransposeBytes;
  struct Params {
    const float* a;
    const float* u;
    uint16_t *dG, *dG_lo, *dU, *dU_lo, *H, *H_lo;
    float l1;
    int ld;
    int rows_alloc;
  };
  const Params& p;
  int m, M, n0;
  float* stage = nullptr;  // this warp's staging buffer
  TW_DEV EpiBackupGrad(const Params& p_, int m_, int M_, int n0_) : p(p_), m(m_), M(M_), n0(n0_) {}

  // Row m's saved a and u over the tile's columns into L2 (rows with saved values).
  TW_DEV void prefetch(int bn) const {
    if (m >= M) return;
    const size_t off = static_cast<size_t>(m) * p.ld + n0;
    for (int i = 0; i < bn; i += 32) {
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.a + off + i));
      if (GATED) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.u + off + i));
    }
  }
  // The warp's 32 rows x 32 fp32 columns of a saved matrix, read four rows per
  // instruction (whole 128-byte row segments); rows at or past `rows` read as 0.
  TW_DEV void load_block(const float* src, int m0, int rows, int col, float4 (&x)[8]) const {
    const int lane = threadIdx.x & 31, sub = lane >> 3, c4 = lane & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 4 * i + sub;
      x[i] = r < rows ? *reinterpret_cast<const float4*>(src + static_cast<size_t>(m0 + r) * p.ld + col + 4 * c4)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // ... then handed back one row per lane through the staging buffer.
  TW_DEV void block_to_rows(const float4 (&x)[8], float (&out)[32]) {
    const int lane = threadIdx.x & 31, sub = lane >> 3, c4 = lane & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) *reinterpret_cast<float4*>(stage + (4 * i + sub) * kEpiStageStride + 4 * c4) = x[i];
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = *reinterpret_cast<const float4*>(stage + lane * kEpiStageStride + 4 * i);
      out[4 * i] = v.x;
      out[4 * i + 1] = v.y;
      out[4 * i + 2] = v.z;
      out[4 * i + 3] = v.w;
    }
    __syncwarp();
  }

  // Every lane of the warp calls it (the loads and stores are warp-cooperative).
  TW_DEV void chunk(int c, const uint32_t (&dh)[32], const uint32_t (&)[32]) {
    const int lane = threadIdx.x & 31;
    const int m0 = m - lane;                           // the warp's first row
    const int rows_out_n = min(32, p.rows_alloc - m0);  // rows of the outputs (zeros past M)
    if (rows_out_n <= 0) return;                       // uniform over the warp
    const int live = max(0, min(32, M - m0));          // rows with saved a and u
    const int col = n0 + c * 32;
    float av[32], uv[32];
    {
      float4 xa[8], xu[8];  // both blocks' loads in flight together
      load_block(p.a, m0, live, col, xa);
      if (GATED) load_block(p.u, m0, live, col, xu);
      block_to_rows(xa, av);
      if (GATED) {
        block_to_rows(xu, uv);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) uv[i] = 0.f;
      }
    }
    // the six outputs, each a bf16 (hi, lo) half of dg, du or h, one at a time
#pragma unroll
    for (int o = 0; o < 6; ++o) {
      if (!GATED && (o == 2 || o == 3)) continue;
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float v2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int k = 2 * i + e;
          const float d = __uint_as_float(dh[k]);
          const bool act = av[k] > 0.f;
          float v;
          if (o < 2)
            v = act ? (GATED ? d * uv[k] : d) + p.l1 : 0.f;  // dg
          else if (o < 4)
            v = act ? d * av[k] : 0.f;                       // du
          else
            v = GATED ? av[k] * uv[k] : av[k];               // h
          if (o & 1) v = v - bf16_lo(pack_bf16x2_rn(v, 0.f));  // the low half: v - bf16(v)
          v2[e] = v;
        }
        w[i] = pack_bf16x2_rn(v2[0], v2[1]);
      }
      uint16_t* dst = o == 0 ? p.dG : o == 1 ? p.dG_lo : o == 2 ? p.dU : o == 3 ? p.dU_lo : o == 4 ? p.H : p.H_lo;
      transposed_rows_bf16(stage, w, m0, rows_out_n, dst + col, p.ld);
    }
  }
  TW_DEV void finish() {}
};

}  // namespace tw

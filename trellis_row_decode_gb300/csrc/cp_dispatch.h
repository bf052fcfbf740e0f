// cp_dispatch.h -- kernel table shared by the instantiation units and the C ABI.
#pragma once

#include "cp_kernels.cuh"
#include "cp_kernels_host.cuh"
#include "cp_kernels_reduce.cuh"
#include "cp_kernels_mixed.cuh"

namespace cpk {

// Stages of the per-warp record ring: one row ahead for HBM-resident tables,
// more rows in flight for tables read over the host link (higher latency).
#ifndef CP_PF_HOST
#define CP_PF_HOST 16
#endif
#ifndef CP_LUTREP_HOST
#define CP_LUTREP_HOST 4
#endif
constexpr int kPfHost = CP_PF_HOST;
constexpr int kLutRepHost = CP_LUTREP_HOST;

using DecodeFn = void (*)(DecodeParams);
using ReduceFn = void (*)(DecodeParams, const float*, uint32_t, uint64_t);
using MixedFn = void (*)(DecodeParams, const uint64_t*);

// Mixed-rate tables (one bit rate per row): the block kernel for a
// chunks-per-lane index (kBlkWarps * mixed_rows_per_warp(cpl_idx) lookups per
// CTA) and the load-time check of the offset table (bad = 1 when a record is
// unusable).
MixedFn mixed_kernel(int cpl_idx);
int mixed_rows_per_warp(int cpl_idx);
void launch_check_mixed(const uint64_t* offsets, uint64_t n_rows, uint32_t d, uint32_t* bad,
                        int sm_count, cudaStream_t s);

// Chunks-per-lane specialisations: index 0 = any d (runtime loop), index i > 0
// = d == 256 * kCplValues[i].
constexpr int kCplVariants = 6;
constexpr int kCplValues[kCplVariants] = {0, 1, 2, 4, 8, 16};

// Rows per warp of the HBM block kernel per chunks-per-lane index: d = 256 and
// 512 (two or four rows per warp step) may take more rows per CTA than the rest.
#ifndef CP_BLK_ROWS_SHORT
#define CP_BLK_ROWS_SHORT 4
#endif
constexpr int kBlkRowsShort = CP_BLK_ROWS_SHORT;
constexpr int block_rows(int cpl_idx) {
  return (cpl_idx == 1 || cpl_idx == 2) ? kBlkRowsShort : kBlkRows;
}
// LUT replicas of the HBM block kernel per chunks-per-lane index: one where a
// warp decodes several short rows per step (the fill per row written weighs more:
// d = 512 table 0.0402 -> 0.0390 ms), kLutRepBlock elsewhere (d = 1024: 1 and 2
// replicas are within noise).
constexpr int block_rep(int cpl_idx) {
  return (cpl_idx == 1 || cpl_idx == 2) ? 1 : kLutRepBlock;
}

inline int cpl_index(uint32_t d) {
  for (int i = 1; i < kCplVariants; ++i)
    if (d == 256u * static_cast<uint32_t>(kCplValues[i])) return i;
  return 0;
}

struct KernelSet {
  DecodeFn dev[2][kCplVariants];    // [layout AoS/SoA][cpl index]: non-persistent block
                                    // kernel, lookup order
  DecodeFn host[2][kCplVariants];   // bucketed order: register-ring kernel for cpl
                                    // indices 1..3 (d <= 1024), cp.async kernel otherwise
  ReduceFn reduce[2][3];            // decode + group readout, d = 256, 512, 1024
};
#ifndef CP_PF_REDUCE
#define CP_PF_REDUCE 2
#endif
constexpr int kPfReduce = CP_PF_REDUCE;

// Host-path kernels for cpl indices 1..3 are lookup_decode_host_kernel (one
// shared stage per warp, kHostWarps warps per CTA).
inline bool host_uses_register_ring(int cpl_idx) { return cpl_idx >= 1 && cpl_idx <= 3; }
#ifndef CP_PF_HOST_REG
#define CP_PF_HOST_REG 4
#endif
constexpr int kPfHostReg = CP_PF_HOST_REG;
// LUT replicas of the register-ring kernel.  The kernel waits on the host link,
// not on LUT bank conflicts, and what shared memory it does not take is L1 that
// holds the records repeats read: 4 replicas (16 KB) against 32 (128 KB) took the
// 2^24-row d = 1024 table from 0.208 to 0.189 ms and the 51 GB one from 0.230
// to 0.215 ms (8 and 16 replicas fall in between).
constexpr int kLutRepHostReg = 4;


// Host-resident tables: lookups are visited bucketed by row-id range so that
// consecutive records of a warp are close in the host address space.
#ifndef CP_BUCKET_BITS
#define CP_BUCKET_BITS 12
#endif
constexpr uint32_t kBucketBits = CP_BUCKET_BITS;      // 4096 ranges (cpx::kBucketBitsHost)
constexpr uint32_t kBucketChunk = 1u << 20;           // lookups per pass

// Hot-row cache construction: records of the m rows `rows` (device ids, sorted)
// copied from the host table alias into `cache` (stride R), and the map
// row + 1 -> slot inserted into keys/vals (ts slots, keys zeroed by the caller).
void launch_cache_build(const uint8_t* table, uint32_t R, const int64_t* rows, uint64_t m,
                        uint8_t* cache, unsigned long long* keys, uint32_t* vals, uint32_t ts,
                        int sm_count, cudaStream_t s);

// Visiting order of n lookups for a host-resident table: perm = the lookups
// grouped by range (id >> shift; range nb: ids outside [0, n_rows)), a counting
// partition (count with the scan in its last CTA, then scatter).  With a cache
// map (cmap_ts > 0) cslot[j] receives the cache slot of idx[j] or 0xFFFFFFFF.
// counts (nb + 2 words: the counts and a completion ticket) must hold zeros on
// entry and holds zeros again afterwards; cursor (nb + 1 words) is scratch.
void launch_bucket_partition(const int64_t* idx, uint64_t n, uint64_t n_rows,
                             const unsigned long long* cmap_keys, const uint32_t* cmap_vals,
                             uint32_t cmap_ts, uint32_t* cslot, uint32_t shift, uint32_t nb,
                             uint32_t* counts, uint32_t* cursor, uint32_t* perm, int sm_count,
                             cudaStream_t s);

KernelSet kernels_k3();
KernelSet kernels_k4();
KernelSet kernels_k5();
KernelSet kernels_k6();

}  // namespace cpk

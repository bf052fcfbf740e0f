// cp_mixed.cu -- mixed-rate tables: load-time check and kernel instantiations.
#include <cstdint>
#include <cuda_runtime.h>

#include "cp_kernels_mixed.cuh"
#include "cp_dispatch.h"

namespace cpk {

__global__ void check_mixed_offsets_kernel(const uint64_t* __restrict__ offsets, uint64_t n_rows,
                                           uint32_t d, uint32_t* __restrict__ bad) {
  const uint64_t T = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t r = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < n_rows;
       r += T) {
    const uint64_t o0 = offsets[r], o1 = offsets[r + 1];
    bool ok = o1 > o0 && (o0 & 1) == 0 && (r != 0 || o0 == 0);
    if (ok) {
      const uint64_t R = o1 - o0;
      ok = R >= 2 && ((R - 2) * 16) % d == 0;
      const uint64_t k = ok ? (R - 2) * 16 / d : 0;
      ok = ok && k >= 3 && k <= 6;
    }
    if (!ok) *bad = 1u;
  }
}

namespace {
// Rows per warp: 8 where a warp decodes several short rows per step (d = 256,
// 512: 0.047 -> 0.045 ms on the 2^24-row d = 512 table), 4 elsewhere (8 took
// d = 1024 from 0.078 to 0.086 ms).
constexpr int kMixedRowsShort = 8;
constexpr int kMixedRows = 4;
}

MixedFn mixed_kernel(int cpl_idx) {
  switch (cpl_idx) {
    case 1: return &lookup_decode_mixed_block_kernel<1, kLutRepBlock, kMixedRowsShort>;
    case 2: return &lookup_decode_mixed_block_kernel<2, kLutRepBlock, kMixedRowsShort>;
    case 3: return &lookup_decode_mixed_block_kernel<4, kLutRepBlock, kMixedRows>;
    case 4: return &lookup_decode_mixed_block_kernel<8, kLutRepBlock, kMixedRows>;
    case 5: return &lookup_decode_mixed_block_kernel<16, kLutRepBlock, kMixedRows>;
    default: return &lookup_decode_mixed_block_kernel<0, kLutRepBlock, kMixedRows>;
  }
}

int mixed_rows_per_warp(int cpl_idx) {
  return (cpl_idx == 1 || cpl_idx == 2) ? kMixedRowsShort : kMixedRows;
}

void launch_check_mixed(const uint64_t* offsets, uint64_t n_rows, uint32_t d, uint32_t* bad,
                        int sm_count, cudaStream_t s) {
  check_mixed_offsets_kernel<<<static_cast<unsigned>(sm_count) * 4, 256, 0, s>>>(offsets, n_rows,
                                                                                  d, bad);
}

}  // namespace cpk

// cp_internal.h -- host-side internals shared by the C ABI translation units.
#pragma once

#include <cstdint>
#include <string>

#include <cuda_runtime.h>

#include "cp.h"
#include "cp_dispatch.h"
#include "cp_geometry.h"

struct cp_table {
  int device;
  int residency;
  int layout;
  uint64_t n_rows;
  uint32_t d;
  uint32_t k;
  uint32_t rec_bytes;     // R
  uint32_t code_bytes;    // d*k/16
  uint32_t soa_stride;    // S
  const uint8_t* rec;     // device-accessible AoS records (HBM, or alias of host memory)
  const uint8_t* soa_codes;
  const uint16_t* soa_alpha;
  uint32_t* lut_dev;      // 512 words
  uint32_t* status_dev;   // 1 word
  void* scratch_dev;      // host-resident tables: see cpx::HostScratch (kBucketChunk capacity)
  const uint64_t* offsets; // mixed-rate tables: record r at [offsets[r], offsets[r+1]), else null
  uint64_t table_bytes;    // mixed-rate tables: offsets[n_rows]
  const uint8_t* cache;   // host-resident tables: device copies of hot records (cache_rows x R)
  uint64_t cache_rows;
  unsigned long long* cmap_keys;   // row id + 1 -> cache slot, open addressing (cmap_ts slots)
  uint32_t* cmap_vals;
  uint32_t cmap_ts;
  uint32_t bucket_shift;  // bucket of row r = r >> bucket_shift
  uint32_t bucket_nb;     // number of row-range buckets
  void* registered;       // host range this handle registered, else nullptr
  int sm_count;
  int max_smem;           // opt-in shared memory per block
  cpk::KernelSet kernels;
};

namespace cpx {

// Device scratch of the host-resident path for passes of up to `capacity`
// lookups: per-range counts (zero between passes) and cursors, the visiting
// order and the cache slot of each lookup.
struct HostScratch {
  uint32_t* counts;       // nb + 1 words, zero on entry and exit of a pass
  uint32_t* cursor;       // nb + 1 words
  uint32_t* perm;         // capacity words
  uint32_t* cslot;        // capacity words: cache slot of each lookup's id (hot-row cache)
  uint32_t capacity;
};

HostScratch host_scratch_layout(void* base, uint32_t capacity, uint32_t nb);

uint32_t stage_bytes(const cp_table* t, bool soa, uint32_t* alpha_slot);
cpk::KernelSet kernels_for(uint32_t k);
void set_error(const std::string& what);
cp_status cuda_fail(cudaError_t e, const char* what);

// Queue one lookup-decode on `stream`.  host_path: the owner/partition pipeline
// of host-resident tables, run in passes of hs->capacity lookups.
cp_status launch_decode(const cp_table* t, const int64_t* idx, uint64_t n, uint16_t* out,
                        cudaStream_t stream, bool host_path, const HostScratch* hs);

}  // namespace cpx

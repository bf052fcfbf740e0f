// cp_bucket.cu -- processing order for host-resident tables.
//
// The pages place the table either in HBM or in pinned host DRAM read over the
// host link ("2비트 코드와 공유 트렐리스로 n-gram 룩업 테이블을 4~8배 압축한다",
// section 전제와 한계).  Over the host link the cost of a random record read
// depends on how far apart successive reads are in the host address space
// (address translation), so the host path visits the lookups grouped by row-id
// range: a counting partition into 2^12 ranges.  Only the visiting order
// changes; every output row is still written at its own lookup position.
//
// Repeated ids are fetched once (the pages name frequency-based caching as a
// lever for the host placement; with Zipf-distributed lookups about half of the
// ids of a replay repeat): a device hash table elects one owner lookup per
// distinct id, only owners are partitioned and decoded, and the other lookups
// copy their owner's finished output row.
#include <cstdint>
#include <cuda_runtime.h>

#include "cp_dispatch.h"

namespace cpk {

namespace {

constexpr uint32_t kNoOwner = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t bucket_of(int64_t r, uint64_t n_rows, uint32_t shift,
                                              uint32_t nb) {
  const uint64_t u = static_cast<uint64_t>(r);
  return (u < n_rows) ? static_cast<uint32_t>(u >> shift) : nb;
}

// First lookup of this warp's first batch of 32 (grid-stride over batches).
__device__ __forceinline__ uint64_t warp_batch0() {
  return (static_cast<uint64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 32;
}

// Lookup j takes part in the partition when it owns its id, or its id is out
// of range (it then writes a zero row).  dup == nullptr: every lookup does.
__device__ __forceinline__ bool visits(const uint32_t* dup, uint64_t j) {
  if (dup == nullptr) return true;
  const uint32_t o = dup[j];
  return o == static_cast<uint32_t>(j) || o == kNoOwner;
}

// dup[j] = the owner lookup of idx[j] (the first to claim the id's slot in an
// open-addressing table of ts = 2^k slots, keys r + 1, 0 = empty), or kNoOwner
// for an id outside [0, n_rows).  Lanes of a warp holding the same id share one
// probe (the group's lowest lane probes); slots are read before any CAS, so the
// lookups of a hot id do not serialise on one atomic.  Probing is bounded by ts;
// a lookup that finds no slot owns itself (still correct, just not deduplicated).
__device__ __forceinline__ uint32_t slot_hash(unsigned long long key, uint32_t ts) {
  return static_cast<uint32_t>((key * 0x9E3779B97F4A7C15ull) >> 32) & (ts - 1);
}

// With a hot-row cache (cmap_ts > 0) the group's lowest lane first looks the id
// up in the cache map (keys r + 1 -> slot) and the group writes cslot[j]; a
// cached id skips the owner table (every one of its lookups owns itself and is
// decoded from the HBM copy, so no row is copied afterwards).
// The same pass counts the lookups that will be visited (owners, and ids out of
// range) per row-range bucket: counts[b] += (a shared-memory histogram per CTA).
__global__ void dedupe_kernel(const int64_t* __restrict__ idx, uint64_t n, uint64_t n_rows,
                              unsigned long long* __restrict__ keys, uint32_t* __restrict__ owner,
                              uint32_t ts, uint32_t* __restrict__ dup,
                              const unsigned long long* __restrict__ cmap_keys,
                              const uint32_t* __restrict__ cmap_vals, uint32_t cmap_ts,
                              uint32_t* __restrict__ cslot, uint32_t shift, uint32_t nb,
                              uint32_t* __restrict__ counts) {
  extern __shared__ uint32_t hist[];                    // nb + 1 bins
  for (uint32_t i = threadIdx.x; i <= nb; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t warps = static_cast<uint64_t>(gridDim.x) * (blockDim.x >> 5);
  for (uint64_t base = warp_batch0(); base < n; base += warps * 32) {
    const uint64_t j = base + lane;
    const int64_t r = (j < n) ? __ldg(idx + j) : -1;
    const bool valid = j < n && static_cast<uint64_t>(r) < n_rows;
    if (j < n && !valid) {
      dup[j] = kNoOwner;
      if (cmap_ts != 0) cslot[j] = kNoOwner;
      atomicAdd(&hist[nb], 1u);
    }
    const uint32_t active = __ballot_sync(0xffffffffu, valid);
    if (!valid) continue;
    const unsigned long long key = static_cast<unsigned long long>(r) + 1ull;
    const uint32_t group = __match_any_sync(active, key);
    const uint32_t leader = __ffs(group) - 1;
    uint32_t o = static_cast<uint32_t>(j);
    uint32_t cs = kNoOwner;
    if (lane == leader && cmap_ts != 0) {
      uint32_t slot = slot_hash(key, cmap_ts);
      for (uint32_t probe = 0; probe < cmap_ts; ++probe) {
        const unsigned long long kk = __ldg(cmap_keys + slot);
        if (kk == key) {
          cs = __ldg(cmap_vals + slot);
          break;
        }
        if (kk == 0ull) break;
        slot = (slot + 1) & (cmap_ts - 1);
      }
    }
    // a cached id needs no owner: each of its lookups decodes from the HBM copy
    cs = __shfl_sync(group, cs, leader);
    if (lane == leader && cs == kNoOwner) {
      uint32_t slot = slot_hash(key, ts);
      for (uint32_t probe = 0; probe < ts; ++probe) {
        unsigned long long cur = __ldcg(keys + slot);
        if (cur == 0ull) {
          cur = atomicCAS(keys + slot, 0ull, key);
          if (cur == 0ull) cur = key;
        }
        if (cur == key) {
          uint32_t w = __ldcg(owner + slot);
          if (w == kNoOwner) {
            w = atomicCAS(owner + slot, kNoOwner, static_cast<uint32_t>(j));
            if (w == kNoOwner) w = static_cast<uint32_t>(j);
          }
          o = w;
          break;
        }
        slot = (slot + 1) & (ts - 1);
      }
    }
    o = (cs == kNoOwner) ? __shfl_sync(group, o, leader) : static_cast<uint32_t>(j);
    dup[j] = o;
    if (o == static_cast<uint32_t>(j)) atomicAdd(&hist[bucket_of(r, n_rows, shift, nb)], 1u);
    if (cmap_ts != 0) cslot[j] = cs;
  }
  __syncthreads();
  for (uint32_t i = threadIdx.x; i <= nb; i += blockDim.x)
    if (hist[i]) atomicAdd(&counts[i], hist[i]);
}

// Cache construction: warp per hot row, 2-byte granules (records are 2-byte
// aligned); then one thread per row inserts row + 1 -> slot.
__global__ void cache_fill_kernel(const uint8_t* __restrict__ table, uint32_t R,
                                  const int64_t* __restrict__ rows, uint64_t m,
                                  uint8_t* __restrict__ cache) {
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t warps = static_cast<uint64_t>(gridDim.x) * (blockDim.x >> 5);
  for (uint64_t s = static_cast<uint64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       s < m; s += warps) {
    const uint16_t* src =
        reinterpret_cast<const uint16_t*>(table + static_cast<uint64_t>(rows[s]) * R);
    uint16_t* dst = reinterpret_cast<uint16_t*>(cache + s * R);
    for (uint32_t i = lane; i < R / 2; i += 32) dst[i] = src[i];
  }
}

__global__ void cache_map_kernel(const int64_t* __restrict__ rows, uint64_t m,
                                 unsigned long long* __restrict__ keys,
                                 uint32_t* __restrict__ vals, uint32_t ts) {
  const uint64_t T = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t s = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; s < m; s += T) {
    const unsigned long long key = static_cast<unsigned long long>(rows[s]) + 1ull;
    uint32_t slot = slot_hash(key, ts);
    for (uint32_t probe = 0; probe < ts; ++probe) {
      const unsigned long long prev = atomicCAS(keys + slot, 0ull, key);
      if (prev == 0ull) {
        vals[slot] = static_cast<uint32_t>(s);
        break;
      }
      slot = (slot + 1) & (ts - 1);
    }
  }
}

// Non-owner lookups copy their owner's decoded row.  A warp reads 32 owner
// entries at once and copies the rows of the non-owners among them one after
// another, each lane loading its (up to) four 16-byte pieces before storing.
__global__ void copy_dups_kernel(const uint32_t* __restrict__ dup, uint64_t n, uint32_t row16,
                                 uint4* __restrict__ out) {
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t warps = static_cast<uint64_t>(gridDim.x) * (blockDim.x >> 5);
  for (uint64_t base = warp_batch0(); base < n; base += warps * 32) {
    const uint64_t j = base + lane;
    const uint32_t o = (j < n) ? __ldg(dup + j) : kNoOwner;
    uint32_t todo = __ballot_sync(0xffffffffu, o != kNoOwner && o != static_cast<uint32_t>(j));
    while (todo) {
      const uint32_t l = __ffs(todo) - 1;
      todo &= todo - 1;
      const uint32_t src_row = __shfl_sync(0xffffffffu, o, l);
      const uint4* src = out + static_cast<uint64_t>(src_row) * row16;
      uint4* dst = out + (base + l) * row16;
      for (uint32_t c0 = 0; c0 < row16; c0 += 128) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t c = c0 + 32 * u + lane;
          if (c < row16) v[u] = __ldcg(src + c);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t c = c0 + 32 * u + lane;
          if (c < row16) __stcs(dst + c, v[u]);
        }
      }
    }
  }
}

// Start of a pass: empty owner table (keys 0, owners 0xFFFFFFFF) of ts slots
// and zero bucket counts.
__global__ void reset_kernel(unsigned long long* __restrict__ keys, uint32_t* __restrict__ owner,
                             uint32_t ts, uint32_t* __restrict__ counts, uint32_t n_counts) {
  const uint32_t T = gridDim.x * blockDim.x;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < ts; i += T) {
    keys[i] = 0ull;
    owner[i] = kNoOwner;
  }
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n_counts; i += T) counts[i] = 0;
}

// In-place exclusive prefix sum of len words, one CTA of 1024 threads.
__global__ void bucket_scan_kernel(uint32_t* __restrict__ counts, uint32_t len) {
  __shared__ uint32_t warp_sum[32];
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t per = (len + blockDim.x - 1) / blockDim.x;
  const uint32_t b0 = tid * per;
  const uint32_t b1 = (b0 + per < len) ? b0 + per : len;
  uint32_t s = 0;
  for (uint32_t i = b0; i < b1; ++i) s += counts[i];
  uint32_t inc = s;                                     // inclusive scan inside the warp
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= static_cast<uint32_t>(o)) inc += v;
  }
  if (lane == 31) warp_sum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t nwarps = blockDim.x >> 5;
    uint32_t w = (lane < nwarps) ? warp_sum[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= static_cast<uint32_t>(o)) w += v;
    }
    if (lane < nwarps) warp_sum[lane] = w;             // inclusive over warps
  }
  __syncthreads();
  uint32_t run = inc - s + (warp > 0 ? warp_sum[warp - 1] : 0);
  for (uint32_t i = b0; i < b1; ++i) {
    const uint32_t v = counts[i];
    counts[i] = run;
    run += v;
  }
}

// perm[cursor[b]++] = j, one atomic per (warp, bucket) group.
__global__ void bucket_scatter_kernel(const int64_t* __restrict__ idx,
                                      const uint32_t* __restrict__ dup,
                                      uint64_t n, uint64_t n_rows, uint32_t shift, uint32_t nb,
                                      uint32_t* __restrict__ cursor, uint32_t* __restrict__ perm) {
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t warps = static_cast<uint64_t>(gridDim.x) * (blockDim.x >> 5);
  for (uint64_t base = warp_batch0(); base < n; base += warps * 32) {
    const uint64_t j = base + lane;
    const bool valid = j < n && visits(dup, j);
    const uint32_t active = __ballot_sync(0xffffffffu, valid);
    if (valid) {
      const uint32_t b = bucket_of(__ldg(idx + j), n_rows, shift, nb);
      const uint32_t group = __match_any_sync(active, b);
      const uint32_t leader = __ffs(group) - 1;
      const uint32_t rank = __popc(group & ((1u << lane) - 1u));
      uint32_t start = 0;
      if (lane == leader) start = atomicAdd(&cursor[b], static_cast<uint32_t>(__popc(group)));
      start = __shfl_sync(group, start, leader);
      perm[start + rank] = static_cast<uint32_t>(j);
    }
  }
}

}  // namespace

void launch_dedupe(const int64_t* idx, uint64_t n, uint64_t n_rows, unsigned long long* keys,
                   uint32_t* owner, uint32_t ts, uint32_t* dup,
                   const unsigned long long* cmap_keys, const uint32_t* cmap_vals,
                   uint32_t cmap_ts, uint32_t* cslot, uint32_t shift, uint32_t nb,
                   uint32_t* counts, int sm_count, cudaStream_t s) {
  reset_kernel<<<static_cast<unsigned>(sm_count) * 2, 512, 0, s>>>(keys, owner, ts, counts,
                                                                  nb + 1);
  dedupe_kernel<<<static_cast<unsigned>(sm_count) * 2, 512, (nb + 1) * sizeof(uint32_t), s>>>(
      idx, n, n_rows, keys, owner, ts, dup, cmap_keys, cmap_vals, cmap_ts, cslot, shift, nb,
      counts);
}

void launch_cache_build(const uint8_t* table, uint32_t R, const int64_t* rows, uint64_t m,
                        uint8_t* cache, unsigned long long* keys, uint32_t* vals, uint32_t ts,
                        int sm_count, cudaStream_t s) {
  cache_fill_kernel<<<static_cast<unsigned>(sm_count) * 4, 512, 0, s>>>(table, R, rows, m, cache);
  cache_map_kernel<<<static_cast<unsigned>(sm_count) * 4, 256, 0, s>>>(rows, m, keys, vals, ts);
}

void launch_bucket_partition(const int64_t* idx, const uint32_t* dup, uint64_t n, uint64_t n_rows,
                             uint32_t shift, uint32_t nb, uint32_t* counts, uint32_t* perm,
                             int sm_count, cudaStream_t s) {
  const unsigned blocks = static_cast<unsigned>(sm_count);
  bucket_scan_kernel<<<1, 1024, 0, s>>>(counts, nb + 1);
  bucket_scatter_kernel<<<blocks, 512, 0, s>>>(idx, dup, n, n_rows, shift, nb, counts, perm);
}

void launch_copy_dups(const uint32_t* dup, uint64_t n, uint32_t d, uint16_t* out, int sm_count,
                      cudaStream_t s) {
  copy_dups_kernel<<<static_cast<unsigned>(sm_count) * 2, 1024, 0, s>>>(
      dup, n, d / 8, reinterpret_cast<uint4*>(out));
}

}  // namespace cpk

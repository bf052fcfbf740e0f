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
// Repeated ids (about half of a Zipf replay's lookups) are visited like any
// other: the lookups of one id fall into the same range and so into the same
// slice of the visiting order, which one SM decodes, so a repeat mostly finds
// the record in that SM's L1 cache.  (Host-memory reads are not kept in L2.)  Ids named in a hot-row cache (frequency-based caching) keep their
// place in that order and read their record from its HBM copy, so every warp
// mixes link reads with cache reads.
#include <cstdint>
#include <cuda_runtime.h>

#include "cp_dispatch.h"

namespace cpk {

namespace {

constexpr uint32_t kNone = 0xFFFFFFFFu;

// Programmatic dependent launch from the count kernel to the scatter kernel:
// the scatter (launched with programmatic stream serialisation) may start once
// every count CTA has signalled, ranks its lookups in shared memory, and waits
// (hardware-managed, no spin in this code) for the count kernel to complete
// before it reads the range starts.  The decode kernel after the scatter is
// launched normally: started early, its CTAs would land on whichever SMs the
// scatter leaves free, and the slices of the visiting order would no longer
// map onto the SMs in order (on a 51 GB table that took the call from 0.21 to
// 2.0 ms: the device's address translation lost its locality).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Range of lookup j: id >> shift; nb for an id outside [0, n_rows) (it writes a
// zero row).
__device__ __forceinline__ uint32_t bucket_of(int64_t r, uint64_t n_rows, uint32_t shift,
                                              uint32_t nb) {
  const uint64_t u = static_cast<uint64_t>(r);
  return (u < n_rows) ? static_cast<uint32_t>(u >> shift) : nb;
}

__device__ __forceinline__ uint32_t slot_hash(unsigned long long key, uint32_t ts) {
  return static_cast<uint32_t>((key * 0x9E3779B97F4A7C15ull) >> 32) & (ts - 1);
}

// Cache slot of id r (map keys r + 1 -> slot, open addressing over cmap_ts
// slots, probing bounded by the table size), or kNone.
__device__ __forceinline__ uint32_t cache_slot(int64_t r, const unsigned long long* cmap_keys,
                                               const uint32_t* cmap_vals, uint32_t cmap_ts) {
  const unsigned long long key = static_cast<unsigned long long>(r) + 1ull;
  uint32_t slot = slot_hash(key, cmap_ts);
  for (uint32_t probe = 0; probe < cmap_ts; ++probe) {
    const unsigned long long kk = __ldg(cmap_keys + slot);
    if (kk == key) return __ldg(cmap_vals + slot);
    if (kk == 0ull) break;
    slot = (slot + 1) & (cmap_ts - 1);
  }
  return kNone;
}

// Partition kernels: CTAs of kPartThreads threads, each taking kPartItems
// consecutive lookups per thread, and per-range arrays of at most kPartBins
// words per thread.  Every loop that waits on memory issues all of a thread's
// loads or atomics before it uses any result, so a thread waits about one
// memory round trip per phase rather than one per item or range.  Both kernels
// are latency-bound: together about 25 us (under ncu) of a 0.19-0.21 ms call
// on the 196,608-lookup replay.
constexpr uint32_t kPartThreads = 512;
constexpr int kPartItems = 4;
constexpr int kPartBins = static_cast<int>(((1u << kBucketBits) + 1 + kPartThreads - 1) / kPartThreads);

// cursor[i] = exclusive prefix sum of counts[0..len) by the whole CTA (thread t
// takes counts [kPartBins t, kPartBins (t + 1))); counts is left holding zeros
// for the next pass.  counts was written by other CTAs' atomics: read at L2.
__device__ void scan_counts(uint32_t* counts, uint32_t* cursor, uint32_t len) {
  __shared__ uint32_t warp_sum[kPartThreads / 32];
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t b0 = tid * kPartBins;
  uint32_t v[kPartBins];
#pragma unroll
  for (int q = 0; q < kPartBins; ++q) v[q] = (b0 + q < len) ? __ldcg(counts + b0 + q) : 0u;
  uint32_t s = 0;
#pragma unroll
  for (int q = 0; q < kPartBins; ++q) s += v[q];
  uint32_t inc = s;                                     // inclusive scan inside the warp
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= static_cast<uint32_t>(o)) inc += x;
  }
  if (lane == 31) warp_sum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    constexpr uint32_t kWarps = kPartThreads / 32;
    uint32_t w = (lane < kWarps) ? warp_sum[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= static_cast<uint32_t>(o)) w += x;
    }
    if (lane < kWarps) warp_sum[lane] = w;             // inclusive over warps
  }
  __syncthreads();
  uint32_t run = inc - s + (warp > 0 ? warp_sum[warp - 1] : 0);
#pragma unroll
  for (int q = 0; q < kPartBins; ++q) {
    if (b0 + q < len) {
      cursor[b0 + q] = run;
      counts[b0 + q] = 0;
    }
    run += v[q];
  }
}

// counts[b] += lookups of range b (a shared-memory histogram per CTA, one
// shared atomic per (warp, range) group).  With a hot-row cache map
// (cmap_ts > 0) it also writes cslot[j], the cache slot of idx[j] or kNone; the
// lanes of a warp holding the same id share one probe.  The CTA that finishes
// last (ticket counts[nb + 1]) turns the counts into the ranges' start
// positions in cursor and sets counts and the ticket back to zero; nothing
// waits for it, the scatter kernel runs after this one.  counts (nb + 2 words)
// must hold zeros on entry.
__global__ void __launch_bounds__(kPartThreads)
    bucket_count_kernel(const int64_t* __restrict__ idx, uint64_t n, uint64_t n_rows,
                        const unsigned long long* __restrict__ cmap_keys,
                        const uint32_t* __restrict__ cmap_vals, uint32_t cmap_ts,
                        uint32_t* __restrict__ cslot, uint32_t shift, uint32_t nb,
                        uint32_t* __restrict__ counts, uint32_t* __restrict__ cursor) {
  pdl_launch_dependents();           // the scatter may start its counting-free part
  extern __shared__ uint32_t hist[];                    // nb + 1 bins
  for (uint32_t i = threadIdx.x; i <= nb; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t j0 = static_cast<uint64_t>(blockIdx.x) * kPartItems * kPartThreads + threadIdx.x;
  int64_t r[kPartItems];
#pragma unroll
  for (int it = 0; it < kPartItems; ++it) {
    const uint64_t j = j0 + static_cast<uint64_t>(it) * kPartThreads;
    r[it] = j < n ? __ldg(idx + j) : -1;
  }
#pragma unroll
  for (int it = 0; it < kPartItems; ++it) {
    const uint64_t j = j0 + static_cast<uint64_t>(it) * kPartThreads;
    const bool in = j < n;
    if (cmap_ts != 0) {
      uint32_t cs = kNone;
      const bool valid = in && static_cast<uint64_t>(r[it]) < n_rows;
      const uint32_t active = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const uint32_t group = __match_any_sync(active, static_cast<unsigned long long>(r[it]));
        const uint32_t leader = __ffs(group) - 1;
        if (lane == leader) cs = cache_slot(r[it], cmap_keys, cmap_vals, cmap_ts);
        cs = __shfl_sync(group, cs, leader);
      }
      if (in) cslot[j] = cs;
    }
    const uint32_t active = __ballot_sync(0xffffffffu, in);
    if (in) {
      const uint32_t b = bucket_of(r[it], n_rows, shift, nb);
      const uint32_t group = __match_any_sync(active, b);
      if (lane == __ffs(group) - 1) atomicAdd(&hist[b], static_cast<uint32_t>(__popc(group)));
    }
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < kPartBins; ++q) {
    const uint32_t i = threadIdx.x + q * kPartThreads;
    if (i <= nb) {
      const uint32_t h = hist[i];
      if (h) atomicAdd(&counts[i], h);
    }
  }
  // the last CTA to finish scans: every CTA's count atomics are ordered before
  // its ticket
  __shared__ uint32_t s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&counts[nb + 1], 1u) == gridDim.x - 1);
  __syncthreads();
  if (s_last) {
    __threadfence();
    scan_counts(counts, cursor, nb + 1);
    if (threadIdx.x == 0) counts[nb + 1] = 0;
  }
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

// perm[cursor[b]++] = j for every lookup j (b its range), the CTA's lookups
// as in the count kernel: a shared-memory histogram gives each lookup its rank
// among the CTA's lookups of its range (one shared atomic per (warp, range)
// group), then one global atomic per range the CTA holds reserves the CTA's
// places.
__global__ void __launch_bounds__(kPartThreads)
    bucket_scatter_kernel(const int64_t* __restrict__ idx, uint64_t n, uint64_t n_rows,
                          uint32_t shift, uint32_t nb, uint32_t* __restrict__ cursor,
                          uint32_t* __restrict__ perm) {
  extern __shared__ uint32_t hist[];                    // nb + 1 bins
  for (uint32_t i = threadIdx.x; i <= nb; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t j0 = static_cast<uint64_t>(blockIdx.x) * kPartItems * kPartThreads + threadIdx.x;
  int64_t r[kPartItems];
#pragma unroll
  for (int it = 0; it < kPartItems; ++it) {
    const uint64_t j = j0 + static_cast<uint64_t>(it) * kPartThreads;
    r[it] = j < n ? __ldg(idx + j) : -1;
  }
  uint32_t bk[kPartItems], rk[kPartItems];
#pragma unroll
  for (int it = 0; it < kPartItems; ++it) {
    const uint64_t j = j0 + static_cast<uint64_t>(it) * kPartThreads;
    const bool in = j < n;
    const uint32_t active = __ballot_sync(0xffffffffu, in);
    bk[it] = nb + 1;                                    // no lookup
    rk[it] = 0;
    if (in) {
      const uint32_t b = bucket_of(r[it], n_rows, shift, nb);
      const uint32_t group = __match_any_sync(active, b);
      const uint32_t leader = __ffs(group) - 1;
      uint32_t start = 0;
      if (lane == leader) start = atomicAdd(&hist[b], static_cast<uint32_t>(__popc(group)));
      start = __shfl_sync(group, start, leader);
      bk[it] = b;
      rk[it] = start + __popc(group & ((1u << lane) - 1u));
    }
  }
  __syncthreads();
  pdl_wait();                        // cursor holds the range starts
  uint32_t base[kPartBins];
#pragma unroll
  for (int q = 0; q < kPartBins; ++q) {
    const uint32_t i = threadIdx.x + q * kPartThreads;
    const uint32_t h = (i <= nb) ? hist[i] : 0u;
    base[q] = h ? atomicAdd(&cursor[i], h) : 0u;
  }
#pragma unroll
  for (int q = 0; q < kPartBins; ++q) {
    const uint32_t i = threadIdx.x + q * kPartThreads;
    if (i <= nb) hist[i] = base[q];
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < kPartItems; ++it) {
    if (bk[it] <= nb) {
      const uint64_t j = j0 + static_cast<uint64_t>(it) * kPartThreads;
      perm[hist[bk[it]] + rk[it]] = static_cast<uint32_t>(j);
    }
  }
}

}  // namespace

void launch_cache_build(const uint8_t* table, uint32_t R, const int64_t* rows, uint64_t m,
                        uint8_t* cache, unsigned long long* keys, uint32_t* vals, uint32_t ts,
                        int sm_count, cudaStream_t s) {
  cache_fill_kernel<<<static_cast<unsigned>(sm_count) * 4, 512, 0, s>>>(table, R, rows, m, cache);
  cache_map_kernel<<<static_cast<unsigned>(sm_count) * 4, 256, 0, s>>>(rows, m, keys, vals, ts);
}

void launch_bucket_partition(const int64_t* idx, uint64_t n, uint64_t n_rows,
                             const unsigned long long* cmap_keys, const uint32_t* cmap_vals,
                             uint32_t cmap_ts, uint32_t* cslot, uint32_t shift, uint32_t nb,
                             uint32_t* counts, uint32_t* cursor, uint32_t* perm, int sm_count,
                             cudaStream_t s) {
  if (n == 0) return;
  (void)sm_count;
  const size_t hist_bytes = (nb + 1) * sizeof(uint32_t);
  const uint64_t per = static_cast<uint64_t>(kPartItems) * kPartThreads;
  const unsigned blocks = static_cast<unsigned>((n + per - 1) / per);
  bucket_count_kernel<<<blocks, kPartThreads, hist_bytes, s>>>(
      idx, n, n_rows, cmap_keys, cmap_vals, cmap_ts, cslot, shift, nb, counts, cursor);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kPartThreads);
  cfg.dynamicSmemBytes = hist_bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, bucket_scatter_kernel, idx, n, n_rows, shift, nb, cursor, perm);
}

}  // namespace cpk

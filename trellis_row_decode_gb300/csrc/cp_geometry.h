// cp_geometry.h -- host-side geometry and argument checks of libcp, in plain
// C++ (no CUDA headers) so that they also build with host sanitizers.
#pragma once

#include <cstddef>
#include <cstdint>

namespace cpx {

constexpr uint64_t kMaxRows = 1ull << 40;
constexpr uint64_t kMaxLookups = 1ull << 40;
#ifndef CP_BUCKET_BITS
#define CP_BUCKET_BITS 12
#endif
constexpr uint32_t kBucketBitsHost = CP_BUCKET_BITS;  // at most 2^12 row ranges

// Geometry accepted by the CUDA path: k in {3,..,6}, d % 8 == 0 in [8, 4096],
// and a whole number of 16-bit words per record (so every record starts
// 2-byte aligned).
inline bool geometry_ok(uint32_t d, uint32_t k) {
  if (k < 3 || k > 6) return false;
  if (d < 8 || d > 4096 || (d % 8) != 0) return false;
  if ((static_cast<uint64_t>(d) * k) % 32 != 0) return false;
  return true;
}

// Code stride of the SoA copy: d*k/16 bytes rounded up to 16.
inline uint32_t soa_stride(uint32_t d, uint32_t k) { return ((d * k / 16) + 15u) & ~15u; }

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Row-range buckets of the host path's visiting order: bucket of row r is
// r >> shift, nb buckets in all (nb <= 2^kBucketBitsHost).  n_rows >= 1.
inline void bucket_params(uint64_t n_rows, uint32_t* shift, uint32_t* nb) {
  uint32_t bits = 0;
  while (bits < 64 && ((n_rows - 1) >> bits) != 0) ++bits;
  *shift = bits > kBucketBitsHost ? bits - kBucketBitsHost : 0;
  *nb = static_cast<uint32_t>(((n_rows - 1) >> *shift) + 1);
}

// Words of one per-range array (nb + 1 ranges and one more word, the counts'
// completion ticket, padded to 64 words).
constexpr size_t host_scratch_count_words(uint32_t nb) { return (nb + 2 + 63) & ~63u; }

// Device scratch of the host path for passes of `capacity` lookups: range
// counts and cursors, then the visiting order and the cache slot per lookup.
constexpr size_t host_scratch_bytes(uint32_t capacity, uint32_t nb) {
  return (2 * host_scratch_count_words(nb) + 2 * static_cast<size_t>(capacity)) *
         sizeof(uint32_t);
}

// Bytes of one shared-memory record stage: a 16-byte prefix (room for the
// spliced code tail below bit 0), the 16-byte aligned span holding the record
// (misalignment <= 14 bytes for AoS), and 16 bytes of slack for the 64-bit
// funnel reads past the code; SoA adds the 4-byte alpha slot in that slack.
inline uint32_t stage_bytes_for(uint32_t prefix, uint32_t code_bytes, uint32_t soa_stride,
                                bool soa, uint32_t* alpha_slot) {
  if (soa) {
    *alpha_slot = prefix + soa_stride + 8;
    return prefix + soa_stride + 16;
  }
  *alpha_slot = 0;
  const uint32_t span = code_bytes + 2 + 14;
  return prefix + ((span + 15u) & ~15u) + 16u;
}

}  // namespace cpx

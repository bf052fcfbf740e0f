// cp_kernels_host.cuh -- host-resident lookup-decode kernel (register ring).
#pragma once

#include "cp_kernels.cuh"

namespace cpk {

// Host-resident variant for records that fit one 16-byte piece per lane
// (d <= 1024).  Reads of pinned host memory over the host link are issued as
// plain 16-byte register loads: asynchronous shared-memory copies of system
// memory hold their issue queue slots for the whole link round trip and throttle
// issue.  Each warp keeps PF rows in flight in a register ring (slots fixed at
// compile time by unrolling) and lands a row into its single shared stage just
// before decoding it.  32 warps per CTA with PF = 4 (64 registers a thread):
// more warps with a shorter ring beat 16 warps with PF = 8 (51 GB table:
// 0.234 -> 0.226 ms, 0.162 -> 0.146 ms with the hot-row cache).
#ifndef CP_HOST_WARPS
#define CP_HOST_WARPS 32
#endif
constexpr int kHostWarps = CP_HOST_WARPS;

// 16-byte piece of which only the first `bytes` (even, < 16) are inside the
// table: 2-byte loads, the rest zero (the table's last record only).
__device__ __forceinline__ uint4 load_partial16(const uint8_t* src, uint32_t bytes) {
  uint64_t lo = 0, hi = 0;
  for (uint32_t b = 0; b < bytes; b += 2) {
    const uint64_t v = __ldg(reinterpret_cast<const uint16_t*>(src + b));
    if (b < 8) lo |= v << (8 * b);
    else hi |= v << (8 * (b - 8));
  }
  return make_uint4(static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32),
                    static_cast<uint32_t>(hi), static_cast<uint32_t>(hi >> 32));
}

// Work distribution: each CTA (one per SM) takes a contiguous slice of the
// visiting order (lookups grouped by row range), so each SM reads from one
// contiguous part of the table, and its warps take chunks of 32 visits of the
// slice from a shared-memory counter, so they finish together.  Handing out
// chunks of the whole order from one global counter balanced the SMs too, but
// let every SM's reads span the whole table, and on a 51 GB table that ran 14
// times slower (the device's address translation for host memory lost its
// locality); fixed ranges per warp left SMs idle 13 % of the time.
template <int K, bool SOA, int PF, int CPL, int REP>
__global__ void __launch_bounds__(kHostWarps * 32, 1)
    lookup_decode_host_kernel(const DecodeParams p) {
  static_assert(CPL >= 1 && CPL <= 4, "one 16-byte piece per lane");
  static_assert(REP >= 4 && REP % 4 == 0, "the LUT fill writes 16-byte groups of replicas");
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const uint32_t lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;

  constexpr int kLutBytes = lut_bytes(REP);
  for (int q = tid; q < kLutEntries * REP / 4; q += blockDim.x) {
    const int e = q / (REP / 4);
    uint32_t v = __ldg(p.lut + (e & 511));
    if (e & 512) v ^= 0x80000000u;
    reinterpret_cast<uint4*>(smem)[q] = make_uint4(v, v, v, v);
  }
  __syncthreads();

  const uint32_t code_bytes = p.code_bytes;
  const uint32_t d = p.d;
  const uint64_t n_rows = p.n_rows;
  const uint64_t stride = p.stride;
  const uintptr_t codes = reinterpret_cast<uintptr_t>(p.codes);
  const uintptr_t tbl_end = codes + p.table_bytes;
  uint8_t* sb = smem + kLutBytes + static_cast<size_t>(warp) * p.stage_bytes + kStagePrefix;

  // each CTA a contiguous slice of the visiting order; its warps take chunks of
  // 32 visits of the slice from a shared-memory counter (a chunk of look-ahead)
  __shared__ uint32_t s_ctr;
  if (tid == 0) s_ctr = 0;
  __syncthreads();
  const uint64_t n_work = p.n;
  const uint64_t c_lo = static_cast<uint64_t>(blockIdx.x) * n_work / gridDim.x;
  const uint64_t c_hi = static_cast<uint64_t>(blockIdx.x + 1) * n_work / gridDim.x;
  constexpr uint32_t kPast = 0xFFFFFFFFu;
  const uint32_t* cslot = p.cslot;
  const uintptr_t cache = reinterpret_cast<uintptr_t>(p.cache);
  const uintptr_t cache_end = cache + p.cache_bytes;
  auto grab = [&]() -> uint64_t {
    uint32_t c = 0;
    if (lane == 0) c = atomicAdd(&s_ctr, 32u);
    return c_lo + __shfl_sync(0xffffffffu, c, 0);
  };
  auto load_batch = [&](uint64_t c, uint32_t& j, int64_t& r, uint32_t& cs) {
    j = kPast;
    r = 0;
    cs = 0xFFFFFFFFu;
    const uint64_t q = c + lane;
    if (q < c_hi) {
      j = __ldg(p.perm + q);
      r = __ldg(p.idx + j);
      if (cslot != nullptr) cs = __ldg(cslot + j);
    }
  };
  uint32_t jb_cur, jb_nxt, cb_cur, cb_nxt;
  int64_t ib_cur, ib_nxt;
  load_batch(grab(), jb_cur, ib_cur, cb_cur);
  load_batch(grab(), jb_nxt, ib_nxt, cb_nxt);
  uint32_t batch = 0;

  uint4 rv[PF];
  uint32_t rm[PF], rj[PF];
  uint16_t ra[PF];

  auto issue = [&](uint32_t q, uint4& v, uint32_t& m, uint32_t& jrow, uint16_t& ab) {
    if (q - batch >= 32) {
      batch += 32;
      ib_cur = ib_nxt;
      jb_cur = jb_nxt;
      cb_cur = cb_nxt;
      load_batch(grab(), jb_nxt, ib_nxt, cb_nxt);
    }
    const int64_t r = __shfl_sync(0xffffffffu, ib_cur, static_cast<int>(q - batch));
    jrow = __shfl_sync(0xffffffffu, jb_cur, static_cast<int>(q - batch));
    const uint32_t cs = __shfl_sync(0xffffffffu, cb_cur, static_cast<int>(q - batch));
    m = 0;
    if (jrow == kPast) return;
    if (static_cast<uint64_t>(r) < n_rows) {
      const bool hot = !SOA && cs != 0xFFFFFFFFu;
      const uintptr_t a = hot ? cache + static_cast<uint64_t>(cs) * stride
                              : codes + static_cast<uint64_t>(r) * stride;
      const uintptr_t end = hot ? cache_end : tbl_end;
      const uintptr_t a0 = a & ~static_cast<uintptr_t>(15);
      const uint32_t mis = static_cast<uint32_t>(a - a0);
      const uint32_t nch = (mis + code_bytes + (SOA ? 0u : 2u) + 15) >> 4;
      if (lane < nch) {
        const uintptr_t src = a0 + 16u * lane;
        if (SOA || end - src >= 16) v = __ldg(reinterpret_cast<const uint4*>(src));
        else v = load_partial16(reinterpret_cast<const uint8_t*>(src),
                                static_cast<uint32_t>(end - src));
      }
      if (SOA) ab = __ldg(p.alpha + r);
      m = 1u | (mis << 8);
    } else if (lane == 0) {
      atomicOr(p.status, 1u);
    }
  };

#pragma unroll
  for (int s = 0; s < PF - 1; ++s) issue(s, rv[s], rm[s], rj[s], ra[s]);

  const uint4 zero = make_uint4(0, 0, 0, 0);
  bool done = false;
  for (uint32_t g = 0; !done; g += PF) {
#pragma unroll
    for (int s = 0; s < PF; ++s) {
      if (!done && rj[s] == kPast) done = true;
      if (!done) {
        const uint32_t i = g + s;
        const int sn = (s + PF - 1) % PF;
        issue(i + PF - 1, rv[sn], rm[sn], rj[sn], ra[sn]);
        const uint32_t m = rm[s];
        uint4* orow = reinterpret_cast<uint4*>(p.out) + static_cast<uint64_t>(rj[s]) * (d >> 3);
        if (m & 1u) {
          const uint32_t mis = m >> 8;
          const uint32_t nch = (mis + code_bytes + (SOA ? 0u : 2u) + 15) >> 4;
          if (lane < nch) *reinterpret_cast<uint4*>(sb + 16u * lane) = rv[s];
          __syncwarp();
          uint8_t* code = sb + mis;
          if (lane == 0)
            *reinterpret_cast<uint16_t*>(code - 2) =
                *reinterpret_cast<const uint16_t*>(code + code_bytes - 2);
          const uint16_t abits = SOA ? ra[s] : *reinterpret_cast<const uint16_t*>(code + code_bytes);
          __syncwarp();
          const float a = __uint_as_float(static_cast<uint32_t>(abits) << 16);
          const uint32_t ex = (abits >> 7) & 0xFFu;
          const uint32_t* w = reinterpret_cast<const uint32_t*>(sb - kStagePrefix);
          const uint32_t boff = (kStagePrefix + mis) * 8;
          if ((abits & 0x7FFFu) == 0 || (ex - 113u) <= 29u) {
            const __half ah = __float2half_rn(a);
            decode_row<K, CPL, true, REP>(w, boff, d, smem, lane, __half_as_ushort(ah), a, orow);
          } else {
            decode_row<K, CPL, false, REP>(w, boff, d, smem, lane, 0, a, orow);
          }
        } else {
          for (uint32_t c = lane; c < (d >> 3); c += 32) __stcs(orow + c, zero);
        }
        __syncwarp();
      }
    }
  }
}

}  // namespace cpk

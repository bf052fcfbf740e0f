// cp_kernels_mixed.cuh -- lookup-decode of a table with one bit rate per row.
//
// The pages try frequency-based bit allocation (a code rate per row chosen from
// access counts) and find its gains inconsistent across text domains
// ("2비트 코드와 공유 트렐리스로 n-gram 룩업 테이블을 4~8배 압축한다", section
// 전제와 한계).  A mixed-rate table stores row r's record (code at rate k_r, then
// the bf16 scale) at bytes [offsets[r], offsets[r+1]); k_r = (R_r - 2) * 16 / d
// follows from the record length, so the offset table is the only extra data.
// The decode steps are the HBM-path kernel's, with the rate dispatched per row: each lane
// loads its batch row's two offsets together with the id, and the decode picks
// decode_row<k> by a warp-uniform switch.
#pragma once

#include "cp_kernels.cuh"

namespace cpk {

// Persistent grid, one CTA of kMaxWarps warps per SM: each row needs three
// dependent loads (id, then its two offsets, then the record), which the batch
// look-ahead of a persistent warp hides; the non-persistent form of the
// single-rate kernel, which starts that chain once per CTA, ran 30 % slower here.
constexpr int kPfMixed = 2;                            // record stages per warp
constexpr int kLutRepMixed = 16;                       // LUT replicas (filled once per SM)

template <int CPL>
__global__ void __launch_bounds__(kMaxWarps * 32, 1)
    lookup_decode_mixed_kernel(const DecodeParams p, const uint64_t* __restrict__ offsets) {
  constexpr int PF = kPfMixed;
  constexpr int REP = kLutRepMixed;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const uint32_t lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  constexpr int kLutBytes = lut_bytes(REP);
  fill_lut<REP>(smem, p.lut, tid, blockDim.x);
  __syncthreads();

  const uint32_t stage_bytes = p.stage_bytes;
  const uint32_t d = p.d;
  const uint64_t n_rows = p.n_rows;
  const uintptr_t codes = reinterpret_cast<uintptr_t>(p.codes);
  const uintptr_t tbl_end = codes + p.table_bytes;
  uint8_t* stages = smem + kLutBytes + static_cast<size_t>(warp) * PF * stage_bytes;
  uint32_t* meta = reinterpret_cast<uint32_t*>(smem + kLutBytes +
                                               static_cast<size_t>(nwarps) * PF * stage_bytes) +
                   warp * PF * 2;
  const uint32_t stages_sa = smem_addr(stages) + kStagePrefix;

  const uint64_t W = static_cast<uint64_t>(gridDim.x) * nwarps;
  const uint64_t gw = static_cast<uint64_t>(blockIdx.x) * nwarps + warp;
  const uint64_t lo = gw * p.n / W;
  const uint64_t hi = (gw + 1) * p.n / W;
  if (lo >= hi) return;
  const uint32_t cnt = static_cast<uint32_t>(hi - lo);

  // ids and their record offsets, 32 rows per batch, one batch of look-ahead
  const int64_t* ids = p.idx + lo;
  auto load_batch = [&](uint32_t q, int64_t& r, uint64_t& o0, uint64_t& o1) {
    r = -1;
    o0 = o1 = 0;
    if (q < cnt) {
      r = __ldg(ids + q);
      if (static_cast<uint64_t>(r) < n_rows) {
        o0 = __ldg(offsets + r);
        o1 = __ldg(offsets + r + 1);
      }
    }
  };
  int64_t ib_cur, ib_nxt;
  uint64_t a_cur, a_nxt, b_cur, b_nxt;
  load_batch(lane, ib_cur, a_cur, b_cur);
  load_batch(lane + 32, ib_nxt, a_nxt, b_nxt);
  uint32_t batch = 0;

  auto issue = [&](uint32_t q) {
    if (q - batch >= 32) {
      batch += 32;
      ib_cur = ib_nxt;
      a_cur = a_nxt;
      b_cur = b_nxt;
      load_batch(batch + 32 + lane, ib_nxt, a_nxt, b_nxt);
    }
    const int src_lane = static_cast<int>(q - batch);
    const int64_t r = __shfl_sync(0xffffffffu, ib_cur, src_lane);
    const uint64_t o0 = __shfl_sync(0xffffffffu, a_cur, src_lane);
    const uint64_t o1 = __shfl_sync(0xffffffffu, b_cur, src_lane);
    const uint32_t st = q & (PF - 1);
    const uint32_t sa = stages_sa + st * stage_bytes;
    uint32_t m = 0;
    if (static_cast<uint64_t>(r) < n_rows) {            // record lengths validated at load
      const uint32_t R = static_cast<uint32_t>(o1 - o0);
      const uint32_t k = (R - 2) * 16 / d;
      const uintptr_t a = codes + o0;
      const uintptr_t a0 = a & ~static_cast<uintptr_t>(15);
      const uint32_t mis = static_cast<uint32_t>(a - a0);
      const uint32_t nch = (mis + R + 15) >> 4;
      for (uint32_t c = lane; c < nch; c += 32) {
        const uintptr_t src = a0 + 16u * c;
        const uintptr_t left = tbl_end - src;
        cp_async16(sa + 16u * c, reinterpret_cast<const void*>(src),
                   left < 16 ? static_cast<uint32_t>(left) : 16u);
      }
      m = 1u | ((k - 3) << 4) | (mis << 8);
    } else if (lane == 0) {
      atomicOr(p.status, 1u);
    }
    if (lane == 0) meta[2 * st] = m;
    cp_async_commit();
  };

#pragma unroll
  for (int q = 0; q < PF - 1; ++q) {
    if (static_cast<uint32_t>(q) < cnt) issue(q);
    else cp_async_commit();
  }

  const uint4 zero = make_uint4(0, 0, 0, 0);
  uint4* orow = reinterpret_cast<uint4*>(p.out) + lo * (d >> 3);
  for (uint32_t i = 0; i < cnt; ++i, orow += (d >> 3)) {
    if (i + PF - 1 < cnt) issue(i + PF - 1);
    else cp_async_commit();
    cp_async_wait<PF - 1>();
    __syncwarp();
    const uint32_t st = i & (PF - 1);
    uint8_t* sb = stages + st * stage_bytes + kStagePrefix;
    const uint32_t m = meta[2 * st];
    if (m & 1u) {
      const uint32_t mis = m >> 8;
      const uint32_t k = 3 + ((m >> 4) & 3u);
      const uint32_t code_bytes = d * k / 16;
      uint8_t* code = sb + mis;
      if (lane == 0)
        *reinterpret_cast<uint16_t*>(code - 2) =
            *reinterpret_cast<const uint16_t*>(code + code_bytes - 2);
      const uint16_t abits = *reinterpret_cast<const uint16_t*>(code + code_bytes);
      __syncwarp();
      const float a = __uint_as_float(static_cast<uint32_t>(abits) << 16);
      const uint32_t ex = (abits >> 7) & 0xFFu;
      const uint32_t* w = reinterpret_cast<const uint32_t*>(sb - kStagePrefix);
      const uint32_t boff = (kStagePrefix + mis) * 8;
      const bool f16 = (abits & 0x7FFFu) == 0 || (ex - 113u) <= 29u;
      const uint16_t ah = f16 ? __half_as_ushort(__float2half_rn(a)) : 0;
#define CP_MIXED_CASE(KK)                                                              \
  case KK:                                                                             \
    if (f16) decode_row<KK, CPL, true, REP>(w, boff, d, smem, lane, ah, a, orow);      \
    else decode_row<KK, CPL, false, REP>(w, boff, d, smem, lane, 0, a, orow);          \
    break;
      switch (k) {
        CP_MIXED_CASE(3)
        CP_MIXED_CASE(4)
        CP_MIXED_CASE(5)
        default:
          CP_MIXED_CASE(6)
      }
#undef CP_MIXED_CASE
    } else {
      for (uint32_t c = lane; c < (d >> 3); c += 32) __stcs(orow + c, zero);
    }
    __syncwarp();
  }
}

// Load-time check of a mixed table: every record length gives k in {3,..,6},
// offsets[0] is 0, and every record starts 2-byte aligned.  bad: set to 1 otherwise.
__global__ void check_mixed_offsets_kernel(const uint64_t* __restrict__ offsets, uint64_t n_rows,
                                           uint32_t d, uint32_t* __restrict__ bad);

}  // namespace cpk

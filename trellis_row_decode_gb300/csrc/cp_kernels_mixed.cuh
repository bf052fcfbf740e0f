// cp_kernels_mixed.cuh -- lookup-decode of a table with one bit rate per row.
//
// The pages try frequency-based bit allocation (a code rate per row chosen from
// access counts) and find its gains inconsistent across text domains
// ("2비트 코드와 공유 트렐리스로 n-gram 룩업 테이블을 4~8배 압축한다", section
// 전제와 한계).  A mixed-rate table stores row r's record (code at rate k_r, then
// the bf16 scale) at bytes [offsets[r], offsets[r+1]); k_r = (R_r - 2) * 16 / d
// follows from the record length, so the offset table is the only extra data.
// The decode steps are the HBM-path kernel's, with the rate taken per row.  Each
// row needs its id, then its two offsets, then its record: the first lanes of a
// warp resolve the warp's rows (id -> offset, rate) before any record is queued.
#pragma once

#include "cp_kernels.cuh"

namespace cpk {

// Steps 4c..4c+3 of a row from x at runtime rate K (the shifts are registers,
// not immediates): one decode body serves every rate of a mixed table, which
// keeps the kernel's code small enough for the instruction cache (a copy per
// rate, with 64 warps per SM in different rates, missed it constantly).
// x = hi:lo holds the chunk's bits from bit 0 of its first window; the window
// of step j starts at bit K j < 32, so one 32-bit funnel shift extracts it.
template <bool F16, int REP>
__device__ __forceinline__ uint4 decode_chunk_rk(uint32_t lo, uint32_t hi, uint32_t K,
                                                 const uint8_t* lut, uint32_t lane4,
                                                 uint16_t a_h, float a) {
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t s = __funnelshift_r(lo, hi, K * j) & 0xFFFFu;
    const uint32_t v = lut_word<REP>(lut, s, lane4);
    o[j] = F16 ? scale_pair_f16(v, a_h) : scale_pair_f32(v, a);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// A staged row at runtime rate K by LPR lanes (sub = this lane's index among
// them), each lane CPL 16-byte chunks c = sub + LPR m whose bit offsets differ by
// K * LPR / 8 whole words, so one shift amount serves all of them (d == LPR * CPL
// * 8); CPL == 0: a loop over the d / 8 chunks with the whole warp.
template <int CPL, bool F16, int REP, int LPR>
__device__ __forceinline__ void decode_row_rk(uint32_t K, const uint32_t* w, uint32_t boff,
                                              uint32_t d, const uint8_t* lut, uint32_t lane,
                                              uint32_t sub, uint16_t a_h, float a, uint4* orow) {
  const uint32_t lane4 = (lane & (REP - 1)) << 2;
  if constexpr (CPL > 0) {
    const uint32_t P0 = boff + K * (4 * sub + 1) - 16;
    const uint32_t* w0 = w + (P0 >> 5);
    const uint32_t sh = P0 & 31;
    const uint32_t step = K * (LPR / 8);                // words between chunks c and c + LPR
#pragma unroll
    for (int m = 0; m < CPL; ++m) {
      const uint64_t x = funnel64(w0[step * m], w0[step * m + 1], sh);
      __stcs(orow + sub + LPR * m,
             decode_chunk_rk<F16, REP>(static_cast<uint32_t>(x), static_cast<uint32_t>(x >> 32), K,
                                       lut, lane4, a_h, a));
    }
  } else {
    for (uint32_t c = lane; c < (d >> 3); c += 32) {
      const uint32_t P = boff + K * (4 * c + 1) - 16;
      const uint64_t x = funnel64(w[P >> 5], w[(P >> 5) + 1], P & 31);
      __stcs(orow + c, decode_chunk_rk<F16, REP>(static_cast<uint32_t>(x),
                                                 static_cast<uint32_t>(x >> 32), K, lut, lane4,
                                                 a_h, a));
    }
  }
}

// Non-persistent decode of a mixed-rate table, the single-rate block kernel's
// work mapping (kBlkWarps warps x ROWS rows per CTA, warp w taking positions
// w, w + kBlkWarps, ...).  Rows shorter than 1024 (d = 256, 512) are decoded
// G = 1024 / d at a time by groups of 32 / G lanes, each row at its own rate (the
// rate is a register of the lane group, so rows of different rates in one warp
// do not diverge).  CPL: chunks per lane of a whole-warp row when d == 256 * CPL,
// else 0.
template <int CPL, int REP, int ROWS>
__global__ void __launch_bounds__(kBlkWarps * 32)
    lookup_decode_mixed_block_kernel(const DecodeParams p, const uint64_t* __restrict__ offsets) {
  constexpr int G = (CPL == 1) ? 4 : (CPL == 2) ? 2 : 1;   // rows side by side in a warp
  constexpr int LPR = 32 / G;                               // lanes per row
  constexpr int CPLG = CPL * G;                             // chunks per lane
  constexpr int STEPS = ROWS / G;
  static_assert(ROWS % G == 0, "rows per warp must be a multiple of the rows per step");
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const uint32_t lane = tid & 31;
  const int warp = tid >> 5;
  const uint32_t slot = lane / LPR;                         // this lane's row within a step
  const uint32_t sub = lane % LPR;
  constexpr int kLutBytes = lut_bytes(REP);
  const uint32_t stage_bytes = p.stage_bytes;
  const uint32_t d = p.d;
  uint8_t* stages = smem + kLutBytes + static_cast<size_t>(warp) * ROWS * stage_bytes;
  const uint32_t stages_sa = smem_addr(stages) + kStagePrefix;
  const uintptr_t codes = reinterpret_cast<uintptr_t>(p.codes);
  const uintptr_t tbl_end = codes + p.table_bytes;

  const uint64_t first = static_cast<uint64_t>(blockIdx.x) * (kBlkWarps * ROWS) + warp;
  const uint64_t n = p.n;
  // lane t resolves the warp's row t: bit 0 = id in range, bits 1..2 = k - 3,
  // bits 4.. = byte offset of the record (record lengths were checked at load)
  uint64_t my_loc = 0;
  if (lane < static_cast<uint32_t>(ROWS)) {
    const uint64_t j = first + static_cast<uint64_t>(lane) * kBlkWarps;
    if (j < n) {
      const int64_t r = __ldg(p.idx + j);
      if (static_cast<uint64_t>(r) < p.n_rows) {
        const uint64_t o0 = __ldg(offsets + r);
        // code bytes c = d k / 16 with k in {3, .., 6} (checked at load), so 16 c
        // = k d: k - 3 by three comparisons (a 64-bit division by the runtime d
        // cost the warp a long instruction sequence per row group)
        const uint32_t c16 = static_cast<uint32_t>(__ldg(offsets + r + 1) - o0 - 2) * 16;
        const uint32_t k3 = (c16 > 3 * d) + (c16 > 4 * d) + (c16 > 5 * d);
        my_loc = (o0 << 4) | (static_cast<uint64_t>(k3) << 1) | 1u;
      } else {
        atomicOr(p.status, 1u);
      }
    }
  }
  uint32_t m[STEPS];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const uint32_t t = s * G + slot;                   // row of this lane's group
    const uint64_t l = __shfl_sync(0xffffffffu, my_loc, static_cast<int>(t));
    m[s] = 0;
    if ((l & 1u) && first + static_cast<uint64_t>(t) * kBlkWarps < n) {
      const uint32_t k = 3 + static_cast<uint32_t>((l >> 1) & 3u);
      const uint32_t R = d * k / 16 + 2;
      const uintptr_t a = codes + (l >> 4);
      const uintptr_t a0 = a & ~static_cast<uintptr_t>(15);
      const uint32_t mis = static_cast<uint32_t>(a - a0);
      const uint32_t nch = (mis + R + 15) >> 4;
      const uint32_t sa = stages_sa + t * stage_bytes;
      for (uint32_t c = sub; c < nch; c += LPR) {
        const uintptr_t src = a0 + 16u * c;
        const uintptr_t left = tbl_end - src;          // > 0: src lies inside the table
        cp_async16(sa + 16u * c, reinterpret_cast<const void*>(src),
                   left < 16 ? static_cast<uint32_t>(left) : 16u);
      }
      m[s] = 1u | ((k - 3) << 4) | (mis << 8);
    }
    cp_async_commit();
  }

  fill_lut<REP>(smem, p.lut, tid, kBlkWarps * 32);
  __syncthreads();

  const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    if (first + static_cast<uint64_t>(s * G) * kBlkWarps >= n) break;   // no row of this step
    cp_async_wait_n(STEPS - 1 - s);
    __syncwarp();
    const uint32_t t = s * G + slot;
    const uint64_t j = first + static_cast<uint64_t>(t) * kBlkWarps;
    uint4* orow = reinterpret_cast<uint4*>(p.out) + j * (d >> 3);
    uint8_t* sb = stages + t * stage_bytes + kStagePrefix;
    const bool has = (m[s] & 1u) != 0;
    const uint32_t mis = m[s] >> 8;
    const uint32_t k = 3 + ((m[s] >> 4) & 3u);
    const uint32_t code_bytes = d * k / 16;
    uint8_t* code = sb + mis;
    // tail-biting splice: the code's last 16 bits just below bit 0
    if (has && sub == 0)
      *reinterpret_cast<uint16_t*>(code - 2) =
          *reinterpret_cast<const uint16_t*>(code + code_bytes - 2);
    __syncwarp();
    if (has) {
      const uint16_t abits = *reinterpret_cast<const uint16_t*>(code + code_bytes);
      const float a = __uint_as_float(static_cast<uint32_t>(abits) << 16);
      const uint32_t ex = (abits >> 7) & 0xFFu;
      const uint32_t* w = reinterpret_cast<const uint32_t*>(sb - kStagePrefix);
      const uint32_t boff = (kStagePrefix + mis) * 8;
      if ((abits & 0x7FFFu) == 0 || (ex - 113u) <= 29u) {   // |alpha| in [2^-14, 2^16) or 0
        const uint16_t ah = __half_as_ushort(__float2half_rn(a));
        decode_row_rk<CPLG, true, REP, LPR>(k, w, boff, d, smem, lane, sub, ah, a, orow);
      } else {
        decode_row_rk<CPLG, false, REP, LPR>(k, w, boff, d, smem, lane, sub, 0, a, orow);
      }
    } else if (j < n) {
      for (uint32_t c = sub; c < (d >> 3); c += LPR) __stcs(orow + c, zero);
    }
  }
}

// Load-time check of a mixed table: every record length gives k in {3,..,6},
// offsets[0] is 0, and every record starts 2-byte aligned.  bad: set to 1 otherwise.
__global__ void check_mixed_offsets_kernel(const uint64_t* __restrict__ offsets, uint64_t n_rows,
                                           uint32_t d, uint32_t* __restrict__ bad);

}  // namespace cpk

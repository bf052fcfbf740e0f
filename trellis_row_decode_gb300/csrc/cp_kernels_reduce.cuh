// cp_kernels_reduce.cuh -- lookup-decode fused with a weighted group readout.
#pragma once

#include "cp_kernels.cuh"

namespace cpk {

// ---------------------------------------------------------------------------
// Decode fused with a weighted readout.  The pages hand the restored rows to
// "the existing readout" ([P4] section 무엇과 다른가); this synthetic readout
// sums each group of `group` consecutive lookups (e.g. the rows of one token and
// layer): out[g] = bf16_rn(acc), acc = fmaf(w_i, float(row_i), acc) over the
// group in lookup order, starting from +0, where row_i is the bf16 row the plain
// lookup-decode would write (zeros for an out-of-range id) and w_i = 1 when no
// weights are given.  Only one bf16 row per group leaves the SM.
// A warp owns a contiguous range of groups; records stream through the same
// cp.async ring; each lane keeps CPL x 8 fp32 accumulators in registers.
#ifndef CP_REDUCE_WARPS
#define CP_REDUCE_WARPS 32
#endif
constexpr int kReduceWarps = CP_REDUCE_WARPS;

// acc (a pair of fp32 accumulators in one 64-bit register) += w2 * v, pairwise
// (fma.rn.f32x2: each lane an fp32 fused multiply-add with one rounding, as fmaf).
__device__ __forceinline__ void fma_pair(unsigned long long& acc, unsigned long long w2,
                                         uint32_t lo_bits, uint32_t hi_bits) {
  unsigned long long v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(lo_bits), "r"(hi_bits));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(w2), "l"(v));
}

__device__ __forceinline__ unsigned long long pair_of(float x) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
  return r;
}

// One chunk (8 coordinates): the bf16 row values, widened exactly, times the
// lookup's weight, added to the four accumulator pairs.
template <int K, bool F16, int REP>
__device__ __forceinline__ void acc_chunk(uint64_t x, const uint8_t* lut, uint32_t lane4,
                                          uint16_t a_h, float a, unsigned long long w2,
                                          unsigned long long* acc) {
  const uint4 o = decode_chunk<K, F16, REP>(x, lut, lane4, a_h, a);
  const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) fma_pair(acc[j], w2, ow[j] << 16, ow[j] & 0xFFFF0000u);
}

template <int K, bool SOA, int PF, int CPL>
__global__ void __launch_bounds__(kReduceWarps * 32, 1)
    lookup_decode_reduce_kernel(const DecodeParams p, const float* __restrict__ weights,
                                uint32_t group, uint64_t n_groups) {
  static_assert(CPL >= 1 && CPL <= 4, "d in {256, 512, 1024}");
  constexpr int REP = 32;
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

  const uint32_t stage_bytes = p.stage_bytes;
  const uint32_t code_bytes = p.code_bytes;
  const uint32_t d = p.d;
  const uint64_t n_rows = p.n_rows;
  const uint64_t stride = p.stride;
  const uintptr_t codes = reinterpret_cast<uintptr_t>(p.codes);
  const uintptr_t tbl_end = codes + p.table_bytes;
  uint8_t* stages = smem + kLutBytes + static_cast<size_t>(warp) * PF * stage_bytes;
  uint32_t* meta = reinterpret_cast<uint32_t*>(smem + kLutBytes +
                                               static_cast<size_t>(nwarps) * PF * stage_bytes) +
                   warp * PF * 2;
  const uint32_t stages_sa = smem_addr(stages) + kStagePrefix;

  const uint64_t W = static_cast<uint64_t>(gridDim.x) * nwarps;
  const uint64_t gw = static_cast<uint64_t>(blockIdx.x) * nwarps + warp;
  const uint64_t g_lo = gw * n_groups / W;
  const uint64_t g_hi = (gw + 1) * n_groups / W;
  if (g_lo >= g_hi) return;
  const uint64_t lo = g_lo * group;                       // first lookup of this warp
  const uint32_t cnt = static_cast<uint32_t>((g_hi - g_lo) * group);

  const int64_t* ids = p.idx + lo;
  int64_t ib_cur = (lane < cnt) ? __ldg(ids + lane) : 0;
  int64_t ib_nxt = (lane + 32 < cnt) ? __ldg(ids + 32 + lane) : 0;
  uint32_t batch = 0;

  auto issue = [&](uint32_t q) {
    if (q - batch >= 32) {
      batch += 32;
      ib_cur = ib_nxt;
      ib_nxt = (batch + 32 + lane < cnt) ? __ldg(ids + batch + 32 + lane) : 0;
    }
    const int64_t r = __shfl_sync(0xffffffffu, ib_cur, static_cast<int>(q - batch));
    const uint32_t st = q & (PF - 1);
    const uint32_t sa = stages_sa + st * stage_bytes;
    uint32_t m = 0;
    if (static_cast<uint64_t>(r) < n_rows) {
      const uintptr_t a = codes + static_cast<uint64_t>(r) * stride;
      const uintptr_t a0 = a & ~static_cast<uintptr_t>(15);
      const uint32_t mis = static_cast<uint32_t>(a - a0);
      const uint32_t nch = (mis + code_bytes + (SOA ? 0u : 2u) + 15) >> 4;
      if (lane < nch) {
        const uintptr_t src = a0 + 16u * lane;
        uint32_t bytes = 16;
        if (!SOA) {
          const uintptr_t left = tbl_end - src;
          bytes = left < 16 ? static_cast<uint32_t>(left) : 16u;
        }
        cp_async16(sa + 16u * lane, reinterpret_cast<const void*>(src), bytes);
      }
      if (SOA && lane == 31) {
        const uint64_t r2 = static_cast<uint64_t>(r) & ~1ull;
        cp_async4(sa - kStagePrefix + p.alpha_slot, p.alpha + r2, (r2 + 1 < n_rows) ? 4u : 2u);
      }
      m = 1u | ((static_cast<uint32_t>(r) & 1u) << 1) | (mis << 8);
    } else if (lane == 0) {
      atomicOr(p.status, 1u);
    }
    if (lane == 0) {
      meta[2 * st] = m;
      meta[2 * st + 1] = __float_as_uint(weights ? __ldg(weights + lo + q) : 1.0f);
    }
    cp_async_commit();
  };

#pragma unroll
  for (int q = 0; q < PF - 1; ++q) {
    if (static_cast<uint32_t>(q) < cnt) issue(q);
    else cp_async_commit();
  }

  unsigned long long acc[CPL][4];                       // fp32 pairs (coordinates 2j, 2j+1)
#pragma unroll
  for (int m = 0; m < CPL; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[m][e] = 0ull;
  uint32_t in_group = 0;
  uint4* orow = reinterpret_cast<uint4*>(p.out) + g_lo * (d >> 3);
  const uint32_t lane4 = lane << 2;

  for (uint32_t i = 0; i < cnt; ++i) {
    if (i + PF - 1 < cnt) issue(i + PF - 1);
    else cp_async_commit();
    cp_async_wait<PF - 1>();
    __syncwarp();
    const uint32_t st = i & (PF - 1);
    uint8_t* sb = stages + st * stage_bytes + kStagePrefix;
    const uint32_t m = meta[2 * st];
    const unsigned long long wgt = pair_of(__uint_as_float(meta[2 * st + 1]));
    if (m & 1u) {
      const uint32_t mis = m >> 8;
      uint8_t* code = sb + mis;
      if (lane == 0)
        *reinterpret_cast<uint16_t*>(code - 2) =
            *reinterpret_cast<const uint16_t*>(code + code_bytes - 2);
      const uint16_t abits = SOA ? *reinterpret_cast<const uint16_t*>(
                                       sb - kStagePrefix + p.alpha_slot + 2 * ((m >> 1) & 1u))
                                 : *reinterpret_cast<const uint16_t*>(code + code_bytes);
      __syncwarp();
      const float a = __uint_as_float(static_cast<uint32_t>(abits) << 16);
      const uint32_t ex = (abits >> 7) & 0xFFu;
      const uint32_t* w = reinterpret_cast<const uint32_t*>(sb - kStagePrefix);
      const uint32_t P0 = (kStagePrefix + mis) * 8 + K * (4 * lane + 1) - 16;
      const uint32_t* w0 = w + (P0 >> 5);
      const uint32_t sh = P0 & 31;
      if ((abits & 0x7FFFu) == 0 || (ex - 113u) <= 29u) {
        const uint16_t ah = __half_as_ushort(__float2half_rn(a));
#pragma unroll
        for (int c = 0; c < CPL; ++c)
          acc_chunk<K, true, REP>(funnel64(w0[4 * K * c], w0[4 * K * c + 1], sh), smem, lane4, ah,
                                  a, wgt, acc[c]);
      } else {
#pragma unroll
        for (int c = 0; c < CPL; ++c)
          acc_chunk<K, false, REP>(funnel64(w0[4 * K * c], w0[4 * K * c + 1], sh), smem, lane4, 0,
                                   a, wgt, acc[c]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) fma_pair(acc[c][e], wgt, 0u, 0u);   // w * (+0) added
    }
    __syncwarp();
    if (++in_group == group) {                            // group complete: one bf16 row
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float lo, hi;
          asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc[c][j]));
          const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
          o[j] = *reinterpret_cast<const uint32_t*>(&r);
        }
        __stcs(orow + lane + 32 * c, make_uint4(o[0], o[1], o[2], o[3]));
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[c][e] = 0ull;
      }
      orow += d >> 3;
      in_group = 0;
    }
  }
}

}  // namespace cpk

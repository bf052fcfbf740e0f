// cp_kernels.cuh -- sm_103a kernels of the CP lookup-decode (internal header).
//
// Pages cited by title: [P4] "2비트 코드와 공유 트렐리스로 n-gram 룩업 테이블을
// 4~8배 압축한다" (onedev.kr/papers/1189).  The kernel is the "fused kernel" of
// section 무엇과 다른가 (how it differs): it fetches only the requested records,
// restores each as e_hat = alpha * f(c) (section 어떻게 동작하나, how it works) and
// writes the rows in the original lookup order, duplicates included.
//
// Work mapping (GB300: 152 SMs, 228 KB shared memory per SM):
//   * one persistent CTA of up to 32 warps per SM; each warp owns a contiguous
//     range of lookups and decodes one row at a time;
//   * the record of a row is copied with 16-byte cp.async (L2 only) into a
//     per-warp ring of PF shared-memory stages, PF-1 rows ahead of the row being
//     decoded, so record latency overlaps decode and stores; the last 16-byte
//     piece of the table is clamped with the copy's source size (zero fill);
//   * the shared LUT (512 fp16 pairs) is expanded in shared memory to 1024
//     entries (the sign of y1 folded in, indexed by hash bits 14..23) and
//     replicated 32 times, word (entry * 32 + lane): every lane reads its own
//     bank, so a warp-wide LUT read is one wavefront;
//   * a lane produces 8 outputs (4 trellis steps, 16 bytes) per chunk; chunk c
//     needs code bits [k(4c+1) - 16, k(4c+4)), at most 34 bits, read from the
//     stage as one 64-bit funnel of two words; chunks with negative start
//     (tail-biting wrap) splice the code's last bits below its first bits;
//   * per step: hash (one IMAD), index (shift + and), one LDS, fp16 -> fp32,
//     two fp32 products by alpha (exact: 8 x 11 significant bits), one
//     cvt.rn.bf16x2; each chunk is one 16-byte streaming store (st.global.cs).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace cpk {

constexpr int kLutEntries = 1024;                  // 512 pairs x sign of y1
constexpr int kLutReplicas = 32;                   // one per lane / bank
constexpr int kLutBytes = kLutEntries * kLutReplicas * 4;   // 128 KB
constexpr int kMaxWarps = 32;

struct DecodeParams {
  const uint8_t* codes;     // AoS: records base; SoA: code array base (16-byte aligned)
  const uint16_t* alpha;    // SoA: alpha array (nullptr for AoS)
  uint64_t n_rows;
  uint64_t table_bytes;     // AoS: n_rows * R, bytes readable from `codes`
  uint32_t d;
  uint32_t stride;          // AoS: record bytes R; SoA: code stride S
  uint32_t code_bytes;      // d * k / 16
  uint32_t stage_bytes;     // bytes of one shared-memory stage (multiple of 16)
  uint32_t alpha_slot;      // SoA: offset of the 4-byte alpha copy inside a stage
  const uint32_t* lut;      // 512 words: fp16 y0 (low half) | fp16 y1 (high half)
  const int64_t* idx;
  uint64_t n;
  uint16_t* out;            // bf16 [n][d], 16-byte aligned
  uint32_t* status;         // bit 0: an id was out of range
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared, L2 only; bytes in [1, 16], rest zero-filled.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_addr(dst)),
               "l"(src), "r"(bytes)
               : "memory");
}

// 4-byte async copy global -> shared; bytes in [0, 4], rest zero-filled.
__device__ __forceinline__ void cp_async4(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_addr(dst)), "l"(src),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// 64 bits of the staged bytes starting at bit P (bit 0 = LSB of byte 0).
// At least 64 - (P & 31) >= 33 of them are meaningful.
__device__ __forceinline__ uint64_t bits64(const uint32_t* w, uint32_t P) {
  const uint32_t i = P >> 5;
  const uint64_t v = (static_cast<uint64_t>(w[i + 1]) << 32) | w[i];
  return v >> (P & 31);
}

// Steps 4c..4c+3 of a row: 8 bf16 outputs (16 bytes).
template <int K>
__device__ __forceinline__ uint4 decode_chunk(uint64_t x, const uint32_t* lut_lane, float a) {
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t s = static_cast<uint32_t>(x >> (K * j)) & 0xFFFFu;
    const uint32_t h = s * s + s;                       // mod 2^32
    const uint32_t e = (h >> 14) & (kLutEntries - 1);   // bit 9 of e = bit 23 of h (sign)
    const uint32_t v = lut_lane[e * kLutReplicas];
    const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&v));
    const __nv_bfloat162 r = __floats2bfloat162_rn(a * y.x, a * y.y);
    o[j] = *reinterpret_cast<const uint32_t*>(&r);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// K: bits per step (3..6).  SOA: read the SoA copy.  PF: stages per warp.
template <int K, bool SOA, int PF>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) lookup_decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* lut_s = reinterpret_cast<uint32_t*>(smem);
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;

  // Shared LUT: entry e -> pair e & 511, y1 negated for e >= 512; 32 copies.
  for (int q = tid; q < kLutEntries * kLutReplicas / 4; q += blockDim.x) {
    const int e = q >> 3;                               // 8 uint4 per entry
    uint32_t v = __ldg(p.lut + (e & 511));
    if (e & 512) v ^= 0x80000000u;
    reinterpret_cast<uint4*>(lut_s)[q] = make_uint4(v, v, v, v);
  }
  __syncthreads();

  uint8_t* stages = smem + kLutBytes + static_cast<size_t>(warp) * PF * p.stage_bytes;
  uint32_t* meta =
      reinterpret_cast<uint32_t*>(smem + kLutBytes + static_cast<size_t>(nwarps) * PF * p.stage_bytes) +
      warp * PF;
  const uint32_t* lut_lane = lut_s + lane;

  const uint64_t W = static_cast<uint64_t>(gridDim.x) * nwarps;
  const uint64_t gw = static_cast<uint64_t>(blockIdx.x) * nwarps + warp;
  const uint64_t lo = gw * p.n / W;
  const uint64_t hi = (gw + 1) * p.n / W;
  if (lo >= hi) return;
  const uint64_t cnt = hi - lo;

  // Row ids, 32 per coalesced load, one batch of look-ahead.
  const int64_t* ids = p.idx + lo;
  int64_t ib_cur = (static_cast<uint64_t>(lane) < cnt) ? __ldg(ids + lane) : 0;
  int64_t ib_nxt = (static_cast<uint64_t>(lane) + 32 < cnt) ? __ldg(ids + 32 + lane) : 0;
  uint64_t batch = 0;

  const uint32_t C = p.d >> 3;                          // 16-byte chunks per row
  const uint32_t Lc = (p.d >> 1) * K;                   // code bits per row

  auto issue = [&](uint64_t q) {
    if (q - batch >= 32) {
      batch += 32;
      ib_cur = ib_nxt;
      ib_nxt = (batch + 32 + lane < cnt) ? __ldg(ids + batch + 32 + lane) : 0;
    }
    const int64_t r = __shfl_sync(0xffffffffu, ib_cur, static_cast<int>(q - batch));
    const uint32_t st = static_cast<uint32_t>(q % PF);
    uint8_t* sb = stages + st * p.stage_bytes;
    uint32_t m = 0;
    if (r >= 0 && static_cast<uint64_t>(r) < p.n_rows) {
      const uint8_t* A = p.codes + static_cast<uint64_t>(r) * p.stride;
      const uintptr_t a = reinterpret_cast<uintptr_t>(A);
      const uintptr_t a0 = a & ~static_cast<uintptr_t>(15);
      const uint32_t mis = static_cast<uint32_t>(a - a0);
      const uint32_t span = mis + p.code_bytes + (SOA ? 0u : 2u);
      const uint32_t nch = (span + 15) >> 4;
      const uintptr_t end = reinterpret_cast<uintptr_t>(p.codes) + p.table_bytes;
      for (uint32_t c = lane; c < nch; c += 32) {
        const uintptr_t src = a0 + 16u * c;
        uint32_t bytes = 16;
        if (!SOA && src + 16 > end) bytes = static_cast<uint32_t>(end - src);
        cp_async16(sb + 16u * c, reinterpret_cast<const void*>(src), bytes);
      }
      if (SOA && lane == 31) {
        const uint64_t r2 = static_cast<uint64_t>(r) & ~1ull;
        const uint32_t bytes = (r2 + 1 < p.n_rows) ? 4u : 2u;
        cp_async4(sb + p.alpha_slot, p.alpha + r2, bytes);
      }
      m = 1u | ((static_cast<uint32_t>(r) & 1u) << 1) | (mis << 8);
    } else if (lane == 0) {
      atomicOr(p.status, 1u);
    }
    if (lane == 0) meta[st] = m;
    cp_async_commit();
  };

#pragma unroll
  for (int q = 0; q < PF - 1; ++q) {
    if (static_cast<uint64_t>(q) < cnt) issue(q);
    else cp_async_commit();
  }

  for (uint64_t i = 0; i < cnt; ++i) {
    const uint64_t q = i + PF - 1;
    if (q < cnt) issue(q);
    else cp_async_commit();
    cp_async_wait<PF - 1>();
    __syncwarp();

    const uint32_t st = static_cast<uint32_t>(i % PF);
    const uint8_t* sb = stages + st * p.stage_bytes;
    const uint32_t m = meta[st];
    uint4* orow = reinterpret_cast<uint4*>(p.out) + (lo + i) * C;
    if (m & 1u) {
      const uint32_t mis = m >> 8;
      uint16_t abits;
      if (SOA) abits = *reinterpret_cast<const uint16_t*>(sb + p.alpha_slot + 2 * ((m >> 1) & 1u));
      else abits = *reinterpret_cast<const uint16_t*>(sb + mis + p.code_bytes);
      const float a = __uint_as_float(static_cast<uint32_t>(abits) << 16);
      const uint32_t* w = reinterpret_cast<const uint32_t*>(sb);
      const uint32_t boff = mis * 8;
      for (uint32_t c = lane; c < C; c += 32) {
        const int32_t pb = K * static_cast<int32_t>(4 * c + 1) - 16;
        uint64_t x;
        if (pb >= 0) {
          x = bits64(w, boff + static_cast<uint32_t>(pb));
        } else {                                        // tail-biting wrap
          const uint32_t nt = static_cast<uint32_t>(-pb);
          const uint64_t tail = bits64(w, boff + Lc - nt) & ((1ull << nt) - 1);
          x = tail | (bits64(w, boff) << nt);
        }
        st_stream(orow + c, decode_chunk<K>(x, lut_lane, a));
      }
    } else {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (uint32_t c = lane; c < C; c += 32) st_stream(orow + c, z);
    }
    __syncwarp();
  }
}

// AoS -> SoA repack: one warp per row, 2-byte granules (records are 2-byte aligned).
__global__ void repack_soa_kernel(const uint8_t* __restrict__ rec, uint64_t n_rows, uint32_t R,
                                  uint32_t code_bytes, uint32_t S, uint8_t* __restrict__ codes,
                                  uint16_t* __restrict__ alpha);

}  // namespace cpk

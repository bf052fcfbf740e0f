// cp_kernels.cuh -- sm_103a kernels of the CP lookup-decode (internal header).
//
// Pages cited by title: [P4] "2비트 코드와 공유 트렐리스로 n-gram 룩업 테이블을
// 4~8배 압축한다" (onedev.kr/papers/1189).  The kernel is the "fused kernel" of
// section 무엇과 다른가 (how it differs): it fetches only the requested records,
// restores each as e_hat = alpha * f(c) (section 어떻게 동작하나, how it works) and
// writes the rows in the original lookup order, duplicates included.
//
// Work mapping (GB300: 152 SMs, 228 KB shared memory per SM):
//   * HBM-resident tables: a non-persistent grid of small CTAs (8 warps, 4 rows
//     per warp, 32 consecutive lookups per CTA).  The hardware block scheduler
//     hands CTAs to SMs as they free up, so the 2 KB row writes advance through
//     the output in a narrow window and SMs that reach memory faster (the
//     imbalance between SMs is systematic on this part) take more CTAs.  With
//     ~40 rows per warp in static ranges, a persistent grid ran 10-20 % longer;
//   * host-resident tables (lookups visited grouped by row range): one
//     persistent CTA per SM over a contiguous slice of that order, a ring of PF
//     records per warp, PF-1 rows ahead of the row being decoded (the register
//     ring kernel of cp_kernels_host.cuh hands its slice to its warps in chunks
//     of 32; the kernel here, for d > 1024, gives each warp a fixed range);
//   * the record of a row is copied with 16-byte cp.async (L2 only) into a
//     shared-memory stage; the block kernel queues all of a warp's rows before
//     the CTA builds its LUT, so record latency overlaps the fill; the last
//     16-byte piece of the table is clamped with the copy's source size (zero
//     fill);
//   * the shared LUT (512 fp16 pairs) is expanded in shared memory to 1024
//     entries (the sign of y1 folded in, indexed by hash bits 14..23) with REP
//     copies of each entry, word (entry * REP + lane % REP).  REP = 32 makes a
//     warp-wide LUT read one wavefront; fewer copies cost bank conflicts (about
//     3 wavefronts at REP = 2) but a smaller fill: the block kernel, which fills
//     once per 32 rows, keeps 2 copies (8 KB); the persistent kernels keep 16
//     (device, filled once per SM) or 4 (host: the shared memory goes to a
//     deeper record ring, since the host link's throughput grows with the bytes
//     in flight);
//   * a record lands 16 bytes into its stage; once it has arrived, lane 0 copies
//     the code's last 16 bits (a whole halfword, since d*k/16 is even) to the
//     two bytes just below code bit 0, so the tail-biting wrap (windows that
//     start below bit 0 take the code's last bits) becomes a plain linear read;
//   * a lane produces 8 outputs (4 trellis steps, 16 bytes) per chunk; chunk c
//     needs code bits [k(4c+1) - 16, k(4c+4)), at most 34 bits, read from the
//     stage as one 64-bit funnel of two words; when d = 256 * CPL every lane
//     owns exactly CPL chunks c = lane + 32m whose bit offsets differ by 128k
//     (4k whole words), so one shift amount serves all of them and every other
//     offset is an immediate;
//   * per step: window (shift + and), hash (one IMAD), LUT byte offset (shift +
//     and, lane OR-ed in), one LDS, then alpha * y for both coordinates as one
//     mixed-precision fma.rn.f32.f16 each (alpha as fp16: exact for |alpha| in
//     [2^-14, 65504] or 0; the fp32 result of fp16 x fp16 is exact) and one
//     cvt.rn.bf16x2.f32; rows whose alpha is outside that range take an fp32
//     multiply path with identical results; each chunk is one 16-byte streaming
//     store (st.global.cs).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace cpk {

constexpr int kLutEntries = 1024;                  // 512 pairs x sign of y1
// Shared-memory LUT bytes with REP replicas (REP = 32: one per lane, no bank
// conflicts, 128 KB; REP = 4: 16 KB, leaving room for more record stages).
__host__ __device__ constexpr int lut_bytes(int rep) { return kLutEntries * rep * 4; }
__host__ __device__ constexpr int log2i(int v) { return v <= 1 ? 0 : 1 + log2i(v / 2); }
#ifndef CP_MAX_WARPS
#define CP_MAX_WARPS 32
#endif
constexpr int kMaxWarps = CP_MAX_WARPS;             // warps per CTA (one CTA per SM)

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
  const uint32_t* perm;     // processing order (PERM kernels): position i decodes lookup perm[i]
  const uint32_t* cslot;    // host path: cache slot per lookup (0xFFFFFFFF: not cached) or null
  const uint8_t* cache;     // host path: device copies of hot records, stride = record bytes
  uint64_t cache_bytes;
  uint64_t n;
  uint16_t* out;            // bf16 [n][d], 16-byte aligned
  uint32_t* status;         // bit 0: an id was out of range
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared, L2 only; bytes in [1, 16], rest zero-filled.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(bytes)
               : "memory");
}

// 4-byte async copy global -> shared; bytes in [0, 4], rest zero-filled.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Exact alpha * (y0, y1) for fp16 alpha: two mixed-precision FMAs with c = -0
// (x + (-0) = x for every x, signed zeros included).
__device__ __forceinline__ uint32_t scale_pair_f16(uint32_t v, uint16_t a_h) {
  float o0, o1;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "fma.rn.f32.f16 %0, lo, %3, %4;\n\tfma.rn.f32.f16 %1, hi, %3, %4;\n\t}"
      : "=f"(o0), "=f"(o1)
      : "r"(v), "h"(a_h), "f"(-0.0f));
  const __nv_bfloat162 r = __floats2bfloat162_rn(o0, o1);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Same result for any bf16 alpha (as fp32): convert, multiply, round.
__device__ __forceinline__ uint32_t scale_pair_f32(uint32_t v, float a) {
  const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&v));
  const __nv_bfloat162 r = __floats2bfloat162_rn(a * y.x, a * y.y);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// LUT word of state s for this lane: entry e = (h >> 14) & 1023 at byte offset
// e * REP * 4, replica (lane % REP); lane4 = (lane % REP) * 4.
template <int REP>
__device__ __forceinline__ uint32_t lut_word(const uint8_t* lut, uint32_t s, uint32_t lane4) {
  constexpr int kSh = log2i(REP * 4);                             // 7 for REP = 32
  const uint32_t h = s * s + s;                                   // mod 2^32
  const uint32_t off = ((h >> (14 - kSh)) & ((kLutEntries - 1) << kSh)) | lane4;
  return *reinterpret_cast<const uint32_t*>(lut + off);
}

// Steps 4c..4c+3 of a row from x (bit 0 = first bit of the first window).
template <int K, bool F16, int REP>
__device__ __forceinline__ uint4 decode_chunk(uint64_t x, const uint8_t* lut,
                                              uint32_t lane4, uint16_t a_h, float a) {
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t s = static_cast<uint32_t>(x >> (K * j)) & 0xFFFFu;
    const uint32_t v = lut_word<REP>(lut, s, lane4);
    o[j] = F16 ? scale_pair_f16(v, a_h) : scale_pair_f32(v, a);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint64_t funnel64(uint32_t lo, uint32_t hi, uint32_t sh) {
  return ((static_cast<uint64_t>(hi) << 32) | lo) >> sh;
}

// Decode one staged row with LPR lanes (sub = this lane's index among them),
// each lane CPL 16-byte chunks c = sub + LPR m, written to orow.  The chunks'
// bit offsets boff + K(4c + 1) - 16 differ by K * LPR / 8 whole words, so one
// shift amount serves all of them.  lane picks the LUT replica.
template <int K, int CPL, bool F16, int REP, int LPR>
__device__ __forceinline__ void decode_row_lanes(const uint32_t* w, uint32_t boff,
                                                 const uint8_t* lut_bytes, uint32_t lane,
                                                 uint32_t sub, uint16_t a_h, float a,
                                                 uint4* orow) {
  static_assert((K * LPR) % 8 == 0, "chunk offsets must be whole words");
  const uint32_t lane4 = (lane & (REP - 1)) << 2;
  const uint32_t P0 = boff + K * (4 * sub + 1) - 16;
  const uint32_t* w0 = w + (P0 >> 5);
  const uint32_t sh = P0 & 31;
#pragma unroll
  for (int m = 0; m < CPL; ++m) {
    constexpr int kStep = K * LPR / 8;                  // words between consecutive chunks
    const uint64_t x = funnel64(w0[kStep * m], w0[kStep * m + 1], sh);
    __stcs(orow + sub + LPR * m, decode_chunk<K, F16, REP>(x, lut_bytes, lane4, a_h, a));
  }
}

// Decode one staged row into orow (16-byte chunks) with the whole warp.  w:
// staged words; boff: bit offset of code bit 0 in the stage (>= 16 bits of
// spliced tail below it).  CPL > 0: d == 256 * CPL.
template <int K, int CPL, bool F16, int REP>
__device__ __forceinline__ void decode_row(const uint32_t* w, uint32_t boff, uint32_t d,
                                           const uint8_t* lut_bytes, uint32_t lane,
                                           uint16_t a_h, float a, uint4* orow) {
  if constexpr (CPL > 0) {
    decode_row_lanes<K, CPL, F16, REP, 32>(w, boff, lut_bytes, lane, lane, a_h, a, orow);
  } else {
    const uint32_t lane4 = (lane & (REP - 1)) << 2;
    const uint32_t C = d >> 3;
    for (uint32_t c = lane; c < C; c += 32) {
      const uint32_t P = boff + K * (4 * c + 1) - 16;
      const uint64_t x = funnel64(w[P >> 5], w[(P >> 5) + 1], P & 31);
      __stcs(orow + c, decode_chunk<K, F16, REP>(x, lut_bytes, lane4, a_h, a));
    }
  }
}

// Non-persistent kernel of the HBM-resident path: a CTA of kBlkWarps warps
// decodes kBlkRows rows per warp, with its own LUT of kLutRepBlock replicas.
#ifndef CP_BLK_WARPS
#define CP_BLK_WARPS 8
#endif
#ifndef CP_BLK_ROWS
#define CP_BLK_ROWS 4
#endif
#ifndef CP_BLK_REP
#define CP_BLK_REP 2
#endif
constexpr int kBlkWarps = CP_BLK_WARPS;
constexpr int kBlkRows = CP_BLK_ROWS;
constexpr int kLutRepBlock = CP_BLK_REP;

// Byte offset of the record data inside a stage (room for the spliced tail).
constexpr uint32_t kStagePrefix = 16;

// Expand the 512 LUT pairs into shared memory: entry e -> pair e & 511 with y1
// negated for e >= 512, REP copies of each entry (word e * REP + replica).
// REP <= 4 (the block kernel fills once per 32 rows): one 8-byte load per two
// source pairs, written with its sign-flipped twin 512 entries on.
template <int REP>
__device__ __forceinline__ void fill_lut(uint8_t* smem, const uint32_t* lut, int tid, int nthreads) {
  static_assert(REP >= 1 && REP <= 32 && (REP & (REP - 1)) == 0, "REP: power of two");
  if constexpr (REP <= 4) {
    // entries e, e + 1 (e even) with values a, b: words [e * REP, (e + 2) * REP)
    auto put = [&](int e, uint32_t a, uint32_t b) {
      if constexpr (REP == 1) {
        reinterpret_cast<uint2*>(smem)[e / 2] = make_uint2(a, b);
      } else if constexpr (REP == 2) {
        reinterpret_cast<uint4*>(smem)[e / 2] = make_uint4(a, a, b, b);
      } else {
        reinterpret_cast<uint4*>(smem)[e] = make_uint4(a, a, a, a);
        reinterpret_cast<uint4*>(smem)[e + 1] = make_uint4(b, b, b, b);
      }
    };
    for (int t = tid; t < kLutEntries / 4; t += nthreads) {        // 256 source word pairs
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(lut) + t);
      put(2 * t, v.x, v.y);
      put(2 * t + kLutEntries / 2, v.x ^ 0x80000000u, v.y ^ 0x80000000u);
    }
  } else {
    for (int q = tid; q < kLutEntries * REP / 4; q += nthreads) {  // REP / 4 uint4 per entry
      const int e = q / (REP / 4);
      uint32_t v = __ldg(lut + (e & 511));
      if (e & 512) v ^= 0x80000000u;
      reinterpret_cast<uint4*>(smem)[q] = make_uint4(v, v, v, v);
    }
  }
}

// Queue the 16-byte cp.async copies of record r into the stage whose data starts
// at shared address sa, with LPR lanes (sub = this lane's index among them; r is
// the same on those lanes).  Returns the stage's meta word: bit 0 = record
// present, bit 1 = r odd (SoA alpha half), bits 8.. = the record's misalignment;
// 0 when r is outside [0, n_rows) (lane sub 0 then sets the status bit).  The
// caller commits the group.  ONE_PASS: the record spans at most LPR pieces.
template <bool SOA, bool ONE_PASS, int LPR = 32>
__device__ __forceinline__ uint32_t issue_record(const DecodeParams& p, int64_t r, uint32_t sa,
                                                 uint32_t sub) {
  if (static_cast<uint64_t>(r) >= p.n_rows) {           // also rejects r < 0
    if (sub == 0) atomicOr(p.status, 1u);
    return 0;
  }
  const uintptr_t codes = reinterpret_cast<uintptr_t>(p.codes);
  const uintptr_t tbl_end = codes + p.table_bytes;
  const uintptr_t a = codes + static_cast<uint64_t>(r) * p.stride;
  const uintptr_t a0 = a & ~static_cast<uintptr_t>(15);
  const uint32_t mis = static_cast<uint32_t>(a - a0);
  const uint32_t nch = (mis + p.code_bytes + (SOA ? 0u : 2u) + 15) >> 4;
  auto copy = [&](uint32_t c) {
    const uintptr_t src = a0 + 16u * c;
    uint32_t bytes = 16;
    if (!SOA) {
      const uintptr_t left = tbl_end - src;             // > 0: src lies inside the table
      bytes = left < 16 ? static_cast<uint32_t>(left) : 16u;
    }
    cp_async16(sa + 16u * c, reinterpret_cast<const void*>(src), bytes);
  };
  if constexpr (ONE_PASS) {
    if (sub < nch) copy(sub);
  } else {
    for (uint32_t c = sub; c < nch; c += LPR) copy(c);
  }
  if (SOA && sub == LPR - 1) {
    const uint64_t r2 = static_cast<uint64_t>(r) & ~1ull;
    // alpha_slot is measured from the stage start, like the decode's read
    cp_async4(sa - kStagePrefix + p.alpha_slot, p.alpha + r2, (r2 + 1 < p.n_rows) ? 4u : 2u);
  }
  return 1u | ((static_cast<uint32_t>(r) & 1u) << 1) | (mis << 8);
}

// Decode the record that has landed in stage sb (data at sb + kStagePrefix) with
// meta word m into orow, or write a row of zeros when m is 0, with LPR lanes
// (sub = this lane's index among them; every lane of the warp must call it, the
// LPR-lane groups each with their own row).  CPL: chunks per lane of the group
// (LPR * CPL * 8 == d), 0 for any d with the whole warp.  valid = false: the
// group has no row (no store).
template <int K, bool SOA, int CPL, int REP, int LPR = 32>
__device__ __forceinline__ void decode_stage(const DecodeParams& p, uint8_t* sb, uint32_t m,
                                             const uint8_t* lut, uint32_t lane, uint32_t sub,
                                             uint4* orow, bool valid) {
  static_assert(CPL > 0 || LPR == 32, "the any-d decode uses the whole warp");
  const uint32_t code_bytes = p.code_bytes;
  const uint32_t d = p.d;
  const bool has = (m & 1u) != 0;
  const uint32_t mis = m >> 8;
  uint8_t* code = sb + kStagePrefix + mis;
  // Tail-biting splice: the code's last 16 bits just below bit 0.
  if (has && sub == 0)
    *reinterpret_cast<uint16_t*>(code - 2) =
        *reinterpret_cast<const uint16_t*>(code + code_bytes - 2);
  __syncwarp();
  if (has) {
    const uint16_t abits = SOA ? *reinterpret_cast<const uint16_t*>(
                                     sb + p.alpha_slot + 2 * ((m >> 1) & 1u))
                               : *reinterpret_cast<const uint16_t*>(code + code_bytes);
    const float a = __uint_as_float(static_cast<uint32_t>(abits) << 16);
    const uint32_t ex = (abits >> 7) & 0xFFu;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(sb);
    const uint32_t boff = (kStagePrefix + mis) * 8;
    const bool f16 = (abits & 0x7FFFu) == 0 || (ex - 113u) <= 29u;  // |alpha| in [2^-14, 2^16) or 0
    if constexpr (CPL > 0) {
      if (f16) {
        const __half ah = __float2half_rn(a);             // exact in this range
        decode_row_lanes<K, CPL, true, REP, LPR>(w, boff, lut, lane, sub, __half_as_ushort(ah), a,
                                                 orow);
      } else {
        decode_row_lanes<K, CPL, false, REP, LPR>(w, boff, lut, lane, sub, 0, a, orow);
      }
    } else {
      if (f16) {
        const __half ah = __float2half_rn(a);
        decode_row<K, 0, true, REP>(w, boff, d, lut, lane, __half_as_ushort(ah), a, orow);
      } else {
        decode_row<K, 0, false, REP>(w, boff, d, lut, lane, 0, a, orow);
      }
    }
  } else if (valid) {
    const uint4 zero = make_uint4(0, 0, 0, 0);
    for (uint32_t c = sub; c < (d >> 3); c += LPR) __stcs(orow + c, zero);
  }
}

// cp.async.wait_group with a count known only after unrolling (0..7; larger
// counts wait for every group, which is also correct).
__device__ __forceinline__ void cp_async_wait_n(int n) {
  switch (n) {
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    case 7: cp_async_wait<7>(); break;
    default: cp_async_wait<0>(); break;
  }
}

// Persistent kernel: one CTA of up to kMaxWarps warps per SM, each warp a
// contiguous range of positions, a ring of PF record stages per warp.
// K: bits per step (3..6).  SOA: read the SoA copy.  PF: stages per warp.
// CPL: chunks per lane when d == 256 * CPL, 0 for any d (runtime loop).
// PERM: lookups are visited in the order p.perm (rows still land at their own
// output position); used to give host-resident tables address locality.
// REP: LUT replicas in shared memory.
template <int K, bool SOA, int PF, int CPL, bool PERM, int REP>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) lookup_decode_kernel(const DecodeParams p) {
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
  // Records up to 496 bytes (d <= 1024 here) fit one 16-byte copy per lane.
  constexpr bool kOnePass = (CPL >= 1 && CPL <= 4);

  uint8_t* stages = smem + kLutBytes + static_cast<size_t>(warp) * PF * stage_bytes;
  // per stage: [0] meta word, [1] output row (PERM)
  uint32_t* meta = reinterpret_cast<uint32_t*>(smem + kLutBytes +
                                               static_cast<size_t>(nwarps) * PF * stage_bytes) +
                   warp * PF * 2;
  const uint32_t stages_sa = smem_addr(stages) + kStagePrefix;

  const uint64_t W = static_cast<uint64_t>(gridDim.x) * nwarps;
  const uint64_t gw = static_cast<uint64_t>(blockIdx.x) * nwarps + warp;
  const uint64_t n_work = p.n;
  const uint64_t lo = gw * n_work / W;
  const uint64_t hi = (gw + 1) * n_work / W;
  if (lo >= hi) return;
  const uint32_t cnt = static_cast<uint32_t>(hi - lo);   // < 2^31 rows per warp (host check)

  // Row ids, 32 per coalesced load, one batch of look-ahead.  With PERM the
  // batch holds positions j = perm[lo + q] and their ids idx[j].
  const int64_t* ids = p.idx + lo;
  const uint32_t* pos = PERM ? p.perm + lo : nullptr;
  auto load_batch = [&](uint32_t q, uint32_t& j, int64_t& r) {
    j = 0;
    r = 0;
    if (q < cnt) {
      if (PERM) {
        j = __ldg(pos + q);
        r = __ldg(p.idx + j);
      } else {
        r = __ldg(ids + q);
      }
    }
  };
  uint32_t jb_cur, jb_nxt;
  int64_t ib_cur, ib_nxt;
  load_batch(lane, jb_cur, ib_cur);
  load_batch(lane + 32, jb_nxt, ib_nxt);
  uint32_t batch = 0;

  auto issue = [&](uint32_t q) {
    if (q - batch >= 32) {
      batch += 32;
      ib_cur = ib_nxt;
      jb_cur = jb_nxt;
      load_batch(batch + 32 + lane, jb_nxt, ib_nxt);
    }
    const int64_t r = __shfl_sync(0xffffffffu, ib_cur, static_cast<int>(q - batch));
    uint32_t jrow = 0;
    if (PERM) jrow = __shfl_sync(0xffffffffu, jb_cur, static_cast<int>(q - batch));
    const uint32_t st = q & (PF - 1);
    const uint32_t m = issue_record<SOA, kOnePass>(p, r, stages_sa + st * stage_bytes, lane);
    if (lane == 0) {
      meta[2 * st] = m;
      if (PERM) meta[2 * st + 1] = jrow;
    }
    cp_async_commit();
  };

#pragma unroll
  for (int q = 0; q < PF - 1; ++q) {
    if (static_cast<uint32_t>(q) < cnt) issue(q);
    else cp_async_commit();
  }

  uint4* orow_seq = reinterpret_cast<uint4*>(p.out) + lo * (d >> 3);
  for (uint32_t i = 0; i < cnt; ++i, orow_seq += (d >> 3)) {
    if (i + PF - 1 < cnt) issue(i + PF - 1);
    else cp_async_commit();
    cp_async_wait<PF - 1>();
    __syncwarp();

    const uint32_t st = i & (PF - 1);
    uint4* orow = PERM ? reinterpret_cast<uint4*>(p.out) +
                             static_cast<uint64_t>(meta[2 * st + 1]) * (d >> 3)
                       : orow_seq;
    decode_stage<K, SOA, CPL, REP>(p, stages + st * stage_bytes, meta[2 * st], smem, lane, lane, orow,
                                   true);
    __syncwarp();
  }
}

// Non-persistent kernel of the HBM-resident path.  CTA b decodes the lookups
// [b * kBlkWarps * ROWS, (b + 1) * kBlkWarps * ROWS): warp w takes positions
// w, w + kBlkWarps, ..., so at every step the CTA writes kBlkWarps consecutive
// rows.  Each warp queues all of its ROWS record copies (one stage each) before
// the CTA expands its LUT, so the record latency overlaps the fill.  The
// hardware block scheduler hands CTAs to SMs as SMs free up, which keeps the
// output writes in a narrow, advancing window of addresses and lets faster SMs
// take more of the work; a persistent grid with static ranges per warp ran
// 10-20 % longer on the same replay.
// Rows shorter than 1024 (d = 256, 512) are decoded G = 1024 / d at a time by
// groups of 32 / G lanes, each lane 4 chunks as at d = 1024: the per-row work
// that does not scale with d (id, record issue, splice, scale) is then shared
// by G rows per warp instruction.
template <int K, bool SOA, int CPL, int REP, int ROWS>
__global__ void __launch_bounds__(kBlkWarps * 32) lookup_decode_block_kernel(const DecodeParams p) {
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
  // Records up to 16 * LPR bytes fit one 16-byte copy per lane of the group:
  // d * k / 16 + 2 + 14 <= d / 2 for k <= 6 and d >= 128.
  constexpr bool kOnePass = (CPL >= 1 && CPL <= 4);
  constexpr int kLutBytes = lut_bytes(REP);
  const uint32_t stage_bytes = p.stage_bytes;
  uint8_t* stages = smem + kLutBytes + static_cast<size_t>(warp) * ROWS * stage_bytes;
  const uint32_t stages_sa = smem_addr(stages) + kStagePrefix;

  const uint64_t first = static_cast<uint64_t>(blockIdx.x) * (kBlkWarps * ROWS) + warp;
  const uint64_t n = p.n;
  int64_t my_id = 0;                                  // lane t: id of the warp's row t
  if (lane < static_cast<uint32_t>(ROWS)) {
    const uint64_t j = first + static_cast<uint64_t>(lane) * kBlkWarps;
    if (j < n) my_id = __ldg(p.idx + j);
  }
  uint32_t m[STEPS];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const uint32_t t = s * G + slot;                  // row of this lane's group
    const int64_t r = __shfl_sync(0xffffffffu, my_id, static_cast<int>(t));
    m[s] = 0;
    if (first + static_cast<uint64_t>(t) * kBlkWarps < n)
      m[s] = issue_record<SOA, kOnePass, LPR>(p, r, stages_sa + t * stage_bytes, sub);
    cp_async_commit();
  }

  fill_lut<REP>(smem, p.lut, tid, kBlkWarps * 32);
  __syncthreads();

#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const uint32_t t = s * G + slot;
    const uint64_t j = first + static_cast<uint64_t>(t) * kBlkWarps;
    if (first + static_cast<uint64_t>(s * G) * kBlkWarps >= n) break;   // no row of this step
    cp_async_wait_n(STEPS - 1 - s);
    __syncwarp();
    decode_stage<K, SOA, CPLG, REP, LPR>(p, stages + t * stage_bytes, m[s], smem, lane, sub,
                                         reinterpret_cast<uint4*>(p.out) + j * (p.d >> 3),
                                         j < n);
  }
}

// AoS -> SoA repack: one warp per row, 2-byte granules (records are 2-byte aligned).
__global__ void repack_soa_kernel(const uint8_t* __restrict__ rec, uint64_t n_rows, uint32_t R,
                                  uint32_t code_bytes, uint32_t S, uint8_t* __restrict__ codes,
                                  uint16_t* __restrict__ alpha);

}  // namespace cpk

// cp_encode.cu -- offline compression on the GPU: tail-biting TCQ encoder.
//
// The pages compress each row as z = sqrt(d) e / |e| coded by a tail-biting
// Gaussian HYB bitshift trellis (TCQ) and restore the norm with
// alpha = |e|_2 / |f(c)|_2 ("2비트 코드와 공유 트렐리스로 n-gram 룩업 테이블을
// 4~8배 압축한다", section 무엇과 다른가).  This is that step for whole tables:
// the two-pass search (a free-start Viterbi on the sequence rotated by T/2
// steps picks the w = 16 - k pre-window bits from its best path, then one
// Viterbi constrained to that w gives a valid tail-biting code).
//
// Precision: z and alpha in fp64 (sums in index order), path metrics in fp32
// (branch cost fl(fl((z0-y0)^2) + fl((z1-y1)^2)), no fused multiply-adds).
// Recursion: the 2^k states with the same low W bits (a group) share their 2^k
// predecessors, so each group picks its survivor once (smallest metric, then
// smallest dropped bits) and every state of the group adds its branch cost;
// one traceback byte per group and step.
//
// Work mapping: one cluster of 4 CTAs x 1024 threads per row (persistent over
// rows).  CTA c owns the 2^14 states whose top two bits are c, 16 per thread,
// held in registers.  The predecessors of a group are 2^K consecutive states, so
// the group minima are local; the 2^W group minima are what every CTA needs for
// the next step and are pushed to all four CTAs through distributed shared
// memory, one cluster barrier per step.  The branch cost depends on the state
// only through its signed LUT entry, so each step first tabulates the 1024
// possible costs in shared memory (replicated against bank conflicts).  The
// traceback bytes (one per group and step) go to a per-cluster global scratch;
// CTA 0 walks them back after each pass from chunks copied into shared memory.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "cp_internal.h"

namespace cpk {

namespace {

#ifndef CP_ENC_THREADS
#define CP_ENC_THREADS 1024
#endif
constexpr int kEncThreads = CP_ENC_THREADS;                    // 512 or 1024
constexpr uint32_t kStates = 1u << 16;
constexpr uint32_t kCluster = 4;
constexpr uint32_t kLocalStates = kStates / kCluster;          // 2^14 per CTA
constexpr int kPerThread = kLocalStates / kEncThreads;        // states per thread (32 or 16)
static_assert(kPerThread == 16 || kPerThread == 32, "512 or 1024 threads");
constexpr int kCostRep = 8;                                    // cost table replicas
constexpr uint32_t kCostBytes = 1024u * kCostRep * 4;          // one step's table

struct EncodeParams {
  const float* e;           // rows x d, fp32
  uint64_t rows;
  uint32_t d;
  const uint32_t* lut;      // 512 words: fp16 y0 | fp16 y1 << 16
  uint8_t* records;         // rows x R
  float* cost;              // rows (optional)
  uint8_t* work;            // per cluster: T x 2^W traceback bytes
  uint64_t work_stride;     // bytes per cluster
};

// Round a positive or zero double to bf16 (one rounding, ties to even).
__device__ __forceinline__ uint16_t double_to_bf16_rne(double x) {
  if (x == 0.0) return 0;
  const unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
  const int ex = static_cast<int>((u >> 52) & 0x7FF) - 1023;       // unbiased exponent
  if (ex < -126) {                  // bf16 subnormal range: multiples of 2^-133
    const long long m = __double2ll_rn(x * 0x1p133);                // exact scaling, RNE
    return static_cast<uint16_t>(m);                                // m == 128: smallest normal
  }
  unsigned long long man = (u & 0xFFFFFFFFFFFFFull) | (1ull << 52);  // 53-bit significand
  // keep 8 significant bits: drop 45, round half to even
  const unsigned long long keep = man >> 45;
  const unsigned long long rest = man & ((1ull << 45) - 1);
  const unsigned long long half = 1ull << 44;
  unsigned long long m8 = keep + ((rest > half || (rest == half && (keep & 1))) ? 1 : 0);
  int e8 = ex;
  if (m8 == 256) {
    m8 = 128;
    e8 += 1;
  }
  if (e8 > 127) return 0x7F80;                                      // overflow -> inf
  return static_cast<uint16_t>(((e8 + 127) << 7) | (m8 & 0x7F));
}

// (y0, y1) of signed LUT entry e (bit 9 = sign of y1) as fp32 (exact fp16 values).
__device__ __forceinline__ float2 entry_y(const uint32_t* lut, uint32_t e) {
  uint32_t v = lut[e & 511];
  if (e & 512) v ^= 0x80000000u;
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

// Signed LUT entry of state s: (h >> 14) & 1023 with h = s*s + s; its bit 9 is
// hash bit 23, the sign of y1.
__device__ __forceinline__ uint32_t state_entry(uint32_t s) { return ((s * s + s) >> 14) & 1023u; }

// fl(fl((z0 - y0)^2) + fl((z1 - y1)^2)), no contraction.
__device__ __forceinline__ float pair_cost(float z0, float z1, float2 y) {
  const float a = __fsub_rn(z0, y.x);
  const float b = __fsub_rn(z1, y.y);
  return __fadd_rn(__fmul_rn(a, a), __fmul_rn(b, b));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// All threads of the cluster; orders shared (local and remote) and global accesses.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// Address of local shared address `a` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_peer2(uint32_t a, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ void st_peer4(uint32_t a, float x, float y, float z, float w) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(x), "f"(y),
               "f"(z), "f"(w)
               : "memory");
}
__device__ __forceinline__ void st_peer(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Word index of group g's minimum in the group-minimum array: 16-byte units are
// XOR-swizzled within blocks of eight, so the 16-byte reads of consecutive
// groups (16 or 32 per thread) are free of bank conflicts across a quarter warp.
__device__ __forceinline__ uint32_t best_word(uint32_t g) {
  const uint32_t u = g >> 2;
  return ((u ^ ((u >> 3) & 7u)) << 2) | (g & 3u);
}

// Lexicographic (value, index) minimum; strict so equal values keep the smaller index.
__device__ __forceinline__ void min_pair(float& v, uint32_t& i, float ov, uint32_t oi) {
  if (ov < v || (ov == v && oi < i)) {
    v = ov;
    i = oi;
  }
}

// Branch costs of step t for the 1024 signed entries, kCostRep copies each
// (entry e, copy r at word e * kCostRep + r).  A warp fills the 1 KB of its 32
// entries with two 16-byte stores per lane, each store instruction covering 512
// contiguous bytes (lane l: entry 16 j + l / 2, copies 4 (l % 2) .. + 3), so no
// store replays on a bank conflict (one 32-byte store per lane replayed every
// store once: 2.6 % of the encoder's time at k = 4); lane l works out the cost
// of entry l and the storing lanes fetch theirs by a shuffle.
__device__ __forceinline__ void build_costs(float* ct, const uint32_t* lut, const float* z,
                                            uint32_t t) {
  static_assert(kCostRep == 8, "two 16-byte pieces per entry");
  const float z0 = z[2 * t], z1 = z[2 * t + 1];
  const uint32_t lane = threadIdx.x & 31u;
#pragma unroll
  for (uint32_t w0 = threadIdx.x & ~31u; w0 < 1024; w0 += kEncThreads) {
    const float cl = pair_cost(z0, z1, entry_y(lut, w0 + lane));
#pragma unroll
    for (uint32_t j = 0; j < 2; ++j) {
      const uint32_t e = w0 + 16 * j + (lane >> 1);
      const float c = __shfl_sync(0xffffffffu, cl, 16 * j + (lane >> 1));
      *reinterpret_cast<float4*>(ct + e * kCostRep + 4 * (lane & 1)) = make_float4(c, c, c, c);
    }
  }
}

// Byte offset of state s's cost in a table, copy (lane % kCostRep).
__device__ __forceinline__ uint32_t cost_off(uint32_t s, uint32_t lane_off) {
  constexpr int kSh = 14 - 5;                          // entry * kCostRep * 4 = entry << 5
  static_assert(kCostRep * 4 == 32, "shift assumes 8 copies");
  return (((s * s + s) >> kSh) & (1023u << 5)) | lane_off;
}

// Per-CTA shared memory (offsets in bytes from the dynamic base).
struct EncSmem {
  uint32_t ct, best, lut, z, code, red, slots, total;
};

__host__ __device__ inline EncSmem enc_smem(uint32_t d, uint32_t k) {
  EncSmem m;
  const uint32_t W = 16 - k;
  m.ct = 0;                                            // 3 x cost table; also fp64 scratch
  m.best = 3 * kCostBytes;                             // 2 x 2^W floats
  m.lut = m.best + 2 * (4u << W);
  m.z = m.lut + 2048;
  m.code = m.z + 4 * d;
  m.red = m.code + ((d * k / 16 + 15) & ~15u);         // 32 floats + 32 words
  m.slots = m.red + 256;                               // 4 floats, 4 words, w, 2 doubles
  m.total = m.slots + 64;
  return m;
}

template <int K>
__global__ void __launch_bounds__(kEncThreads, 1) tcq_encode_kernel(const EncodeParams p) {
  constexpr uint32_t W = 16 - K;
  constexpr uint32_t kMask = (1u << W) - 1;
  // own groups: a thread's states are NG whole groups of GS, or 1/SPLIT of one group
  constexpr int GS = (1 << K) < kPerThread ? (1 << K) : kPerThread;
  constexpr int NG = kPerThread / GS;
  constexpr int SPLIT = (1 << K) / GS;
  // group minima per remote store: 4 when a thread owns several groups (k = 3:
  // two lanes fill a 16-byte unit; the step's remote stores drop from 8 to 2 per
  // thread and the encoder runs 1.8x faster), else 1 (gathering across four lanes
  // costs three shuffles on the critical path and measured 9 % slower)
  constexpr int kGather = NG >= 2 ? 4 : 1;
  extern __shared__ __align__(16) uint8_t smem[];
  const uint32_t d = p.d, T = d / 2, Lc = K * T, code_bytes = Lc / 8;
  const EncSmem L = enc_smem(d, K);
  float* ct = reinterpret_cast<float*>(smem + L.ct);
  float* best = reinterpret_cast<float*>(smem + L.best);
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + L.lut);
  float* z = reinterpret_cast<float*>(smem + L.z);
  uint8_t* code = smem + L.code;
  float* red_v = reinterpret_cast<float*>(smem + L.red);
  uint32_t* red_s = reinterpret_cast<uint32_t*>(smem + L.red + 128);
  float* slot_v = reinterpret_cast<float*>(smem + L.slots);
  uint32_t* slot_s = reinterpret_cast<uint32_t*>(smem + L.slots + 16);
  uint32_t* slot_w = reinterpret_cast<uint32_t*>(smem + L.slots + 32);
  double* sh_d = reinterpret_cast<double*>(smem + L.slots + 48);
  double* scratch = reinterpret_cast<double*>(smem + L.ct);

  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank();
  const uint32_t base = crank * kLocalStates + tid * kPerThread;   // this thread's states
  const uint32_t lane_off = (lane & (kCostRep - 1)) * 4;
  const uint32_t best_sa = smem_u32(best);
  const uint32_t slots_sa = smem_u32(smem + L.slots);
  // per-thread constants: cluster addresses of the group-minimum buffers, own
  // groups' word offsets, the swizzle of the thread's 16-byte reads
  uint32_t peer_best[2][kCluster];
#pragma unroll
  for (uint32_t b = 0; b < 2; ++b)
#pragma unroll
    for (uint32_t c = 0; c < kCluster; ++c) peer_best[b][c] = peer_addr(best_sa + b * (4u << W), c);
  // the thread reads groups (base & kMask) + [0, kPerThread): 16-byte units u0 + q4,
  // all in one block of eight, so their swizzle (u >> 3) & 7 is the same
  const uint32_t u0 = (base & kMask) >> 2;
  const uint32_t rd_swz = (u0 >> 3) & 7u;
  for (uint32_t i = tid; i < 512; i += kEncThreads) lut[i] = p.lut[i];
  uint8_t* tb = p.work + static_cast<uint64_t>(cluster_index()) * p.work_stride;
  __syncthreads();

  float v[kPerThread] = {};

  // Step i of a pass (steps t(1), t(2), ... after the start step t(0)): group
  // minima of v (metrics at t(i-1)) -> traceback bytes and the minima in every
  // CTA's buffer i & 1; then the new metrics at t(i) = tcur.  The cost table of
  // t(i) was built one step earlier (table i % 3); this step builds the one of
  // t(i+1) = tnext and reads its own costs while the cluster barrier completes.
  // Reuse: table (i+1) % 3 and buffer i & 1 were last read at step i-2, before
  // every thread's arrival at step i-1.
  auto step = [&](uint32_t i, uint32_t tcur, uint32_t tnext, bool build_next, bool forced_pass,
                  uint32_t w) {
    const uint32_t buf = i & 1;
    uint32_t tbv[NG];
    float bvs[NG];
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      float bv = v[gi * GS];
      uint32_t by = 0;
#pragma unroll
      for (int y = 1; y < GS; ++y) {
        if (v[gi * GS + y] < bv) {
          bv = v[gi * GS + y];
          by = y;
        }
      }
      if constexpr (SPLIT > 1) {
        by += base & ((1u << K) - 1);
#pragma unroll
        for (int o = 1; o < SPLIT; o <<= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const uint32_t oy = __shfl_xor_sync(0xffffffffu, by, o);
          min_pair(bv, by, ov, oy);
        }
      }
      tbv[gi] = by;
      bvs[gi] = bv;

    }
    // Push the minima to every CTA, kGather consecutive groups per remote store
    // (they share one 8- or 16-byte piece of a swizzled 16-byte unit).  Writer
    // lanes (lane % SPLIT == 0) hold NG consecutive groups each; when a store
    // spans several writers, the first gathers the others' minima (SPLIT lanes
    // apart) by shuffles.
    {
      constexpr int U = NG >= kGather ? 1 : kGather / NG;          // writers per store
      constexpr int kStores = NG >= kGather ? NG / kGather : 1;    // stores per writer
      float q[kGather];
#pragma unroll
      for (int st = 0; st < kStores; ++st) {
#pragma unroll
        for (int m = 0; m < U; ++m)
#pragma unroll
          for (int gi = 0; gi < (NG < kGather ? NG : kGather); ++gi) {
            const float x = bvs[st * kGather + gi];
            q[m * NG + gi] = (m == 0) ? x : __shfl_down_sync(0xffffffffu, x, SPLIT * m);
          }
        if ((lane & (SPLIT * U - 1)) == 0) {
          const uint32_t off = 4 * best_word((base >> K) + st * kGather);
#pragma unroll
          for (uint32_t c = 0; c < kCluster; ++c) {
            const uint32_t a = (buf ? peer_best[1][c] : peer_best[0][c]) + off;
            if constexpr (kGather == 4) st_peer4(a, q[0], q[1], q[2], q[3]);
            else if constexpr (kGather == 2) st_peer2(a, q[0], q[1]);
            else st_peer(a, __float_as_uint(q[0]));
          }
        }
      }
    }
    if (build_next) build_costs(ct + ((i + 1) % 3) * (kCostBytes / 4), lut, z, tnext);
    cluster_arrive();
    // traceback bytes (global) after the arrival, so its release does not wait for them
    if (SPLIT == 1 || (tid & (SPLIT - 1)) == 0) {
      uint8_t* tbi = tb + static_cast<uint64_t>(i) * (kMask + 1) + (base >> K);
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) tbi[gi] = static_cast<uint8_t>(tbv[gi]);
    }
    // own costs at t(i), from the table built before the previous barrier
    const uint8_t* ctb = reinterpret_cast<const uint8_t*>(ct + (i % 3) * (kCostBytes / 4));
#pragma unroll
    for (int q = 0; q < kPerThread; ++q)
      v[q] = *reinterpret_cast<const float*>(ctb + cost_off(base + q, lane_off));
    // forced new bits (second pass): positions >= Lc - W hold w; the new bits
    // (base >> W) are the same for all of the thread's states
    bool dead = false;
    if (forced_pass && K * tcur + K > Lc - W) {
      uint32_t fmask = 0, fval = 0;
      for (uint32_t b = 0; b < K; ++b) {
        const uint32_t pos = K * tcur + b;
        if (pos >= Lc - W) {
          fmask |= 1u << b;
          fval |= ((w >> (pos - (Lc - W))) & 1u) << b;
        }
      }
      dead = ((base >> W) & fmask) != fval;
    }
    cluster_wait();
    const float* bb = best + buf * (1u << W);
#pragma unroll
    for (int q4 = 0; q4 < kPerThread / 4; ++q4) {
      float4 b4 = *reinterpret_cast<const float4*>(bb + 4 * ((u0 + q4) ^ rd_swz));
      if (dead) b4 = make_float4(INFINITY, INFINITY, INFINITY, INFINITY);
      v[4 * q4] = __fadd_rn(b4.x, v[4 * q4]);
      v[4 * q4 + 1] = __fadd_rn(b4.y, v[4 * q4 + 1]);
      v[4 * q4 + 2] = __fadd_rn(b4.z, v[4 * q4 + 2]);
      v[4 * q4 + 3] = __fadd_rn(b4.w, v[4 * q4 + 3]);
    }
  };

  // Cluster-wide argmin of v: smallest finite value, ties to the smaller state;
  // state 0xFFFFFFFF when every metric is infinite.  Ends with a cluster barrier.
  auto argmin = [&](float* best_v) -> uint32_t {
    float bv = INFINITY;
    uint32_t bs = 0xFFFFFFFFu;
#pragma unroll
    for (int q = 0; q < kPerThread; ++q) {
      if (v[q] < bv) {
        bv = v[q];
        bs = base + q;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const uint32_t os = __shfl_xor_sync(0xffffffffu, bs, o);
      min_pair(bv, bs, ov, os);
    }
    if (lane == 0) {
      red_v[warp] = bv;
      red_s[warp] = bs;
    }
    __syncthreads();
    if (warp == 0) {
      constexpr uint32_t kWarps = kEncThreads / 32;
      bv = lane < kWarps ? red_v[lane] : INFINITY;
      bs = lane < kWarps ? red_s[lane] : 0xFFFFFFFFu;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const uint32_t os = __shfl_xor_sync(0xffffffffu, bs, o);
        min_pair(bv, bs, ov, os);
      }
      if (lane < kCluster) {
        st_peer(peer_addr(slots_sa + 4 * crank, lane), __float_as_uint(bv));
        st_peer(peer_addr(slots_sa + 16 + 4 * crank, lane), bs);
      }
    }
    cluster_sync();
    bv = slot_v[0];
    bs = slot_s[0];
#pragma unroll
    for (uint32_t c = 1; c < kCluster; ++c) min_pair(bv, bs, slot_v[c], slot_s[c]);
    *best_v = bv;
    return (bv == INFINITY) ? 0xFFFFFFFFu : bs;
  };

  auto start_costs = [&]() {                          // v = costs of step t(0) (table 0)
#pragma unroll
    for (int q = 0; q < kPerThread; ++q)
      v[q] = *reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(ct) +
                                             cost_off(base + q, lane_off));
  };

  // Traceback by the CTA (rank 0 only): from state s at step index hi down to
  // step index lo + 1, stepping back s <- (g << K) | tb[i][g] (g = low W bits).
  // Chunks of traceback rows are copied into shared memory (the cost tables'
  // space, free between passes) by all threads; thread 0 walks them.  With
  // `emit`, thread 0 also writes the new bits of each step (top K bits of s at
  // step i) into code.  Returns the state at step lo (valid in thread 0).
  auto walk = [&](uint32_t s, uint32_t hi, uint32_t lo, bool emit) -> uint32_t {
    constexpr uint32_t kRowBytes = 1u << W;
    const uint32_t chunk = (3 * kCostBytes) / kRowBytes;
    uint8_t* stage = reinterpret_cast<uint8_t*>(ct);
    for (uint32_t c_hi = hi; c_hi > lo;) {
      const uint32_t c_lo = (c_hi - lo > chunk) ? c_hi - chunk + 1 : lo + 1;
      const uint4* src =
          reinterpret_cast<const uint4*>(tb + static_cast<uint64_t>(c_lo) * kRowBytes);
      const uint32_t n16 = (c_hi - c_lo + 1) * (kRowBytes / 16);
      for (uint32_t q = tid; q < n16; q += kEncThreads)
        reinterpret_cast<uint4*>(stage)[q] = __ldcg(src + q);
      __syncthreads();
      if (tid == 0) {
        for (uint32_t i = c_hi; i >= c_lo; --i) {
          if (emit) {
            const uint32_t x = s >> W;
            for (uint32_t b = 0; b < K; ++b) {
              const uint32_t j = K * i + b;
              if ((x >> b) & 1u) code[j >> 3] |= static_cast<uint8_t>(1u << (j & 7));
            }
          }
          const uint32_t g = s & kMask;
          s = (g << K) | stage[(i - c_lo) * kRowBytes + g];
        }
      }
      __syncthreads();
      c_hi = c_lo - 1;
    }
    return s;
  };

  for (uint64_t r = cluster_index(); r < p.rows; r += cluster_count()) {
    const float* er = p.e + r * d;
    uint8_t* rec = p.records + r * (code_bytes + 2);
    // |e| and z = (float)(e * sqrt(d) / |e|) in fp64, sums in index order
    for (uint32_t q = tid; q < d; q += kEncThreads) {
      const double x = static_cast<double>(er[q]);
      scratch[q] = __dmul_rn(x, x);
    }
    __syncthreads();
    if (tid == 0) {
      double ss = 0.0;
      for (uint32_t q = 0; q < d; ++q) ss = __dadd_rn(ss, scratch[q]);
      const double nrm = __dsqrt_rn(ss);
      sh_d[0] = nrm;
      sh_d[1] = (nrm == 0.0) ? 0.0 : __ddiv_rn(__dsqrt_rn(static_cast<double>(d)), nrm);
    }
    __syncthreads();
    const double nrm = sh_d[0], sc = sh_d[1];
    if (nrm == 0.0) {                                   // zero row: zero code, alpha = 0
      if (crank == 0) {
        for (uint32_t i = tid; i < code_bytes + 2; i += kEncThreads) rec[i] = 0;
        if (tid == 0 && p.cost) p.cost[r] = 0.0f;
      }
      __syncthreads();
      continue;
    }
    for (uint32_t q = tid; q < d; q += kEncThreads)
      z[q] = __double2float_rn(__dmul_rn(static_cast<double>(er[q]), sc));
    __syncthreads();

    // pass 1: free start at step rho = T/2, every state live
    const uint32_t rho = T / 2;
    build_costs(ct, lut, z, rho);
    build_costs(ct + kCostBytes / 4, lut, z, (rho + 1) % T);
    __syncthreads();
    start_costs();
    for (uint32_t i = 1; i < T; ++i)
      step(i, (rho + i) % T, (rho + i + 1) % T, i + 1 < T, false, 0);
    float bestv;
    uint32_t bs = argmin(&bestv);
    if (crank == 0) {                                   // walk back to original step T-1
      const uint32_t s = walk(bs, T - 1, T - 1 - rho, false);
      if (tid == 0)
        for (uint32_t c = 0; c < kCluster; ++c) st_peer(peer_addr(slots_sa + 32, c), s >> K);
    }
    cluster_sync();
    const uint32_t w = *slot_w;                         // the pre-window bits

    // pass 2: constrained to w, starting at step 0
    build_costs(ct, lut, z, 0);
    build_costs(ct + kCostBytes / 4, lut, z, 1);
    __syncthreads();
    start_costs();
#pragma unroll
    for (int q = 0; q < kPerThread; ++q)
      if (((base + q) & kMask) != w) v[q] = INFINITY;
    for (uint32_t i = 1; i < T; ++i) step(i, i, i + 1, i + 1 < T, true, w);
    bs = argmin(&bestv);

    // traceback: new bits of step t are the top K bits of s_t
    if (crank == 0) {
      for (uint32_t i = tid; i < code_bytes; i += kEncThreads) code[i] = 0;
      __syncthreads();
      const uint32_t s0 = walk(bs, T - 1, 0, true);     // state at step 0
      if (tid == 0) {
        const uint32_t x = s0 >> W;
        for (uint32_t b = 0; b < K; ++b)
          if ((x >> b) & 1u) code[b >> 3] |= static_cast<uint8_t>(1u << (b & 7));
      }
    }
    cluster_sync();                                     // traceback bytes free again
    if (crank == 0) {
      // alpha = |e| / |f(c)|, |f|^2 in fp64 over coordinates in order
      for (uint32_t t = tid; t < T; t += kEncThreads) {
        uint32_t st = 0;
        const int32_t first = static_cast<int32_t>(K * (t + 1)) - 16;
        for (int m = 0; m < 16; ++m) {
          int32_t pos = (first + m) % static_cast<int32_t>(Lc);
          if (pos < 0) pos += Lc;
          st |= static_cast<uint32_t>((code[pos >> 3] >> (pos & 7)) & 1u) << m;
        }
        const float2 y = entry_y(lut, state_entry(st));
        const double y0 = y.x, y1 = y.y;
        scratch[2 * t] = __dmul_rn(y0, y0);
        scratch[2 * t + 1] = __dmul_rn(y1, y1);
      }
      __syncthreads();
      if (tid == 0) {
        double fs = 0.0;
        for (uint32_t q = 0; q < 2 * T; ++q) fs = __dadd_rn(fs, scratch[q]);
        const uint16_t ab = double_to_bf16_rne(__ddiv_rn(nrm, __dsqrt_rn(fs)));
        rec[code_bytes] = static_cast<uint8_t>(ab & 0xFF);
        rec[code_bytes + 1] = static_cast<uint8_t>(ab >> 8);
        if (p.cost) p.cost[r] = bestv;
      }
      for (uint32_t i = tid; i < code_bytes; i += kEncThreads) rec[i] = code[i];
      __syncthreads();
    }
  }
  cluster_sync();                                       // no CTA leaves while peers may write to it
}

using EncodeFn = void (*)(EncodeParams);

EncodeFn encode_kernel(uint32_t k) {
  switch (k) {
    case 3: return &tcq_encode_kernel<3>;
    case 4: return &tcq_encode_kernel<4>;
    case 5: return &tcq_encode_kernel<5>;
    default: return &tcq_encode_kernel<6>;
  }
}

}  // namespace

}  // namespace cpk

namespace {

// Launch configuration shared by the encoder entry points: the kernel, its
// shared memory, the clusters in flight for `rows` rows and the traceback
// bytes per cluster.
struct EncLaunch {
  cpk::EncodeFn fn;
  cpk::EncSmem smem;
  uint64_t clusters;
  uint64_t stride;
};

cp_status enc_args_ok(const float* e, uint64_t rows, uint32_t d, uint32_t k,
                      const uint16_t* lut_fp16, const uint8_t* records, const float* cost) {
  if (e == nullptr || records == nullptr || lut_fp16 == nullptr || rows == 0 ||
      !cpx::geometry_ok(d, k) || d < 16 || !cpx::aligned(e, 4) ||
      (cost != nullptr && !cpx::aligned(cost, 4))) {
    cpx::set_error("bad rows/records/LUT pointer or geometry");
    return CP_ERR_INVALID_ARG;
  }
  for (int i = 0; i < 1024; ++i) {
    if ((lut_fp16[i] & 0x7c00u) == 0x7c00u) {
      cpx::set_error("LUT holds a non-finite fp16 value");
      return CP_ERR_FORMAT;
    }
  }
  return CP_OK;
}

cp_status enc_launch_config(uint64_t rows, uint32_t d, uint32_t k, EncLaunch* out,
                            cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr) {
  const uint32_t T = d / 2, W = 16 - k;
  out->smem = cpk::enc_smem(d, k);
  out->fn = cpk::encode_kernel(k);
  cudaError_t err = cudaFuncSetAttribute(reinterpret_cast<const void*>(out->fn),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(out->smem.total));
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cpk::kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  *cfg = cudaLaunchConfig_t{};
  cfg->blockDim = dim3(cpk::kEncThreads);
  cfg->dynamicSmemBytes = out->smem.total;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
  int max_clusters = 0;
  if (err == cudaSuccess) {
    cfg->gridDim = dim3(cpk::kCluster * 64);
    err = cudaOccupancyMaxActiveClusters(&max_clusters, reinterpret_cast<const void*>(out->fn),
                                         cfg);
  }
  if (err != cudaSuccess || max_clusters < 1) {
    if (err == cudaSuccess) err = cudaErrorInvalidConfiguration;
    return cpx::cuda_fail(err, "tcq encoder cluster occupancy");
  }
  out->clusters =
      rows < static_cast<uint64_t>(max_clusters) ? rows : static_cast<uint64_t>(max_clusters);
  out->stride = (static_cast<uint64_t>(T) * (1ull << W) + 255) & ~255ull;
  cfg->gridDim = dim3(static_cast<unsigned>(out->clusters * cpk::kCluster));
  return CP_OK;
}

}  // namespace

extern "C" uint64_t cp_encode_workspace_bytes(uint64_t rows, uint32_t d, uint32_t bits_per_step) {
  if (rows == 0 || !cpx::geometry_ok(d, bits_per_step) || d < 16) return 0;
  EncLaunch el;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  if (enc_launch_config(rows, d, bits_per_step, &el, &cfg, attr) != CP_OK) return 0;
  return el.clusters * el.stride + 2048;
}

extern "C" cp_status cp_encode_rows_ws(const float* e, uint64_t rows, uint32_t d,
                                       uint32_t bits_per_step, const uint16_t* lut_fp16,
                                       uint8_t* records, float* cost, void* workspace,
                                       uint64_t workspace_bytes, void* stream) {
  cp_status st = enc_args_ok(e, rows, d, bits_per_step, lut_fp16, records, cost);
  if (st != CP_OK) return st;
  EncLaunch el;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  st = enc_launch_config(rows, d, bits_per_step, &el, &cfg, attr);
  if (st != CP_OK) return st;
  if (workspace == nullptr || !cpx::aligned(workspace, 256) ||
      workspace_bytes < el.clusters * el.stride + 2048) {
    cpx::set_error("workspace must be 256-byte aligned and hold cp_encode_workspace_bytes bytes");
    return CP_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cfg.stream = s;
  uint32_t* lut_dev =
      reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + el.clusters * el.stride);
  cudaError_t err = cudaMemcpyAsync(lut_dev, lut_fp16, 2048, cudaMemcpyHostToDevice, s);
  cpk::EncodeParams p;
  p.e = e;
  p.rows = rows;
  p.d = d;
  p.lut = lut_dev;
  p.records = records;
  p.cost = cost;
  p.work = static_cast<uint8_t*>(workspace);
  p.work_stride = el.stride;
  if (err == cudaSuccess) err = cudaLaunchKernelEx(&cfg, el.fn, p);
  if (err != cudaSuccess) return cpx::cuda_fail(err, "tcq encoder");
  return CP_OK;
}

extern "C" cp_status cp_encode_rows(const float* e, uint64_t rows, uint32_t d,
                                    uint32_t bits_per_step, const uint16_t* lut_fp16,
                                    uint8_t* records, float* cost, void* stream) {
  cp_status st = enc_args_ok(e, rows, d, bits_per_step, lut_fp16, records, cost);
  if (st != CP_OK) return st;
  const uint64_t bytes = cp_encode_workspace_bytes(rows, d, bits_per_step);
  if (bytes == 0) return CP_ERR_CUDA;                   // occupancy query failed (error set)
  void* mem = nullptr;
  cudaError_t err = cudaMalloc(&mem, bytes);
  if (err != cudaSuccess) {
    cpx::cuda_fail(err, "cudaMalloc(encoder workspace)");
    return CP_ERR_NO_MEMORY;
  }
  st = cp_encode_rows_ws(e, rows, d, bits_per_step, lut_fp16, records, cost, mem, bytes, stream);
  if (st == CP_OK) {
    err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) st = cpx::cuda_fail(err, "tcq encoder");
  }
  cudaFree(mem);
  return st;
}

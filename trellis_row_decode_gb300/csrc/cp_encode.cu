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
// Work mapping: one CTA of 1024 threads per row (persistent over rows); the
// 2^16 path metrics (two 256 KB buffers) and the traceback bytes live in a
// per-CTA global scratch that stays in L2; the LUT and z sit in shared memory.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "cp_internal.h"

namespace cpk {

namespace {

constexpr int kEncThreads = 1024;
constexpr uint32_t kStates = 1u << 16;

struct EncodeParams {
  const float* e;           // rows x d, fp32
  uint64_t rows;
  uint32_t d;
  const uint32_t* lut;      // 512 words: fp16 y0 | fp16 y1 << 16
  uint8_t* records;         // rows x R
  float* cost;              // rows (optional)
  uint8_t* work;            // per CTA: 2 x 2^16 floats, then T x 2^W traceback bytes
  uint64_t work_stride;     // bytes per CTA
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

// (y0, y1) of state s as fp32 (exact fp16 values), the sign of y1 from hash bit 23.
__device__ __forceinline__ float2 state_y(const uint32_t* lut, uint32_t s) {
  const uint32_t h = s * s + s;
  uint32_t v = lut[(h >> 14) & 511];
  if ((h >> 23) & 1u) v ^= 0x80000000u;
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

__device__ __forceinline__ float branch_cost(const uint32_t* lut, const float* z, uint32_t t,
                                             uint32_t s) {
  const float2 y = state_y(lut, s);
  const float a = __fsub_rn(z[2 * t], y.x);
  const float b = __fsub_rn(z[2 * t + 1], y.y);
  return __fadd_rn(__fmul_rn(a, a), __fmul_rn(b, b));
}

// CTA-wide argmin over 2^16 metrics: smallest finite value, ties to the smaller
// state; returns -1 (as 0xFFFFFFFF) when every metric is infinite.
__device__ uint32_t cta_argmin(const float* m, float* red_v, uint32_t* red_s, float* best_out) {
  const uint32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float bv = INFINITY;
  uint32_t bs = 0xFFFFFFFFu;
  for (uint32_t s = tid; s < kStates; s += kEncThreads) {
    const float v = m[s];
    if (v < bv) {                        // states of a thread ascend: strict < keeps the smaller
      bv = v;
      bs = s;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_down_sync(0xffffffffu, bv, o);
    const uint32_t os = __shfl_down_sync(0xffffffffu, bs, o);
    if (ov < bv || (ov == bv && os < bs)) {
      bv = ov;
      bs = os;
    }
  }
  if (lane == 0) {
    red_v[warp] = bv;
    red_s[warp] = bs;
  }
  __syncthreads();
  if (warp == 0) {
    bv = red_v[lane];
    bs = red_s[lane];
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_down_sync(0xffffffffu, bv, o);
      const uint32_t os = __shfl_down_sync(0xffffffffu, bs, o);
      if (ov < bv || (ov == bv && os < bs)) {
        bv = ov;
        bs = os;
      }
    }
    if (lane == 0) {
      red_v[0] = bv;
      red_s[0] = bs;
    }
  }
  __syncthreads();
  const uint32_t r = (red_v[0] == INFINITY) ? 0xFFFFFFFFu : red_s[0];
  *best_out = red_v[0];
  __syncthreads();
  return r;
}

// One pass over steps first+1 .. first+T-1 (mod T), cur holding the metrics of
// the states of step `first`; force_w >= 0 pins new bits in the w region.
template <int K>
__device__ float* viterbi_pass(const uint32_t* lut, const float* z, uint32_t T, uint32_t Lc,
                               float* cur, float* nxt, uint8_t* tb, uint32_t first,
                               int64_t force_w) {
  constexpr uint32_t W = 16 - K;
  constexpr uint32_t kGroups = 1u << W;
  const uint32_t tid = threadIdx.x;
  for (uint32_t i = 1; i < T; ++i) {
    const uint32_t t = (first + i) % T;
    uint32_t fmask = 0, fval = 0;
    if (force_w >= 0) {
      for (uint32_t b = 0; b < K; ++b) {
        const uint32_t pos = K * t + b;
        if (pos >= Lc - W) {
          fmask |= 1u << b;
          fval |= ((static_cast<uint32_t>(force_w) >> (pos - (Lc - W))) & 1u) << b;
        }
      }
    }
    uint8_t* tbi = tb + static_cast<size_t>(i) * kGroups;
    for (uint32_t g = tid; g < kGroups; g += kEncThreads) {
      const float* pr = cur + (static_cast<size_t>(g) << K);
      float best = pr[0];
      uint32_t by = 0;
#pragma unroll
      for (uint32_t y = 1; y < (1u << K); ++y) {
        const float m = pr[y];
        if (m < best) {
          best = m;
          by = y;
        }
      }
      tbi[g] = static_cast<uint8_t>(by);
#pragma unroll 4
      for (uint32_t x = 0; x < (1u << K); ++x) {
        const uint32_t s = (x << W) | g;
        nxt[s] = ((x & fmask) != fval) ? INFINITY : __fadd_rn(best, branch_cost(lut, z, t, s));
      }
    }
    __syncthreads();
    float* tmp = cur;
    cur = nxt;
    nxt = tmp;
  }
  return cur;
}

template <int K>
__global__ void __launch_bounds__(kEncThreads, 1) tcq_encode_kernel(const EncodeParams p) {
  constexpr uint32_t W = 16 - K;
  constexpr uint32_t kGroups = 1u << W;
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem);                  // 512 words
  float* red_v = reinterpret_cast<float*>(smem + 2048);               // 32
  uint32_t* red_s = reinterpret_cast<uint32_t*>(smem + 2048 + 128);   // 32
  double* sh_d = reinterpret_cast<double*>(smem + 2048 + 256);        // 4 doubles
  uint32_t* sh_u = reinterpret_cast<uint32_t*>(smem + 2048 + 288);    // 4 words
  float* z = reinterpret_cast<float*>(smem + 2048 + 304);             // d floats
  uint8_t* code = smem + 2048 + 304 + 4 * p.d;                        // Lc / 8 bytes

  const uint32_t tid = threadIdx.x;
  const uint32_t d = p.d, T = d / 2, Lc = K * T, code_bytes = Lc / 8;
  for (uint32_t i = tid; i < 512; i += kEncThreads) lut[i] = p.lut[i];
  float* cur = reinterpret_cast<float*>(p.work + blockIdx.x * p.work_stride);
  float* nxt = cur + kStates;
  uint8_t* tb = reinterpret_cast<uint8_t*>(nxt + kStates);
  __syncthreads();

  for (uint64_t r = blockIdx.x; r < p.rows; r += gridDim.x) {
    const float* er = p.e + r * d;
    uint8_t* rec = p.records + r * (code_bytes + 2);
    // |e| and z = (float)(e * sqrt(d) / |e|) in fp64, sums in index order
    if (tid == 0) {
      double ss = 0.0;
      for (uint32_t q = 0; q < d; ++q) {
        const double v = static_cast<double>(er[q]);
        ss = __dadd_rn(ss, __dmul_rn(v, v));
      }
      const double nrm = __dsqrt_rn(ss);
      sh_d[0] = nrm;
      sh_d[1] = (nrm == 0.0) ? 0.0 : __ddiv_rn(__dsqrt_rn(static_cast<double>(d)), nrm);
    }
    __syncthreads();
    const double nrm = sh_d[0], sc = sh_d[1];
    if (nrm == 0.0) {                                   // zero row: zero code, alpha = 0
      for (uint32_t i = tid; i < code_bytes + 2; i += kEncThreads) rec[i] = 0;
      if (tid == 0 && p.cost) p.cost[r] = 0.0f;
      __syncthreads();
      continue;
    }
    for (uint32_t q = tid; q < d; q += kEncThreads)
      z[q] = __double2float_rn(__dmul_rn(static_cast<double>(er[q]), sc));
    __syncthreads();

    // pass 1: free start at step rho = T/2, every state live
    const uint32_t rho = T / 2;
    for (uint32_t s = tid; s < kStates; s += kEncThreads) cur[s] = branch_cost(lut, z, rho, s);
    __syncthreads();
    float* fin = viterbi_pass<K>(lut, z, T, Lc, cur, nxt, tb, rho, -1);
    float bestv;
    uint32_t bs = cta_argmin(fin, red_v, red_s, &bestv);
    if (tid == 0) {                                     // walk back to original step T-1
      uint32_t s = bs;
      const uint32_t target = T - 1 - rho;
      for (uint32_t i = T - 1; i > target; --i) {
        const uint32_t g = s & (kGroups - 1);
        s = (g << K) | tb[static_cast<size_t>(i) * kGroups + g];
      }
      sh_u[0] = s >> K;                                 // the pre-window bits w
    }
    __syncthreads();
    const uint32_t w = sh_u[0];

    // pass 2: constrained to w
    float* c2 = (fin == cur) ? nxt : cur;
    float* n2 = fin;
    for (uint32_t s = tid; s < kStates; s += kEncThreads) c2[s] = INFINITY;
    __syncthreads();
    if (tid < (1u << K)) {
      const uint32_t s = w | (tid << W);
      c2[s] = branch_cost(lut, z, 0, s);
    }
    __syncthreads();
    fin = viterbi_pass<K>(lut, z, T, Lc, c2, n2, tb, 0, static_cast<int64_t>(w));
    bs = cta_argmin(fin, red_v, red_s, &bestv);

    // traceback: new bits of step t are the top K bits of s_t
    for (uint32_t i = tid; i < code_bytes; i += kEncThreads) code[i] = 0;
    __syncthreads();
    if (tid == 0) {
      uint32_t s = bs;
      for (int64_t t = T - 1; t >= 0; --t) {
        const uint32_t x = s >> W;
        for (uint32_t b = 0; b < K; ++b) {
          const uint32_t j = K * static_cast<uint32_t>(t) + b;
          if ((x >> b) & 1u) code[j >> 3] |= static_cast<uint8_t>(1u << (j & 7));
        }
        if (t > 0) {
          const uint32_t g = s & (kGroups - 1);
          s = (g << K) | tb[static_cast<size_t>(t) * kGroups + g];
        }
      }
      // alpha = |e| / |f(c)|, |f|^2 in fp64 over coordinates in order
      double fs = 0.0;
      for (uint32_t t = 0; t < T; ++t) {
        uint32_t st = 0;
        const int32_t first = static_cast<int32_t>(K * (t + 1)) - 16;
        for (int m = 0; m < 16; ++m) {
          int32_t pos = (first + m) % static_cast<int32_t>(Lc);
          if (pos < 0) pos += Lc;
          st |= static_cast<uint32_t>((code[pos >> 3] >> (pos & 7)) & 1u) << m;
        }
        const float2 y = state_y(lut, st);
        const double y0 = y.x, y1 = y.y;
        fs = __dadd_rn(fs, __dmul_rn(y0, y0));
        fs = __dadd_rn(fs, __dmul_rn(y1, y1));
      }
      const uint16_t ab = double_to_bf16_rne(__ddiv_rn(nrm, __dsqrt_rn(fs)));
      sh_u[1] = ab;
      if (p.cost) p.cost[r] = bestv;
    }
    __syncthreads();
    for (uint32_t i = tid; i < code_bytes; i += kEncThreads) rec[i] = code[i];
    if (tid == 0) {
      rec[code_bytes] = static_cast<uint8_t>(sh_u[1] & 0xFF);
      rec[code_bytes + 1] = static_cast<uint8_t>(sh_u[1] >> 8);
    }
    __syncthreads();
  }
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

extern "C" cp_status cp_encode_rows(const float* e, uint64_t rows, uint32_t d,
                                    uint32_t bits_per_step, const uint16_t* lut_fp16,
                                    uint8_t* records, float* cost, void* stream) {
  if (e == nullptr || records == nullptr || lut_fp16 == nullptr || rows == 0 ||
      !cpx::geometry_ok(d, bits_per_step) || d < 16 || !cpx::aligned(e, 4) ||
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
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const uint32_t k = bits_per_step, T = d / 2, W = 16 - k;
  const uint64_t ctas = rows < static_cast<uint64_t>(sms) ? rows : static_cast<uint64_t>(sms);
  const uint64_t stride = ((2ull * cpk::kStates * sizeof(float) +
                            static_cast<uint64_t>(T) * (1ull << W)) + 255) & ~255ull;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* mem = nullptr;
  cudaError_t err = cudaMalloc(&mem, ctas * stride + 2048);
  if (err != cudaSuccess) {
    cpx::cuda_fail(err, "cudaMalloc(encoder workspace)");
    return CP_ERR_NO_MEMORY;
  }
  uint32_t* lut_dev = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(mem) + ctas * stride);
  err = cudaMemcpyAsync(lut_dev, lut_fp16, 2048, cudaMemcpyHostToDevice, s);
  cpk::EncodeParams p;
  p.e = e;
  p.rows = rows;
  p.d = d;
  p.lut = lut_dev;
  p.records = records;
  p.cost = cost;
  p.work = static_cast<uint8_t*>(mem);
  p.work_stride = stride;
  const size_t smem = 2048 + 304 + 4ull * d + (k * T) / 8 + 16;
  cpk::EncodeFn fn = cpk::encode_kernel(k);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err == cudaSuccess) {
    void* args[] = {&p};
    err = cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3(static_cast<unsigned>(ctas)),
                           dim3(cpk::kEncThreads), args, smem, s);
  }
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  cudaFree(mem);
  if (err != cudaSuccess) return cpx::cuda_fail(err, "tcq encoder");
  return CP_OK;
}

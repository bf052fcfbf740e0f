// cp_oracle.cpp -- plain, slow CPU oracle for the Conditional Program (CP)
// lookup-decode and its offline encoder.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
// benchmark's CPU-baseline leg load this library.  It shares no code, header,
// table or constant generator with the CUDA library; the two meet only at the
// record bytes, the LUT data file and the index arrays.
//
// Pages cited (by title):
//   [P1] "Two-bit lookup tables shrink DeepSeek's 203 GB memory to 51 GB and
//        cut prefill from 64.66 s to 13.27 s" (ai4snews.wisdomeyes.cn)
//   [P4] "2비트 코드와 공유 트렐리스로 n-gram 룩업 테이블을 4~8배 압축한다"
//        (onedev.kr/papers/1189); sections "어떻게 동작하나" (how it works),
//        "무엇과 다른가" (how it differs), "전제와 한계" (assumptions and limits).
//
// What the pages fix: e_hat_i = alpha_i * f(c_i) with one shared f [P4 how it
// works]; b + 16/d bits per parameter [P4 how it works]; z_i = sqrt(d) e_i/|e_i|
// treated as an N(0,1) source, coded by a tail-biting Gaussian HYB bitshift
// trellis (TCQ) with no per-row rotation, and alpha_i = |e_i|_2 / |f(c_i)|_2
// [P4 how it differs].  The pages leave the trellis constants open; this format
// fixes them as: V = 2 coordinates per step, k = 2b bits per step, an L = 16 bit
// state equal to the 16 code bits ending at bit k(t+1), read cyclically
// (tail-biting); hash h = s*s + s mod 2^32, LUT index (h >> 14) & 511 into a
// 512-entry fp16 2-vector LUT, second coordinate negated when bit 23 of h is set;
// alpha multiplied in fp32 and rounded once to bf16.
//
// Every floating-point reduction below runs in index order in fp64 unless a
// step states fp32; the library must be compiled with -ffp-contract=off so that
// no multiply-add is fused.

#include <cmath>
#include <functional>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

constexpr int kStateBits = 16;          // L
constexpr uint32_t kStates = 1u << kStateBits;

// ---------------------------------------------------------------------------
// Number formats (IEEE binary16 and bfloat16), written from their definitions.
// ---------------------------------------------------------------------------

// binary16 bits -> exact double.
double half_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int ex = (h >> 10) & 0x1f;
  const int man = h & 0x3ff;
  double v;
  if (ex == 0) {
    v = std::ldexp((double)man, -24);                 // subnormal: man * 2^-24
  } else if (ex == 31) {
    v = man ? std::numeric_limits<double>::quiet_NaN()
            : std::numeric_limits<double>::infinity();
  } else {
    v = std::ldexp((double)(1024 + man), ex - 25);    // (1.man) * 2^(ex-15)
  }
  return sign ? -v : v;
}

// Round a finite double to a binary format with p significand bits (implicit
// bit included) whose smallest normal exponent is emin, ties to even.  The
// result is returned as an (exact) double; overflow is the caller's business.
double round_to_format(double x, int p, int emin) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  int e;
  std::frexp(std::fabs(x), &e);       // |x| = m * 2^e, m in [0.5, 1)
  int lead = e - 1;                   // exponent of the leading bit
  if (lead < emin) lead = emin;       // subnormal range: fixed quantum
  const double quantum = std::ldexp(1.0, lead - p + 1);
  return std::nearbyint(x / quantum) * quantum;   // default mode: ties to even
}

// double -> binary16 bits, one rounding (ties to even).
uint16_t double_to_half(double x) {
  if (std::isnan(x)) return 0x7e00;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  const double r = std::fabs(round_to_format(x, 11, -14));
  if (r > 65504.0) return sign | 0x7c00;               // overflow -> inf
  if (r == 0.0) return sign;
  if (r < std::ldexp(1.0, -14)) {                       // subnormal
    return sign | (uint16_t)std::lround(r / std::ldexp(1.0, -24));
  }
  int e;
  const double m = std::frexp(r, &e);                   // r = m * 2^e
  const int ex = e - 1 + 15;
  const int man = (int)std::lround(m * 2048.0) - 1024;  // 11 significant bits
  return sign | (uint16_t)(ex << 10) | (uint16_t)man;
}

// bfloat16 bits -> float (exact).
float bf16_to_float(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// float -> bfloat16 bits, ties to even; NaN -> canonical 0x7fff.
uint16_t float_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fff;
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

// double -> bfloat16 bits with a single rounding (used for the stored alpha).
uint16_t double_to_bf16(double x) {
  if (std::isnan(x)) return 0x7fff;
  const double r = round_to_format(x, 8, -126);
  const double max_bf16 = std::ldexp(255.0, 120);       // (2 - 2^-7) * 2^127
  if (std::fabs(r) > max_bf16) return std::signbit(x) ? 0xff80 : 0x7f80;
  const float f = (float)r;                              // exact: r has <= 8 bits
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

// ---------------------------------------------------------------------------
// Trellis decoder f [P4 how it works / how it differs], constants as above.
// ---------------------------------------------------------------------------

struct Geometry {
  uint32_t d;    // coordinates per row
  uint32_t k;    // bits per 2-coordinate step (k = 2b)
  uint32_t T;    // steps per row = d / 2
  uint32_t Lc;   // code bits per row = d * b = k * T
};

Geometry make_geometry(uint32_t d, uint32_t k) {
  Geometry g;
  g.d = d;
  g.k = k;
  g.T = d / 2;
  g.Lc = k * (d / 2);
  return g;
}

// Code bit j: least significant bit first inside little-endian bytes.
int code_bit(const uint8_t* code, uint64_t j) { return (code[j >> 3] >> (j & 7)) & 1; }

// Cyclic bit position (tail-biting): any integer position reduced mod Lc.
uint64_t cyc(int64_t pos, uint32_t Lc) {
  int64_t r = pos % (int64_t)Lc;
  if (r < 0) r += Lc;
  return (uint64_t)r;
}

// State s_t: the 16 code bits that end at bit k(t+1), oldest bit lowest.
uint32_t window_state(const uint8_t* code, const Geometry& g, uint32_t t) {
  uint32_t s = 0;
  const int64_t first = (int64_t)g.k * (t + 1) - kStateBits;
  for (int m = 0; m < kStateBits; ++m) s |= (uint32_t)code_bit(code, cyc(first + m, g.Lc)) << m;
  return s;
}

// Hashed LUT read for one state: (y0, y1) as exact doubles of fp16 values.
void state_values(uint32_t s, const uint16_t* lut, double* y0, double* y1) {
  const uint32_t h = s * s + s;                 // arithmetic mod 2^32
  const uint32_t idx = (h >> 14) & 511u;
  const bool neg = (h >> 23) & 1u;
  *y0 = half_to_double(lut[2 * idx]);
  const double v1 = half_to_double(lut[2 * idx + 1]);
  *y1 = neg ? -v1 : v1;
}

// f(c): d values, step t gives coordinates 2t and 2t+1.
void decode_f(const uint8_t* code, const Geometry& g, const uint16_t* lut, double* f) {
  for (uint32_t t = 0; t < g.T; ++t) {
    double y0, y1;
    state_values(window_state(code, g, t), lut, &y0, &y1);
    f[2 * t] = y0;
    f[2 * t + 1] = y1;
  }
}

// One reconstructed row: out[q] = bf16_rne(float(alpha) * float(f[q])), the
// product taken in fp32.
void reconstruct_row(const uint8_t* code, uint16_t alpha_bits, const Geometry& g,
                     const uint16_t* lut, uint16_t* out) {
  std::vector<double> f(g.d);
  decode_f(code, g, lut, f.data());
  const float a = bf16_to_float(alpha_bits);
  for (uint32_t q = 0; q < g.d; ++q) {
    const float y = (float)f[q];                // exact: fp16 value
    const float prod = a * y;
    out[q] = float_to_bf16(prod);
  }
}

// ---------------------------------------------------------------------------
// Encoder: tail-biting TCQ search over the trellis [P4 how it differs].
// Distortion D(c) = sum_t (z_2t - y0(s_t))^2 + (z_2t+1 - y1(s_t))^2, fp64,
// summed in t order.
// ---------------------------------------------------------------------------

struct StateTable {
  std::vector<double> y0, y1;
};

StateTable make_state_table(const uint16_t* lut) {
  StateTable st;
  st.y0.resize(kStates);
  st.y1.resize(kStates);
  for (uint32_t s = 0; s < kStates; ++s) state_values(s, lut, &st.y0[s], &st.y1[s]);
  return st;
}

inline double step_cost(const StateTable& st, const double* z, uint32_t t, uint32_t s) {
  const double a = z[2 * t] - st.y0[s];
  const double b = z[2 * t + 1] - st.y1[s];
  const double aa = a * a;
  const double bb = b * b;
  return aa + bb;
}

double distortion(const uint8_t* code, const Geometry& g, const StateTable& st, const double* z) {
  double acc = 0.0;
  for (uint32_t t = 0; t < g.T; ++t) acc = acc + step_cost(st, z, t, window_state(code, g, t));
  return acc;
}

void set_code_bit(uint8_t* code, uint64_t j, int v) {
  if (v) code[j >> 3] |= (uint8_t)(1u << (j & 7));
  else code[j >> 3] &= (uint8_t)~(1u << (j & 7));
}

// Viterbi over the trellis with the W = 16 - k "pre-window" bits w fixed.
// w holds the bits at cyclic positions [Lc - W, Lc) (bit m of w is position
// Lc - W + m).  Steps run in original order t = 0..T-1; the state after step t
// is s_t.  New bits of step t sit at positions [kt, k(t+1)); any of them inside
// the w region is forced.  Survivor rule at a merge: smaller path metric, then
// smaller dropped bits (the predecessor's low k bits), which makes the result
// the smallest code (as a little-endian integer) among equal costs.
// Returns the best cost and writes the code; +inf if no path exists.
// Scratch arrays of one search, reused across the w values of an exact search.
struct ViterbiWork {
  std::vector<double> cur, best_m;
  std::vector<uint16_t> tb, best_drop;   // tb: predecessor state per (t, s)
  std::vector<uint32_t> live, nlive;
  std::vector<uint8_t> seen;
  explicit ViterbiWork(uint32_t T)
      : cur(kStates), best_m(kStates), tb((size_t)T * kStates), best_drop(kStates),
        seen(kStates, 0) {}
};

double viterbi_fixed_w(const double* z, const Geometry& g, const StateTable& st, uint32_t w,
                       uint8_t* code_out, ViterbiWork& wk) {
  const uint32_t k = g.k, T = g.T, Lc = g.Lc;
  const uint32_t W = kStateBits - k;
  const uint32_t xmask = (1u << k) - 1;
  const double inf = std::numeric_limits<double>::infinity();
  std::vector<double>& cur = wk.cur;
  std::vector<uint16_t>& tb = wk.tb;
  std::vector<uint32_t>& live = wk.live;
  std::vector<uint32_t>& nlive = wk.nlive;
  std::vector<uint8_t>& seen = wk.seen;
  std::vector<double>& best_m = wk.best_m;
  std::vector<uint16_t>& best_drop = wk.best_drop;
  live.clear();

  // Step 0: s_0 = w | (x << W); positions [0, k) are never in the w region
  // because Lc >= 16.
  for (uint32_t x = 0; x <= xmask; ++x) {
    const uint32_t s = w | (x << W);
    cur[s] = step_cost(st, z, 0, s);
    live.push_back(s);
  }
  for (uint32_t t = 1; t < T; ++t) {
    // Which new bits are forced by w, and to what.
    uint32_t force_mask = 0, force_val = 0;
    for (uint32_t i = 0; i < k; ++i) {
      const uint64_t pos = (uint64_t)k * t + i;
      if (pos >= (uint64_t)(Lc - W)) {
        force_mask |= 1u << i;
        force_val |= ((w >> (pos - (Lc - W))) & 1u) << i;
      }
    }
    nlive.clear();
    for (uint32_t sp : live) {
      const double mp = cur[sp];
      const uint32_t dropped = sp & xmask;
      for (uint32_t x = 0; x <= xmask; ++x) {
        if ((x & force_mask) != force_val) continue;
        const uint32_t s = (sp >> k) | (x << W);
        const double m = mp + step_cost(st, z, t, s);
        if (!seen[s]) {
          seen[s] = 1;
          nlive.push_back(s);
          best_m[s] = m;
          best_drop[s] = (uint16_t)dropped;
          tb[(size_t)t * kStates + s] = (uint16_t)sp;
        } else if (m < best_m[s] || (m == best_m[s] && dropped < best_drop[s])) {
          best_m[s] = m;
          best_drop[s] = (uint16_t)dropped;
          tb[(size_t)t * kStates + s] = (uint16_t)sp;
        }
      }
    }
    for (uint32_t s : nlive) {
      cur[s] = best_m[s];
      seen[s] = 0;
    }
    live.swap(nlive);
  }
  // Final state: min cost, ties -> smaller state (its high W bits equal w).
  double best = inf;
  uint32_t bs = 0;
  bool found = false;
  for (uint32_t s : live) {
    if (!found || cur[s] < best || (cur[s] == best && s < bs)) {
      best = cur[s];
      bs = s;
      found = true;
    }
  }
  if (!found) return inf;
  // Traceback: the new bits of step t are the top k bits of s_t.
  std::memset(code_out, 0, (Lc + 7) / 8);
  uint32_t s = bs;
  for (int64_t t = T - 1; t >= 0; --t) {
    const uint32_t x = s >> W;
    for (uint32_t i = 0; i < k; ++i) set_code_bit(code_out, (uint64_t)k * t + i, (x >> i) & 1u);
    if (t > 0) s = tb[(size_t)t * kStates + s];
  }
  return best;
}

// Exact tail-biting search: every w, keep the strictly better (so the smaller
// w wins a tie, w being the most significant code bits).
double viterbi_exact(const double* z, const Geometry& g, const StateTable& st, uint8_t* code_out) {
  const uint32_t W = kStateBits - g.k;
  const size_t nb = (g.Lc + 7) / 8;
  std::vector<uint8_t> tmp(nb);
  ViterbiWork wk(g.T);
  double best = std::numeric_limits<double>::infinity();
  for (uint32_t w = 0; w < (1u << W); ++w) {
    const double c = viterbi_fixed_w(z, g, st, w, tmp.data(), wk);
    if (c < best) {
      best = c;
      std::memcpy(code_out, tmp.data(), nb);
    }
  }
  return best;
}

// Two-pass search: a free-start Viterbi on the sequence rotated by T/2 steps
// picks w (read off its path mid-sequence); one constrained Viterbi with that
// w gives a valid tail-biting code whose cost is >= the exact optimum.
double viterbi_two_pass(const double* z, const Geometry& g, const StateTable& st,
                        uint8_t* code_out) {
  const uint32_t k = g.k, T = g.T;
  const uint32_t W = kStateBits - k;
  const uint32_t xmask = (1u << k) - 1;
  const uint32_t rho = T / 2;
  const double inf = std::numeric_limits<double>::infinity();
  std::vector<double> cur(kStates), nxt(kStates);
  std::vector<uint16_t> tb((size_t)T * kStates, 0);
  for (uint32_t s = 0; s < kStates; ++s) cur[s] = step_cost(st, z, rho % T, s);
  for (uint32_t tp = 1; tp < T; ++tp) {
    const uint32_t t = (tp + rho) % T;
    std::fill(nxt.begin(), nxt.end(), inf);
    std::vector<uint16_t> drop(kStates, 0xffff);
    for (uint32_t sp = 0; sp < kStates; ++sp) {
      const uint32_t dropped = sp & xmask;
      for (uint32_t x = 0; x <= xmask; ++x) {
        const uint32_t s = (sp >> k) | (x << W);
        const double m = cur[sp] + step_cost(st, z, t, s);
        if (m < nxt[s] || (m == nxt[s] && dropped < drop[s])) {
          nxt[s] = m;
          drop[s] = (uint16_t)dropped;
          tb[(size_t)tp * kStates + s] = (uint16_t)sp;
        }
      }
    }
    cur.swap(nxt);
  }
  uint32_t bs = 0;
  for (uint32_t s = 1; s < kStates; ++s)
    if (cur[s] < cur[bs]) bs = s;
  // Walk back to rotated step T-1-rho, i.e. original step T-1, whose state is
  // the window [Lc-16, Lc); its top W bits are the w region.
  uint32_t s = bs;
  const uint32_t target = T - 1 - rho;
  for (uint32_t tp = T - 1; tp > target; --tp) s = tb[(size_t)tp * kStates + s];
  const uint32_t w = s >> k;
  ViterbiWork wk(T);
  return viterbi_fixed_w(z, g, st, w, code_out, wk);
}

// ---------------------------------------------------------------------------
// fp32 variant of the encoder (the precision of the GPU encoder; the pages fix
// none).  z comes from the fp64 normalisation rounded to fp32; branch cost
// D = fl(fl((z0 - y0)^2) + fl((z1 - y1)^2)) in fp32 without fused multiply-adds;
// path metrics in fp32.  Recursion per step: the 2^k states that share their
// low W = 16 - k bits (a group g) also share their 2^k predecessors
// (g << k) | y, so the survivor is chosen once per group, smallest predecessor
// metric first, then smallest dropped bits y; every state of the group then
// gets metric fl(min + D(s)).  Since fl(a + D) is monotone in a, the optimum
// equals the minimum over all paths of their fp32 sums accumulated in t order.
// ---------------------------------------------------------------------------

struct StateTableF {
  std::vector<float> y0, y1;
};

StateTableF make_state_table_f(const uint16_t* lut) {
  StateTableF st;
  st.y0.resize(kStates);
  st.y1.resize(kStates);
  for (uint32_t s = 0; s < kStates; ++s) {
    double a, b;
    state_values(s, lut, &a, &b);
    st.y0[s] = (float)a;
    st.y1[s] = (float)b;
  }
  return st;
}

inline float step_cost_f(const StateTableF& st, const float* z, uint32_t t, uint32_t s) {
  const float a = z[2 * t] - st.y0[s];
  const float b = z[2 * t + 1] - st.y1[s];
  const float aa = a * a;
  const float bb = b * b;
  return aa + bb;
}

float distortion_f(const uint8_t* code, const Geometry& g, const StateTableF& st, const float* z) {
  float acc = 0.0f;
  for (uint32_t t = 0; t < g.T; ++t) acc = acc + step_cost_f(st, z, t, window_state(code, g, t));
  return acc;
}

// One Viterbi pass in fp32 over steps t_0 .. t_{T-1} = (first + i) mod T.
// init: metrics of the states before the first transition (step `first`);
// force_w >= 0 constrains new bits in the w region (positions >= Lc - W) to w.
// tb[i * 2^W + g] receives the chosen dropped bits of group g at pass step i.
// Returns the final metrics.
std::vector<float> viterbi_pass_f(const float* z, const Geometry& g, const StateTableF& st,
                                  std::vector<float> cur, uint32_t first, int64_t force_w,
                                  std::vector<uint8_t>& tb) {
  const uint32_t k = g.k, T = g.T, Lc = g.Lc;
  const uint32_t W = kStateBits - k;
  const uint32_t groups = 1u << W;
  const float inf = std::numeric_limits<float>::infinity();
  std::vector<float> nxt(kStates);
  tb.assign((size_t)T * groups, 0);
  for (uint32_t i = 1; i < T; ++i) {
    const uint32_t t = (first + i) % T;
    uint32_t force_mask = 0, force_val = 0;
    if (force_w >= 0) {
      for (uint32_t b = 0; b < k; ++b) {
        const uint64_t pos = (uint64_t)k * t + b;
        if (pos >= (uint64_t)(Lc - W)) {
          force_mask |= 1u << b;
          force_val |= (((uint32_t)force_w >> (pos - (Lc - W))) & 1u) << b;
        }
      }
    }
    for (uint32_t grp = 0; grp < groups; ++grp) {
      float best = cur[(size_t)grp << k];
      uint32_t by = 0;
      for (uint32_t y = 1; y < (1u << k); ++y) {
        const float m = cur[((size_t)grp << k) | y];
        if (m < best) {
          best = m;
          by = y;
        }
      }
      tb[(size_t)i * groups + grp] = (uint8_t)by;
      for (uint32_t x = 0; x < (1u << k); ++x) {
        const uint32_t s = (x << W) | grp;
        nxt[s] = ((x & force_mask) != force_val) ? inf : best + step_cost_f(st, z, t, s);
      }
    }
    cur.swap(nxt);
  }
  return cur;
}

// Smallest finite metric, ties to the smaller state; -1 if none.
int64_t argmin_state_f(const std::vector<float>& m) {
  int64_t bs = -1;
  for (uint32_t s = 0; s < kStates; ++s)
    if (m[s] != std::numeric_limits<float>::infinity() && (bs < 0 || m[s] < m[bs])) bs = s;
  return bs;
}

// Code of the path ending in state `fin` after a constrained pass from step 0.
void traceback_code_f(const Geometry& g, const std::vector<uint8_t>& tb, uint32_t fin,
                      uint8_t* code_out) {
  const uint32_t k = g.k, W = kStateBits - k, groups = 1u << W;
  std::memset(code_out, 0, (g.Lc + 7) / 8);
  uint32_t s = fin;
  for (int64_t t = g.T - 1; t >= 0; --t) {
    const uint32_t x = s >> W;
    for (uint32_t i = 0; i < k; ++i) set_code_bit(code_out, (uint64_t)k * t + i, (x >> i) & 1u);
    if (t > 0) {
      const uint32_t grp = s & (groups - 1);
      s = (grp << k) | tb[(size_t)t * groups + grp];
    }
  }
}

// Constrained fp32 pass with pre-window w; returns the cost (inf if no path).
float viterbi_fixed_w_f(const float* z, const Geometry& g, const StateTableF& st, uint32_t w,
                        uint8_t* code_out) {
  const uint32_t k = g.k, W = kStateBits - k;
  std::vector<float> cur(kStates, std::numeric_limits<float>::infinity());
  for (uint32_t x = 0; x < (1u << k); ++x) {
    const uint32_t s = w | (x << W);
    cur[s] = step_cost_f(st, z, 0, s);
  }
  std::vector<uint8_t> tb;
  const std::vector<float> fin = viterbi_pass_f(z, g, st, cur, 0, (int64_t)w, tb);
  const int64_t bs = argmin_state_f(fin);
  if (bs < 0) return std::numeric_limits<float>::infinity();
  traceback_code_f(g, tb, (uint32_t)bs, code_out);
  return fin[bs];
}

float viterbi_exact_f(const float* z, const Geometry& g, const StateTableF& st, uint8_t* code_out) {
  const uint32_t W = kStateBits - g.k;
  const size_t nb = (g.Lc + 7) / 8;
  std::vector<uint8_t> tmp(nb);
  float best = std::numeric_limits<float>::infinity();
  for (uint32_t w = 0; w < (1u << W); ++w) {
    const float c = viterbi_fixed_w_f(z, g, st, w, tmp.data());
    if (c < best) {
      best = c;
      std::memcpy(code_out, tmp.data(), nb);
    }
  }
  return best;
}

// Two-pass fp32: free-start pass on the sequence rotated by T/2 steps, w read
// off its best path at original step T-1, then one constrained pass.
float viterbi_two_pass_f(const float* z, const Geometry& g, const StateTableF& st,
                         uint8_t* code_out) {
  const uint32_t k = g.k, T = g.T, W = kStateBits - k, groups = 1u << W;
  const uint32_t rho = T / 2;
  std::vector<float> cur(kStates);
  for (uint32_t s = 0; s < kStates; ++s) cur[s] = step_cost_f(st, z, rho % T, s);
  std::vector<uint8_t> tb;
  const std::vector<float> fin = viterbi_pass_f(z, g, st, cur, rho, -1, tb);
  uint32_t s = (uint32_t)argmin_state_f(fin);
  const uint32_t target = T - 1 - rho;
  for (uint32_t i = T - 1; i > target; --i) {
    const uint32_t grp = s & (groups - 1);
    s = (grp << k) | tb[(size_t)i * groups + grp];
  }
  return viterbi_fixed_w_f(z, g, st, s >> k, code_out);
}

// The first pass of the two-pass search on its own (a test hook): a free-start
// fp32 Viterbi over the steps taken in the order rho, rho + 1, ... (mod T), every
// state live at the start.  Returns the best final metric (ties to the smaller
// state) and writes the states of that best path at every original step t.
// Any tail-biting code is one of these paths, so its result never exceeds the
// exact tail-biting cost (a relaxation).
float free_start_f(const float* z, const Geometry& g, const StateTableF& st, uint32_t rho,
                   uint32_t* states) {
  const uint32_t k = g.k, T = g.T, W = kStateBits - k, groups = 1u << W;
  std::vector<float> cur(kStates);
  for (uint32_t s = 0; s < kStates; ++s) cur[s] = step_cost_f(st, z, rho % T, s);
  std::vector<uint8_t> tb;
  const std::vector<float> fin = viterbi_pass_f(z, g, st, cur, rho, -1, tb);
  const int64_t best = argmin_state_f(fin);
  uint32_t s = (uint32_t)best;
  for (int64_t i = T - 1; i >= 0; --i) {
    states[(rho + (uint32_t)i) % T] = s;
    if (i > 0) {
      const uint32_t grp = s & (groups - 1);
      s = (grp << k) | tb[(size_t)i * groups + grp];
    }
  }
  return fin[best];
}

// The same minimum by enumeration (a test hook for small T): every start state
// and every k-bit symbol at each later step, the cost of a path accumulated in
// fp32 in the pass's step order, the first strictly smaller cost kept.
float free_start_brute_f(const float* z, const Geometry& g, const StateTableF& st, uint32_t rho,
                         uint32_t* states) {
  const uint32_t k = g.k, T = g.T, W = kStateBits - k;
  std::vector<uint32_t> path(T), best_path(T);
  float best = std::numeric_limits<float>::infinity();
  std::function<void(uint32_t, uint32_t, float)> extend = [&](uint32_t i, uint32_t s, float acc) {
    path[i] = s;
    if (i + 1 == T) {
      if (acc < best) {
        best = acc;
        best_path = path;
      }
      return;
    }
    const uint32_t t = (rho + i + 1) % T;
    for (uint32_t x = 0; x < (1u << k); ++x) {
      const uint32_t ns = (s >> k) | (x << W);
      extend(i + 1, ns, acc + step_cost_f(st, z, t, ns));
    }
  };
  for (uint32_t s0 = 0; s0 < kStates; ++s0) extend(0, s0, step_cost_f(st, z, rho % T, s0));
  for (uint32_t i = 0; i < T; ++i) states[(rho + i) % T] = best_path[i];
  return best;
}

float brute_force_f(const float* z, const Geometry& g, const StateTableF& st, uint8_t* code_out) {
  const size_t nb = (g.Lc + 7) / 8;
  std::vector<uint8_t> code(nb);
  float best = std::numeric_limits<float>::infinity();
  for (uint64_t c = 0; c < (1ull << g.Lc); ++c) {
    for (size_t b = 0; b < nb; ++b) code[b] = (uint8_t)(c >> (8 * b));
    const float D = distortion_f(code.data(), g, st, z);
    if (D < best) {
      best = D;
      std::memcpy(code_out, code.data(), nb);
    }
  }
  return best;
}

// Brute force over all 2^Lc codes (Lc <= 26): smallest cost, then smallest code.
double brute_force(const double* z, const Geometry& g, const StateTable& st, uint8_t* code_out) {
  const size_t nb = (g.Lc + 7) / 8;
  std::vector<uint8_t> code(nb);
  double best = std::numeric_limits<double>::infinity();
  const uint64_t total = 1ull << g.Lc;
  for (uint64_t c = 0; c < total; ++c) {
    for (size_t b = 0; b < nb; ++b) code[b] = (uint8_t)(c >> (8 * b));
    const double D = distortion(code.data(), g, st, z);
    if (D < best) {
      best = D;
      std::memcpy(code_out, code.data(), nb);
    }
  }
  return best;
}

// ---------------------------------------------------------------------------
// Shared LUT construction: Lloyd k-means on seeded N(0,1) pairs.
// ---------------------------------------------------------------------------

// SplitMix64 (Steele, Lea & Flood 2014): one 64-bit output per counter value.
uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

// Box-Muller transform of two uniforms from the counter stream; u1 in (0, 1].
void normal_pair(uint64_t seed, uint64_t i, double* a, double* b) {
  const uint64_t r1 = splitmix64(seed ^ splitmix64(2 * i));
  const uint64_t r2 = splitmix64(seed ^ splitmix64(2 * i + 1));
  const double u1 = (double)((r1 >> 11) + 1) * 0x1.0p-53;
  const double u2 = (double)(r2 >> 11) * 0x1.0p-53;
  const double rad = std::sqrt(-2.0 * std::log(u1));
  const double th = 2.0 * M_PI * u2;
  *a = rad * std::cos(th);
  *b = rad * std::sin(th);
}

}  // namespace

// ===========================================================================
// C ABI for the Python test harness (ctypes).
// ===========================================================================
extern "C" {

double orc_half_to_double(uint16_t h) { return half_to_double(h); }
uint16_t orc_double_to_half(double x) { return double_to_half(x); }
uint16_t orc_float_to_bf16(float f) { return float_to_bf16(f); }
uint16_t orc_double_to_bf16(double x) { return double_to_bf16(x); }
float orc_bf16_to_float(uint16_t b) { return bf16_to_float(b); }

uint64_t orc_splitmix64(uint64_t x) { return splitmix64(x); }

void orc_normal_pairs(uint64_t seed, uint64_t first, uint64_t count, double* out) {
  for (uint64_t i = 0; i < count; ++i) normal_pair(seed, first + i, &out[2 * i], &out[2 * i + 1]);
}

// Lloyd k-means in 2-D.  Points: n_pairs N(0,1) pairs from the seeded stream.
// Init: the first n_cent points.  Each iteration assigns every point to its
// nearest centroid (squared distance, ties to the lower index) and moves each
// centroid to the mean of its points (an empty cell keeps its centroid).
// Partial sums are formed over fixed blocks of points and combined in block
// order, so the result does not depend on n_threads.  Returns the mean
// squared error per coordinate of the last assignment.  lut_out (optional)
// receives the centroids rounded to fp16, [y0, y1] per entry.
double orc_lloyd_lut(uint64_t seed, uint64_t n_pairs, uint32_t n_cent, uint32_t iters,
                     int n_threads, double* cent_out, uint16_t* lut_out) {
  std::vector<double> pts(2 * n_pairs);
  orc_normal_pairs(seed, 0, n_pairs, pts.data());
  std::vector<double> c(2 * n_cent);
  for (uint32_t j = 0; j < n_cent; ++j) {
    c[2 * j] = pts[2 * j];
    c[2 * j + 1] = pts[2 * j + 1];
  }
  const uint64_t block = 4096;
  const uint64_t nblocks = (n_pairs + block - 1) / block;
  std::vector<double> bsum(nblocks * 2 * n_cent), bdist(nblocks);
  std::vector<uint64_t> bcnt(nblocks * n_cent);
  if (n_threads < 1) n_threads = 1;
  double mse = 0.0;
  for (uint32_t it = 0; it <= iters; ++it) {
    auto work = [&](int tid) {
      for (uint64_t bI = tid; bI < nblocks; bI += n_threads) {
        double* sum = &bsum[bI * 2 * n_cent];
        uint64_t* cnt = &bcnt[bI * n_cent];
        std::fill(sum, sum + 2 * n_cent, 0.0);
        std::fill(cnt, cnt + n_cent, 0);
        double dist = 0.0;
        const uint64_t end = std::min(n_pairs, (bI + 1) * block);
        for (uint64_t i = bI * block; i < end; ++i) {
          const double px = pts[2 * i], py = pts[2 * i + 1];
          uint32_t best = 0;
          double bd = std::numeric_limits<double>::infinity();
          for (uint32_t j = 0; j < n_cent; ++j) {
            const double dx = px - c[2 * j], dy = py - c[2 * j + 1];
            const double dd = dx * dx + dy * dy;
            if (dd < bd) {
              bd = dd;
              best = j;
            }
          }
          sum[2 * best] += px;
          sum[2 * best + 1] += py;
          cnt[best] += 1;
          dist += bd;
        }
        bdist[bI] = dist;
      }
    };
    std::vector<std::thread> th;
    for (int tI = 1; tI < n_threads; ++tI) th.emplace_back(work, tI);
    work(0);
    for (auto& x : th) x.join();
    double total = 0.0;
    for (uint64_t bI = 0; bI < nblocks; ++bI) total += bdist[bI];
    mse = total / (2.0 * (double)n_pairs);
    if (it == iters) break;   // the last pass only measures the distortion
    for (uint32_t j = 0; j < n_cent; ++j) {
      double sx = 0.0, sy = 0.0;
      uint64_t n = 0;
      for (uint64_t bI = 0; bI < nblocks; ++bI) {
        sx += bsum[bI * 2 * n_cent + 2 * j];
        sy += bsum[bI * 2 * n_cent + 2 * j + 1];
        n += bcnt[bI * n_cent + j];
      }
      if (n > 0) {
        c[2 * j] = sx / (double)n;
        c[2 * j + 1] = sy / (double)n;
      }
    }
  }
  if (cent_out) std::memcpy(cent_out, c.data(), sizeof(double) * 2 * n_cent);
  if (lut_out)
    for (uint32_t j = 0; j < 2 * n_cent; ++j) lut_out[j] = double_to_half(c[j]);
  return mse;
}

// Trellis states s_t of one code, t = 0..T-1.
void orc_window_states(const uint8_t* code, uint32_t d, uint32_t k, uint32_t* states) {
  const Geometry g = make_geometry(d, k);
  for (uint32_t t = 0; t < g.T; ++t) states[t] = window_state(code, g, t);
}

// Per-state (hash index, sign) for a list of states.
void orc_state_hash(const uint32_t* states, uint64_t n, uint32_t* idx_out, uint32_t* neg_out) {
  for (uint64_t i = 0; i < n; ++i) {
    const uint32_t s = states[i];
    const uint32_t h = s * s + s;
    idx_out[i] = (h >> 14) & 511u;
    neg_out[i] = (h >> 23) & 1u;
  }
}

// f(c) as exact doubles.
void orc_decode_f(const uint8_t* code, uint32_t d, uint32_t k, const uint16_t* lut, double* f) {
  decode_f(code, make_geometry(d, k), lut, f);
}

// Lookup-decode of n requested rows from AoS records
// [code: d*k/16 bytes][alpha: bf16 little-endian] laid out with stride rec_bytes.
// Output row j (bf16 bits, d per row) is the reconstruction of record idx[j];
// an index outside [0, n_rows) yields a zero row and is counted in the return
// value.  n_threads > 1 splits the lookups into contiguous blocks.
uint64_t orc_lookup_decode(const uint8_t* records, uint64_t n_rows, uint32_t d, uint32_t k,
                           uint64_t rec_bytes, const uint16_t* lut, const int64_t* idx,
                           uint64_t n, uint16_t* out, int n_threads) {
  const Geometry g = make_geometry(d, k);
  const uint64_t code_bytes = (uint64_t)g.Lc / 8;
  if (n_threads < 1) n_threads = 1;
  std::vector<uint64_t> bad(n_threads, 0);
  auto work = [&](int tid) {
    const uint64_t lo = n * tid / n_threads, hi = n * (tid + 1) / n_threads;
    for (uint64_t j = lo; j < hi; ++j) {
      uint16_t* o = out + j * d;
      const int64_t r = idx[j];
      if (r < 0 || (uint64_t)r >= n_rows) {
        std::memset(o, 0, sizeof(uint16_t) * d);
        bad[tid] += 1;
        continue;
      }
      const uint8_t* rec = records + (uint64_t)r * rec_bytes;
      const uint16_t a = (uint16_t)(rec[code_bytes] | (rec[code_bytes + 1] << 8));
      reconstruct_row(rec, a, g, lut, o);
    }
  };
  std::vector<std::thread> th;
  for (int tI = 1; tI < n_threads; ++tI) th.emplace_back(work, tI);
  work(0);
  for (auto& x : th) x.join();
  uint64_t total = 0;
  for (uint64_t b : bad) total += b;
  return total;
}

// Lookup-decode of a table with a bit rate per row (frequency-based bit
// allocation): record r occupies bytes [offsets[r], offsets[r+1]) and its rate
// follows from its length, k_r = (R_r - 2) * 16 / d.  A record whose length
// gives no k in {3, 4, 5, 6} decodes as a zero row and is counted like an
// out-of-range id.  Returns that count.
uint64_t orc_lookup_decode_mixed(const uint8_t* records, const uint64_t* offsets, uint64_t n_rows,
                                 uint32_t d, const uint16_t* lut, const int64_t* idx, uint64_t n,
                                 uint16_t* out) {
  uint64_t bad = 0;
  for (uint64_t j = 0; j < n; ++j) {
    uint16_t* o = out + j * d;
    const int64_t r = idx[j];
    bool ok = r >= 0 && (uint64_t)r < n_rows;
    uint64_t R = 0, k = 0;
    if (ok) {
      R = offsets[r + 1] - offsets[r];
      ok = R >= 2 && ((R - 2) * 16) % d == 0;
      if (ok) k = (R - 2) * 16 / d;
      ok = ok && k >= 3 && k <= 6;
    }
    if (!ok) {
      std::memset(o, 0, sizeof(uint16_t) * d);
      bad += 1;
      continue;
    }
    const Geometry g = make_geometry(d, (uint32_t)k);
    const uint8_t* rec = records + offsets[r];
    const uint64_t cb = R - 2;
    const uint16_t a = (uint16_t)(rec[cb] | (rec[cb + 1] << 8));
    reconstruct_row(rec, a, g, lut, o);
  }
  return bad;
}

// Decode fused with a weighted readout (the pages hand the rows to "the
// existing readout"; this synthetic one sums each group of `group` consecutive
// lookups): out[g][q] = bf16_rne(acc) with acc = 0 (fp32) and, for i in lookup
// order, acc = fmaf(w[g*group + i], float(row_i[q]), acc), where row_i is the
// bf16 row the plain lookup-decode writes (zeros for an out-of-range id) and
// w = 1 when weights is null.  Returns the count of out-of-range ids.
uint64_t orc_lookup_decode_reduce(const uint8_t* records, uint64_t n_rows, uint32_t d, uint32_t k,
                                  uint64_t rec_bytes, const uint16_t* lut, const int64_t* idx,
                                  uint64_t n_groups, uint32_t group, const float* weights,
                                  uint16_t* out, int n_threads) {
  const uint64_t n = n_groups * group;
  std::vector<uint16_t> rows(n * (uint64_t)d);
  const uint64_t bad = orc_lookup_decode(records, n_rows, d, k, rec_bytes, lut, idx, n, rows.data(),
                                         n_threads);
  for (uint64_t g = 0; g < n_groups; ++g) {
    for (uint32_t q = 0; q < d; ++q) {
      float acc = 0.0f;
      for (uint32_t i = 0; i < group; ++i) {
        const uint64_t j = g * group + i;
        const float w = weights ? weights[j] : 1.0f;
        acc = std::fmaf(w, bf16_to_float(rows[j * d + q]), acc);
      }
      out[g * d + q] = float_to_bf16(acc);
    }
  }
  return bad;
}

// D(c) for a code against a normalised row z.
double orc_distortion(const double* z, const uint8_t* code, uint32_t d, uint32_t k,
                      const uint16_t* lut) {
  const Geometry g = make_geometry(d, k);
  const StateTable st = make_state_table(lut);
  return distortion(code, g, st, z);
}

// Search modes for orc_encode_z.
enum { ORC_BRUTE = 0, ORC_EXACT = 1, ORC_TWO_PASS = 2 };

// Best code for a normalised row z under the given mode; returns its cost, or
// -1 when the mode does not apply to this geometry.
double orc_encode_z(const double* z, uint32_t d, uint32_t k, const uint16_t* lut, int mode,
                    uint8_t* code_out) {
  const Geometry g = make_geometry(d, k);
  const StateTable st = make_state_table(lut);
  if (mode == ORC_BRUTE) {
    if (g.Lc > 26) return -1.0;
    return brute_force(z, g, st, code_out);
  }
  if (g.Lc < (uint32_t)kStateBits) return -1.0;
  if (mode == ORC_EXACT) return viterbi_exact(z, g, st, code_out);
  if (mode == ORC_TWO_PASS) return viterbi_two_pass(z, g, st, code_out);
  return -1.0;
}

// Offline compression of rows e (fp64, rows x d) into AoS records
// [code][alpha bf16] [P4 how it differs]:
//   z = sqrt(d) e / |e|; code = search(z); alpha = |e| / |f(code)| (fp64),
//   stored as bf16 (one rounding).  A zero row gets an all-zero code and
//   alpha = 0.  alpha_exact / cost (optional) receive the pre-rounding alpha
//   and the search cost per row.  Rows are split across n_threads.
int orc_encode_rows(const double* e, uint64_t rows, uint32_t d, uint32_t k, const uint16_t* lut,
                    int mode, int n_threads, uint8_t* records, double* alpha_exact,
                    double* cost) {
  const Geometry g = make_geometry(d, k);
  if (g.Lc % 8 != 0) return -1;
  const uint64_t code_bytes = g.Lc / 8;
  const uint64_t rec_bytes = code_bytes + 2;
  const StateTable st = make_state_table(lut);
  if (n_threads < 1) n_threads = 1;
  std::vector<int> fail(n_threads, 0);
  auto work = [&](int tid) {
    std::vector<double> z(d), f(d);
    for (uint64_t r = tid; r < rows; r += n_threads) {
      const double* er = e + r * d;
      uint8_t* rec = records + r * rec_bytes;
      double ss = 0.0;
      for (uint32_t q = 0; q < d; ++q) ss = ss + er[q] * er[q];
      const double nrm = std::sqrt(ss);
      if (nrm == 0.0) {
        std::memset(rec, 0, rec_bytes);
        if (alpha_exact) alpha_exact[r] = 0.0;
        if (cost) cost[r] = 0.0;
        continue;
      }
      const double sc = std::sqrt((double)d) / nrm;
      for (uint32_t q = 0; q < d; ++q) z[q] = er[q] * sc;
      double c;
      if (mode == ORC_BRUTE) c = (g.Lc <= 26) ? brute_force(z.data(), g, st, rec) : -1.0;
      else if (mode == ORC_EXACT) c = viterbi_exact(z.data(), g, st, rec);
      else c = viterbi_two_pass(z.data(), g, st, rec);
      if (c < 0.0) {
        fail[tid] = 1;
        continue;
      }
      decode_f(rec, g, lut, f.data());
      double fs = 0.0;
      for (uint32_t q = 0; q < d; ++q) fs = fs + f[q] * f[q];
      const double alpha = nrm / std::sqrt(fs);
      const uint16_t ab = double_to_bf16(alpha);
      rec[code_bytes] = (uint8_t)(ab & 0xff);
      rec[code_bytes + 1] = (uint8_t)(ab >> 8);
      if (alpha_exact) alpha_exact[r] = alpha;
      if (cost) cost[r] = c;
    }
  };
  std::vector<std::thread> th;
  for (int tI = 1; tI < n_threads; ++tI) th.emplace_back(work, tI);
  work(0);
  for (auto& x : th) x.join();
  for (int f : fail)
    if (f) return -1;
  return 0;
}

// fp32 encoder entry points (see the fp32 variant above).
float orc_distortion_f32(const float* z, const uint8_t* code, uint32_t d, uint32_t k,
                         const uint16_t* lut) {
  const Geometry g = make_geometry(d, k);
  const StateTableF st = make_state_table_f(lut);
  return distortion_f(code, g, st, z);
}

float orc_encode_z_f32(const float* z, uint32_t d, uint32_t k, const uint16_t* lut, int mode,
                       uint8_t* code_out) {
  const Geometry g = make_geometry(d, k);
  const StateTableF st = make_state_table_f(lut);
  if (mode == ORC_BRUTE) return g.Lc > 26 ? -1.0f : brute_force_f(z, g, st, code_out);
  if (g.Lc < (uint32_t)kStateBits) return -1.0f;
  if (mode == ORC_EXACT) return viterbi_exact_f(z, g, st, code_out);
  return viterbi_two_pass_f(z, g, st, code_out);
}

// Rows e (fp32 values, rows x d) -> AoS records with the fp32 two-pass search:
// ss = sum e^2 (fp64, index order), nrm = sqrt(ss), z = (float)(e * (sqrt(d) / nrm));
// alpha = nrm / sqrt(sum f^2) (fp64, index order) rounded once to bf16; a zero
// row gets an all-zero code and alpha = 0.  cost (optional) receives the fp32
// path metric.
float orc_free_start_f(const float* z, uint32_t d, uint32_t k, const uint16_t* lut, uint32_t rho,
                       uint32_t* states) {
  return free_start_f(z, make_geometry(d, k), make_state_table_f(lut), rho, states);
}

float orc_free_start_brute_f(const float* z, uint32_t d, uint32_t k, const uint16_t* lut,
                             uint32_t rho, uint32_t* states) {
  return free_start_brute_f(z, make_geometry(d, k), make_state_table_f(lut), rho, states);
}

int orc_encode_rows_f32(const float* e, uint64_t rows, uint32_t d, uint32_t k, const uint16_t* lut,
                        int n_threads, uint8_t* records, float* cost) {
  const Geometry g = make_geometry(d, k);
  if (g.Lc % 8 != 0 || g.Lc < (uint32_t)kStateBits) return -1;
  const uint64_t code_bytes = g.Lc / 8, rec_bytes = code_bytes + 2;
  const StateTableF st = make_state_table_f(lut);
  if (n_threads < 1) n_threads = 1;
  auto work = [&](int tid) {
    std::vector<float> z(d);
    std::vector<double> f(d);
    for (uint64_t r = tid; r < rows; r += n_threads) {
      const float* er = e + r * d;
      uint8_t* rec = records + r * rec_bytes;
      double ss = 0.0;
      for (uint32_t q = 0; q < d; ++q) ss = ss + (double)er[q] * (double)er[q];
      const double nrm = std::sqrt(ss);
      if (nrm == 0.0) {
        std::memset(rec, 0, rec_bytes);
        if (cost) cost[r] = 0.0f;
        continue;
      }
      const double sc = std::sqrt((double)d) / nrm;
      for (uint32_t q = 0; q < d; ++q) z[q] = (float)((double)er[q] * sc);
      const float c = viterbi_two_pass_f(z.data(), g, st, rec);
      decode_f(rec, g, lut, f.data());
      double fs = 0.0;
      for (uint32_t q = 0; q < d; ++q) fs = fs + f[q] * f[q];
      const uint16_t ab = double_to_bf16(nrm / std::sqrt(fs));
      rec[code_bytes] = (uint8_t)(ab & 0xff);
      rec[code_bytes + 1] = (uint8_t)(ab >> 8);
      if (cost) cost[r] = c;
    }
  };
  std::vector<std::thread> th;
  for (int tI = 1; tI < n_threads; ++tI) th.emplace_back(work, tI);
  work(0);
  for (auto& x : th) x.join();
  return 0;
}

// Two-bit round-to-nearest baseline for one row (the pages do not define it;
// this is the reading used here): a symmetric 4-level midrise grid
// {-3D/2, -D/2, D/2, 3D/2}.  variant 0: D = bf16(absmax / 1.5); variant 1: D
// from a 4000-point search over (0, 2 absmax / 1.5] minimising the row's
// squared error.  ehat receives the reconstruction.
void orc_rtn2(const double* e, uint32_t d, int variant, double* ehat) {
  double amax = 0.0;
  for (uint32_t q = 0; q < d; ++q) amax = std::max(amax, std::fabs(e[q]));
  auto quant = [&](double D, double x) {
    double lvl = std::floor(x / D);
    if (lvl < -2.0) lvl = -2.0;
    if (lvl > 1.0) lvl = 1.0;
    return D * (lvl + 0.5);
  };
  double D = (double)bf16_to_float(double_to_bf16(amax / 1.5));
  if (variant == 1 && amax > 0.0) {
    double best = std::numeric_limits<double>::infinity();
    for (int i = 1; i <= 4000; ++i) {
      const double Dc = (double)bf16_to_float(double_to_bf16(2.0 * amax / 1.5 * i / 4000.0));
      double err = 0.0;
      for (uint32_t q = 0; q < d; ++q) {
        const double r = e[q] - quant(Dc, e[q]);
        err = err + r * r;
      }
      if (err < best) {
        best = err;
        D = Dc;
      }
    }
  }
  for (uint32_t q = 0; q < d; ++q) ehat[q] = (D > 0.0) ? quant(D, e[q]) : 0.0;
}

}  // extern "C"

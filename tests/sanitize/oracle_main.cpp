// Drives the oracle's entry points on small inputs (decode, lookup-decode with
// out-of-range ids, mixed rates, fused readout, exact and two-pass encoders in
// fp64 and fp32, the Lloyd LUT, RTN), built together with oracle/cp_oracle.cpp
// under -fsanitize=address,undefined by tests/test_sanitizers.py.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

extern "C" {
uint64_t orc_splitmix64(uint64_t x);
void orc_normal_pairs(uint64_t seed, uint64_t first, uint64_t count, double* out);
double orc_lloyd_lut(uint64_t seed, uint64_t n_pairs, uint32_t n_cent, uint32_t iters,
                     int n_threads, double* cent_out, uint16_t* lut_out);
void orc_window_states(const uint8_t* code, uint32_t d, uint32_t k, uint32_t* states);
void orc_decode_f(const uint8_t* code, uint32_t d, uint32_t k, const uint16_t* lut, double* f);
uint64_t orc_lookup_decode(const uint8_t* records, uint64_t n_rows, uint32_t d, uint32_t k,
                           uint64_t rec_bytes, const uint16_t* lut, const int64_t* idx,
                           uint64_t n, uint16_t* out, int n_threads);
uint64_t orc_lookup_decode_mixed(const uint8_t* records, const uint64_t* offsets, uint64_t n_rows,
                                 uint32_t d, const uint16_t* lut, const int64_t* idx, uint64_t n,
                                 uint16_t* out);
uint64_t orc_lookup_decode_reduce(const uint8_t* records, uint64_t n_rows, uint32_t d, uint32_t k,
                                  uint64_t rec_bytes, const uint16_t* lut, const int64_t* idx,
                                  uint64_t n_groups, uint32_t group, const float* weights,
                                  uint16_t* out, int n_threads);
double orc_encode_z(const double* z, uint32_t d, uint32_t k, const uint16_t* lut, int mode,
                    uint8_t* code_out);
int orc_encode_rows(const double* e, uint64_t rows, uint32_t d, uint32_t k, const uint16_t* lut,
                    int mode, int n_threads, uint8_t* records, double* alpha_exact, double* cost);
int orc_encode_rows_f32(const float* e, uint64_t rows, uint32_t d, uint32_t k, const uint16_t* lut,
                        int n_threads, uint8_t* records, float* cost);
float orc_encode_z_f32(const float* z, uint32_t d, uint32_t k, const uint16_t* lut, int mode,
                       uint8_t* code_out);
void orc_rtn2(const double* e, uint32_t d, int variant, double* ehat);
}

static uint8_t byte_at(uint64_t seed, uint64_t i) { return orc_splitmix64(seed * 1000003u + i) & 0xFF; }

int main() {
  // a small LUT from a short Lloyd run (also exercises the k-means)
  std::vector<double> cent(1024);
  std::vector<uint16_t> lut(1024);
  orc_lloyd_lut(7, 1u << 12, 512, 2, 2, cent.data(), lut.data());

  // lookup-decode, every rate, rows with ids out of range
  for (uint32_t k = 3; k <= 6; ++k)
    for (uint32_t d : {8u, 16u, 256u, 1024u}) {
      if ((d * k) % 32) continue;
      const uint64_t R = d * k / 16 + 2, n_rows = 37;
      std::vector<uint8_t> rec(n_rows * R);
      for (uint64_t i = 0; i < rec.size(); ++i) rec[i] = byte_at(k * 131 + d, i);
      std::vector<int64_t> idx = {0, 36, -1, 37, 5, 5, 1ll << 40, 20};
      std::vector<uint16_t> out(idx.size() * d);
      const uint64_t bad = orc_lookup_decode(rec.data(), n_rows, d, k, R, lut.data(), idx.data(),
                                             idx.size(), out.data(), 3);
      if (bad != 3) return 2;
      std::vector<uint32_t> st(d / 2);
      orc_window_states(rec.data(), d, k, st.data());
      std::vector<double> f(d);
      orc_decode_f(rec.data(), d, k, lut.data(), f.data());
      std::vector<float> w(8 * 2, 0.5f);
      std::vector<int64_t> gidx = {0, 1, 2, -4, 3, 36, 35, 40};
      std::vector<uint16_t> red(2 * d);
      orc_lookup_decode_reduce(rec.data(), n_rows, d, k, R, lut.data(), gidx.data(), 2, 4,
                               w.data(), red.data(), 2);
    }
  // mixed rates: rows of k = 3..6 at d = 64
  {
    const uint32_t d = 64;
    std::vector<uint64_t> off = {0};
    std::vector<uint8_t> rec;
    for (uint32_t r = 0; r < 12; ++r) {
      const uint32_t k = 3 + r % 4, R = d * k / 16 + 2;
      for (uint32_t i = 0; i < R; ++i) rec.push_back(byte_at(r, i));
      off.push_back(off.back() + R);
    }
    std::vector<int64_t> idx = {0, 11, 3, -2, 12, 7};
    std::vector<uint16_t> out(idx.size() * d);
    if (orc_lookup_decode_mixed(rec.data(), off.data(), 12, d, lut.data(), idx.data(), idx.size(),
                                out.data()) != 2)
      return 3;
  }
  // encoders: brute force and exact at d = 8, two-pass at d = 16 (fp64), and the
  // fp32 encoder (the exact search at d = 16 takes minutes under the sanitizers)
  for (uint32_t d : {8u, 16u}) {
    std::vector<double> z(d);
    std::vector<double> pr(d);
    orc_normal_pairs(3, 0, d / 2, pr.data());
    for (uint32_t q = 0; q < d; ++q) z[q] = pr[q];
    std::vector<uint8_t> code(d * 6 / 16 + 2);
    for (int mode = 0; mode <= 2; ++mode) {
      if (d > 8 && mode != 2) continue;
      if (d == 8 && mode == 2) continue;
      orc_encode_z(z.data(), d, 4, lut.data(), mode, code.data());
    }
    std::vector<float> zf(z.begin(), z.end());
    orc_encode_z_f32(zf.data(), d, 4, lut.data(), d == 8 ? 1 : 2, code.data());
  }
  {
    const uint32_t d = 32, rows = 3;
    std::vector<double> e(rows * d);
    orc_normal_pairs(5, 0, rows * d / 2, e.data());
    std::memset(e.data() + d, 0, d * sizeof(double));            // a zero row
    std::vector<uint8_t> rec(rows * (d * 4 / 16 + 2));
    std::vector<double> ae(rows), cost(rows);
    if (orc_encode_rows(e.data(), rows, d, 4, lut.data(), 2, 2, rec.data(), ae.data(),
                        cost.data()) != 0)
      return 4;
    std::vector<float> ef(e.begin(), e.end()), cf(rows);
    if (orc_encode_rows_f32(ef.data(), rows, d, 4, lut.data(), 2, rec.data(), cf.data()) != 0)
      return 5;
    std::vector<double> eh(d);
    orc_rtn2(e.data(), d, 0, eh.data());
    orc_rtn2(e.data(), d, 1, eh.data());
  }
  std::printf("oracle ok\n");
  return 0;
}

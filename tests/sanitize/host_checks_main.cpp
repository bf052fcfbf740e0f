// Runs libcp's host-side geometry and argument checks (cp_geometry.h) over the
// ranges the C ABI accepts and a margin beyond them, built with
// -fsanitize=address,undefined by tests/test_sanitizers.py.  Exit code 0 and no
// sanitizer report means the arithmetic stayed in range.
#include <cstdio>
#include <cstdint>
#include <cstdlib>

#include "cp_geometry.h"

static int fails = 0;
#define CHECK(c)                                                  \
  do {                                                            \
    if (!(c)) {                                                   \
      std::fprintf(stderr, "check failed: %s (line %d)\n", #c, __LINE__); \
      ++fails;                                                    \
    }                                                             \
  } while (0)

int main() {
  // geometry: accepted exactly when k in 3..6, d % 8 == 0 in [8, 4096], d*k % 32 == 0
  for (uint32_t k = 0; k <= 9; ++k)
    for (uint32_t d = 0; d <= 8200; ++d) {
      const bool ok = cpx::geometry_ok(d, k);
      const bool want = k >= 3 && k <= 6 && d >= 8 && d <= 4096 && d % 8 == 0 && (d * k) % 32 == 0;
      CHECK(ok == want);
      if (ok) {
        const uint32_t S = cpx::soa_stride(d, k);
        CHECK(S % 16 == 0 && S >= d * k / 16 && S < d * k / 16 + 16);
        uint32_t slot = 0;
        const uint32_t sb = cpx::stage_bytes_for(16, d * k / 16, S, false, &slot);
        CHECK(sb % 16 == 0 && sb >= 16 + d * k / 16 + 2 + 14 + 16);
        const uint32_t sbs = cpx::stage_bytes_for(16, d * k / 16, S, true, &slot);
        CHECK(slot + 4 <= sbs);
      }
    }
  CHECK(!cpx::geometry_ok(0xFFFFFFFFu, 4) && !cpx::geometry_ok(1024, 0xFFFFFFFFu));
  // buckets: every row id maps into [0, nb), nb <= 4096, for table sizes up to 2^40
  const uint64_t sizes[] = {1, 2, 3, 7, 4095, 4096, 4097, 65536, 1ull << 24, 198000000ull,
                            (1ull << 32) + 5, cpx::kMaxRows};
  for (uint64_t n_rows : sizes) {
    uint32_t shift = 0, nb = 0;
    cpx::bucket_params(n_rows, &shift, &nb);
    CHECK(nb >= 1 && nb <= (1u << cpx::kBucketBitsHost));
    CHECK(((n_rows - 1) >> shift) == nb - 1);
    CHECK(shift < 64);
  }
  CHECK(cpx::host_scratch_count_words(4096) == 4160);
  CHECK(cpx::host_scratch_count_words(4095) == 4160);   // 4,096 ranges + the ticket word
  CHECK(cpx::host_scratch_count_words(4030) == 4032);
  CHECK(cpx::host_scratch_bytes(1u << 20, 4096) == (2 * 4160 + 2 * (1u << 20)) * 4);
  alignas(16) unsigned char buf[32];
  CHECK(cpx::aligned(buf, 16) && !cpx::aligned(buf + 2, 16) && cpx::aligned(buf + 2, 2));
  if (fails) return 1;
  std::printf("host checks ok\n");
  return 0;
}

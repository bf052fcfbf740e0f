// Instantiations of the lookup-decode kernel for k = 4 bits per trellis step.
#include "cp_kernels.cuh"
#include "cp_dispatch.h"

namespace cpk {

namespace {
template <bool SOA, int PF, bool PERM>
void fill(DecodeFn* row) {
  row[0] = &lookup_decode_kernel<4, SOA, PF, 0, PERM>;
  row[1] = &lookup_decode_kernel<4, SOA, PF, 1, PERM>;
  row[2] = &lookup_decode_kernel<4, SOA, PF, 2, PERM>;
  row[3] = &lookup_decode_kernel<4, SOA, PF, 4, PERM>;
  row[4] = &lookup_decode_kernel<4, SOA, PF, 8, PERM>;
  row[5] = &lookup_decode_kernel<4, SOA, PF, 16, PERM>;
}
}  // namespace

KernelSet kernels_k4() {
  KernelSet s;
  fill<false, kPfDevice, false>(s.dev[0]);
  fill<true, kPfDevice, false>(s.dev[1]);
  fill<false, kPfHost, true>(s.host[0]);
  fill<true, kPfHost, true>(s.host[1]);
  return s;
}

}  // namespace cpk

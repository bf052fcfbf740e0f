// Instantiations of the lookup-decode kernel for k = 6 bits per trellis step.
#include "cp_kernels.cuh"
#include "cp_dispatch.h"

namespace cpk {

KernelSet kernels_k6() {
  KernelSet s;
  s.aos_dev = &lookup_decode_kernel<6, false, kPfDevice>;
  s.soa_dev = &lookup_decode_kernel<6, true, kPfDevice>;
  s.aos_host = &lookup_decode_kernel<6, false, kPfHost>;
  s.soa_host = &lookup_decode_kernel<6, true, kPfHost>;
  return s;
}

}  // namespace cpk

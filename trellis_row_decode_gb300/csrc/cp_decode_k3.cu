// Instantiations of the lookup-decode kernel for k = 3 bits per trellis step.
#include "cp_kernels.cuh"
#include "cp_dispatch.h"

namespace cpk {

KernelSet kernels_k3() {
  KernelSet s;
  s.aos_dev = &lookup_decode_kernel<3, false, kPfDevice>;
  s.soa_dev = &lookup_decode_kernel<3, true, kPfDevice>;
  s.aos_host = &lookup_decode_kernel<3, false, kPfHost>;
  s.soa_host = &lookup_decode_kernel<3, true, kPfHost>;
  return s;
}

}  // namespace cpk

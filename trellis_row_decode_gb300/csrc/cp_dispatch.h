// cp_dispatch.h -- kernel table shared by the instantiation units and the C ABI.
#pragma once

#include "cp_kernels.cuh"

namespace cpk {

// Stages of the per-warp record ring: one row ahead for HBM-resident tables,
// more rows in flight for tables read over the host link (higher latency).
constexpr int kPfDevice = 2;
constexpr int kPfHost = 8;

using DecodeFn = void (*)(DecodeParams);

struct KernelSet {
  DecodeFn aos_dev;
  DecodeFn soa_dev;
  DecodeFn aos_host;
  DecodeFn soa_host;
};

KernelSet kernels_k3();
KernelSet kernels_k4();
KernelSet kernels_k5();
KernelSet kernels_k6();

}  // namespace cpk

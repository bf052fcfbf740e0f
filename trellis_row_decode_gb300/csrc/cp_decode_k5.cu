// Instantiations of the lookup-decode kernel for k = 5 bits per trellis step.
#include "cp_kernels.cuh"
#include "cp_dispatch.h"

namespace cpk {

namespace {
// row[i]: chunks-per-lane index i
template <bool SOA, int PF, bool PERM, int REP>
void fill(DecodeFn* row) {
  row[0] = &lookup_decode_kernel<5, SOA, PF, 0, PERM, REP>;
  row[1] = &lookup_decode_kernel<5, SOA, PF, 1, PERM, REP>;
  row[2] = &lookup_decode_kernel<5, SOA, PF, 2, PERM, REP>;
  row[3] = &lookup_decode_kernel<5, SOA, PF, 4, PERM, REP>;
  row[4] = &lookup_decode_kernel<5, SOA, PF, 8, PERM, REP>;
  row[5] = &lookup_decode_kernel<5, SOA, PF, 16, PERM, REP>;
}

template <bool SOA>
void fill_block(DecodeFn* row) {
  row[0] = &lookup_decode_block_kernel<5, SOA, 0, kLutRepBlock, kBlkRows>;
  row[1] = &lookup_decode_block_kernel<5, SOA, 1, block_rep(1), block_rows(1)>;
  row[2] = &lookup_decode_block_kernel<5, SOA, 2, block_rep(2), block_rows(2)>;
  row[3] = &lookup_decode_block_kernel<5, SOA, 4, kLutRepBlock, kBlkRows>;
  row[4] = &lookup_decode_block_kernel<5, SOA, 8, kLutRepBlock, kBlkRows>;
  row[5] = &lookup_decode_block_kernel<5, SOA, 16, kLutRepBlock, kBlkRows>;
}
}  // namespace

KernelSet kernels_k5() {
  KernelSet s;
  fill_block<false>(s.dev[0]);
  fill_block<true>(s.dev[1]);
  fill<false, kPfHost, true, kLutRepHost>(s.host[0]);
  fill<true, kPfHost, true, kLutRepHost>(s.host[1]);
  s.host[0][1] = &lookup_decode_host_kernel<5, false, kPfHostReg, 1, kLutRepHostReg>;
  s.host[0][2] = &lookup_decode_host_kernel<5, false, kPfHostReg, 2, kLutRepHostReg>;
  s.host[0][3] = &lookup_decode_host_kernel<5, false, kPfHostReg, 4, kLutRepHostReg>;
  s.host[1][1] = &lookup_decode_host_kernel<5, true, kPfHostReg, 1, kLutRepHostReg>;
  s.host[1][2] = &lookup_decode_host_kernel<5, true, kPfHostReg, 2, kLutRepHostReg>;
  s.host[1][3] = &lookup_decode_host_kernel<5, true, kPfHostReg, 4, kLutRepHostReg>;
  s.reduce[0][0] = &lookup_decode_reduce_kernel<5, false, kPfReduce, 1>;
  s.reduce[0][1] = &lookup_decode_reduce_kernel<5, false, kPfReduce, 2>;
  s.reduce[0][2] = &lookup_decode_reduce_kernel<5, false, kPfReduce, 4>;
  s.reduce[1][0] = &lookup_decode_reduce_kernel<5, true, kPfReduce, 1>;
  s.reduce[1][1] = &lookup_decode_reduce_kernel<5, true, kPfReduce, 2>;
  s.reduce[1][2] = &lookup_decode_reduce_kernel<5, true, kPfReduce, 4>;
  return s;
}

}  // namespace cpk

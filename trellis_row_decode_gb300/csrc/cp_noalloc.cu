// cp_noalloc.cu -- host-resident lookup-decode that allocates nothing.
//
// Some callers cannot allocate device memory: a serving runtime whose device
// memory is owned by one pool allocator (a plugin may not call cudaMalloc
// behind its back), code running while allocations would stall other streams
// (cudaMalloc/cudaFree can synchronise the device), or a runtime that forbids
// allocations once it has sized its memory budget.  cp_table_load allocates
// (LUT copy, status word, 32 MB of scratch for host-resident tables), so those
// callers use cp_lookup_decode_host_noalloc instead: it takes the records, the
// LUT, the ids, the output and a status word from the caller, and keeps its own
// scratch (LUT copy, range counts and cursors, visiting order) in one
// file-scope device array, sized for at most kNoAllocMaxLookups lookups per call.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "cp.h"
#include "cp_internal.h"

namespace {

constexpr uint32_t kNoAllocMaxLookups = 1u << 16;
constexpr uint32_t kNoAllocMaxBuckets = 1u << cpk::kBucketBits;
constexpr size_t kLutDevBytes = 512 * sizeof(uint32_t);
constexpr size_t kNoAllocScratchBytes =
    kLutDevBytes + cpx::host_scratch_bytes(kNoAllocMaxLookups, kNoAllocMaxBuckets);

// About 0.5 MB on every GPU that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
unsigned char* g_scratch_addr[kMaxDevices];   // device address of the array, per device

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the host-side name of the array is not a device address).  The
// same set-up clears the range counts, which every call then leaves at zero.
cp_status scratch_for_device(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) {
    cpx::set_error("device ordinal outside the supported range");
    return CP_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cpx::cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    e = cudaMemset(static_cast<unsigned char*>(p) + kLutDevBytes, 0,
                   cpx::host_scratch_count_words(kNoAllocMaxBuckets) * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cpx::cuda_fail(e, "no-alloc scratch clear");
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_scratch_addr[dev];
  return CP_OK;
}

}  // namespace

extern "C" cp_status cp_lookup_decode_host_noalloc(const void* records, uint64_t n_rows,
                                                   uint32_t d, uint32_t bits_per_step,
                                                   const uint16_t* lut_fp16, const int64_t* idx,
                                                   uint64_t n, uint16_t* out, uint32_t* status,
                                                   void* stream) {
  if (records == nullptr || lut_fp16 == nullptr || n_rows == 0 || n_rows > cpx::kMaxRows ||
      !cpx::geometry_ok(d, bits_per_step) || !cpx::aligned(records, 16)) {
    cpx::set_error("bad records pointer/alignment, LUT pointer or geometry");
    return CP_ERR_INVALID_ARG;
  }
  if (n == 0) return CP_OK;
  if (n > kNoAllocMaxLookups) {
    cpx::set_error("more than 65536 lookups in one call: the static scratch of "
                   "cp_lookup_decode_host_noalloc holds one pass of at most 65536");
    return CP_ERR_INVALID_ARG;
  }
  if (idx == nullptr || out == nullptr || status == nullptr || !cpx::aligned(idx, 8) ||
      !cpx::aligned(out, 16) || !cpx::aligned(status, 4)) {
    cpx::set_error("bad ids/output/status pointer or alignment");
    return CP_ERR_INVALID_ARG;
  }
  for (int i = 0; i < 1024; ++i) {
    if ((lut_fp16[i] & 0x7c00u) == 0x7c00u) {
      cpx::set_error("LUT holds a non-finite fp16 value");
      return CP_ERR_FORMAT;
    }
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cpx::cuda_fail(e, "cudaGetDevice");
  unsigned char* scratch = nullptr;
  cp_status st = scratch_for_device(dev, &scratch);
  if (st != CP_OK) return st;

  void* dptr = nullptr;
  e = cudaHostGetDevicePointer(&dptr, const_cast<void*>(records), 0);
  if (e != cudaSuccess) return cpx::cuda_fail(e, "records are not page-locked host memory");
  if (!cpx::aligned(dptr, 16)) {
    cpx::set_error("device alias of the host table is not 16-byte aligned");
    return CP_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = cudaMemcpyAsync(scratch, lut_fp16, 2048, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cpx::cuda_fail(e, "LUT upload");

  cp_table t{};                                         // a view, on the stack
  t.device = dev;
  t.residency = CP_RESIDENT_HOST;
  t.layout = CP_LAYOUT_AOS;
  t.n_rows = n_rows;
  t.d = d;
  t.k = bits_per_step;
  t.code_bytes = d * bits_per_step / 16;
  t.rec_bytes = t.code_bytes + 2;
  t.soa_stride = cpx::soa_stride(d, bits_per_step);
  t.rec = static_cast<const uint8_t*>(dptr);
  t.lut_dev = reinterpret_cast<uint32_t*>(scratch);
  t.status_dev = status;
  t.scratch_dev = scratch + kLutDevBytes;
  cpx::bucket_params(n_rows, &t.bucket_shift, &t.bucket_nb);
  t.kernels = cpx::kernels_for(bits_per_step);
  cudaDeviceGetAttribute(&t.sm_count, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&t.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  // laid out for the largest bucket count, so that the counts (zero between
  // calls) never overlap the cursors of a call on a table with fewer ranges
  const cpx::HostScratch hs =
      cpx::host_scratch_layout(t.scratch_dev, kNoAllocMaxLookups, kNoAllocMaxBuckets);
  return cpx::launch_decode(&t, idx, n, out, s, true, &hs);
}

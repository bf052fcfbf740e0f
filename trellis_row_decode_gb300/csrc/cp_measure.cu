// cp_measure.cu -- read kernels that measure the bandwidth bounding a
// lookup-decode: a streaming read over the host link for a pinned host buffer
// read zero-copy (or from HBM for a device buffer), and a read of scattered
// whole records, the host path's own access pattern without its decode.
#include <cstdint>

#include <cuda_runtime.h>

#include "cp.h"
#include "cp_internal.h"

namespace {

// Written only when the XOR of everything read equals a value no real buffer is
// expected to give; it keeps the loads from being optimised away.
__device__ unsigned long long g_measure_sink;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Grid-stride read of n16 16-byte words, four loads in flight per thread.
__global__ void __launch_bounds__(256) stream_read_kernel(const uint4* __restrict__ p,
                                                          uint64_t n16) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = ld_stream(p + i);
    const uint4 b = ld_stream(p + i + stride);
    const uint4 c = ld_stream(p + i + 2 * stride);
    const uint4 d = ld_stream(p + i + 3 * stride);
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^
           d.z ^ d.w;
  }
  for (; i < n16; i += stride) {
    const uint4 a = ld_stream(p + i);
    acc ^= a.x ^ a.y ^ a.z ^ a.w;
  }
  if (acc == 0x9E3779B9u) g_measure_sink = acc;
}

// Each listed record read once as the 16-byte pieces that cover it (the host
// path's loads), one CTA per SM taking a contiguous slice of the list, each warp
// four records in flight; pieces that would reach past the table are skipped.
__global__ void __launch_bounds__(1024, 1)
    record_read_kernel(const uint8_t* __restrict__ table, uint64_t table_bytes, uint32_t R,
                       const int64_t* __restrict__ rows, uint64_t n) {
  constexpr int kInFlight = 4;
  const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const uint64_t lo = static_cast<uint64_t>(blockIdx.x) * n / gridDim.x;
  const uint64_t hi = static_cast<uint64_t>(blockIdx.x + 1) * n / gridDim.x;
  const uintptr_t base = reinterpret_cast<uintptr_t>(table);
  uint32_t acc = 0;
  for (uint64_t q = lo + warp; q < hi; q += static_cast<uint64_t>(nw) * kInFlight) {
    uint4 v[kInFlight];
#pragma unroll
    for (int s = 0; s < kInFlight; ++s) {
      v[s] = make_uint4(0, 0, 0, 0);
      const uint64_t qq = q + static_cast<uint64_t>(s) * nw;
      if (qq < hi) {
        const uint64_t r = static_cast<uint64_t>(__ldg(rows + qq));
        const uint64_t off = r * R;
        if (r < table_bytes / R) {
          const uint64_t o0 = off & ~static_cast<uint64_t>(15);
          const uint32_t nch = static_cast<uint32_t>(off - o0 + R + 15) >> 4;
          const uint64_t po = o0 + 16u * lane;
          if (lane < nch && po + 16 <= table_bytes) v[s] = ld_stream(reinterpret_cast<const uint4*>(base + po));
        }
      }
    }
#pragma unroll
    for (int s = 0; s < kInFlight; ++s) acc ^= v[s].x ^ v[s].y ^ v[s].z ^ v[s].w;
  }
  if (acc == 0x9E3779B9u) g_measure_sink = acc;
}

// Device address of buf: itself for device memory, its alias for mapped
// page-locked host memory, nullptr otherwise.
const void* device_view(const void* buf, cudaError_t* err) {
  cudaPointerAttributes attr{};
  *err = cudaPointerGetAttributes(&attr, buf);
  if (*err != cudaSuccess) return nullptr;
  if (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged) return buf;
  if (attr.type == cudaMemoryTypeHost && attr.devicePointer != nullptr) return attr.devicePointer;
  return nullptr;
}

}  // namespace

extern "C" cp_status cp_measure_record_read(const void* table, uint64_t table_bytes,
                                            uint32_t record_bytes, const int64_t* rows,
                                            uint64_t n, void* stream) {
  if (table == nullptr || rows == nullptr || record_bytes == 0 || n == 0 || n >= (1ull << 48) ||
      table_bytes < record_bytes || !cpx::aligned(table, 16) || !cpx::aligned(rows, 8)) {
    cpx::set_error("table and rows must be non-null (16- and 8-byte aligned), n in [1, 2^48), "
                   "record_bytes positive, table_bytes at least one record");
    return CP_ERR_INVALID_ARG;
  }
  cudaError_t e = cudaSuccess;
  const void* dptr = device_view(table, &e);
  if (e != cudaSuccess) return cpx::cuda_fail(e, "cudaPointerGetAttributes");
  if (dptr == nullptr) {
    cpx::set_error("table is neither device memory nor mapped page-locked host memory");
    return CP_ERR_INVALID_ARG;
  }
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cpx::cuda_fail(e, "device query");
  uint64_t blocks = static_cast<uint64_t>(sms);
  if (blocks > n) blocks = n;
  record_read_kernel<<<static_cast<unsigned>(blocks), 1024, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(dptr), table_bytes, record_bytes, rows, n);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cpx::cuda_fail(e, "record-read launch");
  return CP_OK;
}

extern "C" cp_status cp_measure_stream_read(const void* buf, uint64_t bytes, void* stream) {
  if (buf == nullptr || bytes == 0 || (bytes % 16) != 0 || !cpx::aligned(buf, 16)) {
    cpx::set_error("buffer must be non-null and 16-byte aligned, bytes a positive multiple of 16");
    return CP_ERR_INVALID_ARG;
  }
  cudaError_t e = cudaSuccess;
  const void* dptr = device_view(buf, &e);
  if (e != cudaSuccess) return cpx::cuda_fail(e, "cudaPointerGetAttributes");
  if (dptr == nullptr) {
    cpx::set_error("buffer is neither device memory nor mapped page-locked host memory");
    return CP_ERR_INVALID_ARG;
  }
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cpx::cuda_fail(e, "device query");
  // 8 CTAs of 256 threads per SM: 2048 threads x 4 loads x 16 B = 128 KB in flight per SM
  const uint64_t n16 = bytes / 16;
  uint64_t blocks = static_cast<uint64_t>(sms) * 8;
  const uint64_t need = (n16 + 255) / 256;
  if (blocks > need) blocks = need;
  stream_read_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(dptr), n16);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cpx::cuda_fail(e, "stream-read launch");
  return CP_OK;
}

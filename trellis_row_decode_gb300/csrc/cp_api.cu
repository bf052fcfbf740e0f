// cp_api.cu -- host side of libcp: validation, table handles, launches.
// The operations are specified in include/cp.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "cp.h"
#include "cp_dispatch.h"
#include "cp_internal.h"

namespace {

thread_local std::string g_last_error;
std::atomic<int> g_fail_alloc{0};
std::atomic<int> g_fail_register{0};

bool take_injected(std::atomic<int>& c) {
  int v = c.load();
  while (v > 0) {
    if (c.compare_exchange_weak(v, v - 1)) return true;
  }
  return false;
}

}  // namespace

static_assert(cpk::kBucketBits == cpx::kBucketBitsHost, "one bucket width on both sides");

namespace cpx {

void set_error(const std::string& what) { g_last_error = what; }

cp_status cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return CP_ERR_CUDA;
}

HostScratch host_scratch_layout(void* base, uint32_t capacity, uint32_t nb) {
  HostScratch h;
  h.capacity = capacity;
  h.counts = static_cast<uint32_t*>(base);
  h.cursor = h.counts + host_scratch_count_words(nb);
  h.perm = h.cursor + host_scratch_count_words(nb);
  h.cslot = h.perm + capacity;
  return h;
}

cpk::KernelSet kernels_for(uint32_t k) {
  switch (k) {
    case 3: return cpk::kernels_k3();
    case 4: return cpk::kernels_k4();
    case 5: return cpk::kernels_k5();
    default: return cpk::kernels_k6();
  }
}

uint32_t stage_bytes(const cp_table* t, bool soa, uint32_t* alpha_slot) {
  return stage_bytes_for(cpk::kStagePrefix, t->code_bytes, t->soa_stride, soa, alpha_slot);
}

cp_status launch_decode(const cp_table* t, const int64_t* idx, uint64_t n, uint16_t* out,
                        cudaStream_t stream, bool host_path, const HostScratch* hs) {
  const bool soa = (t->layout == CP_LAYOUT_SOA);
  const int ci = cpk::cpl_index(t->d);
  cpk::DecodeFn fn = host_path ? t->kernels.host[soa ? 1 : 0][ci] : t->kernels.dev[soa ? 1 : 0][ci];
  cpk::DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.codes = soa ? t->soa_codes : t->rec;
  p.alpha = soa ? t->soa_alpha : nullptr;
  p.n_rows = t->n_rows;
  p.table_bytes = soa ? t->n_rows * t->soa_stride : t->n_rows * t->rec_bytes;
  p.d = t->d;
  p.stride = soa ? t->soa_stride : t->rec_bytes;
  p.code_bytes = t->code_bytes;
  p.stage_bytes = stage_bytes(t, soa, &p.alpha_slot);
  p.lut = t->lut_dev;
  p.idx = idx;
  p.n = n;
  p.out = out;
  p.status = t->status_dev;

  if (!host_path) {
    // Non-persistent grid: kBlkWarps * block_rows(ci) lookups per CTA.
    const int rows = cpk::block_rows(ci);
    const size_t smem = static_cast<size_t>(cpk::lut_bytes(cpk::block_rep(ci))) +
                        static_cast<size_t>(cpk::kBlkWarps) * rows * p.stage_bytes;
    if (smem > static_cast<size_t>(t->max_smem)) {
      g_last_error = "geometry needs more shared memory than the device offers";
      return CP_ERR_INVALID_ARG;
    }
    const uint64_t per_block = static_cast<uint64_t>(cpk::kBlkWarps) * rows;
    const uint64_t blocks = (n + per_block - 1) / per_block;
    if (blocks > 0x7FFFFFFFull) {
      g_last_error = "too many lookups for one launch";
      return CP_ERR_INVALID_ARG;
    }
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    void* args[] = {&p};
    e = cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3(static_cast<unsigned>(blocks)),
                         dim3(cpk::kBlkWarps * 32), args, smem, stream);
    if (e != cudaSuccess) return cuda_fail(e, "lookup-decode launch");
    return CP_OK;
  }
  // Host-resident table: persistent grid.
  const int pf = cpk::kPfHost;
  const bool reg_ring = cpk::host_uses_register_ring(ci);
  int nwarps = reg_ring ? cpk::kHostWarps : cpk::kMaxWarps;
  const size_t lut = cpk::lut_bytes(reg_ring ? cpk::kLutRepHostReg : cpk::kLutRepHost);
  auto smem_for = [&](int w) {
    if (reg_ring) return lut + static_cast<size_t>(w) * p.stage_bytes;   // one stage per warp
    return lut + static_cast<size_t>(w) * pf * p.stage_bytes + static_cast<size_t>(w) * pf * 8;
  };
  while (nwarps > 1 && smem_for(nwarps) > static_cast<size_t>(t->max_smem)) nwarps >>= 1;
  const size_t smem = smem_for(nwarps);
  if (smem > static_cast<size_t>(t->max_smem)) {
    g_last_error = "geometry needs more shared memory than the device offers";
    return CP_ERR_INVALID_ARG;
  }
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  // Persistent grid: one CTA per SM (the LUT takes most of shared memory), or
  // fewer when there are fewer lookups than warps.
  uint64_t blocks = (n + nwarps - 1) / nwarps;
  if (blocks > static_cast<uint64_t>(t->sm_count)) blocks = t->sm_count;
  if (n / (blocks * nwarps) >= (1ull << 31)) {   // rows per warp are counted in 32 bits
    g_last_error = "too many lookups for one launch";
    return CP_ERR_INVALID_ARG;
  }
  // Per pass of at most hs->capacity lookups: partition the lookups by row
  // range, then decode them in that order (each row lands at its own position;
  // repeats of an id read its record from L2).
  const uint64_t cap = hs->capacity;
  const bool cached = t->cache != nullptr && t->cmap_ts != 0;
  for (uint64_t c0 = 0; c0 < n; c0 += cap) {
    const uint64_t m = (n - c0 < cap) ? n - c0 : cap;
    cpk::launch_bucket_partition(idx + c0, m, t->n_rows, cached ? t->cmap_keys : nullptr,
                                 cached ? t->cmap_vals : nullptr, cached ? t->cmap_ts : 0,
                                 hs->cslot, t->bucket_shift, t->bucket_nb, hs->counts,
                                 hs->cursor, hs->perm, t->sm_count, stream);
    cpk::DecodeParams pc = p;
    pc.idx = idx + c0;
    pc.perm = hs->perm;
    if (cached) {
      pc.cslot = hs->cslot;
      pc.cache = t->cache;
      pc.cache_bytes = t->cache_rows * t->rec_bytes;
    }
    pc.n = m;
    pc.out = out + c0 * t->d;
    uint64_t bl = (m + nwarps - 1) / nwarps;
    if (bl > static_cast<uint64_t>(t->sm_count)) bl = t->sm_count;
    void* args[] = {&pc};
    e = cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3(static_cast<unsigned>(bl)),
                         dim3(nwarps * 32), args, smem, stream);
    if (e != cudaSuccess) return cuda_fail(e, "host lookup-decode launch");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "host path launch");
  }
  return CP_OK;
}

}  // namespace cpx

namespace {

using cpx::aligned;
using cpx::cuda_fail;
using cpx::geometry_ok;
using cpx::kernels_for;
using cpx::kMaxLookups;
using cpx::kMaxRows;
using cpx::soa_stride;

// Mixed-rate table: the non-persistent block kernel with the rate taken per row.
cp_status launch_mixed(const cp_table* t, const int64_t* idx, uint64_t n, uint16_t* out,
                       cudaStream_t stream) {
  cpk::DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.codes = t->rec;
  p.n_rows = t->n_rows;
  p.table_bytes = t->table_bytes;
  p.d = t->d;
  p.code_bytes = t->d * 6 / 16;                         // stages sized for the widest rate
  const uint32_t span = p.code_bytes + 2 + 14;
  p.stage_bytes = cpk::kStagePrefix + ((span + 15u) & ~15u) + 16u;
  p.lut = t->lut_dev;
  p.idx = idx;
  p.n = n;
  p.out = out;
  p.status = t->status_dev;
  const int ci = cpk::cpl_index(t->d);
  const int rows = cpk::mixed_rows_per_warp(ci);
  const size_t smem = static_cast<size_t>(cpk::lut_bytes(cpk::kLutRepBlock)) +
                      static_cast<size_t>(cpk::kBlkWarps) * rows * p.stage_bytes;
  if (smem > static_cast<size_t>(t->max_smem)) {
    g_last_error = "geometry needs more shared memory than the device offers";
    return CP_ERR_INVALID_ARG;
  }
  const uint64_t per_block = static_cast<uint64_t>(cpk::kBlkWarps) * rows;
  const uint64_t blocks = (n + per_block - 1) / per_block;
  if (blocks > 0x7FFFFFFFull) {
    g_last_error = "too many lookups for one launch";
    return CP_ERR_INVALID_ARG;
  }
  cpk::MixedFn fn = cpk::mixed_kernel(ci);
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  const uint64_t* offsets = t->offsets;
  void* args[] = {&p, &offsets};
  e = cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3(static_cast<unsigned>(blocks)),
                       dim3(cpk::kBlkWarps * 32), args, smem, stream);
  if (e != cudaSuccess) return cuda_fail(e, "mixed lookup-decode launch");
  return CP_OK;
}

cp_status decode_common(const cp_table* t, const int64_t* idx, uint64_t n, uint16_t* out,
                        void* stream, int want_residency) {
  if (t == nullptr) return CP_ERR_INVALID_ARG;
  if (t->residency != want_residency) {
    g_last_error = want_residency == CP_RESIDENT_DEVICE
                       ? "table is host-resident: use cp_lookup_decode_host"
                       : "table is device-resident: use cp_lookup_decode";
    return CP_ERR_INVALID_ARG;
  }
  if (n == 0) return CP_OK;
  if (n > kMaxLookups || idx == nullptr || out == nullptr || !aligned(idx, 8) ||
      !aligned(out, 16)) {
    g_last_error = "bad ids/output pointer, alignment or count";
    return CP_ERR_INVALID_ARG;
  }
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != t->device) {
    g_last_error = "current device differs from the table's device";
    return CP_ERR_INVALID_ARG;
  }
  if (t->offsets != nullptr) return launch_mixed(t, idx, n, out, static_cast<cudaStream_t>(stream));
  const bool host = want_residency == CP_RESIDENT_HOST;
  cpx::HostScratch hs{};
  if (host) hs = cpx::host_scratch_layout(t->scratch_dev, cpk::kBucketChunk, t->bucket_nb);
  return cpx::launch_decode(t, idx, n, out, static_cast<cudaStream_t>(stream), host,
                            host ? &hs : nullptr);
}

}  // namespace

namespace cpk {

__global__ void repack_soa_kernel(const uint8_t* __restrict__ rec, uint64_t n_rows, uint32_t R,
                                  uint32_t code_bytes, uint32_t S, uint8_t* __restrict__ codes,
                                  uint16_t* __restrict__ alpha) {
  const int lane = threadIdx.x & 31;
  const uint64_t warps = static_cast<uint64_t>(gridDim.x) * (blockDim.x >> 5);
  for (uint64_t r = static_cast<uint64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < n_rows; r += warps) {
    const uint16_t* src = reinterpret_cast<const uint16_t*>(rec + r * R);
    uint16_t* dst = reinterpret_cast<uint16_t*>(codes + r * S);
    for (uint32_t i = lane; i < S / 2; i += 32) dst[i] = (2 * i < code_bytes) ? src[i] : 0;
    if (lane == 0) alpha[r] = src[code_bytes / 2];
  }
}

}  // namespace cpk

extern "C" {

uint64_t cp_record_bytes(uint32_t d, uint32_t bits_per_step) {
  if (!geometry_ok(d, bits_per_step)) return 0;
  return static_cast<uint64_t>(d) * bits_per_step / 16 + 2;
}

uint64_t cp_soa_bytes(uint64_t n_rows, uint32_t d, uint32_t bits_per_step) {
  if (!geometry_ok(d, bits_per_step) || n_rows == 0 || n_rows > kMaxRows) return 0;
  const uint64_t codes = n_rows * soa_stride(d, bits_per_step);
  const uint64_t alph = (n_rows * 2 + 15) & ~15ull;
  return codes + alph;
}

const char* cp_status_string(cp_status s) {
  switch (s) {
    case CP_OK: return "CP_OK";
    case CP_ERR_INVALID_ARG: return "CP_ERR_INVALID_ARG";
    case CP_ERR_INDEX_OOB: return "CP_ERR_INDEX_OOB";
    case CP_ERR_CUDA: return "CP_ERR_CUDA";
    case CP_ERR_NO_MEMORY: return "CP_ERR_NO_MEMORY";
    case CP_ERR_FORMAT: return "CP_ERR_FORMAT";
  }
  return "CP_ERR_UNKNOWN";
}

const char* cp_last_error(void) { return g_last_error.c_str(); }

cp_status cp_test_inject_failure(int kind, int count) {
  if (kind == 1) g_fail_alloc.store(count);
  else if (kind == 2) g_fail_register.store(count);
  else return CP_ERR_INVALID_ARG;
  return CP_OK;
}

void cp_table_free(cp_table* t) {
  if (t == nullptr) return;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != t->device) cudaSetDevice(t->device);
  if (t->lut_dev) cudaFree(t->lut_dev);
  if (t->status_dev) cudaFree(t->status_dev);
  if (t->scratch_dev) cudaFree(t->scratch_dev);
  if (t->cmap_keys) cudaFree(t->cmap_keys);
  if (t->registered) cudaHostUnregister(t->registered);
  if (prev >= 0 && prev != t->device) cudaSetDevice(prev);
  delete t;
}

cp_status cp_table_load(cp_table** out, const void* records, uint64_t n_rows, uint32_t d,
                        uint32_t bits_per_step, const uint16_t* lut_fp16, int residency,
                        int layout, void* soa_dst, void* stream) {
  if (out == nullptr) return CP_ERR_INVALID_ARG;
  *out = nullptr;
  if (records == nullptr || lut_fp16 == nullptr || n_rows == 0 || n_rows > kMaxRows ||
      !geometry_ok(d, bits_per_step) || !aligned(records, 16)) {
    g_last_error = "bad records pointer/alignment, LUT pointer or geometry";
    return CP_ERR_INVALID_ARG;
  }
  if (residency != CP_RESIDENT_DEVICE && residency != CP_RESIDENT_HOST) return CP_ERR_INVALID_ARG;
  if (layout != CP_LAYOUT_AOS && layout != CP_LAYOUT_SOA) return CP_ERR_INVALID_ARG;
  if (layout == CP_LAYOUT_SOA && (soa_dst == nullptr || !aligned(soa_dst, 16))) {
    g_last_error = "CP_LAYOUT_SOA needs a 16-byte aligned soa_dst";
    return CP_ERR_INVALID_ARG;
  }
  if (layout == CP_LAYOUT_AOS && soa_dst != nullptr) return CP_ERR_INVALID_ARG;
  for (int i = 0; i < 1024; ++i) {
    if ((lut_fp16[i] & 0x7c00u) == 0x7c00u) {
      g_last_error = "LUT holds a non-finite fp16 value";
      return CP_ERR_FORMAT;
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  cp_table* t = new (std::nothrow) cp_table();
  if (t == nullptr) return CP_ERR_NO_MEMORY;
  cudaGetDevice(&t->device);
  t->residency = residency;
  t->layout = layout;
  t->n_rows = n_rows;
  t->d = d;
  t->k = bits_per_step;
  t->code_bytes = d * bits_per_step / 16;
  t->rec_bytes = t->code_bytes + 2;
  t->soa_stride = soa_stride(d, bits_per_step);
  t->kernels = kernels_for(bits_per_step);
  cudaDeviceGetAttribute(&t->sm_count, cudaDevAttrMultiProcessorCount, t->device);
  cudaDeviceGetAttribute(&t->max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, t->device);

  cp_status st = CP_OK;
  cudaError_t e;
  if (take_injected(g_fail_alloc)) {
    g_last_error = "injected device allocation failure";
    delete t;
    return CP_ERR_NO_MEMORY;
  }
  e = cudaMalloc(&t->lut_dev, 512 * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMalloc(&t->status_dev, sizeof(uint32_t));
  if (e != cudaSuccess) {
    cuda_fail(e, "cudaMalloc");
    cp_table_free(t);
    return CP_ERR_NO_MEMORY;
  }
  e = cudaMemcpyAsync(t->lut_dev, lut_fp16, 2048, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(t->status_dev, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) {
    st = cuda_fail(e, "LUT upload");
    cp_table_free(t);
    return st;
  }
  const uint64_t table_bytes = n_rows * t->rec_bytes;
  if (residency == CP_RESIDENT_HOST) {
    // row-range buckets of the visiting order: at most 2^kBucketBits of them
    cpx::bucket_params(n_rows, &t->bucket_shift, &t->bucket_nb);
    const size_t bytes = cpx::host_scratch_bytes(cpk::kBucketChunk, t->bucket_nb);
    if (take_injected(g_fail_alloc)) {
      g_last_error = "injected device allocation failure";
      cp_table_free(t);
      return CP_ERR_NO_MEMORY;
    }
    e = cudaMalloc(&t->scratch_dev, bytes);
    if (e != cudaSuccess) {
      cuda_fail(e, "cudaMalloc(bucket scratch)");
      cp_table_free(t);
      return CP_ERR_NO_MEMORY;
    }
    // range counts start at zero; every pass leaves them at zero again
    e = cudaMemsetAsync(t->scratch_dev, 0,
                        cpx::host_scratch_count_words(t->bucket_nb) * sizeof(uint32_t), s);
    if (e != cudaSuccess) {
      st = cuda_fail(e, "scratch clear");
      cp_table_free(t);
      return st;
    }
    void* dptr = nullptr;
    if (take_injected(g_fail_register)) {
      g_last_error = "injected host registration failure";
      cp_table_free(t);
      return CP_ERR_CUDA;
    }
    e = cudaHostGetDevicePointer(&dptr, const_cast<void*>(records), 0);
    if (e != cudaSuccess) {
      cudaGetLastError();   // not page-locked: register it ourselves
      e = cudaHostRegister(const_cast<void*>(records), table_bytes,
                           cudaHostRegisterMapped | cudaHostRegisterReadOnly);
      if (e != cudaSuccess) {   // read-only registration is optional on some systems
        cudaGetLastError();
        e = cudaHostRegister(const_cast<void*>(records), table_bytes, cudaHostRegisterMapped);
      }
      if (e != cudaSuccess) {
        st = cuda_fail(e, "cudaHostRegister");
        cp_table_free(t);
        return st;
      }
      t->registered = const_cast<void*>(records);
      e = cudaHostGetDevicePointer(&dptr, const_cast<void*>(records), 0);
      if (e != cudaSuccess) {
        st = cuda_fail(e, "cudaHostGetDevicePointer");
        cp_table_free(t);
        return st;
      }
    }
    t->rec = static_cast<const uint8_t*>(dptr);
    if (!aligned(t->rec, 16)) {
      g_last_error = "device alias of the host table is not 16-byte aligned";
      cp_table_free(t);
      return CP_ERR_INVALID_ARG;
    }
  } else {
    t->rec = static_cast<const uint8_t*>(records);
  }
  if (layout == CP_LAYOUT_SOA) {
    uint8_t* codes = static_cast<uint8_t*>(soa_dst);
    if (residency == CP_RESIDENT_HOST) {
      void* dptr = nullptr;
      e = cudaHostGetDevicePointer(&dptr, soa_dst, 0);
      if (e != cudaSuccess) {
        st = cuda_fail(e, "cudaHostGetDevicePointer(soa_dst)");
        cp_table_free(t);
        return st;
      }
      codes = static_cast<uint8_t*>(dptr);
    }
    t->soa_codes = codes;
    t->soa_alpha = reinterpret_cast<const uint16_t*>(codes + n_rows * t->soa_stride);
    const uint64_t warps = n_rows < (1ull << 22) ? n_rows : (1ull << 22);
    const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
    cpk::repack_soa_kernel<<<blocks, 256, 0, s>>>(t->rec, n_rows, t->rec_bytes, t->code_bytes,
                                                  t->soa_stride, codes,
                                                  const_cast<uint16_t*>(t->soa_alpha));
    e = cudaGetLastError();
    if (e != cudaSuccess) {
      st = cuda_fail(e, "SoA repack launch");
      cp_table_free(t);
      return st;
    }
  }
  *out = t;
  return CP_OK;
}

cp_status cp_lookup_decode(const cp_table* t, const int64_t* idx, uint64_t n, uint16_t* out,
                           void* stream) {
  return decode_common(t, idx, n, out, stream, CP_RESIDENT_DEVICE);
}

cp_status cp_lookup_decode_host(const cp_table* t, const int64_t* idx, uint64_t n,
                                uint16_t* out, void* stream) {
  return decode_common(t, idx, n, out, stream, CP_RESIDENT_HOST);
}

cp_status cp_table_load_mixed(cp_table** out, const void* records, const uint64_t* offsets,
                              uint64_t n_rows, uint32_t d, const uint16_t* lut_fp16, void* stream) {
  if (out == nullptr) return CP_ERR_INVALID_ARG;
  *out = nullptr;
  if (records == nullptr || offsets == nullptr || lut_fp16 == nullptr || n_rows == 0 ||
      n_rows > kMaxRows || d < 32 || d > 4096 || d % 32 != 0 || !aligned(records, 16) ||
      !aligned(offsets, 8)) {
    cpx::set_error("bad records/offsets pointer or alignment, LUT pointer or geometry");
    return CP_ERR_INVALID_ARG;
  }
  for (int i = 0; i < 1024; ++i) {
    if ((lut_fp16[i] & 0x7c00u) == 0x7c00u) {
      cpx::set_error("LUT holds a non-finite fp16 value");
      return CP_ERR_FORMAT;
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cp_table* t = new (std::nothrow) cp_table();
  if (t == nullptr) return CP_ERR_NO_MEMORY;
  cudaGetDevice(&t->device);
  t->residency = CP_RESIDENT_DEVICE;
  t->layout = CP_LAYOUT_AOS;
  t->n_rows = n_rows;
  t->d = d;
  t->k = 0;
  t->rec = static_cast<const uint8_t*>(records);
  t->offsets = offsets;
  cudaDeviceGetAttribute(&t->sm_count, cudaDevAttrMultiProcessorCount, t->device);
  cudaDeviceGetAttribute(&t->max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, t->device);
  if (take_injected(g_fail_alloc)) {
    cpx::set_error("injected device allocation failure");
    delete t;
    return CP_ERR_NO_MEMORY;
  }
  cudaError_t e = cudaMalloc(&t->lut_dev, 512 * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMalloc(&t->status_dev, sizeof(uint32_t));
  if (e != cudaSuccess) {
    cuda_fail(e, "cudaMalloc");
    cp_table_free(t);
    return CP_ERR_NO_MEMORY;
  }
  e = cudaMemcpyAsync(t->lut_dev, lut_fp16, 2048, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(t->status_dev, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) {
    cp_status st = cuda_fail(e, "LUT upload");
    cp_table_free(t);
    return st;
  }
  // every record length must give a rate in {3,..,6}; read the table's end
  cpk::launch_check_mixed(offsets, n_rows, d, t->status_dev, t->sm_count, s);
  uint32_t bad = 0;
  uint64_t end = 0;
  e = cudaMemcpyAsync(&bad, t->status_dev, sizeof(bad), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&end, offsets + n_rows, sizeof(end), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(t->status_dev, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cp_status st = cuda_fail(e, "mixed table check");
    cp_table_free(t);
    return st;
  }
  if (bad) {
    cpx::set_error("a record length gives no bit rate in {3, 4, 5, 6} bits per step");
    cp_table_free(t);
    return CP_ERR_FORMAT;
  }
  t->table_bytes = end;
  *out = t;
  return CP_OK;
}

cp_status cp_table_set_cache(cp_table* t, const int64_t* hot_rows, uint64_t m, void* cache,
                             void* stream) {
  if (t == nullptr) return CP_ERR_INVALID_ARG;
  if (t->residency != CP_RESIDENT_HOST || t->layout != CP_LAYOUT_AOS ||
      !cpk::host_uses_register_ring(cpk::cpl_index(t->d))) {
    cpx::set_error(
        "the hot-row cache applies to host-resident AoS tables with d = 256, 512 or 1024");
    return CP_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (t->cmap_keys != nullptr) {            // drop the previous cache (after pending work)
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    cudaFree(t->cmap_keys);
    t->cmap_keys = nullptr;
    t->cmap_vals = nullptr;
    t->cmap_ts = 0;
    t->cache = nullptr;
    t->cache_rows = 0;
  }
  if (m == 0) return CP_OK;
  if (hot_rows == nullptr || cache == nullptr || !aligned(cache, 16) || m > (1ull << 30) ||
      m > t->n_rows) {
    cpx::set_error("bad hot-row list, cache pointer/alignment or count");
    return CP_ERR_INVALID_ARG;
  }
  std::vector<int64_t> rows(hot_rows, hot_rows + m);
  std::sort(rows.begin(), rows.end());            // ascending: link-friendly copy order
  for (uint64_t i = 0; i < m; ++i) {
    if (rows[i] < 0 || static_cast<uint64_t>(rows[i]) >= t->n_rows ||
        (i > 0 && rows[i] == rows[i - 1])) {
      cpx::set_error("hot rows must be distinct ids in [0, n_rows)");
      return CP_ERR_INVALID_ARG;
    }
  }
  uint32_t ts = 1024;
  while (ts < 2 * m) ts <<= 1;
  if (take_injected(g_fail_alloc)) {
    cpx::set_error("injected device allocation failure");
    return CP_ERR_NO_MEMORY;
  }
  void* mem = nullptr;
  const size_t bytes = static_cast<size_t>(ts) * (sizeof(unsigned long long) + sizeof(uint32_t)) +
                       m * sizeof(int64_t);
  cudaError_t e = cudaMalloc(&mem, bytes);
  if (e != cudaSuccess) {
    cuda_fail(e, "cudaMalloc(cache map)");
    return CP_ERR_NO_MEMORY;
  }
  unsigned long long* keys = static_cast<unsigned long long*>(mem);
  uint32_t* vals = reinterpret_cast<uint32_t*>(keys + ts);
  int64_t* rows_dev = reinterpret_cast<int64_t*>(vals + ts);
  e = cudaMemsetAsync(keys, 0, ts * sizeof(unsigned long long), s);
  if (e == cudaSuccess)   // pageable source: returns once the data is staged
    e = cudaMemcpyAsync(rows_dev, rows.data(), m * sizeof(int64_t), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) {
    cudaFree(mem);
    return cuda_fail(e, "cache map upload");
  }
  cpk::launch_cache_build(t->rec, t->rec_bytes, rows_dev, m, static_cast<uint8_t*>(cache), keys,
                          vals, ts, t->sm_count, s);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    cudaFree(mem);
    return cuda_fail(e, "cache build launch");
  }
  e = cudaStreamSynchronize(s);                  // rows_dev must stay valid until then
  if (e != cudaSuccess) {
    cudaFree(mem);
    return cuda_fail(e, "cache build");
  }
  t->cmap_keys = keys;
  t->cmap_vals = vals;
  t->cmap_ts = ts;
  t->cache = static_cast<const uint8_t*>(cache);
  t->cache_rows = m;
  return CP_OK;
}

cp_status cp_lookup_decode_reduce(const cp_table* t, const int64_t* idx, uint64_t n_groups,
                                  uint32_t group, const float* weights, uint16_t* out,
                                  void* stream) {
  if (t == nullptr) return CP_ERR_INVALID_ARG;
  if (t->residency != CP_RESIDENT_DEVICE || t->offsets != nullptr) {
    cpx::set_error("the fused readout needs a device-resident single-rate table");
    return CP_ERR_INVALID_ARG;
  }
  if (n_groups == 0) return CP_OK;
  const int ci = cpk::cpl_index(t->d);
  if (ci < 1 || ci > 3) {
    cpx::set_error("the fused readout supports d = 256, 512 or 1024");
    return CP_ERR_INVALID_ARG;
  }
  if (group == 0 || n_groups > kMaxLookups / group || idx == nullptr || out == nullptr ||
      !aligned(idx, 8) || !aligned(out, 16) || (weights != nullptr && !aligned(weights, 4))) {
    cpx::set_error("bad ids/weights/output pointer, alignment or counts");
    return CP_ERR_INVALID_ARG;
  }
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != t->device) {
    cpx::set_error("current device differs from the table's device");
    return CP_ERR_INVALID_ARG;
  }
  const bool soa = (t->layout == CP_LAYOUT_SOA);
  cpk::DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.codes = soa ? t->soa_codes : t->rec;
  p.alpha = soa ? t->soa_alpha : nullptr;
  p.n_rows = t->n_rows;
  p.table_bytes = soa ? t->n_rows * t->soa_stride : t->n_rows * t->rec_bytes;
  p.d = t->d;
  p.stride = soa ? t->soa_stride : t->rec_bytes;
  p.code_bytes = t->code_bytes;
  p.stage_bytes = cpx::stage_bytes(t, soa, &p.alpha_slot);
  p.lut = t->lut_dev;
  p.idx = idx;
  p.n = n_groups * group;
  p.out = out;
  p.status = t->status_dev;
  const int nwarps = cpk::kReduceWarps;
  const size_t smem = static_cast<size_t>(cpk::lut_bytes(32)) +
                      static_cast<size_t>(nwarps) * cpk::kPfReduce * (p.stage_bytes + 8);
  if (smem > static_cast<size_t>(t->max_smem)) return CP_ERR_INVALID_ARG;
  cpk::ReduceFn fn = t->kernels.reduce[soa ? 1 : 0][ci - 1];
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  uint64_t blocks = (n_groups + nwarps - 1) / nwarps;
  if (blocks > static_cast<uint64_t>(t->sm_count)) blocks = t->sm_count;
  if ((n_groups / (blocks * nwarps) + 1) * group >= (1ull << 31)) {
    cpx::set_error("too many lookups for one launch");
    return CP_ERR_INVALID_ARG;
  }
  void* args[] = {&p, &weights, &group, &n_groups};
  e = cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3(static_cast<unsigned>(blocks)),
                       dim3(nwarps * 32), args, smem, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fused readout launch");
  return CP_OK;
}

cp_status cp_get_status(const cp_table* t, void* stream) {
  if (t == nullptr) return CP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t h = 0;
  e = cudaMemcpyAsync(&h, t->status_dev, sizeof(h), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(t->status_dev, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status readback");
  return (h & 1u) ? CP_ERR_INDEX_OOB : CP_OK;
}

}  // extern "C"

// Shared helpers of libmoe_dp (device and host side).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_dp.h"

namespace moe {

inline int dtype_bytes(int dtype) { return dtype == MOE_BF16 ? 2 : (dtype == MOE_F32 ? 4 : 0); }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Launch-status mapping used by every entry point after its launches.
inline moe_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int num_sms();  // cached per device (host.cpp)

// Programmatic dependent launch: every kernel of the library is launched with
// programmatic stream serialization, so its launch may overlap the end of the
// kernel before it on the stream.  Each kernel starts with grid_dep_wait(),
// which returns once the earlier kernels on the stream have completed and
// their memory is visible, before it touches global memory; it then calls
// grid_dep_launch() so that the next kernel can start launching.  MOE_PDL=0
// in the environment turns the overlap off (plain stream order).
bool pdl_enabled();  // host.cpp

__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

inline void set_pdl_attr(cudaLaunchAttribute& a) {
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
}

// kernel<<<grid, block, smem, stream>>>(args...) with the dependent-launch
// attribute; the result is also left for cudaGetLastError.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  set_pdl_attr(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Replica pointer table passed by value as a kernel argument.
struct ReplicaPtrs {
  const void* p[MOE_MAX_REPLICAS];
};

// ------------------------------------------------------------------ device
__device__ __forceinline__ void flag(uint32_t* status, uint32_t bit) {
  if (status != nullptr) atomicOr(status, bit);
}

// Segment r containing global row g: largest r with offsets[r] <= g (offsets
// non-decreasing, offsets[0] = 0, g < offsets[R]).
__device__ __forceinline__ int find_segment(const int32_t* offsets, int R, int64_t g) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((int64_t)offsets[mid] <= g)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// bf16x2 <-> float2 packing (round to nearest even)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

}  // namespace moe

// DP gather and DP scatter: packed row copies between the replicas' token
// segments and the global buffer.
//
// SGLang chapter 17, section "两种 gather: all_reduce 与 all_gather": the
// global buffer is zero-filled and each replica writes its rows at its start
// row; on one device the all-reduce that follows adds nothing, so the gather
// is a copy plus zero padding.  Section "scatter: 把 MoE 的输出还回本副本":
// the scatter cuts the buffer back by the same counts.
//
// Design: one warp per global row, 16-byte vectors, several vectors in flight
// per lane; replica pointers travel by value in the kernel arguments, the
// counts and offsets are read once per block into shared memory.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void copy_row(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                         int vpr, int lane) {
  for (int v0 = lane; v0 < vpr; v0 += 32 * kUnroll) {
    uint4 t[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      int v = v0 + u * 32;
      if (v < vpr) t[u] = ld_nc(src + v);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      int v = v0 + u * 32;
      if (v < vpr) dst[v] = t[u];
    }
  }
}

__device__ __forceinline__ void zero_row(uint4* __restrict__ dst, int vpr, int lane) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int v = lane; v < vpr; v += 32) dst[v] = z;
}

__global__ void __launch_bounds__(kWarps * 32)
    dp_gather_kernel(ReplicaPtrs src, const int32_t* __restrict__ counts,
                     const int32_t* __restrict__ offsets, int R, int64_t rows, int vpr,
                     uint4* __restrict__ global, uint32_t* status) {
  __shared__ int32_t s_off[MOE_MAX_REPLICAS + 1];
  __shared__ int32_t s_cnt[MOE_MAX_REPLICAS];
  for (int i = threadIdx.x; i <= R; i += blockDim.x) {
    s_off[i] = offsets[i];
    if (i < R) s_cnt[i] = counts[i];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  for (int64_t g = warp0; g < rows; g += nwarps) {
    int r = find_segment(s_off, R, g);
    int64_t i = g - s_off[r];
    int64_t seg = (int64_t)s_off[r + 1] - s_off[r];
    int64_t c = s_cnt[r];
    if (c > seg) {
      if (i == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
      c = seg;
    }
    if (c > 0 && src.p[r] == nullptr) {
      if (i == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
      c = 0;
    }
    uint4* dst = global + g * vpr;
    if (i >= 0 && i < c)
      copy_row(static_cast<const uint4*>(src.p[r]) + i * vpr, dst, vpr, lane);
    else
      zero_row(dst, vpr, lane);
  }
}

__global__ void __launch_bounds__(kWarps * 32)
    dp_scatter_kernel(const uint4* __restrict__ global, const int32_t* __restrict__ counts,
                      const int32_t* __restrict__ offsets, int R, int64_t rows, int vpr,
                      ReplicaPtrs dst, uint32_t* status) {
  __shared__ int32_t s_off[MOE_MAX_REPLICAS + 1];
  __shared__ int32_t s_cnt[MOE_MAX_REPLICAS];
  for (int i = threadIdx.x; i <= R; i += blockDim.x) {
    s_off[i] = offsets[i];
    if (i < R) s_cnt[i] = counts[i];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  for (int64_t g = warp0; g < rows; g += nwarps) {
    int r = find_segment(s_off, R, g);
    int64_t i = g - s_off[r];
    int64_t seg = (int64_t)s_off[r + 1] - s_off[r];
    int64_t c = s_cnt[r];
    if (c > seg) {
      if (i == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
      c = seg;
    }
    if (c > 0 && dst.p[r] == nullptr) {
      if (i == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
      c = 0;
    }
    if (i >= 0 && i < c)
      copy_row(global + g * vpr,
               static_cast<uint4*>(const_cast<void*>(dst.p[r])) + i * vpr, vpr, lane);
  }
}

moe_status check_common(const int32_t* d_counts, const int32_t* d_offsets, int R, int64_t rows,
                        int H, int dtype, const void* d_global) {
  if (R < 1 || R > MOE_MAX_REPLICAS || rows < 0 || rows > INT32_MAX || H < 1)
    return MOE_ERR_INVALID_ARG;
  int eb = dtype_bytes(dtype);
  if (eb == 0) return MOE_ERR_UNSUPPORTED;
  if (((int64_t)H * eb) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;  // nothing to move; data pointers may be null
  if (d_counts == nullptr || d_offsets == nullptr || d_global == nullptr || !aligned16(d_global))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int grid_for_rows(int64_t rows) {
  int64_t want = (rows + kWarps - 1) / kWarps;
  int64_t cap = (int64_t)num_sms() * 16;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_dp_gather(const void* const* local, const int32_t* d_counts,
                                    const int32_t* d_offsets, int R, int64_t rows, int H,
                                    int dtype, void* d_global, uint32_t* d_status, void* stream) {
  moe_status st = check_common(d_counts, d_offsets, R, rows, H, dtype, d_global);
  if (st != MOE_OK || rows == 0) return st;
  if (local == nullptr) return MOE_ERR_INVALID_ARG;
  ReplicaPtrs ptrs;
  for (int r = 0; r < R; ++r) {
    if (local[r] != nullptr && !aligned16(local[r])) return MOE_ERR_INVALID_ARG;
    ptrs.p[r] = local[r];
  }
  const int vpr = (int)((int64_t)H * dtype_bytes(dtype) / 16);
  dp_gather_kernel<<<grid_for_rows(rows), kWarps * 32, 0, as_stream(stream)>>>(
      ptrs, d_counts, d_offsets, R, rows, vpr, static_cast<uint4*>(d_global), d_status);
  return launch_status();
}

extern "C" moe_status moe_dp_scatter(const void* d_global, const int32_t* d_counts,
                                     const int32_t* d_offsets, int R, int64_t rows, int H,
                                     int dtype, void* const* local, uint32_t* d_status,
                                     void* stream) {
  moe_status st = check_common(d_counts, d_offsets, R, rows, H, dtype, d_global);
  if (st != MOE_OK || rows == 0) return st;
  if (local == nullptr) return MOE_ERR_INVALID_ARG;
  ReplicaPtrs ptrs;
  for (int r = 0; r < R; ++r) {
    if (local[r] != nullptr && !aligned16(local[r])) return MOE_ERR_INVALID_ARG;
    ptrs.p[r] = local[r];
  }
  const int vpr = (int)((int64_t)H * dtype_bytes(dtype) / 16);
  dp_scatter_kernel<<<grid_for_rows(rows), kWarps * 32, 0, as_stream(stream)>>>(
      static_cast<const uint4*>(d_global), d_counts, d_offsets, R, rows, vpr, ptrs, d_status);
  return launch_status();
}

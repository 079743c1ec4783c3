// Combine: un-permute the expert outputs and apply the top-k weights.
//
// vLLM chapter 27 (Dual Batch Overlap), figure "MoE 模块化内核的
// PrepareAndFinalize 块结构": after MM2 the rows are un-permuted and finalize
// applies the top-k weights.  Token row g receives
//   out[g] = sum_{j<k} w[g, j] * y[inv[g, j]]
// accumulated in float32 in j order and rounded once; rows whose inv entries
// are all -1 (pad rows) are zero.  No float atomics: each output row has one
// owner warp, so the result is deterministic.
//
// Design: one warp per output row; the row is walked in chunks of
// 32 lanes x kUnroll 16-byte vectors; for each chunk the k source rows are
// read (k * kUnroll independent loads per lane in flight) and accumulated in
// registers.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kUnroll = 2;

__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <bool BF16>
__global__ void __launch_bounds__(kWarps * 32)
    combine_kernel(const uint4* __restrict__ ys, const int32_t* __restrict__ inv,
                   const float* __restrict__ w, int64_t rows, int k, int vpr, int64_t cap,
                   uint4* __restrict__ out, uint32_t* status) {
  constexpr int EPV = BF16 ? 8 : 4;  // elements per 16-byte vector
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  for (int64_t g = warp0; g < rows; g += nwarps) {
    int32_t my_d = -1;
    float my_w = 0.f;
    if (lane < k) {
      my_d = inv[g * k + lane];
      my_w = w[g * k + lane];
      if (my_d >= cap) {
        flag(status, MOE_DEV_BAD_COUNTS);
        my_d = -1;
      }
    }
    uint4* dst = out + g * vpr;
    for (int v0 = lane; v0 < vpr; v0 += 32 * kUnroll) {
      float acc[kUnroll][EPV];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[u][e] = 0.f;
      for (int j = 0; j < k; ++j) {
        const int32_t d = __shfl_sync(0xffffffffu, my_d, j);
        const float wj = __shfl_sync(0xffffffffu, my_w, j);
        if (d < 0) continue;
        const uint4* src = ys + (int64_t)d * vpr;
        uint4 t[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          int v = v0 + u * 32;
          if (v < vpr) t[u] = ld_nc(src + v);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const uint32_t q[4] = {t[u].x, t[u].y, t[u].z, t[u].w};
          if (BF16) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc[u][2 * e] = fmaf(wj, bf16lo(q[e]), acc[u][2 * e]);
              acc[u][2 * e + 1] = fmaf(wj, bf16hi(q[e]), acc[u][2 * e + 1]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[u][e] = fmaf(wj, __uint_as_float(q[e]), acc[u][e]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        int v = v0 + u * 32;
        if (v >= vpr) continue;
        uint4 r;
        if (BF16) {
          r.x = pack_bf16x2(acc[u][0], acc[u][1]);
          r.y = pack_bf16x2(acc[u][2], acc[u][3]);
          r.z = pack_bf16x2(acc[u][4], acc[u][5]);
          r.w = pack_bf16x2(acc[u][6], acc[u][7]);
        } else {
          r.x = __float_as_uint(acc[u][0]);
          r.y = __float_as_uint(acc[u][1]);
          r.z = __float_as_uint(acc[u][2]);
          r.w = __float_as_uint(acc[u][3]);
        }
        dst[v] = r;
      }
    }
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_combine(const void* d_out_sorted, const int32_t* d_inv, const float* d_w,
                                  int64_t rows, int k, int H, int dtype, int64_t cap,
                                  void* d_global_out, uint32_t* d_status, void* stream) {
  if (rows < 0 || rows > INT32_MAX || k < 1 || k > MOE_MAX_TOPK || H < 1 || cap < 0)
    return MOE_ERR_INVALID_ARG;
  int eb = dtype_bytes(dtype);
  if (eb == 0) return MOE_ERR_UNSUPPORTED;
  if (((int64_t)H * eb) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (d_inv == nullptr || d_w == nullptr || d_global_out == nullptr ||
      (d_out_sorted == nullptr && cap > 0))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(d_out_sorted) || !aligned16(d_global_out)) return MOE_ERR_INVALID_ARG;
  const int vpr = (int)((int64_t)H * eb / 16);
  int64_t want = (rows + kWarps - 1) / kWarps;
  int64_t lim = (int64_t)num_sms() * 16;
  int grid = (int)(want < lim ? want : lim);
  cudaStream_t s = as_stream(stream);
  if (dtype == MOE_BF16)
    combine_kernel<true><<<grid, kWarps * 32, 0, s>>>(
        static_cast<const uint4*>(d_out_sorted), d_inv, d_w, rows, k, vpr, cap,
        static_cast<uint4*>(d_global_out), d_status);
  else
    combine_kernel<false><<<grid, kWarps * 32, 0, s>>>(
        static_cast<const uint4*>(d_out_sorted), d_inv, d_w, rows, k, vpr, cap,
        static_cast<uint4*>(d_global_out), d_status);
  return launch_status();
}

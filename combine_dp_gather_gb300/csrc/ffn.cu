// moe_grouped_ffn entry point and its float32 CUDA-core path.
//
// The float32 path serves fp32 layers (small, latency-bound shapes): one thread
// per output element, float32 accumulation in index order.  bf16 layers go to
// the tcgen05 kernel in ffn_tc.cu.
#include "common.cuh"
#include "ffn_internal.h"

namespace moe {
namespace {

constexpr int TS = 32;

__device__ __forceinline__ int slot_of_row(const int32_t* offsets, int lo, int hi, int64_t d) {
  // largest s in [lo, hi) with offsets[s] <= d (offsets non-decreasing)
  int a = lo, b = hi - 1;
  while (a < b) {
    int mid = (a + b + 1) >> 1;
    if ((int64_t)offsets[mid] <= d)
      a = mid;
    else
      b = mid - 1;
  }
  return a;
}

// MM1 + SwiGLU: h[d, i] = silu(x[d] . Wg_s[i]) * (x[d] . Wu_s[i]).
// Block: 32 rows x 32 outputs.
__global__ void __launch_bounds__(TS * 8)
    ffn1_f32_kernel(const float* __restrict__ xs, const int32_t* __restrict__ offsets, int lo,
                    int hi, int64_t cap, const float* __restrict__ wgu, int H, int I,
                    float* __restrict__ h) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  const int64_t r0 = (int64_t)blockIdx.y * TS;
  const int i = blockIdx.x * TS + (threadIdx.x & (TS - 1));
  const int64_t begin = offsets[lo], end = offsets[hi] < cap ? offsets[hi] : cap;
  for (int rr = threadIdx.x >> 5; rr < TS; rr += blockDim.x >> 5) {
    const int64_t d = r0 + rr;
    if (d < begin || d >= end || i >= I) continue;
    const int s = slot_of_row(offsets, lo, hi, d);
    const float* x = xs + d * H;
    const float* wg = wgu + ((int64_t)s * 2 * I + i) * H;
    const float* wu = wgu + ((int64_t)s * 2 * I + I + i) * H;
    float g = 0.f, u = 0.f;
    for (int k = 0; k < H; ++k) {
      g = fmaf(x[k], wg[k], g);
      u = fmaf(x[k], wu[k], u);
    }
    h[d * I + i] = g / (1.0f + expf(-g)) * u;
  }
}

// MM2: y[d, o] = h[d] . Wd_s[o].
__global__ void __launch_bounds__(TS * 8)
    ffn2_f32_kernel(const float* __restrict__ h, const int32_t* __restrict__ offsets, int lo,
                    int hi, int64_t cap, const float* __restrict__ wd, int H, int I,
                    float* __restrict__ ys) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  const int64_t r0 = (int64_t)blockIdx.y * TS;
  const int o = blockIdx.x * TS + (threadIdx.x & (TS - 1));
  const int64_t begin = offsets[lo], end = offsets[hi] < cap ? offsets[hi] : cap;
  for (int rr = threadIdx.x >> 5; rr < TS; rr += blockDim.x >> 5) {
    const int64_t d = r0 + rr;
    if (d < begin || d >= end || o >= H) continue;
    const int s = slot_of_row(offsets, lo, hi, d);
    const float* a = h + d * I;
    const float* w = wd + ((int64_t)s * H + o) * I;
    float y = 0.f;
    for (int k = 0; k < I; ++k) y = fmaf(a[k], w[k], y);
    ys[d * H + o] = y;
  }
}

}  // namespace

moe_status launch_ffn_simt_f32(const FfnArgs& a, cudaStream_t s) {
  if (a.slot_hi <= a.slot_lo || a.cap <= 0) return MOE_OK;
  dim3 block(TS * 8);
  dim3 g1((a.I + TS - 1) / TS, (unsigned)((a.cap + TS - 1) / TS));
  launch(ffn1_f32_kernel, g1, block, 0, s, static_cast<const float*>(a.xs), a.offsets, a.slot_lo,
         a.slot_hi, a.cap, static_cast<const float*>(a.wgu), a.H, a.I, static_cast<float*>(a.h));
  dim3 g2((a.H + TS - 1) / TS, (unsigned)((a.cap + TS - 1) / TS));
  launch(ffn2_f32_kernel, g2, block, 0, s, static_cast<const float*>(a.h), a.offsets, a.slot_lo,
         a.slot_hi, a.cap, static_cast<const float*>(a.wd), a.H, a.I, static_cast<float*>(a.ys));
  return launch_status();
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_grouped_ffn_ws_bytes(int64_t cap, int I, int dtype) {
  int eb = dtype_bytes(dtype);
  if (cap < 0 || I < 1 || eb == 0) return 0;
  return (size_t)(cap * (int64_t)I * eb);
}

extern "C" moe_status moe_grouped_ffn(const void* d_sorted, const int32_t* d_offsets_P, int P,
                                      int slot_lo, int slot_hi, int64_t cap,
                                      const void* d_w_gate_up, const void* d_w_down, int H, int I,
                                      int dtype, void* d_out_sorted, void* d_ws, size_t ws_bytes,
                                      uint32_t* d_status, void* stream) {
  if (P < 1 || slot_lo < 0 || slot_hi > P || slot_lo > slot_hi || cap < 0 || cap > INT32_MAX ||
      H < 1 || I < 1)
    return MOE_ERR_INVALID_ARG;
  int eb = dtype_bytes(dtype);
  if (eb == 0) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_BF16 && (H % 256 != 0 || I % 128 != 0 || P > MOE_MAX_SLOTS))
    return MOE_ERR_UNSUPPORTED;
  if (cap == 0 || slot_lo == slot_hi) return MOE_OK;
  if (d_sorted == nullptr || d_offsets_P == nullptr || d_w_gate_up == nullptr ||
      d_w_down == nullptr || d_out_sorted == nullptr || d_ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_grouped_ffn_ws_bytes(cap, I, dtype)) return MOE_ERR_CAPACITY;
  if (!aligned16(d_sorted) || !aligned16(d_out_sorted) || !aligned16(d_ws) ||
      !aligned16(d_w_gate_up) || !aligned16(d_w_down))
    return MOE_ERR_INVALID_ARG;
  FfnArgs a{d_sorted, d_offsets_P, P, slot_lo, slot_hi, cap, d_w_gate_up, d_w_down,
            H, I, d_out_sorted, d_ws, d_status};
  cudaStream_t s = as_stream(stream);
  if (dtype == MOE_BF16) {
    if ((int64_t)P * 2 * I > INT32_MAX || (int64_t)P * H > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    int major = 0, minor = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
    return launch_ffn_tc(a, s);
  }
  return launch_ffn_simt_f32(a, s);
}

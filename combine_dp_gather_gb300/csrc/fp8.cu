// FP8 (e4m3, UE8M0 group scales) quantisation: per-token groups of 128, 128 x
// 128 weight blocks, and the dispatch that quantises the rows it permutes.
//
// SGLang chapter 17, section "prefll 侧的一个必要步骤:per-token-group 量化":
// before dispatch the hidden states are quantised in groups of 128 features
// (the same 128 as expert_alignment) with UE8M0 scale factors.  The scale and
// rounding rules are in fp8.cuh.
#include "common.cuh"
#include "fp8.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kSeg = 1024;  // elements per warp segment: 32 lanes x 32 values

// 32 consecutive values of a row starting at element e0 (16-byte aligned).
template <bool BF16>
__device__ __forceinline__ void load32(const void* row, int64_t e0, float (&v)[32]) {
  if (BF16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(row) + e0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 t = __ldg(p + i);
      const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * i + 2 * j] = bf16lo(w[j]);
        v[8 * i + 2 * j + 1] = bf16hi(w[j]);
      }
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(row) + e0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 t = __ldg(p + i);
      v[4 * i] = t.x;
      v[4 * i + 1] = t.y;
      v[4 * i + 2] = t.z;
      v[4 * i + 3] = t.w;
    }
  }
}

// The lane's 32 values of a 128-value group held by its lane quad -> codes and
// the group's scale exponent.  Every lane of the warp must call it (the quad
// maximum uses shuffles); lanes without data pass zeros.
__device__ __forceinline__ int quantise32(const float (&v)[32], uint4 (&codes)[2]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int e = fp8_scale_exp(quad_max(amax));
  const float inv = pow2i(-e);
  uint32_t c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    c[i] = e4m3x4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
  codes[0] = make_uint4(c[0], c[1], c[2], c[3]);
  codes[1] = make_uint4(c[4], c[5], c[6], c[7]);
  return e;
}

// One warp per (row, 1024-value segment).
template <bool BF16>
__global__ void __launch_bounds__(kWarps * 32)
    quant_groups_kernel(const void* __restrict__ x, int64_t n, int K, uint8_t* __restrict__ q,
                        uint8_t* __restrict__ scales) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  const int lane = threadIdx.x & 31;
  const int segs = (K + kSeg - 1) / kSeg;
  const int64_t items = n * segs;
  const int64_t eb = BF16 ? 2 : 4;
  for (int64_t w = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); w < items;
       w += (int64_t)gridDim.x * kWarps) {
    const int64_t r = w / segs;
    const int64_t e0 = (w - r * segs) * kSeg + lane * 32;
    const bool have = e0 < K;  // whole quads: K is a multiple of 128
    float v[32];
    if (have)
      load32<BF16>(static_cast<const uint8_t*>(x) + r * K * eb, e0, v);
    else
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
    uint4 c[2];
    const int e = quantise32(v, c);
    if (have) {
      uint4* dst = reinterpret_cast<uint4*>(q + r * K + e0);
      dst[0] = c[0];
      dst[1] = c[1];
      if ((lane & 3) == 0) scales[r * (K / 128) + e0 / 128] = (uint8_t)(e + 127);
    }
  }
}

// One block of 256 threads per 128 x 128 block; thread t covers row t/2,
// columns (t%2)*64 .. +63 of the block.
template <bool BF16>
__global__ void __launch_bounds__(256)
    quant_blocks_kernel(const void* __restrict__ w, int K, uint8_t* __restrict__ q,
                        uint8_t* __restrict__ scales) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  __shared__ float wmax[8];
  const int br = blockIdx.y, bc = blockIdx.x, t = threadIdx.x;
  const int64_t r = (int64_t)br * 128 + (t >> 1);
  const int64_t c0 = (int64_t)bc * 128 + (t & 1) * 64;
  const int64_t eb = BF16 ? 2 : 4;
  const uint8_t* row = static_cast<const uint8_t*>(w) + r * K * eb;
  float v[64];
  {
    float a[32];
    load32<BF16>(row, c0, a);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = a[i];
    load32<BF16>(row, c0 + 32, a);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[32 + i] = a[i];
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((t & 31) == 0) wmax[t >> 5] = amax;
  __syncthreads();
  amax = wmax[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, wmax[i]);
  const int e = fp8_scale_exp(amax);
  const float inv = pow2i(-e);
  uint4* dst = reinterpret_cast<uint4*>(q + r * K + c0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float* s = v + 16 * i;
    dst[i] = make_uint4(e4m3x4(s[0] * inv, s[1] * inv, s[2] * inv, s[3] * inv),
                        e4m3x4(s[4] * inv, s[5] * inv, s[6] * inv, s[7] * inv),
                        e4m3x4(s[8] * inv, s[9] * inv, s[10] * inv, s[11] * inv),
                        e4m3x4(s[12] * inv, s[13] * inv, s[14] * inv, s[15] * inv));
  }
  if (t == 0) scales[(int64_t)br * (K / 128) + bc] = (uint8_t)(e + 127);
}

// Dispatch copy with quantisation: one warp per (source row, segment); the
// segment is quantised once and written to the row's k destinations.
template <bool BF16>
__global__ void __launch_bounds__(kWarps * 32)
    dispatch_copy_fp8_kernel(const void* __restrict__ xg, const int32_t* __restrict__ inv,
                             int64_t rows, int k, int H, int64_t cap, uint8_t* __restrict__ xq,
                             uint8_t* __restrict__ xscale) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  const int lane = threadIdx.x & 31;
  const int segs = (H + kSeg - 1) / kSeg;
  const int64_t items = rows * segs;
  const int64_t eb = BF16 ? 2 : 4;
  for (int64_t w = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); w < items;
       w += (int64_t)gridDim.x * kWarps) {
    const int64_t g = w / segs;
    const int64_t e0 = (w - g * segs) * kSeg + lane * 32;
    int32_t my_d = lane < k ? inv[g * k + lane] : -1;
    if (my_d >= cap) my_d = -1;
    if (__ballot_sync(0xffffffffu, my_d >= 0) == 0) continue;  // pad row
    const bool have = e0 < H;
    float v[32];
    if (have)
      load32<BF16>(static_cast<const uint8_t*>(xg) + g * H * eb, e0, v);
    else
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.0f;
    uint4 c[2];
    const int e = quantise32(v, c);
    for (int j = 0; j < k; ++j) {
      const int32_t d = __shfl_sync(0xffffffffu, my_d, j);
      if (d < 0 || !have) continue;
      uint4* dst = reinterpret_cast<uint4*>(xq + (int64_t)d * H + e0);
      dst[0] = c[0];
      dst[1] = c[1];
      if ((lane & 3) == 0) xscale[(int64_t)d * (H / 128) + e0 / 128] = (uint8_t)(e + 127);
    }
  }
}

// Alignment padding rows: zero codes, scale byte 127 (2^0).
__global__ void __launch_bounds__(256)
    dispatch_pad_fp8_kernel(const int32_t* __restrict__ counts_P,
                            const int32_t* __restrict__ offsets_P, int P, int H, int64_t cap,
                            uint8_t* __restrict__ xq, uint8_t* __restrict__ xscale) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  const int s = blockIdx.x;
  if (s >= P) return;
  int64_t a = (int64_t)offsets_P[s] + counts_P[s];
  int64_t b = offsets_P[s + 1];
  if (b > cap) b = cap;
  const int vpr = H / 16;
  for (int64_t d = a; d < b; ++d) {
    uint4* row = reinterpret_cast<uint4*>(xq + d * H);
    for (int v = threadIdx.x; v < vpr; v += blockDim.x) row[v] = make_uint4(0, 0, 0, 0);
    for (int g = threadIdx.x; g < H / 128; g += blockDim.x) xscale[d * (H / 128) + g] = 127;
  }
}

int grid_for(int64_t items) {
  const int64_t want = (items + kWarps - 1) / kWarps;
  const int64_t lim = (int64_t)num_sms() * 8;
  return (int)(want < lim ? (want > 0 ? want : 1) : lim);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_quantize_fp8_groups(const void* d_x, int64_t n, int K, int dtype,
                                              uint8_t* d_q, uint8_t* d_scales, void* stream) {
  if (n < 0 || K < 128 || K % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (dtype_bytes(dtype) == 0) return MOE_ERR_UNSUPPORTED;
  if (n == 0) return MOE_OK;
  if (d_x == nullptr || d_q == nullptr || d_scales == nullptr || !aligned16(d_x) || !aligned16(d_q))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  const int64_t items = n * ((K + kSeg - 1) / kSeg);
  if (dtype == MOE_BF16)
    launch(quant_groups_kernel<true>, grid_for(items), kWarps * 32, 0, s, d_x, n, K, d_q, d_scales);
  else
    launch(quant_groups_kernel<false>, grid_for(items), kWarps * 32, 0, s, d_x, n, K, d_q,
           d_scales);
  return launch_status();
}

extern "C" moe_status moe_quantize_fp8_blocks(const void* d_w, int64_t R, int K, int dtype,
                                              uint8_t* d_q, uint8_t* d_scales, void* stream) {
  if (R < 0 || R % 128 != 0 || K < 128 || K % 128 != 0 || R / 128 > 65535)
    return MOE_ERR_INVALID_ARG;
  if (dtype_bytes(dtype) == 0) return MOE_ERR_UNSUPPORTED;
  if (R == 0) return MOE_OK;
  if (d_w == nullptr || d_q == nullptr || d_scales == nullptr || !aligned16(d_w) || !aligned16(d_q))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  dim3 grid((unsigned)(K / 128), (unsigned)(R / 128));
  if (dtype == MOE_BF16)
    launch(quant_blocks_kernel<true>, grid, 256, 0, s, d_w, K, d_q, d_scales);
  else
    launch(quant_blocks_kernel<false>, grid, 256, 0, s, d_w, K, d_q, d_scales);
  return launch_status();
}

extern "C" moe_status moe_dispatch_fp8(const void* d_global, const int32_t* d_ids, int64_t rows,
                                       int k, int H, int dtype, int E, int P,
                                       const int32_t* d_l2p, const int32_t* d_nrep, int X,
                                       int align, int64_t cap, int32_t* d_counts_P,
                                       int32_t* d_offsets_P, int32_t* d_perm, int32_t* d_inv,
                                       uint8_t* d_sorted_q, uint8_t* d_sorted_scales, void* d_ws,
                                       size_t ws_bytes, uint32_t* d_status, void* stream) {
  if (H < 128 || H % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (dtype_bytes(dtype) == 0) return MOE_ERR_UNSUPPORTED;
  if (rows > 0 && (d_global == nullptr || !aligned16(d_global))) return MOE_ERR_INVALID_ARG;
  if (cap > 0 && (d_sorted_q == nullptr || d_sorted_scales == nullptr || !aligned16(d_sorted_q)))
    return MOE_ERR_INVALID_ARG;
  // counts, offsets, permutation and inverse map (no rows moved)
  moe_status st = moe_dispatch(nullptr, d_ids, rows, k, H, dtype, E, P, d_l2p, d_nrep, X, align,
                               cap, d_counts_P, d_offsets_P, d_perm, d_inv, nullptr, d_ws,
                               ws_bytes, d_status, stream);
  if (st != MOE_OK) return st;
  cudaStream_t s = as_stream(stream);
  if (rows > 0) {
    const int64_t items = rows * ((H + kSeg - 1) / kSeg);
    if (dtype == MOE_BF16)
      launch(dispatch_copy_fp8_kernel<true>, grid_for(items), kWarps * 32, 0, s, d_global, d_inv,
             rows, k, H, cap, d_sorted_q, d_sorted_scales);
    else
      launch(dispatch_copy_fp8_kernel<false>, grid_for(items), kWarps * 32, 0, s, d_global, d_inv,
             rows, k, H, cap, d_sorted_q, d_sorted_scales);
  }
  if (align > 1 && cap > 0)
    launch(dispatch_pad_fp8_kernel, P, 256, 0, s, d_counts_P, d_offsets_P, P, H, cap, d_sorted_q,
           d_sorted_scales);
  return launch_status();
}

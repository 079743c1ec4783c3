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
// Design: one warp per (output row, segment of 64 16-byte vectors); the k
// source rows are read kBatch at a time with every load of a batch in flight
// and accumulated in registers.
//
// moe_combine_scatter runs the DP scatter in the same kernel (SGLang chapter
// 17, section "scatter: 把 MoE 的输出还回本副本"): a combined row of replica r's
// segment goes straight to replica r's output, so the global buffer need not
// be written and read back; pad rows are then skipped.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kUnroll = 2;                // 16-byte vectors per lane per segment
constexpr int kSegVecs = 32 * kUnroll;    // vectors per warp segment of a row
constexpr int kBatch = 4;                 // source rows loaded together

__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <bool BF16>
__device__ __forceinline__ void fma_vec(float* acc, const uint4& t, float wj) {
  const uint32_t q[4] = {t.x, t.y, t.z, t.w};
  if (BF16) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc[2 * e] = fmaf(wj, bf16lo(q[e]), acc[2 * e]);
      acc[2 * e + 1] = fmaf(wj, bf16hi(q[e]), acc[2 * e + 1]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] = fmaf(wj, __uint_as_float(q[e]), acc[e]);
  }
}

// One warp per (output row, segment of 64 vectors).  Source rows are taken
// kBatch at a time with all kBatch x kUnroll loads in flight, then added in j
// order, so the result does not depend on the batching.
// Replica outputs of the fused scatter (SCATTER = true).
struct ScatterArgs {
  ReplicaPtrs dst;
  const int32_t* counts;
  const int32_t* offsets;
  int R;
};

template <bool BF16, bool SCATTER>
__global__ void __launch_bounds__(kWarps * 32)
    combine_kernel(const uint4* __restrict__ ys, const int32_t* __restrict__ inv,
                   const float* __restrict__ w, int64_t rows, int k, int vpr, int64_t cap,
                   uint4* __restrict__ out, const __grid_constant__ ScatterArgs sc,
                   uint32_t* status) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  constexpr int EPV = BF16 ? 8 : 4;  // elements per 16-byte vector
  __shared__ int32_t s_off[SCATTER ? MOE_MAX_REPLICAS + 1 : 1];
  __shared__ int32_t s_cnt[SCATTER ? MOE_MAX_REPLICAS : 1];
  if (SCATTER) {
    for (int i = threadIdx.x; i <= sc.R; i += blockDim.x) {
      s_off[i] = sc.offsets[i];
      if (i < sc.R) s_cnt[i] = sc.counts[i];
    }
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  const int segs = (vpr + kSegVecs - 1) / kSegVecs;
  const int64_t items = rows * segs;
  for (int64_t item = warp0; item < items; item += nwarps) {
    const int64_t g = item / segs;
    const int v0 = (int)(item - g * segs) * kSegVecs;
    uint4* rdst = nullptr;  // the row in its replica's output (fused scatter)
    if (SCATTER) {
      const int r = find_segment(s_off, sc.R, g);
      const int64_t i = g - s_off[r];
      const int64_t seg = (int64_t)s_off[r + 1] - s_off[r];
      int64_t c = s_cnt[r];
      if (c > seg) {
        if (i == 0 && v0 == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
        c = seg;
      }
      if (c > 0 && sc.dst.p[r] == nullptr) {
        if (i == 0 && v0 == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
        c = 0;
      }
      if (i >= 0 && i < c)
        rdst = static_cast<uint4*>(const_cast<void*>(sc.dst.p[r])) + i * vpr;
      else if (out == nullptr)
        continue;  // a pad row with nowhere to go
    }
    int32_t my_d = -1;
    float my_w = 0.f;
    if (lane < k) {
      my_d = inv[g * k + lane];
      my_w = w[g * k + lane];
      if (my_d >= cap) {
        if (v0 == 0) flag(status, MOE_DEV_BAD_COUNTS);
        my_d = -1;
      }
    }
    float acc[kUnroll][EPV];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int e = 0; e < EPV; ++e) acc[u][e] = 0.f;
    for (int j0 = 0; j0 < k; j0 += kBatch) {
      uint4 t[kBatch][kUnroll];
      int32_t d[kBatch];
      float wj[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int j = j0 + b;
        d[b] = __shfl_sync(0xffffffffu, my_d, j & 31);
        wj[b] = __shfl_sync(0xffffffffu, my_w, j & 31);
        if (j >= k) d[b] = -1;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + u * 32 + lane;
          t[b][u] = make_uint4(0, 0, 0, 0);
          if (d[b] >= 0 && v < vpr) t[b][u] = ld_nc(ys + (int64_t)d[b] * vpr + v);
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (d[b] < 0) continue;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) fma_vec<BF16>(acc[u], t[b][u], wj[b]);
      }
    }
    uint4* dst = out != nullptr ? out + g * vpr : nullptr;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = v0 + u * 32 + lane;
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
      if (dst != nullptr) dst[v] = r;
      if (SCATTER && rdst != nullptr) rdst[v] = r;
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
  const int64_t items = rows * ((vpr + kSegVecs - 1) / kSegVecs);
  int64_t want = (items + kWarps - 1) / kWarps;
  int64_t lim = (int64_t)num_sms() * 8;
  int grid = (int)(want < lim ? want : lim);
  cudaStream_t s = as_stream(stream);
  ScatterArgs none = {};
  if (dtype == MOE_BF16)
    launch(combine_kernel<true, false>, grid, kWarps * 32, 0, s,
           static_cast<const uint4*>(d_out_sorted), d_inv, d_w, rows, k, vpr, cap,
           static_cast<uint4*>(d_global_out), none, d_status);
  else
    launch(combine_kernel<false, false>, grid, kWarps * 32, 0, s,
           static_cast<const uint4*>(d_out_sorted), d_inv, d_w, rows, k, vpr, cap,
           static_cast<uint4*>(d_global_out), none, d_status);
  return launch_status();
}

extern "C" moe_status moe_combine_scatter(const void* d_out_sorted, const int32_t* d_inv,
                                          const float* d_w, int64_t rows, int k, int H, int dtype,
                                          int64_t cap, const int32_t* d_counts,
                                          const int32_t* d_offsets, int R, void* const* local,
                                          void* d_global_out, uint32_t* d_status, void* stream) {
  if (rows < 0 || rows > INT32_MAX || k < 1 || k > MOE_MAX_TOPK || H < 1 || cap < 0 || R < 1 ||
      R > MOE_MAX_REPLICAS)
    return MOE_ERR_INVALID_ARG;
  int eb = dtype_bytes(dtype);
  if (eb == 0) return MOE_ERR_UNSUPPORTED;
  if (((int64_t)H * eb) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (d_inv == nullptr || d_w == nullptr || d_counts == nullptr || d_offsets == nullptr ||
      local == nullptr || (d_out_sorted == nullptr && cap > 0))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(d_out_sorted) || (d_global_out != nullptr && !aligned16(d_global_out)))
    return MOE_ERR_INVALID_ARG;
  ScatterArgs sc;
  for (int r = 0; r < R; ++r) {
    if (local[r] != nullptr && !aligned16(local[r])) return MOE_ERR_INVALID_ARG;
    sc.dst.p[r] = local[r];
  }
  sc.counts = d_counts;
  sc.offsets = d_offsets;
  sc.R = R;
  const int vpr = (int)((int64_t)H * eb / 16);
  const int64_t items = rows * ((vpr + kSegVecs - 1) / kSegVecs);
  int64_t want = (items + kWarps - 1) / kWarps;
  int64_t lim = (int64_t)num_sms() * 8;
  int grid = (int)(want < lim ? want : lim);
  cudaStream_t s = as_stream(stream);
  if (dtype == MOE_BF16)
    launch(combine_kernel<true, true>, grid, kWarps * 32, 0, s,
           static_cast<const uint4*>(d_out_sorted), d_inv, d_w, rows, k, vpr, cap,
           static_cast<uint4*>(d_global_out), sc, d_status);
  else
    launch(combine_kernel<false, true>, grid, kWarps * 32, 0, s,
           static_cast<const uint4*>(d_out_sorted), d_inv, d_w, rows, k, vpr, cap,
           static_cast<uint4*>(d_global_out), sc, d_status);
  return launch_status();
}

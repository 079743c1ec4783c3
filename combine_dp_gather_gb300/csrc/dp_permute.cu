// DP gather and DP scatter: packed row copies between the replicas' token
// segments and the global buffer.
//
// SGLang chapter 17, section "两种 gather: all_reduce 与 all_gather": the
// global buffer is zero-filled and each replica writes its rows at its start
// row; on one device the all-reduce that follows adds nothing, so the gather
// is a copy plus zero padding.  Section "scatter: 把 MoE 的输出还回本副本":
// the scatter cuts the buffer back by the same counts.
//
// Design: one warp per (row, segment of 32 x kUnroll 16-byte vectors), so a
// 14 KB row is spread over 7 warps and every lane has all its loads in flight
// at once (one memory round trip per segment); replica pointers travel by
// value in the kernel arguments, counts and offsets are read once per block
// into shared memory.
//
// The gather can also route its rows on the way (moe_dp_gather_route): one
// warp per global row takes the top-k of the row's router logits straight from
// its replica (route_row.cuh), so the routing needs no launch of its own.
#include "common.cuh"
#include "route_row.cuh"

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

constexpr int kSegVecs = 32 * kUnroll;  // vectors per warp segment

// Copy (src != nullptr) or zero one warp segment [v0, v0 + kSegVecs) of a row.
__device__ __forceinline__ void copy_seg(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                         int v0, int vpr, int lane) {
  uint4 t[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    int v = v0 + u * 32 + lane;
    t[u] = make_uint4(0, 0, 0, 0);
    if (src != nullptr && v < vpr) t[u] = ld_nc(src + v);
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    int v = v0 + u * 32 + lane;
    if (v < vpr) dst[v] = t[u];
  }
}

// One row tensor of the gather: the replicas' pointers, 16-byte vectors per
// row, the global buffer.  A plane with vpr == 0 is absent.
struct GatherPlane {
  ReplicaPtrs src;
  int vpr;
  uint4* global;
};

// Routing of the gathered rows from the replicas' router logits (float32
// [counts[r], E] per replica) into ids / w [rows, k + n_shared].
struct RoutePlan {
  ReplicaPtrs src;
  int E, k, n_shared, renorm;
  int32_t* ids;
  float* w;
};

// Routing of global row g (row i of replica r, whose first c rows are real) by
// one warp; rows of a replica without a logits pointer are flagged and padded.
template <int EPL>
__device__ __forceinline__ void route_global_row(const RoutePlan& rt, int r, int64_t i, int64_t c,
                                                 int64_t g, int lane, uint32_t* status) {
  const int kk = rt.k + rt.n_shared;
  bool real = i >= 0 && i < c;
  if (real && rt.src.p[r] == nullptr) {
    if (i == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
    real = false;
  }
  if (real)
    route_row<(EPL > 0 ? EPL : 1)>(static_cast<const float*>(rt.src.p[r]) + i * rt.E, rt.E, rt.k,
                                   rt.n_shared, rt.renorm, rt.ids + g * kk, rt.w + g * kk, lane);
  else
    route_pad_row(kk, rt.ids + g * kk, rt.w + g * kk, lane);
}

// Items are (global row, segment) over the segments of plane a then plane b,
// so one launch gathers two row tensors of the same replicas (hidden states
// and router logits) with the same per-row replica lookup.  With EPL > 0 the
// first `rows` items are the rows' routing (one warp each; EPL experts per lane).
template <int EPL>
__global__ void __launch_bounds__(kWarps * 32)
    dp_gather_kernel(const __grid_constant__ GatherPlane a, const __grid_constant__ GatherPlane b,
                     const __grid_constant__ RoutePlan rt, const int32_t* __restrict__ counts,
                     const int32_t* __restrict__ offsets, int R, int64_t rows,
                     uint32_t* status) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
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
  const int segs_a = (a.vpr + kSegVecs - 1) / kSegVecs;
  const int segs = segs_a + (b.vpr + kSegVecs - 1) / kSegVecs;
  const int64_t route_items = EPL > 0 ? rows : 0;
  const int64_t items = route_items + rows * segs;
  for (int64_t w = warp0; w < items; w += nwarps) {
    if (EPL > 0 && w < route_items) {
      const int64_t g = w;
      const int r = find_segment(s_off, R, g);
      const int64_t i = g - s_off[r];
      const int64_t seg = (int64_t)s_off[r + 1] - s_off[r];
      int64_t c = s_cnt[r];
      if (c > seg) {
        if (i == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
        c = seg;
      }
      route_global_row<EPL>(rt, r, i, c, g, lane, status);
      continue;
    }
    const int64_t wi = w - route_items;
    const int64_t g = wi / segs;
    const int j = (int)(wi - g * segs);
    const GatherPlane& pl = j < segs_a ? a : b;
    const int v0 = (j < segs_a ? j : j - segs_a) * kSegVecs;
    int r = find_segment(s_off, R, g);
    int64_t i = g - s_off[r];
    int64_t seg = (int64_t)s_off[r + 1] - s_off[r];
    int64_t c = s_cnt[r];
    if (c > seg) {
      if (i == 0 && v0 == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
      c = seg;
    }
    if (c > 0 && pl.src.p[r] == nullptr) {
      if (i == 0 && v0 == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
      c = 0;
    }
    const uint4* from =
        (i >= 0 && i < c) ? static_cast<const uint4*>(pl.src.p[r]) + i * pl.vpr : nullptr;
    copy_seg(from, pl.global + g * pl.vpr, v0, pl.vpr, lane);
  }
}

__global__ void __launch_bounds__(kWarps * 32)
    dp_scatter_kernel(const uint4* __restrict__ global, const int32_t* __restrict__ counts,
                      const int32_t* __restrict__ offsets, int R, int64_t rows, int vpr,
                      ReplicaPtrs dst, uint32_t* status) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
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
  const int segs = (vpr + kSegVecs - 1) / kSegVecs;
  const int64_t items = rows * segs;
  for (int64_t w = warp0; w < items; w += nwarps) {
    const int64_t g = w / segs;
    const int v0 = (int)(w - g * segs) * kSegVecs;
    int r = find_segment(s_off, R, g);
    int64_t i = g - s_off[r];
    int64_t seg = (int64_t)s_off[r + 1] - s_off[r];
    int64_t c = s_cnt[r];
    if (c > seg) {
      if (i == 0 && v0 == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
      c = seg;
    }
    if (c > 0 && dst.p[r] == nullptr) {
      if (i == 0 && v0 == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
      c = 0;
    }
    if (i >= 0 && i < c)
      copy_seg(global + g * vpr, static_cast<uint4*>(const_cast<void*>(dst.p[r])) + i * vpr, v0,
               vpr, lane);
  }
}

// ------------------------------------------------------------------ fused
// Residual add + RMSNorm + DP gather (SGLang chapter 17, section "边界判定的融合",
// _reduce_update_read_dp_gather: update the residual with the hidden states,
// read the FFN input as RMSNorm of the updated residual, then gather it).
// One block per global row; each thread keeps up to kNormVecs 16-byte vectors
// of the row in registers, so the row is read once and written twice
// (updated residual, normed row in the global buffer).
constexpr int kNormThreads = 256;
constexpr int kNormVecs = 4;  // 16-byte vectors per thread: rows up to 16 KB

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const uint32_t q[4] = {v.x, v.y, v.z, v.w};
  if (BF16) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = bf16lo(q[e]);
      f[2 * e + 1] = bf16hi(q[e]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) f[e] = __uint_as_float(q[e]);
  }
}
template <bool BF16>
__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 r;
  if (BF16) {
    r.x = pack_bf16x2(f[0], f[1]);
    r.y = pack_bf16x2(f[2], f[3]);
    r.z = pack_bf16x2(f[4], f[5]);
    r.w = pack_bf16x2(f[6], f[7]);
  } else {
    r.x = __float_as_uint(f[0]);
    r.y = __float_as_uint(f[1]);
    r.z = __float_as_uint(f[2]);
    r.w = __float_as_uint(f[3]);
  }
  return r;
}

template <bool BF16, int EPL>
__global__ void __launch_bounds__(kNormThreads)
    dp_gather_add_rmsnorm_kernel(const __grid_constant__ ReplicaPtrs hidden,
                                 const __grid_constant__ ReplicaPtrs residual,
                                 const uint4* __restrict__ gamma, float eps,
                                 const int32_t* __restrict__ counts,
                                 const int32_t* __restrict__ offsets, int R, int64_t rows, int H,
                                 int vpr, uint4* __restrict__ global,
                                 const __grid_constant__ GatherPlane side,
                                 const __grid_constant__ RoutePlan rt, uint32_t* status) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  constexpr int EPV = BF16 ? 8 : 4;
  __shared__ int32_t s_off[MOE_MAX_REPLICAS + 1];
  __shared__ int32_t s_cnt[MOE_MAX_REPLICAS];
  __shared__ float s_part[kNormThreads / 32];
  for (int i = threadIdx.x; i <= R; i += blockDim.x) {
    s_off[i] = offsets[i];
    if (i < R) s_cnt[i] = counts[i];
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int64_t g = blockIdx.x; g < rows; g += gridDim.x) {
    const int r = find_segment(s_off, R, g);
    const int64_t i = g - s_off[r];
    int64_t c = s_cnt[r];
    const int64_t seg = (int64_t)s_off[r + 1] - s_off[r];
    if (c > seg) {
      if (i == 0 && threadIdx.x == 0) flag(status, MOE_DEV_BAD_COUNTS);
      c = seg;
    }
    if (c > 0 && (hidden.p[r] == nullptr || residual.p[r] == nullptr)) {
      if (i == 0 && threadIdx.x == 0) flag(status, MOE_DEV_BAD_COUNTS);
      c = 0;
    }
    uint4* dst = global + g * vpr;
    // the side plane (router logits) of the same row: copied, or zero for a pad row
    if (side.vpr > 0) {
      const bool real = i >= 0 && i < c;
      const bool have = real && side.src.p[r] != nullptr;
      if (real && !have && i == 0 && threadIdx.x == 0) flag(status, MOE_DEV_BAD_COUNTS);
      const uint4* srow = have ? static_cast<const uint4*>(side.src.p[r]) + i * side.vpr : nullptr;
      for (int v = threadIdx.x; v < side.vpr; v += blockDim.x)
        side.global[g * side.vpr + v] = srow != nullptr ? ld_nc(srow + v) : make_uint4(0, 0, 0, 0);
    }
    if (!(i >= 0 && i < c)) {  // pad row (block-uniform)
      for (int v = threadIdx.x; v < vpr; v += blockDim.x) dst[v] = make_uint4(0, 0, 0, 0);
      if (EPL > 0 && wid == kNormThreads / 32 - 1) route_global_row<EPL>(rt, r, i, c, g, lane, status);
      continue;
    }
    const uint4* hrow = static_cast<const uint4*>(hidden.p[r]) + i * vpr;
    uint4* rrow = static_cast<uint4*>(const_cast<void*>(residual.p[r])) + i * vpr;
    float x[kNormVecs][EPV];
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < kNormVecs; ++u) {
      const int v = threadIdx.x + u * kNormThreads;
      if (v < vpr) {
        float a[EPV], b[EPV];
        unpack8<BF16>(hrow[v], a);
        unpack8<BF16>(rrow[v], b);
#pragma unroll
        for (int e = 0; e < EPV; ++e) x[u][e] = a[e] + b[e];   // float32 add
        const uint4 stored = pack8<BF16>(x[u]);                   // round once
        rrow[v] = stored;                                          // updated residual
        unpack8<BF16>(stored, x[u]);                               // the norm reads it
#pragma unroll
        for (int e = 0; e < EPV; ++e) ss = fmaf(x[u][e], x[u][e], ss);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) s_part[wid] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += s_part[w];
    __syncthreads();  // s_part is reused by the next row
    const float inv = rsqrtf(tot / (float)H + eps);
#pragma unroll
    for (int u = 0; u < kNormVecs; ++u) {
      const int v = threadIdx.x + u * kNormThreads;
      if (v < vpr) {
        float gm[EPV], y[EPV];
        unpack8<BF16>(gamma[v], gm);
#pragma unroll
        for (int e = 0; e < EPV; ++e) y[e] = x[u][e] * inv * gm[e];
        dst[v] = pack8<BF16>(y);
      }
    }
    // the row's routing by the last warp, from the replica's logits
    if (EPL > 0 && wid == kNormThreads / 32 - 1) route_global_row<EPL>(rt, r, i, c, g, lane, status);
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

bool make_plane(const void* const* local, int R, int H, int dtype, void* d_global,
                GatherPlane* pl) {
  if (local == nullptr) return false;
  for (int r = 0; r < R; ++r) {
    if (local[r] != nullptr && !aligned16(local[r])) return false;
    pl->src.p[r] = local[r];
  }
  pl->vpr = (int)((int64_t)H * dtype_bytes(dtype) / 16);
  pl->global = static_cast<uint4*>(d_global);
  return true;
}

int segments(int vpr) { return (vpr + kSegVecs - 1) / kSegVecs; }

int grid_for_items(int64_t items) {
  int64_t want = (items + kWarps - 1) / kWarps;
  int64_t cap = (int64_t)num_sms() * 8;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

int grid_for_rows(int64_t rows, int vpr, int vpr2 = 0) {
  return grid_for_items(rows * (segments(vpr) + segments(vpr2)));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_dp_gather(const void* const* local, const int32_t* d_counts,
                                    const int32_t* d_offsets, int R, int64_t rows, int H,
                                    int dtype, void* d_global, uint32_t* d_status, void* stream) {
  moe_status st = check_common(d_counts, d_offsets, R, rows, H, dtype, d_global);
  if (st != MOE_OK || rows == 0) return st;
  GatherPlane a, b;
  if (!make_plane(local, R, H, dtype, d_global, &a)) return MOE_ERR_INVALID_ARG;
  b.vpr = 0;
  b.global = nullptr;
  launch(dp_gather_kernel<0>, grid_for_rows(rows, a.vpr), kWarps * 32, 0, as_stream(stream), a,
         b, RoutePlan{}, d_counts, d_offsets, R, rows, d_status);
  return launch_status();
}

extern "C" moe_status moe_dp_gather2(const void* const* local_a, int H_a, int dtype_a,
                                     void* d_global_a, const void* const* local_b, int H_b,
                                     int dtype_b, void* d_global_b, const int32_t* d_counts,
                                     const int32_t* d_offsets, int R, int64_t rows,
                                     uint32_t* d_status, void* stream) {
  moe_status st = check_common(d_counts, d_offsets, R, rows, H_a, dtype_a, d_global_a);
  if (st != MOE_OK) return st;
  st = check_common(d_counts, d_offsets, R, rows, H_b, dtype_b, d_global_b);
  if (st != MOE_OK || rows == 0) return st;
  GatherPlane a, b;
  if (!make_plane(local_a, R, H_a, dtype_a, d_global_a, &a) ||
      !make_plane(local_b, R, H_b, dtype_b, d_global_b, &b))
    return MOE_ERR_INVALID_ARG;
  launch(dp_gather_kernel<0>, grid_for_rows(rows, a.vpr, b.vpr), kWarps * 32, 0,
         as_stream(stream), a, b, RoutePlan{}, d_counts, d_offsets, R, rows, d_status);
  return launch_status();
}

extern "C" moe_status moe_dp_gather_route(const void* const* local_x, int H, int dtype,
                                          void* d_global_x, const void* const* local_logits, int E,
                                          void* d_global_logits, int k, int renormalize,
                                          int n_shared, const int32_t* d_counts,
                                          const int32_t* d_offsets, int R, int64_t rows,
                                          int32_t* d_ids, float* d_w, uint32_t* d_status,
                                          void* stream) {
  moe_status st = check_common(d_counts, d_offsets, R, rows, H, dtype, d_global_x);
  if (st != MOE_OK) return st;
  if (E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E || n_shared < 0 ||
      k + n_shared > MOE_MAX_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (d_global_logits != nullptr) {
    st = check_common(d_counts, d_offsets, R, rows, E, MOE_F32, d_global_logits);
    if (st != MOE_OK) return st;
  }
  if (rows == 0) return MOE_OK;
  if (local_logits == nullptr || d_ids == nullptr || d_w == nullptr) return MOE_ERR_INVALID_ARG;
  GatherPlane a, b;
  if (!make_plane(local_x, R, H, dtype, d_global_x, &a)) return MOE_ERR_INVALID_ARG;
  if (d_global_logits != nullptr) {
    if (!make_plane(local_logits, R, E, MOE_F32, d_global_logits, &b)) return MOE_ERR_INVALID_ARG;
  } else {
    b.vpr = 0;
    b.global = nullptr;
  }
  RoutePlan rt;
  for (int r = 0; r < R; ++r) {
    if (reinterpret_cast<uintptr_t>(local_logits[r]) % alignof(float) != 0)
      return MOE_ERR_INVALID_ARG;
    rt.src.p[r] = local_logits[r];
  }
  rt.E = E;
  rt.k = k;
  rt.n_shared = n_shared;
  rt.renorm = renormalize != 0;
  rt.ids = d_ids;
  rt.w = d_w;
  const int grid = grid_for_items(rows * (1 + segments(a.vpr) + segments(b.vpr)));
  cudaStream_t s = as_stream(stream);
  switch (route_epl(E)) {
    case 1:
      launch(dp_gather_kernel<1>, grid, kWarps * 32, 0, s, a, b, rt, d_counts, d_offsets, R, rows,
             d_status);
      break;
    case 2:
      launch(dp_gather_kernel<2>, grid, kWarps * 32, 0, s, a, b, rt, d_counts, d_offsets, R, rows,
             d_status);
      break;
    case 4:
      launch(dp_gather_kernel<4>, grid, kWarps * 32, 0, s, a, b, rt, d_counts, d_offsets, R, rows,
             d_status);
      break;
    case 8:
      launch(dp_gather_kernel<8>, grid, kWarps * 32, 0, s, a, b, rt, d_counts, d_offsets, R, rows,
             d_status);
      break;
    case 16:
      launch(dp_gather_kernel<16>, grid, kWarps * 32, 0, s, a, b, rt, d_counts, d_offsets, R,
             rows, d_status);
      break;
    default:
      launch(dp_gather_kernel<32>, grid, kWarps * 32, 0, s, a, b, rt, d_counts, d_offsets, R,
             rows, d_status);
      break;
  }
  return launch_status();
}

namespace moe {
namespace {
template <bool BF16, int EPL>
void launch_norm(int grid, cudaStream_t s, const ReplicaPtrs& hp, const ReplicaPtrs& rp,
                 const void* d_gamma, float eps, const int32_t* d_counts, const int32_t* d_offsets,
                 int R, int64_t rows, int H, int vpr, void* d_global, const GatherPlane& side,
                 const RoutePlan& rt, uint32_t* d_status) {
  launch(dp_gather_add_rmsnorm_kernel<BF16, EPL>, grid, kNormThreads, 0, s, hp, rp,
         static_cast<const uint4*>(d_gamma), eps, d_counts, d_offsets, R, rows, H, vpr,
         static_cast<uint4*>(d_global), side, rt, d_status);
}

template <bool BF16>
void launch_norm_epl(int epl, int grid, cudaStream_t s, const ReplicaPtrs& hp,
                     const ReplicaPtrs& rp, const void* d_gamma, float eps,
                     const int32_t* d_counts, const int32_t* d_offsets, int R, int64_t rows, int H,
                     int vpr, void* d_global, const GatherPlane& side, const RoutePlan& rt,
                     uint32_t* d_status) {
#define MOE_NORM_CASE(N)                                                                       \
  case N:                                                                                      \
    launch_norm<BF16, N>(grid, s, hp, rp, d_gamma, eps, d_counts, d_offsets, R, rows, H, vpr, \
                         d_global, side, rt, d_status);                                        \
    break;
  switch (epl) {
    MOE_NORM_CASE(0)
    MOE_NORM_CASE(1)
    MOE_NORM_CASE(2)
    MOE_NORM_CASE(4)
    MOE_NORM_CASE(8)
    MOE_NORM_CASE(16)
    default:
      launch_norm<BF16, 32>(grid, s, hp, rp, d_gamma, eps, d_counts, d_offsets, R, rows, H, vpr,
                            d_global, side, rt, d_status);
      break;
  }
#undef MOE_NORM_CASE
}

moe_status gather_add_rmsnorm(const void* const* local_hidden, void* const* local_residual,
                              const void* d_gamma, float eps, const GatherPlane& side,
                              const RoutePlan* rt, const int32_t* d_counts,
                              const int32_t* d_offsets, int R, int64_t rows, int H, int dtype,
                              void* d_global, uint32_t* d_status, void* stream) {
  if (local_hidden == nullptr || local_residual == nullptr || d_gamma == nullptr ||
      !aligned16(d_gamma) || !(eps >= 0.f))
    return MOE_ERR_INVALID_ARG;
  const int vpr = (int)((int64_t)H * dtype_bytes(dtype) / 16);
  if (vpr > kNormThreads * kNormVecs) return MOE_ERR_UNSUPPORTED;  // rows above 16 KB
  ReplicaPtrs hp, rp;
  for (int r = 0; r < R; ++r) {
    if ((local_hidden[r] != nullptr && !aligned16(local_hidden[r])) ||
        (local_residual[r] != nullptr && !aligned16(local_residual[r])))
      return MOE_ERR_INVALID_ARG;
    hp.p[r] = local_hidden[r];
    rp.p[r] = local_residual[r];
  }
  const int64_t lim = (int64_t)num_sms() * 8;
  const int grid = (int)(rows < lim ? rows : lim);
  const int epl = rt != nullptr ? route_epl(rt->E) : 0;
  const RoutePlan none{};
  const RoutePlan& plan = rt != nullptr ? *rt : none;
  if (dtype == MOE_BF16)
    launch_norm_epl<true>(epl, grid, as_stream(stream), hp, rp, d_gamma, eps, d_counts, d_offsets,
                          R, rows, H, vpr, d_global, side, plan, d_status);
  else
    launch_norm_epl<false>(epl, grid, as_stream(stream), hp, rp, d_gamma, eps, d_counts,
                           d_offsets, R, rows, H, vpr, d_global, side, plan, d_status);
  return launch_status();
}
}  // namespace
}  // namespace moe

extern "C" moe_status moe_dp_gather_add_rmsnorm(const void* const* local_hidden,
                                                void* const* local_residual, const void* d_gamma,
                                                float eps, const int32_t* d_counts,
                                                const int32_t* d_offsets, int R, int64_t rows,
                                                int H, int dtype, void* d_global,
                                                uint32_t* d_status, void* stream) {
  moe_status st = check_common(d_counts, d_offsets, R, rows, H, dtype, d_global);
  if (st != MOE_OK || rows == 0) return st;
  GatherPlane none;
  none.vpr = 0;
  none.global = nullptr;
  return gather_add_rmsnorm(local_hidden, local_residual, d_gamma, eps, none, nullptr, d_counts,
                            d_offsets, R, rows, H, dtype, d_global, d_status, stream);
}

extern "C" moe_status moe_dp_gather_add_rmsnorm2(const void* const* local_hidden,
                                                 void* const* local_residual, const void* d_gamma,
                                                 float eps, const void* const* local_b, int H_b,
                                                 int dtype_b, void* d_global_b,
                                                 const int32_t* d_counts, const int32_t* d_offsets,
                                                 int R, int64_t rows, int H, int dtype,
                                                 void* d_global, uint32_t* d_status,
                                                 void* stream) {
  moe_status st = check_common(d_counts, d_offsets, R, rows, H, dtype, d_global);
  if (st != MOE_OK) return st;
  st = check_common(d_counts, d_offsets, R, rows, H_b, dtype_b, d_global_b);
  if (st != MOE_OK || rows == 0) return st;
  GatherPlane side;
  if (!make_plane(local_b, R, H_b, dtype_b, d_global_b, &side)) return MOE_ERR_INVALID_ARG;
  return gather_add_rmsnorm(local_hidden, local_residual, d_gamma, eps, side, nullptr, d_counts,
                            d_offsets, R, rows, H, dtype, d_global, d_status, stream);
}

extern "C" moe_status moe_dp_gather_add_rmsnorm_route(
    const void* const* local_hidden, void* const* local_residual, const void* d_gamma, float eps,
    const void* const* local_logits, int E, void* d_global_logits, int k, int renormalize,
    int n_shared, int32_t* d_ids, float* d_w, const int32_t* d_counts, const int32_t* d_offsets,
    int R, int64_t rows, int H, int dtype, void* d_global, uint32_t* d_status, void* stream) {
  moe_status st = check_common(d_counts, d_offsets, R, rows, H, dtype, d_global);
  if (st != MOE_OK) return st;
  if (E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E || n_shared < 0 ||
      k + n_shared > MOE_MAX_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (d_global_logits != nullptr) {
    st = check_common(d_counts, d_offsets, R, rows, E, MOE_F32, d_global_logits);
    if (st != MOE_OK) return st;
  }
  if (rows == 0) return MOE_OK;
  if (local_logits == nullptr || d_ids == nullptr || d_w == nullptr) return MOE_ERR_INVALID_ARG;
  GatherPlane side;
  if (d_global_logits != nullptr) {
    if (!make_plane(local_logits, R, E, MOE_F32, d_global_logits, &side))
      return MOE_ERR_INVALID_ARG;
  } else {
    side.vpr = 0;
    side.global = nullptr;
  }
  RoutePlan rt;
  for (int r = 0; r < R; ++r) {
    if (reinterpret_cast<uintptr_t>(local_logits[r]) % alignof(float) != 0)
      return MOE_ERR_INVALID_ARG;
    rt.src.p[r] = local_logits[r];
  }
  rt.E = E;
  rt.k = k;
  rt.n_shared = n_shared;
  rt.renorm = renormalize != 0;
  rt.ids = d_ids;
  rt.w = d_w;
  return gather_add_rmsnorm(local_hidden, local_residual, d_gamma, eps, side, &rt, d_counts,
                            d_offsets, R, rows, H, dtype, d_global, d_status, stream);
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
  launch(dp_scatter_kernel, grid_for_rows(rows, vpr), kWarps * 32, 0, as_stream(stream),
         static_cast<const uint4*>(d_global), d_counts, d_offsets, R, rows, vpr, ptrs, d_status);
  return launch_status();
}

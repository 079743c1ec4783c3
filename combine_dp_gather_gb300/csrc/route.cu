// Top-k routing: for every real row of the global buffer, the k experts with
// the largest router logits (equal logits: lower id first), best first, and
// their softmax weights.
//
// SGLang chapter 17 names the result TopKOutput{topk_ids, topk_weights}
// (sections "normal dispatch 的调用链" and "Two-batch Overlap"); the scoring
// is softmax routing, renormalised over the k chosen experts unless asked
// otherwise.  Rows past counts[r] inside replica r's segment are padding:
// id -1, weight 0.
//
// Shared experts (vLLM chapter 27, section "共享专家: 在被让出的空档里干活": every
// token also goes through them): expert E + s is listed after the k routed ids
// of every real row with weight 1, so dispatch, the grouped FFN and combine
// treat it as one more slot.
//
// Design: one warp per row (route_row.cuh).
#include "route_row.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;

template <int EPL>
__global__ void __launch_bounds__(kWarps * 32)
    route_topk_kernel(const float* __restrict__ logits, int64_t rows, int E, int k, int renorm,
                      int n_shared, const int32_t* __restrict__ counts,
                      const int32_t* __restrict__ offsets, int R, int32_t* __restrict__ ids,
                      float* __restrict__ w, uint32_t* status) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  const int kk = k + n_shared;  // row stride of ids / w
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
    int64_t c = s_cnt[r];
    int64_t seg = (int64_t)s_off[r + 1] - s_off[r];
    if (c > seg) {
      if (i == 0 && lane == 0) flag(status, MOE_DEV_BAD_COUNTS);
      c = seg;
    }
    if (!(i >= 0 && i < c)) {
      route_pad_row(kk, ids + g * kk, w + g * kk, lane);
      continue;
    }
    route_row<EPL>(logits + g * E, E, k, n_shared, renorm, ids + g * kk, w + g * kk, lane);
  }
}

template <int EPL>
void launch_route(const float* logits, int64_t rows, int E, int k, int renorm, int n_shared,
                  const int32_t* counts, const int32_t* offsets, int R, int32_t* ids, float* w,
                  uint32_t* status, cudaStream_t s) {
  int64_t want = (rows + kWarps - 1) / kWarps;
  int64_t cap = (int64_t)num_sms() * 8;
  int grid = (int)(want < cap ? want : cap);
  launch(route_topk_kernel<EPL>, grid, kWarps * 32, 0, s, logits, rows, E, k, renorm, n_shared,
         counts, offsets, R, ids, w, status);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_route_topk_shared(const float* d_logits, int64_t rows, int E, int k,
                                            int renormalize, int n_shared,
                                            const int32_t* d_counts, const int32_t* d_offsets,
                                            int R, int32_t* d_ids, float* d_w, uint32_t* d_status,
                                            void* stream) {
  if (rows < 0 || rows > INT32_MAX || R < 1 || R > MOE_MAX_REPLICAS) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E || n_shared < 0 ||
      k + n_shared > MOE_MAX_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (d_logits == nullptr || d_counts == nullptr || d_offsets == nullptr || d_ids == nullptr ||
      d_w == nullptr)
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  const int ns = n_shared;
  if (E <= 32)
    launch_route<1>(d_logits, rows, E, k, renormalize, ns, d_counts, d_offsets, R, d_ids, d_w,
                     d_status, s);
  else if (E <= 64)
    launch_route<2>(d_logits, rows, E, k, renormalize, ns, d_counts, d_offsets, R, d_ids, d_w,
                     d_status, s);
  else if (E <= 128)
    launch_route<4>(d_logits, rows, E, k, renormalize, ns, d_counts, d_offsets, R, d_ids, d_w,
                     d_status, s);
  else if (E <= 256)
    launch_route<8>(d_logits, rows, E, k, renormalize, ns, d_counts, d_offsets, R, d_ids, d_w,
                     d_status, s);
  else if (E <= 512)
    launch_route<16>(d_logits, rows, E, k, renormalize, ns, d_counts, d_offsets, R, d_ids, d_w,
                      d_status, s);
  else
    launch_route<32>(d_logits, rows, E, k, renormalize, ns, d_counts, d_offsets, R, d_ids, d_w,
                      d_status, s);
  return launch_status();
}

extern "C" moe_status moe_route_topk(const float* d_logits, int64_t rows, int E, int k,
                                     int renormalize, const int32_t* d_counts,
                                     const int32_t* d_offsets, int R, int32_t* d_ids, float* d_w,
                                     uint32_t* d_status, void* stream) {
  return moe_route_topk_shared(d_logits, rows, E, k, renormalize, 0, d_counts, d_offsets, R,
                               d_ids, d_w, d_status, stream);
}

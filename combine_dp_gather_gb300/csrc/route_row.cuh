// One row of top-k routing by one warp: the k experts with the largest router
// logits (equal logits: lower id first), best first, and their softmax
// weights (renormalised over the k chosen, or the full-softmax probabilities),
// then the shared experts with weight 1.
//
// SGLang chapter 17 names the result TopKOutput{topk_ids, topk_weights}
// (sections "normal dispatch 的调用链" and "Two-batch Overlap"); vLLM chapter 27,
// section "共享专家: 在被让出的空档里干活": every token also goes through the shared
// experts.
//
// Lane l holds experts l, l+32, ... (coalesced 128-byte loads); k rounds of a
// warp arg-max on (logit desc, id asc) pick the experts; lane j keeps the j-th
// pick; the weights use expf in float32 and sum in pick order.  Used by the
// routing kernel and by the DP gather that routes its rows on the way.
#pragma once

#include <float.h>

#include "common.cuh"

namespace moe {

// Experts per lane for E experts (the template argument of route_row).
inline int route_epl(int E) {
  return E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : E <= 512 ? 16 : 32;
}

// Pad row: id -1, weight 0 in every column of ids / w.
__device__ __forceinline__ void route_pad_row(int kk, int32_t* ids_row, float* w_row, int lane) {
  if (lane < kk) {
    ids_row[lane] = -1;
    w_row[lane] = 0.f;
  }
}

// Real row: lr points at its E logits; ids_row / w_row have k + n_shared columns.
template <int EPL>
__device__ __forceinline__ void route_row(const float* __restrict__ lr, int E, int k,
                                          int n_shared, int renorm, int32_t* ids_row,
                                          float* w_row, int lane) {
  const int kk = k + n_shared;
  float v[EPL];
#pragma unroll
  for (int t = 0; t < EPL; ++t) {
    int e = lane + 32 * t;
    v[t] = e < E ? lr[e] : -FLT_MAX;
  }
  uint32_t taken = 0;
  float my_val = 0.f;
  int my_id = -1;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = INT32_MAX;
#pragma unroll
    for (int t = 0; t < EPL; ++t) {
      int e = lane + 32 * t;
      bool cand = e < E && !((taken >> t) & 1u);
      if (cand && (v[t] > bv || (v[t] == bv && e < bi))) {
        bv = v[t];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == (bi & 31)) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_val = bv;
      my_id = bi;
    }
  }
  const float top = __shfl_sync(0xffffffffu, my_val, 0);
  float ex = lane < k ? expf(my_val - top) : 0.f;
  float denom = 0.f;
  if (renorm) {
    for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, ex, j);
  } else {
    float part = 0.f;
#pragma unroll
    for (int t = 0; t < EPL; ++t) {
      int e = lane + 32 * t;
      if (e < E) part += expf(v[t] - top);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    denom = part;
  }
  if (lane < k) {
    ids_row[lane] = my_id;
    w_row[lane] = ex / denom;
  } else if (lane < kk) {  // shared experts: always selected, weight 1
    ids_row[lane] = E + (lane - k);
    w_row[lane] = 1.f;
  }
}

}  // namespace moe

// Host-side helpers of libmoe_dp: global-buffer layout, padding-mode rule,
// status names and workspace sizes.  Pure integer code, no CUDA calls except
// the cached SM count.
#include <cuda_runtime.h>
#include <limits.h>
#include <mutex>
#include <stdint.h>
#include <stdlib.h>

#include "moe_dp.h"

namespace moe {

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("MOE_PDL");
    return !(v != nullptr && v[0] == '0' && v[1] == 0);
  }();
  return on;
}

int num_sms() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace moe

extern "C" {

// SGLang chapter 17, sections "本 rank 的切片位置怎么算" and "DpPaddingMode";
// zdszero "DP", section "跳过同步: 用约定代替通信".
moe_status moe_dp_layout(const int32_t* counts, int R, int mode, int static_bound,
                         int tokens_per_req, int32_t* offsets, int64_t* rows) {
  if (counts == nullptr || offsets == nullptr || rows == nullptr) return MOE_ERR_INVALID_ARG;
  if (R < 1 || R > MOE_MAX_REPLICAS) return MOE_ERR_INVALID_ARG;
  int32_t mx = 0;
  for (int r = 0; r < R; ++r) {
    if (counts[r] < 0) return MOE_ERR_INVALID_ARG;
    if (counts[r] > mx) mx = counts[r];
  }
  int64_t seg = 0;
  if (mode == MOE_PAD_MAX) {
    seg = mx;
  } else if (mode == MOE_PAD_STATIC) {
    if (static_bound < 0 || tokens_per_req < 1) return MOE_ERR_INVALID_ARG;
    seg = (int64_t)static_bound * tokens_per_req;
    if (mx > seg) return MOE_ERR_BOUND_EXCEEDED;
  } else if (mode != MOE_PAD_SUM) {
    return MOE_ERR_INVALID_ARG;
  }
  int64_t pos = 0;
  for (int r = 0; r < R; ++r) {
    if (pos > INT32_MAX) return MOE_ERR_INVALID_ARG;
    offsets[r] = (int32_t)pos;
    pos += (mode == MOE_PAD_SUM) ? counts[r] : seg;
  }
  if (pos > INT32_MAX) return MOE_ERR_INVALID_ARG;
  offsets[R] = (int32_t)pos;
  *rows = pos;
  return MOE_OK;
}

// SGLang chapter 17, section "DpPaddingMode" (get_dp_padding_mode).
int moe_dp_padding_mode(const int32_t* counts, int R, int gather_width, int is_extend_in_batch,
                        int max_len_with_idle) {
  if (counts == nullptr || R < 1) return -1;
  int64_t sum = 0;
  int32_t mx = counts[0], mn = counts[0];
  for (int r = 0; r < R; ++r) {
    if (counts[r] < 0) return -1;
    sum += counts[r];
    mx = counts[r] > mx ? counts[r] : mx;
    mn = counts[r] < mn ? counts[r] : mn;
  }
  if (is_extend_in_batch && gather_width > 1)
    return (max_len_with_idle && mn == 0) ? MOE_PAD_MAX : MOE_PAD_SUM;
  return (2 * sum >= (int64_t)mx * gather_width) ? MOE_PAD_MAX : MOE_PAD_SUM;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_CAPACITY: return "capacity too small";
    case MOE_ERR_BOUND_EXCEEDED: return "static bound exceeded";
    case MOE_ERR_DEVICE_INPUT: return "invalid device input";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_UNSUPPORTED: return "unsupported dtype, shape or device";
    default: return "unknown status";
  }
}

// SGLang chapter 17, section "不均衡的代价与冗余专家的思路" (compute_utilization_rate).
double moe_balancedness(const int64_t* loads, int n) {
  if (loads == nullptr || n < 1) return -1.0;
  int64_t sum = 0, mx = 0;
  for (int i = 0; i < n; ++i) {
    if (loads[i] < 0) return -1.0;
    sum += loads[i];
    mx = loads[i] > mx ? loads[i] : mx;
  }
  const double mean = (double)sum / (double)n;
  return (mean + 1e-5) / ((double)mx + 1e-5);
}

// SGLang chapter 17, section "逻辑与物理的两套映射": contiguous slot ranges per EP rank.
moe_status moe_range_loads(const int32_t* counts, int n, int n_ranges, int64_t* loads) {
  if (counts == nullptr || loads == nullptr || n < 1 || n_ranges < 1 || n % n_ranges != 0)
    return MOE_ERR_INVALID_ARG;
  const int per = n / n_ranges;
  for (int r = 0; r < n_ranges; ++r) {
    int64_t sum = 0;
    for (int i = r * per; i < (r + 1) * per; ++i) {
      if (counts[i] < 0) return MOE_ERR_INVALID_ARG;
      sum += counts[i];
    }
    loads[r] = sum;
  }
  return MOE_OK;
}

// SGLang chapter 17, sections "逻辑与物理的两套映射" and "推理时怎么选副本":
// per-slot counts summed over each logical expert's replicas.
moe_status moe_logical_counts(const int32_t* counts_P, const int32_t* p2l, int P, int E,
                              int64_t* counts_E) {
  if (counts_P == nullptr || p2l == nullptr || counts_E == nullptr || P < 1 || E < 1)
    return MOE_ERR_INVALID_ARG;
  for (int e = 0; e < E; ++e) counts_E[e] = 0;
  for (int s = 0; s < P; ++s) {
    if (counts_P[s] < 0 || p2l[s] < 0 || p2l[s] >= E) return MOE_ERR_INVALID_ARG;
    counts_E[p2l[s]] += counts_P[s];
  }
  return MOE_OK;
}

int64_t moe_dispatch_cap_bound(int64_t rows, int k, int P, int align) {
  if (rows < 0 || k < 1 || P < 1 || align < 1) return -1;
  return rows * k + (int64_t)P * (align - 1);
}

}  // extern "C"

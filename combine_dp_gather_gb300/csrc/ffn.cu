// moe_grouped_ffn entry point and its float32 CUDA-core path.
//
// The float32 path serves fp32 layers (small, latency-bound shapes): one thread
// per output element, float32 accumulation in index order.  bf16 layers go to
// the tcgen05 kernel in ffn_tc.cu.
#include <mutex>

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

// ---------------------------------------------------------------------------
// Grouped FFN with the combine and the DP scatter in the down projection's
// epilogue (vLLM chapter 27, figure "MoE 模块化内核的 PrepareAndFinalize 块结构":
// MM2, then finalize applies the top-k weights; SGLang chapter 17, section
// "scatter: 把 MoE 的输出还回本副本").  Workspace: h [cap, I] in the layer dtype,
// then (bf16) one int32 arrival counter per (global row, 256-feature n-tile).

namespace {

size_t fuse_h_bytes(int64_t cap, int I, int eb) {
  return ((size_t)(cap * (int64_t)I * eb) + 255) & ~(size_t)255;
}

}  // namespace

extern "C" size_t moe_grouped_ffn_combine_ws_bytes(int64_t cap, int64_t rows, int H, int I,
                                                   int dtype) {
  const int eb = dtype_bytes(dtype);
  if (cap < 0 || rows < 0 || H < 1 || I < 1 || eb == 0) return 0;
  if (dtype != MOE_BF16) return fuse_h_bytes(cap, I, eb);  // no counters on the float32 path
  if (H % kFuseBlock != 0) return 0;
  return fuse_h_bytes(cap, I, eb) + (size_t)rows * (size_t)(H / kFuseBlock) * sizeof(int32_t);
}

extern "C" int moe_grouped_ffn_combine_in_epilogue(int64_t cap, int P, int dtype) {
  if (cap < 1 || P < 1 || dtype != MOE_BF16) return 0;
  FfnArgs a = {};
  a.cap = cap;
  a.P = P;
  return ffn_uses_pair_kernel(a) ? 0 : 1;
}

extern "C" moe_status moe_grouped_ffn_combine(
    const void* d_sorted, const int32_t* d_offsets_P, int P, int slot_lo, int slot_hi, int64_t cap,
    const void* d_w_gate_up, const void* d_w_down, int H, int I, int dtype, void* d_out_sorted,
    const int32_t* d_perm, const int32_t* d_inv, const float* d_w, int64_t rows, int k,
    const int32_t* d_counts, const int32_t* d_offsets, int R, void* const* local,
    void* d_global_out, void* d_ws, size_t ws_bytes, uint32_t* d_status, void* stream) {
  if (P < 1 || slot_lo < 0 || slot_hi > P || slot_lo > slot_hi || cap < 0 || cap > INT32_MAX ||
      H < 1 || I < 1 || rows < 0 || rows > INT32_MAX || k < 1 || k > MOE_MAX_TOPK || R < 1 ||
      R > MOE_MAX_REPLICAS)
    return MOE_ERR_INVALID_ARG;
  const int eb = dtype_bytes(dtype);
  if (eb == 0) return MOE_ERR_UNSUPPORTED;
  if (((int64_t)H * eb) % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (dtype == MOE_BF16 && (H % kFuseBlock != 0 || I % 128 != 0 || P > MOE_MAX_SLOTS))
    return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  if (d_inv == nullptr || d_w == nullptr || d_counts == nullptr || d_offsets == nullptr ||
      local == nullptr || d_ws == nullptr || (cap > 0 && (d_sorted == nullptr ||
      d_offsets_P == nullptr || d_w_gate_up == nullptr || d_w_down == nullptr ||
      d_out_sorted == nullptr || d_perm == nullptr)))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_grouped_ffn_combine_ws_bytes(cap, rows, H, I, dtype)) return MOE_ERR_CAPACITY;
  if (!aligned16(d_sorted) || !aligned16(d_out_sorted) || !aligned16(d_ws) ||
      !aligned16(d_w_gate_up) || !aligned16(d_w_down) ||
      (d_global_out != nullptr && !aligned16(d_global_out)))
    return MOE_ERR_INVALID_ARG;
  for (int r = 0; r < R; ++r)
    if (local[r] != nullptr && !aligned16(local[r])) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  void* h = d_ws;
  if (dtype != MOE_BF16) {
    // float32 layers (CUDA-core FFN): the FFN, then the combine + scatter launch
    if (cap > 0 && slot_lo < slot_hi) {
      FfnArgs a{d_sorted, d_offsets_P, P, slot_lo, slot_hi, cap, d_w_gate_up, d_w_down,
                H, I, d_out_sorted, h, d_status};
      const moe_status st = launch_ffn_simt_f32(a, s);
      if (st != MOE_OK) return st;
    }
    return moe_combine_scatter(d_out_sorted, d_inv, d_w, rows, k, H, dtype, cap, d_counts,
                               d_offsets, R, local, d_global_out, d_status, stream);
  }
  if ((int64_t)P * 2 * I > INT32_MAX || (int64_t)P * H > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
  FuseArgs f = {};
  f.perm = d_perm;
  f.inv = d_inv;
  f.w = d_w;
  f.cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(d_ws) + fuse_h_bytes(cap, I, eb));
  f.rows = rows;
  f.kk = k;
  f.nblk = H / kFuseBlock;
  f.H = H;
  f.R = R;
  f.counts = d_counts;
  f.offsets = d_offsets;
  f.global_out = static_cast<__nv_bfloat16*>(d_global_out);
  for (int r = 0; r < R; ++r) f.dst.p[r] = local[r];
  if (cap == 0 || slot_lo == slot_hi) {
    // no expert rows: every real row's combine is an empty sum
    return moe_combine_scatter(d_out_sorted, d_inv, d_w, rows, k, H, dtype, cap, d_counts,
                               d_offsets, R, local, d_global_out, d_status, stream);
  }
  FfnArgs a{d_sorted, d_offsets_P, P, slot_lo, slot_hi, cap, d_w_gate_up, d_w_down,
            H, I, d_out_sorted, h, d_status};
  if (ffn_uses_pair_kernel(a)) {
    // Many rows per slot: the pair kernel's down projection already moves its
    // weights and rows at about 0.8 of the HBM roofline, and a combine in its
    // epilogue must read the same expert rows back, so it only lengthened the
    // epilogue (measured: MM2 2.11 ms fused against 1.65 + 0.18 ms for MM2 and
    // the combine launch at 8192 tokens).  The combine runs as its own launch.
    const moe_status st = launch_ffn_tc(a, s);
    if (st != MOE_OK) return st;
    return moe_combine_scatter(d_out_sorted, d_inv, d_w, rows, k, H, dtype, cap, d_counts,
                               d_offsets, R, local, d_global_out, d_status, stream);
  }
  a.fuse = &f;
  return launch_ffn_tc(a, s);
}

// ---------------------------------------------------------------------------
// Grouped FFN of a skewed layer split by slot over two streams: the slots with
// at least hot_rows rows run on the pair kernel (weights as M) on hot_sms SMs
// of stream_hot, the others on the single-SM kernel (tokens as M) on the rest
// of the SMs of `stream`, at the same time.  SGLang chapter 17, section
// "Two-batch Overlap" and vLLM chapter 27 (Dual Batch Overlap, its SM control):
// two streams keep different kinds of work in flight together; here it is the
// hot slots' tensor-bound GEMMs beside the cold slots' weight stream, and every
// weight tile is still read once.

namespace {

// Fork and join events of the split FFN, created once per device on first use
// (never inside a call that is being captured, if the first call on the device
// runs eagerly).  The mutex keeps each record + wait pair together when several
// host threads call on one device.
struct SplitEvents {
  std::mutex mu;
  cudaEvent_t fork = nullptr, join = nullptr;
};

SplitEvents* split_events(int dev) {
  static std::mutex mu;
  static SplitEvents* cache[64] = {nullptr};
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == nullptr) {
    SplitEvents* e = new SplitEvents();
    if (cudaEventCreateWithFlags(&e->fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&e->join, cudaEventDisableTiming) != cudaSuccess) {
      delete e;
      return nullptr;
    }
    cache[dev] = e;
  }
  return cache[dev];
}

}  // namespace

extern "C" moe_status moe_grouped_ffn_split(const void* d_sorted, const int32_t* d_offsets_P,
                                            int P, int slot_lo, int slot_hi, int64_t cap,
                                            const void* d_w_gate_up, const void* d_w_down, int H,
                                            int I, int dtype, void* d_out_sorted, void* d_ws,
                                            size_t ws_bytes, int hot_rows, int hot_sms,
                                            uint32_t* d_status, void* stream, void* stream_hot) {
  if (P < 1 || slot_lo < 0 || slot_hi > P || slot_lo > slot_hi || cap < 0 || cap > INT32_MAX ||
      H < 1 || I < 1 || hot_rows < 1)
    return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (H % 256 != 0 || I % 128 != 0 || P > MOE_MAX_SLOTS) return MOE_ERR_UNSUPPORTED;
  if (cap == 0 || slot_lo == slot_hi) return MOE_OK;
  if (d_sorted == nullptr || d_offsets_P == nullptr || d_w_gate_up == nullptr ||
      d_w_down == nullptr || d_out_sorted == nullptr || d_ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_grouped_ffn_ws_bytes(cap, I, dtype)) return MOE_ERR_CAPACITY;
  if (!aligned16(d_sorted) || !aligned16(d_out_sorted) || !aligned16(d_ws) ||
      !aligned16(d_w_gate_up) || !aligned16(d_w_down))
    return MOE_ERR_INVALID_ARG;
  if ((int64_t)P * 2 * I > INT32_MAX || (int64_t)P * H > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
  const int sms = num_sms();
  if (hot_sms < 2 || hot_sms % 2 != 0 || hot_sms > sms - 2) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  cudaStream_t sh = stream_hot != nullptr ? as_stream(stream_hot) : s;
  FfnArgs hot{d_sorted, d_offsets_P, P, slot_lo, slot_hi, cap, d_w_gate_up, d_w_down,
              H, I, d_out_sorted, d_ws, d_status};
  FfnArgs cold = hot;
  hot.min_slot_rows = hot_rows;
  hot.sm_budget = hot_sms;
  cold.max_slot_rows = hot_rows - 1;
  cold.sm_budget = sms - hot_sms;
  if (sh == s) {  // one stream: the two parts one after the other
    const moe_status st = launch_ffn_tc_swap(hot, s);
    return st != MOE_OK ? st : launch_ffn_tc_single(cold, s);
  }
  // fork: stream_hot starts after everything already on `stream`; join: `stream`
  // continues after both parts
  SplitEvents* ev = split_events(dev);
  if (ev == nullptr) return MOE_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(ev->mu);
    if (cudaEventRecord(ev->fork, s) != cudaSuccess ||
        cudaStreamWaitEvent(sh, ev->fork, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  moe_status st = launch_ffn_tc_swap(hot, sh);
  const moe_status st2 = launch_ffn_tc_single(cold, s);
  if (st == MOE_OK) st = st2;
  // the join is recorded whatever happened, so `stream` never runs ahead of work
  // already queued on stream_hot
  std::lock_guard<std::mutex> lock(ev->mu);
  if (cudaEventRecord(ev->join, sh) != cudaSuccess ||
      cudaStreamWaitEvent(s, ev->join, 0) != cudaSuccess)
    st = MOE_ERR_CUDA;
  return st;
}

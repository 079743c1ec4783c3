// moe_dispatch_noalloc: the dispatch of moe_dispatch with its per-chunk
// histogram workspace held in a fixed-size array that the library itself
// places in device memory, so the caller never has to allocate scratch.
//
// Who needs it: code that may not allocate device memory at the point where
// it dispatches tokens -- e.g. a plugin running inside another framework's
// enqueue callback, where the host framework owns every device allocation, or
// a latency-critical decode loop that must never hit cudaMalloc/cudaFree,
// which can synchronise the device and stall the pipeline.  Those callers
// still own and pass every input and output buffer; only the scratch moves
// into the library.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// this library holds MOE_NOALLOC_SCRATCH_BYTES of it until the process exits.
// In host code its name is only a host-side stand-in, so the host looks up
// the real device address with cudaGetSymbolAddress once per device (with
// that device current) and passes that address on.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_dispatch_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// Device address of g_dispatch_scratch on the current device, looked up on
// the first call made on that device and cached.
void* scratch_on_current_device(moe_status* st) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *st = MOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr) {
      *st = MOE_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

// moe_dispatch's own argument checks, applied before the scratch-size check so
// that an invalid call returns what moe_dispatch returns for it, whatever its
// size.
moe_status check_dispatch_args(const void* d_global, const int32_t* d_ids, int64_t rows, int k,
                               int H, int dtype, int E, int P, const int32_t* d_l2p,
                               const int32_t* d_nrep, int X, int align, int64_t cap,
                               const int32_t* d_counts_P, const int32_t* d_offsets_P,
                               const int32_t* d_perm, const int32_t* d_inv,
                               const void* d_sorted) {
  if (d_counts_P == nullptr || d_offsets_P == nullptr ||
      (rows > 0 && (d_ids == nullptr || d_inv == nullptr)) || (cap > 0 && d_perm == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (rows < 0 || k < 1 || k > MOE_MAX_TOPK || E < 1 || P < 1 || P > MOE_MAX_SLOTS ||
      E > MOE_MAX_SLOTS || align < 1 || cap < 0)
    return MOE_ERR_INVALID_ARG;
  if (rows * k > INT32_MAX || cap > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if ((d_l2p == nullptr) != (d_nrep == nullptr)) return MOE_ERR_INVALID_ARG;
  if (d_l2p == nullptr && P != E) return MOE_ERR_INVALID_ARG;
  if (d_l2p != nullptr && X < 1) return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (d_global != nullptr || d_sorted != nullptr)) {
    if (d_global == nullptr || d_sorted == nullptr || H < 1) return MOE_ERR_INVALID_ARG;
    const int eb = moe::dtype_bytes(dtype);
    if (eb == 0) return MOE_ERR_UNSUPPORTED;
    if (((int64_t)H * eb) % 16 != 0 || !moe::aligned16(d_global) || !moe::aligned16(d_sorted))
      return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_dispatch_noalloc(const void* d_global, const int32_t* d_ids,
                                           int64_t rows, int k, int H, int dtype, int E, int P,
                                           const int32_t* d_l2p, const int32_t* d_nrep, int X,
                                           int align, int64_t cap, int32_t* d_counts_P,
                                           int32_t* d_offsets_P, int32_t* d_perm, int32_t* d_inv,
                                           void* d_sorted, uint32_t* d_status, void* stream) {
  const moe_status bad = check_dispatch_args(d_global, d_ids, rows, k, H, dtype, E, P, d_l2p,
                                             d_nrep, X, align, cap, d_counts_P, d_offsets_P,
                                             d_perm, d_inv, d_sorted);
  if (bad != MOE_OK) return bad;
  if (moe_dispatch_ws_bytes(rows, k, E) > (size_t)MOE_NOALLOC_SCRATCH_BYTES)
    return MOE_ERR_CAPACITY;  // rows * k pairs over E experts need more than the fixed scratch
  moe_status st = MOE_OK;
  void* scratch = scratch_on_current_device(&st);
  if (scratch == nullptr) return st;
  // The histogram kernel writes every entry it later reads, so the scratch
  // needs no clearing between calls.
  return moe_dispatch(d_global, d_ids, rows, k, H, dtype, E, P, d_l2p, d_nrep, X, align, cap,
                      d_counts_P, d_offsets_P, d_perm, d_inv, d_sorted, scratch,
                      (size_t)MOE_NOALLOC_SCRATCH_BYTES, d_status, stream);
}

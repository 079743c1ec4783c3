// Dispatch: a deterministic, stable counting sort of the routed (row, j)
// pairs by physical expert slot, plus the row permute that builds the
// per-slot contiguous buffers.
//
// SGLang chapter 17, section "normal dispatch 的调用链": get_dispatch_layout
// counts tokens per expert; expert_alignment rounds each expert's count up to
// a multiple of 128 for the grouped GEMM.  Sections "逻辑与物理的两套映射" and
// "推理时怎么选副本": a logical expert lives in num_valid physical slots
// (logical_to_all_physical_map); without an all-to-all every rank must pick
// the same replica for a token.  The pick here: occurrence p of logical expert
// l, counted in (row, j) order, goes to replica p mod num_valid[l], at
// position p / num_valid[l] inside that slot -- the stable (slot, row, j)
// order needs no second sort.
//
// Kernels (all deterministic: integer shared-memory atomics only where the
// result does not depend on their order):
//   1. hist   one block per chunk of kChunk pairs: per-chunk logical histogram
//   2. scan   one block: per-expert exclusive scan over chunks, per-slot
//             counts from the replica rule, aligned exclusive scan -> offsets
//   3. rank   one warp per chunk, its ids loaded up front, then 32 pairs per
//             step in order: __match_any_sync groups equal ids, popc of the
//             lower lanes gives the in-step rank, a shared running count
//             carries it across steps
//   4. copy   one warp per (source row, 2 KB segment): the segment is read
//             once and written to the row's k destinations, 16-byte vectors
//   5. pad    (align > 1) zero the alignment rows and mark them perm = -1
#include "common.cuh"

namespace moe {
namespace {

constexpr int kChunk = 1024;  // routed pairs per chunk

inline int64_t n_chunks(int64_t pairs) { return (pairs + kChunk - 1) / kChunk; }

__global__ void __launch_bounds__(256)
    dispatch_hist_kernel(const int32_t* __restrict__ ids, int64_t pairs, int E,
                         int32_t* __restrict__ hist, uint32_t* status) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  extern __shared__ int32_t s_h[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_h[e] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kChunk;
  for (int t = threadIdx.x; t < kChunk; t += blockDim.x) {
    int64_t q = base + t;
    if (q >= pairs) break;
    int32_t l = ids[q];
    if (l >= 0 && l < E)
      atomicAdd(&s_h[l], 1);
    else if (l != -1)
      flag(status, MOE_DEV_BAD_EXPERT_ID);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = s_h[e];
}

// Block-wide exclusive scan of one value per thread (blockDim.x == 1024).
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* s_warp,
                                                        int32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int32_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int32_t t = s_warp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += y;
    }
    s_warp[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  int32_t excl = x - v + (wid > 0 ? s_warp[wid - 1] : 0);
  *total = s_warp[31];
  return excl;
}

__global__ void __launch_bounds__(1024)
    dispatch_scan_kernel(int32_t* __restrict__ hist, int64_t chunks, int E, int P,
                         const int32_t* __restrict__ l2p, const int32_t* __restrict__ nrep, int X,
                         int align, int64_t cap, int32_t* __restrict__ counts_P,
                         int32_t* __restrict__ offsets_P, uint32_t* status) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  __shared__ int32_t s_cnt[MOE_MAX_SLOTS];    // per logical expert
  __shared__ int32_t s_slot[MOE_MAX_SLOTS];   // per physical slot
  __shared__ int32_t s_claim[MOE_MAX_SLOTS];
  __shared__ int32_t s_warp[32];
  // per-expert exclusive scan over chunks (in place: hist becomes chunk bases),
  // kScanBatch chunks' counts loaded together so their loads overlap
  constexpr int kScanBatch = 16;
  for (int l = threadIdx.x; l < E; l += blockDim.x) {
    int32_t run = 0;
    for (int64_t c0 = 0; c0 < chunks; c0 += kScanBatch) {
      int32_t t[kScanBatch];
#pragma unroll
      for (int i = 0; i < kScanBatch; ++i) t[i] = c0 + i < chunks ? hist[(c0 + i) * E + l] : 0;
#pragma unroll
      for (int i = 0; i < kScanBatch; ++i) {
        if (c0 + i < chunks) hist[(c0 + i) * E + l] = run;
        run += t[i];
      }
    }
    s_cnt[l] = run;
  }
  for (int s = threadIdx.x; s < P; s += blockDim.x) {
    s_slot[s] = 0;
    s_claim[s] = 0;
  }
  __syncthreads();
  if (l2p == nullptr) {
    for (int s = threadIdx.x; s < P; s += blockDim.x) s_slot[s] = s_cnt[s];
  } else {
    for (int l = threadIdx.x; l < E; l += blockDim.x) {
      int32_t nv = nrep[l];
      int32_t cl = s_cnt[l];
      if (nv < 1 || nv > X) {
        if (cl > 0) flag(status, MOE_DEV_BAD_MAP);
        continue;
      }
      for (int r = 0; r < nv; ++r) {
        int32_t slot = l2p[(int64_t)l * X + r];
        if (slot < 0 || slot >= P || atomicAdd(&s_claim[slot], 1) != 0) {
          flag(status, MOE_DEV_BAD_MAP);
          continue;
        }
        s_slot[slot] = cl > r ? (cl - 1 - r) / nv + 1 : 0;
      }
    }
  }
  __syncthreads();
  // aligned exclusive scan over slots (P <= 1024, one slot per thread)
  const int s = threadIdx.x;
  int32_t cnt = s < P ? s_slot[s] : 0;
  int32_t padded = (int32_t)(((int64_t)cnt + align - 1) / align * align);
  int32_t total = 0;
  int32_t excl = block_exclusive_scan(padded, s_warp, &total);
  if (s < P) {
    counts_P[s] = cnt;
    offsets_P[s] = excl;
  }
  if (s == 0) {
    offsets_P[P] = total;
    if ((int64_t)total > cap) flag(status, MOE_DEV_CAPACITY);
  }
}

// Slot and in-slot position of occurrence p of logical expert l (replica rule
// of the header: occurrence p goes to replica p mod num_valid, position
// p div num_valid).  Returns false for a bad map entry.
__device__ __forceinline__ bool place(int32_t l, int32_t p, const int32_t* l2p,
                                      const int32_t* nrep, int X, int P, int32_t* slot,
                                      int32_t* pos) {
  if (l2p == nullptr) {
    *slot = l;
    *pos = p;
    return true;
  }
  const int32_t nv = nrep[l];
  if (nv < 1 || nv > X) return false;
  *slot = l2p[(int64_t)l * X + p % nv];
  *pos = p / nv;
  return *slot >= 0 && *slot < P;
}

// Rank the pairs of one warp's segment in order: __match_any_sync groups equal
// ids in a 32-pair step, popc of the lower lanes gives the in-step rank,
// run[l] carries the count of l across steps.  idv holds the segment's ids.
template <int STEPS>
__device__ __forceinline__ void rank_segment(const int32_t (&idv)[STEPS], int64_t base,
                                             int64_t end, int k, int E, int32_t* run,
                                             const int32_t* l2p, const int32_t* nrep, int X,
                                             int P, const int32_t* offP, int64_t cap,
                                             int32_t* __restrict__ perm,
                                             int32_t* __restrict__ inv, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    if (base + s * 32 >= end) break;  // warp-uniform
    const int64_t q = base + s * 32 + lane;
    const int32_t l = idv[s];
    const bool valid = l >= 0 && l < E;
    const uint32_t mask = __match_any_sync(0xffffffffu, valid ? l : -1);
    const int rank = __popc(mask & lt);
    int32_t p = 0;
    if (valid) p = run[l] + rank;
    __syncwarp();
    if (valid && rank == __popc(mask) - 1) run[l] += __popc(mask);
    __syncwarp();
    if (q >= end) continue;
    int32_t dest = -1, slot = 0, pos = 0;
    if (valid) {
      if (place(l, p, l2p, nrep, X, P, &slot, &pos)) {
        const int64_t d = (int64_t)offP[slot] + pos;
        if (d < cap && d < offP[slot + 1]) {
          dest = (int32_t)d;
          perm[d] = (int32_t)(q / k);
        } else {
          flag(status, MOE_DEV_CAPACITY);
        }
      }
    }
    inv[q] = dest;
  }
}

// kRankWarps warps per chunk, each ranking a consecutive quarter of it: the
// warps' per-expert counts (shared-memory histograms) give each warp its start
// within the chunk's base counts, so the in-order ranking takes 8 steps per
// warp instead of 32.  The slot offsets and the replica tables are staged in
// shared memory first, so the ranking touches only registers and shared memory.
constexpr int kRankWarps = 4;
constexpr int kRankSteps = kChunk / 32 / kRankWarps;

__global__ void __launch_bounds__(kRankWarps * 32)
    dispatch_rank_kernel(const int32_t* __restrict__ ids, int64_t pairs, int k, int E,
                         const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ l2p,
                         const int32_t* __restrict__ nrep, int X, int P,
                         const int32_t* __restrict__ offsets_P, int64_t cap,
                         int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                         int stage_map, uint32_t* status) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  extern __shared__ int32_t smem[];
  int32_t* s_run = smem;                      // [kRankWarps][E] per-warp counts, then starts
  int32_t* s_off = s_run + kRankWarps * E;    // [P + 1]
  int32_t* s_nrep = s_off + P + 1;            // [E]   (map only)
  int32_t* s_l2p = s_nrep + E;                // [E*X] (map only)
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t cbase = (int64_t)blockIdx.x * kChunk;
  const int64_t cend = cbase + kChunk < pairs ? cbase + kChunk : pairs;
  const int64_t base = cbase + (int64_t)wid * (kChunk / kRankWarps);
  const int64_t wend = base + kChunk / kRankWarps;
  const int64_t end = wend < cend ? wend : cend;  // may be <= base in the last chunk
  int32_t idv[kRankSteps];
#pragma unroll
  for (int s = 0; s < kRankSteps; ++s) {
    const int64_t q = base + s * 32 + lane;
    idv[s] = q < end ? ids[q] : -1;
  }
  for (int i = threadIdx.x; i < kRankWarps * E; i += blockDim.x) s_run[i] = 0;
  for (int i = threadIdx.x; i <= P; i += blockDim.x) s_off[i] = offsets_P[i];
  const int32_t* m_l2p = l2p;
  const int32_t* m_nrep = nrep;
  if (l2p != nullptr && stage_map) {
    for (int i = threadIdx.x; i < E; i += blockDim.x) s_nrep[i] = nrep[i];
    for (int i = threadIdx.x; i < E * X; i += blockDim.x) s_l2p[i] = l2p[i];
    m_l2p = s_l2p;
    m_nrep = s_nrep;
  }
  __syncthreads();
  int32_t* my_run = s_run + wid * E;
#pragma unroll
  for (int s = 0; s < kRankSteps; ++s) {
    const int32_t l = idv[s];
    if (l >= 0 && l < E) atomicAdd(&my_run[l], 1);
  }
  __syncthreads();
  // each warp starts where the chunk's earlier warps end, from the chunk base
  const int32_t* cb = chunk_base + (int64_t)blockIdx.x * E;
  for (int l = threadIdx.x; l < E; l += blockDim.x) {
    int32_t run = cb[l];
#pragma unroll
    for (int w = 0; w < kRankWarps; ++w) {
      const int32_t t = s_run[w * E + l];
      s_run[w * E + l] = run;
      run += t;
    }
  }
  __syncthreads();
  rank_segment<kRankSteps>(idv, base, end, k, E, my_run, m_l2p, m_nrep, X, P, s_off, cap, perm,
                           inv, status);
}

// Small problems (<= kSmallPairs routed pairs, tables within kSmallSmemBytes) in one CTA:
// per-warp histograms, per-expert scan over warps, slot counts and aligned
// offsets, then each warp ranks its own segment -- one launch instead of three.
constexpr int kSmallWarps = 32;
constexpr int kSmallSteps = 8;   // 32-pair steps per warp segment (above 8192 pairs the
                                 // chunked kernels, four warps per 1024 pairs, are faster)
constexpr int64_t kSmallPairs = (int64_t)kSmallWarps * kSmallSteps * 32;
constexpr size_t kSmallSmemBytes = 48 * 1024;  // per-warp histograms + slot tables

__global__ void __launch_bounds__(kSmallWarps * 32)
    dispatch_small_kernel(const int32_t* __restrict__ ids, int64_t pairs, int k, int E, int P,
                          const int32_t* __restrict__ l2p, const int32_t* __restrict__ nrep,
                          int X, int align, int64_t cap, int32_t* __restrict__ counts_P,
                          int32_t* __restrict__ offsets_P, int32_t* __restrict__ perm,
                          int32_t* __restrict__ inv, int stage_map, uint32_t* status) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  extern __shared__ int32_t smem[];
  int32_t* s_hist = smem;                           // [kSmallWarps][E]
  int32_t* s_off = s_hist + kSmallWarps * E;        // [P + 1]
  int32_t* s_slot = s_off + P + 1;                  // [P]
  int32_t* s_claim = s_slot + P;                    // [P]
  int32_t* s_cnt = s_claim + P;                     // [E]
  int32_t* s_nrep = s_cnt + E;                      // [E]   (map staged only)
  int32_t* s_l2p = s_nrep + E;                      // [E*X] (map staged only)
  __shared__ int32_t s_warp[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kSmallWarps * E; i += blockDim.x) s_hist[i] = 0;
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    s_slot[i] = 0;
    s_claim[i] = 0;
  }
  // the replica tables, read by every rank step, from shared memory when they fit
  const int32_t* m_l2p = l2p;
  const int32_t* m_nrep = nrep;
  if (l2p != nullptr && stage_map) {
    for (int i = threadIdx.x; i < E; i += blockDim.x) s_nrep[i] = nrep[i];
    for (int i = threadIdx.x; i < E * X; i += blockDim.x) s_l2p[i] = l2p[i];
    m_l2p = s_l2p;
    m_nrep = s_nrep;
  }
  // warp segments of whole 32-pair steps
  const int64_t seg = ((pairs + kSmallWarps - 1) / kSmallWarps + 31) / 32 * 32;
  const int64_t base = (int64_t)wid * seg;
  const int64_t end = base + seg < pairs ? base + seg : pairs;
  int32_t idv[kSmallSteps];
#pragma unroll
  for (int s = 0; s < kSmallSteps; ++s) {
    const int64_t q = base + s * 32 + lane;
    idv[s] = (s * 32 < seg && q < end) ? ids[q] : -1;
  }
  __syncthreads();
  int32_t* my_hist = s_hist + wid * E;
#pragma unroll
  for (int s = 0; s < kSmallSteps; ++s) {
    const int32_t l = idv[s];
    const int64_t q = base + s * 32 + lane;
    if (l >= 0 && l < E)
      atomicAdd(&my_hist[l], 1);
    else if (l != -1 && q < end)
      flag(status, MOE_DEV_BAD_EXPERT_ID);
  }
  __syncthreads();
  // per-expert exclusive scan over warps (hist becomes each warp's base)
  for (int l = threadIdx.x; l < E; l += blockDim.x) {
    int32_t run = 0;
    for (int w = 0; w < kSmallWarps; ++w) {
      const int32_t t = s_hist[w * E + l];
      s_hist[w * E + l] = run;
      run += t;
    }
    s_cnt[l] = run;
  }
  __syncthreads();
  if (l2p == nullptr) {
    for (int sl = threadIdx.x; sl < P; sl += blockDim.x) s_slot[sl] = s_cnt[sl];
  } else {
    for (int l = threadIdx.x; l < E; l += blockDim.x) {
      const int32_t nv = nrep[l];
      const int32_t cl = s_cnt[l];
      if (nv < 1 || nv > X) {
        if (cl > 0) flag(status, MOE_DEV_BAD_MAP);
        continue;
      }
      for (int r = 0; r < nv; ++r) {
        const int32_t slot = l2p[(int64_t)l * X + r];
        if (slot < 0 || slot >= P || atomicAdd(&s_claim[slot], 1) != 0) {
          flag(status, MOE_DEV_BAD_MAP);
          continue;
        }
        s_slot[slot] = cl > r ? (cl - 1 - r) / nv + 1 : 0;
      }
    }
  }
  __syncthreads();
  {
    const int sl = threadIdx.x;  // P <= MOE_MAX_SLOTS = blockDim.x
    const int32_t cnt = sl < P ? s_slot[sl] : 0;
    const int32_t padded = (int32_t)(((int64_t)cnt + align - 1) / align * align);
    int32_t total = 0;
    const int32_t excl = block_exclusive_scan(padded, s_warp, &total);
    if (sl < P) {
      counts_P[sl] = cnt;
      offsets_P[sl] = excl;
      s_off[sl] = excl;
    }
    if (sl == 0) {
      offsets_P[P] = total;
      s_off[P] = total;
      if ((int64_t)total > cap) flag(status, MOE_DEV_CAPACITY);
    }
  }
  __syncthreads();
  rank_segment<kSmallSteps>(idv, base, end, k, E, my_hist, m_l2p, m_nrep, X, P, s_off, cap,
                            perm, inv, status);
}

__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

constexpr int kCopyWarps = 8;
constexpr int kCopyUnroll = 4;
constexpr int kSegVecs = 32 * kCopyUnroll;  // vectors per warp segment of a row

// One warp per (source row, segment): the segment is read once (every lane's
// loads in flight together) and written to the row's k destinations.
__global__ void __launch_bounds__(kCopyWarps * 32)
    dispatch_copy_kernel(const uint4* __restrict__ xg, const int32_t* __restrict__ inv,
                         int64_t rows, int k, int vpr, int64_t cap, uint4* __restrict__ xs) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * kCopyWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kCopyWarps;
  const int segs = (vpr + kSegVecs - 1) / kSegVecs;
  const int64_t items = rows * segs;
  for (int64_t w = warp0; w < items; w += nwarps) {
    const int64_t g = w / segs;
    const int v0 = (int)(w - g * segs) * kSegVecs;
    int32_t my_d = lane < k ? inv[g * k + lane] : -1;
    if (my_d >= cap) my_d = -1;
    if (__ballot_sync(0xffffffffu, my_d >= 0) == 0) continue;  // pad row
    const uint4* src = xg + g * vpr;
    uint4 t[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < vpr) t[u] = ld_nc(src + v);
    }
    for (int j = 0; j < k; ++j) {
      const int32_t d = __shfl_sync(0xffffffffu, my_d, j);
      if (d < 0) continue;
      uint4* dst = xs + (int64_t)d * vpr;
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vpr) dst[v] = t[u];
      }
    }
  }
}

__global__ void __launch_bounds__(256)
    dispatch_pad_kernel(const int32_t* __restrict__ counts_P, const int32_t* __restrict__ offsets_P,
                        int P, int vpr, int64_t cap, int32_t* __restrict__ perm,
                        uint4* __restrict__ xs) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  const int s = blockIdx.x;
  if (s >= P) return;
  int64_t a = (int64_t)offsets_P[s] + counts_P[s];
  int64_t b = offsets_P[s + 1];
  if (b > cap) b = cap;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int64_t d = a; d < b; ++d) {
    if (threadIdx.x == 0) perm[d] = -1;
    if (xs != nullptr)
      for (int v = threadIdx.x; v < vpr; v += blockDim.x) xs[d * vpr + v] = z;
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_dispatch_ws_bytes(int64_t rows, int k, int E) {
  if (rows < 0 || k < 1 || E < 1) return 0;
  int64_t chunks = n_chunks(rows * k);
  if (chunks < 1) chunks = 1;
  return (size_t)(chunks * E * (int64_t)sizeof(int32_t));
}

extern "C" moe_status moe_dispatch(const void* d_global, const int32_t* d_ids, int64_t rows,
                                   int k, int H, int dtype, int E, int P, const int32_t* d_l2p,
                                   const int32_t* d_nrep, int X, int align, int64_t cap,
                                   int32_t* d_counts_P, int32_t* d_offsets_P, int32_t* d_perm,
                                   int32_t* d_inv, void* d_sorted, void* d_ws, size_t ws_bytes,
                                   uint32_t* d_status, void* stream) {
  if (d_counts_P == nullptr || d_offsets_P == nullptr || d_ws == nullptr ||
      (rows > 0 && (d_ids == nullptr || d_inv == nullptr)) || (cap > 0 && d_perm == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (rows < 0 || k < 1 || k > MOE_MAX_TOPK || E < 1 || P < 1 || P > MOE_MAX_SLOTS ||
      E > MOE_MAX_SLOTS || align < 1 || cap < 0)
    return MOE_ERR_INVALID_ARG;
  if (rows * k > INT32_MAX || cap > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if ((d_l2p == nullptr) != (d_nrep == nullptr)) return MOE_ERR_INVALID_ARG;
  if (d_l2p == nullptr && P != E) return MOE_ERR_INVALID_ARG;
  if (d_l2p != nullptr && X < 1) return MOE_ERR_INVALID_ARG;
  const bool move_rows = rows > 0 && (d_global != nullptr || d_sorted != nullptr);
  int vpr = 0;
  if (move_rows) {
    if (d_global == nullptr || d_sorted == nullptr || H < 1) return MOE_ERR_INVALID_ARG;
    int eb = dtype_bytes(dtype);
    if (eb == 0) return MOE_ERR_UNSUPPORTED;
    if (((int64_t)H * eb) % 16 != 0 || !aligned16(d_global) || !aligned16(d_sorted))
      return MOE_ERR_INVALID_ARG;
    vpr = (int)((int64_t)H * eb / 16);
  }
  if (ws_bytes < moe_dispatch_ws_bytes(rows, k, E)) return MOE_ERR_CAPACITY;
  cudaStream_t s = as_stream(stream);
  const int64_t pairs = rows * k;
  const int64_t chunks = n_chunks(pairs);
  int32_t* hist = static_cast<int32_t*>(d_ws);
  const size_t small_smem =
      sizeof(int32_t) * ((size_t)kSmallWarps * E + (P + 1) + 2 * (size_t)P + E);
  const size_t small_map = d_l2p != nullptr ? sizeof(int32_t) * ((size_t)E + (size_t)E * X) : 0;
  if (pairs <= kSmallPairs && small_smem <= kSmallSmemBytes) {
    const int stage = small_map > 0 && small_smem + small_map <= kSmallSmemBytes;
    const size_t smem = small_smem + (stage ? small_map : 0);
    launch(dispatch_small_kernel, 1, kSmallWarps * 32, smem, s, d_ids, pairs, k, E, P, d_l2p,
           d_nrep, X, align, cap, d_counts_P, d_offsets_P, d_perm, d_inv, stage, d_status);
  } else if (chunks == 0) {
    launch(dispatch_scan_kernel, 1, 1024, 0, s, hist, 0, E, P, d_l2p, d_nrep, X, align, cap,
           d_counts_P, d_offsets_P, d_status);
  } else {
    launch(dispatch_hist_kernel, (unsigned)chunks, 256, E * sizeof(int32_t), s, d_ids, pairs, E,
           hist, d_status);
    launch(dispatch_scan_kernel, 1, 1024, 0, s, hist, chunks, E, P, d_l2p, d_nrep, X, align, cap,
           d_counts_P, d_offsets_P, d_status);
    // replica tables staged in shared memory when they fit (else read from global)
    const int stage_map = d_l2p != nullptr && (int64_t)E * X <= 4096;
    const size_t smem = sizeof(int32_t) * ((size_t)kRankWarps * E + (P + 1) +
                                           (stage_map ? E + (size_t)E * X : 0));
    launch(dispatch_rank_kernel, (unsigned)chunks, kRankWarps * 32, smem, s, d_ids, pairs, k, E,
           hist, d_l2p, d_nrep, X, P, d_offsets_P, cap, d_perm, d_inv, stage_map, d_status);
  }
  if (move_rows && rows > 0) {
    const int64_t items = rows * ((vpr + kSegVecs - 1) / kSegVecs);
    int64_t want = (items + kCopyWarps - 1) / kCopyWarps;
    int64_t lim = (int64_t)num_sms() * 8;
    launch(dispatch_copy_kernel, (unsigned)(want < lim ? want : lim), kCopyWarps * 32, 0, s,
           static_cast<const uint4*>(d_global), d_inv, rows, k, vpr, cap,
           static_cast<uint4*>(d_sorted));
  }
  if (align > 1) {
    launch(dispatch_pad_kernel, P, 256, 0, s, d_counts_P, d_offsets_P, P, vpr, cap, d_perm,
           move_rows ? static_cast<uint4*>(d_sorted) : nullptr);
  }
  return launch_status();
}

// Grouped SwiGLU expert FFN on the 5th-generation tensor cores (sm_103a).
//
// SGLang chapter 17, opening sections: a DeepSeek-V3 expert has gate_proj and
// up_proj [2048, 7168] and down_proj [7168, 2048] (weights stored [out, in]);
// section "normal dispatch 的调用链": the experts run as a grouped GEMM over
// the per-expert contiguous rows.  vLLM chapter 27, figure "MoE 模块化内核的
// PrepareAndFinalize 块结构": MM1, activation, MM2.
//
// Two launches of one persistent, warp-specialised kernel:
//   MM1 + SwiGLU:  acc[M x 256] = xs_tile . [Wg rows n..n+127 ; Wu rows n..n+127]^T
//                  h[:, n..n+127] = bf16( silu(acc[:, 0:128]) * acc[:, 128:256] )
//   MM2:           acc[M x 256] = h_tile . Wd[rows n..n+255]^T
//                  ys[:, n..n+255] = bf16(acc)
// Work units are (slot, n-tile, m-group) with the m-groups of one slot and
// n-tile adjacent, so units running at the same time share the weight tile
// through L2; unit counts come from the device-side slot offsets, so the host
// never synchronises after dispatch.  A unit's rows start at the slot's first
// row (no alignment needed); rows past the slot's end are computed from
// whatever follows and never stored.
//
// CL = 2 (chosen when the sorted buffer holds >= 192 rows per slot on
// average): a cluster of two CTAs on two SMs runs one M = 256 MMA
// (tcgen05.mma.cta_group::2).  Each CTA holds its own 128 rows of A and one
// 128-row half of the weight tile B in shared memory; the MMA reads both
// CTAs' halves.  Per SM and 64-deep k-block that is 32 KB written by TMA and
// 32 KB read by the tensor core, against 48 + 48 KB for one 128 x 256 tile per
// SM (CL = 1), whose shared-memory traffic caps the tensor pipe near two
// thirds of its rate.  A pair launch covers whole 256-row groups (and a last
// group more than half full); a second, single-SM launch covers each slot's
// remaining <= 128 rows as one 128-row tile, so a slot of 256 + t rows costs
// one group plus one half-size tile instead of two groups.  With few rows per
// slot (decode) the weight stream is the whole cost and the single-SM kernel
// (CL = 1, 4 stages of 48 KB) keeps more weight bytes in flight per SM, so
// the launcher picks by rows per slot.
//
// Roles (192 threads, one CTA per SM):
//   warp 0    TMA producer (both CTAs): own A box 64x128 and own B box 64x128
//             per stage, 128-byte swizzle; completion is signalled on the
//             leader CTA's "full" barrier; 6-stage ring (32 KB per stage)
//   warp 1    TMEM allocation (512 columns: two 128x256 fp32 accumulators per
//             CTA); in the leader CTA lane 0 issues the MMAs (M=256, N=256,
//             K=16, bf16 -> fp32) and tcgen05.commit, multicast to both CTAs
//             to release stages and publish accumulators
//   warps 2-5 epilogue (both CTAs): tcgen05.ld 32 columns at a time from the
//             warp's TMEM lane quarter, activation, bf16 pack, 64-byte row
//             stores; one arrival per warp on the leader's "accumulator free"
//             barrier
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel sets
// MOE_DEV_TIMEOUT, the other roles stop at their next wait, TMEM is freed and
// the kernel returns.
#include <mutex>

#include "common.cuh"
#include "ffn_internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

// The pair kernel (CL = 2) needs a full 256-row group per unit to pay off;
// below this many rows per slot on average the single-SM kernel (CL = 1)
// streams the weights faster (decode-sized batches).
#ifndef MOE_FFN_PAIR_ROWS
#define MOE_FFN_PAIR_ROWS 192
#endif
constexpr int64_t kPairRowsPerSlot = MOE_FFN_PAIR_ROWS;
#ifndef MOE_FFN_SWAP
#define MOE_FFN_SWAP 1
#endif

constexpr int BM = 128;  // rows per CTA
constexpr int BN = 256;  // accumulator columns
constexpr int BK = 64;   // 64 bf16 = 128 bytes = one swizzle row
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BOX_BYTES = 128 * BK * 2;  // one 64 x 128 TMA box
constexpr int THREADS = 192;

template <int CL>
struct Cfg {
  static constexpr int B_BYTES = (BN / CL) * BK * 2;  // this CTA's share of the B tile
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = CL == 2 ? 6 : 4;
  static constexpr int M = BM * CL;
  static constexpr uint32_t IDESC = idesc_bf16(M, BN);
};

constexpr int MAX_STAGES = 6;
struct SmemLayout {
  // stage buffers come first (1024-byte aligned base)
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t total_units;
  int32_t warp_sums[THREADS / 32];
  int32_t pref[MOE_MAX_SLOTS + 1];  // unit prefix over the slot range
  int32_t mt[MOE_MAX_SLOTS];        // 128-row m-tiles per slot in this launch
  int32_t row_base[MOE_MAX_SLOTS];  // first row of the slot this launch covers
  int32_t row_end[MOE_MAX_SLOTS];   // one past the last row it covers
};
template <int CL>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)Cfg<CL>::STAGES * Cfg<CL>::STAGE_BYTES + sizeof(SmemLayout);
}

// Which rows of each slot a launch covers.  kAllRows: every row, in groups of
// CL m-tiles.  kPairGroups (CL = 2): whole 256-row groups, plus the last
// partial group only when it is more than half full.  kTailRows (CL = 1): the
// <= 128 rows kPairGroups leaves, as one 128-row tile.  kPairGroups followed
// by kTailRows covers every row exactly once.
enum Part { kAllRows = 0, kPairGroups = 1, kTailRows = 2 };

__host__ __device__ __forceinline__ int32_t pair_groups(int64_t rows) {
  return (int32_t)(rows / 256 + ((rows % 256) > 128 ? 1 : 0));
}

struct TcParams {
  const int32_t* offsets;
  int part;
  int slot_lo, nslots;
  int64_t cap;
  int num_kb;
  int n_tiles;
  int b_rows_per_slot;
  int b_tile_step;
  int b_second;
  int out_ld;
  int out_tile_cols;
  __nv_bfloat16* out;
  uint32_t* status;
};

// Work unit u -> (slot, m-group, n-tile) through the prefix over the slot range.
// An m-group is CL consecutive 128-row m-tiles (one per CTA of the cluster).
struct Unit {
  int slot, mg, n;
};
__device__ __forceinline__ Unit decode_unit(const SmemLayout& L, int nslots, int u, int CL) {
  int lo = 0, hi = nslots - 1;
  while (lo < hi) {  // largest s with pref[s] <= u
    int mid = (lo + hi + 1) >> 1;
    if (L.pref[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int local = u - L.pref[lo];
  const int groups = (L.mt[lo] + CL - 1) / CL;
  Unit r;
  r.slot = lo;
  r.mg = local % groups;
  r.n = local / groups;
  return r;
}

template <bool SWIGLU, int CL>
__global__ void __launch_bounds__(THREADS, 1)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const TcParams p) {
  using C = Cfg<CL>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  SmemLayout& L = *reinterpret_cast<SmemLayout*>(stage_base + (size_t)STAGES * C::STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = CL > 1 ? cluster_ctarank() : 0u;
  const bool leader = crank == 0;
  const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;

  // ---- unit table: m-tiles per slot, exclusive prefix of units
  {
    const int per = (p.nslots + THREADS - 1) / THREADS;
    const int s0 = threadIdx.x * per;
    int32_t local = 0;
    for (int i = 0; i < per; ++i) {
      int s = s0 + i;
      if (s < p.nslots) {
        const int64_t o0 = p.offsets[p.slot_lo + s];
        int64_t rows = (int64_t)p.offsets[p.slot_lo + s + 1] - o0;
        if (rows < 0) rows = 0;
        int64_t base = 0, end = rows;
        if (p.part == kPairGroups) {
          end = (int64_t)pair_groups(rows) * 256;
          if (end > rows) end = rows;
        } else if (p.part == kTailRows) {
          base = (int64_t)pair_groups(rows) * 256;
          if (base > rows) base = rows;
        }
        const int32_t mt = end > base ? (int32_t)((end - base + BM - 1) / BM) : 0;
        L.mt[s] = mt;
        L.row_base[s] = (int32_t)(o0 + base);
        L.row_end[s] = (int32_t)(o0 + end);
        local += (mt + CL - 1) / CL * p.n_tiles;
      }
    }
    int32_t x = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) L.warp_sums[warp] = x;
    if (threadIdx.x == 0) {
      L.abort_flag = 0;
      for (int i = 0; i < STAGES; ++i) {
        mbar_init(smem_u32(&L.full[i]), 1);   // leader: its producer's expect_tx
        mbar_init(smem_u32(&L.empty[i]), 1);  // the leader's MMA commit
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(smem_u32(&L.tmem_full[i]), 1);
        mbar_init(smem_u32(&L.tmem_empty[i]), 4 * CL);  // one per epilogue warp of the pair
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<CL>(smem_u32(&L.tmem_base));  // whole warp, both CTAs
    __syncthreads();
    int32_t before = 0;
    for (int w = 0; w < warp; ++w) before += L.warp_sums[w];
    int32_t run = before + x - local;  // exclusive prefix of this thread's group
    for (int i = 0; i < per; ++i) {
      int s = s0 + i;
      if (s < p.nslots) {
        L.pref[s] = run;
        run += (L.mt[s] + CL - 1) / CL * p.n_tiles;
      }
    }
    if (threadIdx.x == THREADS - 1) {
      int32_t tot = 0;
      for (int w = 0; w < THREADS / 32; ++w) tot += L.warp_sums[w];
      L.pref[p.nslots] = tot;
      L.total_units = tot;
    }
    fence_before();
    if (CL > 1)
      cluster_sync();  // the leader's barriers exist before the peer signals them
    else
      __syncthreads();
    fence_after();
  }
  const int total = L.total_units;
  const uint32_t tmem_base = L.tmem_base;
  volatile int32_t* abort_flag = &L.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_act = policy_evict_last();
    const uint64_t pol_w = policy_evict_first();
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    uint32_t it = 0;
    for (int u = cid; u < total; u += ncl) {
      const Unit un = decode_unit(L, p.nslots, u, CL);
      const int slot = p.slot_lo + un.slot;
      const int32_t row0 = L.row_base[un.slot] + (un.mg * CL + (int)crank) * BM;
      const int32_t brow1 = slot * p.b_rows_per_slot + un.n * p.b_tile_step;
      const int32_t brow2 = brow1 + p.b_second;
      bool ok = true;
      for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
        const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
        if (!wait_bar(smem_u32(&L.empty[st]), ph ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full_local = smem_u32(&L.full[st]);
          const uint32_t full = CL > 1 ? map_to_rank(full_local, 0) : full_local;
          const uint32_t sa = smem_u32(stage_base + (size_t)st * C::STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          if (leader) mbar_arrive_expect_tx(full_local, CL * C::STAGE_BYTES);
          tma_load_2d<CL>(sa, &tmA, kb * BK, row0, full, pol_act);
          if (CL == 1) {
            tma_load_2d<CL>(sb, &tmB, kb * BK, brow1, full, pol_w);
            tma_load_2d<CL>(sb + B_BOX_BYTES, &tmB, kb * BK, brow2, full, pol_w);
          } else {
            tma_load_2d<CL>(sb, &tmB, kb * BK, crank ? brow2 : brow1, full, pol_w);
          }
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    // drain: every "stage free" arrival bound for this CTA (the leader's MMA
    // commits, which follow the loads they consumed) has happened before exit
    for (uint32_t j = (it >= STAGES ? it - STAGES : 0); j < it; ++j) {
      const uint32_t st = j % STAGES, ph = (j / STAGES) & 1u;
      if (!wait_bar(smem_u32(&L.empty[st]), ph, abort_flag, p.status)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    if (leader) {
      uint32_t it = 0, local_tile = 0;
      for (int u = cid; u < total; u += ncl, ++local_tile) {
        const uint32_t acc = local_tile & 1u, acc_ph = (local_tile >> 1) & 1u;
        if (!wait_bar(smem_u32(&L.tmem_empty[acc]), acc_ph ^ 1u, abort_flag, p.status)) break;
        fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
          if (!wait_bar(smem_u32(&L.full[st]), ph, abort_flag, p.status)) {
            ok = false;
            break;
          }
          fence_after();
          if (lane == 0) {
            const uint32_t sa = smem_u32(stage_base + (size_t)st * C::STAGE_BYTES);
            const uint64_t adesc = sw128_desc(sa);
            const uint64_t bdesc = sw128_desc(sa + A_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes per K=16 step in the swizzle row
              mma<CL>(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, C::IDESC, (kb | kk) != 0);
            commit<CL>(smem_u32(&L.empty[st]));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) commit<CL>(smem_u32(&L.tmem_full[acc]));
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    const int row_in_tile = quad * 32 + lane;
    uint32_t local_tile = 0;
    for (int u = cid; u < total; u += ncl, ++local_tile) {
      const Unit un = decode_unit(L, p.nslots, u, CL);
      const int64_t row0 = (int64_t)L.row_base[un.slot] + (int64_t)(un.mg * CL + (int)crank) * BM;
      const int64_t row_end = L.row_end[un.slot];
      const uint32_t acc = local_tile & 1u, acc_ph = (local_tile >> 1) & 1u;
      if (!wait_bar(smem_u32(&L.tmem_full[acc]), acc_ph, abort_flag, p.status)) break;
      fence_after();
      const int64_t row = row0 + row_in_tile;
      const bool valid = row < row_end && row < p.cap;
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * BN;
      __nv_bfloat16* orow = p.out + row * p.out_ld + (int64_t)un.n * p.out_tile_cols;
      if (SWIGLU) {
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t g[32], v[32];
          tmem_ld32(taddr + c, g);
          tmem_ld32(taddr + 128 + c, v);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float g0 = __uint_as_float(g[2 * e]), g1 = __uint_as_float(g[2 * e + 1]);
            float u0 = __uint_as_float(v[2 * e]), u1 = __uint_as_float(v[2 * e + 1]);
            float h0 = g0 / (1.0f + expf(-g0)) * u0;
            float h1 = g1 / (1.0f + expf(-g1)) * u1;
            pk[e] = pack_bf16x2(h0, h1);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t y[32];
          tmem_ld32(taddr + c, y);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(y[2 * e]), __uint_as_float(y[2 * e + 1]));
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t bar = smem_u32(&L.tmem_empty[acc]);
        if (CL == 1)
          mbar_arrive(bar);
        else
          mbar_arrive_cluster(map_to_rank(bar, 0));  // the leader's barrier
      }
    }
  }

  fence_before();
  // No CTA may leave while its peer can still signal its barriers or read its
  // shared memory through the pair MMA.
  if (CL > 1)
    cluster_sync();
  else
    __syncthreads();
  fence_after();
  if (warp == 1) tmem_dealloc<CL>(tmem_base);
}

// ------------------------------------------------------------- host side
template <int CL>
cudaLaunchConfig_t launch_cfg(int clusters, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL * clusters);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem_bytes<CL>();
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Per device and cluster size: raise the dynamic shared-memory limit and find
// how many clusters fit at once (the persistent grid must be fully resident).
template <int CL>
bool device_setup(int* max_clusters) {
  static std::mutex mu;
  static int clusters[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (clusters[dev] == 0) {
    const int bytes = (int)smem_bytes<CL>();
    if (cudaFuncSetAttribute(ffn_tc_kernel<true, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess ||
        cudaFuncSetAttribute(ffn_tc_kernel<false, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess)
      return false;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = launch_cfg<CL>(num_sms() / CL, nullptr, attr);
    int c1 = 0, c2 = 0;
    if (cudaOccupancyMaxActiveClusters(&c1, ffn_tc_kernel<true, CL>, &cfg) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&c2, ffn_tc_kernel<false, CL>, &cfg) != cudaSuccess)
      return false;
    const int n = c1 < c2 ? c1 : c2;
    if (n < 1) return false;
    clusters[dev] = n;
  }
  *max_clusters = clusters[dev];
  return true;
}

template <bool SWIGLU, int CL>
cudaError_t launch(const CUtensorMap& mA, const CUtensorMap& mB, const TcParams& p, int clusters,
                   cudaStream_t s) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_cfg<CL>(clusters, s, attr);
  return cudaLaunchKernelEx(&cfg, ffn_tc_kernel<SWIGLU, CL>, mA, mB, p);
}

// One launch of MM1 + SwiGLU (gemm1) or MM2 over the rows `part` selects.
template <int CL>
moe_status run_ffn(const FfnArgs& a, const CUtensorMap& mA, const CUtensorMap& mB, int part,
                   bool gemm1, cudaStream_t s) {
  const int nslots = a.slot_hi - a.slot_lo;
  int max_clusters = 0;
  if (!device_setup<CL>(&max_clusters)) return MOE_ERR_CUDA;
  // upper bound of m-groups over the slot range (device-side counts unknown here)
  const int64_t m_bound = part == kTailRows ? nslots
                                            : ((a.cap + BM - 1) / BM + nslots) / CL + nslots;
  TcParams p;
  p.offsets = a.offsets;
  p.part = part;
  p.slot_lo = a.slot_lo;
  p.nslots = nslots;
  p.cap = a.cap;
  p.status = a.status;
  if (gemm1) {
    p.num_kb = a.H / BK;
    p.n_tiles = a.I / 128;
    p.b_rows_per_slot = 2 * a.I;
    p.b_tile_step = 128;
    p.b_second = a.I;
    p.out_ld = a.I;
    p.out_tile_cols = 128;
    p.out = static_cast<__nv_bfloat16*>(a.h);
  } else {
    p.num_kb = a.I / BK;
    p.n_tiles = a.H / BN;
    p.b_rows_per_slot = a.H;
    p.b_tile_step = BN;
    p.b_second = 128;
    p.out_ld = a.H;
    p.out_tile_cols = BN;
    p.out = static_cast<__nv_bfloat16*>(a.ys);
  }
  const int64_t bound = m_bound * p.n_tiles;
  const int clusters = (int)(bound < max_clusters ? bound : max_clusters);
  const cudaError_t e = gemm1 ? launch<true, CL>(mA, mB, p, clusters, s)
                              : launch<false, CL>(mA, mB, p, clusters, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

moe_status launch_ffn_tc(const FfnArgs& a, cudaStream_t s) {
  const int nslots = a.slot_hi - a.slot_lo;
  if (nslots <= 0 || a.cap <= 0) return MOE_OK;
  CUtensorMap mA1, mB1, mA2, mB2;
  if (!make_map(&mA1, a.xs, (uint64_t)a.H, (uint64_t)a.cap, 128) ||
      !make_map(&mB1, a.wgu, (uint64_t)a.H, (uint64_t)a.P * 2 * a.I, 128) ||
      !make_map(&mA2, a.h, (uint64_t)a.I, (uint64_t)a.cap, 128) ||
      !make_map(&mB2, a.wd, (uint64_t)a.I, (uint64_t)a.P * a.H, 128))
    return MOE_ERR_CUDA;
  // rows per slot the sorted buffer can hold on average, over the whole layer
  const int64_t rows_per_slot = a.cap / (a.P > 0 ? a.P : 1);
  moe_status st;
  if (rows_per_slot >= kPairRowsPerSlot) {
#if MOE_FFN_SWAP
    return launch_ffn_tc_swap(a, s);
#endif
    // pair groups on two SMs, then each slot's short remainder on one SM
    if ((st = run_ffn<2>(a, mA1, mB1, kPairGroups, true, s)) != MOE_OK) return st;
    if ((st = run_ffn<1>(a, mA1, mB1, kTailRows, true, s)) != MOE_OK) return st;
    if ((st = run_ffn<2>(a, mA2, mB2, kPairGroups, false, s)) != MOE_OK) return st;
    return run_ffn<1>(a, mA2, mB2, kTailRows, false, s);
  }
  if ((st = run_ffn<1>(a, mA1, mB1, kAllRows, true, s)) != MOE_OK) return st;
  return run_ffn<1>(a, mA2, mB2, kAllRows, false, s);
}

}  // namespace moe

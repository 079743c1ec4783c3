// Grouped SwiGLU expert FFN on the 5th-generation tensor cores (sm_103a):
// tokens as the MMA's M operand, one SM per tile (few tokens per slot).
//
// SGLang chapter 17, opening sections: a DeepSeek-V3 expert has gate_proj and
// up_proj [2048, 7168] and down_proj [7168, 2048] (weights stored [out, in]);
// section "normal dispatch 的调用链": the experts run as a grouped GEMM over
// the per-expert contiguous rows.  vLLM chapter 27, figure "MoE 模块化内核的
// PrepareAndFinalize 块结构": MM1, activation, MM2.
//
// Two launches of one persistent, warp-specialised kernel:
//   MM1 + SwiGLU:  acc[128 x 256] = xs_tile . [Wg rows n..n+127 ; Wu rows n..n+127]^T
//                  h[:, n..n+127] = bf16( silu(acc[:, 0:128]) * acc[:, 128:256] )
//   MM2:           acc[128 x 256] = h_tile . Wd[rows n..n+255]^T
//                  ys[:, n..n+255] = bf16(acc)
// Work units are (slot, n-tile, m-tile) with the m-tiles of one slot and
// n-tile adjacent, so units running at the same time share the weight tile
// through L2; unit counts come from the device-side slot offsets, so the host
// never synchronises after dispatch.  A unit's rows start at the slot's first
// row (no alignment needed); rows past the slot's end are computed from
// whatever follows and never stored.
//
// With few rows per slot (decode) the weight stream is the whole cost: four
// 48 KB stages keep 128 KB of weights in flight per SM.  From 192 sorted rows
// per slot on average the launcher hands the layer to the pair kernel with
// the weights as M (ffn_tc_swap.cu), which reads each weight tile once per
// slot whatever the slot's row count.
//
// Roles (192 threads, one CTA per SM):
//   warp 0    TMA producer: A box 64x128 (rows) and two B boxes 64x128 (the
//             weight tile) per stage, 128-byte swizzle; 4-stage ring
//   warp 1    TMEM allocation (512 columns: two 128x256 fp32 accumulators);
//             lane 0 issues the MMAs (M=128, N=256, K=16, bf16 -> fp32) and
//             tcgen05.commit to release stages and publish accumulators
//   warps 2-5 epilogue: tcgen05.ld 32 columns at a time from the warp's TMEM
//             lane quarter, activation (fast exp and divide), bf16 pack, 64-byte
//             row stores; a warp whose 32 rows lie past the slot's end (most of
//             them at decode) skips straight to its arrival on the
//             "accumulator free" barrier
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel sets
// MOE_DEV_TIMEOUT, the other roles stop at their next wait, TMEM is freed and
// the kernel returns.
//
// With FUSE (moe_grouped_ffn_combine) the MM2 epilogue also combines: after a
// thread has stored its row of the n-tile, it counts the row in on the token's
// counter for that n-tile with one acquire-release atomic (fuse_combine.cuh);
// the warp then runs the weighted sum of every token whose count its rows
// completed, one 16-byte vector of the 256 features per lane, straight into the
// replica rows.  The token of each row is loaded before the accumulator wait and
// the replica table sits in shared memory, so the combine adds a few memory
// round trips to the epilogue after the accumulator is handed back.
#include <mutex>

#include "common.cuh"
#include "ffn_internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

// Rows per slot on average from which the pair kernel with the weights as M
// takes over (below it, this kernel streams the weights faster).
#ifndef MOE_FFN_PAIR_ROWS
#define MOE_FFN_PAIR_ROWS 192
#endif
constexpr int64_t kPairRowsPerSlot = MOE_FFN_PAIR_ROWS;

constexpr int BM = 128;  // rows per tile
constexpr int BN = 256;  // accumulator columns
constexpr int BK = 64;   // 64 bf16 = 128 bytes = one swizzle row
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BOX_BYTES = 128 * BK * 2;  // one 64 x 128 TMA box
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int STAGES = 4;
constexpr int THREADS = 192;
constexpr uint32_t IDESC = idesc_bf16(BM, BN);

struct SmemLayout {
  // stage buffers come first (1024-byte aligned base)
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t total_units;
  int32_t warp_sums[THREADS / 32];
  int32_t pref[MOE_MAX_SLOTS + 1];  // unit prefix over the slot range
  int32_t mt[MOE_MAX_SLOTS];        // 128-row m-tiles per slot
  int32_t row_base[MOE_MAX_SLOTS];  // first row of the slot
  int32_t row_end[MOE_MAX_SLOTS];   // one past its last row
  int32_t r_off[MOE_MAX_REPLICAS + 1];  // FUSE: replica offsets and counts
  int32_t r_cnt[MOE_MAX_REPLICAS];
};
constexpr size_t smem_bytes() { return 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(SmemLayout); }

struct TcParams {
  const int32_t* offsets;
  int slot_lo, nslots;
  int32_t min_slot_rows, max_slot_rows;  // slots outside [min, max] rows get no units
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

// Work unit u -> (slot, m-tile, n-tile) through the prefix over the slot range.
struct Unit {
  int slot, mt, n;
};
__device__ __forceinline__ Unit decode_unit(const SmemLayout& L, int nslots, int u) {
  int lo = 0, hi = nslots - 1;
  while (lo < hi) {  // largest s with pref[s] <= u
    int mid = (lo + hi + 1) >> 1;
    if (L.pref[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int local = u - L.pref[lo];
  const int tiles = L.mt[lo];
  Unit r;
  r.slot = lo;
  r.mt = local % tiles;
  r.n = local / tiles;
  return r;
}

template <bool SWIGLU, bool FUSE>
__global__ void __launch_bounds__(THREADS, 1)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const TcParams p, const __grid_constant__ FuseArgs f) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  SmemLayout& L = *reinterpret_cast<SmemLayout*>(stage_base + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
        if (rows < 0 || rows < p.min_slot_rows || rows > p.max_slot_rows) rows = 0;
        const int32_t mt = (int32_t)((rows + BM - 1) / BM);
        L.mt[s] = mt;
        L.row_base[s] = (int32_t)o0;
        L.row_end[s] = (int32_t)(o0 + rows);
        local += mt * p.n_tiles;
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
        mbar_init(smem_u32(&L.full[i]), 1);   // the producer's expect_tx
        mbar_init(smem_u32(&L.empty[i]), 1);  // the MMA commit
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(smem_u32(&L.tmem_full[i]), 1);
        mbar_init(smem_u32(&L.tmem_empty[i]), 4);  // one per epilogue warp
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<1>(smem_u32(&L.tmem_base));  // whole warp
    if constexpr (FUSE) {
      for (int i = threadIdx.x; i <= f.R; i += THREADS) {
        L.r_off[i] = f.offsets[i];
        if (i < f.R) L.r_cnt[i] = f.counts[i];
      }
    }
    __syncthreads();
    int32_t before = 0;
    for (int w = 0; w < warp; ++w) before += L.warp_sums[w];
    int32_t run = before + x - local;  // exclusive prefix of this thread's group
    for (int i = 0; i < per; ++i) {
      int s = s0 + i;
      if (s < p.nslots) {
        L.pref[s] = run;
        run += L.mt[s] * p.n_tiles;
      }
    }
    if (threadIdx.x == THREADS - 1) {
      int32_t tot = 0;
      for (int w = 0; w < THREADS / 32; ++w) tot += L.warp_sums[w];
      L.pref[p.nslots] = tot;
      L.total_units = tot;
    }
    fence_before();
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
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const Unit un = decode_unit(L, p.nslots, u);
      const int slot = p.slot_lo + un.slot;
      const int32_t row0 = L.row_base[un.slot] + un.mt * BM;
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
          const uint32_t full = smem_u32(&L.full[st]);
          const uint32_t sa = smem_u32(stage_base + (size_t)st * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          mbar_arrive_expect_tx(full, STAGE_BYTES);
          tma_load_2d<1>(sa, &tmA, kb * BK, row0, full, pol_act);
          tma_load_2d<1>(sb, &tmB, kb * BK, brow1, full, pol_w);
          tma_load_2d<1>(sb + B_BOX_BYTES, &tmB, kb * BK, brow2, full, pol_w);
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    // drain: every "stage free" arrival (the MMA commits, which follow the
    // loads they consumed) has happened before exit
    for (uint32_t j = (it >= STAGES ? it - STAGES : 0); j < it; ++j) {
      const uint32_t st = j % STAGES, ph = (j / STAGES) & 1u;
      if (!wait_bar(smem_u32(&L.empty[st]), ph, abort_flag, p.status)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t it = 0, local_tile = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++local_tile) {
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
          const uint32_t sa = smem_u32(stage_base + (size_t)st * STAGE_BYTES);
          const uint64_t adesc = sw128_desc(sa);
          const uint64_t bdesc = sw128_desc(sa + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes per K=16 step in the swizzle row
            mma<1>(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, IDESC, (kb | kk) != 0);
          commit<1>(smem_u32(&L.empty[st]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) commit<1>(smem_u32(&L.tmem_full[acc]));
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    const int row_in_tile = quad * 32 + lane;
    uint32_t local_tile = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++local_tile) {
      const Unit un = decode_unit(L, p.nslots, u);
      const int64_t row0 = (int64_t)L.row_base[un.slot] + (int64_t)un.mt * BM;
      const int64_t row_end = L.row_end[un.slot];
      const uint32_t acc = local_tile & 1u, acc_ph = (local_tile >> 1) & 1u;
      const int64_t row = row0 + row_in_tile;
      const bool valid = row < row_end && row < p.cap;
      int64_t g = -1;  // FUSE: the token of this row, loaded while the MMAs run
      if constexpr (!SWIGLU && FUSE) {
        if (valid) g = f.perm[row];
      }
      if (!wait_bar(smem_u32(&L.tmem_full[acc]), acc_ph, abort_flag, p.status)) break;
      fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * BN;
      __nv_bfloat16* orow = p.out + row * p.out_ld + (int64_t)un.n * p.out_tile_cols;
      // a warp whose 32 rows all lie past the slot's end has nothing to store
      const bool any = row0 + quad * 32 < row_end && row0 + quad * 32 < p.cap;
      if (!any) {
      } else if (SWIGLU) {
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
            float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
            float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
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
      if (lane == 0) mbar_arrive(smem_u32(&L.tmem_empty[acc]));
      if constexpr (!SWIGLU && FUSE) {
        if (any) {
          // the arrival releases this thread's row of the tile and acquires the
          // rows of the token's earlier arrivals
          const bool own = g >= 0 && g < f.rows && fuse_arrive(f, g, un.n, p.status);
          const uint32_t owners = __ballot_sync(0xffffffffu, own);
          __syncwarp();  // the owners' acquires come before every lane's reads
          for (uint32_t m = owners; m != 0; m &= m - 1) {
            const int64_t gg = __shfl_sync(0xffffffffu, g, __ffs(m) - 1);
            fuse_combine_vec(f, p.out, p.cap, gg, un.n * BN + lane * 8, L.r_off, L.r_cnt,
                             p.status);
          }
        }
      }
    }
    if constexpr (!SWIGLU && FUSE)
      fuse_zero_pad_rows(f, L.r_off, L.r_cnt, (int64_t)blockIdx.x * 4 + (warp - 2),
                         (int64_t)gridDim.x * 4, lane);
  }

  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) tmem_dealloc<1>(tmem_base);
}

// ------------------------------------------------------------- host side
// Per device: raise the dynamic shared-memory limit and find how many CTAs fit
// at once (the persistent grid must be fully resident).
bool device_setup(int* max_ctas) {
  static std::mutex mu;
  static int ctas[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (ctas[dev] == 0) {
    const int bytes = (int)smem_bytes();
    if (cudaFuncSetAttribute(ffn_tc_kernel<true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(ffn_tc_kernel<false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(ffn_tc_kernel<false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
      return false;
    int b1 = 0, b2 = 0, b3 = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, ffn_tc_kernel<true, false>, THREADS,
                                                      bytes) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b2, ffn_tc_kernel<false, false>, THREADS,
                                                      bytes) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b3, ffn_tc_kernel<false, true>, THREADS,
                                                      bytes) != cudaSuccess)
      return false;
    int b = b1 < b2 ? b1 : b2;
    b = b < b3 ? b : b3;
    const int n = b * num_sms();
    if (n < 1) return false;
    ctas[dev] = n;
  }
  *max_ctas = ctas[dev];
  return true;
}

// One launch of MM1 + SwiGLU (gemm1) or MM2.
moe_status run_ffn(const FfnArgs& a, const CUtensorMap& mA, const CUtensorMap& mB, bool gemm1,
                   cudaStream_t s) {
  const int nslots = a.slot_hi - a.slot_lo;
  int max_ctas = 0;
  if (!device_setup(&max_ctas)) return MOE_ERR_CUDA;
  // upper bound of m-tiles over the slot range (device-side counts unknown here)
  const int64_t m_bound = (a.cap + BM - 1) / BM + nslots;
  TcParams p;
  p.offsets = a.offsets;
  p.slot_lo = a.slot_lo;
  p.nslots = nslots;
  p.min_slot_rows = a.min_slot_rows;
  p.max_slot_rows = a.max_slot_rows;
  if (a.sm_budget > 0 && a.sm_budget < max_ctas) max_ctas = a.sm_budget;
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
  const int grid = (int)(bound < max_ctas ? bound : max_ctas);
  const FuseArgs none = {};
  if (gemm1) {
    launch(ffn_tc_kernel<true, false>, grid, THREADS, smem_bytes(), s, mA, mB, p, none);
  } else if (a.fuse != nullptr) {
    launch(ffn_tc_kernel<false, true>, grid, THREADS, smem_bytes(), s, mA, mB, p, *a.fuse);
  } else {
    launch(ffn_tc_kernel<false, false>, grid, THREADS, smem_bytes(), s, mA, mB, p, none);
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

bool ffn_uses_pair_kernel(const FfnArgs& a) {
  // rows per slot the sorted buffer can hold on average, over the whole layer
  return a.cap / (a.P > 0 ? a.P : 1) >= kPairRowsPerSlot;
}

moe_status launch_ffn_tc(const FfnArgs& a, cudaStream_t s) {
  const int nslots = a.slot_hi - a.slot_lo;
  if (nslots <= 0 || a.cap <= 0) return MOE_OK;
  if (ffn_uses_pair_kernel(a)) return launch_ffn_tc_swap(a, s);
  return launch_ffn_tc_single(a, s);
}

moe_status launch_ffn_tc_single(const FfnArgs& a, cudaStream_t s) {
  const int nslots = a.slot_hi - a.slot_lo;
  if (nslots <= 0 || a.cap <= 0) return MOE_OK;
  CUtensorMap mA1, mB1, mA2, mB2;
  if (!make_map(&mA1, a.xs, (uint64_t)a.H, (uint64_t)a.cap, 128) ||
      !make_map(&mB1, a.wgu, (uint64_t)a.H, (uint64_t)a.P * 2 * a.I, 128) ||
      !make_map(&mA2, a.h, (uint64_t)a.I, (uint64_t)a.cap, 128) ||
      !make_map(&mB2, a.wd, (uint64_t)a.I, (uint64_t)a.P * a.H, 128))
    return MOE_ERR_CUDA;
  moe_status st = run_ffn(a, mA1, mB1, true, s);
  if (st != MOE_OK) return st;
  return run_ffn(a, mA2, mB2, false, s);
}

}  // namespace moe

// Grouped SwiGLU expert FFN on the 5th-generation tensor cores (sm_103a).
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
// Work tiles are (slot, n-tile, m-tile) with the m-tiles of one slot and
// n-tile adjacent, so CTAs running at the same time share the weight tile
// through L2; tile counts come from the device-side slot offsets, so the host
// never synchronises after dispatch.  A tile's rows start at the slot's
// first row (no alignment needed); rows past the slot's end are computed
// from whatever follows and never stored.
//
// Roles (192 threads, one CTA per SM):
//   warp 0    TMA producer: A box 64x128 and two B boxes 64x128 per stage,
//             128-byte swizzle, 4-stage mbarrier ring (48 KB per stage)
//   warp 1    allocates 512 TMEM columns (two 128x256 fp32 accumulators);
//             lane 0 issues tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32)
//             and tcgen05.commit to release stages and publish accumulators
//   warps 2-5 epilogue: tcgen05.ld 32 columns at a time from the warp's TMEM
//             lane quarter, activation, bf16 pack, 64-byte row stores
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel sets
// MOE_DEV_TIMEOUT, the other roles stop at their next wait, TMEM is freed and
// the kernel returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "ffn_internal.h"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // 64 bf16 = 128 bytes = one swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_HALF_BYTES = 128 * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

// instruction descriptor, kind::f16: D f32, A bf16, B bf16, both K-major,
// N = 256, M = 128
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

struct SmemLayout {
  // stage buffers come first (1024-byte aligned base)
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t total_tiles;
  int32_t warp_sums[THREADS / 32];
  int32_t pref[MOE_MAX_SLOTS + 1];  // tile prefix over the slot range
  int32_t mt[MOE_MAX_SLOTS];        // m-tiles per slot
};
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(SmemLayout);

struct TcParams {
  const int32_t* offsets;
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

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; the whole warp calls it and gets one warp-uniform answer.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag,
                                         uint32_t* status) {
  bool ok = mbar_try_wait(bar, parity);
  if (!ok) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(bar, parity)) {
        ok = true;
        break;
      }
      if ((it & 63u) == 0) {
        if (*abort_flag) break;
        if (globaltimer_ns() - t0 > kTimeoutNs) {
          flag(status, MOE_DEV_TIMEOUT);
          *abort_flag = 1;
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (SBO), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;              // LBO (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;    // SBO
  d |= (uint64_t)1 << 46;              // version
  d |= (uint64_t)2 << 61;              // SWIZZLE_128B
  return d;
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Tile t -> (slot, m-tile, n-tile) through the prefix over the slot range.
struct Tile {
  int slot, m, n;
};
__device__ __forceinline__ Tile decode_tile(const SmemLayout& L, int nslots, int t) {
  int lo = 0, hi = nslots - 1;
  while (lo < hi) {  // largest s with pref[s] <= t
    int mid = (lo + hi + 1) >> 1;
    if (L.pref[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  int local = t - L.pref[lo];
  int mt = L.mt[lo];
  Tile r;
  r.slot = lo;
  r.m = local % mt;
  r.n = local / mt;
  return r;
}

template <bool SWIGLU>
__global__ void __launch_bounds__(THREADS, 1)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  SmemLayout& L = *reinterpret_cast<SmemLayout*>(stage_base + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- tile table: m-tiles per slot, exclusive prefix of tiles
  {
    const int per = (p.nslots + THREADS - 1) / THREADS;
    const int s0 = threadIdx.x * per;
    int32_t local = 0;
    for (int i = 0; i < per; ++i) {
      int s = s0 + i;
      if (s < p.nslots) {
        int64_t rows = (int64_t)p.offsets[p.slot_lo + s + 1] - p.offsets[p.slot_lo + s];
        int32_t mt = rows > 0 ? (int32_t)((rows + BM - 1) / BM) : 0;
        L.mt[s] = mt;
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
        mbar_init(smem_u32(&L.full[i]), 1);
        mbar_init(smem_u32(&L.empty[i]), 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(smem_u32(&L.tmem_full[i]), 1);
        mbar_init(smem_u32(&L.tmem_empty[i]), 128);
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {  // whole warp allocates the accumulators
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(&L.tmem_base)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
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
      L.total_tiles = tot;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  const int total = L.total_tiles;
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
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode_tile(L, p.nslots, t);
      const int slot = p.slot_lo + tl.slot;
      const int32_t row0 = p.offsets[slot] + tl.m * BM;
      const int32_t brow1 = slot * p.b_rows_per_slot + tl.n * p.b_tile_step;
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
          tma_load_2d(sa, &tmA, kb * BK, row0, full, pol_act);
          tma_load_2d(sb, &tmB, kb * BK, brow1, full, pol_w);
          tma_load_2d(sb + B_HALF_BYTES, &tmB, kb * BK, brow2, full, pol_w);
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    // drain: every load issued must land before the CTA can exit
    for (uint32_t j = (it >= STAGES ? it - STAGES : 0); j < it; ++j) {
      const uint32_t st = j % STAGES, ph = (j / STAGES) & 1u;
      volatile int32_t never = 0;
      if (!wait_bar(smem_u32(&L.full[st]), ph, &never, p.status)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t it = 0, local_tile = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++local_tile) {
      const uint32_t acc = local_tile & 1u, acc_ph = (local_tile >> 1) & 1u;
      if (!wait_bar(smem_u32(&L.tmem_empty[acc]), acc_ph ^ 1u, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      bool ok = true;
      for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
        const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
        if (!wait_bar(smem_u32(&L.full[st]), ph, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = smem_u32(stage_base + (size_t)st * STAGE_BYTES);
          const uint64_t adesc = sw128_desc(sa);
          const uint64_t bdesc = sw128_desc(sa + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes per K=16 step inside the swizzle row
            tc_mma(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, IDESC, (kb | kk) != 0);
          tc_commit(smem_u32(&L.empty[st]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(smem_u32(&L.tmem_full[acc]));
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    const int row_in_tile = quad * 32 + lane;
    uint32_t local_tile = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++local_tile) {
      const Tile tl = decode_tile(L, p.nslots, t);
      const int slot = p.slot_lo + tl.slot;
      const int64_t row0 = (int64_t)p.offsets[slot] + (int64_t)tl.m * BM;
      const int64_t row_end = p.offsets[slot + 1];
      const uint32_t acc = local_tile & 1u, acc_ph = (local_tile >> 1) & 1u;
      if (!wait_bar(smem_u32(&L.tmem_full[acc]), acc_ph, abort_flag, p.status)) break;
      tc_fence_after();
      const int64_t row = row0 + row_in_tile;
      const bool valid = row < row_end && row < p.cap;
      const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * BN;
      __nv_bfloat16* orow = p.out + row * p.out_ld + (int64_t)tl.n * p.out_tile_cols;
      if (SWIGLU) {
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c, g);
          tmem_ld32(taddr + 128 + c, u);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float g0 = __uint_as_float(g[2 * e]), g1 = __uint_as_float(g[2 * e + 1]);
            float u0 = __uint_as_float(u[2 * e]), u1 = __uint_as_float(u[2 * e + 1]);
            float h0 = g0 / (1.0f + expf(-g0)) * u0;
            float h1 = g1 / (1.0f + expf(-g1)) * u1;
            pk[e] = pack_bf16x2(h0, h1);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
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
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&L.tmem_empty[acc]));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D bf16 tensor [outer, inner] row-major, box 64 x 128, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool set_smem_attr() {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    if (cudaFuncSetAttribute(ffn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(ffn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess)
      return false;
    done[dev] = true;
  }
  return true;
}

}  // namespace

moe_status launch_ffn_tc(const FfnArgs& a, cudaStream_t s) {
  const int nslots = a.slot_hi - a.slot_lo;
  if (nslots <= 0 || a.cap <= 0) return MOE_OK;
  if (!set_smem_attr()) return MOE_ERR_CUDA;
  CUtensorMap mA1, mB1, mA2, mB2;
  if (!make_map(&mA1, a.xs, (uint64_t)a.H, (uint64_t)a.cap) ||
      !make_map(&mB1, a.wgu, (uint64_t)a.H, (uint64_t)a.P * 2 * a.I) ||
      !make_map(&mA2, a.h, (uint64_t)a.I, (uint64_t)a.cap) ||
      !make_map(&mB2, a.wd, (uint64_t)a.I, (uint64_t)a.P * a.H))
    return MOE_ERR_CUDA;
  const int64_t m_bound = (a.cap + BM - 1) / BM + nslots;
  const int sms = num_sms();

  TcParams p1;
  p1.offsets = a.offsets;
  p1.slot_lo = a.slot_lo;
  p1.nslots = nslots;
  p1.cap = a.cap;
  p1.num_kb = a.H / BK;
  p1.n_tiles = a.I / 128;
  p1.b_rows_per_slot = 2 * a.I;
  p1.b_tile_step = 128;
  p1.b_second = a.I;
  p1.out_ld = a.I;
  p1.out_tile_cols = 128;
  p1.out = static_cast<__nv_bfloat16*>(a.h);
  p1.status = a.status;
  int64_t bound1 = m_bound * p1.n_tiles;
  int grid1 = (int)(bound1 < sms ? bound1 : sms);
  ffn_tc_kernel<true><<<grid1, THREADS, SMEM_BYTES, s>>>(mA1, mB1, p1);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;

  TcParams p2 = p1;
  p2.num_kb = a.I / BK;
  p2.n_tiles = a.H / BN;
  p2.b_rows_per_slot = a.H;
  p2.b_tile_step = BN;
  p2.b_second = 128;
  p2.out_ld = a.H;
  p2.out_tile_cols = BN;
  p2.out = static_cast<__nv_bfloat16*>(a.ys);
  int64_t bound2 = m_bound * p2.n_tiles;
  int grid2 = (int)(bound2 < sms ? bound2 : sms);
  ffn_tc_kernel<false><<<grid2, THREADS, SMEM_BYTES, s>>>(mA2, mB2, p2);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace moe

// Grouped SwiGLU expert FFN on FP8 operands (e4m3 codes with UE8M0 scales per
// 128-value group) on the tcgen05 tensor cores (sm_103a).
//
// SGLang chapter 17, section "prefll 侧的一个必要步骤:per-token-group 量化":
// tokens enter the grouped GEMM as FP8 in groups of 128 features with UE8M0
// scale factors (DeepGEMM's 1x128 fine-grained scaling); the expert weights
// carry one scale per 128 x 128 block.  Opening sections: a DeepSeek-V3 expert
// has gate/up [2048, 7168] and down [7168, 2048].
//
// One 128-deep k-block is exactly one scale block of both operands, so each
// k-block's four MMAs (kind::f8f6f4, K = 32 each) write a fresh fp32 partial
// in tensor memory, and the epilogue warps add it into fp32 registers scaled
// by 2^(e_token + e_weight):
//   acc[row, t] += 2^(ex[t, kb] + ew[row / 128, kb]) * partial_kb[row, t]
// The weights are the MMA's M operand (two 128-row MMAs per K step, 256 rows
// and one 32 KB TMA box per stage) and up to 64 of a slot's tokens its N (one
// weight pass serves them all; a second token group would stream the weights
// from DRAM again), so the accumulators of a unit live in registers: each
// epilogue thread owns two weight rows and 32 token columns.
//   MM1 + SwiGLU: unit = (slot, 128 features f, token group); A = gate rows
//                 f..f+127 and the same up rows (one 3-D TMA box), two MMAs
//                 per K step; the epilogue forms h = silu(gate) * up and
//                 quantises it per token over its 128 features (one group),
//                 writing codes and the scale byte for the down projection.
//   MM2:          unit = (slot, 256 output rows, token group): two MMAs per K
//                 step on the two 128-row halves; bf16 output.
// With few tokens per slot (decode) the weight stream is the whole cost, and
// FP8 weights halve it.
//
// Both GEMMs run in one persistent launch.  The producer of each CTA claims the
// next unit from a ticket in the workspace (all MM1 units of the call, then all
// MM2 units, each in slot order) and hands it to the other roles through a
// four-entry ring in shared memory.  An SM that finishes its last MM1 unit early
// goes on with MM2 units, so neither GEMM leaves a partly empty last round of
// SMs.  An MM2 unit reads h, so its producer (and its epilogue, which reads the
// scale bytes) first waits until every MM1 unit of the slot has been counted.
//
// Roles (352 threads, one CTA per SM):
//   warp 0    TMA producer: weight box + token box per stage
//   warp 1    TMEM allocation; lane 0 issues the MMAs and commits (stage free,
//             partial ready); partials rotate through four TMEM buffers
//   warps 2-9 epilogue, two warps per TMEM lane quarter (token columns 0-31 and
//             32-63): per k-block tcgen05.ld of the partials, release, scale and
//             accumulate; per unit SwiGLU + quantisation or bf16 out
//   warp 10   publisher: makes each MM1 unit's h visible to the other CTAs (a
//             gpu-scope fence, which waits for the stores) and counts it for its
//             slot, off the epilogue's path
// The epilogue's work sets the pace once the weight stream is fast enough, so it
// is kept small: a warp whose columns hold no token of the unit only releases
// the buffer; the others scale only the columns that hold tokens (in groups of
// 8), with packed fp32x2 FMAs, and at the unit's end apply SwiGLU (fast exp and
// divide) and the per-token quantisation to those columns only.  A k-block's factor
// 2^(e_token + e_weight) depends on the token and on which 128-row half of the
// tile a row is in, not on the row, so each lane forms its token's two factors
// once and the warp reads them back from shared memory as broadcasts.
// Every wait (mbarriers and slot counts) is bounded (globaltimer); on expiry
// the kernel sets MOE_DEV_TIMEOUT, the other roles stop at their next wait,
// TMEM is freed and the kernel returns.
#include <mutex>

#include "common.cuh"
#include "ffn_internal.h"
#include "fp8.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BK = 128;     // fp8 values per k-block = one 128-byte swizzle row = one scale group
constexpr int NT = 64;      // tokens per unit
constexpr int CT = 32;      // token columns per epilogue warp
constexpr int THREADS = 352;
constexpr int NPB = 4;      // TMEM partial buffers: the MMAs run up to 4 k-blocks ahead of the epilogue

// tcgen05.wait::ld that also names the destination registers of the load it
// waits for, so the compiler cannot move a use of them above the wait.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// (a0, a1) += (x0, x1) * (f[0], f[1]) as one packed fp32x2 FMA (each lane rounded
// as fmaf); f is a shared-memory pair at the same address in every lane.
__device__ __forceinline__ void fma2_shared(float& a0, float& a1, uint32_t x0, uint32_t x1,
                                            const float* f) {
  uint64_t a, x, g;
  asm volatile("ld.shared.b64 %0, [%1];"
               : "=l"(g)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(f)))
               : "memory");
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(x0), "r"(x1));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(x), "l"(g));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
}

struct F8Cfg {
  static constexpr int A_ROWS = 256;  // 128 gate + 128 up rows, or 256 down rows
  static constexpr int A_BYTES = A_ROWS * BK;
  static constexpr int B_BYTES = NT * BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 5;
  static constexpr int PCOLS = 2 * NT;  // partial columns per buffer (two MMAs)
};
constexpr int UQ = 4;  // claimed units in flight between the producer and the other roles

// Scheduler words at the end of the workspace (int32): the unit ticket, the
// CTAs that have finished, a reserved word, then per slot of the call the
// MM1 units finished (counted once per epilogue column group).
constexpr int kTicket = 0, kDone = 1, kReady = 3;
constexpr int kSyncWords = kReady + MOE_MAX_SLOTS;

struct F8Smem {
  uint64_t full[F8Cfg::STAGES];
  uint64_t empty[F8Cfg::STAGES];
  uint64_t pfull[NPB];
  uint64_t pempty[NPB];
  uint64_t ufull[UQ];   // a claimed unit id is in uring
  uint64_t uempty[UQ];  // the MMA warp and the eight epilogue warps have read it
  int32_t uring[UQ];
  int32_t h_stored;     // epilogue warps that have stored an MM1 unit's h (8 per unit)
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t last_cta;
  int32_t total1, total;
  int32_t warp_sums[THREADS / 32];
  float wmax[2][4][CT];              // per epilogue warp: token maxima of h
  alignas(16) float fac[8][2][CT];   // per epilogue warp: this k-block's token factors
  int32_t pref[MOE_MAX_SLOTS + 1];   // token-group prefix over the slot range
  int32_t row0[MOE_MAX_SLOTS];
  int32_t rows[MOE_MAX_SLOTS];
};
constexpr size_t f8_smem_bytes() {
  return 1024 + (size_t)F8Cfg::STAGES * F8Cfg::STAGE_BYTES + sizeof(F8Smem);
}

// One of the two GEMMs: MM1 (gate/up + SwiGLU, K = H) or MM2 (down, K = I).
struct F8Phase {
  int num_kb;              // K / 128
  int n_tiles;             // weight tiles per slot (128 features of gate + up, or 256 rows)
  int out_ld;              // output row length: I (h codes) or H (y)
  int wscale_rows;         // weight scale rows per slot: 2I/128 or H/128
  int blk_mul, blk_off;    // weight blocks of tile t: t*blk_mul and t*blk_mul + blk_off
  const uint8_t* xscale;   // token scale bytes [cap, K / 128]
  const uint8_t* wscale;   // weight scale bytes [P, wscale_rows, K / 128]
};

struct F8Params {
  const int32_t* offsets;
  int slot_lo, nslots;
  int32_t max_slot_rows;   // slots with more rows get no units (another kernel's)
  int64_t cap;
  int H;
  F8Phase ph[2];
  uint8_t* hq;             // h codes [cap, I]
  uint8_t* hscale;         // h scale bytes [cap, I / 128]
  __nv_bfloat16* y;        // [cap, H]
  int32_t* sync;           // scheduler words
  uint32_t* status;
};

// Token-row tensor maps with boxes of 16, 32, 48 and 64 rows (N = 16 .. 64).
struct TokMaps {
  CUtensorMap m[NT / 16];
  __host__ __device__ const CUtensorMap& operator[](int i) const { return m[i]; }
};

__host__ __device__ __forceinline__ int32_t token_groups(int32_t rows) {
  return rows > 0 ? (rows + NT - 1) / NT : 0;
}

struct F8Unit {
  int ph;    // 0: MM1 + SwiGLU, 1: MM2
  int slot, tile;
  int32_t tok0, ntok;
  int N;  // MMA width: tokens rounded up to 16
};
// Unit u of the call: MM1 units first (slot-major, then tile, then token
// group), then the MM2 units in the same order.
__device__ __forceinline__ F8Unit decode_unit(const F8Smem& L, const F8Params& p, int u) {
  F8Unit r;
  r.ph = u >= L.total1 ? 1 : 0;
  const int v = r.ph ? u - L.total1 : u;
  const int nt = p.ph[r.ph].n_tiles;
  int lo = 0, hi = p.nslots - 1;
  while (lo < hi) {  // largest s with pref[s] * nt <= v
    const int mid = (lo + hi + 1) >> 1;
    if (L.pref[mid] * nt <= v)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int local = v - L.pref[lo] * nt;
  const int32_t T = L.rows[lo];
  const int32_t g = token_groups(T);
  r.slot = lo;
  r.tile = local / g;
  const int32_t grp = local % g;
  r.tok0 = L.row0[lo] + grp * NT;
  const int32_t left = T - grp * NT;
  r.ntok = left < NT ? left : NT;
  r.N = (r.ntok + 15) & ~15;
  return r;
}

__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t* a) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(int32_t* a, int32_t v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
// Generic-proxy writes and async-proxy (TMA) reads of global memory ordered.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ int32_t ld_acquire_cta(const int32_t* a) {
  int32_t v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(a)) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_cta_add(int32_t* a, int32_t v) {
  asm volatile("red.release.cta.shared::cta.add.s32 [%0], %1;" ::"r"(smem_u32(a)), "r"(v)
               : "memory");
}
// Bounded wait of a whole warp until *ctr >= target (acquire); warp-uniform.
template <bool SHARED>
__device__ bool wait_count_t(const int32_t* ctr, int32_t target, volatile int32_t* abort_flag,
                             uint32_t* status) {
  if (__all_sync(0xffffffffu, (SHARED ? ld_acquire_cta(ctr) : ld_acquire_gpu(ctr)) >= target))
    return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (!SHARED) __nanosleep(100);
    if (__all_sync(0xffffffffu, (SHARED ? ld_acquire_cta(ctr) : ld_acquire_gpu(ctr)) >= target))
      return true;
    if ((i & 63u) == 0) {
      bool stop = *abort_flag != 0;
      if (!stop && globaltimer_ns() - t0 > kTimeoutNs) {
        if ((threadIdx.x & 31) == 0) {
          flag(status, MOE_DEV_TIMEOUT);
          *abort_flag = 1;
        }
        stop = true;
      }
      if (__any_sync(0xffffffffu, stop)) return false;
    }
  }
}
// a global counter written by other CTAs / a shared counter of this CTA
__device__ __forceinline__ bool wait_count(const int32_t* ctr, int32_t target,
                                           volatile int32_t* abort_flag, uint32_t* status) {
  return wait_count_t<false>(ctr, target, abort_flag, status);
}
__device__ __forceinline__ bool wait_count_cta(const int32_t* ctr, int32_t target,
                                               volatile int32_t* abort_flag, uint32_t* status) {
  return wait_count_t<true>(ctr, target, abort_flag, status);
}

// Both GEMMs of the grouped FFN in one persistent launch.  A CTA claims units
// from a global ticket: all MM1 units, then all MM2 units; an MM2 unit of a
// slot first waits until that slot's MM1 units have written h.  Every ticket
// below an MM2 ticket is an MM1 unit held by a running CTA, and an MM1 unit
// waits on nothing, so the waits always end.  The claim order balances the two
// GEMMs' unequal units over the SMs (a CTA that finishes its last MM1 unit early
// goes on with MM2 units).
__global__ void __launch_bounds__(THREADS, 1)
    ffn_fp8_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ TokMaps tmB1,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ TokMaps tmB2,
                   const F8Params p) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  using C = F8Cfg;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  F8Smem& L = *reinterpret_cast<F8Smem*>(stage_base + (size_t)STAGES * C::STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- slot table: token groups per slot, exclusive prefix
  {
    const int per = (p.nslots + THREADS - 1) / THREADS;
    const int s0 = threadIdx.x * per;
    int32_t local = 0;
    for (int i = 0; i < per; ++i) {
      const int s = s0 + i;
      if (s < p.nslots) {
        const int32_t o0 = p.offsets[p.slot_lo + s];
        int32_t rows = p.offsets[p.slot_lo + s + 1] - o0;
        if (rows < 0 || rows > p.max_slot_rows) rows = 0;
        L.row0[s] = o0;
        L.rows[s] = rows;
        local += token_groups(rows);
      }
    }
    int32_t x = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) L.warp_sums[warp] = x;
    if (threadIdx.x == 0) {
      L.abort_flag = 0;
      L.h_stored = 0;
      for (int i = 0; i < STAGES; ++i) {
        mbar_init(smem_u32(&L.full[i]), 1);   // the producer's expect_tx
        mbar_init(smem_u32(&L.empty[i]), 1);  // the MMA commit
      }
      for (int i = 0; i < NPB; ++i) {
        mbar_init(smem_u32(&L.pfull[i]), 1);   // the MMA commit
        mbar_init(smem_u32(&L.pempty[i]), 8);  // every epilogue warp
      }
      for (int i = 0; i < UQ; ++i) {
        mbar_init(smem_u32(&L.ufull[i]), 1);   // the producer
        mbar_init(smem_u32(&L.uempty[i]), 10);  // MMA, eight epilogue and the publisher warp
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<1>(smem_u32(&L.tmem_base));
    __syncthreads();
    int32_t before = 0;
    for (int w = 0; w < warp; ++w) before += L.warp_sums[w];
    int32_t run = before + x - local;
    for (int i = 0; i < per; ++i) {
      const int s = s0 + i;
      if (s < p.nslots) {
        L.pref[s] = run;
        run += token_groups(L.rows[s]);
      }
    }
    if (threadIdx.x == THREADS - 1) {
      int32_t tot = 0;
      for (int w = 0; w < THREADS / 32; ++w) tot += L.warp_sums[w];
      L.pref[p.nslots] = tot;
      L.total1 = tot * p.ph[0].n_tiles;
      L.total = tot * (p.ph[0].n_tiles + p.ph[1].n_tiles);
    }
    fence_before();
    __syncthreads();
    fence_after();
  }
  const int total = L.total;
  const uint32_t tmem_base = L.tmem_base;
  volatile int32_t* abort_flag = &L.abort_flag;
  int32_t* ready = p.sync + kReady;
  const int32_t ready_per_group = p.ph[0].n_tiles;  // MM1 units per token group

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_tok = policy_evict_last();
    const uint64_t pol_w = policy_evict_first();
    uint32_t it = 0;
    for (uint32_t q = 0;; ++q) {
      const uint32_t rs = q % UQ, rph = (q / UQ) & 1u;
      if (!wait_bar(smem_u32(&L.uempty[rs]), rph ^ 1u, abort_flag, p.status)) break;
      int u = 0;
      if (lane == 0) {
        u = atomicAdd(p.sync + kTicket, 1);
        if (u < 0 || u >= total) u = -1;  // no unit left
        L.uring[rs] = u;
        mbar_arrive(smem_u32(&L.ufull[rs]));
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u < 0) break;
      const F8Unit un = decode_unit(L, p, u);
      if (un.ph == 1) {  // h of the slot written by the MM1 units (any CTA)
        if (!wait_count(ready + un.slot, ready_per_group * token_groups(L.rows[un.slot]),
                        abort_flag, p.status))
          break;
        fence_proxy_async_global();
      }
      const int32_t slot = p.slot_lo + un.slot;
      const CUtensorMap* bmap = un.ph ? &tmB2[(un.N >> 4) - 1] : &tmB1[(un.N >> 4) - 1];
      const uint32_t tx = (uint32_t)(C::A_BYTES + un.N * BK);
      const int num_kb = p.ph[un.ph].num_kb;
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
        if (!wait_bar(smem_u32(&L.empty[st]), ph ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full = smem_u32(&L.full[st]);
          const uint32_t sa = smem_u32(stage_base + (size_t)st * C::STAGE_BYTES);
          const uint32_t sb = sa + C::A_BYTES;
          const int32_t kc = kb * BK;
          mbar_arrive_expect_tx(full, tx);
          if (un.ph == 0)
            tma_load_3d<1>(sa, &tmA1, kc, un.tile * 128, 2 * slot, full, pol_w);
          else
            tma_load_2d<1>(sa, &tmA2, kc, slot * p.H + un.tile * 256, full, pol_w);
          tma_load_2d<1>(sb, bmap, kc, un.tok0, full, pol_tok);
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    for (uint32_t j = (it >= STAGES ? it - STAGES : 0); j < it; ++j) {
      const uint32_t st = j % STAGES, ph = (j / STAGES) & 1u;
      if (!wait_bar(smem_u32(&L.empty[st]), ph, abort_flag, p.status)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t it = 0;
    for (uint32_t q = 0;; ++q) {
      const uint32_t rs = q % UQ, rph = (q / UQ) & 1u;
      if (!wait_bar(smem_u32(&L.ufull[rs]), rph, abort_flag, p.status)) break;
      const int u = L.uring[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&L.uempty[rs]));
      if (u < 0) break;
      const F8Unit un = decode_unit(L, p, u);
      const uint32_t idesc = idesc_e4m3(128, un.N);
      const int num_kb = p.ph[un.ph].num_kb;
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
        const uint32_t pb = it % NPB, pph = (it / NPB) & 1u;
        if (!wait_bar(smem_u32(&L.full[st]), ph, abort_flag, p.status) ||
            !wait_bar(smem_u32(&L.pempty[pb]), pph ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        fence_after();
        if (lane == 0) {
          const uint32_t sa = smem_u32(stage_base + (size_t)st * C::STAGE_BYTES);
          const uint64_t adesc = sw128_desc(sa);
          const uint64_t adesc_up = sw128_desc(sa + 128 * BK);
          const uint64_t bdesc = sw128_desc(sa + C::A_BYTES);
          const uint32_t d = tmem_base + pb * C::PCOLS;
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {  // +32 bytes per K=32 step in the swizzle row
            mma_e4m3(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, kk != 0);
            mma_e4m3(d + NT, adesc_up + 2 * kk, bdesc + 2 * kk, idesc, kk != 0);
          }
          commit<1>(smem_u32(&L.empty[st]));
          commit<1>(smem_u32(&L.pfull[pb]));
        }
        __syncwarp();
      }
      if (!ok) break;
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;          // TMEM lanes 32q .. 32q+31 = weight rows of the tile
    const int cg = (warp - 2) >> 2;  // token columns 32cg .. 32cg+31 of the unit
    const uint32_t lanes = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(cg * CT);
    const uint32_t bar_id = 1u + (uint32_t)cg;  // the four warps of this column group
    float* fac0 = L.fac[warp - 2][0];  // factors of the first half (gate rows / rows 0-127)
    float* fac1 = L.fac[warp - 2][1];  // and of the second (up rows / rows 128-255)
    uint32_t it = 0;
    for (uint32_t qu = 0;; ++qu) {
      const uint32_t rs = qu % UQ, rph = (qu / UQ) & 1u;
      bool ok = wait_bar(smem_u32(&L.ufull[rs]), rph, abort_flag, p.status);
      const int u = ok ? L.uring[rs] : -1;
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(smem_u32(&L.uempty[rs]));
      F8Unit un{};
      if (ok && u >= 0) {
        un = decode_unit(L, p, u);
        if (un.ph == 1)  // the scale bytes of h are read below
          ok = wait_count(ready + un.slot, ready_per_group * token_groups(L.rows[un.slot]),
                          abort_flag, p.status);
      }
      // the column group's four warps go on, or stop, together (named barriers below)
      ok = named_all(bar_id, 128, ok);
      if (!ok || u < 0) break;
      const bool swiglu = un.ph == 0;
      const F8Phase& P = p.ph[un.ph];
      const int32_t slot = p.slot_lo + un.slot;
      const int t0 = cg * CT;  // first token of this warp's columns
      const bool act = t0 < un.ntok;
      const int ncol = un.ntok - t0;  // columns of this warp that hold tokens (if act)
      // scale bytes, loaded one k-block ahead: lane j holds token t0 + j's byte,
      // every lane the weight blocks' bytes
      const int64_t trow = (int64_t)un.tok0 + t0 + lane;
      const bool tv = t0 + lane < un.ntok && trow < p.cap;
      const uint8_t* xs_row = P.xscale + (tv ? trow : 0) * P.num_kb;
      const int64_t wb0 = (int64_t)slot * P.wscale_rows + un.tile * P.blk_mul;
      const uint8_t* ws0 = P.wscale + wb0 * P.num_kb;
      const uint8_t* ws1 = P.wscale + (wb0 + P.blk_off) * P.num_kb;
      uint32_t nx = tv ? xs_row[0] : 127u, nw0 = ws0[0], nw1 = ws1[0];
      float acc0[CT], acc1[CT];
#pragma unroll
      for (int j = 0; j < CT; ++j) acc0[j] = acc1[j] = 0.0f;
      for (int kb = 0; kb < P.num_kb; ++kb, ++it) {
        const uint32_t ex = nx, ew0 = nw0, ew1 = nw1;
        if (kb + 1 < P.num_kb) {
          nx = tv ? xs_row[kb + 1] : 127u;
          nw0 = ws0[kb + 1];
          nw1 = ws1[kb + 1];
        }
        const uint32_t pb = it % NPB, pph = (it / NPB) & 1u;
        if (!wait_bar(smem_u32(&L.pfull[pb]), pph, abort_flag, p.status)) {
          ok = false;
          it += P.num_kb - kb;
          break;
        }
        fence_after();
        if (!act) {  // no token of the unit in this warp's columns
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&L.pempty[pb]));
          continue;
        }
        const float cx_mine = pow2i((int)ex - 127);
        uint32_t r[32];
        tmem_ld32(lanes + pb * C::PCOLS, r);
        __syncwarp();  // the previous k-block's factors have been read
        fac0[lane] = cx_mine * pow2i((int)ew0 - 127);
        fac1[lane] = cx_mine * pow2i((int)ew1 - 127);
        __syncwarp();
        tmem_wait_ld_regs(r);
#pragma unroll
        for (int g = 0; g < CT; g += 8)
          if (g < ncol)
#pragma unroll
            for (int j = g; j < g + 8; j += 2)
              fma2_shared(acc0[j], acc0[j + 1], r[j], r[j + 1], &fac0[j]);
        tmem_ld32(lanes + pb * C::PCOLS + NT, r);
        tmem_wait_ld_regs(r);
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&L.pempty[pb]));
#pragma unroll
        for (int g = 0; g < CT; g += 8)
          if (g < ncol)
#pragma unroll
            for (int j = g; j < g + 8; j += 2)
              fma2_shared(acc1[j], acc1[j + 1], r[j], r[j + 1], &fac1[j]);
      }
      ok = named_all(bar_id, 128, ok);  // the group's four warps leave together
      if (!ok) break;
      if (swiglu) {
        const int feat = un.tile * 128 + q * 32 + lane;
        // h = silu(gate) * up, then per token one scale over its 128 features; only
        // the column groups of 8 that hold tokens are computed
        float m[CT];
#pragma unroll
        for (int g = 0; g < CT; g += 8) {
          if (g < ncol) {
#pragma unroll
            for (int j = g; j < g + 8; ++j) {
              acc0[j] = __fdividef(acc0[j], 1.0f + __expf(-acc0[j])) * acc1[j];
              m[j] = fabsf(acc0[j]);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
              for (int j = g; j < g + 8; ++j)
                m[j] = fmaxf(m[j], __shfl_xor_sync(0xffffffffu, m[j], off));
            if (lane == 0)
#pragma unroll
              for (int j = g; j < g + 8; ++j) L.wmax[cg][q][j] = m[j];
          }
        }
        named_sync(bar_id, 128);
#pragma unroll
        for (int j = 0; j < CT; ++j) {
          if (j >= ncol) continue;
          const float amax = fmaxf(fmaxf(L.wmax[cg][0][j], L.wmax[cg][1][j]),
                                   fmaxf(L.wmax[cg][2][j], L.wmax[cg][3][j]));
          const int e = fp8_scale_exp(amax);
          const int64_t row = (int64_t)un.tok0 + t0 + j;
          if (t0 + j < un.ntok && row < p.cap) {
            p.hq[row * P.out_ld + feat] = (uint8_t)(e4m3x4(acc0[j] * pow2i(-e), 0.f, 0.f, 0.f) & 0xFFu);
            if (q == 0 && lane == 0)
              p.hscale[row * (P.out_ld / 128) + un.tile] = (uint8_t)(e + 127);
          }
        }
        // this warp's h is stored; the publisher warp makes it visible to the MM2
        // units of other CTAs
        __syncwarp();
        if (lane == 0) red_release_cta_add(&L.h_stored, 1);
        named_sync(bar_id, 128);  // the maxima are read before the next unit writes them
      } else {
        const int feat = un.tile * 256 + q * 32 + lane;  // and feat + 128 (second half)
#pragma unroll
        for (int j = 0; j < CT; ++j) {
          if (j >= ncol) continue;
          const int64_t row = (int64_t)un.tok0 + t0 + j;
          if (t0 + j < un.ntok && row < p.cap) {
            p.y[row * P.out_ld + feat] = __float2bfloat16_rn(acc0[j]);
            p.y[row * P.out_ld + feat + 128] = __float2bfloat16_rn(acc1[j]);
          }
        }
      }
    }
  }

  else {
    // ------------------------------------------------------------ publisher
    int32_t mm1_units = 0;
    for (uint32_t qu = 0;; ++qu) {
      const uint32_t rs = qu % UQ, rph = (qu / UQ) & 1u;
      if (!wait_bar(smem_u32(&L.ufull[rs]), rph, abort_flag, p.status)) break;
      const int u = L.uring[rs];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&L.uempty[rs]));
      if (u < 0) break;
      if (u >= L.total1) continue;  // an MM2 unit publishes nothing
      const F8Unit un = decode_unit(L, p, u);
      ++mm1_units;
      if (!wait_count_cta(&L.h_stored, 8 * mm1_units, abort_flag, p.status)) break;
      if (lane == 0) {
        __threadfence();              // the eight warps' h stores, at gpu scope
        fence_proxy_async_global();   // and for the TMA loads that read them
        red_release_gpu_add(ready + un.slot, 1);
      }
      __syncwarp();
    }
  }

  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) tmem_dealloc<1>(tmem_base);
  // The last CTA out checks the scheduler words against this call's units and
  // clears them for the next call.  Every other CTA has made its last claim and
  // count before adding itself to kDone.
  if (threadIdx.x == 0) {
    __threadfence();
    L.last_cta = atomicAdd(p.sync + kDone, 1) == (int)gridDim.x - 1;
    __threadfence();
  }
  __syncthreads();
  if (L.last_cta) {
    const bool timed_out =
        p.status != nullptr && (ld_acquire_gpu(reinterpret_cast<const int32_t*>(p.status)) &
                                (int32_t)MOE_DEV_TIMEOUT) != 0;
    bool bad = false;
    for (int s = threadIdx.x; s < p.nslots; s += THREADS) {
      if (ld_acquire_gpu(ready + s) != ready_per_group * token_groups(L.rows[s])) bad = true;
      ready[s] = 0;
    }
    if (threadIdx.x == 0) {
      // each CTA's producer claimed every unit ticket once and one ticket past the end
      if (ld_acquire_gpu(p.sync + kTicket) != total + (int)gridDim.x) bad = true;
      p.sync[kTicket] = 0;
      p.sync[kDone] = 0;
    }
    if (bad && !timed_out) flag(p.status, MOE_DEV_BAD_WORKSPACE);
    __threadfence();
  }
}

// ------------------------------------------------------------- host side
bool f8_setup(int* max_ctas) {
  static std::mutex mu;
  static int ctas[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (ctas[dev] == 0) {
    const int bytes = (int)f8_smem_bytes();
    if (cudaFuncSetAttribute(ffn_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess)
      return false;
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, ffn_fp8_kernel, THREADS, bytes) !=
            cudaSuccess ||
        b < 1)
      return false;
    ctas[dev] = b * num_sms();
  }
  *max_ctas = ctas[dev];
  return true;
}

struct F8Args {
  const uint8_t *xq, *xscale;
  const int32_t* offsets;
  int P, slot_lo, slot_hi;
  int64_t cap;
  const uint8_t *wguq, *wgus, *wdq, *wds;
  int H, I;
  uint8_t *hq, *hs;
  __nv_bfloat16* y;
  int32_t* sync;
  uint32_t* status;
  int32_t max_slot_rows;
};

moe_status run_f8(const F8Args& a, cudaStream_t s) {
  int max_ctas = 0;
  if (!f8_setup(&max_ctas)) return MOE_ERR_CUDA;
  CUtensorMap mA1, mA2;
  TokMaps mB1, mB2;
  bool ok = make_map_u8_gate_up(&mA1, a.wguq, a.H, a.I, a.P, 128) &&
            make_map_u8(&mA2, a.wdq, a.I, (uint64_t)a.P * a.H, 256);
  for (int i = 0; i < NT / 16 && ok; ++i)
    ok = make_map_u8(&mB1.m[i], a.xq, a.H, (uint64_t)a.cap, 16u * (i + 1)) &&
         make_map_u8(&mB2.m[i], a.hq, a.I, (uint64_t)a.cap, 16u * (i + 1));
  if (!ok) return MOE_ERR_CUDA;
  F8Params p;
  p.offsets = a.offsets;
  p.slot_lo = a.slot_lo;
  p.nslots = a.slot_hi - a.slot_lo;
  p.max_slot_rows = a.max_slot_rows;
  p.cap = a.cap;
  p.H = a.H;
  F8Phase& m1 = p.ph[0];
  m1.num_kb = a.H / BK;
  m1.n_tiles = a.I / 128;
  m1.out_ld = a.I;
  m1.wscale_rows = 2 * a.I / 128;
  m1.blk_mul = 1;
  m1.blk_off = a.I / 128;
  m1.xscale = a.xscale;
  m1.wscale = a.wgus;
  F8Phase& m2 = p.ph[1];
  m2.num_kb = a.I / BK;
  m2.n_tiles = a.H / 256;
  m2.out_ld = a.H;
  m2.wscale_rows = a.H / 128;
  m2.blk_mul = 2;
  m2.blk_off = 1;
  m2.xscale = a.hs;
  m2.wscale = a.wds;
  p.hq = a.hq;
  p.hscale = a.hs;
  p.y = a.y;
  p.sync = a.sync;
  p.status = a.status;
  // upper bound of units (device-side counts unknown here)
  const int64_t bound = (a.cap / NT + p.nslots) * (int64_t)(m1.n_tiles + m2.n_tiles);
  const int grid = (int)(bound < max_ctas ? bound : max_ctas);
  launch(ffn_fp8_kernel, grid, THREADS, f8_smem_bytes(), s, mA1, mB1, mA2, mB2, p);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Workspace: h codes [cap, I], h scale bytes [cap, I/128], then (the pair
// kernel's path) h in fp32 [cap, I], then the scheduler's words.
size_t hscale_offset(int64_t cap, int I) { return ((size_t)cap * I + 255) & ~(size_t)255; }
size_t h32_offset(int64_t cap, int I) {
  return (hscale_offset(cap, I) + (size_t)cap * (I / 128) + 255) & ~(size_t)255;
}
size_t sync_offset(int64_t cap, int I) {
  return (h32_offset(cap, I) + (size_t)cap * I * sizeof(float) + 255) & ~(size_t)255;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_grouped_ffn_fp8_ws_bytes(int64_t cap, int I) {
  if (cap < 0 || I < 128 || I % 128 != 0) return 0;
  return sync_offset(cap, I) + sizeof(int32_t) * kSyncWords;
}

extern "C" moe_status moe_grouped_ffn_fp8(const uint8_t* d_sorted_q,
                                          const uint8_t* d_sorted_scales,
                                          const int32_t* d_offsets_P, int P, int slot_lo,
                                          int slot_hi, int64_t cap, const uint8_t* d_w_gate_up_q,
                                          const uint8_t* d_w_gate_up_scales,
                                          const uint8_t* d_w_down_q,
                                          const uint8_t* d_w_down_scales, int H, int I,
                                          void* d_out_sorted, void* d_ws, size_t ws_bytes,
                                          uint32_t* d_status, void* stream) {
  if (P < 1 || P > MOE_MAX_SLOTS || slot_lo < 0 || slot_hi > P || slot_lo > slot_hi || cap < 0 ||
      cap > INT32_MAX || H < 256 || H % 256 != 0 || I < 128 || I % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if ((int64_t)P * H > INT32_MAX || (int64_t)2 * P * I > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (cap == 0 || slot_lo == slot_hi) return MOE_OK;
  if (d_sorted_q == nullptr || d_sorted_scales == nullptr || d_offsets_P == nullptr ||
      d_w_gate_up_q == nullptr || d_w_gate_up_scales == nullptr || d_w_down_q == nullptr ||
      d_w_down_scales == nullptr || d_out_sorted == nullptr || d_ws == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(d_sorted_q) || !aligned16(d_w_gate_up_q) || !aligned16(d_w_down_q) ||
      !aligned16(d_out_sorted) || !aligned16(d_ws))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_grouped_ffn_fp8_ws_bytes(cap, I)) return MOE_ERR_CAPACITY;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
  auto aligned4 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 3u) == 0; };
  const bool pair_ok = H % 512 == 0 && I % 512 == 0 && aligned4(d_sorted_scales) &&
                       aligned4(d_w_gate_up_scales) && aligned4(d_w_down_scales);
  // many rows per slot: every slot on SM pairs with block-scaled MMAs; a
  // skewed layer (fewer rows per slot on average, EPLB): its slots of 192 or
  // more rows there, the others on the single-SM kernel after them
  const bool all_pair = pair_ok && ffn_fp8_uses_pair_kernel(cap, P, H, I);
  const bool split = pair_ok && !all_pair && ffn_fp8_splits_slots(cap, P, H, I);
  if (all_pair || split) {
    uint8_t* ws = static_cast<uint8_t*>(d_ws);
    F8SwapArgs f;
    f.xq = d_sorted_q;
    f.xs = d_sorted_scales;
    f.offsets = d_offsets_P;
    f.P = P;
    f.slot_lo = slot_lo;
    f.slot_hi = slot_hi;
    f.cap = cap;
    f.wguq = d_w_gate_up_q;
    f.wgus = d_w_gate_up_scales;
    f.wdq = d_w_down_q;
    f.wds = d_w_down_scales;
    f.H = H;
    f.I = I;
    f.h32 = reinterpret_cast<float*>(ws + h32_offset(cap, I));
    f.hq = ws;
    f.hs = ws + hscale_offset(cap, I);
    f.y = static_cast<__nv_bfloat16*>(d_out_sorted);
    f.status = d_status;
    f.min_slot_rows = split ? kFp8PairRows : 0;
    const moe_status st = launch_ffn_fp8_swap(f, as_stream(stream));
    if (st != MOE_OK || !split) return st;
  }
  F8Args a;
  a.xq = d_sorted_q;
  a.xscale = d_sorted_scales;
  a.offsets = d_offsets_P;
  a.P = P;
  a.slot_lo = slot_lo;
  a.slot_hi = slot_hi;
  a.cap = cap;
  a.wguq = d_w_gate_up_q;
  a.wgus = d_w_gate_up_scales;
  a.wdq = d_w_down_q;
  a.wds = d_w_down_scales;
  a.H = H;
  a.I = I;
  a.hq = static_cast<uint8_t*>(d_ws);
  a.hs = static_cast<uint8_t*>(d_ws) + hscale_offset(cap, I);
  a.y = static_cast<__nv_bfloat16*>(d_out_sorted);
  a.sync = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(d_ws) + sync_offset(cap, I));
  a.status = d_status;
  a.max_slot_rows = split ? kFp8PairRows - 1 : INT32_MAX;
  return run_f8(a, as_stream(stream));
}

// Grouped SwiGLU expert FFN on FP8 operands with the expert weights as the
// MMA's M operand (sm_103a, two-SM tcgen05 pairs, block-scaled MMA): the FP8
// path for many tokens per slot.
//
// SGLang chapter 17, section "prefll 侧的一个必要步骤:per-token-group 量化":
// tokens enter the grouped GEMM as e4m3 in groups of 128 features with UE8M0
// scale factors, and the expert weights carry one scale per 128 x 128 block.
// Opening sections: a DeepSeek-V3 expert has gate/up [2048, 7168] and down
// [7168, 2048].  Each GEMM sums, per output, 2^(e_token + e_block) times the
// e4m3 products of every 128-deep block in fp32 (moe_grouped_ffn_fp8).
//
// The structure is that of the bf16 pair kernel (ffn_tc_swap.cu): one unit is
// (slot, weight tile, token group of up to 320 tokens), the weight rows fill
// the pair's M = 256 (128 per SM) and the tokens are N, so every weight tile
// crosses HBM once per slot.  A stage holds one 128-deep k-block: 128 e4m3 per
// row are one 128-byte swizzle row, so the boxes have the bf16 kernel's bytes
// and twice its depth.  The MMA is tcgen05.mma.cta_group::2.kind::mxf8f6f4.
// block_scale.scale_vec::1X: the tensor core applies the scales itself, so
// the fp32 accumulators stay in tensor memory for the whole unit and the
// epilogue runs once per unit (no per-block promotion).
//
// Scale factors sit in tensor memory: scale of row r of 128 in lane r mod 32 of
// every lane quarter, column r / 32, one 32-bit cell holding four scale bytes;
// the MMA picks one byte per instruction (the descriptor's scale-factor IDs).
// A cell here holds the bytes of four consecutive k-blocks -- exactly one
// 32-bit word of a row of the scale arrays -- and every K = 32 step of k-block
// j of the four takes byte j.  Each CTA holds the scales of its 128 weight rows
// (rows 0-63 of an MM1 tile are gate rows, 64-127 up rows: two blocks) and
// those of all N token columns of each MMA, in the MMA's column order.  Four
// scale warps per CTA (one per lane quarter) write a slot per four k-blocks
// with tcgen05.st into a four-slot ring of 16 columns (weights 4, first MMA's
// tokens 8, second MMA's 4), from words loaded a slot ahead, and report it to
// the leader's "scales ready" barrier; the MMA commit after the slot's fourth
// k-block frees it in both CTAs.
//
// Tensor memory: two accumulator halves of 224 columns, each with a 96-column
// head for the other half's unit's tail (the bf16 kernel's scheme with 256 and
// 64), then the scale ring (columns 448-511).  A unit's first MMA takes up to
// 224 tokens, the second the rest (up to 96).
//
//   MM1 + SwiGLU: as the bf16 kernel; h is written in fp32 and quantised per
//                 token over groups of 128 features by its own launch
//                 (moe_quantize_fp8_groups): its e4m3 codes are those of the
//                 exact activations except where one lies within fp32 rounding
//                 of a rounding tie (a bf16 copy of h would move many more).
//   MM2:          bf16 output rows, as the bf16 kernel.
//
// Roles (448 threads, one CTA per SM, clusters of two):
//   warp 0      TMA producer (both CTAs): weight box and token box per stage
//   warp 1      TMEM allocation; in the leader CTA lane 0 issues the MMAs
//   warps 2-9   epilogue
//   warps 10-13 scale warps
// Every wait is bounded (globaltimer); on expiry the kernel sets
// MOE_DEV_TIMEOUT, the other roles stop at their next wait, TMEM is freed and
// the kernel returns.
#include "common.cuh"
#include "ffn_internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BK = 128;                         // 128 e4m3 = one 128-byte swizzle row = one scale group
constexpr int A_ROWS = 128;                     // weight rows per CTA
constexpr int A_BYTES = A_ROWS * BK;            // 16 KB
constexpr int NMAX = 320;                       // tokens per unit
constexpr int N0_MAX = 224;                     // largest N of the first MMA (one TMEM half)
constexpr int B_ROWS = NMAX / 2;                // token rows per CTA
constexpr int B_BYTES = B_ROWS * BK;            // 20 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 36 KB
constexpr int STAGES = 5;
constexpr int THREADS = 448;
constexpr int SF_WARP0 = 10;                    // warps 10-13: scale factors
constexpr int HALF_COLS = 224;                  // one TMEM half: a unit's main accumulator
constexpr int HEAD_COLS = 96;                   // head of a half: the other half's unit's tail
constexpr int SF_BASE = 2 * HALF_COLS;          // scale ring: columns 448-511
constexpr int SF_STAGES = 4;                    // slots of four k-blocks each
constexpr int SF_COLS = 16;                     // per slot: weights 0-3, tokens of MMA 0 4-11, of MMA 1 12-15
constexpr int SFB0 = 4, SFB1 = 12;
static_assert(SF_BASE + SF_STAGES * SF_COLS <= 512, "tensor memory columns");
constexpr int EPI_WARPS = 8;                    // two per TMEM lane quarter
constexpr int XCH_BYTES = 32 * 32 * 4;          // per epilogue warp: 32 lanes x 32 fp32
constexpr int NUM_BOXES = B_ROWS / 8;           // token boxes of 8, 16, ..., 160 rows

struct Maps {
  CUtensorMap a;              // e4m3 weights: MM1 3-D box 128 x 64 x 2 (gate, up), MM2 box 128 x 128
  CUtensorMap b[NUM_BOXES];   // e4m3 tokens, box 128 x 8(i+1)
};

struct SwapParams {
  const int32_t* offsets;
  int slot_lo, nslots;
  int32_t min_slot_rows, max_slot_rows;  // slots outside [min, max] rows get no units
  int64_t cap;
  int num_kb;
  int n_tiles;          // weight tiles per slot
  int gemm1;            // MM1: weight box at (k, row in the gate/up half, 2 * slot)
  int a_rows_per_slot;  // MM2: H rows of the down projection per slot
  int a_tile_step;      // weight rows per tile and pair: 128 features (MM1) or 256 rows (MM2)
  int a_cta_step;       // first weight row of CTA 1 within a tile: 64 (MM1) or 128 (MM2)
  int out_ld;
  void* out;            // MM1: float h; MM2: bf16 y
  uint32_t* status;
  // scale bytes: weights [slot][block][k-group], tokens [row][k-group]
  const uint8_t* a_scale;
  int a_blocks;         // 128-row weight blocks per slot (2I/128 or H/128)
  int a_up_block;       // MM1: block of up row 0 within the slot (I/128); MM2: 0
  const uint8_t* b_scale;
  int k_groups;         // 128-deep k-blocks of the GEMM (= num_kb)
};

struct SmemLayout {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t sf_full[SF_STAGES];   // leader: both CTAs' scale warps wrote the slot
  uint64_t sf_empty[SF_STAGES];  // the leader's MMA commit (multicast): the slot was read
  uint64_t tmem_full[2];    // per unit parity: the unit's MMAs are done
  uint64_t tmem_empty[4];   // per TMEM region (head 0, rest 0, head 1, rest 1): drained
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t total_units;
  int32_t warp_sums[THREADS / 32];
  int32_t pref[MOE_MAX_SLOTS + 1];  // unit prefix over the slot range
  int32_t row0[MOE_MAX_SLOTS];      // first sorted row of the slot
  int32_t rows[MOE_MAX_SLOTS];      // tokens of the slot
};
constexpr size_t kEpiBytes = (size_t)EPI_WARPS * XCH_BYTES;
constexpr size_t smem_bytes() {
  return 1024 + (size_t)STAGES * STAGE_BYTES + kEpiBytes + sizeof(SmemLayout);
}
static_assert(smem_bytes() <= 232448, "shared memory per CTA");

__host__ __device__ __forceinline__ int32_t token_groups(int32_t rows) {
  return rows > 0 ? (rows + NMAX - 1) / NMAX : 0;
}

struct SUnit {
  int slot, tile;
  int32_t tok0;  // first sorted row of the token group
  int32_t ntok;  // tokens in the group (1..NMAX)
  int N0, N1;    // MMA widths: tokens rounded up to 16, split at 224
};
// Unit u -> (slot, tile, token group).  The token groups of one (slot, tile)
// are adjacent, then the tiles of one slot, so units running at the same time
// share weight tiles or token rows through L2.
__device__ __forceinline__ SUnit decode_unit(const SmemLayout& L, int nslots, int u) {
  int lo = 0, hi = nslots - 1;
  while (lo < hi) {  // largest s with pref[s] <= u
    const int mid = (lo + hi + 1) >> 1;
    if (L.pref[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int local = u - L.pref[lo];
  const int32_t T = L.rows[lo];
  const int32_t g = token_groups(T);
  SUnit r;
  r.slot = lo;
  r.tile = local / g;
  const int32_t grp = local % g;
  r.tok0 = L.row0[lo] + grp * NMAX;
  const int32_t left = T - grp * NMAX;
  r.ntok = left < NMAX ? left : NMAX;
  const int N = (r.ntok + 15) & ~15;
  r.N0 = N < N0_MAX ? N : N0_MAX;
  r.N1 = N - r.N0;
  return r;
}

// Token of accumulator column `col` of the unit's first (buf 0) or second
// (buf 1) MMA, relative to the group's first row: CTA c holds rows
// [c*h, (c+1)*h), h = N/2; the first MMA reads rows [0, N0/2) of each CTA,
// the second rows [N0/2, h).  -1 where the column is past the MMA's width.
__device__ __forceinline__ int col_token(const SUnit& un, int buf, int col) {
  const int h = (un.N0 + un.N1) >> 1;
  const int w = buf ? un.N1 : un.N0, half = w >> 1, base = buf ? un.N0 >> 1 : 0;
  if (col >= w) return -1;
  return col < half ? base + col : h + base + (col - half);
}

// Block-scaled e4m3 MMA of the pair: D (+)= (A . sA) (B . sB)^T, K = 32.
__device__ __forceinline__ void mma_f8bs(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// Instruction descriptor of kind::mxf8f6f4 with block scales: A and B e4m3,
// both K-major, UE8M0 scales (bit 23), N >> 3 at bit 17, M >> 4 at bit 24; the
// scale byte of each cell the MMA takes (0-3) at bits 29-30 for A and 4-5 for B.
__host__ __device__ constexpr uint32_t idesc_f8bs(int M, int N) {
  return ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_sf_byte(uint32_t idesc, uint32_t j) {
  return idesc | (j << 29) | (j << 4);
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c,
                                         uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::
                   "r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
               "r"(v[7])
               : "memory");
}
// wait_bar with a cluster-scope acquire (the peer CTA's scale warps arrive too).
__device__ __forceinline__ bool try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool wait_bar_cl(uint32_t bar, uint32_t parity,
                                            volatile int32_t* abort_flag, uint32_t* status) {
  bool ok = try_wait_cl(bar, parity);
  if (!ok) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
      if (try_wait_cl(bar, parity)) {
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

template <bool SWIGLU>
__global__ void __launch_bounds__(THREADS, 1)
    ffn_f8swap_kernel(const __grid_constant__ Maps maps, const SwapParams p) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  float* xch = reinterpret_cast<float*>(stage_base + (size_t)STAGES * STAGE_BYTES);
  SmemLayout& L = *reinterpret_cast<SmemLayout*>(reinterpret_cast<uint8_t*>(xch) + kEpiBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;
  const int cid = blockIdx.x / 2, ncl = gridDim.x / 2;

  // ---- unit table: token groups per slot, exclusive prefix of units
  {
    const int per = (p.nslots + THREADS - 1) / THREADS;
    const int s0 = threadIdx.x * per;
    int32_t local = 0;
    for (int i = 0; i < per; ++i) {
      const int s = s0 + i;
      if (s < p.nslots) {
        const int32_t o0 = p.offsets[p.slot_lo + s];
        int32_t rows = p.offsets[p.slot_lo + s + 1] - o0;
        if (rows < 0 || rows < p.min_slot_rows || rows > p.max_slot_rows) rows = 0;
        L.row0[s] = o0;
        L.rows[s] = rows;
        local += token_groups(rows) * p.n_tiles;
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
      for (int i = 0; i < STAGES; ++i) {
        mbar_init(smem_u32(&L.full[i]), 1);   // leader: its producer's expect_tx
        mbar_init(smem_u32(&L.empty[i]), 1);  // the leader's MMA commit
      }
      for (int i = 0; i < SF_STAGES; ++i) {
        mbar_init(smem_u32(&L.sf_full[i]), 8);   // leader: 4 scale warps of each CTA
        mbar_init(smem_u32(&L.sf_empty[i]), 1);  // the leader's MMA commit
      }
      for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&L.tmem_full[i]), 1);
      for (int i = 0; i < 4; ++i)
        mbar_init(smem_u32(&L.tmem_empty[i]), 2 * EPI_WARPS);  // every epilogue warp of the pair
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<2>(smem_u32(&L.tmem_base));  // whole warp, both CTAs
    __syncthreads();
    int32_t before = 0;
    for (int w = 0; w < warp; ++w) before += L.warp_sums[w];
    int32_t run = before + x - local;
    for (int i = 0; i < per; ++i) {
      const int s = s0 + i;
      if (s < p.nslots) {
        L.pref[s] = run;
        run += token_groups(L.rows[s]) * p.n_tiles;
      }
    }
    if (threadIdx.x == THREADS - 1) {
      int32_t tot = 0;
      for (int w = 0; w < THREADS / 32; ++w) tot += L.warp_sums[w];
      L.pref[p.nslots] = tot;
      L.total_units = tot;
    }
    fence_before();
    cluster_sync();  // the leader's barriers exist before the peer signals them
    fence_after();
  }
  const int total = L.total_units;
  const uint32_t tmem_base = L.tmem_base;
  volatile int32_t* abort_flag = &L.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_tok = policy_evict_last();
    const uint64_t pol_w = policy_evict_first();
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.a))
                   : "memory");
    }
    uint32_t it = 0;
    for (int u = cid; u < total; u += ncl) {
      const SUnit un = decode_unit(L, p.nslots, u);
      const int32_t wrow = un.tile * p.a_tile_step + (int32_t)crank * p.a_cta_step;
      const int32_t slot = p.slot_lo + un.slot;
      const int h = (un.N0 + un.N1) >> 1;  // token rows of this CTA
      const int32_t brow = un.tok0 + (int32_t)crank * h;
      const CUtensorMap* bmap = &maps.b[(h >> 3) - 1];
      const uint32_t tx = 2u * (uint32_t)(A_BYTES + h * BK);  // both CTAs
      bool ok = true;
      for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
        const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
        if (!wait_bar(smem_u32(&L.empty[st]), ph ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full_local = smem_u32(&L.full[st]);
          const uint32_t full = map_to_rank(full_local, 0);
          const uint32_t sa = smem_u32(stage_base + (size_t)st * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          const int32_t kc = kb * BK;
          if (leader) mbar_arrive_expect_tx(full_local, tx);
          if (p.gemm1)
            tma_load_3d<2>(sa, &maps.a, kc, wrow, 2 * slot, full, pol_w);
          else
            tma_load_2d<2>(sa, &maps.a, kc, slot * p.a_rows_per_slot + wrow, full, pol_w);
          tma_load_2d<2>(sb, bmap, kc, brow, full, pol_tok);
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
      uint32_t it = 0, seq = 0;
      uint32_t uses[4] = {0, 0, 0, 0};  // earlier uses of each TMEM region
      for (int u = cid; u < total; u += ncl, ++seq) {
        const SUnit un = decode_unit(L, p.nslots, u);
        const uint32_t hm = seq & 1u;  // the unit's half; its tail goes to the other head
        // this half's head and rest, and for a tail the other half's head
        auto take = [&](uint32_t r) {
          const bool got = wait_bar(smem_u32(&L.tmem_empty[r]), (uses[r] & 1u) ^ 1u, abort_flag,
                                    p.status);
          ++uses[r];
          return got;
        };
        if (!take(2 * hm) || !take(2 * hm + 1) || (un.N1 && !take(2 * (hm ^ 1u)))) break;
        fence_after();
        const uint32_t d0 = tmem_base + hm * HALF_COLS;
        const uint32_t d1 = tmem_base + (hm ^ 1u) * HALF_COLS;
        const uint32_t id0 = idesc_f8bs(256, un.N0);
        const uint32_t id1 = idesc_f8bs(256, un.N1 ? un.N1 : 16);
        const uint32_t boff1 = (uint32_t)(un.N0 >> 1) * BK;
        bool ok = true;
        for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
          const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
          const uint32_t bt = it >> 2, j = it & 3u;  // scale slot use and its byte
          const uint32_t sf = bt % SF_STAGES, phs = (bt / SF_STAGES) & 1u;
          if (!wait_bar(smem_u32(&L.full[st]), ph, abort_flag, p.status) ||
              (j == 0 && !wait_bar_cl(smem_u32(&L.sf_full[sf]), phs, abort_flag, p.status))) {
            ok = false;
            break;
          }
          fence_after();
          if (lane == 0) {
            const uint32_t sfa = tmem_base + SF_BASE + sf * SF_COLS;
            const uint32_t i0 = idesc_sf_byte(id0, j), i1 = idesc_sf_byte(id1, j);
            const uint32_t sa = smem_u32(stage_base + (size_t)st * STAGE_BYTES);
            const uint64_t adesc = sw128_desc(sa);
            const uint64_t bdesc0 = sw128_desc(sa + A_BYTES);
            const uint64_t bdesc1 = sw128_desc(sa + A_BYTES + boff1);
#pragma unroll
            for (int kk = 0; kk < BK / 32; ++kk) {  // +32 bytes per K=32 step in the swizzle row
              mma_f8bs(d0, adesc + 2 * kk, bdesc0 + 2 * kk, i0, sfa, sfa + SFB0, (kb | kk) != 0);
              if (un.N1)
                mma_f8bs(d1, adesc + 2 * kk, bdesc1 + 2 * kk, i1, sfa, sfa + SFB1,
                         (kb | kk) != 0);
            }
            commit<2>(smem_u32(&L.empty[st]));
            if (j == 3) commit<2>(smem_u32(&L.sf_empty[sf]));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) commit<2>(smem_u32(&L.tmem_full[hm]));
        __syncwarp();
      }
    }
  } else if (warp >= SF_WARP0) {
    // ------------------------------------------------------------ scale warps
    // this warp writes lane quarter (warp & 3) of every slot of the scale ring
    const uint32_t lanes = tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t it = 0;
    bool ok = true;
    for (int u = cid; u < total && ok; u += ncl) {
      const SUnit un = decode_unit(L, p.nslots, u);
      const int32_t slot = p.slot_lo + un.slot;
      const int32_t wrow = un.tile * p.a_tile_step + (int32_t)crank * p.a_cta_step;
      // weight blocks of this CTA's rows 0-63 and 64-127 (MM1: gate and up)
      const int blk0 = wrow / 128, blk1 = p.gemm1 ? p.a_up_block + wrow / 128 : wrow / 128;
      const uint8_t* arow0 = p.a_scale + ((int64_t)slot * p.a_blocks + blk0) * p.k_groups;
      const uint8_t* arow1 = p.a_scale + ((int64_t)slot * p.a_blocks + blk1) * p.k_groups;
      // token of column lane + 32c of each MMA (-1: no token there)
      const int ncol0 = (un.N0 + 31) >> 5, ncol1 = (un.N1 + 31) >> 5;
      int64_t r0[7], r1[3];
#pragma unroll
      for (int c = 0; c < 7; ++c) {
        const int t = c < ncol0 ? col_token(un, 0, lane + 32 * c) : -1;
        const int64_t d = (int64_t)un.tok0 + t;
        r0[c] = (t >= 0 && t < un.ntok && d < p.cap) ? d : -1;
      }
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        const int t = c < ncol1 ? col_token(un, 1, lane + 32 * c) : -1;
        const int64_t d = (int64_t)un.tok0 + t;
        r1[c] = (t >= 0 && t < un.ntok && d < p.cap) ? d : -1;
      }
      // scale words of k-blocks g .. g+3 (one word per row: a byte per k-block),
      // loaded a batch ahead of the one being written
      struct Words {
        uint32_t a[2], t0[7], t1[3];
      };
      auto load = [&](int g, Words& w) {
        w.a[0] = __ldg(reinterpret_cast<const uint32_t*>(arow0 + g));
        w.a[1] = __ldg(reinterpret_cast<const uint32_t*>(arow1 + g));
#pragma unroll
        for (int c = 0; c < 7; ++c)
          w.t0[c] = r0[c] >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(p.b_scale +
                                                                         r0[c] * p.k_groups + g))
                               : 0x7F7F7F7Fu;
#pragma unroll
        for (int c = 0; c < 3; ++c)
          w.t1[c] = r1[c] >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(p.b_scale +
                                                                         r1[c] * p.k_groups + g))
                               : 0x7F7F7F7Fu;
      };
      Words cur, nxt;
      load(0, cur);
      for (int g = 0; g < p.num_kb && ok; g += 4, ++it) {
        if (g + 4 < p.num_kb) load(g + 4, nxt);
        const uint32_t sf = it % SF_STAGES, ph = (it / SF_STAGES) & 1u;
        if (!wait_bar(smem_u32(&L.sf_empty[sf]), ph ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t base = lanes + SF_BASE + sf * SF_COLS;
        tmem_st4(base, cur.a[0], cur.a[0], cur.a[1], cur.a[1]);
        uint32_t v0[8];
#pragma unroll
        for (int c = 0; c < 7; ++c) v0[c] = cur.t0[c];
        v0[7] = 0x7F7F7F7Fu;
        tmem_st8(base + SFB0, v0);
        tmem_st4(base + SFB1, cur.t1[0], cur.t1[1], cur.t1[2], 0x7F7F7F7Fu);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(map_to_rank(smem_u32(&L.sf_full[sf]), 0));
        cur = nxt;
      }
    }
    // drain: the MMA commits that free this CTA's slots have all arrived
    for (uint32_t j = (it >= SF_STAGES ? it - SF_STAGES : 0); j < it && ok; ++j) {
      const uint32_t sf = j % SF_STAGES, ph = (j / SF_STAGES) & 1u;
      if (!wait_bar(smem_u32(&L.sf_empty[sf]), ph, abort_flag, p.status)) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lanes this warp may read: 32q .. 32q+31
    const int grp = (warp - 2) >> 2;   // two warps per lane quarter take alternate chunks
    const int e = grp * 4 + q, e_peer = grp * 4 + (q ^ 2);
    float* xmine = xch + e * (XCH_BYTES / 4);
    float* xpeer = xch + e_peer * (XCH_BYTES / 4);
    const uint32_t bar_id = 1u + (uint32_t)(q & 1) + 2u * (uint32_t)grp;  // lanes q and q ^ 2
    uint32_t seq = 0;
    for (int u = cid; u < total; u += ncl, ++seq) {
      const SUnit un = decode_unit(L, p.nslots, u);
      const uint32_t hm = seq & 1u;  // the unit's half; its tail is in the other head
      bool ok = wait_bar(smem_u32(&L.tmem_full[hm]), (seq >> 1) & 1u, abort_flag, p.status);
      // the gate and up warps of a feature range leave together, or the one
      // still in the chunk loop would wait for its partner forever
      if (SWIGLU) ok = named_all(bar_id, 64, ok);
      if (!ok) break;
      fence_after();
      const uint32_t lanes = tmem_base + ((uint32_t)(q * 32) << 16);
      // chunk c = 32 accumulator columns: first the ntail chunks of the tail
      // (second MMA, head of the other half), then the main part's (first MMA,
      // this unit's half) from its first column
      const int ntail = (un.N1 + 31) >> 5;
      const int nmain = (un.N0 + 31) >> 5;
      const int nch = ntail + nmain;
      auto chunk_buf = [&](int c) { return c < ntail ? 1 : 0; };  // which MMA (col_token)
      auto chunk_col = [&](int c) { return 32 * (c < ntail ? c : c - ntail); };
      auto chunk_addr = [&](int c) {
        return lanes + (c < ntail ? hm ^ 1u : hm) * HALF_COLS + (uint32_t)chunk_col(c);
      };
      // regions of this unit in chunk order: tail (other head), head, rest of
      // this half; each goes back to the MMA issuer once this warp has loaded
      // its last chunk of it (the regions the MMA issuer waited on)
      const int head_end = ntail + (nmain < HEAD_COLS / 32 ? nmain : HEAD_COLS / 32);
      auto r_end = [&](int i) { return i == 0 ? ntail : (i == 1 ? head_end : nch); };
      auto r_id = [&](int i) { return i == 0 ? 2 * (hm ^ 1u) : 2 * hm + (uint32_t)(i - 1); };
      int freed = un.N1 ? 0 : 1;  // regions 0 .. freed-1 handed back (no tail: none to hand)
      auto release = [&](int next_chunk) {
        const int from = freed;
        while (freed < 3 && next_chunk >= r_end(freed)) ++freed;
        if (freed == from) return;
        fence_before();
        __syncwarp();
        if (lane == 0)
          for (int i = from; i < freed; ++i)
            mbar_arrive_cluster(map_to_rank(smem_u32(&L.tmem_empty[r_id(i)]), 0));
      };
      // 32 columns x 32 features of this warp -> token rows of `out`, 16-byte
      // stores through a staging tile (`wstg`, a hand-over buffer no longer read)
      auto store_block = [&](const float (&v)[32], int c, int feat, __nv_bfloat16* wstg) {
#pragma unroll
        for (int j = 0; j < 32; ++j) wstg[j * 32 + lane] = __float2bfloat16_rn(v[j]);
        __syncwarp();
        const int buf = chunk_buf(c), col = chunk_col(c);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int vi = lane + 32 * i, j = vi >> 2, part = vi & 3;
          const int t = col_token(un, buf, col + j);
          const int64_t row = (int64_t)un.tok0 + t;
          if (t >= 0 && t < un.ntok && row >= 0 && row < p.cap)
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + row * p.out_ld +
                                      feat + part * 8) =
                *reinterpret_cast<const uint4*>(wstg + j * 32 + part * 8);
        }
        __syncwarp();
      };
      // the same in fp32 (MM1's h): 128 bytes per token row, 8 stores of 16
      auto store_block_f32 = [&](const float (&v)[32], int c, int feat, float* wstg) {
#pragma unroll
        for (int j = 0; j < 32; ++j) wstg[j * 32 + lane] = v[j];
        __syncwarp();
        const int buf = chunk_buf(c), col = chunk_col(c);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int vi = lane + 32 * i, j = vi >> 3, part = vi & 7;
          const int t = col_token(un, buf, col + j);
          const int64_t row = (int64_t)un.tok0 + t;
          if (t >= 0 && t < un.ntok && row >= 0 && row < p.cap)
            *reinterpret_cast<uint4*>(static_cast<float*>(p.out) + row * p.out_ld + feat +
                                      part * 4) =
                *reinterpret_cast<const uint4*>(wstg + j * 32 + part * 4);
        }
        __syncwarp();
      };
      if (SWIGLU) {
        const bool is_gate = q < 2;
        const int feat = un.tile * 128 + (int)crank * 64 + (q & 1) * 32;
#pragma unroll 1
        for (int c = 2 * grp; c < nch; c += 4) {
          const bool has2 = c + 1 < nch;
          uint32_t v0[32], v1[32];
          tmem_ld32(chunk_addr(c), v0);
          if (has2) tmem_ld32(chunk_addr(c + 1), v1);
          tmem_wait_ld();
          release(c + 4);
          // the gate warp computes chunk c, the up warp chunk c + 1; each hands
          // the other the values it lacks
          if (is_gate) {
            if (has2) {
#pragma unroll
              for (int j = 0; j < 32; ++j) xmine[j * 32 + lane] = __uint_as_float(v1[j]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) xmine[j * 32 + lane] = __uint_as_float(v0[j]);
          }
          named_sync(bar_id, 64);
          const int cc = is_gate ? c : c + 1;
          if (cc < nch) {
            float hv[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float g = is_gate ? __uint_as_float(v0[j]) : xpeer[j * 32 + lane];
              const float up = is_gate ? xpeer[j * 32 + lane] : __uint_as_float(v1[j]);
              hv[j] = __fdividef(g, 1.0f + __expf(-g)) * up;
            }
            // the partner's hand-over is in registers now: stage there
            store_block_f32(hv, cc, feat, xpeer);
          }
          named_sync(bar_id, 64);  // the partner has read this warp's hand-over
        }
      } else {
        const int feat = un.tile * 256 + (int)crank * 128 + q * 32;
#pragma unroll 1
        for (int c = grp; c < nch; c += 2) {
          uint32_t v[32];
          tmem_ld32(chunk_addr(c), v);
          tmem_wait_ld();
          release(c + 2);
          float y[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(v[j]);
          store_block(y, c, feat, reinterpret_cast<__nv_bfloat16*>(xmine));
        }
      }
      release(nch);  // whatever this warp had no chunk of
    }
  }

  fence_before();
  // No CTA may leave while its peer can still signal its barriers or read its
  // shared memory through the pair MMA.
  cluster_sync();
  fence_after();
  if (warp == 1) tmem_dealloc<2>(tmem_base);
}

// ------------------------------------------------------------- host side
cudaLaunchConfig_t launch_cfg(int clusters, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem_bytes();
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}
cudaLaunchConfig_t launch_cfg_pdl(int clusters, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = launch_cfg(clusters, s, attr);
  set_pdl_attr(attr[1]);
  cfg.numAttrs = 2;
  return cfg;
}

// Per device: raise the dynamic shared-memory limit and find how many pairs
// fit at once (the persistent grid must be fully resident).
bool device_setup(int* max_clusters) {
  static std::mutex mu;
  static int clusters[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (clusters[dev] == 0) {
    const int bytes = (int)smem_bytes();
    if (cudaFuncSetAttribute(ffn_f8swap_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess ||
        cudaFuncSetAttribute(ffn_f8swap_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
      return false;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = launch_cfg(num_sms() / 2, nullptr, attr);
    int c1 = 0, c2 = 0;
    if (cudaOccupancyMaxActiveClusters(&c1, ffn_f8swap_kernel<true>, &cfg) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&c2, ffn_f8swap_kernel<false>, &cfg) != cudaSuccess)
      return false;
    const int n = c1 < c2 ? c1 : c2;
    if (n < 1) return false;
    clusters[dev] = n;
  }
  *max_clusters = clusters[dev];
  return true;
}

moe_status run_f8swap(const F8SwapArgs& a, const Maps& m, bool gemm1, cudaStream_t s) {
  int max_clusters = 0;
  if (!device_setup(&max_clusters)) return MOE_ERR_CUDA;
  SwapParams p;
  p.offsets = a.offsets;
  p.slot_lo = a.slot_lo;
  p.nslots = a.slot_hi - a.slot_lo;
  p.min_slot_rows = a.min_slot_rows;
  p.max_slot_rows = INT32_MAX;
  p.cap = a.cap;
  p.status = a.status;
  p.gemm1 = gemm1 ? 1 : 0;
  if (gemm1) {
    p.num_kb = a.H / BK;
    p.n_tiles = a.I / 128;
    p.a_rows_per_slot = 0;
    p.a_tile_step = 128;
    p.a_cta_step = 64;
    p.out_ld = a.I;
    p.out = a.h32;
    p.a_scale = a.wgus;
    p.a_blocks = 2 * a.I / 128;
    p.a_up_block = a.I / 128;
    p.b_scale = a.xs;
  } else {
    p.num_kb = a.I / BK;
    p.n_tiles = a.H / 256;
    p.a_rows_per_slot = a.H;
    p.a_tile_step = 256;
    p.a_cta_step = 128;
    p.out_ld = a.H;
    p.out = a.y;
    p.a_scale = a.wds;
    p.a_blocks = a.H / 128;
    p.a_up_block = 0;
    p.b_scale = a.hs;
  }
  p.k_groups = p.num_kb;
  // upper bound of units (device-side counts unknown here)
  const int64_t bound = (a.cap / NMAX + p.nslots) * (int64_t)p.n_tiles;
  const int clusters = (int)(bound < max_clusters ? bound : max_clusters);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_cfg_pdl(clusters, s, attr);
  const cudaError_t e = gemm1 ? cudaLaunchKernelEx(&cfg, ffn_f8swap_kernel<true>, m, p)
                              : cudaLaunchKernelEx(&cfg, ffn_f8swap_kernel<false>, m, p);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

bool ffn_fp8_uses_pair_kernel(int64_t cap, int P, int H, int I) {
  // many rows per slot, and the scale words of four k-blocks 4-byte aligned
  return P > 0 && cap / P >= kFp8PairRows && H % 512 == 0 && I % 512 == 0;
}
bool ffn_fp8_splits_slots(int64_t cap, int P, int H, int I) {
  return P > 0 && cap / P >= 32 && cap / P < kFp8PairRows && cap >= kFp8PairRows &&
         H % 512 == 0 && I % 512 == 0;
}

moe_status launch_ffn_fp8_swap(const F8SwapArgs& a, cudaStream_t s) {
  if (a.slot_hi <= a.slot_lo || a.cap <= 0) return MOE_OK;
  Maps m1, m2;
  bool ok = make_map_u8_gate_up(&m1.a, a.wguq, (uint64_t)a.H, (uint64_t)a.I, (uint64_t)a.P, 64) &&
            make_map_u8(&m2.a, a.wdq, (uint64_t)a.I, (uint64_t)a.P * a.H, 128);
  for (int i = 0; i < NUM_BOXES && ok; ++i)
    ok = make_map_u8(&m1.b[i], a.xq, (uint64_t)a.H, (uint64_t)a.cap, 8u * (i + 1)) &&
         make_map_u8(&m2.b[i], a.hq, (uint64_t)a.I, (uint64_t)a.cap, 8u * (i + 1));
  if (!ok) return MOE_ERR_CUDA;
  moe_status st = run_f8swap(a, m1, true, s);
  if (st != MOE_OK) return st;
  // h: per-token groups of 128 features, rounded from fp32
  st = moe_quantize_fp8_groups(a.h32, a.cap, a.I, MOE_F32, a.hq, a.hs, s);
  if (st != MOE_OK) return st;
  return run_f8swap(a, m2, false, s);
}

}  // namespace moe

// Grouped SwiGLU expert FFN with the expert weights as the MMA's M operand
// (sm_103a, two-SM tcgen05 pairs).
//
// SGLang chapter 17, opening sections: a DeepSeek-V3 expert has gate_proj and
// up_proj [2048, 7168] and down_proj [7168, 2048] (weights stored [out, in]);
// section "normal dispatch 的调用链": the experts run as a grouped GEMM over
// the per-expert contiguous rows.  vLLM chapter 27, figure "MoE 模块化内核的
// PrepareAndFinalize 块结构": MM1, activation, MM2.
//
// The products are computed transposed, D^T = W . X^T: the weight rows fill
// the MMA's M = 256 (128 per SM of the pair) and a slot's tokens are its N.
// One work unit is (slot, weight tile, token group) and covers up to 320 of
// the slot's tokens with one or two MMAs per K step (N <= 256: one; above, the
// last 64 tokens in a second MMA so that no MMA is narrower than 64 columns),
// so every weight tile crosses HBM once per slot however many tokens the slot
// has, and a ragged token count costs N rounded up to 16 columns rather than
// a second weight pass.  (With tokens as M, a slot of 256 + t rows needs a
// second 128- or 256-row tile that streams the whole weight tile again.)
// Each operand moves as ONE TMA box per stage and CTA (small extra boxes cost
// far more than their bytes): CTA c takes the contiguous token rows
// [c*N/2, (c+1)*N/2) of the group through a map whose box is exactly N/2
// rows high; the first MMA reads its first N0/2 rows, the second the rest, so
// accumulator column j of the first MMA is token j (j < N0/2) or N/2 + j - N0/2.
//
//   MM1 + SwiGLU: CTA c of the pair holds gate rows f+64c .. f+64c+63 and the
//                 up rows of the same features (A, 128 rows, one 3-D box over
//                 [slot, gate|up, row, k]); TMEM lanes 0-63 hold gate, 64-127
//                 up.  The epilogue warps of lanes q and q+2 trade one
//                 32-column chunk through shared memory and each computes
//                 h = silu(gate) * up for one of the two chunks.
//   MM2:          CTA c holds down-projection rows f+128c .. f+128c+127.
// The epilogue stages each 32-token x 32-feature block through shared memory
// (in a hand-over buffer already read) and writes token rows with 16-byte
// stores (h and ys stay [tokens, features]).
//
// TMEM (512 fp32 columns per SM) is two halves of 256 columns, each a "head"
// (its first 64 columns) and a "rest".  Units alternate halves: unit s puts
// its first N0 <= 256 tokens in half s % 2 and its tail (N1 = 64 tokens) in
// the head of the other half.  The epilogue reads the tail, then the main
// part from its first column, and hands each of the three regions back as
// soon as its warps have loaded their last chunk of it; the next unit needs
// only its own half (the rest was freed a unit ago, the head holds this
// unit's tail) and the head of this unit's half for its tail, so its MMAs
// start after the first few chunks of this epilogue instead of all of it.
// Token rows past the slot's end are computed from whatever follows and never
// stored; rows past the buffer read as zero.
//
// Roles (320 threads, one CTA per SM, clusters of two):
//   warp 0    TMA producer (both CTAs): one weight box (128 rows) and one
//             token box (N/2 rows) per stage, completion on the leader CTA's
//             "full" barrier; 5-stage ring
//   warp 1    TMEM allocation; in the leader CTA lane 0 issues the MMAs
//             (cta_group::2, bf16 -> fp32) and the commits, multicast to both
//   warps 2-9 epilogue (both CTAs): two warps per TMEM lane quarter take
//             alternate chunks (MM2) or chunk pairs (MM1)
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel sets
// MOE_DEV_TIMEOUT, the other roles stop at their next wait, TMEM is freed and
// the kernel returns.
#include "common.cuh"
#include "ffn_internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BK = 64;                          // 64 bf16 = one 128-byte swizzle row
constexpr int A_ROWS = 128;                     // weight rows per CTA
constexpr int A_BYTES = A_ROWS * BK * 2;        // 16 KB
constexpr int NMAX = 320;                       // tokens per unit
constexpr int N_INSTR = 256;                    // largest N of one MMA
constexpr int B_ROWS = NMAX / 2;                // token rows per CTA
constexpr int B_BYTES = B_ROWS * BK * 2;        // 20 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 36 KB
constexpr int STAGES = 5;
constexpr int THREADS = 320;
constexpr int HALF_COLS = 256;                  // one TMEM half: a unit's main accumulator
constexpr int HEAD_COLS = 64;                   // head of a half: the other half's unit's tail
constexpr int EPI_WARPS = 8;                    // two per TMEM lane quarter
constexpr int XCH_BYTES = 32 * 32 * 4;          // per epilogue warp: 32 lanes x 32 fp32
constexpr int NUM_BOXES = B_ROWS / 8;           // token boxes of 8, 16, ..., 160 rows

struct Maps {
  CUtensorMap a;              // weights: MM1 3-D box 64 x 64 x 2 (gate, up), MM2 box 64 x 128
  CUtensorMap b[NUM_BOXES];   // tokens, box 64 x 8(i+1)
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
  __nv_bfloat16* out;
  uint32_t* status;
};

struct SmemLayout {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
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
  int N0, N1;    // MMA widths: tokens rounded up to 16; above 256, N1 = 64
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
  // A tail MMA rereads all 128 weight rows from shared memory whatever its
  // width, so a 16-column tail costs nearly what a 64-column one does: give
  // the tail the whole head.
  r.N1 = N > N_INSTR ? HEAD_COLS : 0;
  r.N0 = N - r.N1;
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

template <bool SWIGLU>
__global__ void __launch_bounds__(THREADS, 1)
    ffn_swap_kernel(const __grid_constant__ Maps maps, const SwapParams p) {
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
      const uint32_t tx = 2u * (uint32_t)(A_BYTES + h * BK * 2);  // both CTAs
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
        const uint32_t id0 = idesc_bf16(256, un.N0);
        const uint32_t id1 = idesc_bf16(256, un.N1 ? un.N1 : 16);
        const uint32_t boff1 = (uint32_t)(un.N0 >> 1) * BK * 2;
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
            const uint64_t bdesc0 = sw128_desc(sa + A_BYTES);
            const uint64_t bdesc1 = sw128_desc(sa + A_BYTES + boff1);
            // +32 bytes per K=16 step in the swizzle row.  The tail test stays outside
            // the K steps: a branch between the MMA issues, even one never taken, cost
            // the tensor pipe ~45% of its rate.
            if (un.N1) {
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                mma<2>(d0, adesc + 2 * kk, bdesc0 + 2 * kk, id0, (kb | kk) != 0);
                mma<2>(d1, adesc + 2 * kk, bdesc1 + 2 * kk, id1, (kb | kk) != 0);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk)
                mma<2>(d0, adesc + 2 * kk, bdesc0 + 2 * kk, id0, (kb | kk) != 0);
            }
            commit<2>(smem_u32(&L.empty[st]));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) commit<2>(smem_u32(&L.tmem_full[hm]));
        __syncwarp();
      }
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
            *reinterpret_cast<uint4*>(p.out + row * p.out_ld + feat + part * 8) =
                *reinterpret_cast<const uint4*>(wstg + j * 32 + part * 8);
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
            store_block(hv, cc, feat, reinterpret_cast<__nv_bfloat16*>(xpeer));
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
    if (cudaFuncSetAttribute(ffn_swap_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess ||
        cudaFuncSetAttribute(ffn_swap_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes) != cudaSuccess)
      return false;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = launch_cfg(num_sms() / 2, nullptr, attr);
    int c1 = 0, c2 = 0;
    if (cudaOccupancyMaxActiveClusters(&c1, ffn_swap_kernel<true>, &cfg) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&c2, ffn_swap_kernel<false>, &cfg) != cudaSuccess)
      return false;
    const int n = c1 < c2 ? c1 : c2;
    if (n < 1) return false;
    clusters[dev] = n;
  }
  *max_clusters = clusters[dev];
  return true;
}

moe_status run_swap(const FfnArgs& a, const Maps& m, bool gemm1, cudaStream_t s) {
  int max_clusters = 0;
  if (!device_setup(&max_clusters)) return MOE_ERR_CUDA;
  if (a.sm_budget > 0 && a.sm_budget / 2 < max_clusters) max_clusters = a.sm_budget / 2;
  if (max_clusters < 1) return MOE_ERR_INVALID_ARG;
  SwapParams p;
  p.offsets = a.offsets;
  p.slot_lo = a.slot_lo;
  p.nslots = a.slot_hi - a.slot_lo;
  p.min_slot_rows = a.min_slot_rows;
  p.max_slot_rows = a.max_slot_rows;
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
    p.out = static_cast<__nv_bfloat16*>(a.h);
  } else {
    p.num_kb = a.I / BK;
    p.n_tiles = a.H / 256;
    p.a_rows_per_slot = a.H;
    p.a_tile_step = 256;
    p.a_cta_step = 128;
    p.out_ld = a.H;
    p.out = static_cast<__nv_bfloat16*>(a.ys);
  }
  // upper bound of units (device-side counts unknown here)
  const int64_t bound = (a.cap / NMAX + p.nslots) * (int64_t)p.n_tiles;
  const int clusters = (int)(bound < max_clusters ? bound : max_clusters);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_cfg_pdl(clusters, s, attr);
  const cudaError_t e = gemm1 ? cudaLaunchKernelEx(&cfg, ffn_swap_kernel<true>, m, p)
                              : cudaLaunchKernelEx(&cfg, ffn_swap_kernel<false>, m, p);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

moe_status launch_ffn_tc_swap(const FfnArgs& a, cudaStream_t s) {
  if (a.slot_hi <= a.slot_lo || a.cap <= 0) return MOE_OK;
  Maps m1, m2;
  bool ok = make_map_gate_up(&m1.a, a.wgu, (uint64_t)a.H, (uint64_t)a.I, (uint64_t)a.P, 64) &&
            make_map(&m2.a, a.wd, (uint64_t)a.I, (uint64_t)a.P * a.H, 128);
  for (int i = 0; i < NUM_BOXES && ok; ++i)
    ok = make_map(&m1.b[i], a.xs, (uint64_t)a.H, (uint64_t)a.cap, 8u * (i + 1)) &&
         make_map(&m2.b[i], a.h, (uint64_t)a.I, (uint64_t)a.cap, 8u * (i + 1));
  if (!ok) return MOE_ERR_CUDA;
  moe_status st = run_swap(a, m1, true, s);
  if (st != MOE_OK) return st;
  return run_swap(a, m2, false, s);
}

}  // namespace moe

// Combine + DP scatter fused into the down projection's epilogue (bf16).
//
// vLLM chapter 27, figure "MoE 模块化内核的 PrepareAndFinalize 块结构": after
// MM2 the rows are un-permuted and finalize applies the top-k weights; SGLang
// chapter 17, section "scatter: 把 MoE 的输出还回本副本": each replica gets its
// rows of the combined buffer back.  Token row g receives
//   out[g] = sum_{j<k} w[g, j] * y[inv[g, j]]
// in float32, j ascending, rounded once -- exactly what combine_kernel computes.
//
// A token's k expert rows come from k different MM2 units, so the sum cannot
// happen in any one unit's registers.  Instead every unit still writes its rows
// of y and then counts itself in for each of its (token, feature block) cells
// on an integer counter, with one atomic that releases its stores and acquires
// the earlier arrivals' (atom.acq_rel.gpu).  The unit whose
// arrival completes the count (the token's number of routed slots) owns the
// cell: it reads the token's k rows of that block back (its own included) and
// writes the weighted sum in j order to the token's replica row.  Which unit
// wins changes nothing in the result, so the output is deterministic and equal
// bit for bit to the separate combine.  Nobody waits on a counter: the last
// arrival simply does the work, so the scheme cannot stall.
//
// Counters live in the caller's workspace, start at zero and are put back to
// zero by their owner; a counter found above its target (a workspace that was
// not cleared, e.g. after a call that timed out) sets MOE_DEV_BAD_WORKSPACE.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kFuseBlock = 256;  // features per counter cell: one MM2 n-tile

struct FuseArgs {
  const int32_t* perm;  // [cap] global row of each sorted row (-1: alignment pad)
  const int32_t* inv;   // [rows, kk] sorted row of each (row, j) (-1: none)
  const float* w;       // [rows, kk] top-k weights
  int32_t* cnt;         // [rows, nblk] arrival counters
  int64_t rows;         // global rows
  int kk;               // routed slots per row (k + shared experts)
  int nblk;             // counter cells per row = H / kFuseBlock
  int H;
  int R;
  const int32_t* counts;   // [R] replica counts (device)
  const int32_t* offsets;  // [R + 1] replica offsets (device)
  __nv_bfloat16* global_out;  // optional [rows, H]: the combined global buffer
  ReplicaPtrs dst;            // replica r's output [counts[r], H]
};

// Strong gpu-scope load of 16 bytes that bypasses L1: rows written by other
// SMs in this kernel are read from L2.
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Routed slots of global row g (entries of inv that point at a sorted row).
__device__ __forceinline__ int fuse_target(const FuseArgs& f, int64_t g) {
  int n = 0;
  const int32_t* iv = f.inv + g * f.kk;
  for (int j = 0; j < f.kk; ++j) n += iv[j] >= 0;
  return n;
}

// atomicAdd with release and acquire semantics at gpu scope: the calling
// thread's earlier stores are visible to whoever reads the counter after it,
// and what the earlier arrivals stored is visible to this thread after it.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

// Count one arrival on cell (g, blk) after this thread's stores of the cell;
// true if it completes the cell, which is then reset to zero for the next call.
__device__ __forceinline__ bool fuse_arrive(const FuseArgs& f, int64_t g, int blk,
                                            uint32_t* status) {
  const int n = fuse_target(f, g);
  int32_t* c = f.cnt + g * f.nblk + blk;
  const int old = atom_add_acq_rel_gpu(c, 1);
  if (old + 1 == n) {
    *c = 0;  // every arrival of this call has happened
    return true;
  }
  if (old >= n) flag(status, MOE_DEV_BAD_WORKSPACE);
  return false;
}

// One lane's 8 features [f0, f0 + 8) of token g: sum_j w[g, j] * y[inv[g, j]]
// in j order (eight source rows in flight at a time), rounded once, written to
// the replica row of g (and to the global buffer when kept).  r_off / r_cnt
// are the replica offsets and counts (a shared-memory copy).
__device__ __forceinline__ void fuse_combine_vec(const FuseArgs& f, const __nv_bfloat16* ys,
                                                 int64_t cap, int64_t g, int f0,
                                                 const int32_t* r_off, const int32_t* r_cnt,
                                                 uint32_t* status) {
  constexpr int B = 8;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  const int32_t* iv = f.inv + g * f.kk;
  const float* wv = f.w + g * f.kk;
  for (int j0 = 0; j0 < f.kk; j0 += B) {
    uint4 t[B];
    int32_t d[B];
    float wj[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int j = j0 + b;
      d[b] = j < f.kk ? iv[j] : -1;
      wj[b] = j < f.kk ? wv[j] : 0.f;
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (d[b] >= cap) {
        flag(status, MOE_DEV_BAD_COUNTS);
        d[b] = -1;
      }
      t[b] = make_uint4(0, 0, 0, 0);
      if (d[b] >= 0) t[b] = ld_cg_v4(ys + (int64_t)d[b] * f.H + f0);
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (d[b] < 0) continue;
      const uint32_t q[4] = {t[b].x, t[b].y, t[b].z, t[b].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[2 * e] = fmaf(wj[b], bf16lo(q[e]), acc[2 * e]);
        acc[2 * e + 1] = fmaf(wj[b], bf16hi(q[e]), acc[2 * e + 1]);
      }
    }
  }
  uint4 r;
  r.x = pack_bf16x2(acc[0], acc[1]);
  r.y = pack_bf16x2(acc[2], acc[3]);
  r.z = pack_bf16x2(acc[4], acc[5]);
  r.w = pack_bf16x2(acc[6], acc[7]);
  if (f.global_out != nullptr)
    *reinterpret_cast<uint4*>(f.global_out + g * f.H + f0) = r;
  const int rr = find_segment(r_off, f.R, g);
  const int64_t i = g - r_off[rr];
  const int64_t seg = (int64_t)r_off[rr + 1] - r_off[rr];
  const int64_t c = r_cnt[rr];
  if (c > seg || (c > 0 && f.dst.p[rr] == nullptr)) {
    flag(status, MOE_DEV_BAD_COUNTS);
    return;
  }
  if (i < c)
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(const_cast<void*>(f.dst.p[rr])) +
                              i * f.H + f0) = r;
}

// Zero the pad rows (rows of no replica's tokens) of the kept global buffer;
// `worker` of `nworkers` warps, each lane 16 bytes at a time.
__device__ __forceinline__ void fuse_zero_pad_rows(const FuseArgs& f, const int32_t* r_off,
                                                   const int32_t* r_cnt, int64_t worker,
                                                   int64_t nworkers, int lane) {
  if (f.global_out == nullptr) return;
  const int vpr = f.H / 8;
  for (int64_t g = worker; g < f.rows; g += nworkers) {
    const int rr = find_segment(r_off, f.R, g);
    int64_t c = r_cnt[rr];
    const int64_t seg = (int64_t)r_off[rr + 1] - r_off[rr];
    if (c > seg) c = seg;
    if (g - r_off[rr] < c) continue;
    uint4* row = reinterpret_cast<uint4*>(f.global_out + g * f.H);
    for (int v = lane; v < vpr; v += 32) row[v] = make_uint4(0, 0, 0, 0);
  }
}

}  // namespace moe

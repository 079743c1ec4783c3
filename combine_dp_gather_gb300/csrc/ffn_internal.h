// Internal launchers of the grouped SwiGLU expert FFN (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fuse_combine.cuh"
#include "moe_dp.h"

namespace moe {

struct FfnArgs {
  const void* xs;       // [cap, H] sorted rows
  const int32_t* offsets;  // [P + 1]
  int P, slot_lo, slot_hi;
  int64_t cap;
  const void* wgu;      // [P, 2I, H]
  const void* wd;       // [P, H, I]
  int H, I;
  void* ys;             // [cap, H]
  void* h;              // [cap, I] workspace
  uint32_t* status;
  // non-null: the down projection's epilogue also combines each token's rows and
  // scatters them to the replicas (tokens-as-M kernel only; the pair kernel
  // ignores it)
  const FuseArgs* fuse = nullptr;
  // slot filter by rows (device-side counts): the kernel serves only the slots
  // with min_slot_rows <= rows <= max_slot_rows
  int32_t min_slot_rows = 0;
  int32_t max_slot_rows = INT32_MAX;
  // SMs the persistent grid may use (0: every resident CTA)
  int sm_budget = 0;
};

// bf16 operands on the tcgen05 tensor cores (TMA-fed, TMEM accumulators).
moe_status launch_ffn_tc(const FfnArgs& a, cudaStream_t s);
// True if launch_ffn_tc hands this call to the pair kernel (many rows per slot).
bool ffn_uses_pair_kernel(const FfnArgs& a);
// The two kernels directly, whatever the rows per slot (slot filter and SM
// budget from the args): tokens as M on single SMs, weights as M on pairs.
moe_status launch_ffn_tc_single(const FfnArgs& a, cudaStream_t s);
// The same with the weights as the MMA's M operand and tokens as N, on pairs
// of SMs (many tokens per slot).
moe_status launch_ffn_tc_swap(const FfnArgs& a, cudaStream_t s);
// float32 on the CUDA cores.
moe_status launch_ffn_simt_f32(const FfnArgs& a, cudaStream_t s);

// FP8 operands on SM pairs with the weights as M and block-scaled MMAs (many
// rows per slot): MM1 + SwiGLU into float h32, its per-token-group
// quantisation into hq / hs, MM2 into bf16 y.
struct F8SwapArgs {
  const uint8_t* xq;     // [cap, H] e4m3 rows, sorted by slot
  const uint8_t* xs;     // [cap, H/128] their scale bytes
  const int32_t* offsets;  // [P + 1]
  int P, slot_lo, slot_hi;
  int64_t cap;
  const uint8_t* wguq;   // [P, 2I, H] e4m3
  const uint8_t* wgus;   // [P, 2I/128, H/128]
  const uint8_t* wdq;    // [P, H, I] e4m3
  const uint8_t* wds;    // [P, H/128, I/128]
  int H, I;
  float* h32;            // [cap, I] workspace
  uint8_t* hq;           // [cap, I] workspace
  uint8_t* hs;           // [cap, I/128] workspace
  __nv_bfloat16* y;      // [cap, H]
  uint32_t* status;
  int32_t min_slot_rows = 0;  // slots with fewer rows get no units
};
// Rows per slot from which a slot goes to the FP8 pair kernel.
constexpr int32_t kFp8PairRows = 192;
// True for many rows per slot (kFp8PairRows on average) with H and I multiples
// of 512 (the scale words of four k-blocks are then 4-byte aligned); the caller
// also checks that the scale arrays are.
bool ffn_fp8_uses_pair_kernel(int64_t cap, int P, int H, int I);
// True for a layer with fewer rows per slot on average but enough (32) that
// some slots may hold kFp8PairRows or more: those run on the pair kernel, the
// rest on the single-SM FP8 kernel.
bool ffn_fp8_splits_slots(int64_t cap, int P, int H, int I);
moe_status launch_ffn_fp8_swap(const F8SwapArgs& a, cudaStream_t s);

}  // namespace moe

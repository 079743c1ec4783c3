// Router gate GEMM fused ahead of top-k selection (sm_103a, tcgen05).
//
// SGLang chapter 17, section "Two-batch Overlap": the MoE operations run
// op_gate and then op_select_experts: the gate projects each token's hidden
// state onto the experts (here logits[g, e] = sum_h x[g, h] * W_r[e, h] + b[e],
// a linear gate with an optional per-expert bias, bf16 operands, fp32
// accumulation; section "推理时怎么“选副本”": expert selection takes the router
// logits together with a per-expert correction bias) and the top-k
// selection follows (moe_route_topk's rule: k largest logits, equal logits
// lower id first, softmax weights over the k or over all experts).
//
// Fused path (many rows, k <= 8): one CTA per 128-row tile, M = 128 rows,
// N = E experts (a multiple of 32, <= 256), K = H; the accumulator is one token row per TMEM
// lane, so each epilogue thread streams its row's E logits out of tensor
// memory 32 at a time into a register top-k list and never writes the logits
// (unless asked to).  Split path (few rows, or k > 8): CTAs also split K,
// write fp32 partial logits, a second kernel sums the partials in a fixed
// order (deterministic), and the top-k kernel of moe_route_topk selects.
//
// Roles (192 threads): warp 0 TMA producer (x box 64 x 128, W_r box 64 x E),
// warp 1 TMEM allocation + MMA issue (lane 0), warps 2-5 epilogue.  Every
// mbarrier wait is bounded (globaltimer); on expiry the kernel sets
// MOE_DEV_TIMEOUT and returns.
#include <float.h>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int THREADS = 192;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;     // 16 KB of token rows
constexpr int B_BYTES = 256 * BK * 2;    // up to 256 gate rows
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int KS_MAX = 16;               // K splits of the split path
constexpr int KMAX_FUSED = 8;            // k of the fused top-k

struct RSmem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t off[MOE_MAX_REPLICAS + 1];
  int32_t cnt[MOE_MAX_REPLICAS];
  float bias[256];
};
constexpr size_t r_smem_bytes() { return 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(RSmem); }

struct RParams {
  int64_t rows;
  int H, E, k, renorm, n_shared;
  int num_kb, kb_per;
  const int32_t* counts;
  const int32_t* offsets;
  int R;
  int32_t* ids;
  float* w;
  float* logits;   // fused: optional [rows, E] copy of the logits
  float* partial;  // split: [ks][rows][E]
  const float* bias;  // [E] or null
  uint32_t* status;
};

// (v, e) into a descending top-K list; scanning e ascending keeps equal
// logits in id order (a tie never displaces an earlier entry).
template <int K>
__device__ __forceinline__ void topk_insert(float (&tv)[K], int (&ti)[K], float v, int e) {
  if (!(v > tv[K - 1])) return;
  float cv = v;
  int ce = e;
#pragma unroll
  for (int j = 0; j < K; ++j) {
    if (cv > tv[j]) {
      const float t = tv[j];
      const int u = ti[j];
      tv[j] = cv;
      ti[j] = ce;
      cv = t;
      ce = u;
    }
  }
}

// K > 0: fused top-K epilogue; K == 0: partial logits of K split blockIdx.y.
template <int K>
__global__ void __launch_bounds__(THREADS, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const RParams p) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  RSmem& L = *reinterpret_cast<RSmem*>(stage_base + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, ks = blockIdx.y;
  const int kb0 = ks * p.kb_per;
  const int kb1 = kb0 + p.kb_per < p.num_kb ? kb0 + p.kb_per : p.num_kb;
  if (K > 0) {
    for (int i = threadIdx.x; i <= p.R; i += THREADS) {
      L.off[i] = p.offsets[i];
      if (i < p.R) L.cnt[i] = p.counts[i];
    }
    for (int e = threadIdx.x; e < p.E; e += THREADS)
      L.bias[e] = p.bias != nullptr ? p.bias[e] : 0.0f;
  }
  if (threadIdx.x == 0) {
    L.abort_flag = 0;
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&L.full[i]), 1);
      mbar_init(smem_u32(&L.empty[i]), 1);
    }
    mbar_init(smem_u32(&L.acc_full), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc<1>(smem_u32(&L.tmem_base));
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem_base = L.tmem_base;
  volatile int32_t* abort_flag = &L.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_x = policy_evict_first();
    const uint64_t pol_w = policy_evict_last();
    const uint32_t tx = (uint32_t)(A_BYTES + p.E * BK * 2);
    uint32_t it = 0;
    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
      if (!wait_bar(smem_u32(&L.empty[st]), ph ^ 1u, abort_flag, p.status)) break;
      if (lane == 0) {
        const uint32_t full = smem_u32(&L.full[st]);
        const uint32_t sa = smem_u32(stage_base + (size_t)st * STAGE_BYTES);
        mbar_arrive_expect_tx(full, tx);
        tma_load_2d<1>(sa, &tmA, kb * BK, tile * BM, full, pol_x);
        tma_load_2d<1>(sa + A_BYTES, &tmB, kb * BK, 0, full, pol_w);
      }
      __syncwarp();
    }
    for (uint32_t j = (it >= STAGES ? it - STAGES : 0); j < it; ++j) {
      const uint32_t st = j % STAGES, ph = (j / STAGES) & 1u;
      if (!wait_bar(smem_u32(&L.empty[st]), ph, abort_flag, p.status)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16(BM, p.E);
    uint32_t it = 0;
    bool ok = true;
    for (int kb = kb0; kb < kb1; ++kb, ++it) {
      const uint32_t st = it % STAGES, ph = (it / STAGES) & 1u;
      if (!wait_bar(smem_u32(&L.full[st]), ph, abort_flag, p.status)) {
        ok = false;
        break;
      }
      fence_after();
      if (lane == 0) {
        const uint32_t sa = smem_u32(stage_base + (size_t)st * STAGE_BYTES);
        const uint64_t adesc = sw128_desc(sa), bdesc = sw128_desc(sa + A_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma<1>(tmem_base, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
        commit<1>(smem_u32(&L.empty[st]));
      }
      __syncwarp();
    }
    if (ok && lane == 0) commit<1>(smem_u32(&L.acc_full));
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int64_t g = (int64_t)tile * BM + q * 32 + lane;  // this thread's token row
    const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
    const bool ok = wait_bar(smem_u32(&L.acc_full), 0, abort_flag, p.status);
    if (ok) {
      fence_after();
      const int nch = p.E / 32;
      if (K == 0) {
        float* dst = p.partial + ((int64_t)ks * p.rows + g) * p.E;
        for (int c = 0; c < nch; ++c) {
          uint32_t r[32];
          tmem_ld32(taddr + 32 * c, r);
          tmem_wait_ld();
          if (g < p.rows) {
            float4* d4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              d4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                  __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
          }
        }
      } else {
        constexpr int KK = K > 0 ? K : 1;
        // real row?  (rows past counts[r] in replica r's segment are padding)
        bool real = false;
        if (g < p.rows) {
          const int r = find_segment(L.off, p.R, g);
          const int64_t i = g - L.off[r];
          int64_t c = L.cnt[r];
          const int64_t seg = (int64_t)L.off[r + 1] - L.off[r];
          if (c > seg) {
            if (i == 0) flag(p.status, MOE_DEV_BAD_COUNTS);
            c = seg;
          }
          real = i >= 0 && i < c;
        }
        float tv[KK];
        int ti[KK];
#pragma unroll
        for (int j = 0; j < KK; ++j) {
          tv[j] = -INFINITY;
          ti[j] = INT32_MAX;
        }
        float m = -INFINITY, ssum = 0.0f;  // running max and sum of exp (full softmax)
        for (int c = 0; c < nch; ++c) {
          uint32_t r[32];
          tmem_ld32(taddr + 32 * c, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float v = __uint_as_float(r[i]) + L.bias[32 * c + i];
            r[i] = __float_as_uint(v);
            topk_insert<KK>(tv, ti, v, 32 * c + i);
            if (!p.renorm) {
              if (v > m) {
                ssum = ssum * expf(m - v) + 1.0f;
                m = v;
              } else {
                ssum += expf(v - m);
              }
            }
          }
          if (p.logits != nullptr && g < p.rows) {
            float4* d4 = reinterpret_cast<float4*>(p.logits + g * p.E + 32 * c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              d4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                  __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
          }
        }
        if (g < p.rows) {
          const int kk = p.k + p.n_shared;
          int32_t* idr = p.ids + g * kk;
          float* wr = p.w + g * kk;
          if (!real) {
            for (int j = 0; j < kk; ++j) {
              idr[j] = -1;
              wr[j] = 0.0f;
            }
          } else {
            // moe_route_topk's arithmetic: exp relative to the best logit, the
            // k terms summed in pick order (renormalised) or every expert's
            float ex[KK], denom = 0.0f;
#pragma unroll
            for (int j = 0; j < KK; ++j) {
              ex[j] = expf(tv[j] - tv[0]);
              denom += ex[j];
            }
            if (!p.renorm) denom = ssum * expf(m - tv[0]);
#pragma unroll
            for (int j = 0; j < KK; ++j) {
              idr[j] = ti[j];
              wr[j] = ex[j] / denom;
            }
            for (int s2 = 0; s2 < p.n_shared; ++s2) {
              idr[KK + s2] = p.E + s2;
              wr[KK + s2] = 1.0f;
            }
          }
        }
      }
    }
  }

  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) tmem_dealloc<1>(tmem_base);
}

// logits[i] = sum over ks ascending of partial[ks][i], then + bias[e]
// (float4 per thread; E is a multiple of 4).
__global__ void __launch_bounds__(256)
    router_reduce_kernel(const float4* __restrict__ partial, int64_t n4, int ks, int E,
                         const float* __restrict__ bias, float4* __restrict__ logits) {
  grid_dep_wait();    // earlier kernels on the stream are complete
  grid_dep_launch();  // the next kernel may start its launch
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 a = partial[i];
    for (int s = 1; s < ks; ++s) {
      const float4 b = partial[(int64_t)s * n4 + i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    if (bias != nullptr) {
      const int e = (int)((i * 4) % E);
      a.x += bias[e];
      a.y += bias[e + 1];
      a.z += bias[e + 2];
      a.w += bias[e + 3];
    }
    logits[i] = a;
  }
}

struct Plan {
  bool fused;
  int ks, kb_per;
};
Plan make_plan(int64_t rows, int H, int k) {
  const int64_t tiles = (rows + BM - 1) / BM;
  const int num_kb = H / BK;
  const int sms = num_sms();
  if (k <= KMAX_FUSED && tiles * 4 >= sms) return {true, 1, num_kb};
  int64_t ks = sms / (tiles > 0 ? tiles : 1);
  if (ks < 1) ks = 1;
  if (ks > KS_MAX) ks = KS_MAX;
  if (ks > num_kb) ks = num_kb;
  const int kb_per = (int)((num_kb + ks - 1) / ks);
  return {false, (num_kb + kb_per - 1) / kb_per, kb_per};
}

bool r_setup() {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    const int bytes = (int)r_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(router_gemm_kernel<0>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
#define MOE_SET(K)                                                                              \
  if (e == cudaSuccess)                                                                         \
    e = cudaFuncSetAttribute(router_gemm_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             bytes);
    MOE_SET(1) MOE_SET(2) MOE_SET(3) MOE_SET(4) MOE_SET(5) MOE_SET(6) MOE_SET(7) MOE_SET(8)
#undef MOE_SET
    if (e != cudaSuccess) return false;
    done[dev] = true;
  }
  return true;
}

size_t split_ws(int64_t rows, int E, int ks) {
  return (((size_t)ks + 1) * (size_t)rows * E * sizeof(float) + 255) & ~(size_t)255;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_route_gemm_ws_bytes(int64_t rows, int H, int E, int k) {
  if (rows <= 0 || H < BK || H % BK != 0 || E < 32 || E > 256 || E % 32 != 0 || k < 1) return 0;
  const Plan pl = make_plan(rows, H, k);
  return pl.fused ? 0 : split_ws(rows, E, pl.ks);
}

extern "C" moe_status moe_route_gemm_topk(const void* d_x, const void* d_w_router,
                                          const float* d_bias, int64_t rows, int H, int E, int k,
                                          int renormalize, int n_shared,
                                          const int32_t* d_counts, const int32_t* d_offsets,
                                          int R, int32_t* d_ids, float* d_w, float* d_logits,
                                          void* d_ws, size_t ws_bytes, uint32_t* d_status,
                                          void* stream) {
  if (rows < 0 || rows > INT32_MAX || R < 1 || R > MOE_MAX_REPLICAS) return MOE_ERR_INVALID_ARG;
  if (H < BK || H % BK != 0 || E < 32 || E > 256 || E % 32 != 0 || k < 1 || k > E ||
      n_shared < 0 || k + n_shared > MOE_MAX_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (d_x == nullptr || d_w_router == nullptr || d_counts == nullptr || d_offsets == nullptr ||
      d_ids == nullptr || d_w == nullptr || !aligned16(d_x) || !aligned16(d_w_router) ||
      (d_logits != nullptr && !aligned16(d_logits)))
    return MOE_ERR_INVALID_ARG;
  const Plan pl = make_plan(rows, H, k);
  if (!pl.fused && (d_ws == nullptr || !aligned16(d_ws) || ws_bytes < split_ws(rows, E, pl.ks)))
    return d_ws == nullptr ? MOE_ERR_INVALID_ARG : MOE_ERR_CAPACITY;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
  if (!r_setup()) return MOE_ERR_CUDA;
  CUtensorMap mA, mB;
  if (!make_map(&mA, d_x, (uint64_t)H, (uint64_t)rows, 128) ||
      !make_map(&mB, d_w_router, (uint64_t)H, (uint64_t)E, (uint32_t)E))
    return MOE_ERR_CUDA;
  RParams p;
  p.rows = rows;
  p.H = H;
  p.E = E;
  p.k = k;
  p.renorm = renormalize;
  p.n_shared = n_shared;
  p.num_kb = H / BK;
  p.kb_per = pl.kb_per;
  p.counts = d_counts;
  p.offsets = d_offsets;
  p.R = R;
  p.ids = d_ids;
  p.w = d_w;
  p.logits = d_logits;
  p.partial = static_cast<float*>(d_ws);
  p.bias = d_bias;
  p.status = d_status;
  cudaStream_t s = as_stream(stream);
  const unsigned tiles = (unsigned)((rows + BM - 1) / BM);
  const size_t smem = r_smem_bytes();
  if (pl.fused) {
    switch (k) {
#define MOE_CASE(K)                                                                  \
  case K:                                                                            \
    launch(router_gemm_kernel<K>, dim3(tiles, 1), THREADS, smem, s, mA, mB, p); \
    break;
      MOE_CASE(1) MOE_CASE(2) MOE_CASE(3) MOE_CASE(4) MOE_CASE(5) MOE_CASE(6) MOE_CASE(7)
      MOE_CASE(8)
#undef MOE_CASE
      default:
        return MOE_ERR_INVALID_ARG;
    }
    return launch_status();
  }
  launch(router_gemm_kernel<0>, dim3(tiles, (unsigned)pl.ks), THREADS, smem, s, mA, mB, p);
  float* logits = d_logits != nullptr
                      ? d_logits
                      : static_cast<float*>(d_ws) + (size_t)pl.ks * (size_t)rows * E;
  const int64_t n4 = rows * (int64_t)E / 4;
  int64_t blocks = (n4 + 255) / 256;
  const int64_t lim = (int64_t)num_sms() * 8;
  launch(router_reduce_kernel, (unsigned)(blocks < lim ? blocks : lim), 256, 0, s,
         static_cast<const float4*>(d_ws), n4, pl.ks, E, d_bias, reinterpret_cast<float4*>(logits));
  if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
  return moe_route_topk_shared(logits, rows, E, k, renormalize, n_shared, d_counts, d_offsets, R,
                               d_ids, d_w, d_status, stream);
}

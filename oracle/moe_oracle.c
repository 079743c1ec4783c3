/*
 * moe_oracle.c -- plain, slow CPU oracle of the MoE layer between DP attention
 * and expert parallelism.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * bench use it.  It shares no code, header, table or helper with the CUDA
 * library; both sides only receive the same seeded inputs.
 *
 * Arithmetic is done in double precision.  Every loop runs in the order the
 * definition states (rows ascending, k-slots ascending, reduction index
 * ascending); nothing is blocked, fused or reordered.  OpenMP is used only to
 * split independent output rows between threads in the FFN, which changes no
 * result.
 *
 * Sources (pages of the web text this project follows):
 *   [P1] "SGLang 源码完全拆解(十七): DP Attention 与专家并行" (SGLang source
 *        walkthrough, chapter 17: DP attention and expert parallelism).
 *   [P2] "vLLM 源码完全拆解(二十七): Dual Batch Overlap".
 *   [P4] "DP" (zdszero, data_parallelism): DP vs TP, MLP sync, static bound.
 *
 * Parity status of each function is stated in its comment; the pins live in
 * tests/test_oracle_pins.py.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_CAPACITY 2
#define ORC_ERR_BOUND 3
#define ORC_ERR_INPUT 4

#define ORC_PAD_SUM 0
#define ORC_PAD_MAX 1
#define ORC_PAD_STATIC 2

/* ------------------------------------------------------------------------ */
/* Layout of the global buffer.                                              */
/*                                                                          */
/* [P1] section "本 rank 的切片位置怎么算" (where this rank's slice starts):   */
/*   replica r starts at the sum of the token counts of replicas 0..r-1     */
/*   (a cumulative sum, replica 0 at row 0).                                 */
/* [P1] section "DpPaddingMode: 补齐到最长还是补齐到总和":                    */
/*   MAX_LEN pads every replica to max(global_num_tokens) so that all        */
/*   segments have equal length (all_gather layout: replica r at r*max);     */
/*   SUM_LEN sizes the buffer as the sum of the counts, segments back to     */
/*   back at the cumulative-sum offsets.                                     */
/* [P4] section "跳过同步: 用约定代替通信" (static bound B): every rank        */
/*   assumes every rank holds B requests, offset = rank * B; a rank above B  */
/*   is an error.  [P4] section "整体流程" states that decode counts are     */
/*   request counts, multiplied by tokens per request (draft + 1) inside the */
/*   forward, so the token offset of replica r is r * B * tokens_per_req.    */
/* Parity: pinned (closed forms, concatenation, golden fixtures).            */
/* ------------------------------------------------------------------------ */
int orc_dp_layout(const int32_t *counts, int R, int mode, int static_bound,
                  int tokens_per_req, int32_t *offsets, int64_t *rows_out) {
  if (R < 1 || counts == NULL || offsets == NULL || rows_out == NULL) return ORC_ERR_ARG;
  for (int r = 0; r < R; ++r)
    if (counts[r] < 0) return ORC_ERR_ARG;
  int64_t start = 0;
  if (mode == ORC_PAD_SUM) {
    for (int r = 0; r < R; ++r) {
      offsets[r] = (int32_t)start;
      start += counts[r];
    }
  } else if (mode == ORC_PAD_MAX) {
    int32_t mx = 0;
    for (int r = 0; r < R; ++r)
      if (counts[r] > mx) mx = counts[r];
    for (int r = 0; r < R; ++r) {
      offsets[r] = (int32_t)start;
      start += mx;
    }
  } else if (mode == ORC_PAD_STATIC) {
    if (static_bound < 0 || tokens_per_req < 1) return ORC_ERR_ARG;
    int64_t seg = (int64_t)static_bound * tokens_per_req;
    for (int r = 0; r < R; ++r)
      if (counts[r] > seg) return ORC_ERR_BOUND;
    for (int r = 0; r < R; ++r) {
      offsets[r] = (int32_t)start;
      start += seg;
    }
  } else {
    return ORC_ERR_ARG;
  }
  if (start > INT32_MAX) return ORC_ERR_ARG;
  offsets[R] = (int32_t)start;
  *rows_out = start;
  return ORC_OK;
}

/* [P1] section "DpPaddingMode", the get_dp_padding_mode rule, with the two
 * backend-specific branches (pplx, DeepEP v2) left out because no a2a
 * backend exists here:
 *   prefill in the batch and gather width > 1:
 *       MAX if the idle-aware flag is set and some replica has 0 tokens,
 *       else SUM;
 *   otherwise MAX iff 2 * sum >= max * width (the cheaper communication).
 * Parity: pinned (hand-worked golden table). */
int orc_dp_padding_mode(const int32_t *counts, int R, int gather_width,
                        int is_extend_in_batch, int max_len_with_idle) {
  int64_t sum = 0;
  int32_t mx = 0, mn = INT32_MAX;
  for (int r = 0; r < R; ++r) {
    sum += counts[r];
    if (counts[r] > mx) mx = counts[r];
    if (counts[r] < mn) mn = counts[r];
  }
  if (is_extend_in_batch && gather_width > 1) {
    if (max_len_with_idle && R > 0 && mn == 0) return ORC_PAD_MAX;
    return ORC_PAD_SUM;
  }
  if (sum * 2 >= (int64_t)mx * gather_width) return ORC_PAD_MAX;
  return ORC_PAD_SUM;
}

/* Row g of the global buffer carries a real token iff it lies in the first
 * counts[r] rows of the segment that starts at offsets[r]; the remaining rows
 * of a MAX or static-bound segment are padding.  Pad rows are not routed. */
void orc_valid_rows(const int32_t *counts, const int32_t *offsets, int R, int64_t rows,
                    uint8_t *valid) {
  for (int64_t g = 0; g < rows; ++g) valid[g] = 0;
  for (int r = 0; r < R; ++r)
    for (int32_t i = 0; i < counts[r]; ++i) valid[(int64_t)offsets[r] + i] = 1;
}

/* [P1] section "两种 gather: all_reduce 与 all_gather", path one: the global
 * buffer is filled with zeros, then each replica's tokens are copied to rows
 * [start, start + count).  With one device the all-reduce that follows sums
 * one non-zero contribution per row, so the result is that copy.
 * Rows are opaque byte strings of row_bytes bytes.  Parity: pinned
 * (gather then scatter is the identity; SUM equals concatenation). */
void orc_dp_gather(const void *const *local, const int32_t *counts, const int32_t *offsets,
                   int R, int64_t rows, int64_t row_bytes, void *global) {
  memset(global, 0, (size_t)(rows * row_bytes));
  for (int r = 0; r < R; ++r)
    for (int32_t i = 0; i < counts[r]; ++i)
      memcpy((char *)global + ((int64_t)offsets[r] + i) * row_bytes,
             (const char *)local[r] + (int64_t)i * row_bytes, (size_t)row_bytes);
}

/* [P1] section "scatter: 把 MoE 的输出还回本副本": the global buffer is cut
 * back into per-replica pieces by the same global_num_tokens that placed
 * them.  Parity: pinned (identity with gather). */
void orc_dp_scatter(const void *global, const int32_t *counts, const int32_t *offsets, int R,
                    int64_t row_bytes, void *const *local) {
  for (int r = 0; r < R; ++r)
    for (int32_t i = 0; i < counts[r]; ++i)
      memcpy((char *)local[r] + (int64_t)i * row_bytes,
             (const char *)global + ((int64_t)offsets[r] + i) * row_bytes, (size_t)row_bytes);
}

/* ------------------------------------------------------------------------ */
/* Top-k routing.  [P1] (TopKOutput{topk_ids, topk_weights} produced by       */
/* select_experts, section "normal dispatch 的调用链" and the TBO operation  */
/* list) names the output but not the scoring.  Reading taken: softmax       */
/* routing.  The k experts with the largest logits are chosen (largest      */
/* probability, the same order); equal logits go to the lower expert id;     */
/* ids are listed best first.  With renormalize the weights are the softmax */
/* over the k chosen logits, else the full softmax probabilities of the      */
/* chosen experts.  Pad rows get id -1 and weight 0.                         */
/* Parity: pinned (brute force over all k-subsets, scipy softmax, k=1, k=E). */
/* ------------------------------------------------------------------------ */
/* Shared experts: [P2] section "共享专家: 在被让出的空档里干活" -- a shared
 * expert's input bypasses routing; every token goes through it and its output
 * is added to the routed mixture.  Reading taken: shared expert s is logical
 * expert E + s, listed after the k routed ids of every real row with weight 1,
 * so dispatch, the grouped FFN and combine treat it as one more slot.
 * ids / w are [rows, k + n_shared].  Parity: pinned (dense per-token sum). */
int orc_route_topk_shared(const float *logits, int64_t rows, int E, int k, int renormalize,
                          int n_shared, const uint8_t *valid, int32_t *ids, double *w);
int orc_route_topk_routed(const float *logits, int64_t rows, int E, int k, int renormalize,
                          const uint8_t *valid, int32_t *ids, double *w);

int orc_route_topk(const float *logits, int64_t rows, int E, int k, int renormalize,
                   const uint8_t *valid, int32_t *ids, double *w) {
  return orc_route_topk_shared(logits, rows, E, k, renormalize, 0, valid, ids, w);
}

int orc_route_topk_shared(const float *logits, int64_t rows, int E, int k, int renormalize,
                          int n_shared, const uint8_t *valid, int32_t *ids_out, double *w_out) {
  if (E < 1 || k < 1 || k > E || n_shared < 0) return ORC_ERR_ARG;
  const int kk = k + n_shared;
  int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)(rows > 0 ? rows * k : 1));
  double *w = (double *)malloc(sizeof(double) * (size_t)(rows > 0 ? rows * k : 1));
  if (ids == NULL || w == NULL) {
    free(ids);
    free(w);
    return ORC_ERR_ARG;
  }
  int st = orc_route_topk_routed(logits, rows, E, k, renormalize, valid, ids, w);
  for (int64_t g = 0; g < rows && st == ORC_OK; ++g) {
    for (int j = 0; j < k; ++j) {
      ids_out[g * kk + j] = ids[g * k + j];
      w_out[g * kk + j] = w[g * k + j];
    }
    for (int s = 0; s < n_shared; ++s) {
      ids_out[g * kk + k + s] = valid[g] ? E + s : -1;
      w_out[g * kk + k + s] = valid[g] ? 1.0 : 0.0;
    }
  }
  free(ids);
  free(w);
  return st;
}

int orc_route_topk_routed(const float *logits, int64_t rows, int E, int k, int renormalize,
                          const uint8_t *valid, int32_t *ids, double *w) {
  if (E < 1 || k < 1 || k > E) return ORC_ERR_ARG;
  uint8_t *taken = (uint8_t *)malloc((size_t)E);
  if (taken == NULL) return ORC_ERR_ARG;
  for (int64_t g = 0; g < rows; ++g) {
    const float *l = logits + g * E;
    if (!valid[g]) {
      for (int j = 0; j < k; ++j) {
        ids[g * k + j] = -1;
        w[g * k + j] = 0.0;
      }
      continue;
    }
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict: ties keep the lower id */
      }
      taken[best] = 1;
      ids[g * k + j] = best;
    }
    double lmax = (double)l[ids[g * k]];
    double denom = 0.0;
    if (renormalize) {
      for (int j = 0; j < k; ++j) denom += exp((double)l[ids[g * k + j]] - lmax);
    } else {
      for (int e = 0; e < E; ++e) denom += exp((double)l[e] - lmax);
    }
    for (int j = 0; j < k; ++j) w[g * k + j] = exp((double)l[ids[g * k + j]] - lmax) / denom;
  }
  free(taken);
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Dispatch: sort the routed (row, j) pairs by expert slot into contiguous    */
/* per-slot buffers.                                                         */
/* [P1] section "normal dispatch 的调用链": get_dispatch_layout computes the  */
/*   tokens per expert; expert_alignment=128 rounds each expert's token      */
/*   count up to a multiple of 128 for the grouped GEMM tiles.               */
/* [P1] section "逻辑与物理的两套映射": logical_to_all_physical_map[E, X]      */
/*   with num_valid[E] lists the physical slots that hold a logical expert.  */
/* [P1] section "推理时怎么选副本": every rank must pick the same physical     */
/*   replica for a token (rank_invariant) when no a2a backend exists.        */
/* Reading taken for the replica choice: the occurrences of a logical expert */
/* are counted in (row, j) order and occurrence p goes to replica            */
/* p mod num_valid (round robin, the same on every simulated rank).          */
/* The order inside a slot is by (row, j): a stable sort by (slot, row, j).   */
/* Align pad positions get perm = -1.                                        */
/* Parity: pinned (Python sort with a tuple key on tiny inputs, bijection,   */
/* per-expert conservation, alignment).                                      */
/* ------------------------------------------------------------------------ */
typedef struct {
  int32_t slot, row, j;
} orc_key;

static int orc_key_cmp(const void *a, const void *b) {
  const orc_key *x = (const orc_key *)a, *y = (const orc_key *)b;
  if (x->slot != y->slot) return x->slot < y->slot ? -1 : 1;
  if (x->row != y->row) return x->row < y->row ? -1 : 1;
  if (x->j != y->j) return x->j < y->j ? -1 : 1;
  return 0;
}

int orc_dispatch(const int32_t *ids, int64_t rows, int k, int E, int P, const int32_t *l2p,
                 const int32_t *nrep, int X, int align, int64_t cap, int32_t *counts,
                 int32_t *offsets, int32_t *perm, int32_t *inv) {
  if (k < 1 || E < 1 || P < 1 || align < 1) return ORC_ERR_ARG;
  if (l2p == NULL && P != E) return ORC_ERR_ARG;
  int64_t n = rows * k;
  orc_key *keys = (orc_key *)malloc(sizeof(orc_key) * (size_t)(n > 0 ? n : 1));
  int64_t *seen = (int64_t *)calloc((size_t)E, sizeof(int64_t));
  if (keys == NULL || seen == NULL) {
    free(keys);
    free(seen);
    return ORC_ERR_ARG;
  }
  int64_t m = 0;
  int status = ORC_OK;
  for (int s = 0; s < P; ++s) counts[s] = 0;
  for (int64_t g = 0; g < rows && status == ORC_OK; ++g) {
    for (int j = 0; j < k; ++j) {
      int32_t l = ids[g * k + j];
      inv[g * k + j] = -1;
      if (l < 0) continue; /* pad row: not routed */
      if (l >= E) {
        status = ORC_ERR_INPUT;
        break;
      }
      int32_t slot = l;
      if (l2p != NULL) {
        int32_t nv = nrep[l];
        if (nv < 1 || nv > X) {
          status = ORC_ERR_INPUT;
          break;
        }
        int64_t p = seen[l]++;
        slot = l2p[(int64_t)l * X + (int32_t)(p % nv)];
        if (slot < 0 || slot >= P) {
          status = ORC_ERR_INPUT;
          break;
        }
      }
      counts[slot] += 1;
      keys[m].slot = slot;
      keys[m].row = (int32_t)g;
      keys[m].j = j;
      ++m;
    }
  }
  if (status == ORC_OK) {
    int64_t acc = 0;
    for (int s = 0; s < P; ++s) {
      offsets[s] = (int32_t)acc;
      acc += ((int64_t)counts[s] + align - 1) / align * align;
    }
    offsets[P] = (int32_t)acc;
    if (acc > cap) status = ORC_ERR_CAPACITY;
  }
  if (status == ORC_OK) {
    qsort(keys, (size_t)m, sizeof(orc_key), orc_key_cmp);
    for (int64_t d = 0; d < cap; ++d) perm[d] = -1;
    /* walk the sorted keys; within a slot they occupy consecutive positions
     * starting at the slot's offset */
    int64_t i = 0;
    for (int s = 0; s < P; ++s) {
      for (int32_t c = 0; c < counts[s]; ++c, ++i) {
        int64_t d = (int64_t)offsets[s] + c;
        perm[d] = keys[i].row;
        inv[(int64_t)keys[i].row * k + keys[i].j] = (int32_t)d;
      }
    }
  }
  free(keys);
  free(seen);
  return status;
}

/* xs[d] = xg[perm[d]], or a zero row where perm[d] = -1 (align padding).
 * Rows are opaque byte strings. */
void orc_permute_rows(const void *xg, const int32_t *perm, int64_t n, int64_t row_bytes,
                      void *xs) {
  for (int64_t d = 0; d < n; ++d) {
    if (perm[d] < 0)
      memset((char *)xs + d * row_bytes, 0, (size_t)row_bytes);
    else
      memcpy((char *)xs + d * row_bytes, (const char *)xg + (int64_t)perm[d] * row_bytes,
             (size_t)row_bytes);
  }
}

/* ------------------------------------------------------------------------ */
/* Expert FFN (SwiGLU) of one expert slot over n rows.                        */
/* [P1] opening sections: a DeepSeek-V3 expert has gate_proj [2048, 7168],   */
/*   up_proj of the same size and down_proj [7168, 2048], i.e. weights are   */
/*   stored [out, in].                                                        */
/* [P2] figure "MoE 模块化内核的 PrepareAndFinalize 块结构": permute, MM1,     */
/*   activation, MM2, unpermute.                                             */
/* SwiGLU: a = silu(x Wg^T) * (x Wu^T), y = a Wd^T, silu(g) = g / (1 + e^-g). */
/* wgu holds the gate rows 0..I-1 followed by the up rows I..2I-1.           */
/* Everything in double, sums in index order, no intermediate rounding.     */
/* Parity: pinned against numpy float64 matmul + scipy expit on small cases. */
/* ------------------------------------------------------------------------ */
void orc_expert_ffn(const float *x, int64_t n, int H, int I, const float *wgu, const float *wd,
                    double *y) {
#pragma omp parallel
  {
    double *a = (double *)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
      const float *xr = x + r * H;
      for (int i = 0; i < I; ++i) {
        const float *wg = wgu + (int64_t)i * H;
        const float *wu = wgu + (int64_t)(I + i) * H;
        double gsum = 0.0, usum = 0.0;
        for (int h = 0; h < H; ++h) {
          gsum += (double)xr[h] * (double)wg[h];
          usum += (double)xr[h] * (double)wu[h];
        }
        a[i] = gsum / (1.0 + exp(-gsum)) * usum;
      }
      for (int o = 0; o < H; ++o) {
        const float *wdo = wd + (int64_t)o * I;
        double ysum = 0.0;
        for (int i = 0; i < I; ++i) ysum += a[i] * (double)wdo[i];
        y[r * H + o] = ysum;
      }
    }
    free(a);
  }
}

/* ------------------------------------------------------------------------ */
/* Combine.  [P2] figure "MoE 模块化内核的 PrepareAndFinalize 块结构":        */
/* finalize applies the top-k weights while un-permuting: token row g        */
/* receives sum_j w[g, j] * ys[inv[g, j]], j ascending.  Pad rows (inv = -1  */
/* everywhere) are zero.  Parity: pinned (identity experts with weights      */
/* summing to 1 give the input back; numpy einsum on random inputs).         */
/* ------------------------------------------------------------------------ */
void orc_combine(const double *ys, const int32_t *inv, const double *w, int64_t rows, int k,
                 int H, double *out) {
  for (int64_t g = 0; g < rows; ++g) {
    double *o = out + g * H;
    for (int h = 0; h < H; ++h) o[h] = 0.0;
    for (int j = 0; j < k; ++j) {
      int32_t d = inv[g * k + j];
      if (d < 0) continue;
      const double *src = ys + (int64_t)d * H;
      double wj = w[g * k + j];
      for (int h = 0; h < H; ++h) o[h] += wj * src[h];
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Residual add + RMSNorm fused ahead of the DP gather.                      */
/* [P1] section "边界判定的融合" (_reduce_update_read_dp_gather): after the    */
/* attention-TP sum (nothing to sum on one device) the hidden states are     */
/* added into the residual ("update", written back in place), the FFN input  */
/* is read as RMSNorm of the updated residual ("read"), and that input is    */
/* DP-gathered.  Reading taken: the add is done in float32 and rounded once  */
/* to the layer's element type (this rounding decides stored bits, so it is  */
/* done in the same precision as the kernel: float32 add, then round to      */
/* nearest even); the norm reads the stored residual:                        */
/*   y = r / sqrt(mean(r^2) + eps) * gamma   (double here).                  */
/* Rows are float32 (bf16 layers arrive widened; round_bf16 = 1 asks for the */
/* bf16 rounding of the updated residual).                                   */
/* Parity: pinned (numpy restatement of RMSNorm, zero residual, gamma = 1).  */
/* ------------------------------------------------------------------------ */
static float orc_round_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return x; /* inf / nan unchanged */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  u &= 0xffff0000u;
  float y;
  memcpy(&y, &u, 4);
  return y;
}

void orc_add_rmsnorm(const float *hidden, float *residual, const float *gamma, int64_t n, int H,
                     double eps, int round_bf16, double *y) {
  for (int64_t r = 0; r < n; ++r) {
    const float *h = hidden + r * H;
    float *res = residual + r * H;
    double ss = 0.0;
    for (int c = 0; c < H; ++c) {
      float s = h[c] + res[c];
      if (round_bf16) s = orc_round_bf16(s);
      res[c] = s;
      ss += (double)s * (double)s;
    }
    double inv = 1.0 / sqrt(ss / H + eps);
    for (int c = 0; c < H; ++c) y[r * H + c] = (double)res[c] * inv * (double)gamma[c];
  }
}

/* ------------------------------------------------------------------------ */
/* FP8 path.                                                                */
/*                                                                          */
/* [P1] section "prefll 侧的一个必要步骤:per-token-group 量化": before        */
/*   dispatch the hidden states are quantised to FP8 in groups of 128       */
/*   consecutive features of one token (the group size is fixed at 128, the */
/*   same number as expert_alignment); with DeepGEMM the scale factors are  */
/*   UE8M0, i.e. powers of two, for its 1x128 fine-grained scaling.          */
/* Readings (the pages leave these open):                                    */
/*   * the FP8 format is e4m3 without infinities (max 448), round to        */
/*     nearest with ties to even, saturating at +-448;                      */
/*   * a group's scale is the smallest power of two 2^e with                 */
/*     amax <= 448 * 2^e (amax = largest magnitude in the group; e = 0 for  */
/*     an all-zero group), stored as the byte e + 127; codes are            */
/*     e4m3(x / 2^e);                                                       */
/*   * expert weights use the same rule on 128 x 128 blocks (output rows x  */
/*     input features), gate and up rows in separate blocks;               */
/*   * the SwiGLU activation h is quantised the same way (groups of 128     */
/*     intermediate features per token) before the down projection;        */
/*   * the GEMM sums dequantised products: for output (m, n),               */
/*     sum over k-blocks b of 2^(ea[m,b] + ew[n/128,b]) *                   */
/*     sum_{k in b} e4m3(qa[m,k]) * e4m3(qw[n,k]).                           */
/* Parity: pinned (e4m3 against torch's float8_e4m3fn conversion, the scale */
/* rule's closed form, the FFN against an independent numpy evaluation).   */
/* ------------------------------------------------------------------------ */
uint8_t orc_e4m3_encode(double x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  if (isnan(a)) return 0x7F;
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);       /* saturate */
  if (a < 0.015625) {                                  /* below 2^-6: steps of 2^-9 */
    double m = rint(a * 512.0);                        /* 0 .. 8; 8 is 2^-6 (code 0x08) */
    return (uint8_t)(sign | (uint8_t)m);
  }
  int E;
  double f = frexp(a, &E);                             /* a = f * 2^E, f in [0.5, 1) */
  int e = E - 1;                                       /* a = (2f) * 2^e, 2f in [1, 2) */
  double mant = rint((2.0 * f - 1.0) * 8.0);           /* 3 fraction bits, 0 .. 8 */
  if (mant == 8.0) {
    mant = 0.0;
    e += 1;
  }
  int field = e + 7;
  if (field > 15 || (field == 15 && mant == 7.0)) return (uint8_t)(sign | 0x7E);
  return (uint8_t)(sign | (uint8_t)(field << 3) | (uint8_t)mant);
}

double orc_e4m3_decode(uint8_t c) {
  int field = (c >> 3) & 15, mant = c & 7;
  double s = (c & 0x80) ? -1.0 : 1.0;
  if (field == 15 && mant == 7) return NAN;
  if (field == 0) return s * ldexp((double)mant, -9);
  return s * ldexp(1.0 + mant / 8.0, field - 7);
}

int orc_ue8m0_exp(double amax) {
  if (!(amax > 0.0)) return 0;
  int E;
  double f = frexp(amax, &E);          /* amax = f * 2^E; 448 = 0.875 * 2^9 */
  int e = E - 9 + (f > 0.875 ? 1 : 0);
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

void orc_e4m3_encode_array(const double *x, int64_t n, uint8_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(x[i]);
}
void orc_e4m3_decode_array(const uint8_t *c, int64_t n, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(c[i]);
}
void orc_ue8m0_exp_array(const double *amax, int64_t n, int32_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_ue8m0_exp(amax[i]);
}

/* Groups of 128 along each row of x [n, K] (K a multiple of 128):
 * q [n, K] codes, sexp [n, K / 128] scale bytes (e + 127). */
void orc_quant_groups(const double *x, int64_t n, int K, uint8_t *q, uint8_t *sexp) {
  const int G = K / 128;
  for (int64_t r = 0; r < n; ++r) {
    for (int g = 0; g < G; ++g) {
      const double *xs = x + r * K + (int64_t)g * 128;
      double amax = 0.0;
      for (int i = 0; i < 128; ++i)
        if (fabs(xs[i]) > amax) amax = fabs(xs[i]);
      int e = orc_ue8m0_exp(amax);
      sexp[r * G + g] = (uint8_t)(e + 127);
      for (int i = 0; i < 128; ++i) q[r * K + (int64_t)g * 128 + i] = orc_e4m3_encode(ldexp(xs[i], -e));
    }
  }
}

/* 128 x 128 blocks of w [R, K] (R and K multiples of 128):
 * q [R, K] codes, sexp [R / 128, K / 128] scale bytes. */
void orc_quant_blocks(const double *w, int64_t R, int K, uint8_t *q, uint8_t *sexp) {
  const int G = K / 128;
  for (int64_t br = 0; br < R / 128; ++br) {
    for (int g = 0; g < G; ++g) {
      double amax = 0.0;
      for (int64_t r = br * 128; r < br * 128 + 128; ++r)
        for (int i = 0; i < 128; ++i) {
          double v = fabs(w[r * K + (int64_t)g * 128 + i]);
          if (v > amax) amax = v;
        }
      int e = orc_ue8m0_exp(amax);
      sexp[br * G + g] = (uint8_t)(e + 127);
      for (int64_t r = br * 128; r < br * 128 + 128; ++r)
        for (int i = 0; i < 128; ++i)
          q[r * K + (int64_t)g * 128 + i] = orc_e4m3_encode(ldexp(w[r * K + (int64_t)g * 128 + i], -e));
    }
  }
}

/* orc_e4m3_decode of every code, so the dot products below look values up
 * instead of decoding each product's operands again. */
static double orc_e4m3_table[256];
static int orc_e4m3_table_ready = 0;
static void orc_e4m3_table_init(void) {
  if (orc_e4m3_table_ready) return;
  for (int c = 0; c < 256; ++c) orc_e4m3_table[c] = orc_e4m3_decode((uint8_t)c);
  orc_e4m3_table_ready = 1;
}

/* One dequantised dot product of FP8 rows a, w of length K: sum over
 * 128-blocks b of 2^(ea[b] + ew[b]) * sum_{k in b} e4m3(a_k) * e4m3(w_k). */
static double orc_fp8_dot(const uint8_t *a, const uint8_t *ea, const uint8_t *w,
                          const uint8_t *ew, int K) {
  double total = 0.0;
  for (int b = 0; b < K / 128; ++b) {
    double s = 0.0;
    for (int k = b * 128; k < b * 128 + 128; ++k) s += orc_e4m3_table[a[k]] * orc_e4m3_table[w[k]];
    total += ldexp(s, ((int)ea[b] - 127) + ((int)ew[b] - 127));
  }
  return total;
}

/* SwiGLU FFN of one expert on FP8 operands.
 *   xq [n, H] codes, xe [n, H/128] scale bytes (token groups)
 *   wguq [2I, H] codes, wgue [2I/128, H/128] (gate rows 0..I-1, up rows I..2I-1)
 *   wdq [H, I] codes, wde [H/128, I/128]
 *   y [n, H] double.  h is quantised per token in groups of 128 before MM2. */
void orc_expert_ffn_fp8(const uint8_t *xq, const uint8_t *xe, int64_t n, int H, int I,
                        const uint8_t *wguq, const uint8_t *wgue, const uint8_t *wdq,
                        const uint8_t *wde, double *y) {
  const int GH = H / 128, GI = I / 128;
  orc_e4m3_table_init();
#pragma omp parallel
  {
    double *a = (double *)malloc(sizeof(double) * (size_t)I);
    uint8_t *aq = (uint8_t *)malloc((size_t)I);
    uint8_t *ae = (uint8_t *)malloc((size_t)GI);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
      const uint8_t *xr = xq + r * H, *xer = xe + r * GH;
      for (int i = 0; i < I; ++i) {
        double g = orc_fp8_dot(xr, xer, wguq + (int64_t)i * H, wgue + (int64_t)(i / 128) * GH, H);
        double u = orc_fp8_dot(xr, xer, wguq + (int64_t)(I + i) * H,
                               wgue + (int64_t)((I + i) / 128) * GH, H);
        a[i] = g / (1.0 + exp(-g)) * u;
      }
      orc_quant_groups(a, 1, I, aq, ae);
      for (int o = 0; o < H; ++o)
        y[r * H + o] = orc_fp8_dot(aq, ae, wdq + (int64_t)o * I, wde + (int64_t)(o / 128) * GI, I);
    }
    free(a);
    free(aq);
    free(ae);
  }
}

/* ------------------------------------------------------------------------ */
/* Router GEMM.  [P1] section "Two-batch Overlap" lists the MoE operations   */
/* op_gate then op_select_experts: the gate projects each token's hidden     */
/* state onto the experts and top-k selection follows; section "推理时怎么    */
/* “选副本”" hands select_experts the router logits together with a          */
/* per-expert correction bias.  Reading: a linear gate with an optional      */
/* per-expert bias, logits[g, e] = sum_h x[g, h] * w[e, h] + b[e]            */
/* (w [E, H], h ascending, the bias added once after the sum; bias NULL is   */
/* the gate without bias); selection is orc_route_topk on these logits.     */
/* Parity: pinned (numpy matmul plus bias; a zero gate returns the bias;     */
/* a bias that reorders two experts moves the top-1).                        */
/* ------------------------------------------------------------------------ */
void orc_router_logits(const float *x, int64_t rows, int H, const float *w, int E,
                       const float *bias, double *logits) {
  for (int64_t g = 0; g < rows; ++g)
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int h = 0; h < H; ++h) s += (double)x[g * H + h] * (double)w[(int64_t)e * H + h];
      if (bias != NULL) s += (double)bias[e];
      logits[g * E + e] = s;
    }
}

/* Host threads the oracle's parallel loops use (the timed CPU baseline runs it
 * once on every core and once on one).  n < 1 leaves the default. */
void orc_set_threads(int n) {
  if (n >= 1) omp_set_num_threads(n);
}

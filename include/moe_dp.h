/*
 * moe_dp.h -- C ABI of libmoe_dp, the GB300 (sm_103a) MoE layer that sits
 * between data-parallel attention and expert parallelism, run on one GPU.
 *
 * One layer is six stream-ordered device calls:
 *
 *   moe_dp_gather    per-replica token segments  -> one global buffer
 *   moe_route_topk   router logits               -> top-k expert ids + weights
 *   moe_dispatch     ids (+ expert map)          -> per-slot counts/offsets,
 *                                                   permutation, sorted rows
 *   moe_grouped_ffn  sorted rows + expert weights -> SwiGLU expert outputs
 *   moe_combine      expert outputs + weights    -> token-order outputs
 *   moe_dp_scatter   global buffer               -> per-replica segments
 *
 * plus host helpers for the global-buffer layout (moe_dp_layout,
 * moe_dp_padding_mode) and workspace sizing.
 *
 * Sources of the operations (web pages this library follows):
 *   [P1] "SGLang 源码完全拆解(十七): DP Attention 与专家并行" -- SGLang source
 *        walkthrough, chapter 17: DP attention and expert parallelism.
 *   [P2] "vLLM 源码完全拆解(二十七): Dual Batch Overlap".
 *   [P4] "DP" (zdszero, data_parallelism): DP vs TP, MLP sync, static bound.
 *
 * Conventions (every entry point):
 *   - Ownership: the caller owns every buffer.  The library allocates no
 *     memory and keeps no state between calls, except a per-process cache of
 *     the driver's tensor-map encoder and of SM counts.
 *   - "d_" pointers are device pointers; "h_" or unprefixed array pointers
 *     are host pointers.  Shapes are row-major.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream) and never synchronise the
 *     host.
 *   - Host-checkable errors (null pointers, bad sizes, unsupported dtype or
 *     shape) return an error status before anything is launched.  A failed
 *     launch returns MOE_ERR_CUDA.
 *   - Data-dependent errors found on the device (an expert id outside
 *     [0, E), a bad map entry, capacity exceeded, a count larger than its
 *     segment, a bounded wait that gave up) are OR-ed into *d_status as
 *     MOE_DEV_* bits.  The caller zeroes *d_status before a layer and reads
 *     it after synchronising.  Kernels skip the offending accesses; they
 *     never trap.
 *   - Rows move as 16-byte vectors: the row width in bytes of every copied
 *     or combined tensor must be a multiple of 16 and every base pointer
 *     16-byte aligned.
 */
#ifndef MOE_DP_H
#define MOE_DP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,     /* null pointer, negative or inconsistent size */
  MOE_ERR_CAPACITY = 2,        /* a caller-provided buffer is too small */
  MOE_ERR_BOUND_EXCEEDED = 3,  /* a replica count exceeds the static bound */
  MOE_ERR_DEVICE_INPUT = 4,    /* reserved for callers mapping MOE_DEV_* bits */
  MOE_ERR_TIMEOUT = 5,         /* reserved for callers mapping MOE_DEV_TIMEOUT */
  MOE_ERR_CUDA = 6,            /* a CUDA runtime call or launch failed */
  MOE_ERR_UNSUPPORTED = 7      /* dtype / shape / device not supported */
} moe_status;

/* Global-buffer padding modes: [P1] section "DpPaddingMode" (MAX_LEN, SUM_LEN)
 * and [P4] section "跳过同步: 用约定代替通信" (static bound B). */
typedef enum { MOE_PAD_SUM = 0, MOE_PAD_MAX = 1, MOE_PAD_STATIC = 2 } moe_pad_mode;

/* Element types: MOE_F32 rows are float32; MOE_BF16 rows are bfloat16 with
 * float32 accumulation wherever the layer sums. */
typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Bits OR-ed into the device status word. */
#define MOE_DEV_BAD_EXPERT_ID 0x1u /* routed id outside [-1, E) */
#define MOE_DEV_BAD_MAP 0x2u       /* num_valid outside [1, X] or slot outside [0, P) */
#define MOE_DEV_CAPACITY 0x4u      /* padded slot total exceeds cap */
#define MOE_DEV_TIMEOUT 0x8u       /* a bounded device wait gave up */
#define MOE_DEV_BAD_COUNTS 0x10u   /* a replica count exceeds its segment, or an
                                      index points outside its buffer */
#define MOE_DEV_BAD_WORKSPACE 0x20u /* a grouped-FFN workspace's scheduler words were
                                        not zero at the call (they are cleared) */

#define MOE_MAX_REPLICAS 256 /* R limit (replica pointers travel as kernel arguments) */
#define MOE_MAX_SLOTS 1024   /* P limit of the grouped FFN's tile scheduler */
#define MOE_MAX_EXPERTS 1024 /* E limit of moe_route_topk */
#define MOE_MAX_TOPK 32      /* k limit */

/* ========================================================================
 * Host helpers (pure integer; no CUDA call, usable without a GPU)
 * ======================================================================== */

/* Offsets of the replicas' segments in the global buffer.
 * [P1] section "本 rank 的切片位置怎么算" (get_dp_local_info): replica r starts
 * at the exclusive prefix sum of the counts.  [P1] section "DpPaddingMode":
 * MAX pads each replica to the largest count (offset r * max), SUM packs them
 * back to back.  [P4] section "跳过同步": with a static bound B every replica
 * gets B requests of tokens_per_req tokens (offset r * B * tokens_per_req;
 * [P4] section "整体流程" for requests times draft + 1).
 *   counts          host int32[R], tokens per replica (>= 0; 0 = idle replica)
 *   R               1 .. MOE_MAX_REPLICAS
 *   mode            moe_pad_mode
 *   static_bound    B (requests per replica), used by MOE_PAD_STATIC only
 *   tokens_per_req  >= 1, used by MOE_PAD_STATIC only
 *   offsets         host int32[R + 1] out; offsets[R] = rows
 *   rows            host out, global buffer rows (real + padding)
 * Returns MOE_ERR_BOUND_EXCEEDED if a count exceeds B * tokens_per_req,
 * MOE_ERR_INVALID_ARG for negative counts or a total above INT32_MAX. */
moe_status moe_dp_layout(const int32_t* counts, int R, int mode, int static_bound,
                         int tokens_per_req, int32_t* offsets, int64_t* rows);

/* The padding-mode heuristic of [P1] section "DpPaddingMode"
 * (get_dp_padding_mode) without its a2a-backend branches: with prefill in the
 * batch and gather_width > 1 it returns SUM (MAX if max_len_with_idle and some
 * count is 0); otherwise MAX iff 2 * sum(counts) >= max(counts) * gather_width.
 * Returns a moe_pad_mode, or -1 on invalid arguments. */
int moe_dp_padding_mode(const int32_t* counts, int R, int gather_width, int is_extend_in_batch,
                        int max_len_with_idle);

/* Human-readable name of a moe_status value (static storage). */
const char* moe_status_string(int status);

/* Upper bound of the dispatch capacity: every routed (row, j) pair plus
 * alignment padding, rows * k + P * (align - 1). */
int64_t moe_dispatch_cap_bound(int64_t rows, int k, int P, int align);

/* Bytes of device workspace moe_dispatch needs for rows x k routed pairs over
 * E logical experts (per-chunk histograms). */
size_t moe_dispatch_ws_bytes(int64_t rows, int k, int E);

/* Bytes of device workspace moe_grouped_ffn needs: the SwiGLU activations
 * h[cap, I] in the layer dtype. */
size_t moe_grouped_ffn_ws_bytes(int64_t cap, int I, int dtype);

/* EPLB load report, [P1] section "不均衡的代价与冗余专家的思路"
 * (compute_utilization_rate): balancedness of per-rank token loads,
 * (mean + 1e-5) / (max + 1e-5); 1 is perfect balance, the 1e-5 keeps an
 * all-idle layer at 1.
 *   loads  host int64[n], tokens per simulated EP rank (>= 0)
 * Returns the balancedness in (0, 1], or -1.0 for a null array, n < 1 or a
 * negative load. */
double moe_balancedness(const int64_t* loads, int n);

/* Token loads of n_ranges contiguous, equal ranges of n slots (the simulated
 * EP ranks of [P1] section "逻辑与物理的两套映射": rank r holds slots
 * [r * n / n_ranges, (r + 1) * n / n_ranges)).
 *   counts  host int32[n], tokens per slot (>= 0)
 *   loads   host int64[n_ranges] out
 * Returns MOE_ERR_INVALID_ARG for null arrays, n_ranges < 1, n not a multiple
 * of n_ranges or a negative count. */
moe_status moe_range_loads(const int32_t* counts, int n, int n_ranges, int64_t* loads);

/* Tokens per logical expert from tokens per physical slot: the sum over each
 * logical expert's replicas ([P1] section "逻辑与物理的两套映射",
 * physical_to_logical_map; the scatter_add of per-slot counts into logical
 * counts in section "推理时怎么选副本").
 *   counts_P  host int32[P], tokens per slot (>= 0)
 *   p2l       host int32[P], logical expert of each slot, in [0, E)
 *   counts_E  host int64[E] out
 * Returns MOE_ERR_INVALID_ARG for null arrays, P < 1, E < 1, a negative count
 * or a map entry outside [0, E). */
moe_status moe_logical_counts(const int32_t* counts_P, const int32_t* p2l, int P, int E,
                              int64_t* counts_E);

/* ========================================================================
 * Device calls
 * ======================================================================== */

/* DP gather: copy replica r's counts[r] rows to global rows
 * [offsets[r], offsets[r] + counts[r]) and zero every other row.
 * [P1] section "两种 gather: all_reduce 与 all_gather" (path one: fill the
 * global buffer with zeros, copy the local segment at its start row; on one
 * device the all-reduce adds nothing else).
 *   local      HOST array of R device pointers; local[r] is [counts[r], H]
 *   d_counts   device int32[R]; d_offsets device int32[R + 1] (moe_dp_layout)
 *   rows       global rows (= offsets[R]); H row width in elements
 *   d_global   device [rows, H] out
 * A count larger than its segment sets MOE_DEV_BAD_COUNTS and copies only the
 * rows that fit. */
moe_status moe_dp_gather(const void* const* local, const int32_t* d_counts,
                         const int32_t* d_offsets, int R, int64_t rows, int H, int dtype,
                         void* d_global, uint32_t* d_status, void* stream);

/* moe_dp_gather of two row tensors of the same replicas in one launch (e.g.
 * the hidden states and the router logits of each token): tensor a is
 * [counts[r], H_a] of dtype_a per replica into d_global_a [rows, H_a], tensor b
 * likewise; counts, offsets, zero pad rows and error behaviour as
 * moe_dp_gather, whose result each output equals bit for bit. */
moe_status moe_dp_gather2(const void* const* local_a, int H_a, int dtype_a, void* d_global_a,
                          const void* const* local_b, int H_b, int dtype_b, void* d_global_b,
                          const int32_t* d_counts, const int32_t* d_offsets, int R, int64_t rows,
                          uint32_t* d_status, void* stream);

/* moe_dp_gather of the hidden states with the top-k routing of the gathered
 * rows in the same launch: for every global row the result of moe_dp_gather
 * (into d_global_x) and of moe_route_topk_shared on the row's router logits
 * (into d_ids / d_w), both bit for bit.  The routing reads each real row's
 * logits from its replica (local_logits[r] is float32 [counts[r], E]), so
 * they need not be gathered; with d_global_logits != NULL they are also
 * gathered there (float32 [rows, E], E a multiple of 4).
 *   local_x, H, dtype, d_global_x   as moe_dp_gather
 *   E, k, renormalize, n_shared     as moe_route_topk_shared
 *   d_ids int32 / d_w float32 [rows, k + n_shared] out
 * Argument checks and device errors are those of the two entry points. */
moe_status moe_dp_gather_route(const void* const* local_x, int H, int dtype, void* d_global_x,
                               const void* const* local_logits, int E, void* d_global_logits,
                               int k, int renormalize, int n_shared, const int32_t* d_counts,
                               const int32_t* d_offsets, int R, int64_t rows, int32_t* d_ids,
                               float* d_w, uint32_t* d_status, void* stream);

/* Residual add + RMSNorm fused ahead of the DP gather.  [P1] section
 * "边界判定的融合" (_reduce_update_read_dp_gather): the attention output is added
 * into the residual ("update", written back in place) and the FFN input is read
 * as RMSNorm of the updated residual ("read") before the DP gather; with one
 * device there is no attention-TP sum to complete.  For each real row i of
 * replica r:
 *   residual[r][i] = round(hidden[r][i] + residual[r][i])   (float32 add)
 *   global[offsets[r] + i] = round(res / sqrt(mean(res^2) + eps) * gamma)
 * where res is the stored (rounded) residual; pad rows of the global buffer
 * are zero.
 *   local_hidden    HOST array of R device pointers, [counts[r], H]
 *   local_residual  HOST array of R device pointers, [counts[r], H], updated
 *   d_gamma         device [H] norm weight, layer dtype
 *   eps             >= 0
 *   other arguments as moe_dp_gather; rows of at most 16 KB (H <= 8192 bf16,
 *   4096 fp32), else MOE_ERR_UNSUPPORTED. */
moe_status moe_dp_gather_add_rmsnorm(const void* const* local_hidden, void* const* local_residual,
                                     const void* d_gamma, float eps, const int32_t* d_counts,
                                     const int32_t* d_offsets, int R, int64_t rows, int H,
                                     int dtype, void* d_global, uint32_t* d_status, void* stream);

/* moe_dp_gather_add_rmsnorm plus the plain gather of a second row tensor of the
 * same replicas in the same launch (e.g. the router logits of each token):
 * local_b[r] is [counts[r], H_b] of dtype_b, gathered into d_global_b
 * [rows, H_b] bit for bit as moe_dp_gather would; the first tensor is added,
 * normed and gathered as moe_dp_gather_add_rmsnorm.  Argument checks and error
 * behaviour are those of the two entry points. */
moe_status moe_dp_gather_add_rmsnorm2(const void* const* local_hidden,
                                      void* const* local_residual, const void* d_gamma, float eps,
                                      const void* const* local_b, int H_b, int dtype_b,
                                      void* d_global_b, const int32_t* d_counts,
                                      const int32_t* d_offsets, int R, int64_t rows, int H,
                                      int dtype, void* d_global, uint32_t* d_status,
                                      void* stream);

/* moe_dp_gather_add_rmsnorm with the top-k routing of every global row in the
 * same launch: ids / w as moe_route_topk_shared computes them from each row's
 * router logits, read from the row's replica (local_logits[r] float32
 * [counts[r], E]); with d_global_logits != NULL the logits are also gathered
 * there (E a multiple of 4).  Checks and errors as the two entry points. */
moe_status moe_dp_gather_add_rmsnorm_route(const void* const* local_hidden,
                                           void* const* local_residual, const void* d_gamma,
                                           float eps, const void* const* local_logits, int E,
                                           void* d_global_logits, int k, int renormalize,
                                           int n_shared, int32_t* d_ids, float* d_w,
                                           const int32_t* d_counts, const int32_t* d_offsets,
                                           int R, int64_t rows, int H, int dtype, void* d_global,
                                           uint32_t* d_status, void* stream);

/* Top-k routing of every real row of the global buffer.  [P1] names the
 * result TopKOutput{topk_ids, topk_weights} (sections "normal dispatch 的调用链"
 * and "Two-batch Overlap"); the scoring is softmax routing: the k largest
 * logits win (equal logits: lower expert id first), listed best first; with
 * renormalize the weights are the softmax of the k chosen logits, else the
 * full softmax probabilities of the chosen experts.  Pad rows (not among the
 * first counts[r] rows of their segment) get id -1 and weight 0.
 *   d_logits  device float32[rows, E], finite values
 *   E         1 .. MOE_MAX_EXPERTS; k 1 .. min(E, MOE_MAX_TOPK)
 *   d_ids     device int32[rows, k] out; d_w device float32[rows, k] out */
moe_status moe_route_topk(const float* d_logits, int64_t rows, int E, int k, int renormalize,
                          const int32_t* d_counts, const int32_t* d_offsets, int R,
                          int32_t* d_ids, float* d_w, uint32_t* d_status, void* stream);

/* Router gate GEMM fused ahead of top-k.  [P1] section "Two-batch Overlap"
 * lists op_gate then op_select_experts: the gate projects each token onto the
 * experts and top-k selection follows; section "推理时怎么“选副本”": expert
 * selection takes the router logits together with a per-expert correction
 * bias.  Here:
 *   logits[g, e] = sum_h x[g, h] * W_r[e, h] + b[e]   (bf16 operands, fp32 sums)
 * and the selection, weights, pad rows and shared experts are exactly those
 * of moe_route_topk_shared on these logits.
 *   d_x         device bf16 [rows, H], the gathered rows (16-byte aligned)
 *   d_w_router  device bf16 [E, H]; E a multiple of 32 up to 256; H of 64
 *   d_bias      device float32 [E] per-expert bias, or NULL (none)
 *   d_logits    device float32 [rows, E] out, or NULL (not needed)
 *   d_ws        workspace of moe_route_gemm_ws_bytes(rows, H, E, k) bytes
 *               (0 when the fused path runs; may then be NULL)
 * Many rows and k <= 8: one kernel, the top-k taken from tensor memory.
 * Otherwise K is split over more CTAs and the partial logits are summed in
 * a fixed order before the top-k kernel (the result does not depend on
 * scheduling).  sm_103 only. */
size_t moe_route_gemm_ws_bytes(int64_t rows, int H, int E, int k);
moe_status moe_route_gemm_topk(const void* d_x, const void* d_w_router, const float* d_bias,
                               int64_t rows, int H, int E, int k, int renormalize, int n_shared,
                               const int32_t* d_counts, const int32_t* d_offsets, int R,
                               int32_t* d_ids, float* d_w, float* d_logits, void* d_ws,
                               size_t ws_bytes, uint32_t* d_status, void* stream);

/* moe_route_topk plus n_shared shared experts.  [P2] section "共享专家: 在被让出的
 * 空档里干活": a shared expert's input bypasses routing and its output is added
 * to the routed mixture.  Every real row lists its k routed ids followed by
 * the shared experts E .. E + n_shared - 1 with weight 1; pad rows get -1 / 0
 * in all k + n_shared columns.  d_ids and d_w are [rows, k + n_shared];
 * k + n_shared <= MOE_MAX_TOPK.  Dispatch then runs over E + n_shared logical
 * experts, the weights hold the shared experts as the last slots, and combine
 * adds them with weight 1. */
moe_status moe_route_topk_shared(const float* d_logits, int64_t rows, int E, int k,
                                 int renormalize, int n_shared, const int32_t* d_counts,
                                 const int32_t* d_offsets, int R, int32_t* d_ids, float* d_w,
                                 uint32_t* d_status, void* stream);

/* Dispatch: stable sort of the routed (row, j) pairs by physical expert slot.
 * [P1] section "normal dispatch 的调用链" (get_dispatch_layout: tokens per
 * expert; expert_alignment rounds each expert's count up to a multiple of
 * 128 for the grouped GEMM).  [P1] sections "逻辑与物理的两套映射" and
 * "推理时怎么选副本" (logical_to_all_physical_map[E, X] with num_valid[E];
 * one rank-invariant replica per token): occurrence p of logical expert l,
 * counted in (row, j) order, goes to replica p mod num_valid[l].
 *   d_global   device [rows, H] rows to permute (may be NULL: indices only)
 *   d_ids      device int32[rows, k]; -1 marks a pad row
 *   E, P       logical experts, physical slots (P == E when d_l2p is NULL)
 *   d_l2p      device int32[E, X] slot of each replica, or NULL
 *   d_nrep     device int32[E] replicas per logical expert, or NULL
 *   align      >= 1; each slot's count is rounded up to a multiple of align
 *   cap        rows of d_perm / d_sorted (moe_dispatch_cap_bound suffices)
 * Outputs (device): d_counts_P int32[P] tokens per slot; d_offsets_P
 * int32[P + 1] slot starts (exclusive scan of the rounded counts);
 * d_perm int32[cap] source row of each sorted position (-1 at alignment
 * padding; defined for positions < d_offsets_P[P]); d_inv int32[rows, k]
 * sorted position of each (row, j) (-1 for pad rows); d_sorted [cap, H]
 * permuted rows (alignment padding rows zeroed).
 *   d_ws, ws_bytes   workspace of at least moe_dispatch_ws_bytes(rows, k, E)
 * Device errors: MOE_DEV_BAD_EXPERT_ID, MOE_DEV_BAD_MAP, MOE_DEV_CAPACITY (no
 * write goes past cap). */
moe_status moe_dispatch(const void* d_global, const int32_t* d_ids, int64_t rows, int k, int H,
                        int dtype, int E, int P, const int32_t* d_l2p, const int32_t* d_nrep,
                        int X, int align, int64_t cap, int32_t* d_counts_P,
                        int32_t* d_offsets_P, int32_t* d_perm, int32_t* d_inv, void* d_sorted,
                        void* d_ws, size_t ws_bytes, uint32_t* d_status, void* stream);

/* Grouped SwiGLU expert FFN over the sorted rows of slots [slot_lo, slot_hi)
 * (one contiguous slot range stands for one EP rank).  For each slot s and
 * each row x in [offsets[s], offsets[s + 1]):
 *   h = silu(x Wg_s^T) * (x Wu_s^T),  y = h Wd_s^T
 * ([P1] opening sections: gate_proj and up_proj are [I, H], down_proj is
 * [H, I]; [P2] figure "MoE 模块化内核的 PrepareAndFinalize 块结构": MM1,
 * activation, MM2.)
 *   d_sorted     device [cap, H]
 *   d_offsets_P  device int32[P + 1] from moe_dispatch
 *   d_w_gate_up  device [P, 2I, H]: gate rows 0..I-1, up rows I..2I-1
 *   d_w_down     device [P, H, I]
 *   d_out_sorted device [cap, H] out; rows of other slots are not written
 *   d_ws         workspace >= moe_grouped_ffn_ws_bytes(cap, I, dtype)
 * MOE_BF16 runs on the tcgen05 tensor cores (fp32 accumulation in tensor
 * memory, h rounded to bf16) and needs H % 256 == 0, I % 128 == 0 and
 * P <= MOE_MAX_SLOTS; MOE_F32 runs a CUDA-core kernel (fp32 throughout). */
moe_status moe_grouped_ffn(const void* d_sorted, const int32_t* d_offsets_P, int P, int slot_lo,
                           int slot_hi, int64_t cap, const void* d_w_gate_up,
                           const void* d_w_down, int H, int I, int dtype, void* d_out_sorted,
                           void* d_ws, size_t ws_bytes, uint32_t* d_status, void* stream);

/* The grouped FFN of a skewed layer, split by slot over two streams with an SM
 * budget: slots with at least hot_rows rows run on the pair kernel (expert
 * weights as the MMA's M operand on two-SM pairs, each weight tile read once
 * per 320 tokens) on hot_sms SMs of stream_hot, all other slots on the
 * single-SM kernel (tokens as M) on the remaining SMs of `stream`, at the same
 * time; the result is what moe_grouped_ffn computes.  [P1] section "Two-batch
 * Overlap" and [P2] (Dual Batch Overlap, its SM control): two streams keep
 * different work in flight together -- here the hot slots' tensor-bound GEMMs
 * beside the cold slots' weight stream, with every weight tile still read once.
 * Arguments as moe_grouped_ffn (bf16 only), plus:
 *   hot_rows    >= 1: a slot with at least this many rows is hot
 *   hot_sms     SMs of the hot part: even, 2 .. (SM count - 2)
 *   stream_hot  second stream (void* cudaStream_t); it waits for the work queued
 *               on `stream` before the call, and `stream` waits for it after.
 *               NULL or equal to `stream`: the two parts run one after the other.
 * The fork and join use two events the library creates on the first call on a
 * device and keeps until exit (make that first call outside stream capture);
 * the call can then be captured into a CUDA graph, where the fork and join
 * become graph edges.
 * The rounding order of a slot's sums can differ between the two kernels, so
 * the output equals moe_grouped_ffn within the bf16 tolerance, not bit for bit. */
moe_status moe_grouped_ffn_split(const void* d_sorted, const int32_t* d_offsets_P, int P,
                                 int slot_lo, int slot_hi, int64_t cap, const void* d_w_gate_up,
                                 const void* d_w_down, int H, int I, int dtype,
                                 void* d_out_sorted, void* d_ws, size_t ws_bytes, int hot_rows,
                                 int hot_sms, uint32_t* d_status, void* stream, void* stream_hot);

/* Combine: un-permute and apply the top-k weights.
 * [P2] figure "MoE 模块化内核的 PrepareAndFinalize 块结构" (finalize applies
 * the top-k weights): out[row] = sum_{j<k} w[row, j] * y[inv[row, j]],
 * accumulated in float32 in j order and rounded once; rows whose inv entries
 * are all -1 (pad rows) are zero.
 *   d_out_sorted device [cap, H]; d_inv device int32[rows, k];
 *   d_w device float32[rows, k]; d_global_out device [rows, H] out.
 * An inv entry >= cap sets MOE_DEV_BAD_COUNTS and is skipped. */
moe_status moe_combine(const void* d_out_sorted, const int32_t* d_inv, const float* d_w,
                       int64_t rows, int k, int H, int dtype, int64_t cap, void* d_global_out,
                       uint32_t* d_status, void* stream);

/* DP scatter: copy global rows [offsets[r], offsets[r] + counts[r]) back to
 * replica r.  [P1] section "scatter: 把 MoE 的输出还回本副本" (reduce_scatterv
 * split by the same global_num_tokens that placed the rows).
 *   local  HOST array of R device pointers; local[r] is [counts[r], H] out */
moe_status moe_dp_scatter(const void* d_global, const int32_t* d_counts, const int32_t* d_offsets,
                          int R, int64_t rows, int H, int dtype, void* const* local,
                          uint32_t* d_status, void* stream);

/* moe_combine followed by moe_dp_scatter in one launch: each combined row of
 * replica r's segment (global row offsets[r] + i, i < counts[r]) is written
 * straight to local[r] row i, bit for bit what the two calls produce.  With
 * d_global_out non-NULL the combined global buffer [rows, H] (pad rows zero)
 * is written as well; with NULL it is not, and pad rows are skipped.
 *   arguments as moe_combine and moe_dp_scatter (local: HOST array of R device
 *   pointers, local[r] [counts[r], H] out). */
moe_status moe_combine_scatter(const void* d_out_sorted, const int32_t* d_inv, const float* d_w,
                               int64_t rows, int k, int H, int dtype, int64_t cap,
                               const int32_t* d_counts, const int32_t* d_offsets, int R,
                               void* const* local, void* d_global_out, uint32_t* d_status,
                               void* stream);

/* The grouped FFN with the combine and the DP scatter after it, as one call:
 * the result of moe_grouped_ffn followed by moe_combine_scatter.  [P2] figure
 * "MoE 模块化内核的 PrepareAndFinalize 块结构" (MM2, then finalize applies the
 * top-k weights to the un-permuted rows); [P1] section "scatter: 把 MoE 的输出
 * 还回本副本".  With few rows per slot (under 192 on average, the tokens-as-M
 * kernel: decode) the combine runs in the down projection's epilogue: each MM2
 * unit still writes its rows of d_out_sorted, then counts itself in on a
 * per-(token, 256-feature tile) integer counter in the workspace; the unit that
 * completes a token's count sums the token's rows of the tile in j order in
 * float32, rounds once and writes the replica row -- the same bits as
 * moe_combine_scatter, whichever unit wins, and one launch fewer.  With more
 * rows per slot (the pair kernel: prefill) the combine is its own launch after
 * the FFN, which measured faster there.
 * Arguments as moe_grouped_ffn, plus:
 *   d_perm      device int32[cap] from moe_dispatch (global row of each sorted row)
 *   d_inv, d_w  device [rows, k] from moe_dispatch / the routing (k = routed slots
 *               per row, shared experts included)
 *   d_counts, d_offsets, R, local, d_global_out   as moe_combine_scatter (pad rows
 *               of d_global_out are written zero)
 *   d_ws        workspace of moe_grouped_ffn_combine_ws_bytes(cap, rows, H, I, dtype)
 *               bytes: h [cap, I], then (bf16) rows x H/256 int32 counters.  The
 *               counters must be zero before the first call (e.g. a zero-filled
 *               workspace); every call that completes leaves them zero.  A call that
 *               set MOE_DEV_TIMEOUT may leave them non-zero: zero them again.  A
 *               counter found above its target sets MOE_DEV_BAD_WORKSPACE.
 * With slot ranges, a token's rows are combined by whichever call completes
 * them: the calls of one layer step must together cover every slot that holds
 * a routed row, and none may run concurrently with another on the same
 * workspace.  bf16 runs on the tensor-core kernels (H a multiple of 256);
 * float32 layers run the CUDA-core FFN and then moe_combine_scatter. */
size_t moe_grouped_ffn_combine_ws_bytes(int64_t cap, int64_t rows, int H, int I, int dtype);
/* 1 if moe_grouped_ffn_combine on a sorted buffer of cap rows over P slots runs
 * the combine inside the down projection's epilogue (one launch fewer), 0 if it
 * runs it as its own launch after the FFN.  Host only, no CUDA call. */
int moe_grouped_ffn_combine_in_epilogue(int64_t cap, int P, int dtype);
moe_status moe_grouped_ffn_combine(const void* d_sorted, const int32_t* d_offsets_P, int P,
                                   int slot_lo, int slot_hi, int64_t cap,
                                   const void* d_w_gate_up, const void* d_w_down, int H, int I,
                                   int dtype, void* d_out_sorted, const int32_t* d_perm,
                                   const int32_t* d_inv, const float* d_w, int64_t rows, int k,
                                   const int32_t* d_counts, const int32_t* d_offsets, int R,
                                   void* const* local, void* d_global_out, void* d_ws,
                                   size_t ws_bytes, uint32_t* d_status, void* stream);

/* Same as moe_dispatch, but allocates nothing and takes no workspace: the
 * per-chunk histograms live in a fixed device array inside the library.
 * The pages have no counterpart; this entry point exists for callers that
 * cannot allocate device memory where they dispatch (a plugin whose host
 * framework owns all device allocations, or a decode loop that must not call
 * cudaMalloc/cudaFree because they can synchronise the device).
 *   Arguments and outputs: as moe_dispatch, without d_ws / ws_bytes.
 *   Limit: moe_dispatch_ws_bytes(rows, k, E) <= MOE_NOALLOC_SCRATCH_BYTES
 *          (65536 chunk-histogram entries, e.g. 262144 routed pairs at E = 256);
 *          larger problems return MOE_ERR_CAPACITY before anything runs.
 *   Set-up: the first call on each device looks up the array's device address
 *          (cudaGetSymbolAddress) with that device current; make that first
 *          call before any stream capture.
 *   Sharing: every call on a device uses the same array, which keeps the last
 *          call's contents (each call overwrites what it reads, so nothing
 *          has to be cleared); calls that overlap on the GPU (different
 *          streams, or different host threads) race on it and must be
 *          serialised by the caller.
 *   The array occupies MOE_NOALLOC_SCRATCH_BYTES on every GPU that loads the
 *   library until the process exits. */
#define MOE_NOALLOC_SCRATCH_BYTES (256u * 1024u)
moe_status moe_dispatch_noalloc(const void* d_global, const int32_t* d_ids, int64_t rows, int k,
                                int H, int dtype, int E, int P, const int32_t* d_l2p,
                                const int32_t* d_nrep, int X, int align, int64_t cap,
                                int32_t* d_counts_P, int32_t* d_offsets_P, int32_t* d_perm,
                                int32_t* d_inv, void* d_sorted, uint32_t* d_status, void* stream);

/* ------------------------------------------------------------------ FP8 path
 * [P1] section "prefll 侧的一个必要步骤:per-token-group 量化": before dispatch
 * the hidden states are quantised to FP8 in groups of 128 consecutive
 * features of one token (the same 128 as expert_alignment) with UE8M0 scale
 * factors for DeepGEMM's 1x128 fine-grained scaling.  Here:
 *   codes   e4m3 (no infinities, max 448), round to nearest with ties to
 *           even, saturating at +-448; one byte per value;
 *   scales  per group of 128 values the smallest power of two 2^e with
 *           amax <= 448 * 2^e (e = 0 for an all-zero group), stored as the
 *           byte e + 127; code = e4m3(x / 2^e), value = e4m3 * 2^e.
 * Expert weights use the same rule on 128 x 128 blocks (output rows x input
 * features); gate and up rows of [P, 2I, H] fall in separate blocks. */

/* Per-token groups: x [n, K] (K a multiple of 128, MOE_BF16 or MOE_F32,
 * 16-byte aligned) -> d_q uint8[n, K] codes, d_scales uint8[n, K / 128]. */
moe_status moe_quantize_fp8_groups(const void* d_x, int64_t n, int K, int dtype, uint8_t* d_q,
                                   uint8_t* d_scales, void* stream);

/* 128 x 128 blocks: w [R, K] (R and K multiples of 128) -> d_q uint8[R, K],
 * d_scales uint8[R / 128, K / 128] (row-major over blocks).  Weights of all
 * slots quantise as one [P * rows, K] matrix. */
moe_status moe_quantize_fp8_blocks(const void* d_w, int64_t R, int K, int dtype, uint8_t* d_q,
                                   uint8_t* d_scales, void* stream);

/* moe_dispatch whose permuted rows are quantised on the way: every routed
 * copy of row g is the per-token-group FP8 quantisation of d_global row g.
 *   d_sorted_q       device uint8[cap, H] codes (16-byte aligned)
 *   d_sorted_scales  device uint8[cap, H / 128] scale bytes
 * H must be a multiple of 128.  Alignment padding rows get zero codes and
 * scale byte 127.  Counts, offsets, perm, inv and errors as moe_dispatch. */
moe_status moe_dispatch_fp8(const void* d_global, const int32_t* d_ids, int64_t rows, int k,
                            int H, int dtype, int E, int P, const int32_t* d_l2p,
                            const int32_t* d_nrep, int X, int align, int64_t cap,
                            int32_t* d_counts_P, int32_t* d_offsets_P, int32_t* d_perm,
                            int32_t* d_inv, uint8_t* d_sorted_q, uint8_t* d_sorted_scales,
                            void* d_ws, size_t ws_bytes, uint32_t* d_status, void* stream);

/* Workspace of moe_grouped_ffn_fp8: the FP8 SwiGLU activation (codes and
 * scale bytes) of cap rows, the fp32 activation of cap rows (the path for many
 * rows per slot), then the scheduler's words: the last
 * 4 * (3 + MOE_MAX_SLOTS) bytes.  They must be zero before the first call on a
 * workspace (e.g. a zero-filled allocation); every call leaves them zero.  A
 * call that finds them otherwise sets MOE_DEV_BAD_WORKSPACE (its output is then
 * not valid) and clears them.  One call at a time per workspace. */
size_t moe_grouped_ffn_fp8_ws_bytes(int64_t cap, int I);

/* Grouped SwiGLU FFN on FP8 operands (moe_grouped_ffn's computation): per
 * slot s in [slot_lo, slot_hi) and row x, with every GEMM summing
 * 2^(e_row + e_weight_block) * (e4m3 products) over 128-deep blocks in fp32:
 *   h = silu(x . Wg_s^T) * (x . Wu_s^T), quantised per token in groups of
 *   128 features; y = h . Wd_s^T, rounded to bf16.
 *   d_sorted_q, d_sorted_scales   moe_dispatch_fp8's output
 *   d_w_gate_up_q [P, 2I, H], d_w_gate_up_scales [P, 2I/128, H/128]
 *   d_w_down_q [P, H, I], d_w_down_scales [P, H/128, I/128]
 *   d_out_sorted  device bf16 [cap, H] out (rows of the slot range)
 * H a multiple of 256, I a multiple of 128; sm_103 only (else
 * MOE_ERR_UNSUPPORTED).  With few rows per slot both GEMMs run in one launch:
 * CTAs claim the MM1 units and then the MM2 units in order, and an MM2 unit
 * waits (bounded, else MOE_DEV_TIMEOUT) until its slot's h is written.  With
 * 192 or more rows per slot on average (cap / P), H and I multiples of 512 and
 * 4-byte aligned scale arrays, the GEMMs run on SM pairs with the weights as the
 * MMA's M operand and block-scaled MMAs (the scales applied by the tensor cores,
 * accumulators in tensor memory for a whole unit of up to 320 tokens): MM1 +
 * SwiGLU writes h in fp32 to the workspace, one launch quantises it per token
 * (groups of 128 features, as moe_quantize_fp8_groups), MM2 follows.  With 32 to
 * 191 rows per slot on average (a skewed layer, e.g. EPLB) the slots of 192 or
 * more rows take that path and the others the one-launch kernel after it. */
moe_status moe_grouped_ffn_fp8(const uint8_t* d_sorted_q, const uint8_t* d_sorted_scales,
                               const int32_t* d_offsets_P, int P, int slot_lo, int slot_hi,
                               int64_t cap, const uint8_t* d_w_gate_up_q,
                               const uint8_t* d_w_gate_up_scales, const uint8_t* d_w_down_q,
                               const uint8_t* d_w_down_scales, int H, int I, void* d_out_sorted,
                               void* d_ws, size_t ws_bytes, uint32_t* d_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_DP_H */

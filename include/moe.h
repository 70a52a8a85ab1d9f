/*
 * moe.h — C ABI of the sparse mixture-of-experts feed-forward layer (libmoe.so).
 *
 * The layer, as the Mixtral 8x7B pages define it ("Mixtral of Experts", xyznot.com
 * summary, section "Método (con las ecuaciones clave)"; blog.csdn.net post
 * "《Mixtral of Experts》Mixtral 8x7B：稀疏专家混合模型的突破性进展", section
 * "MOE数学公式"):
 *
 *     l    = x · W_g                       router logits, W_g in R^{d x n}
 *     G(x) = Softmax(TopK(l))              TopK keeps the K largest logits, the rest -> -inf
 *     y    = sum_i G(x)_i · E_i(x)         E_i(x) = w2_i · (SiLU(w1_i · x) ⊙ (w3_i · x))
 *
 * Only the K experts with a non-zero gate are evaluated, on the group of tokens routed
 * to them, and their outputs return to the original token positions ("Mixtral 8x7B:
 * 疎な専門家混合言語モデル", ja.news.hada.io, sections "MoEレイヤーの計算方式" and
 * "実装と推論効率").
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers (cudaMalloc / torch CUDA memory) unless
 *     stated otherwise; the caller owns every buffer, including the workspace.  The
 *     library allocates nothing and frees nothing.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  No call synchronises except moe_check_device_error().
 *   - Arguments are validated on the host before anything is launched.  On a non-OK
 *     status no kernel was launched and no output was written, except MOE_ERR_CUDA
 *     (a launch failed part-way; outputs are undefined).
 *   - Layouts are dense row-major with no padding:
 *       x, residual, y   [T, d]        activations
 *       w_gate           [d, n]        router weight (logits = x · w_gate)
 *       w1, w3           [n, f, d]     expert gate / up projections, out x in
 *       w2               [n, d, f]     expert down projection, out x in
 *       topk_idx         [T, k] int32  chosen experts, descending logit, ties -> lower index
 *       topk_w           [T, k] fp32   their gate values (sum to 1 per token)
 *       expert_offsets   [n + 1] int32 exclusive prefix sum of per-expert counts
 *       perm             [T*k] int32   perm[p] = assignment a = t*k + slot at position p,
 *                                      positions ordered by (expert, a)
 *       inv_perm         [T*k] int32   inv_perm[a] = position of assignment a
 *       y_perm           [T*k, d]      expert outputs E_e(x_t), one row per position p
 *   - dtype MOE_F32: x, w_gate, w1, w3, w2, residual, y_perm, y are float32.
 *     dtype MOE_BF16: they are bfloat16; products accumulate in fp32; the intermediate
 *     SiLU(a)⊙b and y_perm are rounded to bf16.  logit_bias, logits and topk_w are
 *     always float32.
 *   - Supported sizes: T >= 0, d >= 1, f >= 1, 1 <= k <= n <= 32, T*k < 2^31.  Tensor
 *     pointers must be 16-byte aligned.  MOE_BF16 experts run on the tensor cores when
 *     d % 64 == 0 and f % 64 == 0, otherwise on an fp32 CUDA-core kernel.
 *   - Device status: kernels report a timed-out wait or a bad expert index by setting bits
 *     of a status word in the first 256 bytes of the workspace.  The bits stay set until
 *     moe_check_device_error() reads and clears them, so a new workspace must start with
 *     those 256 bytes zeroed (cudaMemset once, or one moe_check_device_error call).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, bad dtype       */
  MOE_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement                  */
  MOE_ERR_WORKSPACE = 3,   /* workspace null or smaller than moe_workspace_size()           */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed                          */
  MOE_ERR_TIMEOUT = 5,     /* a kernel wait ran past its limit; the kernel gave up cleanly  */
  MOE_ERR_DEVICE_INDEX = 6 /* a kernel met an expert index outside [0, n)                   */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Human-readable name of a status code.  Never NULL. */
const char* moe_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int moe_version(void);

/*
 * Bytes of device workspace needed by moe_layer_forward (and enough for
 * moe_permute and moe_grouped_swiglu) for these sizes.  Returns 0 for invalid sizes.
 * The workspace holds a status header, the router outputs, the permutation, the
 * expert-ordered copy of x, the SwiGLU intermediate [T*k, f] and y_perm [T*k, d].  Apart
 * from the status header (see above) it needs no initialisation.
 */
size_t moe_workspace_size(int T, int d, int f, int n, int k, int dtype);

/*
 * Router and gate: logits l = x · w_gate (+ logit_bias), TopK, softmax over the K
 * kept logits ("Mixtral of Experts", Método, eq. G; blog.csdn.net MOE数学公式 §2.1-§2.3).
 *   x          [T, d]   dtype
 *   w_gate     [d, n]   dtype
 *   logit_bias [n] fp32, nullable: added to the logits before TopK and softmax
 *   topk_idx   [T, k] int32 out
 *   topk_w     [T, k] fp32 out
 *   logits     [T, n] fp32 out, nullable (biased logits, fp32 accumulation)
 * One warp per token (one block per token for batches of at most 1024 tokens with
 * n = 8 bf16); fp32 accumulation of the products.
 */
moe_status moe_router_topk(const void* x, const void* w_gate, const float* logit_bias, int T, int d,
                           int n, int k, int dtype, int32_t* topk_idx, float* topk_w, float* logits,
                           void* stream);

/*
 * Group the T*k assignments by expert: counts per expert, exclusive prefix sum into
 * expert_offsets, and a stable rank that yields perm / inv_perm (see layouts above).
 * Deterministic and bit-exact: within one expert, assignments keep ascending a = t*k+slot.
 *   topk_idx       [T, k] int32 in (values must be in [0, n))
 *   expert_offsets [n+1] int32 out; perm, inv_perm [T*k] int32 out
 *   ws, ws_bytes   workspace of at least moe_workspace_size(T, 64, 64, n, k, MOE_BF16)
 *                  bytes (only its status header and, for large T*k, per-block counts
 *                  are used)
 * An index outside [0, n) is reported by moe_check_device_error() as
 * MOE_ERR_DEVICE_INDEX.  Its assignment goes to a trailing bucket after the last expert:
 * expert_offsets[n] then counts only the valid assignments, the positions
 * [expert_offsets[n], T*k) hold the bad ones in ascending a, and perm / inv_perm remain a
 * permutation of [0, T*k), so later calls never index out of bounds with them.  The
 * experts skip the trailing bucket; what moe_combine reads for those slots is unspecified.
 */
moe_status moe_permute(const int32_t* topk_idx, int T, int k, int n, int32_t* expert_offsets,
                       int32_t* perm, int32_t* inv_perm, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_permute without a workspace.  The pages have no counterpart to this entry point; it
 * serves callers that cannot allocate device memory at all and have no workspace to hand
 * over — for example code that runs while a stream is being captured into a CUDA graph, or
 * inside a host runtime's enqueue callback, where cudaMalloc is not allowed.  Same inputs,
 * outputs and results as moe_permute.  Its scratch (a status word and the per-block counts)
 * is a fixed 34,048-byte array inside libmoe.so, which every GPU that loads the library
 * keeps until the process exits.
 *   - T*k must be at most 4,194,304; larger sizes return MOE_ERR_UNSUPPORTED.
 *   - The first call in a CUDA context (per device, and again after cudaDeviceReset or a
 *     switch to another context) looks up the array's device address with that context
 *     current; make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents (each call
 *     clears the part that must start at zero).  Calls that may overlap on the GPU (for
 *     instance on two streams with no ordering between them) race: results are undefined.
 *   - Expert indices outside [0, n) go to the trailing bucket as in moe_permute; nothing
 *     reports them here (moe_permute reports them through its workspace).
 */
moe_status moe_permute_noalloc(const int32_t* topk_idx, int T, int k, int n,
                               int32_t* expert_offsets, int32_t* perm, int32_t* inv_perm,
                               void* stream);

/*
 * The experts: for every expert e with rows p in [offsets[e], offsets[e+1]) and token
 * t = perm[p] / k,   y_perm[p] = w2_e · (SiLU(w1_e · x_t) ⊙ (w3_e · x_t))
 * ("Mixtral of Experts", Método: SwiGLU experts; ja.news.hada.io MoEレイヤーの計算方式:
 * experts with a zero gate are not computed).  Gate weights are NOT applied here.
 *   x [T, d], w1/w3 [n, f, d], w2 [n, d, f]: dtype;  y_perm [T*k, d]: dtype out
 *   perm, expert_offsets: as produced by moe_permute (read on the device; the host never
 *   sees the per-expert counts, so the call needs no synchronisation)
 * MOE_BF16 (d, f multiples of 64) runs two persistent tcgen05 grouped GEMMs (w1|w3 with
 * SiLU⊙ fused, then w2) fed by TMA; otherwise an fp32 CUDA-core kernel runs.
 *   ws, ws_bytes: at least moe_workspace_size(T, d, f, n, k, dtype) bytes.
 */
moe_status moe_grouped_swiglu(const void* x, const int32_t* perm, const int32_t* expert_offsets,
                              const void* w1, const void* w3, const void* w2, int T, int d, int f,
                              int n, int k, int dtype, void* y_perm, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * The two halves of moe_grouped_swiglu, for callers that keep the intermediate themselves
 * or time the projections separately.  Together they compute exactly moe_grouped_swiglu.
 *   moe_expert_up:   h[p] = SiLU(w1_e · x_t) ⊙ (w3_e · x_t),  t = perm[p] / k
 *                    h [T*k, f] dtype out (bf16: rounded once).  ws as for moe_grouped_swiglu
 *                    (holds the expert-ordered copy of x).
 *   moe_expert_down: y_perm[p] = w2_e · h[p]      (ws: only its status header is used)
 */
moe_status moe_expert_up(const void* x, const int32_t* perm, const int32_t* expert_offsets,
                         const void* w1, const void* w3, int T, int d, int f, int n, int k,
                         int dtype, void* h, void* ws, size_t ws_bytes, void* stream);
moe_status moe_expert_down(const void* h, const int32_t* expert_offsets, const void* w2, int T,
                           int d, int f, int n, int k, int dtype, void* y_perm, void* ws,
                           size_t ws_bytes, void* stream);

/*
 * Gate-weighted sum back in token order ("Mixtral of Experts", Método, eq. y):
 *   y[t] = sum_{slot<k} topk_w[t, slot] · y_perm[inv_perm[t*k + slot]]  (+ residual[t])
 * fp32 accumulation in ascending slot order (deterministic), one rounding to dtype.
 *   residual [T, d] dtype, nullable.   y may alias residual.
 */
moe_status moe_combine(const void* y_perm, const int32_t* inv_perm, const float* topk_w,
                       const void* residual, int T, int d, int k, int dtype, void* y, void* stream);

/*
 * Row-wise RMSNorm with unit weight, x[t] = h[t] / sqrt(mean(h[t]^2) + eps), fp32 math,
 * one rounding to dtype.  Not part of the pages' layer; used by stacked layers
 * h <- h + MoE(RMSNorm(h)).   x may not alias h.
 */
moe_status moe_rmsnorm(const void* h, int T, int d, float eps, int dtype, void* x, void* stream);

/*
 * One whole MoE layer: router_topk -> permute -> grouped_swiglu -> combine, all on
 * `stream`, no host synchronisation (the sequence can be captured in a CUDA graph).
 *   residual          [T, d] nullable: y = residual + MoE(x)
 *   topk_idx_out      [T, k] int32 nullable: copy of the chosen experts
 *   expert_offsets_out[n+1] int32 nullable: copy of the per-expert offsets
 *   ws, ws_bytes      at least moe_workspace_size(T, d, f, n, k, dtype) bytes
 */
moe_status moe_layer_forward(const void* x, const void* w_gate, const float* logit_bias,
                             const void* w1, const void* w3, const void* w2, const void* residual,
                             int T, int d, int f, int n, int k, int dtype, void* y,
                             int32_t* topk_idx_out, int32_t* expert_offsets_out, void* ws,
                             size_t ws_bytes, void* stream);

/*
 * Backward of the layer y = MoE(x) (without residual; with y = r + MoE(x) the residual's
 * gradient is dy itself): the gradients of L = <dy, y> by the chain rule through the pages'
 * definition ("Mixtral of Experts", Método, eqs. G and y; blog.csdn.net MOE数学公式 §2).
 * TopK is piecewise constant, so only the K kept logits of each token get gradient, through
 * the softmax over them:  dl_k = G_k (dG_k - sum_j G_j dG_j),  dG_k = <dy, E_{e_k}(x)>.
 * The routing is recomputed from x, w_gate and logit_bias with the forward's kernels (the
 * same selection and gates as moe_layer_forward on the same inputs).
 *   x, dy           [T, d] dtype        inputs of the forward / gradient of its output
 *   w_gate [d, n], w1, w3 [n, f, d], w2 [n, d, f] dtype;  logit_bias [n] fp32 nullable
 *   dx              [T, d] dtype out    fp32 accumulation, one rounding
 *   dw_gate         [d, n] fp32 out
 *   dlogit_bias     [n] fp32 out, nullable
 *   dw1, dw3        [n, f, d] dtype out; dw2 [n, d, f] dtype out (fp32 accumulation over the
 *                   expert's rows, one rounding; experts without rows get zeros)
 *   ws, ws_bytes    at least moe_backward_workspace_size(T, d, f, n, k, dtype) bytes, its
 *                   first 256 bytes zeroed as for every workspace (status word)
 * Every output is overwritten (not accumulated into).  The expert GEMMs run in an
 * expert-padded row order (every expert's rows padded with zero rows to a multiple of 128):
 * on tcgen05 for MOE_BF16 with d % 64 == 0 and f % 64 == 0, otherwise on CUDA cores (fp32
 * products; bf16 storage rounds the intermediates to bf16 as the tensor-core path does).
 */
size_t moe_backward_workspace_size(int T, int d, int f, int n, int k, int dtype);
moe_status moe_layer_backward(const void* x, const void* w_gate, const float* logit_bias,
                              const void* w1, const void* w3, const void* w2, const void* dy,
                              int T, int d, int f, int n, int k, int dtype, void* dx,
                              float* dw_gate, float* dlogit_bias, void* dw1, void* dw3, void* dw2,
                              void* ws, size_t ws_bytes, void* stream);

/*
 * Training pair: a forward that keeps what the backward needs, and the backward that uses it
 * instead of recomputing the routing and the expert inputs a = x w1ᵀ, b = x w3ᵀ (the
 * recompute is a quarter of moe_layer_backward's expert FLOPs).  Same results as
 * moe_layer_forward / moe_layer_backward on the same inputs.
 *   moe_train_saved_size   bytes of the `saved` buffer for these sizes (0 where the pair is
 *                          not implemented: only MOE_BF16 with d % 64 == 0 and f % 64 == 0)
 *   moe_layer_forward_train   moe_layer_forward (same arguments; no topk_idx_out /
 *                          expert_offsets_out) that also fills `saved` (caller-owned device
 *                          memory, 16-byte aligned): the routing (TopK indices and gates, the
 *                          grouping) and a | b in bf16, rows in the expert-padded order
 *   moe_layer_backward_saved  moe_layer_backward from `saved` (left unchanged, reusable) with
 *                          the same x, weights and dy; no logit_bias (the routing is saved)
 * Other dtypes or shapes return MOE_ERR_UNSUPPORTED.
 */
size_t moe_train_saved_size(int T, int d, int f, int n, int k, int dtype);
moe_status moe_layer_forward_train(const void* x, const void* w_gate, const float* logit_bias,
                                   const void* w1, const void* w3, const void* w2,
                                   const void* residual, int T, int d, int f, int n, int k,
                                   int dtype, void* y, void* saved, size_t saved_bytes, void* ws,
                                   size_t ws_bytes, void* stream);
moe_status moe_layer_backward_saved(const void* x, const void* w_gate, const void* w1,
                                    const void* w3, const void* w2, const void* dy, int T, int d,
                                    int f, int n, int k, int dtype, const void* saved,
                                    size_t saved_bytes, void* dx, float* dw_gate,
                                    float* dlogit_bias, void* dw1, void* dw3, void* dw2, void* ws,
                                    size_t ws_bytes, void* stream);

/*
 * Causal grouped-query attention, the attention sub-block's core (the pages: 32 attention
 * heads and 8 key-value heads at hidden size 4096, i.e. head dimension 128, over the full
 * dense 32k context; "Mixtral of Experts", Método; newsflash.city digest):
 *     out[t, h] = sum_{s <= t, same sequence} softmax_s(q[t, h] · k[s, g] / sqrt(dh)) v[s, g]
 * with g = h / (hq / hkv).  The pages give no positional encoding; positions enter through
 * the causal mask only.
 *   q, out      [T, hq, dh] bf16;   k, v  [T, hkv, dh] bf16   (dense, 16-byte aligned)
 *   seq_len     0: the T tokens are one sequence; > 0: sequences of seq_len tokens (the last
 *               may be shorter), attention never crosses a sequence boundary
 *   ws          any workspace of at least 256 bytes (its status word reports timeouts)
 * fp32 scores and softmax (online, exp2), P rounded to bf16 for the P·V product, fp32
 * accumulation in TMEM, one rounding of the output.  Only dtype MOE_BF16 with dh = 128 is
 * implemented (MOE_ERR_UNSUPPORTED otherwise).
 */
moe_status moe_attention_gqa(const void* q, const void* k, const void* v, int T, int seq_len,
                             int hq, int hkv, int dh, int dtype, void* out, void* ws,
                             size_t ws_bytes, void* stream);

/*
 * Routing statistics of one layer from its TopK selections (newsflash.city digest,
 * "路径分析", Table 5: how often consecutive tokens are sent to the same expert;
 * "Mixtral of Experts" (xyznot.com summary), "Limitaciones": 28.4% first-choice repetition
 * at layer 15 against 12.5% for random assignment).
 *   topk_idx      [T, k] int32 in, as written by moe_router_topk
 *   seq_len       0: the T tokens form one sequence; > 0: sequences of seq_len tokens (the
 *                 last may be shorter) and no pair crosses a sequence boundary
 *   expert_counts [n] int64 out: assignments routed to each expert (the layer's load)
 *   pair_counts   [3] int64 out: { consecutive pairs (t, t+1) inside a sequence,
 *                 pairs with equal first-choice experts,
 *                 pairs whose k chosen experts share at least one expert }
 * Both outputs are overwritten (8-byte aligned device memory; topk_idx 4-byte aligned).
 * An index outside [0, n) is left out of expert_counts (their sum then falls short of
 * T*k) and out of the shared-expert test; first choices are compared as stored.
 * No workspace; stream-ordered like every call here.
 */
moe_status moe_routing_stats(const int32_t* topk_idx, int T, int k, int n, int seq_len,
                             int64_t* expert_counts, int64_t* pair_counts, void* stream);

/*
 * One decoder layer of the Mixtral stack: Mistral 7B's layer with the feed-forward sub-block
 * replaced by the MoE layer ("Mixtral of Experts", Método: 32 query heads, 8 key-value heads,
 * hidden 4096, so head dimension 128):
 *     a  = RMSNorm(h)
 *     h1 = h + attention_gqa(a wqᵀ, a wkᵀ, a wvᵀ) woᵀ        (moe_attention_gqa, dh = 128)
 *     y  = h1 + MoE(RMSNorm(h1))                              (moe_layer_forward)
 * The pages name neither the normalisation nor a positional encoding: RMSNorm with unit
 * weight (eps) before each sub-block, and no positional encoding.
 *   h, y      [T, d] bf16 (y may alias h)
 *   wq        [hq*128, d], wk / wv [hkv*128, d], wo [d, hq*128] bf16 (out x in)
 *   w_gate, logit_bias, w1, w3, w2, k, n, f: as for moe_layer_forward
 *   seq_len   tokens per sequence for the attention (0: one sequence)
 *   topk_idx_out [T, k] int32, nullable: the MoE sub-block's expert choices
 *   ws        at least moe_decoder_workspace_size(...) bytes; status header as usual
 * bf16 only, d and f multiples of 64 (the tensor-core path); otherwise MOE_ERR_UNSUPPORTED.
 * The projections run on the grouped tensor-core GEMM with one group holding every row.
 */
size_t moe_decoder_workspace_size(int T, int d, int f, int n, int k, int hq, int hkv);
moe_status moe_decoder_layer_forward(const void* h, const void* wq, const void* wk, const void* wv,
                                     const void* wo, const void* w_gate, const float* logit_bias,
                                     const void* w1, const void* w3, const void* w2, int T, int d,
                                     int f, int n, int k, int hq, int hkv, int seq_len, float eps,
                                     int dtype, void* y, int32_t* topk_idx_out, void* ws,
                                     size_t ws_bytes, void* stream);

/*
 * Expert parallelism (EP): the layer spread over G GPUs by experts.  Tokens an expert must
 * process go to the GPU holding it and its outputs return to the original token positions
 * (newsflash.city digest, section "专家层的混合"; ja.news.hada.io, section "実装と推論効率").
 * Rank g of G holds the experts [g*E, (g+1)*E), E = n/G.  A layer pass on rank g is:
 * moe_router_topk and moe_permute on its own tokens; moe_gather_rows of x into grouping
 * order; an all-to-all of the per-expert counts and an all-to-all-v of the rows (the
 * caller's collective library, e.g. NCCL); moe_ep_regroup; moe_gather_rows into the
 * experts' order; moe_expert_up / moe_expert_down with the local experts' weights (k = 1,
 * n = E); moe_gather_rows back to receive order; the reverse all-to-all-v; moe_combine.
 *
 * moe_ep_regroup: the receive buffer of rank g holds, source after source (s = 0..G-1),
 * each source's rows for g's experts in the source's order (local expert j = 0..E-1, then
 * assignment).  Orders them by local expert, then source:
 *   recv_counts   [G, E] int32 in (device): rows from source s for local expert j
 *   R             total rows = sum of recv_counts (known to the caller, who sized the
 *                 buffers with it); positions at or past R are never written
 *   local_offsets [E+1] int32 out: exclusive prefix sum of the local experts' rows
 *   row_map       [R] int32 out: row_map[p] = receive-buffer row at grouped position p
 *   inv_row_map   [R] int32 out: inv_row_map[q] = grouped position of receive row q
 * Negative counts count as 0.  Bit-exact (integer only), deterministic.
 */
moe_status moe_ep_regroup(const int32_t* recv_counts, int G, int E, int R, int32_t* local_offsets,
                          int32_t* row_map, int32_t* inv_row_map, void* stream);

/*
 * Row gather by an index vector:  dst[p] = src[index[p] / k]  for p < rows.
 *   src [rows_src, row_bytes] in; index [rows] int32 in; dst [rows, row_bytes] out.
 * An index outside [0, rows_src * k) gives a zero row (no read out of bounds).  16-byte
 * vectors when row_bytes and both pointers allow it.  Used by the EP sequence above.
 */
moe_status moe_gather_rows(const void* src, int rows_src, const int32_t* index, int rows, int k,
                           size_t row_bytes, void* dst, void* stream);

/*
 * Synchronise `stream`, read the device status word that the kernels of the last calls
 * using this workspace may have set, and clear it.  Returns MOE_OK, MOE_ERR_TIMEOUT or
 * MOE_ERR_DEVICE_INDEX (or MOE_ERR_CUDA if the synchronisation itself failed).
 */
moe_status moe_check_device_error(void* ws, size_t ws_bytes, void* stream);

/*
 * Wait limit, in nanoseconds, of every bounded wait inside the tensor-core kernels
 * (default 2e9).  A wait that runs past it makes its kernel stop cleanly and set
 * MOE_ERR_TIMEOUT.  Process-wide; takes effect at the next launch.  0 restores the default.
 */
void moe_set_wait_limit_ns(unsigned long long ns);

/*
 * Which form of the tensor-core expert GEMMs the bf16 calls use (process-wide; takes effect
 * at the next launch):
 *   MOE_TC_FORM_AUTO    (default) for batches of at most 64 tokens (decode), the swapped
 *                       form of both forward GEMMs: the weights are the 128-row side of
 *                       every MMA and the expert's token rows, in blocks of 16-64 rows, the
 *                       other side, so that each SM keeps more weight bytes in flight.  Else
 *                       the CTA-pair form (tcgen05 cta_group::2, 256-row tiles over two SMs)
 *                       for the down-projection (w2) when the experts average at least 256
 *                       rows (T*k >= 256*n) and for the up-projection (w1|w3 with SwiGLU) when
 *                       they average at least 512 (T*k >= 512*n); the single-CTA form (128-row
 *                       tiles) otherwise.  The forward that keeps a|b for the backward
 *                       (moe_layer_forward_train) never takes the swapped form for its
 *                       up-projection.  In the backward the weight-gradient GEMMs (dW1, dW3,
 *                       dW2: 256-row tiles of dW) always take the pair form and the other
 *                       backward GEMMs the single form.
 *   MOE_TC_FORM_SINGLE  always the single-CTA form
 *   MOE_TC_FORM_PAIR    always the CTA-pair form for the forward GEMMs and the weight
 *                       gradients (where the device can co-schedule pairs)
 *   MOE_TC_FORM_SWAP    the swapped form for the forward GEMMs at any batch size (token
 *                       blocks of 64 rows above 64 tokens; an expert's weights are read once
 *                       per block); the AUTO rules elsewhere
 * The single-CTA and pair forms accumulate K in the same ascending order, so their outputs
 * are identical; the swapped form agrees with them within the rounding of the fp32 sums.
 * Returns MOE_ERR_INVALID_ARG for any other value.
 */
enum { MOE_TC_FORM_AUTO = 0, MOE_TC_FORM_SINGLE = 1, MOE_TC_FORM_PAIR = 2, MOE_TC_FORM_SWAP = 3 };
moe_status moe_set_tc_form(int form);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */

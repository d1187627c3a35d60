/*
 * mtgr.h -- C ABI of libmtgr.so: one MTGR HSTU layer (Group LayerNorm, UQKV
 * projection + SiLU, jagged HSTU attention under the dynamic mixed mask,
 * LayerNorm(O) ⊙ U, output projection + residual), forward and backward,
 * as hand-written CUDA kernels for B300 (sm_103a); a stack of layers run
 * forward in one call for ranking; and the host-side construction of training
 * batches (stochastic length, token-balanced ranks).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Ownership.  Every pointer argument is caller-owned.  Tensor arguments are
 *   DEVICE pointers (current device) unless the comment says "host".  The
 *   library allocates no device memory of its own: scratch comes from the
 *   caller's `workspace`, sized by the matching *_workspace_size() query
 *   (mtgr_group_layernorm_bwd_noalloc uses a fixed array inside the library).
 * Streams.  Every call enqueues work on `stream` (a cudaStream_t; NULL = the
 *   legacy default stream) and returns without synchronising.
 * Layout.  Row-major.  T tokens of B users, user b owning rows
 *   offsets[b] .. offsets[b+1]-1 (int32 offsets[B+1], offsets[0] = 0,
 *   offsets[B] = T), ordered User*, Seq*, RealTime*, Cand* inside a user;
 *   gid[t] in {0 User, 1 Seq, 2 RealTime, 3 Cand} (uint8); ts[t] int64 seconds.
 *   Head h of a [T, H*d_h] activation occupies columns h*d_h .. h*d_h+d_h-1.
 * Types.  MTGR_BF16: the layer's inputs, outputs and weights bf16, statistics
 *   fp32, weight / GLN-parameter gradients fp32, fp32 accumulation throughout;
 *   inside the layer the tensor-core operands and everything saved or passed
 *   between steps are f16 (11 significand bits against bf16's 8; see
 *   mtgr_hstu_layer_bwd for the gradients' scaling).  MTGR_F16: the
 *   forward-only inference variant, f16 activations and weights.  MTGR_F32:
 *   everything fp32.  gamma/beta are fp32 in every mode.
 * Errors.  A non-zero mtgr_status means nothing was enqueued, except
 *   MTGR_ERR_CUDA, which reports a launch failure; mtgr_last_error() returns a
 *   thread-local message.  Malformed device metadata is not checked by the
 *   compute calls (that would need a host round trip): call
 *   mtgr_validate_batch() once per batch.  Kernels never trap; they clamp
 *   offsets to [0, T], so malformed metadata gives wrong numbers, not faults.
 *
 * The operations follow these pages on MTGR (Meituan's generative-style ranking
 * model):
 *  - marovi.ai, "MTGR: Industrial-Scale Generative Recommendation Framework in
 *    Meituan/es", section "Métodos": sample D = [U, S, R, (C,I)_1..K], block
 *    update Ṽ = silu(KᵀQ)/(N_U+N_S+N_R+N_I) · M · V.
 *  - paper-daily.com, "MTGR：美团外卖生成式推荐Scaling Law落地实践", sections
 *    "模型怎么搭" (linear + SiLU -> U,Q,K,V; SiLU(QKᵀ) without softmax; normalise
 *    the aggregate, gate with U, final linear; Group LayerNorm) and
 *    "训练数据怎么组织，掩码怎么设" (jagged user rows, raw timestamps, mask).
 *  - fun-rec chapter 7.3 "MTGR：混合范式建模", §7.3.3 (GLN formula) and
 *    §7.3.4 (the three dynamic-masking rules).
 */
#ifndef MTGR_H_
#define MTGR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MTGR_API __attribute__((visibility("default")))
#else
#define MTGR_API
#endif

typedef struct CUstream_st* mtgr_stream_t; /* == cudaStream_t */

typedef enum {
  MTGR_OK = 0,
  MTGR_ERR_INVALID_ARG = -1,     /* a scalar argument or pointer is invalid */
  MTGR_ERR_BAD_OFFSETS = -2,     /* reported through the status word only */
  MTGR_ERR_BAD_GROUP_ORDER = -3, /* reported through the status word only */
  MTGR_ERR_UNSUPPORTED = -4,     /* shape / dtype / device not supported */
  MTGR_ERR_CUDA = -5,            /* a CUDA runtime call failed */
  MTGR_ERR_TIMEOUT = -6,         /* reported through the status word only */
  MTGR_ERR_WORKSPACE = -7        /* workspace missing or smaller than queried */
} mtgr_status;

/* MTGR_F16 is the inference variant (the pages serve in FP16, paper-daily
 * "计算量涨了 65 倍…"): activations, weights and the layer's outputs in f16.
 * It is accepted by mtgr_group_layernorm_fwd, mtgr_layer_workspace_size,
 * mtgr_hstu_layer_fwd and mtgr_hstu_stack_fwd (the layer's saved state is
 * then f16 too); the attention and backward entry points return
 * MTGR_ERR_UNSUPPORTED for it. */
typedef enum { MTGR_F32 = 0, MTGR_BF16 = 1, MTGR_F16 = 2 } mtgr_dtype;

/* Bits of the int32 device status word written by mtgr_validate_batch and
 * OR-ed by kernels that give up a bounded wait. */
#define MTGR_STATUS_BAD_OFFSETS 1
#define MTGR_STATUS_BAD_GROUP_ORDER 2
#define MTGR_STATUS_BAD_GROUP_ID 4
#define MTGR_STATUS_TIMEOUT 8

/* Thread-local description of the last non-OK status. */
MTGR_API const char* mtgr_last_error(void);
/* Library version (major*10000 + minor*100 + patch). */
MTGR_API int mtgr_version(void);

/* Kernel tracing (host side).  While enabled, every kernel launch of the
 * library is bracketed by two CUDA events recorded on the launching stream.
 * mtgr_trace_report() waits for the recorded events, then writes per kernel
 * name (up to max_entries, each name truncated to name_len-1 bytes into
 * names[k*name_len]) the summed device time in ms and the launch count, and
 * returns the number of distinct names (-1 on a CUDA error).  The events are
 * pooled and reused after mtgr_trace_reset(). */
MTGR_API void mtgr_trace_enable(int on);
MTGR_API void mtgr_trace_reset(void);
MTGR_API int mtgr_trace_report(int max_entries, char* names, int name_len, double* total_ms, int32_t* launches);

/* ------------------------------------------------------------------------- */
/* Batch metadata                                                             */
/* ------------------------------------------------------------------------- */

/* Check the jagged metadata on the device (sample layout of the marovi.ai
 * "Métodos" section; token order of fun-rec §7.3.1): offsets[0] = 0,
 * non-decreasing, offsets[B] = T; gid <= 3; inside a segment the group ids do
 * not decrease (User*, Seq*, RealTime*, Cand*).  Writes the MTGR_STATUS_* bits
 * into *status_word (device int32, overwritten, 0 = valid). */
MTGR_API mtgr_status mtgr_validate_batch(const int32_t* offsets, int32_t B, const uint8_t* gid, int64_t T,
                                int32_t* status_word, mtgr_stream_t stream);

/* Dynamic mixed mask, integer export (fun-rec §7.3.4 rules 1-3): cnt[t]
 * (device int32 [T]) = number of keys row t may attend to inside its user;
 * *total_pairs (device int64, overwritten) = sum over t.  Rule reading:
 * User/Seq keys are seen by every row; a RealTime key j is seen by RealTime
 * rows i with ts_j <= ts_i and by candidate rows i with ts_j < ts_i; a
 * candidate key is seen only by itself. */
/* Copies to counts_host[0..3] (host memory) the plan counts that the last
 * attention or layer call on `workspace` (device memory; a layer workspace
 * holds its attention workspace first) left there for a batch of B users:
 * the work items of the forward, of the dK/dV pass and of the dQ pass, and 1
 * when that backward kept its dS tiles (mtgr_attn_ds_store_size), else 0.
 * Synchronises `stream`.  For inspection and tests. */
MTGR_API mtgr_status mtgr_debug_plan_counts(const void* workspace, int32_t B, int32_t* counts_host,
                                            mtgr_stream_t stream);

MTGR_API mtgr_status mtgr_debug_visible_counts(const int32_t* offsets, int32_t B, const uint8_t* gid, const int64_t* ts,
                                      int64_t T, int32_t* cnt, int64_t* total_pairs, mtgr_stream_t stream);

/* Self-check of the timeout path.  Launches one CTA that takes tensor memory
 * and waits on an mbarrier that nothing completes, with the same bounded waits
 * the tcgen05 kernels use (limit 2 s of %globaltimer).  When they give up it
 * ORs MTGR_STATUS_TIMEOUT into *status_word (device int32, not cleared), frees
 * its tensor memory and returns; nothing faults or hangs and the context stays
 * usable.  Asynchronous on stream; takes about 2 s of one SM. */
MTGR_API mtgr_status mtgr_debug_wait_timeout(int32_t* status_word, mtgr_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Group LayerNorm (fun-rec §7.3.3: GLN(x_i) = (x_i - μ)/σ · γ_g(i) + β_g(i);  */
/* paper-daily "模型怎么搭": one set of normalisation parameters per token      */
/* class).  μ, σ² are per token over its D features (biased variance,          */
/* σ = sqrt(σ² + eps)); gamma/beta are fp32 [4, D], row g for group g.         */
/* ------------------------------------------------------------------------- */

/* x, y: [T, D] (dtype).  mean, rstd: fp32 [T] (may be NULL).  D % 8 == 0,
 * D <= 8192. */
MTGR_API mtgr_status mtgr_group_layernorm_fwd(const void* x, void* y, float* mean, float* rstd, const uint8_t* gid,
                                     const float* gamma, const float* beta, int64_t T, int32_t D, float eps,
                                     mtgr_dtype dtype, mtgr_stream_t stream);

MTGR_API size_t mtgr_group_layernorm_bwd_workspace_size(int64_t T, int32_t D);

/* dx = GLN'(x)ᵀ dy (+ dx_residual when non-NULL, same dtype as dx);
 * dgamma, dbeta: fp32 [4, D], overwritten.  mean/rstd from the forward. */
MTGR_API mtgr_status mtgr_group_layernorm_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
                                     const uint8_t* gid, const float* gamma, const void* dx_residual, void* dx,
                                     float* dgamma, float* dbeta, int64_t T, int32_t D, mtgr_dtype dtype,
                                     void* workspace, size_t workspace_bytes, mtgr_stream_t stream);

/* Same result as mtgr_group_layernorm_bwd, for callers that cannot allocate
 * device memory when they call it (a framework whose allocator owns all device
 * memory, a process that reserved its memory up front, a latency-critical step
 * that must not allocate) and so cannot pass a workspace.  The pages have no
 * counterpart: this is a packaging variant, not a step of the method.
 * The per-block dγ/dβ partial sums go to one fixed 10 MiB device array inside
 * the library (held by every device that loads the library until the process
 * exits).  Nothing is allocated: no cudaMalloc, cudaFree or allocating library
 * call.  Limit: D <= 4096 (a launch uses at most 2,621,440 / (8*D) blocks: the
 * full grid of two blocks per SM on a 148-SM B300 up to D = 1107, fewer above);
 * larger D returns MTGR_ERR_UNSUPPORTED with a message.  The first call on each
 * device looks up the array's device address (cudaGetSymbolAddress, with that
 * device current) and keeps it for later calls; make that first call before any
 * stream capture.  The kept address is not valid after cudaDeviceReset (the
 * context that held the array is gone): do not call this again after a reset
 * in the same process.  Every call
 * shares the array and overwrites the part it reads, so no clearing is needed,
 * but calls that overlap on the GPU (other streams, other host threads) race on
 * it: serialise them.  Arguments, layouts and errors as mtgr_group_layernorm_bwd. */
MTGR_API mtgr_status mtgr_group_layernorm_bwd_noalloc(const void* dy, const void* x, const float* mean,
                                             const float* rstd, const uint8_t* gid, const float* gamma,
                                             const void* dx_residual, void* dx, float* dgamma, float* dbeta,
                                             int64_t T, int32_t D, mtgr_dtype dtype, mtgr_stream_t stream);

/* ------------------------------------------------------------------------- */
/* HSTU attention (marovi.ai "Métodos" block formula; paper-daily "模型怎么搭")  */
/*   s_ij = q_i·k_j / sqrt(d_h);  A_ij = M_ij · silu(s_ij) / n_u;              */
/*   O_i = Σ_j A_ij v_j;  Y_i = LayerNorm(O_i) ⊙ u_i,                          */
/* per head, over the keys j of row i's own user; n_u = that user's token     */
/* count; LayerNorm over all H*d_h features of the row, no affine, eps inside  */
/* the square root; M is the dynamic mixed mask (see visible counts above).    */
/* ------------------------------------------------------------------------- */

/* Workspace for mtgr_hstu_attn_fwd / _bwd (jagged tile schedule, dO and the
 * dQ accumulator).  Its first 4 bytes are the call's device status word
 * (MTGR_STATUS_* bits; cleared by each call, set if a bounded wait gave up). */
MTGR_API size_t mtgr_attn_workspace_size(int32_t B, int64_t T, int32_t n_heads, int32_t d_h, mtgr_dtype dtype);

/* Extra workspace with which the MTGR_BF16 backward (mtgr_hstu_attn_bwd,
 * mtgr_hstu_layer_bwd) keeps its dS tiles: one 128 x 128 f16 tile (32 KB) per
 * head and per (query tile, key tile) of each user's tile grid,
 * n_heads * sum_b ceil(n_b/128)^2 tiles plus 1024 bytes of alignment, where
 * n_b = offsets_host[b+1] - offsets_host[b] (offsets_host: the batch's B+1
 * offsets in HOST memory).  0 for other dtypes or d_h, or for bad offsets.
 * A backward whose workspace holds at least this many bytes beyond its
 * required size copies each dS tile of the dK/dV pass to HBM and forms dQ =
 * dS K from the stored tiles (one product per tile pair) instead of
 * recomputing S and dP (three); the gradients are the same up to f32
 * summation order.  The device decides from the metadata it was given: when
 * the tiles of the batch do not fit the extra bytes, the recomputing pass
 * runs.  Derivation of the backward: marovi.ai "Métodos" block formula. */
MTGR_API size_t mtgr_attn_ds_store_size(const int32_t* offsets_host, int32_t B, int32_t n_heads, int32_t d_h,
                                        mtgr_dtype dtype);

/* q, k, v, u: [T, *] with row stride ld_in elements (e.g. views into one
 * [T, 4*H*d_h] buffer).  In the MTGR_BF16 path the tensor-core operands are
 * f16: q, k, v are first copied to f16 (exact for values in the f16 normal
 * range, |x| in [6.1e-5, 65504]) and P, dO, dS are rounded to f16 (11
 * significand bits) instead of bf16 (8).  y: [T, H*d_h] dense (dtype).  o_saved:
 * [T, H*d_h], O before the gate (needed by the backward): f16 in the MTGR_BF16
 * path (11 significand bits; O is an average of V rows, far inside the f16
 * range), fp32 in the MTGR_F32 path.  ln_mean, ln_rstd: fp32 [T].
 * Supported: MTGR_BF16 with d_h in {64, 128} (tcgen05 tensor-core path) and
 * MTGR_F32 with d_h <= 128, d_h % 4 == 0 (fp32 CUDA-core path). */
MTGR_API mtgr_status mtgr_hstu_attn_fwd(const void* q, const void* k, const void* v, const void* u, int64_t ld_in,
                               const int32_t* offsets, int32_t B, const uint8_t* gid, const int64_t* ts,
                               int64_t T, int32_t n_heads, int32_t d_h, float eps, void* y, void* o_saved,
                               float* ln_mean, float* ln_rstd, mtgr_dtype dtype, void* workspace,
                               size_t workspace_bytes, mtgr_stream_t stream);

/* Backward of mtgr_hstu_attn_fwd for upstream dy [T, H*d_h].  Writes dq, dk,
 * dv, du (row stride ld_grad elements; every row of every segment is
 * overwritten).  silu'(s) = σ(s)(1 + s(1 - σ(s))).  When dsilu_uqkv is not
 * NULL it is a [T, 4*H*d_h] multiplier (dtype, row stride ld_grad, which must
 * then be 4*H*d_h; column blocks U, Q, K, V, each head-major) and every
 * gradient is also multiplied elementwise by its block.  The layer passes
 * silu'(z) of its UQKV pre-activation z, which fuses the SiLU backward of the
 * projection into this call.  Workspace: mtgr_attn_workspace_size; with
 * mtgr_attn_ds_store_size more bytes the MTGR_BF16 backward keeps its dS
 * tiles and forms dQ from them. */
MTGR_API mtgr_status mtgr_hstu_attn_bwd(const void* dy, const void* q, const void* k, const void* v, const void* u,
                               int64_t ld_in, const void* o_saved, const float* ln_mean, const float* ln_rstd,
                               const int32_t* offsets, int32_t B, const uint8_t* gid, const int64_t* ts,
                               int64_t T, int32_t n_heads, int32_t d_h, void* dq, void* dk, void* dv, void* du,
                               int64_t ld_grad, const void* dsilu_uqkv, mtgr_dtype dtype, void* workspace,
                               size_t workspace_bytes, mtgr_stream_t stream);

/* ------------------------------------------------------------------------- */
/* One HSTU layer (paper-daily "模型怎么搭"; paper-daily deep reading §2       */
/* "统一 HSTU 编码 + Group LayerNorm"):                                       */
/*   xn = GLN(x);  z = xn · W_uqkv;  [U|Q|K|V] = silu(z);                      */
/*   Y = LayerNorm(attention(Q,K,V)) ⊙ U;  x' = x + Y · W_o.                   */
/* ------------------------------------------------------------------------- */
typedef struct {
  int32_t d_model;      /* D; multiple of 64 */
  int32_t n_heads;      /* H */
  int32_t d_h;          /* head dim; H*d_h multiple of 64 */
  const void* w_uqkv;   /* [D, 4*H*d_h] (dtype): column blocks U, Q, K, V */
  const void* w_o;      /* [H*d_h, D] (dtype) */
  const float* gamma;   /* [4, D] fp32 */
  const float* beta;    /* [4, D] fp32 */
  float eps_gln;        /* 1e-5 */
  float eps_ln;         /* 1e-5 */
  /* Optional, MTGR_BF16 only: f16 copies of w_uqkv and w_o (same shapes,
   * 16-byte aligned, caller-owned), as written by mtgr_layer_weights_to_f16.
   * When both are set the layer's tensor-core operands are read from them;
   * when both are NULL (zero-initialised struct) every forward and backward
   * call converts the weights into its workspace first (two kernels).  The
   * caller keeps them equal to the bf16 weights: refresh them after every
   * weight update (inference with fixed weights converts once).  Setting
   * only one is MTGR_ERR_INVALID_ARG; the other dtypes ignore them. */
  const void* w_uqkv_f16;
  const void* w_o_f16;
} mtgr_layer_weights;

/* f16 copies of a MTGR_BF16 layer's w_uqkv and w_o into caller-owned device
 * buffers of D*4*H*d_h and H*d_h*D f16 elements (16-byte aligned).  Each
 * value is the bf16 weight rounded to f16 (exact in f16's normal range).
 * Reads only d_model, n_heads, d_h, w_uqkv and w_o of *w. */
MTGR_API mtgr_status mtgr_layer_weights_to_f16(const mtgr_layer_weights* w, void* w_uqkv_f16, void* w_o_f16,
                                      mtgr_stream_t stream);

typedef struct {        /* written by the forward, read by the backward: f16 in the MTGR_BF16 and
                           MTGR_F16 paths (11 significand bits between the steps), fp32 in MTGR_F32 */
  void* xn;             /* [T, D] GLN output */
  void* dsilu;          /* [T, 4*H*d_h] silu'(z) at the UQKV pre-activation z: the only
                           use the backward makes of z */
  void* uqkv;           /* [T, 4*H*d_h] silu(z) (the attention's tensor-core operands) */
  void* o;              /* [T, H*d_h] attention output before the gate */
  void* y;              /* [T, H*d_h] gate output */
  float* gln_mean;      /* [T] */
  float* gln_rstd;      /* [T] */
  float* ln_mean;       /* [T] */
  float* ln_rstd;       /* [T] */
} mtgr_layer_saved;

typedef struct {        /* fp32, overwritten */
  float* dw_uqkv;       /* [D, 4*H*d_h] */
  float* dw_o;          /* [H*d_h, D] */
  float* dgamma;        /* [4, D] */
  float* dbeta;         /* [4, D] */
} mtgr_layer_grads;

MTGR_API size_t mtgr_layer_workspace_size(int32_t B, int64_t T, int32_t d_model, int32_t n_heads, int32_t d_h,
                                 mtgr_dtype dtype);

/* x, x_out: [T, D] (dtype; may not alias). */
MTGR_API mtgr_status mtgr_hstu_layer_fwd(const mtgr_layer_weights* w, const void* x, void* x_out,
                                const mtgr_layer_saved* saved, const int32_t* offsets, int32_t B,
                                const uint8_t* gid, const int64_t* ts, int64_t T, mtgr_dtype dtype,
                                void* workspace, size_t workspace_bytes, mtgr_stream_t stream);

/* A stack of n_layers layers run forward for ranking (paper-daily deep reading
 * §2: 22 layers at d_model 1024), in one call: layer l reads layer l-1's
 * output; the last layer writes x_out.  w: host array of n_layers weight sets,
 * all with the same d_model, n_heads, d_h.  act: [T, D] scratch (dtype,
 * distinct from x and x_out) when n_layers > 1.  saved: one set of buffers
 * that every layer overwrites (inference keeps nothing between layers); its
 * dsilu is neither written nor required (may be NULL), since nothing runs a
 * backward on it, which saves the UQKV projection a second output.  The
 * attention work lists are built once for all layers (they depend only on the
 * batch).  Workspace: mtgr_layer_workspace_size of one layer.  The call
 * allocates nothing and never synchronises, so it can be captured in a CUDA
 * Graph. */
MTGR_API mtgr_status mtgr_hstu_stack_fwd(const mtgr_layer_weights* w, int32_t n_layers, const void* x, void* x_out,
                                void* act, const mtgr_layer_saved* saved, const int32_t* offsets, int32_t B,
                                const uint8_t* gid, const int64_t* ts, int64_t T, mtgr_dtype dtype,
                                void* workspace, size_t workspace_bytes, mtgr_stream_t stream);

/* Chunked candidate scoring of one ranking request, the history encoded once
 * (paper-daily "MTGR：美团外卖生成式推荐Scaling Law落地实践", inference: the user
 * profile and the thousand behaviour tokens are encoded once and every
 * candidate shares that result; fun-rec chapter 7.3, §7.3.1).  A request is one
 * user: n_hist history rows (User*, Seq*, RealTime*) followed by n_cand
 * candidate rows; gid, ts: device [n_hist + n_cand] for the whole request.
 * Under the dynamic mixed mask a history row sees history rows only and a
 * candidate sees the history and itself, so the history's activations at every
 * layer are those of the whole request, and a chunk of candidates scored
 * against them gives exactly the rows it would get in the whole request.  n_u
 * is the whole request's token count n_hist + n_cand in both calls.
 * cache: device, mtgr_stack_cache_size() bytes, caller-owned: layer l's
 * [U|Q|K|V] (f16, [n_hist + chunk][4*H*d_h]) at byte offset
 * l * (n_hist + chunk) * 4*H*d_h * 2, history rows first, then room for one
 * chunk; after all layers' rows, the f16 copies of every layer's weights that
 * the MTGR_BF16 chunk calls use (made once by the history call).  The weights
 * must not change between the history call and the chunk calls.
 * Workspace: mtgr_stack_chunk_workspace_size().  MTGR_BF16 or MTGR_F16
 * only (16-bit tensor-core path); same error rules as the layer calls.
 *
 * mtgr_hstu_stack_hist_fwd: the n_layers layers on the history rows; x_hist
 *   [n_hist, D] (dtype); act: [2][n_hist, D] scratch (dtype, each half 256-byte
 *   aligned in size).  Fills the history rows of every layer's cache.
 * mtgr_hstu_stack_cand_fwd: the n_layers layers on candidates c0 .. c0+c-1
 *   (c <= chunk): x_cand [c, D] -> x_out [c, D]; act: [c, D] scratch (dtype)
 *   when n_layers > 1; x_cand, x_out, act distinct.  Overwrites the chunk rows
 *   of the cache, so chunks run one after the other on one cache. */
MTGR_API size_t mtgr_stack_cache_size(int32_t n_layers, int32_t n_hist, int32_t chunk, int32_t d_model,
                                      int32_t n_heads, int32_t d_h);
MTGR_API size_t mtgr_stack_chunk_workspace_size(int32_t n_hist, int32_t chunk, int32_t d_model, int32_t n_heads,
                                                int32_t d_h, mtgr_dtype dtype);
MTGR_API mtgr_status mtgr_hstu_stack_hist_fwd(const mtgr_layer_weights* w, int32_t n_layers, const void* x_hist,
                                              void* act, void* cache, int32_t chunk, const uint8_t* gid,
                                              const int64_t* ts, int32_t n_hist, int32_t n_cand, mtgr_dtype dtype,
                                              void* workspace, size_t workspace_bytes, mtgr_stream_t stream);
MTGR_API mtgr_status mtgr_hstu_stack_cand_fwd(const mtgr_layer_weights* w, int32_t n_layers, const void* x_cand,
                                              void* x_out, void* act, void* cache, int32_t chunk, const uint8_t* gid,
                                              const int64_t* ts, int32_t n_hist, int32_t n_cand, int32_t c0,
                                              int32_t c, mtgr_dtype dtype, void* workspace, size_t workspace_bytes,
                                              mtgr_stream_t stream);

/* dx_out: [T, D] upstream gradient; dx: [T, D] (dtype), includes the residual path.
 * MTGR_BF16: the layer runs its products on f16 operands (exact f16 copies of
 * the bf16 weights, f16 activations) and carries its gradients in f16 scaled
 * by a power of two s chosen from max|dx_out| (so that f16's range holds them
 * whatever the loss scale; an all-zero or non-finite dx_out uses s = 1); dx,
 * dw_*, dgamma and dbeta leave scaled back.  The scaling is exact.
 * Workspace: mtgr_layer_workspace_size; with mtgr_attn_ds_store_size more
 * bytes the attention backward keeps its dS tiles (see there). */
MTGR_API mtgr_status mtgr_hstu_layer_bwd(const mtgr_layer_weights* w, const void* x, const mtgr_layer_saved* saved,
                                const void* dx_out, void* dx, const mtgr_layer_grads* grads,
                                const int32_t* offsets, int32_t B, const uint8_t* gid, const int64_t* ts,
                                int64_t T, mtgr_dtype dtype, void* workspace, size_t workspace_bytes,
                                mtgr_stream_t stream);

/* Dense upstream gradient from its nonzero rows.  A loss on the candidate tokens
 * only (fun-rec §7.3.1: every candidate is scored from its own position) makes
 * dx' zero on every other row, so a training step need only move the
 * candidates' rows to the GPU.  dst [T, D] (dtype, device) is zeroed, then
 * dst[rows[k], :] = src[k, :] for k < n; src [n, D] (dtype, device), rows
 * (device int32 [n], distinct); a row outside [0, T) is skipped.  D * element
 * size must be a multiple of 16 bytes; src and dst 16-byte aligned. */
MTGR_API mtgr_status mtgr_expand_rows(const void* src, const int32_t* rows, int64_t n, void* dst, int64_t T,
                                      int32_t D, mtgr_dtype dtype, mtgr_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Training batches (host side: plain host arrays, no device work, no stream). */
/* ------------------------------------------------------------------------- */

/* Stochastic length (paper-daily "MTGR：美团外卖生成式推荐Scaling Law落地实践",
 * "计算量涨了 65 倍…": training shortens long user sequences by sampling a piece
 * of them; scoring keeps the whole sequence).  Reading: per user the User,
 * RealTime and candidate tokens are kept; a Seq run longer than max_seq is cut
 * to the max_seq consecutive Seq tokens starting at Seq position
 * draws[u] mod (n_S - max_seq + 1), so the caller supplies the randomness
 * (one uint64 per user).  offsets (host int32 [B+1], offsets[0] = 0,
 * offsets[B] = T) and gid (host uint8 [T], User*, Seq*, RealTime*, Cand* per
 * segment) describe the batch.  Writes keep (host int32, capacity T: the kept
 * token indices, ascending), new_offsets (host int32 [B+1]) and *new_T.  The
 * caller gathers its per-token arrays with keep.  Returns
 * MTGR_ERR_BAD_OFFSETS / MTGR_ERR_BAD_GROUP_ORDER for bad metadata,
 * MTGR_ERR_INVALID_ARG for bad scalars or NULL pointers; nothing is written
 * then. */
MTGR_API mtgr_status mtgr_stochastic_length(const int32_t* offsets, int32_t B, const uint8_t* gid, int64_t T,
                                            int32_t max_seq, const uint64_t* draws, int32_t* keep,
                                            int32_t* new_offsets, int64_t* new_T);

/* Token-balanced per-GPU batches (zzxanthony.github.io "MTGR：工业级生成式推荐框架",
 * §11.3 "Dynamic batch size 做负载均衡": each GPU's batch size follows the
 * sequence lengths so that every GPU computes about the same, and gradients are
 * weighted by each GPU's batch size).  Reading: users keep their arrival order
 * and are cut into n_ranks contiguous groups whose largest token count is the
 * smallest possible; among such cuts, each rank in turn takes as many users as
 * fit, leaving at least one user for every later rank when B >= n_ranks (with
 * fewer users than ranks the last ranks are empty).  tokens: host int64 [B]
 * (tokens of each user, >= 0).  Writes rank_first (host int32 [n_ranks+1]:
 * rank r owns users rank_first[r] .. rank_first[r+1]-1), rank_tokens (host
 * int64 [n_ranks]) and grad_weight (host double [n_ranks] = users of the rank /
 * B).  MTGR_ERR_INVALID_ARG for bad scalars, negative tokens or NULL pointers. */
MTGR_API mtgr_status mtgr_token_balanced_split(const int64_t* tokens, int32_t B, int32_t n_ranks,
                                               int32_t* rank_first, int64_t* rank_tokens, double* grad_weight);

#ifdef __cplusplus
}
#endif
#endif /* MTGR_H_ */

/*
 * tpffn.h -- C ABI of the GB300 tensor-parallel feed-forward library
 * (libtpffn.so).
 *
 * The operation is the Megatron tensor-parallel FFN sublayer of
 * "7.9 Tensor and pipeline parallelism (TP, PP)" (AI/ML Theory), §2.1
 * "The FFN, sharded":  y = sum_t W2^(t) sigma(W1^(t) x), W1 (and W3 for the
 * SwiGLU form of "S17 Tensor & Pipeline Parallelism", listing "the megatron
 * pattern") split along its output dimension and W2 along its input
 * dimension into T_p shards.  All T_p shards run on the calling GPU as
 * virtual ranks; the g-operator all-reduce of the forward pass and the
 * f-operator all-reduce of dx in the backward pass are on-device sums of the
 * shard partials taken in the fixed order t = 0..T_p-1, so every result is
 * bit-identical from run to run.  The row-parallel attention output
 * projection of §2.2 "Attention, sharded" is the same path with no first
 * matrix (activation TP_ACT_NONE).
 *
 * Conventions
 *   - Row-major storage.  Weights are [out_features][in_features]:
 *     W1, W3: [d_ff][d];  W2: [d][d_ff].  Activations are [n_tokens][features]
 *     (the transpose of the column-vector form on the page, applied to n
 *     tokens): h = sigma(x W1^T), y = h W2^T.
 *   - Element type is the plan's dtype: TP_BF16 (bf16 storage, fp32
 *     accumulation on tcgen05 tensor cores) or TP_F32 (fp32 throughout,
 *     SIMT FMA).  fp32 partial buffers are fp32 in both.
 *   - Every device buffer is owned by the caller; the plan owns host metadata
 *     only.  Calls never allocate device memory.  All work is enqueued on the
 *     given stream and runs asynchronously; pointers must stay valid until it
 *     has finished.
 *   - Device pointers must be 16-byte aligned (TP_ERR_ALIGN otherwise).
 *   - Status codes are returned; nothing is thrown across the ABI.  A
 *     launch failure returns TP_ERR_CUDA.  A device-side bounded wait that
 *     expires is recorded in the workspace's error word and read back by
 *     tp_ffn_last_device_error() (or returned directly under TP_FLAG_SYNC).
 */
#ifndef TPFFN_H
#define TPFFN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TPFFN_API __attribute__((visibility("default")))
#else
#define TPFFN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same object as cudaStream_t); NULL = legacy stream. */
typedef struct CUstream_st* tp_stream_t;

typedef struct tp_ffn_plan tp_ffn_plan;

/* Status codes. */
enum {
  TP_OK = 0,
  TP_ERR_INVALID = 1,      /* bad argument: NULL, shape, divisibility, size */
  TP_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement   */
  TP_ERR_CUDA = 3,         /* a CUDA call or kernel launch failed           */
  TP_ERR_TIMEOUT = 4,      /* a device-side bounded wait expired            */
  TP_ERR_ALIGN = 5         /* pointer not 16-byte aligned                    */
};

/* Activation between the two matrices. */
enum {
  TP_ACT_NONE = 0,       /* no first matrix: row-parallel linear only (W_O) */
  TP_ACT_GELU_TANH = 1,  /* h = gelu_tanh(x W1^T + b1)                      */
  TP_ACT_SWIGLU = 2      /* h = silu(x W1^T) * (x W3^T)                      */
};

/* Storage dtype. */
enum { TP_F32 = 0, TP_BF16 = 1 };

/* Packed weight buffers (tp_ffn_packed_bytes). */
enum { TP_PACK_COLUMNS = 0, TP_PACK_ROWS = 1 };

/* Flags for tp_ffn_fwd / tp_ffn_bwd / tp_ffn_workspace_bytes. */
enum {
  TP_SUM_STANDALONE = 0,  /* shard GEMMs write fp32 partials, then a separate
                             streaming kernel sums them in order t = 0..T_p-1 */
  TP_SUM_FUSED = 1,       /* one GEMM accumulates shard after shard into the
                             same tensor-memory accumulator (K order: shard 0's
                             hidden units first); no partials are written     */
  TP_FLAG_SYNC = 2,       /* synchronize the stream before returning and
                             report device-side errors as the return value   */
  TP_FLAG_TIMING = 4,     /* record CUDA events around every kernel of the
                             call (read with tp_ffn_kernel_times)            */
  TP_SUM_OVERLAP = 8,     /* standalone sum overlapped with compute: the
                             row-sharded GEMM and the shard-sum run in 4 token
                             chunks, the sum of chunk i on a second stream
                             (owned by the plan) while the GEMM of chunk i+1
                             runs on the call's stream; the call's stream waits
                             for the last sum before anything later on it.
                             Results are bit-identical to TP_SUM_STANDALONE.
                             TP_ERR_INVALID together with TP_SUM_FUSED.
                             This puts on the device the "hidden behind
                             compute" argument of "7.9 Tensor and pipeline
                             parallelism (TP, PP)", §2.4-2.5              */
  TP_FLAG_DEBUG_SKIP_LOAD = 1 << 16  /* test hook: the first tensor-core GEMM
                             of the call never issues its first operand load,
                             so its consumer's bounded wait expires and the
                             call reports TP_ERR_TIMEOUT (bf16 plans only)    */
};

/* ---------------------------------------------------------------- plans */

/* Create a plan for an FFN of model width d and hidden width d_ff split into
 * T_p shards of s = d_ff / T_p hidden units ("7.9 Tensor and pipeline
 * parallelism (TP, PP)", §2.1: shard t holds rows [t*s, (t+1)*s) of W1/W3 and
 * the same columns of W2).
 *   act   : TP_ACT_GELU_TANH or TP_ACT_SWIGLU (TP_ACT_NONE: see
 *           tp_attn_out_plan_create; here d_ff is then the input width).
 *   dtype : TP_BF16 or TP_F32.
 * Errors: TP_ERR_INVALID if out is NULL, d < 1, d_ff < 1, T_p < 1,
 * d_ff % T_p != 0, or act/dtype unknown.  TP_ERR_UNSUPPORTED for a bf16 plan
 * whose widths break the 16-byte row rule of the tensor-memory-access unit:
 * d % 8 != 0, or (act NONE) s % 8 != 0.
 * On success *out receives a plan to be released with tp_ffn_plan_destroy. */
TPFFN_API int tp_ffn_plan_create(tp_ffn_plan** out, int64_t d, int64_t d_ff, int T_p, int act, int dtype);

/* Plan for the row-parallel attention output projection ("7.9 Tensor and
 * pipeline parallelism (TP, PP)", §2.2 "Attention, sharded"): shard t owns
 * heads [t*n_heads/T_p, (t+1)*n_heads/T_p) and the matching input columns of
 * W_O [d_model][n_heads*head_dim]; y = sum_t c^(t) W_O^(t)T, with c the
 * concatenated head outputs.  Validates the divisibility rule of
 * "S17 Tensor & Pipeline Parallelism" ("Attention shards by head, and GQA
 * caps the degree"): TP_ERR_INVALID unless n_heads % T_p == 0 and
 * n_kv_heads % T_p == 0.  The resulting plan has act TP_ACT_NONE,
 * d = d_model and d_ff = n_heads * head_dim. */
TPFFN_API int tp_attn_out_plan_create(tp_ffn_plan** out, int64_t d_model, int n_heads, int n_kv_heads,
                            int64_t head_dim, int T_p, int dtype);

/* Release a plan (NULL is a no-op). */
TPFFN_API void tp_ffn_plan_destroy(tp_ffn_plan* plan);

/* Read back a plan's shape.  s = d_ff / T_p; s_pad = hidden units per shard
 * after padding (multiple of 8; multiple of 128 for SwiGLU).  Any output
 * pointer may be NULL.  TP_ERR_INVALID if plan is NULL. */
TPFFN_API int tp_ffn_plan_info(const tp_ffn_plan* plan, int64_t* d, int64_t* d_ff, int* T_p, int* act,
                     int* dtype, int64_t* s, int64_t* s_pad);

/* ------------------------------------------------------------ buffer sizes */

/* Bytes of a packed weight buffer (0 on a NULL plan or unknown `which`).
 *   TP_PACK_COLUMNS : GELU  [T_p][s_pad][d]        shard t row j = W1 row t*s+j
 *                     SwiGLU [T_p][s_pad/128][2][128][d]: block b holds W1 rows
 *                            t*s+128b.. then W3 rows t*s+128b.. (interleaved so
 *                            one 256-row tile yields matching a and g columns)
 *                     NONE  0 (no first matrix)
 *   TP_PACK_ROWS    : [T_p][d][s_pad]  element (t,c,j) = W2[c][t*s+j]
 * Rows j >= s of a shard are zero. */
TPFFN_API size_t tp_ffn_packed_bytes(const tp_ffn_plan* plan, int which);

/* Bytes of the activations the forward pass saves for the backward pass, for
 * n_tokens tokens (0 for act NONE):
 *   GELU  : z [T_p][n][s_pad], then h [T_p][n][s_pad]
 *   SwiGLU: ag [T_p][n][2*s_pad] (a and g interleaved in 128-column blocks,
 *           like TP_PACK_COLUMNS), then h [T_p][n][s_pad]
 * each region starting on a 256-byte boundary, elements of the plan dtype. */
TPFFN_API size_t tp_ffn_saved_bytes(const tp_ffn_plan* plan, int64_t n_tokens);

/* Bytes of scratch that one tp_ffn_fwd or tp_ffn_bwd call with these flags
 * needs for n_tokens tokens (one buffer of this size serves both).  It holds
 * the device error word (first 4 bytes), the hidden activations when nothing
 * is saved, the fp32 shard partials of the standalone sum, the backward's
 * hidden gradients, the fp32 K parts of split GEMMs (decode-sized SwiGLU up
 * GEMMs; weight-gradient GEMMs of problems with few output tiles; the last
 * wave of a forward GEMM (up, or fused-sum down), one 256 x 256 fp32 block
 * per SM pair --
 * sized from the current device's SM count) and the bias-gradient reduction
 * scratch.  Query it on the device that will run the calls. */
TPFFN_API size_t tp_ffn_workspace_bytes(const tp_ffn_plan* plan, int64_t n_tokens, int flags);

/* ---------------------------------------------------------------- packing */

/* shard_columns for all T_p shards at once ("S17 Tensor & Pipeline
 * Parallelism", listing "the megatron pattern": W1 and W3 keep d_ff/world of
 * their output rows per rank).  W1, W3: [d_ff][d] device, plan dtype (W3
 * required for SwiGLU, ignored otherwise).  packed: TP_PACK_COLUMNS bytes.
 * TP_ERR_INVALID for act NONE or NULL pointers. */
TPFFN_API int tp_ffn_shard_columns(const tp_ffn_plan* plan, const void* W1, const void* W3, void* packed,
                         tp_stream_t stream);

/* shard_rows for all T_p shards: W2 [d][d_ff] device -> TP_PACK_ROWS layout
 * (each shard's d_ff/T_p input columns made contiguous). */
TPFFN_API int tp_ffn_shard_rows(const tp_ffn_plan* plan, const void* W2, void* packed, tp_stream_t stream);

/* Inverses of the two packers (for weight gradients, which the backward pass
 * returns in packed layout).  Padding rows are dropped. */
TPFFN_API int tp_ffn_unshard_columns(const tp_ffn_plan* plan, const void* packed, void* W1, void* W3,
                           tp_stream_t stream);
TPFFN_API int tp_ffn_unshard_rows(const tp_ffn_plan* plan, const void* packed, void* W2, tp_stream_t stream);

/* ----------------------------------------------------------------- forward */

/* Forward pass of all T_p shards and the g-operator shard-sum.
 *   x        : [n][d] (act NONE: [n][d_ff], the concatenated head outputs)
 *   w13p     : TP_PACK_COLUMNS buffer (NULL for act NONE)
 *   w2p      : TP_PACK_ROWS buffer
 *   b1       : [d_ff] or NULL (GELU only; TP_ERR_UNSUPPORTED otherwise)
 *   b2       : [d] or NULL, added once after the shard-sum
 *   y        : [n][d] output, plan dtype
 *   partials : [T_p][n][d] fp32 or NULL.  If given, the shard partials
 *              y^(t) = h^(t) W2^(t)T are written there (standalone sum only;
 *              TP_ERR_INVALID together with TP_SUM_FUSED)
 *   saved    : tp_ffn_saved_bytes buffer for a later tp_ffn_bwd, or NULL for
 *              inference
 *   workspace: tp_ffn_workspace_bytes(plan, n, flags) bytes (>= that many,
 *              given in workspace_bytes; TP_ERR_INVALID if smaller)
 * n == 0 returns TP_OK without enqueueing work. */
TPFFN_API int tp_ffn_fwd(const tp_ffn_plan* plan, int64_t n_tokens, const void* x, const void* w13p,
               const void* w2p, const void* b1, const void* b2, void* y, float* partials,
               void* saved, void* workspace, size_t workspace_bytes, int flags, tp_stream_t stream);

/* ---------------------------------------------------------------- backward */

/* Backward pass: the g operator is the identity here, each shard computes its
 * own hidden gradient and weight gradients (no cross-shard sum: every shard
 * owns its weights), and the f operator sums the dx partials in order
 * t = 0..T_p-1.
 *   x, w13p, w2p : as given to tp_ffn_fwd;  saved: filled by tp_ffn_fwd
 *   dy       : [n][d] upstream gradient
 *   dx       : [n][d] (act NONE: [n][d_ff]; shard t writes its own head
 *              columns and no sum is taken)
 *   dx_partials : [T_p][n][d] fp32 or NULL (standalone only, not for NONE)
 *   dw13p    : TP_PACK_COLUMNS-layout gradient of W1/W3 (NULL for NONE)
 *   dw2p     : TP_PACK_ROWS-layout gradient of W2
 *   db1      : [d_ff] or NULL (GELU only);  db2: [d] or NULL
 * Gradients are written (not accumulated), in the plan dtype. */
TPFFN_API int tp_ffn_bwd(const tp_ffn_plan* plan, int64_t n_tokens, const void* x, const void* w13p,
               const void* w2p, const void* saved, const void* dy, void* dx, float* dx_partials,
               void* dw13p, void* dw2p, void* db1, void* db2, void* workspace,
               size_t workspace_bytes, int flags, tp_stream_t stream);

/* ------------------------------------------------------- sequence parallel */

/* Sequence-parallel forms ("7.9 Tensor and pipeline parallelism (TP, PP)",
 * §2.5 "Sequence parallelism"; "Parallelism II: model", "Sequence and context
 * parallelism"): outside the tensor-parallel region each of the T_p virtual
 * ranks holds the token slice [t*n/T_p, (t+1)*n/T_p) of the activations, and
 * the all-reduce becomes an all-gather before the column-sharded GEMM plus a
 * reduce-scatter after the row-sharded GEMM (the same bytes).
 *   x_slices, y_slices, dy_slices, dx_slices: host arrays of T_p device
 *   pointers, slice t = [n/T_p][features] (features: d, or d_ff for act NONE
 *   inputs and dx).  TP_ERR_INVALID unless n % T_p == 0 and T_p <= 64.
 * The forward gathers x, runs tp_ffn_fwd's path and writes row-slice t of
 * y = sum_t y^(t) (+ b2) into y_slices[t]: with TP_SUM_STANDALONE the ordered
 * shard-sum itself writes each slice (reduce-scatter); with TP_SUM_FUSED the
 * fused GEMM's result is scattered.  The backward gathers x and dy and
 * reduce-scatters dx the same way; weight and bias gradients are as in
 * tp_ffn_bwd.  Results are bit-identical to tp_ffn_fwd / tp_ffn_bwd on the
 * concatenated tensors.  TP_SUM_OVERLAP is not supported (TP_ERR_INVALID).
 * workspace: tp_ffn_seq_parallel_workspace_bytes(plan, n, flags) bytes. */
TPFFN_API size_t tp_ffn_seq_parallel_workspace_bytes(const tp_ffn_plan* plan, int64_t n_tokens, int flags);
TPFFN_API int tp_ffn_fwd_seq_parallel(const tp_ffn_plan* plan, int64_t n_tokens, const void* const* x_slices,
                                      const void* w13p, const void* w2p, const void* b1, const void* b2,
                                      void* const* y_slices, void* saved, void* workspace, size_t workspace_bytes,
                                      int flags, tp_stream_t stream);
TPFFN_API int tp_ffn_bwd_seq_parallel(const tp_ffn_plan* plan, int64_t n_tokens, const void* const* x_slices,
                                      const void* w13p, const void* w2p, const void* saved,
                                      const void* const* dy_slices, void* const* dx_slices, void* dw13p,
                                      void* dw2p, void* db1, void* db2, void* workspace, size_t workspace_bytes,
                                      int flags, tp_stream_t stream);

/* ------------------------------------------------------- attention sublayer
 *
 * The whole head-sharded self-attention sublayer of "7.9 Tensor and pipeline
 * parallelism (TP, PP)", §2.2 "Attention, sharded": shard t owns the query
 * heads [t*H/T_p, (t+1)*H/T_p) and the key/value heads [t*Hkv/T_p, ...) (the
 * divisibility rule of "S17 Tensor & Pipeline Parallelism", "Attention shards
 * by head, and GQA caps the degree"; query head h reads key/value head
 * h / (H/Hkv)).  Per shard: column-sharded projections q, k, v = x W^(t)T,
 * scaled dot-product attention of each of its heads (s = q k^T / sqrt(hd),
 * optional causal mask, softmax, o = p v), and the row-sharded output
 * projection y^(t) = c^(t) W_O^(t)T of its head outputs c^(t); y is the sum
 * of the T_p shards in the order t = 0..T_p-1 (the g operator).  Backward: dc
 * per shard (no sum), the attention gradients, dx = sum_t of the shards'
 * q/k/v input gradients in the order t = 0..T_p-1 (the f operator), and the
 * weight gradients of every shard.
 *
 * Tokens: B sequences of S tokens, sequence b in rows b*S .. b*S+S-1 of every
 * [B*S][...] buffer.  All buffers bf16 row-major unless stated; every pointer
 * 16-byte aligned (TP_ERR_ALIGN otherwise).
 *
 * Packed projection weights ("wqkv", [T_p * slice][d]): shard t's slice of
 * slice = (H + 2*Hkv)/T_p * hd rows is [Wq rows of its query heads | Wk rows
 * of its key heads | Wv rows of its value heads].  The packed q/k/v buffer
 * ("qkv", [B*S][T_p * slice]) has the same column order: it is x wqkv^T.
 * The packed output projection is the W_O packing of tp_attn_out_plan_create.
 */
typedef struct tp_attn_plan tp_attn_plan;

/* d_model: model width (multiple of 8); head_dim: 128 only (the tensor-core
 * kernels' tile); causal: 1 for the decoder mask (key j visible to query i
 * iff j <= i), 0 for none; dtype: TP_BF16 only.
 * Errors: TP_ERR_INVALID for NULL out, non-positive sizes, or when T_p does
 * not divide n_heads and n_kv_heads or n_kv_heads does not divide n_heads;
 * TP_ERR_UNSUPPORTED for head_dim != 128, d_model % 8 != 0 or TP_F32. */
TPFFN_API int tp_attn_plan_create(tp_attn_plan** out, int64_t d_model, int n_heads, int n_kv_heads,
                                  int64_t head_dim, int T_p, int causal, int dtype);
TPFFN_API void tp_attn_plan_destroy(tp_attn_plan* plan);
/* qkv_width = T_p * slice; slice, and its query / key widths sq = H/T_p*hd,
 * sk = Hkv/T_p*hd (any pointer may be NULL). */
TPFFN_API int tp_attn_plan_info(const tp_attn_plan* plan, int64_t* qkv_width, int64_t* slice, int64_t* sq,
                                int64_t* sk);

/* TP_PACK_COLUMNS: bytes of wqkv; TP_PACK_ROWS: bytes of the packed W_O. */
TPFFN_API size_t tp_attn_packed_bytes(const tp_attn_plan* plan, int which);
/* Wq [H*hd][d], Wk, Wv [Hkv*hd][d], Wo [d][H*hd] (row-major [out][in]) into
 * the packed forms, and back. */
TPFFN_API int tp_attn_shard_weights(const tp_attn_plan* plan, const void* Wq, const void* Wk, const void* Wv,
                                    const void* Wo, void* wqkv, void* wo_packed, tp_stream_t stream);
TPFFN_API int tp_attn_unshard_weights(const tp_attn_plan* plan, const void* wqkv, const void* wo_packed, void* Wq,
                                      void* Wk, void* Wv, void* Wo, tp_stream_t stream);

/* Activations the forward saves for the backward, in one buffer of
 * tp_attn_saved_bytes(plan, B, S) bytes: qkv [B*S][qkv_width] at *qkv_off,
 * the head outputs c [B*S][H*hd] at *c_off, and the log-sum-exp of every
 * softmax row, fp32 [B*H][S_pad] with S_pad = S rounded up to 128, in the
 * base-2 domain (log2 of sum_j 2^(s_ij log2 e)), at *lse_off. */
TPFFN_API size_t tp_attn_saved_bytes(const tp_attn_plan* plan, int64_t B, int64_t S);
TPFFN_API int tp_attn_saved_offsets(const tp_attn_plan* plan, int64_t B, int64_t S, size_t* qkv_off,
                                    size_t* c_off, size_t* lse_off);
/* Workspace of every tp_attn_* pass for this shape and these flags. */
TPFFN_API size_t tp_attn_workspace_bytes(const tp_attn_plan* plan, int64_t B, int64_t S, int flags);

/* Forward: y [B*S][d] from x [B*S][d]; fills `saved`.  Flags as tp_ffn_fwd
 * (TP_SUM_* choose how the output projection sums its shards).
 * Launches: q/k/v GEMM, attention kernel, output-projection GEMM (+ sum). */
TPFFN_API int tp_attn_fwd(const tp_attn_plan* plan, int64_t B, int64_t S, const void* x, const void* wqkv,
                          const void* wo_packed, void* y, void* saved, void* workspace, size_t workspace_bytes,
                          int flags, tp_stream_t stream);
/* Backward from dy [B*S][d]: dx [B*S][d]; dwqkv (packed like wqkv) and
 * dwo_packed (packed like W_O) are overwritten with this call's gradients. */
TPFFN_API int tp_attn_bwd(const tp_attn_plan* plan, int64_t B, int64_t S, const void* x, const void* wqkv,
                          const void* wo_packed, const void* saved, const void* dy, void* dx, void* dwqkv,
                          void* dwo_packed, void* workspace, size_t workspace_bytes, int flags, tp_stream_t stream);

/* The attention core alone, on a caller's packed qkv [B*S][qkv_width]:
 * o [B*S][H*hd] (head h in columns [h*hd, (h+1)*hd)) and lse as in `saved`.
 * Backward: dqkv [B*S][qkv_width] (packed like qkv) from dO [B*S][H*hd],
 * given the forward's o and lse.  workspace: tp_attn_workspace_bytes. */
TPFFN_API int tp_attn_core_fwd(const tp_attn_plan* plan, int64_t B, int64_t S, const void* qkv, void* o,
                               float* lse, void* workspace, size_t workspace_bytes, int flags, tp_stream_t stream);
TPFFN_API int tp_attn_core_bwd(const tp_attn_plan* plan, int64_t B, int64_t S, const void* qkv, const void* o,
                               const float* lse, const void* dO, void* dqkv, void* workspace,
                               size_t workspace_bytes, int flags, tp_stream_t stream);

/* Diagnostics of attention calls, as their tp_ffn_* counterparts. */
TPFFN_API int tp_attn_kernel_times(const tp_attn_plan* plan, int max, const char** names, float* ms);
TPFFN_API int tp_attn_last_launch_count(const tp_attn_plan* plan);

/* ------------------------------------------------ forward without allocation */

/* Size of the library's static scratch array (32 MiB).  A GPU holds this
 * much device memory from the moment the library's static-scratch module is
 * loaded on it until the process exits (see "Set-up" below). */
#define TPFFN_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

/* Forward pass for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point: it exists for callers
 * that must not call cudaMalloc, or any allocator, when they run the layer.
 * Examples are a serving engine that reserves all of its device memory at
 * start-up and forbids allocation while it handles requests, a plugin whose
 * host framework owns the allocator, or a loop whose latency budget leaves
 * no room for an allocation that might block.
 *
 * It computes what tp_ffn_fwd computes with TP_SUM_STANDALONE, saved = NULL
 * and partials = NULL, with the same kernels, so its y is bit-identical to
 * that call's.  The caller still passes the inputs (x, w13p, w2p, b1, b2)
 * and the output y, with the meanings and layouts of tp_ffn_fwd.  The
 * scratch (error word, hidden activations, fp32 shard partials, the decode
 * K-split parts) lives in one file-scope device array of
 * TPFFN_STATIC_SCRATCH_BYTES.  This call allocates nothing: no cudaMalloc,
 * no cudaFree, no allocating library call.
 *   - Limit: returns TP_ERR_UNSUPPORTED, without enqueueing work, when
 *     tp_ffn_workspace_bytes(plan, n_tokens, TP_SUM_STANDALONE) exceeds
 *     TPFFN_STATIC_SCRATCH_BYTES (for example above 76 tokens for the
 *     Llama-3-70B-shaped decode FFN: d 8192, d_ff 28672, T_p 8, SwiGLU).
 *   - Set-up: every call looks up the array's device address
 *     (cudaGetSymbolAddress, on the current device).  Under CUDA's lazy
 *     module loading, the runtime's default, the first look-up on a device
 *     loads the module that holds the array, and the device reserves
 *     TPFFN_STATIC_SCRATCH_BYTES then.  A call with n_tokens = 0 does only
 *     that set-up (x, w13p, w2p, b1, b2, y and stream are not read) and
 *     returns TP_OK: make it once per device, with that device current,
 *     during start-up -- before the caller reserves its device memory and
 *     before any stream capture.  Likewise, kernels of the library that
 *     have not run yet on a device are loaded on their first launch; one
 *     ordinary call at start-up (tp_ffn_fwd, or this one) loads them.
 *   - Sharing: every call, on any stream, uses the same array, which keeps
 *     the previous call's contents; the call clears the error word it needs
 *     zeroed, and overwrites the rest.  Calls that overlap on the GPU (for
 *     example on two streams) race on the array: serialise them.
 *   - Errors: argument and launch errors as in tp_ffn_fwd; TP_ERR_CUDA when
 *     the address look-up fails.  The device error word sits inside the
 *     array and is not exposed, so a device-side timeout is not reported by
 *     this entry point. */
TPFFN_API int tp_ffn_fwd_static_scratch(const tp_ffn_plan* plan, int64_t n_tokens, const void* x,
                                        const void* w13p, const void* w2p, const void* b1, const void* b2,
                                        void* y, tp_stream_t stream);

/* ------------------------------------------------------------- diagnostics */

/* Wait for the stream, then read the error word a previous call left in this
 * workspace: TP_OK, TP_ERR_TIMEOUT (a bounded device wait expired) or
 * TP_ERR_CUDA (the stream reported an error). */
TPFFN_API int tp_ffn_last_device_error(const tp_ffn_plan* plan, const void* workspace, tp_stream_t stream);

/* Human-readable name of a status code (static storage). */
TPFFN_API const char* tp_ffn_status_string(int status);

/* Calls made with TP_FLAG_TIMING append one (kernel name, start, stop) event
 * record per launch to the plan.  This waits for the recorded events, copies
 * up to `max` (name, elapsed milliseconds) pairs in launch order, and clears
 * the list.  Returns the number of launches recorded since the last read
 * (may exceed max), or -1 on a NULL plan.  names point to static strings. */
TPFFN_API int tp_ffn_kernel_times(const tp_ffn_plan* plan, int max, const char** names, float* ms);

/* Number of kernel launches the most recent fwd/bwd call on this plan
 * enqueued (-1 on a NULL plan). */
TPFFN_API int tp_ffn_last_launch_count(const tp_ffn_plan* plan);

#ifdef __cplusplus
}
#endif
#endif /* TPFFN_H */

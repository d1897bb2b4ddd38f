/*
 * tt_ops.h -- op-level C ABI: the individual kernels tt_gpt2_step is built
 * from, callable on their own (tests check each one against a CPU reference;
 * small programs can build their own training steps from them).
 *
 * Every call enqueues on the context's stream and takes device pointers.
 * `dtype` selects the storage type of activations and weights: TT_FP32 (all
 * fp32) or TT_BF16 (bf16 storage, fp32 arithmetic).  Parameter gradients,
 * LayerNorm statistics, log-sum-exp values and losses are always fp32.
 * Scratch memory, where a call needs it, is bump-allocated from the context's
 * arena (reset the arena between calls to reclaim it); TT_ERR_ARENA_OOM if
 * it does not fit.  All matrices are row-major and contiguous.
 */
#ifndef TT_OPS_H
#define TT_OPS_H

#include "tt.h"

#ifdef __cplusplus
extern "C" {
#endif

/* GEMM engine selection: 0 = automatic (tcgen05 tensor cores whenever the
 * operands allow: bf16, 16-byte aligned rows; else SIMT, and the two-CTA
 * pair form wherever the M-tile count allows), 1 = SIMT only, 2 = tensor
 * cores with one CTA per 128-row tile (no pair form).  Returns TT_ERR_ARG
 * for any other value. */
tt_status tt_ctx_set_gemm_backend(tt_ctx* ctx, int backend);

/* Limit of every bounded device-side wait of the tensor-core kernels
 * launched through this context, in SM clock cycles (clock64).  cycles <= 0
 * restores the default, 4e9 cycles (about 2 s).  A wait that runs out sets
 * the context's timeout flag and a code naming the wait; the kernel lets its
 * copies and MMAs already issued finish, frees its tensor memory and returns;
 * every kernel that sees the flag gives up at its next wait; and the next
 * call that synchronises (tt_ctx_sync, a step with a loss pointer) returns
 * TT_ERR_TIMEOUT with the code in tt_last_error.  tt_ctx_reset clears the
 * flag; the context is usable again.  Below 1e6 cycles the waits look at
 * the clock on every poll, so a wait that is not complete within a few
 * hundred cycles of its start runs out (the form used to exercise the
 * timeout path).  The pages' boundary reports failure by status codes
 * (microcrad page, 反向传播); this is how a device-side wait reports one. */
tt_status tt_ctx_set_wait_limit(tt_ctx* ctx, long long cycles);

/* Linear layer forward (tinytorch 三.3 MatMul with the [out, in] weight
 * layout of 八.5):  u = x W^T + b;  y = gelu(u) if gelu (tanh form, tinytorch
 * 三.4) else u;  y += residual if residual != NULL.
 *   x [M,K], W [N,K], b [N] or NULL, residual [M,N] or NULL, y [M,N];
 *   pre [M,N]: receives u when gelu != 0 (required then), else ignored. */
tt_status tt_op_linear_fwd(tt_ctx* ctx, tt_dtype dtype, const void* x, const void* W,
                           const void* b, const void* residual, void* y, void* pre,
                           int M, int K, int N, int gelu);

/* Input gradient of a linear layer (tinytorch 三.3: dA = dC B^T):
 *   dx = dy W, times gelu'(pre) elementwise if pre != NULL (the gradient is
 *   then taken through the GELU that produced this layer's input from pre);
 *   accumulate != 0 adds into dx instead of overwriting.
 *   dy [M,N], W [N,K], pre [M,K] or NULL, dx [M,K]. */
tt_status tt_op_linear_bwd_dx(tt_ctx* ctx, tt_dtype dtype, const void* dy, const void* W,
                              const void* pre, void* dx, int M, int K, int N, int accumulate);

/* Weight and bias gradients (tinytorch 三.3: dB = A^T dC), fp32, overwritten:
 *   dW[N,K] = dy^T x,  db[N] = column sums of dy (db may be NULL).
 *   Deterministic: fixed split of the token dimension and fixed-order sums. */
tt_status tt_op_linear_bwd_dw(tt_ctx* ctx, tt_dtype dtype, const void* dy, const void* x,
                              float* dW, float* db, int M, int K, int N);

/* Causal self-attention forward (Forge page, 最硬的一关: scores scaled by
 * 1/sqrt(d_k), future masked with -inf).  qkv [B*T, 3C] with columns
 * [q | k | v] each [H, C/H]; y [B*T, C]; lse [B, H, T] fp32 receives the
 * log-sum-exp of each score row (saved for the backward). */
tt_status tt_op_attention_fwd(tt_ctx* ctx, tt_dtype dtype, const void* qkv, void* y,
                              float* lse, int B, int T, int C, int H);

/* Attention backward: dqkv [B*T, 3C] is overwritten.  Needs the forward's
 * y and lse; probabilities are recomputed, no T x T matrix is stored. */
tt_status tt_op_attention_bwd(tt_ctx* ctx, tt_dtype dtype, const void* qkv, const void* y,
                              const float* lse, const void* dy, void* dqkv,
                              int B, int T, int C, int H);

/* LayerNorm forward over the last dimension (biased variance, eps = 1e-5):
 *   y = (x - mean) * rstd * w + b;  mean, rstd [M] fp32. */
tt_status tt_op_layernorm_fwd(tt_ctx* ctx, tt_dtype dtype, const void* x, const void* w,
                              const void* b, void* y, float* mean, float* rstd, int M, int C);

/* LayerNorm backward: dx (+)= rstd (g - mean(g) - xhat mean(g xhat)), g = dy w;
 * dw = sum_rows dy xhat, db = sum_rows dy (fp32, overwritten, deterministic). */
tt_status tt_op_layernorm_bwd(tt_ctx* ctx, tt_dtype dtype, const void* x, const void* w,
                              const float* mean, const float* rstd, const void* dy, void* dx,
                              float* dw, float* db, int M, int C, int accumulate);

/* Fused log-softmax cross entropy, forward and backward in one pass over the
 * logits (tinytorch 三.5, Forge 核心组件清单).  logits [M, ld] (ld >= V; the
 * columns V..ld-1 are padding and are masked out) are REPLACED by
 *   dlogits = (softmax(z) - onehot(target)) * dscale      (pad columns: 0)
 * row_loss [M] receives log-sum-exp - z[target]; mean_loss[0] receives the
 * mean over the M rows (deterministic fixed-order sum).  dscale is usually 1/M. */
tt_status tt_op_xent(tt_ctx* ctx, tt_dtype dtype, void* logits, const int32_t* targets,
                     float* row_loss, float* mean_loss, int M, int V, int ld, float dscale);

/* Token + position embedding: x[b*T+t] = wte[tokens[b*T+t]] + wpe[t]. */
tt_status tt_op_embed_fwd(tt_ctx* ctx, tt_dtype dtype, const void* wte, const void* wpe,
                          const int32_t* tokens, void* x, int B, int T, int C, int V);

/* Embedding backward, deterministic (no floating-point atomics):
 *   dwte[v] += sum of dx rows whose token is v, in increasing position order
 *   (dwte is ACCUMULATED into, so that a tied LM-head gradient written first
 *   is kept); dwpe[t] = sum_b dx[b*T+t] for t < T and 0 for T <= t < maxT. */
tt_status tt_op_embed_bwd(tt_ctx* ctx, tt_dtype dtype, const void* dx, const int32_t* tokens,
                          float* dwte, float* dwpe, int B, int T, int C, int V, int maxT);

/* ------------------------------------------------------ allocation-free call
 * The pages have no counterpart to this entry point.  It serves callers of
 * this library that cannot allocate device memory: a program whose GPU memory
 * is owned by another allocator (for example a framework's caching allocator
 * or a server that budgets all memory when it starts) must not have a library
 * call cudaMalloc behind its back, and such a caller cannot create a tt_ctx
 * either, because a context's arena is one cudaMalloc.
 *
 * tt_linear_bwd_dw_noalloc computes the same weight and bias gradients as
 * tt_op_linear_bwd_dw in bf16 mode (tensor cores, deterministic split-K):
 *   dW[N,K] = dy^T x (fp32, overwritten),  db[N] = column sums of dy (fp32,
 *   overwritten; db may be NULL),  dy [M,N] and x [M,K] bf16 row-major,
 *   16-byte aligned, N and K multiples of 8.
 * It takes a stream (a cudaStream_t; NULL = legacy default stream) instead
 * of a context and allocates nothing -- no cudaMalloc, no cudaFree, no
 * allocating library routine.  Its scratch is one fixed array of
 * TT_NOALLOC_SCRATCH_BYTES (32 MiB + 256 B) of device memory inside this
 * library, held by every GPU that loads the library until the process exits:
 * 256 B of device flags, TT_NOALLOC_SPLIT_FLOATS floats of split-K partial
 * sums (always enough on GPUs with up to 192 SMs) and TT_NOALLOC_BIAS_FLOATS
 * floats of bias partial sums.
 * Returns TT_ERR_ARG for a NULL pointer, a non-positive size, operands the
 * tensor-core path cannot take, or when db != NULL and the bias partial sums,
 * ceil(M / 256) * N floats, exceed TT_NOALLOC_BIAS_FLOATS (for M = 32768 that
 * allows N <= 16384); TT_ERR_CUDA if a CUDA call fails.  It returns before the
 * GPU finishes; a device-side wait that times out leaves dW undefined and is
 * not reported by this call.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, once per device, with that device current); make
 * that first call before any stream capture begins.  Every call shares the
 * one array and it keeps the last call's contents: nothing in it needs to
 * start at zero except the flags, which each call clears on its stream, since
 * every scratch element a call reads is written earlier in that call.  Calls
 * that overlap on the GPU (on different streams, or from threads without
 * ordering between them) race on the array: issue them on one stream. */
#define TT_NOALLOC_SPLIT_FLOATS 6291456u
#define TT_NOALLOC_BIAS_FLOATS 2097152u
#define TT_NOALLOC_SCRATCH_BYTES (256u + 4u * (TT_NOALLOC_SPLIT_FLOATS + TT_NOALLOC_BIAS_FLOATS))
tt_status tt_linear_bwd_dw_noalloc(void* stream, const void* dy, const void* x, float* dW,
                                   float* db, int M, int K, int N);

#ifdef __cplusplus
}
#endif
#endif /* TT_OPS_H */

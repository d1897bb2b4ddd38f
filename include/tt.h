/*
 * tt.h -- C ABI of the arena-allocated autograd GPT-2 training step (sm_103a).
 *
 * One context owns one device arena (a single cudaMalloc) and one host-side
 * tape.  A training step is: tt_ctx_reset, tt_gpt2_step (forward, then the
 * tape replayed backwards), tt_adamw.  Every activation, saved tensor and
 * activation gradient of the step is bump-allocated from the arena; the
 * caller owns the parameters, gradients, optimizer moments and token buffers.
 *
 * Pages the calls follow (cited by title and section):
 *  - "不用PyTorch，一个头文件就能训练GPT-2：Arena内存池+自动微分的C++实现"
 *    (tinytorch): 三.1 the arena (TensorContext with a bump offset and
 *    Reset()), 三.3 forward records op and inputs / backward walks back,
 *    三.6 the GPT-2 model, 三.7 the loop (ZeroGrad, Backward, Adam with
 *    bias correction and step+1).
 *  - "17岁少年用C++从零构建深度学习框架Forge，精确复现GPT-2": 核心组件清单
 *    (AdamW with decoupled weight decay, fused log-softmax cross entropy).
 *  - "microcrad": 反向传播 (backward returns 0 on success and -1 on failure),
 *    内存管理 (release is NULL-safe), 关于 magic 字段的说明 (a magic number
 *    guards against stale handles).
 *
 * Conventions for every call:
 *  - Status: 0 (TT_OK) on success, a negative tt_status on failure; the
 *    message of the last failure is kept in the context (tt_last_error).
 *  - Pointers marked "device" must be device memory of the current CUDA
 *    device (for example torch tensors); "host" pointers are host memory.
 *  - Work is enqueued on the context's stream (tt_ctx_set_stream; default:
 *    the legacy default stream).  Calls return before the GPU finishes unless
 *    stated otherwise.
 *  - All sizes are in elements unless the name says bytes.
 */
#ifndef TT_H
#define TT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TT_OK = 0,
    TT_ERR = -1,            /* generic failure (the microcrad convention) */
    TT_ERR_ARG = -2,        /* bad argument: NULL pointer, size, shape, token id */
    TT_ERR_ARENA_OOM = -3,  /* the step's exact arena plan exceeds the arena; nothing was launched */
    TT_ERR_CUDA = -4,       /* a CUDA runtime call failed (message in tt_last_error) */
    TT_ERR_TIMEOUT = -5,    /* a bounded device-side wait gave up; results are undefined */
    TT_ERR_NONFINITE = -6,  /* the loss is NaN or Inf */
    TT_ERR_STALE = -7,      /* the handle is not a live context (magic check) */
    TT_ERR_STATE = -8       /* call out of order (e.g. a step before tt_ctx_set_model) */
} tt_status;

typedef enum { TT_FP32 = 0, TT_BF16 = 1, TT_FP16 = 2 } tt_dtype;

/* GPT-2 architecture.  V is the real vocabulary; the device pads the LM-head
 * width internally to a multiple of 128 (50257 -> 50304), the pad logits
 * being masked to -inf.  Requirements: C % H == 0, C % 64 == 0, C <= 1024,
 * maxT >= 1.  dtype TT_FP32: every tensor fp32; TT_BF16: bf16 weights,
 * activations and activation gradients with fp32 accumulation, fp32 LayerNorm
 * statistics, softmax, loss and parameter gradients (needs C / H == 64).
 * TT_FP16: the same split with IEEE half storage (the mixed precision of the
 * dl-scratch page, 3.4): a 10-bit mantissa but a 5-bit exponent, so small
 * activation gradients underflow unless the loss is scaled
 * (tt_gpt2_step_ex's loss_scale).  The half step runs on the SIMT kernels
 * (the tensor-core kernels are bf16).  tt_gpt2_eval takes it too; the
 * op-level calls and tt_gpt2_generate take TT_FP32 and TT_BF16 only. */
typedef struct {
    int L, C, H, V, maxT;
    tt_dtype dtype;
} tt_gpt2_config;

typedef struct tt_ctx tt_ctx;

/* ---------------------------------------------------------------- context */

/* Create a context whose arena holds arena_bytes of device memory (one
 * cudaMalloc on the current device).  *out receives the handle.  Returns
 * TT_ERR_ARG for out == NULL or arena_bytes == 0, TT_ERR_CUDA if the
 * allocation fails.  (tinytorch 三.1: TensorContext(arena_size).) */
tt_status tt_ctx_create(size_t arena_bytes, tt_ctx** out);

/* Free the arena.  NULL-safe; a stale handle is ignored.  The small host-side
 * handle is kept with its magic number poisoned, so that any later call
 * through it returns TT_ERR_STALE instead of touching freed memory. */
void tt_ctx_destroy(tt_ctx* ctx);

/* Enqueue all further work on `stream` (a cudaStream_t, e.g.
 * torch.cuda.current_stream().cuda_stream; NULL = legacy default stream). */
tt_status tt_ctx_set_stream(tt_ctx* ctx, void* stream);

/* Fix the model this context trains.  Validates the config (TT_ERR_ARG). */
tt_status tt_ctx_set_model(tt_ctx* ctx, const tt_gpt2_config* cfg);

/* Rewind the arena offset to 0 and clear the tape: every arena tensor of the
 * previous step becomes invalid (tinytorch 三.1 Reset()).  Also clears the
 * device error flags.  Call it before each step. */
tt_status tt_ctx_reset(tt_ctx* ctx);

/* Wait for the context's stream, then read the device error flags of the
 * work enqueued since the last reset: TT_ERR_ARG (a token id out of range),
 * TT_ERR_TIMEOUT (a bounded wait gave up), TT_ERR_NONFINITE (loss), else TT_OK. */
tt_status tt_ctx_sync(tt_ctx* ctx);

size_t tt_ctx_arena_capacity(const tt_ctx* ctx);   /* bytes; 0 for a bad handle */
size_t tt_ctx_arena_used(const tt_ctx* ctx);       /* bytes in use since the last reset */
size_t tt_ctx_arena_high_water(const tt_ctx* ctx); /* largest use since creation */

/* Number of kernels this context has launched since creation (for launch
 * accounting; library copies and memsets are not counted). */
uint64_t tt_ctx_launch_count(const tt_ctx* ctx);

/* Per-op timing (tracing).  While on, every kernel group the context launches
 * is bracketed by CUDA events on the context's stream and tagged with its op
 * kind and its algorithmic FLOPs and bytes (the method's own work: each
 * operand read once, each result written once).  tt_ctx_profile_read
 * synchronizes the stream and returns one row per op kind seen since
 * profiling was switched on (at most max_rows), then clears the records. */
typedef struct {
    char name[24];      /* op kind, e.g. "gemm_fwd", "attn_bwd", "xent" */
    uint64_t calls;     /* bracketed groups */
    double ms;          /* summed device time */
    double flops;       /* summed algorithmic FLOPs */
    double bytes;       /* summed algorithmic DRAM bytes */
} tt_op_profile;

tt_status tt_ctx_set_profiling(tt_ctx* ctx, int on);
int tt_ctx_profile_read(tt_ctx* ctx, tt_op_profile* rows, int max_rows);

/* Message of the last failure on this context ("" if none).  Never NULL. */
const char* tt_last_error(const tt_ctx* ctx);

/* --------------------------------------------------------- model layout */

/* Number of elements of the flat parameter vector.  Order (fixed): wte[V,C],
 * wpe[maxT,C], then for each layer {ln1_w[C], ln1_b[C], qkv_w[3C,C],
 * qkv_b[3C], proj_w[C,C], proj_b[C], ln2_w[C], ln2_b[C], fc_w[4C,C],
 * fc_b[4C], fcproj_w[C,4C], fcproj_b[C]}, then lnf_w[C], lnf_b[C].  Weight
 * matrices are [out, in] row-major (y = x W^T + b).  QKV output columns are
 * [q | k | v], each split [H, C/H] head-major.  The LM head is tied to wte. */
size_t tt_gpt2_num_params(const tt_gpt2_config* cfg);

/* Offset and size of one tensor: which = 0 wte, 1 wpe, 2..13 the per-layer
 * tensors in the order above (layer = 0..L-1), 14 lnf_w, 15 lnf_b. */
tt_status tt_gpt2_param_offset(const tt_gpt2_config* cfg, int layer, int which,
                               size_t* off, size_t* numel);

/* Exact number of arena bytes tt_gpt2_step needs for a B x T batch (the same
 * allocation sequence, run without launching).  0 for an invalid config. */
size_t tt_gpt2_arena_bytes(const tt_gpt2_config* cfg, int B, int T);

/* ------------------------------------------------------------- training */

/* One forward + backward pass of the GPT-2 step over a B x T batch
 * (tinytorch 三.6-三.7; the tape records every op of the forward and is
 * replayed in reverse record order, a reverse topological order).
 *   params  device, flat (tt_gpt2_num_params elements), fp32 in TT_FP32 mode,
 *           bf16 in TT_BF16 mode, half in TT_FP16 mode.  Read only.
 *   grads   device fp32, flat, same layout.  OVERWRITTEN with
 *           d(mean loss)/d(params) (no separate zeroing is needed).
 *   tokens, targets  int32 [B*T] row-major (b, t); device OR host memory (host
 *           buffers are staged into the arena with cudaMemcpyAsync).  targets
 *           are the next tokens; ids must lie in [0, V).
 *   loss    host float*: if non-NULL the call synchronizes the stream, stores
 *           the mean cross-entropy over all B*T positions and checks the error
 *           flags; if NULL the call does not synchronize (read the loss later
 *           with tt_ctx_loss_device / tt_ctx_sync).
 * Errors: TT_ERR_ARG (B <= 0, T <= 0, T > maxT, NULL pointer, or -- with a
 * non-NULL loss -- a token id out of range); TT_ERR_ARENA_OOM from the host
 * plan before anything is launched; TT_ERR_STATE without a model.  After an
 * error the gradients are undefined and the context is usable after a reset.
 * The arena is NOT reset by this call. */
tt_status tt_gpt2_step(tt_ctx* ctx, const void* params, float* grads,
                       const int32_t* tokens, const int32_t* targets,
                       int B, int T, float* loss);

/* Device pointers to the last step's mean loss (1 float) and per-position
 * losses (B*T floats, row-major).  Valid until the next reset. */
tt_status tt_ctx_loss_device(const tt_ctx* ctx, const float** mean_loss,
                             const float** row_losses);

/* Copy the last step's per-position losses (n <= B*T floats) to dst, which
 * may be host or device memory; synchronizes the context's stream. */
tt_status tt_ctx_copy_row_losses(tt_ctx* ctx, float* dst, size_t n);

/* ---------------------------------------------------------------- step variants
 * Gradient accumulation, global gradient-norm clipping and dynamic loss
 * scaling, with every decision taken on the device (no host round trip):
 *  - accumulation: gradients add up (+=) over micro-batches as they do over a
 *    tensor's consumers (tinytorch 三.3; NumPy framework page 3.2);
 *  - clipping: the global norm clip of the dl-scratch page (3.2, clip_grad_norm_
 *    applied to the separate gradient storage), with the usual coefficient
 *    min(1, max_norm / (norm + 1e-6));
 *  - loss scaling: the dl-scratch page's 3.4 (the loss is multiplied by a scale
 *    before the backward; an Inf/NaN gradient halves the scale and the update
 *    is skipped; after a run of clean steps the scale grows by a small factor).
 * A typical loop: tt_ctx_reset, tt_gpt2_step_ex (first micro-batch without
 * TT_STEP_ACCUMULATE, the rest with it), tt_grad_stats, tt_adamw_ex,
 * tt_loss_scale_update. */

/* tt_gpt2_step_ex flag: add this step's parameter gradients to grads instead
 * of overwriting them. */
#define TT_STEP_ACCUMULATE 1

/* tt_gpt2_step with options.  flags: 0 or TT_STEP_ACCUMULATE (other bits:
 * TT_ERR_ARG).  loss_scale: device float or NULL; when given, the gradients
 * are those of (mean loss) * (*loss_scale), read on the device when the step
 * runs (the reported loss is unscaled). */
tt_status tt_gpt2_step_ex(tt_ctx* ctx, const void* params, float* grads, const int32_t* tokens,
                          const int32_t* targets, int B, int T, int flags, const float* loss_scale,
                          float* loss);

/* Global gradient statistics, on the device: stats[0] = sqrt(sum_i (g_i /
 * s)^2) and stats[1] = 1 if that sum is not finite (an Inf or NaN gradient, or
 * one whose square overflows), else 0; s = *loss_scale when loss_scale is not
 * NULL, else 1.  grads: device fp32 [n]; stats: device float[2].  The sum is
 * taken in a fixed order (per-thread float sums, per-block partials added in
 * double).  Uses a few KB of the arena for the partial sums. */
tt_status tt_grad_stats(tt_ctx* ctx, const float* grads, size_t n, const float* loss_scale, float* stats);

/* AdamW (as tt_adamw) on the gradient g * k, k = (1 / *loss_scale when
 * loss_scale is not NULL) * (min(1, max_norm / (stats[0] + 1e-6)) when
 * max_norm > 0).  step: device int, the number of updates taken so far; the
 * update uses t = *step + 1 and then advances *step.  With stats given and
 * stats[1] != 0 the whole update is skipped: master, params_lowp, m, v and
 * *step keep their values.  max_norm > 0 needs stats (else TT_ERR_ARG). */
tt_status tt_adamw_ex(tt_ctx* ctx, float* master, void* params_lowp, const float* grads, float* m,
                      float* v, size_t n, float lr, float beta1, float beta2, float eps,
                      float weight_decay, int* step, const float* stats, float max_norm,
                      const float* loss_scale);

/* Dynamic loss scale, on the device (loss_scale: device float; clean_steps:
 * device int): after an overflow step (stats[1] != 0) *loss_scale *= backoff
 * and *clean_steps = 0; after a clean step ++*clean_steps, and when it
 * reaches window, *loss_scale *= growth and *clean_steps = 0.  The dl-scratch
 * page's values are backoff 0.5, window 1000, growth 1.001.  TT_ERR_ARG for
 * window < 1, growth < 1 or backoff outside (0, 1). */
tt_status tt_loss_scale_update(tt_ctx* ctx, float* loss_scale, int* clean_steps, const float* stats, int window,
                               float growth, float backoff);

/* One AdamW step over n flat elements (tinytorch 三.7 Adam with bias
 * correction; Forge: weight decay decoupled from the gradient):
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   master -= lr * ( m/(1-b1^step) / (sqrt(v/(1-b2^step)) + eps) + wd * master )
 * master, grads, m, v: device fp32 [n] (m, v start at zero).  params_lowp:
 * device 16-bit [n] copy written from the updated master (round to nearest
 * even): half when the context's model (tt_ctx_set_model) is TT_FP16, bf16
 * otherwise; or NULL (TT_FP32 mode trains the master directly).  step >= 1.
 * Every element decays.  Pointers must be 16-byte aligned. */
tt_status tt_adamw(tt_ctx* ctx, float* master, void* params_lowp, const float* grads,
                   float* m, float* v, size_t n, float lr, float beta1, float beta2,
                   float eps, float weight_decay, int step);

/* dst[i] = bf16(src[i]) (round to nearest even); device pointers, n elements.
 * Used to make the bf16 parameter copy of a freshly initialized master. */
tt_status tt_cast_f32_to_bf16(tt_ctx* ctx, const float* src, void* dst, size_t n);

/* dst[i] = half(src[i]) (round to nearest even; beyond 65504 it is +-inf);
 * device pointers, n elements.  The half copy of the master for TT_FP16. */
tt_status tt_cast_f32_to_f16(tt_ctx* ctx, const float* src, void* dst, size_t n);

/* ------------------------------------------------------------- inference */

/* The forward pass and the mean cross entropy only, no gradients: the
 * validation loss the tinytorch page's training loop evaluates every 40 steps
 * (三.7, 八.3).  Arguments as for tt_gpt2_step without grads; the arena needs
 * at most tt_gpt2_arena_bytes(cfg, B, T).  The logits buffer of the arena is
 * overwritten by the fused cross entropy, as in the step.  The arena is NOT
 * reset by this call. */
tt_status tt_gpt2_eval(tt_ctx* ctx, const void* params, const int32_t* tokens,
                       const int32_t* targets, int B, int T, float* loss);

/* Exact number of arena bytes tt_gpt2_generate needs (the same allocation
 * sequence, run without launching); 0 for invalid arguments. */
size_t tt_gpt2_generate_arena_bytes(const tt_gpt2_config* cfg, int B, int T_prompt, int n_new);

/* Greedy generation with a key/value cache (tinytorch 八.3 generates text
 * after training; the Forge page, 性能瓶颈与未来路线图, names the key/value
 * cache: each new token's query against the cached keys of the earlier
 * positions, instead of recomputing every position).
 *   prompt  int32 [B, T_prompt] row-major, device or host memory; ids in [0, V).
 *   out     int32 [B, T_prompt + n_new] row-major, device or host memory:
 *           receives the prompt followed by n_new tokens, each the first index
 *           of the largest logit given everything before it (greedy).
 *   T_prompt >= 1, n_new >= 0, T_prompt + n_new <= maxT.
 * The prompt runs through the training forward once (prefill), which fills a
 * per-layer cache [B, maxT, 2C] in the arena; every further token is one
 * decode step on the device.  The call synchronizes the stream.  Errors:
 * TT_ERR_ARG for bad shapes, NULL pointers or a prompt id out of range;
 * TT_ERR_ARENA_OOM from the host plan before anything is launched.  The
 * arena is NOT reset by this call. */
tt_status tt_gpt2_generate(tt_ctx* ctx, const void* params, const int32_t* prompt, int B,
                           int T_prompt, int n_new, int32_t* out);

#ifdef __cplusplus
}
#endif
#endif /* TT_H */

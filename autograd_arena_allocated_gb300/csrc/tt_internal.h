// tt_internal.h -- shared declarations of the native runtime and its kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stddef.h>

#include <string>
#include <vector>
#include <utility>

#include "../../include/tt.h"
#include "../../include/tt_ops.h"
#include "../../include/tt_graph.h"

namespace tt {

// ------------------------------------------------------------ device flags
// Error flags written by kernels (never a trap or fault); read back by the host.
enum DeviceFlag : int {
    FLAG_BAD_TOKEN = 0,  // a token/target id outside [0, V)
    FLAG_TIMEOUT = 1,    // a bounded mbarrier wait gave up
    FLAG_NONFINITE = 2,  // non-finite loss
    FLAG_SITE = 3,       // which bounded wait gave up first (kernel-specific code)
    FLAG_COUNT = 4
};

// ------------------------------------------------------------ launch context
// What every kernel launcher needs: the stream, the flag buffer, and a counter
// of launches (launch accounting for the benchmark).
struct Launch {
    cudaStream_t stream = nullptr;
    int* flags = nullptr;  // device int[FLAG_COUNT]
    uint64_t* launches = nullptr;
    bool dry = false;      // plan only: allocate, launch nothing
    int gemm_backend = 0;  // 0 auto, 1 SIMT only
    int num_sms = 148;
    bool pdl = false;      // programmatic dependent launch (kernels launched by launch_k or the GEMM)
    bool f16 = false;      // 16-bit storage is IEEE half, not bf16 (the model's TT_FP16 mode)
    bool no_pair = false;  // tensor-core GEMMs without the two-CTA pair form
    long long wait_cycles = 4000000000LL;  // limit of every bounded device-side wait (clock64 cycles)
    void count() const { if (launches) ++*launches; }
};

// ------------------------------------------------------------ dependent launch
// Programmatic dependent launch: a kernel launched by launch_k with L.pdl set
// may be scheduled while the kernel before it on the stream is finishing.
// Every such kernel calls pdl_enter() before it touches global memory: the
// wait returns once the previous grid has completed and its writes are
// visible, so stream order holds for every read and write; the trigger lets
// the next kernel be scheduled once all of this grid's CTAs have started.
// Both instructions are no-ops in a kernel launched without the attribute.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
    pdl_wait();
    pdl_trigger();
}

template <typename... KArgs, typename... Args>
inline void launch_k(const Launch& L, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute at[1];
    if (L.pdl) {
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
    }
    cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
#endif

// ------------------------------------------------------------ per-device set-up
// Kernel attributes (the dynamic shared-memory limit) and occupancy results
// belong to one device: a process that drives several GPUs must set them once
// on each, with that device current.  PerDevice keeps one state per device
// ordinal: 0 not yet done, 1 done, -1 failed (or a cached value >= 0 for
// `value`).  Two host threads racing on the same device may both run the
// set-up; it is idempotent.
constexpr int kMaxDevices = 64;

inline int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return d;
}

struct PerDevice {
    volatile int state[kMaxDevices] = {};
    // runs f() (returning bool) once for the current device; its result is kept
    template <class F>
    bool once(F&& f) {
        const int d = current_device();
        if (d < 0 || d >= kMaxDevices) return f();
        if (state[d] == 0) state[d] = f() ? 1 : -1;
        return state[d] == 1;
    }
    // runs f() (returning int >= 0) once for the current device; its value is kept
    template <class F>
    int value(F&& f) {
        const int d = current_device();
        if (d < 0 || d >= kMaxDevices) return f();
        if (state[d] == 0) state[d] = f() + 1;
        return state[d] - 1;
    }
};

// ------------------------------------------------------------ GEMM
// Logical contraction D[m,n] = sum_k A(m,k) B(n,k) with
//   A(m,k) = a_kmajor ? A[m*lda + k] : A[k*lda + m]
//   B(n,k) = b_kmajor ? B[n*ldb + k] : B[k*ldb + n]
// and an epilogue.  The three forms the step uses:
//   FWD: A = x [M,K] (K-major), B = W [N,K] (K-major), D = y [M,N]
//   DX : A = dy [M,N'] (K-major), B(n,k) = W[k,n] (MN-major), D = dx
//   DW : A(n,m) = dy[m,n] (MN-major), B(k,m) = x[m,k] (MN-major), D = dW fp32
enum EpiKind : int {
    EPI_STORE = 0,   // D = acc (+ bias) (+ residual)
    EPI_GELU = 1,    // aux = acc + bias (pre-activation), D = gelu(aux)
    EPI_DGELU = 2,   // D = acc * gelu'(aux)
};

struct GemmArgs {
    const void* A = nullptr; long long lda = 0; bool a_kmajor = true;
    const void* B = nullptr; long long ldb = 0; bool b_kmajor = true;
    int M = 0, N = 0, K = 0;
    int a_rows = 0;          // valid extent of A's MN dimension (rows beyond read as 0); 0 = M
    int b_rows = 0;          // valid extent of B's MN dimension (rows beyond read as 0); 0 = N
    int k_valid = 0;         // valid extent of K (beyond reads as 0); 0 = K
    bool in_bf16 = true;     // operand storage: bf16 or fp32
    bool in_f16 = false;     // with in_bf16: the 16-bit storage is IEEE half (SIMT kernel only)
    void* D = nullptr; long long ldd = 0; bool d_f32 = false;
    int n_store = 0;         // columns >= n_store are not stored; 0 = N
    int epi = EPI_STORE;
    const void* bias = nullptr;      // [N], same storage type as operands
    const void* residual = nullptr;  // [M, ldd] same type as D
    void* aux = nullptr;             // EPI_GELU: out pre-activation; EPI_DGELU: in
    bool accumulate = false;         // D += result
    // optional: column sums of the result over each 32-row slice,
    // colsum_part[m / 32][n] (gemm_colsum_rows(M) rows); *colsum_done is set
    // when the kernel wrote them (the tensor-core GELU' epilogue does)
    float* colsum_part = nullptr;
    bool* colsum_done = nullptr;
};
inline int gemm_colsum_rows(int M) { return ((M + 127) / 128) * 4; }

// Runs the GEMM; `workspace` (fp32, may be needed for split-K of the DW form)
// is sized by gemm_workspace_floats.  Returns false on unsupported arguments.
bool gemm(const Launch& L, const GemmArgs& g, float* workspace, size_t workspace_floats);
size_t gemm_workspace_floats(const Launch& L, const GemmArgs& g);
bool gemm_tc_eligible(const GemmArgs& g);
bool gemm_tc_launch(const Launch& L, const GemmArgs& g, float* workspace, size_t workspace_floats);
size_t gemm_tc_workspace_floats(const Launch& L, const GemmArgs& g);
void gemm_simt_launch(const Launch& L, const GemmArgs& g);

// ------------------------------------------------------------ other kernels
void launch_embed_fwd(const Launch& L, bool bf16, const void* wte, const void* wpe,
                      const int32_t* tok, void* x, int B, int T, int C, int V);
// scratch: the stable sort of positions by token id plus chunk partial sums
size_t embed_bwd_scratch_bytes(int M, int C);
void launch_embed_bwd(const Launch& L, bool bf16, const void* dx, const int32_t* tok,
                      float* dwte, float* dwpe, int B, int T, int C, int V, int maxT,
                      void* scratch, bool acc_params = false);

size_t layernorm_bwd_scratch_floats(int M, int C);
void launch_layernorm_fwd(const Launch& L, bool bf16, const void* x, const void* w,
                          const void* b, void* y, float* mean, float* rstd, int M, int C);
// dres (may be NULL): also the column sums of the finished dx -- the bias
// gradient of the linear layer that produced x (the bf16 vector kernel forms
// them on the way; the others in a second pass)
void launch_layernorm_bwd(const Launch& L, bool bf16, const void* x, const void* w,
                          const float* mean, const float* rstd, const void* dy, void* dx,
                          float* dw, float* db, int M, int C, bool accumulate, float* scratch,
                          bool acc_params = false, float* dres = nullptr);

// dz = (softmax - onehot) * dscale (* *scale_dev when given: a device loss scale)
void launch_xent(const Launch& L, bool bf16, void* logits, const int32_t* targets,
                 float* row_loss, float* mean_loss, int M, int V, int ld, float dscale,
                 const float* scale_dev = nullptr);

size_t colsum_scratch_floats(int M, int N);
void launch_colsum(const Launch& L, bool bf16, const void* x, int M, int N, float* out,
                   float* scratch, bool acc = false);

void launch_adamw(const Launch& L, float* master, void* lowp, const float* g,
                  float* m, float* v, size_t n, float lr, float b1, float b2, float eps,
                  float wd, int step);
void launch_cast_bf16(const Launch& L, const float* src, __nv_bfloat16* dst, size_t n);
void launch_cast_f16(const Launch& L, const float* src, __half* dst, size_t n);
// global gradient statistics: stats[0] = ||g / scale||_2, stats[1] = 1 if not finite
size_t grad_stats_scratch_doubles(const Launch& L);
void launch_grad_stats(const Launch& L, const float* g, size_t n, const float* scale_dev, float* stats,
                       double* scratch);
// AdamW whose gradient is g / scale * clip, skipped when stats[1] != 0; t = *step + 1
void launch_adamw_ex(const Launch& L, float* master, void* lowp, const float* g, float* m, float* v,
                     size_t n, float lr, float b1, float b2, float eps, float wd, int* step, const float* stats,
                     float max_norm, const float* scale_dev);
void launch_loss_scale_update(const Launch& L, float* scale, int* clean, const float* stats, int window,
                              float growth, float backoff);

size_t attention_bwd_scratch_floats(int B, int T, int C, int H);
void launch_attention_fwd(const Launch& L, bool bf16, const void* qkv, void* y, float* lse,
                          int B, int T, int C, int H);
// dbias (may be NULL): also the column sums of dqkv -- the qkv layer's bias
// gradient (accumulated into when acc_bias)
void launch_attention_bwd(const Launch& L, bool bf16, const void* qkv, const void* y,
                          const float* lse, const void* dy, void* dqkv, int B, int T, int C,
                          int H, float* scratch, float* dbias = nullptr, bool acc_bias = false);
// bandwidth-oriented bf16 kernels (kernels_bf16.cu); false = shape not taken
bool launch_ln_fwd_bf16(const Launch& L, const void* x, const void* w, const void* b, void* y,
                        float* mean, float* rstd, int M, int C);
bool launch_ln_bwd_bf16(const Launch& L, const void* x, const void* w, const float* mean,
                        const float* rstd, const void* dy, void* dx, float* dw, float* db, int M,
                        int C, bool accumulate, float* scratch, bool acc_params = false,
                        float* dres = nullptr);
size_t ln_bwd_bf16_scratch_floats(int C);
bool launch_xent_bf16(const Launch& L, void* logits, const int32_t* targets, float* row_loss, int M,
                      int V, int ld, float dscale, const float* scale_dev = nullptr);
bool launch_colsum_bf16(const Launch& L, const void* x, int M, int N, float* part);
// out[c] = sum of the G rows of part[G][ncols] (fixed order); columns [0, split)
// go to out_a, [split, 2 split) to out_b, [2 split, 3 split) to out_c
void launch_sum_rows(const Launch& L, const float* part, int G, int ncols, int split, float* out_a,
                     float* out_b, bool acc = false, float* out_c = nullptr);
size_t embed_chunk_scratch_floats(int M, int C);
bool launch_embed_chunks(const Launch& L, bool bf16, const void* dx, const int32_t* keys,
                         const int32_t* vals, int M, int C, int V, float* dwte, float* scratch);

// tcgen05 attention (attn_tc.cu); false = not taken (then the mma.sync path runs)
bool attention_tc_eligible(bool bf16, int C, int H);
bool launch_attention_fwd_tc(const Launch& L, const void* qkv, void* y, float* lse, int B, int T,
                             int C, int H);
// bpart (may be NULL): per (sequence, 128-row tile) row of 3C column sums of
// dqkv over the tile's rows (the qkv bias gradient's partials)
bool launch_attention_bwd_tc(const Launch& L, const void* qkv, const void* y, const float* lse,
                             const void* dy, void* dqkv, int B, int T, int C, int H, float* Dlt,
                             float* bpart = nullptr);

// decoding with a key/value cache (decode.cu); cache per layer [B, maxT, 2C].
// The decode-step kernels read the newest position from device memory
// (pos_dev); the step's last linear layer advances it (advance != nullptr).
bool launch_kv_fill(const Launch& L, bool bf16, const void* qkv, void* cache, int B, int Tn, int C, int t0,
                    int maxT);
void launch_set_int(const Launch& L, int* p, int v);  // *p = v
void launch_add_int(const Launch& L, int* p, int v);  // *p += v
void launch_embed_at(const Launch& L, bool bf16, const void* wte, const void* wpe, const int32_t* tok,
                     int ld_tok, const int* pos_dev, void* x, int B, int C, int V);
// attention of the newest query against keys 0..pos (at most max_keys), which
// also writes the newest key and value into the cache; part holds
// decode_attn_scratch_floats() floats, counters B*H ints that start at zero
// (and are left at zero)
int decode_attn_splits(int max_keys);
size_t decode_attn_scratch_floats(int B, int H, int max_keys);
bool launch_decode_attn(const Launch& L, bool bf16, const void* qkv, void* cache, void* y, int B, int H, int C,
                        const int* pos_dev, int max_keys, int maxT, float* part, int* counters);
// greedy choice over stored logits into out[b][col_dev ? *col_dev : col]
void launch_argmax(const Launch& L, bool bf16, const void* z, long long row_stride, int rows, int V, int32_t* out,
                   int ld_out, int col, const int* col_dev);
// decode-step linear layers (M <= 16 rows); false = shape not taken.  With
// ln_w/ln_b (bf16 only, K <= 1024) the rows of A go through LayerNorm first.
bool launch_gemm_skinny(const Launch& L, bool bf16, const void* A, const void* W, const void* bias, const void* res,
                        void* D, void* pre, int M, int N, int K, int ldd, int n_store, bool gelu, int* advance,
                        const void* ln_w = nullptr, const void* ln_b = nullptr);
// bf16 LM head with the greedy choice folded in: keys[m * skinny_pick_ctas(N) + cta]
// holds each CTA's largest (logit, -index) key of row m; launch_pick reduces them
int skinny_pick_ctas(int N);
bool launch_gemm_skinny_pick(const Launch& L, const void* A, const void* W, int M, int N, int K,
                             unsigned long long* keys, int* advance, const void* ln_w = nullptr,
                             const void* ln_b = nullptr);
void launch_pick(const Launch& L, const unsigned long long* keys, int nct, int rows, int32_t* tok, int ld_tok,
                 const int* pos_dev);

// the generic tensor graph (graph.cu), fp32
constexpr int G_ZERO_MAX = 32;
struct GZeroList {  // buffers to zero in one launch (passed by value)
    float* p[G_ZERO_MAX];
    long long n[G_ZERO_MAX];
    int count;
};
void launch_g_zero_many(const Launch& L, const GZeroList& l);
void launch_g_matmul(const Launch& L, const float* X, long long xi, long long xk, const float* Y, long long yk,
                     long long yj, float* C, int M, int N, int K, bool accumulate);
void launch_g_add(const Launch& L, const float* a, const float* b, float* c, long long n, int bcols);
void launch_g_mul(const Launch& L, const float* a, const float* b, float* c, long long n);
void launch_g_gelu(const Launch& L, const float* a, float* c, long long n);
void launch_g_softmax(const Launch& L, const float* z, float* p, int rows, int cols);
void launch_g_xent(const Launch& L, const float* p, const int32_t* y, int rows, int cols, float* loss);
void launch_g_fill(const Launch& L, float* d, long long n, float v);
void launch_g_acc(const Launch& L, float* d, const float* s, long long n);
void launch_g_colsum_acc(const Launch& L, const float* dC, int rows, int cols, float* db);
void launch_g_mul_bwd(const Launch& L, const float* dc, const float* a, const float* b, float* ga, float* gb,
                      long long n);
void launch_g_gelu_bwd(const Launch& L, const float* dc, const float* a, float* ga, long long n);
void launch_g_softmax_bwd(const Launch& L, const float* p, const float* dp, float* dz, int rows, int cols);
void launch_g_xent_bwd(const Launch& L, const float* p, const int32_t* y, const float* dloss, int rows, int cols,
                       float* dp);
void launch_g_softmax_xent_bwd(const Launch& L, const float* p, const int32_t* y, const float* dloss, int rows,
                               int cols, float* dz);
void launch_g_sgd(const Launch& L, float* w, const float* g, long long n, float lr);

bool attention_mma_eligible(bool bf16, int C, int H);
void launch_attention_fwd_mma(const Launch& L, const void* qkv, void* y, float* lse,
                              int B, int T, int C, int H);
void launch_attention_bwd_mma(const Launch& L, const void* qkv, const void* y,
                              const float* lse, const void* dy, void* dqkv, int B, int T,
                              int C, int H, float* scratch);

}  // namespace tt

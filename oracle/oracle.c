/*
 * oracle.c -- the reference ("oracle") GPT-2 training step: plain, slow,
 * obviously-correct CPU code in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py may load or call this library.  It shares no
 * code, header, table or helper with the CUDA path, and it includes nothing
 * from that path.
 *
 * Pages followed (cited by title and section):
 *   [TT]    "不用PyTorch，一个头文件就能训练GPT-2：Arena内存池+自动微分的C++实现"
 *           (the tinytorch page): 三.1 Arena, 三.2 Tensor, 三.3 autograd and MatMul,
 *           三.4 GELU, 三.5 Softmax+CrossEntropy, 三.6 GPT-2 model, 三.7 training loop (Adam),
 *           八.1 and 八.5 the small classifier trained by SGD through the generic tensor API.
 *   [FORGE] "17岁少年用C++从零构建深度学习框架Forge，精确复现GPT-2": 核心组件清单
 *           (GELU tanh form, fused log-softmax CE, AdamW decoupled decay) and
 *           最硬的一关 (causal -inf mask, 1/sqrt(d_k), LayerNorm eps/variance).
 *   [NPF]   the NumPy framework page ("为什么我要从零写一个深度学习框架"):
 *           3.2 gradient accumulation, 4.2 finite-difference check, 4.3 graph trace.
 *   [MCRAD] the "microcrad" page: Values 的工作原理, 操作, 反向传播 (topological
 *           backward returning 0 / -1).
 *   [DLS]   "从零手写C++深度学习框架：Tensor设计、Autograd与CUDA优化实战" (the
 *           dl-scratch page): 3.2 clip_grad_norm_ on the gradient storage, 3.4
 *           dynamic loss scaling (halve on Inf/NaN, grow after a run of clean steps).
 *
 * Readings taken where the pages are silent or garbled (each is listed in
 * the design notes of the repository):
 *   - loss = mean over all B*T positions, targets = tokens shifted by one
 *     ([TT] 三.6 takes only the last position in a "simplified" sketch);
 *   - GELU backward = exact derivative of the tanh form ([TT] 三.4 prints the
 *     erf-GELU derivative, which does not match its own forward);
 *   - position embedding is indexed by position t ([TT] 三.6 is garbled);
 *   - the LM head is tied to the token embedding;
 *   - LayerNorm: biased variance, eps = 1e-5 inside the square root;
 *   - AdamW: eps = 1e-8, p -= lr*(mhat/(sqrt(vhat)+eps) + wd*p), every tensor
 *     decays, step t is 1-based ([TT] 三.7 uses step+1);
 *   - MatMul is C = A B with B [K, N] ([TT] 三.3); the classifier's weights are
 *     therefore W1 [3, 32] and W2 [32, 3] ([TT] 八.5 declares them [32, 3] and
 *     [3, 32], which does not compose with that MatMul);
 *   - the classifier's SGD update is p[i] -= lr * g[i] for every element;
 *   - gradient clipping is the global L2 norm clip with coefficient
 *     min(1, max_norm / (norm + 1e-6)) ([DLS] 3.2 names clip_grad_norm_ only);
 *   - loss scaling multiplies the loss by the scale, an overflow skips the
 *     update and halves the scale, and every window-th clean step in a row
 *     multiplies it by the growth factor ([DLS] 3.4: halve; x1.001 after
 *     1000 clean steps).
 *
 * Parity pins: every exported function is pinned by tests/test_oracle_*.py
 * against closed forms, worked examples printed on the pages, library
 * routines (torch float64 functional ops, torch.optim.AdamW) or central
 * finite differences.  No function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Configuration and the flat parameter layout                              */
/* ------------------------------------------------------------------------ */

typedef struct {
    int L, C, H, V, maxT;
} or_config;

/* Offsets of the parameter tensors inside the flat vector, in the fixed
 * order: wte[V,C], wpe[maxT,C], per layer {ln1_w, ln1_b, qkv_w[3C,C], qkv_b,
 * proj_w[C,C], proj_b, ln2_w, ln2_b, fc_w[4C,C], fc_b, fcproj_w[C,4C],
 * fcproj_b}, then lnf_w, lnf_b.  The oracle computes this on its own. */
typedef struct {
    size_t wte, wpe;
    size_t ln1w, ln1b, qkvw, qkvb, projw, projb, ln2w, ln2b, fcw, fcb, fpw, fpb;
    size_t layer_stride, layers_begin;
    size_t lnfw, lnfb, total;
} or_layout;

static or_layout or_make_layout(const or_config* c) {
    or_layout o;
    size_t C = (size_t)c->C;
    size_t at = 0;
    o.wte = at;  at += (size_t)c->V * C;
    o.wpe = at;  at += (size_t)c->maxT * C;
    o.layers_begin = at;
    /* offsets relative to the start of a layer */
    size_t r = 0;
    o.ln1w = r;  r += C;
    o.ln1b = r;  r += C;
    o.qkvw = r;  r += 3 * C * C;
    o.qkvb = r;  r += 3 * C;
    o.projw = r; r += C * C;
    o.projb = r; r += C;
    o.ln2w = r;  r += C;
    o.ln2b = r;  r += C;
    o.fcw = r;   r += 4 * C * C;
    o.fcb = r;   r += 4 * C;
    o.fpw = r;   r += 4 * C * C;
    o.fpb = r;   r += C;
    o.layer_stride = r;
    at += (size_t)c->L * r;
    o.lnfw = at; at += C;
    o.lnfb = at; at += C;
    o.total = at;
    return o;
}

OR_EXPORT size_t or_num_params(int L, int C, int H, int V, int maxT) {
    or_config c = {L, C, H, V, maxT};
    return or_make_layout(&c).total;
}

/* which: 0 wte, 1 wpe, 2..13 the per-layer tensors in order, 14 lnf_w, 15 lnf_b */
OR_EXPORT int or_param_offset(int L, int C, int H, int V, int maxT, int layer, int which,
                              size_t* off, size_t* numel) {
    or_config c = {L, C, H, V, maxT};
    or_layout o = or_make_layout(&c);
    size_t Cz = (size_t)C;
    size_t base = o.layers_begin + (size_t)layer * o.layer_stride;
    switch (which) {
    case 0: *off = o.wte; *numel = (size_t)V * Cz; return 0;
    case 1: *off = o.wpe; *numel = (size_t)maxT * Cz; return 0;
    case 14: *off = o.lnfw; *numel = Cz; return 0;
    case 15: *off = o.lnfb; *numel = Cz; return 0;
    default: break;
    }
    if (layer < 0 || layer >= L || which < 2 || which > 13) return -1;
    switch (which) {
    case 2: *off = base + o.ln1w; *numel = Cz; break;
    case 3: *off = base + o.ln1b; *numel = Cz; break;
    case 4: *off = base + o.qkvw; *numel = 3 * Cz * Cz; break;
    case 5: *off = base + o.qkvb; *numel = 3 * Cz; break;
    case 6: *off = base + o.projw; *numel = Cz * Cz; break;
    case 7: *off = base + o.projb; *numel = Cz; break;
    case 8: *off = base + o.ln2w; *numel = Cz; break;
    case 9: *off = base + o.ln2b; *numel = Cz; break;
    case 10: *off = base + o.fcw; *numel = 4 * Cz * Cz; break;
    case 11: *off = base + o.fcb; *numel = 4 * Cz; break;
    case 12: *off = base + o.fpw; *numel = 4 * Cz * Cz; break;
    case 13: *off = base + o.fpb; *numel = Cz; break;
    }
    return 0;
}

OR_EXPORT void or_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

OR_EXPORT int or_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Host arena ([TT] 三.1): every tensor of a step is cut from big blocks by  */
/* bumping an offset; one reset releases everything.  Blocks are chained so */
/* that earlier pointers stay valid when a new block is needed.             */
/* ------------------------------------------------------------------------ */

typedef struct or_block {
    struct or_block* next;
    size_t cap, off;
    double data[];
} or_block;

typedef struct {
    or_block* head;
    size_t bytes_in_use;
} or_arena;

static double* ar_new(or_arena* a, size_t n) {
    size_t need = n ? n : 1;
    need = (need + 7) & ~(size_t)7; /* keep 64-byte granularity */
    if (!a->head || a->head->off + need > a->head->cap) {
        size_t cap = need > ((size_t)1 << 24) ? need : ((size_t)1 << 24); /* 128 MB blocks */
        or_block* b = (or_block*)malloc(sizeof(or_block) + cap * sizeof(double));
        if (!b) abort();
        b->next = a->head;
        b->cap = cap;
        b->off = 0;
        a->head = b;
    }
    double* p = a->head->data + a->head->off;
    a->head->off += need;
    a->bytes_in_use += need * sizeof(double);
    memset(p, 0, n * sizeof(double));
    return p;
}

static void ar_reset(or_arena* a) {
    or_block* b = a->head;
    while (b) {
        or_block* nx = b->next;
        free(b);
        b = nx;
    }
    a->head = NULL;
    a->bytes_in_use = 0;
}

/* ------------------------------------------------------------------------ */
/* Op arithmetic.  Each op has a forward and a backward; backward functions */
/* ACCUMULATE (+=) into the input gradients, because one tensor can feed     */
/* several consumers ([TT] 三.3, [NPF] 3.2).                                 */
/* ------------------------------------------------------------------------ */

/* y[m,n] = sum_k x[m,k] * W[n,k] + b[n]; W is stored [out,in] ([TT] 八.5
 * allocates W1 as {neurons, variables}); b may be NULL. */
OR_EXPORT void or_linear_fwd(const double* x, const double* W, const double* b,
                             int M, int K, int N, double* y) {
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; m++) {
        const double* xr = x + (size_t)m * K;
        for (int n = 0; n < N; n++) {
            const double* wr = W + (size_t)n * K;
            double s = 0.0;
            for (int k = 0; k < K; k++) s += xr[k] * wr[k];
            y[(size_t)m * N + n] = s + (b ? b[n] : 0.0);
        }
    }
}

/* dx += dy * W ; dW += dy^T * x ; db += column sums of dy  ([TT] 三.3 MatMul backward) */
OR_EXPORT void or_linear_bwd(const double* x, const double* W, const double* dy,
                             int M, int K, int N, double* dx, double* dW, double* db) {
    if (dx) {
#pragma omp parallel for schedule(static)
        for (int m = 0; m < M; m++) {
            double* dxr = dx + (size_t)m * K;
            for (int n = 0; n < N; n++) {
                double g = dy[(size_t)m * N + n];
                const double* wr = W + (size_t)n * K;
                for (int k = 0; k < K; k++) dxr[k] += g * wr[k];
            }
        }
    }
    if (dW) {
#pragma omp parallel for schedule(static)
        for (int n = 0; n < N; n++) {
            double* dwr = dW + (size_t)n * K;
            for (int m = 0; m < M; m++) {
                double g = dy[(size_t)m * N + n];
                const double* xr = x + (size_t)m * K;
                for (int k = 0; k < K; k++) dwr[k] += g * xr[k];
            }
        }
    }
    if (db) {
        for (int n = 0; n < N; n++) {
            double s = 0.0;
            for (int m = 0; m < M; m++) s += dy[(size_t)m * N + n];
            db[n] += s;
        }
    }
}

/* LayerNorm over the last dimension: subtract the mean, divide by the
 * standard deviation, scale and shift ([TT] 四, LayerNorm row).  Biased
 * variance, eps inside the root.  Two passes: mean, then mean((x-mu)^2). */
OR_EXPORT void or_layernorm_fwd(const double* x, const double* w, const double* b,
                                int M, int C, double eps,
                                double* y, double* mean, double* rstd) {
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; m++) {
        const double* xr = x + (size_t)m * C;
        double mu = 0.0;
        for (int c = 0; c < C; c++) mu += xr[c];
        mu /= C;
        double var = 0.0;
        for (int c = 0; c < C; c++) var += (xr[c] - mu) * (xr[c] - mu);
        var /= C;
        double rs = 1.0 / sqrt(var + eps);
        for (int c = 0; c < C; c++)
            y[(size_t)m * C + c] = (xr[c] - mu) * rs * w[c] + b[c];
        mean[m] = mu;
        rstd[m] = rs;
    }
}

/* Chain rule through y = xhat*w + b with xhat = (x - mu)*rstd:
 *   dw += sum_m dy*xhat,  db += sum_m dy,
 *   dx += rstd * (g - mean(g) - xhat*mean(g*xhat)),  g = dy*w. */
OR_EXPORT void or_layernorm_bwd(const double* x, const double* w, const double* mean,
                                const double* rstd, const double* dy, int M, int C,
                                double* dx, double* dw, double* db) {
    if (dx) {
#pragma omp parallel for schedule(static)
        for (int m = 0; m < M; m++) {
            const double* xr = x + (size_t)m * C;
            const double* dyr = dy + (size_t)m * C;
            double mg = 0.0, mgx = 0.0;
            for (int c = 0; c < C; c++) {
                double xh = (xr[c] - mean[m]) * rstd[m];
                double g = dyr[c] * w[c];
                mg += g;
                mgx += g * xh;
            }
            mg /= C;
            mgx /= C;
            for (int c = 0; c < C; c++) {
                double xh = (xr[c] - mean[m]) * rstd[m];
                double g = dyr[c] * w[c];
                dx[(size_t)m * C + c] += rstd[m] * (g - mg - xh * mgx);
            }
        }
    }
#pragma omp parallel for schedule(static)
    for (int c = 0; c < C; c++) {
        double sw = 0.0, sb = 0.0;
        for (int m = 0; m < M; m++) {
            double xh = (x[(size_t)m * C + c] - mean[m]) * rstd[m];
            sw += dy[(size_t)m * C + c] * xh;
            sb += dy[(size_t)m * C + c];
        }
        if (dw) dw[c] += sw;
        if (db) db[c] += sb;
    }
}

/* GELU, tanh approximation ([TT] 三.4, [FORGE] 核心组件清单):
 *   g(u) = 0.5 u (1 + tanh(k (u + 0.044715 u^3))),  k = sqrt(2/pi). */
#define OR_GELU_A 0.044715
static double or_gelu_k(void) { return sqrt(2.0 / M_PI); }

OR_EXPORT void or_gelu_fwd(const double* u, size_t n, double* g) {
    double k = or_gelu_k();
    for (size_t i = 0; i < n; i++) {
        double x = u[i];
        g[i] = 0.5 * x * (1.0 + tanh(k * (x + OR_GELU_A * x * x * x)));
    }
}

/* Exact derivative of the tanh form (reading: [TT] 三.4 prints the erf
 * derivative, which does not belong to its own forward):
 *   g'(u) = 0.5 (1 + tau) + 0.5 u (1 - tau^2) k (1 + 3 a u^2),  tau = tanh(k(u + a u^3)). */
OR_EXPORT void or_gelu_bwd(const double* u, const double* dg, size_t n, double* du) {
    double k = or_gelu_k();
    for (size_t i = 0; i < n; i++) {
        double x = u[i];
        double tau = tanh(k * (x + OR_GELU_A * x * x * x));
        double d = 0.5 * (1.0 + tau) + 0.5 * x * (1.0 - tau * tau) * k * (1.0 + 3.0 * OR_GELU_A * x * x);
        du[i] += dg[i] * d;
    }
}

/* Causal multi-head self-attention ([FORGE] 最硬的一关: scores divided by
 * sqrt(d_k), future positions masked with -inf; softmax with max
 * subtraction, [TT] 四).  qkv is [B*T, 3C] with columns [q | k | v], each
 * split [H, hd] head-major.  P is saved as [B, H, T, T] (masked entries 0).
 * lse (may be NULL) receives, per [B, H, T] row, the natural log of the
 * softmax denominator taken over the scaled scores: m + ln(sum exp(s - m)),
 * the normaliser the backward needs to rebuild P from the scores. */
OR_EXPORT void or_attention_fwd(const double* qkv, int B, int T, int C, int H,
                                double* y, double* P, double* lse) {
    int hd = C / H;
    double scale = 1.0 / sqrt((double)hd);
    size_t ld = (size_t)3 * C;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < H; h++) {
            double* Pbh = P + ((size_t)b * H + h) * (size_t)T * T;
            for (int t = 0; t < T; t++) {
                const double* q = qkv + ((size_t)b * T + t) * ld + (size_t)h * hd;
                double* prow = Pbh + (size_t)t * T;
                double mx = -INFINITY;
                for (int s = 0; s < T; s++) {
                    if (s > t) { prow[s] = -INFINITY; continue; }
                    const double* kk = qkv + ((size_t)b * T + s) * ld + C + (size_t)h * hd;
                    double d = 0.0;
                    for (int i = 0; i < hd; i++) d += q[i] * kk[i];
                    prow[s] = d * scale;
                    if (prow[s] > mx) mx = prow[s];
                }
                double sum = 0.0;
                for (int s = 0; s < T; s++) {
                    prow[s] = (s > t) ? 0.0 : exp(prow[s] - mx);
                    sum += prow[s];
                }
                for (int s = 0; s < T; s++) prow[s] /= sum;
                if (lse) lse[((size_t)b * H + h) * T + t] = mx + log(sum);
                double* yr = y + ((size_t)b * T + t) * C + (size_t)h * hd;
                for (int i = 0; i < hd; i++) {
                    double acc = 0.0;
                    for (int s = 0; s <= t; s++)
                        acc += prow[s] * qkv[((size_t)b * T + s) * ld + 2 * (size_t)C + (size_t)h * hd + i];
                    yr[i] = acc;
                }
            }
        }
    }
}

/* Backward of y = P V with P = softmax(q k^T / sqrt(hd)) (masked):
 *   dV += P^T dY;  dP = dY V^T;  dS = P o (dP - rowsum(P o dP));
 *   dQ += dS K / sqrt(hd);  dK += dS^T Q / sqrt(hd). */
OR_EXPORT void or_attention_bwd(const double* qkv, const double* P, const double* dy,
                                int B, int T, int C, int H, double* dqkv) {
    int hd = C / H;
    double scale = 1.0 / sqrt((double)hd);
    size_t ld = (size_t)3 * C;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < H; h++) {
            const double* Pbh = P + ((size_t)b * H + h) * (size_t)T * T;
            double* dP = (double*)calloc((size_t)T, sizeof(double));
            for (int t = 0; t < T; t++) {
                const double* prow = Pbh + (size_t)t * T;
                const double* dyr = dy + ((size_t)b * T + t) * C + (size_t)h * hd;
                /* dP[t,s] = dy_t . v_s, and dv_s += P[t,s] dy_t */
                double dot = 0.0;
                for (int s = 0; s <= t; s++) {
                    const double* v = qkv + ((size_t)b * T + s) * ld + 2 * (size_t)C + (size_t)h * hd;
                    double* dv = dqkv + ((size_t)b * T + s) * ld + 2 * (size_t)C + (size_t)h * hd;
                    double d = 0.0;
                    for (int i = 0; i < hd; i++) {
                        d += dyr[i] * v[i];
                        dv[i] += prow[s] * dyr[i];
                    }
                    dP[s] = d;
                    dot += prow[s] * d;
                }
                const double* q = qkv + ((size_t)b * T + t) * ld + (size_t)h * hd;
                double* dq = dqkv + ((size_t)b * T + t) * ld + (size_t)h * hd;
                for (int s = 0; s <= t; s++) {
                    double ds = prow[s] * (dP[s] - dot) * scale;
                    const double* kk = qkv + ((size_t)b * T + s) * ld + C + (size_t)h * hd;
                    double* dk = dqkv + ((size_t)b * T + s) * ld + C + (size_t)h * hd;
                    for (int i = 0; i < hd; i++) {
                        dq[i] += ds * kk[i];
                        dk[i] += ds * q[i];
                    }
                }
            }
            free(dP);
        }
    }
}

/* Fused log-softmax cross entropy ([TT] 三.5, [FORGE] 核心组件清单):
 *   loss_m = log(sum_v exp(z[m,v])) - z[m, y_m]  (max subtracted first),
 *   loss   = (1/M) sum_m loss_m;
 * if dz is given: dz[m,v] += dloss * (softmax(z_m)[v] - [v == y_m]) / M. */
OR_EXPORT double or_xent(const double* z, const int* targets, int M, int V,
                         double* row_loss, double* dz, double dloss) {
    double total = 0.0;
    double* rl = row_loss ? row_loss : (double*)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1));
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; m++) {
        const double* zr = z + (size_t)m * V;
        double mx = -INFINITY;
        for (int v = 0; v < V; v++) if (zr[v] > mx) mx = zr[v];
        double sum = 0.0;
        for (int v = 0; v < V; v++) sum += exp(zr[v] - mx);
        double lse = mx + log(sum);
        rl[m] = lse - zr[targets[m]];
        if (dz) {
            double* dr = dz + (size_t)m * V;
            for (int v = 0; v < V; v++) {
                double p = exp(zr[v] - lse);
                dr[v] += dloss * (p - (v == targets[m] ? 1.0 : 0.0)) / M;
            }
        }
    }
    for (int m = 0; m < M; m++) total += rl[m];
    if (!row_loss) free(rl);
    return M > 0 ? total / M : 0.0;
}

/* Token + position embedding ([TT] 三.6): x[b*T+t] = wte[tok] + wpe[t]. */
OR_EXPORT void or_embed_fwd(const double* wte, const double* wpe, const int* tok,
                            int B, int T, int C, double* x) {
    for (int b = 0; b < B; b++)
        for (int t = 0; t < T; t++) {
            size_t m = (size_t)b * T + t;
            for (int c = 0; c < C; c++)
                x[m * C + c] = wte[(size_t)tok[m] * C + c] + wpe[(size_t)t * C + c];
        }
}

/* Rows are added to the table gradients in increasing position order. */
OR_EXPORT void or_embed_bwd(const double* dx, const int* tok, int B, int T, int C,
                            double* dwte, double* dwpe) {
    for (int b = 0; b < B; b++)
        for (int t = 0; t < T; t++) {
            size_t m = (size_t)b * T + t;
            for (int c = 0; c < C; c++) {
                dwte[(size_t)tok[m] * C + c] += dx[m * C + c];
                dwpe[(size_t)t * C + c] += dx[m * C + c];
            }
        }
}

/* AdamW, one step t >= 1 ([TT] 三.7 Adam with bias correction, step+1;
 * [FORGE] 核心组件清单: weight decay decoupled from the gradient update):
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   p -= lr * ( (m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps) + wd * p ). */
OR_EXPORT void or_adamw(double* p, const double* g, double* m, double* v, size_t n,
                        double lr, double b1, double b2, double eps, double wd, int t) {
    double c1 = 1.0 - pow(b1, t);
    double c2 = 1.0 - pow(b2, t);
    for (size_t i = 0; i < n; i++) {
        m[i] = b1 * m[i] + (1.0 - b1) * g[i];
        v[i] = b2 * v[i] + (1.0 - b2) * g[i] * g[i];
        double mh = m[i] / c1;
        double vh = v[i] / c2;
        p[i] -= lr * (mh / (sqrt(vh) + eps) + wd * p[i]);
    }
}

/* ------------------------------------------------------------------------ */
/* Update-side variants ([DLS] 3.2: the global norm clip applied to the     */
/* separate gradient storage; 3.4: dynamic loss scaling; accumulation of     */
/* gradients over micro-batches is the += of [TT] 三.3).                     */
/* ------------------------------------------------------------------------ */

/* sqrt(sum_i (g_i / scale)^2); *nonfinite = 1 if the sum is Inf or NaN. */
OR_EXPORT double or_grad_norm(const double* g, size_t n, double scale, int* nonfinite) {
    double s = 0.0;
    for (size_t i = 0; i < n; i++) {
        double x = g[i] / scale;
        s += x * x;
    }
    if (nonfinite) *nonfinite = isfinite(s) ? 0 : 1;
    return sqrt(s);
}

/* The clip coefficient of a global norm clip: min(1, max_norm / (norm + 1e-6)). */
OR_EXPORT double or_clip_coef(double norm, double max_norm) {
    double c = max_norm / (norm + 1e-6);
    return c < 1.0 ? c : 1.0;
}

/* AdamW step t on the gradient g / scale, clipped to max_norm (max_norm <= 0:
 * no clip), skipped entirely (returns 1, nothing changed) when the unscaled
 * gradient is not finite; returns 0 after an update. */
OR_EXPORT int or_adamw_ex(double* p, const double* g, double* m, double* v, size_t n, double lr, double b1,
                          double b2, double eps, double wd, int t, double scale, double max_norm) {
    int bad = 0;
    double norm = or_grad_norm(g, n, scale, &bad);
    if (bad) return 1;
    double k = 1.0 / scale;
    if (max_norm > 0.0) k *= or_clip_coef(norm, max_norm);
    double* ge = (double*)malloc(sizeof(double) * (n ? n : 1));
    for (size_t i = 0; i < n; i++) ge[i] = g[i] * k;
    or_adamw(p, ge, m, v, n, lr, b1, b2, eps, wd, t);
    free(ge);
    return 0;
}

/* Dynamic loss scale ([DLS] 3.4): an overflow multiplies the scale by backoff
 * and restarts the count of clean steps; a clean step counts, and the
 * window-th clean step in a row multiplies the scale by growth and restarts
 * the count. */
OR_EXPORT void or_loss_scale_update(double* scale, int* clean, int overflow, int window, double growth,
                                    double backoff) {
    if (overflow) {
        *scale *= backoff;
        *clean = 0;
    } else if (++*clean >= window) {
        *scale *= growth;
        *clean = 0;
    }
}

/* ------------------------------------------------------------------------ */
/* Tensor tape ([TT] 三.2-三.3: each tensor records the op and the inputs   */
/* that made it).  Backward replays the records in reverse record order,    */
/* which is a reverse topological order ([MCRAD] 反向传播, [NPF] 3.2), so a */
/* tensor with several consumers receives all of its gradient before its    */
/* own backward runs.                                                        */
/* ------------------------------------------------------------------------ */

typedef struct {
    double* v;     /* values */
    double* g;     /* gradient, allocated zeroed on first use */
    size_t n;
} otensor;

enum { OP_EMBED = 1, OP_LAYERNORM, OP_LINEAR, OP_GELU, OP_ADD, OP_ATTENTION, OP_XENT };

typedef struct {
    int op;
    otensor *a, *b, *c; /* inputs (unused ones NULL) */
    otensor* out;
    double *s0, *s1;    /* saved statistics (LN mean/rstd, attention P) */
    const int* idx;     /* tokens or targets */
    int M, K, N;        /* shapes: rows, inner, outer */
    int B, T, H;
} orecord;

typedef struct {
    or_arena arena;
    orecord* rec;
    int n, cap;
} otape;

static otensor* ot_new(otape* tp, size_t n) {
    otensor* t = (otensor*)ar_new(&tp->arena, (sizeof(otensor) + 7) / 8);
    t->v = ar_new(&tp->arena, n);
    t->g = NULL;
    t->n = n;
    return t;
}

static otensor* ot_wrap(otape* tp, double* v, double* g, size_t n) {
    otensor* t = (otensor*)ar_new(&tp->arena, (sizeof(otensor) + 7) / 8);
    t->v = v;
    t->g = g;
    t->n = n;
    return t;
}

static double* ot_grad(otape* tp, otensor* t) {
    if (!t->g) t->g = ar_new(&tp->arena, t->n);
    return t->g;
}

static orecord* tp_push(otape* tp, int op) {
    if (tp->n == tp->cap) {
        tp->cap = tp->cap ? 2 * tp->cap : 64;
        tp->rec = (orecord*)realloc(tp->rec, sizeof(orecord) * (size_t)tp->cap);
    }
    orecord* r = &tp->rec[tp->n++];
    memset(r, 0, sizeof(*r));
    r->op = op;
    return r;
}

static otensor* tp_embed(otape* tp, otensor* wte, otensor* wpe, const int* tok, int B, int T, int C) {
    otensor* out = ot_new(tp, (size_t)B * T * C);
    or_embed_fwd(wte->v, wpe->v, tok, B, T, C, out->v);
    orecord* r = tp_push(tp, OP_EMBED);
    r->a = wte; r->b = wpe; r->out = out; r->idx = tok; r->B = B; r->T = T; r->N = C;
    return out;
}

static otensor* tp_layernorm(otape* tp, otensor* x, otensor* w, otensor* b, int M, int C) {
    otensor* out = ot_new(tp, (size_t)M * C);
    double* mean = ar_new(&tp->arena, (size_t)M);
    double* rstd = ar_new(&tp->arena, (size_t)M);
    or_layernorm_fwd(x->v, w->v, b->v, M, C, 1e-5, out->v, mean, rstd);
    orecord* r = tp_push(tp, OP_LAYERNORM);
    r->a = x; r->b = w; r->c = b; r->out = out; r->s0 = mean; r->s1 = rstd; r->M = M; r->N = C;
    return out;
}

static otensor* tp_linear(otape* tp, otensor* x, otensor* W, otensor* b, int M, int K, int N) {
    otensor* out = ot_new(tp, (size_t)M * N);
    or_linear_fwd(x->v, W->v, b ? b->v : NULL, M, K, N, out->v);
    orecord* r = tp_push(tp, OP_LINEAR);
    r->a = x; r->b = W; r->c = b; r->out = out; r->M = M; r->K = K; r->N = N;
    return out;
}

static otensor* tp_gelu(otape* tp, otensor* u) {
    otensor* out = ot_new(tp, u->n);
    or_gelu_fwd(u->v, u->n, out->v);
    orecord* r = tp_push(tp, OP_GELU);
    r->a = u; r->out = out;
    return out;
}

static otensor* tp_add(otape* tp, otensor* a, otensor* b) {
    otensor* out = ot_new(tp, a->n);
    for (size_t i = 0; i < a->n; i++) out->v[i] = a->v[i] + b->v[i];
    orecord* r = tp_push(tp, OP_ADD);
    r->a = a; r->b = b; r->out = out;
    return out;
}

static otensor* tp_attention(otape* tp, otensor* qkv, int B, int T, int C, int H) {
    otensor* out = ot_new(tp, (size_t)B * T * C);
    double* P = ar_new(&tp->arena, (size_t)B * H * T * T);
    or_attention_fwd(qkv->v, B, T, C, H, out->v, P, NULL);
    orecord* r = tp_push(tp, OP_ATTENTION);
    r->a = qkv; r->out = out; r->s0 = P; r->B = B; r->T = T; r->N = C; r->H = H;
    return out;
}

static otensor* tp_xent(otape* tp, otensor* z, const int* targets, int M, int V, double* row_loss) {
    otensor* out = ot_new(tp, 1);
    double* rl = ar_new(&tp->arena, (size_t)M);
    out->v[0] = or_xent(z->v, targets, M, V, rl, NULL, 0.0);
    if (row_loss) memcpy(row_loss, rl, sizeof(double) * (size_t)M);
    orecord* r = tp_push(tp, OP_XENT);
    r->a = z; r->out = out; r->idx = targets; r->M = M; r->N = V;
    return out;
}

static void tp_backward_record(otape* tp, orecord* r) {
    double* dy = r->out->g;
    if (!dy) return; /* nothing flows into this op */
    switch (r->op) {
    case OP_EMBED:
        or_embed_bwd(dy, r->idx, r->B, r->T, r->N, ot_grad(tp, r->a), ot_grad(tp, r->b));
        break;
    case OP_LAYERNORM:
        or_layernorm_bwd(r->a->v, r->b->v, r->s0, r->s1, dy, r->M, r->N,
                         ot_grad(tp, r->a), ot_grad(tp, r->b), ot_grad(tp, r->c));
        break;
    case OP_LINEAR:
        or_linear_bwd(r->a->v, r->b->v, dy, r->M, r->K, r->N, ot_grad(tp, r->a),
                      ot_grad(tp, r->b), r->c ? ot_grad(tp, r->c) : NULL);
        break;
    case OP_GELU:
        or_gelu_bwd(r->a->v, dy, r->a->n, ot_grad(tp, r->a));
        break;
    case OP_ADD: {
        double* da = ot_grad(tp, r->a);
        double* db = ot_grad(tp, r->b);
        for (size_t i = 0; i < r->out->n; i++) { da[i] += dy[i]; db[i] += dy[i]; }
        break;
    }
    case OP_ATTENTION:
        or_attention_bwd(r->a->v, r->s0, dy, r->B, r->T, r->N, r->H, ot_grad(tp, r->a));
        break;
    case OP_XENT:
        or_xent(r->a->v, r->idx, r->M, r->N, NULL, ot_grad(tp, r->a), dy[0]);
        break;
    }
}

/* Seed d(loss)/d(loss) = 1 and walk the tape backwards. */
static void tp_backward(otape* tp, otensor* loss) {
    ot_grad(tp, loss)[0] = 1.0;
    for (int i = tp->n - 1; i >= 0; i--) tp_backward_record(tp, &tp->rec[i]);
}

static void tp_free(otape* tp) {
    ar_reset(&tp->arena);
    free(tp->rec);
    tp->rec = NULL;
    tp->n = tp->cap = 0;
}

/* ------------------------------------------------------------------------ */
/* GPT-2 training step ([TT] 三.6 model, 三.7 loop steps 2-3)               */
/* ------------------------------------------------------------------------ */

/* The model's forward ([TT] 三.6) on the tape: embedding, L pre-LN blocks,
 * final LayerNorm and the tied LM head.  Parameter tensors point straight into
 * the flat vectors (and their gradients into G, when given).  Returns the
 * logits [B*T, V]. */
static otensor* tp_gpt2_forward(otape* tp, const or_config* cfg, const or_layout* o,
                                const double* params, double* G, const int* tokens, int B, int T) {
    const int L = cfg->L, C = cfg->C, H = cfg->H, V = cfg->V, maxT = cfg->maxT;
    const int M = B * T;
#define PARAM(off, n) ot_wrap(tp, (double*)params + (off), G ? G + (off) : NULL, (n))
    size_t Cz = (size_t)C;
    otensor* wte = PARAM(o->wte, (size_t)V * Cz);
    otensor* wpe = PARAM(o->wpe, (size_t)maxT * Cz);
    otensor* x = tp_embed(tp, wte, wpe, tokens, B, T, C);
    for (int l = 0; l < L; l++) {
        size_t base = o->layers_begin + (size_t)l * o->layer_stride;
        otensor* ln1w = PARAM(base + o->ln1w, Cz);
        otensor* ln1b = PARAM(base + o->ln1b, Cz);
        otensor* qkvw = PARAM(base + o->qkvw, 3 * Cz * Cz);
        otensor* qkvb = PARAM(base + o->qkvb, 3 * Cz);
        otensor* projw = PARAM(base + o->projw, Cz * Cz);
        otensor* projb = PARAM(base + o->projb, Cz);
        otensor* ln2w = PARAM(base + o->ln2w, Cz);
        otensor* ln2b = PARAM(base + o->ln2b, Cz);
        otensor* fcw = PARAM(base + o->fcw, 4 * Cz * Cz);
        otensor* fcb = PARAM(base + o->fcb, 4 * Cz);
        otensor* fpw = PARAM(base + o->fpw, 4 * Cz * Cz);
        otensor* fpb = PARAM(base + o->fpb, Cz);
        /* pre-LN block: LN -> attention -> residual -> LN -> MLP -> residual */
        otensor* h = tp_layernorm(tp, x, ln1w, ln1b, M, C);
        otensor* qkv = tp_linear(tp, h, qkvw, qkvb, M, C, 3 * C);
        otensor* a = tp_attention(tp, qkv, B, T, C, H);
        otensor* p = tp_linear(tp, a, projw, projb, M, C, C);
        otensor* x1 = tp_add(tp, x, p);
        otensor* h2 = tp_layernorm(tp, x1, ln2w, ln2b, M, C);
        otensor* u = tp_linear(tp, h2, fcw, fcb, M, C, 4 * C);
        otensor* g = tp_gelu(tp, u);
        otensor* f = tp_linear(tp, g, fpw, fpb, M, 4 * C, C);
        x = tp_add(tp, x1, f);
    }
    otensor* lnfw = PARAM(o->lnfw, Cz);
    otensor* lnfb = PARAM(o->lnfb, Cz);
    otensor* hf = tp_layernorm(tp, x, lnfw, lnfb, M, C);
    /* tied LM head: logits = hf * wte^T */
    return tp_linear(tp, hf, wte, NULL, M, C, V);
#undef PARAM
}

/* Forward + backward of one batch.  params: flat [num_params] in the fixed
 * layout; grads (optional): overwritten with d(mean loss)/d(params);
 * row_loss (optional): [B*T] per-position losses.  Returns the mean loss,
 * or NAN on bad arguments. */
OR_EXPORT double or_gpt2_step(int L, int C, int H, int V, int maxT,
                              const double* params, const int* tokens, const int* targets,
                              int B, int T, double* grads, double* row_loss) {
    if (B <= 0 || T <= 0 || T > maxT || C % H != 0) return NAN;
    for (size_t i = 0; i < (size_t)B * T; i++)
        if (tokens[i] < 0 || tokens[i] >= V || targets[i] < 0 || targets[i] >= V) return NAN;
    or_config cfg = {L, C, H, V, maxT};
    or_layout o = or_make_layout(&cfg);
    otape tp;
    memset(&tp, 0, sizeof(tp));
    double* G = grads;
    if (G) memset(G, 0, sizeof(double) * o.total);
    otensor* z = tp_gpt2_forward(&tp, &cfg, &o, params, G, tokens, B, T);
    otensor* loss = tp_xent(&tp, z, targets, B * T, V, row_loss);
    double lv = loss->v[0];
    if (G) tp_backward(&tp, loss);
    tp_free(&tp);
    return lv;
}

/* The logits of each sequence's last position, [B][V] (the distribution the
 * next token is drawn from when generating; [TT] 八.3 generates text after
 * training).  Returns 0, or -1 on bad arguments. */
OR_EXPORT int or_gpt2_logits_last(int L, int C, int H, int V, int maxT, const double* params,
                                  const int* tokens, int B, int T, double* logits_last) {
    if (B <= 0 || T <= 0 || T > maxT || C % H != 0 || !logits_last) return -1;
    for (size_t i = 0; i < (size_t)B * T; i++)
        if (tokens[i] < 0 || tokens[i] >= V) return -1;
    or_config cfg = {L, C, H, V, maxT};
    or_layout o = or_make_layout(&cfg);
    otape tp;
    memset(&tp, 0, sizeof(tp));
    otensor* z = tp_gpt2_forward(&tp, &cfg, &o, params, NULL, tokens, B, T);
    for (int b = 0; b < B; b++)
        memcpy(logits_last + (size_t)b * V, z->v + ((size_t)b * T + (T - 1)) * V, sizeof(double) * (size_t)V);
    tp_free(&tp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Generic tensor ops of the library API ([TT] 三.2-三.5) and the small      */
/* classifier trained by SGD ([TT] 八.1 and 八.5: three features, a hidden   */
/* GELU layer, three classes).  Gradients are accumulated (+=), as [TT] 三.3 */
/* requires for a tensor with several consumers.                            */
/* ------------------------------------------------------------------------ */

/* C[M,N] = A[M,K] B[K,N]: B is [K,N] row-major ([TT] 三.3 MatMulForward). */
OR_EXPORT void or_matmul(const double* A, const double* B, int M, int K, int N, double* C) {
    for (int i = 0; i < M; i++)
        for (int j = 0; j < N; j++) {
            double s = 0.0;
            for (int k = 0; k < K; k++) s += A[(size_t)i * K + k] * B[(size_t)k * N + j];
            C[(size_t)i * N + j] = s;
        }
}

/* dA += dC B^T and dB += A^T dC ([TT] 三.3 MatMulBackward); either may be NULL. */
OR_EXPORT void or_matmul_bwd(const double* A, const double* B, const double* dC, int M, int K, int N,
                             double* dA, double* dB) {
    if (dA)
        for (int i = 0; i < M; i++)
            for (int k = 0; k < K; k++) {
                double s = 0.0;
                for (int j = 0; j < N; j++) s += dC[(size_t)i * N + j] * B[(size_t)k * N + j];
                dA[(size_t)i * K + k] += s;
            }
    if (dB)
        for (int k = 0; k < K; k++)
            for (int j = 0; j < N; j++) {
                double s = 0.0;
                for (int i = 0; i < M; i++) s += A[(size_t)i * K + k] * dC[(size_t)i * N + j];
                dB[(size_t)k * N + j] += s;
            }
}

/* C[r, c] = A[r, c] + b[c] (a bias row added to every row); backward
 * dA += dC, db[c] += sum_r dC[r, c]. */
OR_EXPORT void or_add_row(const double* A, const double* b, int R, int Cc, double* C) {
    for (int r = 0; r < R; r++)
        for (int c = 0; c < Cc; c++) C[(size_t)r * Cc + c] = A[(size_t)r * Cc + c] + b[c];
}
OR_EXPORT void or_add_row_bwd(const double* dC, int R, int Cc, double* dA, double* db) {
    for (int r = 0; r < R; r++)
        for (int c = 0; c < Cc; c++) {
            if (dA) dA[(size_t)r * Cc + c] += dC[(size_t)r * Cc + c];
            if (db) db[c] += dC[(size_t)r * Cc + c];
        }
}

/* Softmax of each row, the row maximum subtracted before exp ([TT] 四,
 * Softmax 数值稳定性). */
OR_EXPORT void or_softmax_rows(const double* Z, int R, int Cc, double* P) {
    for (int r = 0; r < R; r++) {
        const double* z = Z + (size_t)r * Cc;
        double* p = P + (size_t)r * Cc;
        double mx = -INFINITY, sum = 0.0;
        for (int c = 0; c < Cc; c++) if (z[c] > mx) mx = z[c];
        for (int c = 0; c < Cc; c++) { p[c] = exp(z[c] - mx); sum += p[c]; }
        for (int c = 0; c < Cc; c++) p[c] /= sum;
    }
}

/* Jacobian-vector product of the row softmax: dZ += P o (dP - <P, dP>). */
OR_EXPORT void or_softmax_rows_bwd(const double* P, const double* dP, int R, int Cc, double* dZ) {
    for (int r = 0; r < R; r++) {
        const double* p = P + (size_t)r * Cc;
        const double* dp = dP + (size_t)r * Cc;
        double dot = 0.0;
        for (int c = 0; c < Cc; c++) dot += p[c] * dp[c];
        for (int c = 0; c < Cc; c++) dZ[(size_t)r * Cc + c] += p[c] * (dp[c] - dot);
    }
}

/* CrossEntropy of probabilities ([TT] 三.2 probs.CrossEntropy(y)):
 *   loss = -(1/R) sum_r log P[r, y_r];  dP[r, y_r] += -dloss / (R P[r, y_r]). */
OR_EXPORT double or_xent_probs(const double* P, const int* y, int R, int Cc, double* dP, double dloss) {
    double s = 0.0;
    for (int r = 0; r < R; r++) {
        double pr = P[(size_t)r * Cc + y[r]];
        s -= log(pr);
        if (dP) dP[(size_t)r * Cc + y[r]] += -dloss / (R * pr);
    }
    return R > 0 ? s / R : 0.0;
}

/* The classifier of [TT] 八.5, on a fixed batch of R rows:
 *   h = gelu(x W1 + b1),  z = h W2 + b2,  p = softmax(z),  loss = CE(p, y),
 * then the gradients of W1 [nin,nh], b1 [nh], W2 [nh,nout], b2 [nout] and
 * SGD p -= lr g.  losses[s] is the loss of step s before its update.  With
 * grads != NULL the gradients of the last step are copied there (W1, b1,
 * W2, b2 in that order). */
OR_EXPORT void or_mlp_sgd(const double* x, const int* y, int R, int nin, int nh, int nout, double* W1, double* b1,
                          double* W2, double* b2, double lr, int steps, double* losses, double* grads) {
    const size_t n1 = (size_t)nin * nh, n2 = (size_t)nh * nout;
    double* a = (double*)calloc((size_t)R * nh, sizeof(double));   /* x W1 */
    double* u = (double*)calloc((size_t)R * nh, sizeof(double));   /* + b1 */
    double* h = (double*)calloc((size_t)R * nh, sizeof(double));   /* gelu */
    double* m = (double*)calloc((size_t)R * nout, sizeof(double)); /* h W2 */
    double* z = (double*)calloc((size_t)R * nout, sizeof(double)); /* + b2 */
    double* p = (double*)calloc((size_t)R * nout, sizeof(double));
    double* dp = (double*)calloc((size_t)R * nout, sizeof(double));
    double* dz = (double*)calloc((size_t)R * nout, sizeof(double));
    double* dh = (double*)calloc((size_t)R * nh, sizeof(double));
    double* du = (double*)calloc((size_t)R * nh, sizeof(double));
    double* gW1 = (double*)calloc(n1, sizeof(double));
    double* gb1 = (double*)calloc((size_t)nh, sizeof(double));
    double* gW2 = (double*)calloc(n2, sizeof(double));
    double* gb2 = (double*)calloc((size_t)nout, sizeof(double));
    for (int s = 0; s < steps; s++) {
        or_matmul(x, W1, R, nin, nh, a);
        or_add_row(a, b1, R, nh, u);
        or_gelu_fwd(u, (size_t)R * nh, h);
        or_matmul(h, W2, R, nh, nout, m);
        or_add_row(m, b2, R, nout, z);
        or_softmax_rows(z, R, nout, p);
        memset(dp, 0, sizeof(double) * (size_t)R * nout);
        memset(dz, 0, sizeof(double) * (size_t)R * nout);
        memset(dh, 0, sizeof(double) * (size_t)R * nh);
        memset(du, 0, sizeof(double) * (size_t)R * nh);
        memset(gW1, 0, sizeof(double) * n1);
        memset(gb1, 0, sizeof(double) * (size_t)nh);
        memset(gW2, 0, sizeof(double) * n2);
        memset(gb2, 0, sizeof(double) * (size_t)nout);
        double loss = or_xent_probs(p, y, R, nout, dp, 1.0);
        if (losses) losses[s] = loss;
        or_softmax_rows_bwd(p, dp, R, nout, dz);
        or_add_row_bwd(dz, R, nout, NULL, gb2);
        or_matmul_bwd(h, W2, dz, R, nh, nout, dh, gW2);
        or_gelu_bwd(u, dh, (size_t)R * nh, du);
        or_add_row_bwd(du, R, nh, NULL, gb1);
        or_matmul_bwd(x, W1, du, R, nin, nh, NULL, gW1);
        for (size_t i = 0; i < n1; i++) W1[i] -= lr * gW1[i];
        for (int i = 0; i < nh; i++) b1[i] -= lr * gb1[i];
        for (size_t i = 0; i < n2; i++) W2[i] -= lr * gW2[i];
        for (int i = 0; i < nout; i++) b2[i] -= lr * gb2[i];
    }
    if (grads && steps > 0) {
        memcpy(grads, gW1, sizeof(double) * n1);
        memcpy(grads + n1, gb1, sizeof(double) * (size_t)nh);
        memcpy(grads + n1 + nh, gW2, sizeof(double) * n2);
        memcpy(grads + n1 + nh + n2, gb2, sizeof(double) * (size_t)nout);
    }
    free(a); free(u); free(h); free(m); free(z); free(p); free(dp); free(dz); free(dh); free(du);
    free(gW1); free(gb1); free(gW2); free(gb2);
}

/* ------------------------------------------------------------------------ */
/* Scalar tape ([MCRAD] Values 的工作原理 / 操作 / 反向传播; [NPF] 4.3).      */
/* Nodes live in one growable pool (the arena replaces reference counting); */
/* handles are indices.  backward: depth-first topological sort with a      */
/* visited mark, seed grad = 1, reverse walk applying the chain rule.       */
/* ------------------------------------------------------------------------ */

enum { SV_LEAF = 0, SV_ADD, SV_MUL, SV_POW, SV_EXP, SV_LOG };

typedef struct {
    double data, grad, extra;
    int op, nprev, prev[2];
} ovalue;

static ovalue* sv_pool = NULL;
static int sv_n = 0, sv_cap = 0;

static int sv_new(double data, int op, int nprev, int p0, int p1, double extra) {
    if (sv_n == sv_cap) {
        sv_cap = sv_cap ? 2 * sv_cap : 256;
        sv_pool = (ovalue*)realloc(sv_pool, sizeof(ovalue) * (size_t)sv_cap);
    }
    ovalue* v = &sv_pool[sv_n];
    v->data = data; v->grad = 0.0; v->extra = extra; v->op = op;
    v->nprev = nprev; v->prev[0] = p0; v->prev[1] = p1;
    return sv_n++;
}

static int sv_ok(int i) { return i >= 0 && i < sv_n; }

OR_EXPORT void or_val_reset(void) { sv_n = 0; }
OR_EXPORT int or_val_leaf(double d) { return sv_new(d, SV_LEAF, 0, -1, -1, 0.0); }
OR_EXPORT int or_val_add(int a, int b) {
    if (!sv_ok(a) || !sv_ok(b)) return -1;
    return sv_new(sv_pool[a].data + sv_pool[b].data, SV_ADD, 2, a, b, 0.0);
}
OR_EXPORT int or_val_mul(int a, int b) {
    if (!sv_ok(a) || !sv_ok(b)) return -1;
    return sv_new(sv_pool[a].data * sv_pool[b].data, SV_MUL, 2, a, b, 0.0);
}
OR_EXPORT int or_val_pow(int a, double e) {
    if (!sv_ok(a)) return -1;
    return sv_new(pow(sv_pool[a].data, e), SV_POW, 1, a, -1, e);
}
OR_EXPORT int or_val_exp(int a) {
    if (!sv_ok(a)) return -1;
    return sv_new(exp(sv_pool[a].data), SV_EXP, 1, a, -1, 0.0);
}
OR_EXPORT int or_val_log(int a) {
    if (!sv_ok(a)) return -1;
    return sv_new(log(sv_pool[a].data), SV_LOG, 1, a, -1, 0.0);
}
OR_EXPORT double or_val_data(int a) { return sv_ok(a) ? sv_pool[a].data : NAN; }
OR_EXPORT double or_val_grad(int a) { return sv_ok(a) ? sv_pool[a].grad : NAN; }

/* Returns 0 on success, -1 on a bad root (as the microcrad page specifies). */
OR_EXPORT int or_val_backward(int root) {
    if (!sv_ok(root)) return -1;
    char* seen = (char*)calloc((size_t)sv_n, 1);
    int* order = (int*)malloc(sizeof(int) * (size_t)sv_n);
    int* stack = (int*)malloc(sizeof(int) * (size_t)sv_n * 3);
    int* state = (int*)calloc((size_t)sv_n, sizeof(int));
    int n_order = 0, sp = 0;
    /* iterative post-order DFS: a node is emitted after all of its operands */
    stack[sp++] = root;
    while (sp > 0) {
        int v = stack[sp - 1];
        if (!seen[v]) {
            seen[v] = 1;
            for (int i = sv_pool[v].nprev - 1; i >= 0; i--) {
                int p = sv_pool[v].prev[i];
                if (!seen[p]) stack[sp++] = p;
            }
        } else {
            sp--;
            if (!state[v]) {
                state[v] = 1;
                order[n_order++] = v;
            }
        }
    }
    for (int i = 0; i < sv_n; i++) sv_pool[i].grad = 0.0;
    sv_pool[root].grad = 1.0;
    for (int i = n_order - 1; i >= 0; i--) {
        ovalue* v = &sv_pool[order[i]];
        double g = v->grad;
        switch (v->op) {
        case SV_ADD:
            sv_pool[v->prev[0]].grad += g;
            sv_pool[v->prev[1]].grad += g;
            break;
        case SV_MUL:
            sv_pool[v->prev[0]].grad += g * sv_pool[v->prev[1]].data;
            sv_pool[v->prev[1]].grad += g * sv_pool[v->prev[0]].data;
            break;
        case SV_POW: {
            double b = sv_pool[v->prev[0]].data;
            sv_pool[v->prev[0]].grad += g * v->extra * pow(b, v->extra - 1.0);
            break;
        }
        case SV_EXP:
            sv_pool[v->prev[0]].grad += g * v->data;
            break;
        case SV_LOG:
            sv_pool[v->prev[0]].grad += g / sv_pool[v->prev[0]].data;
            break;
        default:
            break;
        }
    }
    free(seen); free(order); free(stack); free(state);
    return 0;
}

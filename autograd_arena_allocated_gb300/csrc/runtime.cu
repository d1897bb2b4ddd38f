// runtime.cu -- the native runtime behind include/tt.h and include/tt_ops.h:
// the context, its device arena, the host-side tape, the GPT-2 step built on
// that tape, AdamW, and the op-level entry points.
//
// Arena (tinytorch page, 三.1): one cudaMalloc per context; tensors are cut by
// bumping an offset (256-byte aligned); tt_ctx_reset rewinds the offset.  A
// 256-byte header at the start holds the device error flags and is never
// rewound.  Scratch needed by one kernel is bumped and released right after
// the launch (stream order guarantees the next user of that memory runs later).
//
// Tape (tinytorch 三.2-三.3, microcrad 反向传播): every forward op records its
// kind, input and output tensors, the parameters it read and what it saved.
// Backward walks the records in reverse record order -- a reverse topological
// order, so a tensor has received every contribution to its gradient before
// its producer's record runs.  Gradients of activations live in the arena:
// the first contribution allocates and overwrites, later ones accumulate
// (a residual branch reuses the buffer of the gradient flowing through it).
//
// The whole step can be run "dry": the same allocation sequence with no
// launches, which gives the exact arena requirement before anything runs.
#include "tt_internal.h"

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <unordered_set>

using namespace tt;

static constexpr uint64_t TT_MAGIC = 0x7474617265676e61ULL;  // live context
static constexpr uint64_t TT_DEAD = 0xdeaddeaddeaddeadULL;    // destroyed
static constexpr size_t ARENA_ALIGN = 256;
static constexpr size_t ARENA_HEADER = 256;  // flags live here

struct TapeTensor {
    void* data = nullptr;
    void* grad = nullptr;
    long long rows = 0, cols = 0;
    int producer = -1;       // record index
    int consumers = 0;
    int first_consumer = -1;  // record index of the first record that read it
    bool grad_is_pre = false;  // grad holds d/d(pre-activation) of a GELU producer
};

enum RecKind { R_EMBED, R_LN, R_LINEAR, R_ATTN, R_XENT };

struct Record {
    RecKind kind;
    int in = -1, out = -1, res = -1;
    void* pre = nullptr;  // GELU pre-activation (LINEAR with gelu)
    const void* W = nullptr;
    const void* b = nullptr;
    float* dW = nullptr;
    float* db = nullptr;
    const void* wpe = nullptr;
    float* dwpe = nullptr;
    float* mean = nullptr;
    float* rstd = nullptr;
    float* lse = nullptr;
    const int32_t* idx = nullptr;
    int M = 0, K = 0, N = 0;
    int B = 0, T = 0, H = 0, V = 0, maxT = 0;
    // LINEAR extras (tied LM head)
    int b_rows = 0, n_store = 0;
    long long ldy = 0;
    bool gelu = false;
    // LINEAR: the bias gradient was produced by the backward of a consumer of
    // this layer's output (it is the column sum of that output's gradient)
    bool db_fused = false;
};

// ------------------------------------------------------------------ profiling
enum ProfKind : int {
    PK_GEMM_FWD, PK_GEMM_DX, PK_GEMM_DW, PK_COLSUM, PK_ATTN_FWD, PK_ATTN_BWD, PK_LN_FWD,
    PK_LN_BWD, PK_XENT, PK_EMBED_FWD, PK_EMBED_BWD, PK_ADAMW, PK_CAST, PK_COUNT
};
static const char* const PROF_NAMES[PK_COUNT] = {
    "gemm_fwd", "gemm_dx", "gemm_dw", "colsum", "attn_fwd", "attn_bwd", "ln_fwd",
    "ln_bwd", "xent", "embed_fwd", "embed_bwd", "adamw", "cast"};

struct ProfEntry {
    int kind;
    double flops, bytes;
    cudaEvent_t e0, e1;
};

// A node of the generic tensor graph: its value and gradient in the arena,
// the op that makes it and its inputs (tinytorch 三.2).
enum GOp : int { G_LEAF = 0, G_MATMUL, G_ADD, G_ADD_ROW, G_MUL, G_GELU, G_SOFTMAX, G_XENT };
struct GNode {
    int op = G_LEAF;
    int type = TT_NODE_F32;
    int ndim = 0;
    int shape[4] = {1, 1, 1, 1};
    long long n = 0;
    void* data = nullptr;
    float* grad = nullptr;  // null for int32 nodes
    int in0 = -1, in1 = -1;
    int uses = 0;           // nodes that take this one as an input
};

struct tt_ctx {
    uint64_t magic = TT_MAGIC;
    int device = 0;
    char* arena = nullptr;
    size_t cap = 0, off = ARENA_HEADER, high = ARENA_HEADER;
    cudaStream_t stream = nullptr;
    uint64_t launches = 0;
    int num_sms = 148;
    int gemm_backend = 0;
    long long wait_cycles = 4000000000LL;  // bounded-wait limit of the tensor-core kernels
    bool has_model = false;
    tt_gpt2_config cfg{};
    bool dry = false;
    bool oom = false;
    std::vector<TapeTensor> tensors;
    std::vector<Record> tape;
    std::unordered_set<const float*> grad_written;
    float* loss_dev = nullptr;
    float* row_loss_dev = nullptr;
    std::string err;
    bool profiling = false;
    std::vector<ProfEntry> prof;
    std::vector<cudaEvent_t> event_pool;
    // the generic tensor graph (tt_graph.h): nodes made since the last reset
    std::vector<struct GNode> gnodes;
    uint32_t gepoch = 0;
    // step variants (tt_gpt2_step_ex): parameter gradients added to the
    // caller's buffers, and the device loss scale that seeds the backward
    bool accum_params = false;
    const float* loss_scale_dev = nullptr;
    // a recording of graph calls (tt_capture_begin / tt_capture_end / tt_replay)
    bool capturing = false;
    cudaStream_t cap_stream = nullptr, saved_stream = nullptr;
    cudaGraphExec_t recording = nullptr;
    uint64_t rec_launches = 0, cap_launches0 = 0;
};

// Brackets the launches of one op with events when profiling is on.
struct ProfScope {
    tt_ctx* c;
    int idx = -1;
    static cudaEvent_t take(tt_ctx* c) {
        if (!c->event_pool.empty()) {
            cudaEvent_t e = c->event_pool.back();
            c->event_pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        cudaEventCreate(&e);
        return e;
    }
    ProfScope(tt_ctx* c_, int kind, double flops, double bytes) : c(c_) {
        if (!c->profiling || c->dry || c->oom) return;
        ProfEntry e{kind, flops, bytes, take(c), take(c)};
        cudaEventRecord(e.e0, c->stream);
        c->prof.push_back(e);
        idx = (int)c->prof.size() - 1;
    }
    ~ProfScope() {
        if (idx >= 0) cudaEventRecord(c->prof[idx].e1, c->stream);
    }
};

// ------------------------------------------------------------------ helpers
static bool live(const tt_ctx* c) { return c && c->magic == TT_MAGIC; }

// Graph handles carry an 11-bit epoch, new for every context and every reset,
// so that a handle of an earlier epoch or of another context is refused.
static uint32_t next_graph_epoch() {
    static std::atomic<uint32_t> e{0};
    uint32_t v;
    do { v = (e.fetch_add(1) + 1) & 0x7FF; } while (v == 0);
    return v;
}

static tt_status fail(tt_ctx* c, tt_status s, const char* fmt, ...) {
    if (c) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        c->err = buf;
    }
    return s;
}

// Programmatic dependent launch for every kernel that supports it (each such
// kernel waits for its predecessor before touching global memory), unless
// TT_PDL=0 is in the environment (for comparisons).
static bool pdl_enabled() {
    static const bool on = [] {
        const char* e = getenv("TT_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

static Launch launch_of(tt_ctx* c) {
    Launch L;
    L.pdl = pdl_enabled();
    L.stream = c->stream;
    L.flags = (int*)c->arena;
    L.launches = &c->launches;
    L.dry = c->dry;
    L.gemm_backend = c->gemm_backend == 1 ? 1 : 0;
    L.no_pair = c->gemm_backend == 2;
    L.wait_cycles = c->wait_cycles;
    L.num_sms = c->num_sms;
    L.f16 = c->has_model && c->cfg.dtype == TT_FP16;
    return L;
}

// the op-level calls name their own dtype (never TT_FP16), whatever the model
static Launch op_launch(tt_ctx* c) {
    Launch L = launch_of(c);
    L.f16 = false;
    return L;
}

// Bump allocation; in dry mode only the offsets move.
static void* arena_alloc(tt_ctx* c, size_t bytes) {
    size_t at = (c->off + ARENA_ALIGN - 1) & ~(ARENA_ALIGN - 1);
    size_t end = at + ((bytes + ARENA_ALIGN - 1) & ~(ARENA_ALIGN - 1));
    if (end > c->cap) {
        c->oom = true;
        c->off = end;  // keep counting so that a dry run reports the full need
        c->high = std::max(c->high, end);
        return nullptr;
    }
    c->off = end;
    c->high = std::max(c->high, end);
    return c->dry ? (void*)(uintptr_t)(0x100000ull + at) : (void*)(c->arena + at);
}

static size_t esize(tt_dtype d) { return d == TT_FP32 ? 4 : 2; }

// record `rec` reads tensor t
static void add_consumer(tt_ctx* c, int t, int rec) {
    TapeTensor& x = c->tensors[t];
    if (x.first_consumer < 0) x.first_consumer = rec;
    x.consumers++;
}

static int new_tensor(tt_ctx* c, long long rows, long long cols, size_t elem) {
    TapeTensor t;
    t.rows = rows;
    t.cols = cols;
    t.data = arena_alloc(c, (size_t)(rows * cols) * elem);
    c->tensors.push_back(t);
    return (int)c->tensors.size() - 1;
}

// ------------------------------------------------------------------ GEMM dispatch
namespace tt {
size_t gemm_workspace_floats(const Launch& L, const GemmArgs& g) {
    if (L.gemm_backend == 0 && gemm_tc_eligible(g)) return gemm_tc_workspace_floats(L, g);
    return 0;
}

bool gemm(const Launch& L, const GemmArgs& g, float* ws, size_t ws_floats) {
    if (L.gemm_backend == 0 && gemm_tc_eligible(g)) return gemm_tc_launch(L, g, ws, ws_floats);
    gemm_simt_launch(L, g);
    return true;
}
}  // namespace tt

// run a GEMM with its split-K workspace bumped from the arena and released after
static bool run_gemm(tt_ctx* c, const GemmArgs& g, int kind) {
    const double es = g.in_bf16 ? 2.0 : 4.0;
    ProfScope ps(c, kind, 2.0 * g.M * g.N * (double)g.K,
                 es * ((double)g.M * g.K + (double)g.N * g.K) + (g.d_f32 ? 4.0 : es) * (double)g.M * g.N);
    Launch L = launch_of(c);
    size_t mark = c->off;
    size_t wsf = gemm_workspace_floats(L, g);
    float* ws = wsf ? (float*)arena_alloc(c, wsf * sizeof(float)) : nullptr;
    bool ok = c->oom ? c->dry : gemm(L, g, ws, wsf);
    c->off = mark;
    return ok;
}

// ------------------------------------------------------------------ forward ops (record + launch)
static int op_embed(tt_ctx* c, const void* wte, const void* wpe, float* dwte, float* dwpe,
                    const int32_t* tok, int B, int T) {
    const tt_gpt2_config& m = c->cfg;
    const bool bf = m.dtype != TT_FP32;  // 16-bit storage (bf16 or half)
    int out = new_tensor(c, (long long)B * T, m.C, esize(m.dtype));
    ProfScope ps(c, PK_EMBED_FWD, 0.0, 3.0 * B * T * m.C * esize(m.dtype) + 4.0 * B * T);
    if (!c->oom) launch_embed_fwd(launch_of(c), bf, wte, wpe, tok, c->tensors[out].data, B, T, m.C, m.V);
    Record r;
    r.kind = R_EMBED;
    r.out = out;
    r.W = wte;
    r.dW = dwte;
    r.wpe = wpe;
    r.dwpe = dwpe;
    r.idx = tok;
    r.B = B; r.T = T; r.N = m.C; r.V = m.V; r.maxT = m.maxT;
    c->tape.push_back(r);
    c->tensors[out].producer = (int)c->tape.size() - 1;
    return out;
}

static int op_layernorm(tt_ctx* c, int x, const void* w, const void* b, float* dw, float* db) {
    const tt_gpt2_config& m = c->cfg;
    const bool bf = m.dtype != TT_FP32;  // 16-bit storage (bf16 or half)
    const int M = (int)c->tensors[x].rows, C = m.C;
    int out = new_tensor(c, M, C, esize(m.dtype));
    float* mean = (float*)arena_alloc(c, (size_t)M * 4);
    float* rstd = (float*)arena_alloc(c, (size_t)M * 4);
    ProfScope ps(c, PK_LN_FWD, 0.0, 2.0 * M * C * esize(m.dtype) + 8.0 * M);
    if (!c->oom)
        launch_layernorm_fwd(launch_of(c), bf, c->tensors[x].data, w, b, c->tensors[out].data, mean,
                             rstd, M, C);
    Record r;
    r.kind = R_LN;
    r.in = x; r.out = out; r.W = w; r.b = b; r.dW = dw; r.db = db;
    r.mean = mean; r.rstd = rstd; r.M = M; r.N = C;
    c->tape.push_back(r);
    add_consumer(c, x, (int)c->tape.size() - 1);
    c->tensors[out].producer = (int)c->tape.size() - 1;
    return out;
}

// y = x W^T + b (+ residual) or gelu(x W^T + b)
static int op_linear(tt_ctx* c, int x, const void* W, const void* b, float* dW, float* db, int N,
                     int res, bool gelu, int b_rows = 0, int n_store = 0) {
    const tt_gpt2_config& m = c->cfg;
    const bool bf = m.dtype != TT_FP32;  // 16-bit storage (bf16 or half)
    const size_t es = esize(m.dtype);
    const int M = (int)c->tensors[x].rows, K = (int)c->tensors[x].cols;
    int out = new_tensor(c, M, N, es);
    void* pre = gelu ? arena_alloc(c, (size_t)M * N * es) : nullptr;
    if (!c->oom) {
        GemmArgs g;
        g.A = c->tensors[x].data; g.lda = K; g.a_kmajor = true;
        g.B = W; g.ldb = K; g.b_kmajor = true;
        g.M = M; g.N = N; g.K = K;
        g.b_rows = b_rows;
        g.in_bf16 = bf;
        g.in_f16 = m.dtype == TT_FP16;
        g.D = c->tensors[out].data; g.ldd = N; g.d_f32 = !bf;
        g.n_store = n_store;
        g.epi = gelu ? EPI_GELU : EPI_STORE;
        g.bias = b;
        g.residual = res >= 0 ? c->tensors[res].data : nullptr;
        g.aux = pre;
        if (!run_gemm(c, g, PK_GEMM_FWD)) c->err = "linear forward: GEMM launch failed";
    }
    Record r;
    r.kind = R_LINEAR;
    r.in = x; r.out = out; r.res = res; r.pre = pre;
    r.W = W; r.b = b; r.dW = dW; r.db = db;
    r.M = M; r.K = K; r.N = N; r.b_rows = b_rows; r.n_store = n_store; r.gelu = gelu;
    c->tape.push_back(r);
    add_consumer(c, x, (int)c->tape.size() - 1);
    if (res >= 0) add_consumer(c, res, (int)c->tape.size() - 1);
    c->tensors[out].producer = (int)c->tape.size() - 1;
    return out;
}

static int op_attention(tt_ctx* c, int qkv, int B, int T) {
    const tt_gpt2_config& m = c->cfg;
    const bool bf = m.dtype != TT_FP32;  // 16-bit storage (bf16 or half)
    const int M = B * T;
    int out = new_tensor(c, M, m.C, esize(m.dtype));
    float* lse = (float*)arena_alloc(c, (size_t)B * m.H * T * 4);
    // causal: QK^T and PV over the T(T+1)/2 unmasked pairs
    const double pairs = (double)B * m.H * T * (T + 1) / 2.0;
    ProfScope ps(c, PK_ATTN_FWD, 4.0 * pairs * (m.C / m.H),
                 (3.0 + 1.0) * M * m.C * esize(m.dtype) + 4.0 * B * m.H * T);
    if (!c->oom)
        launch_attention_fwd(launch_of(c), bf, c->tensors[qkv].data, c->tensors[out].data, lse, B, T,
                             m.C, m.H);
    Record r;
    r.kind = R_ATTN;
    r.in = qkv; r.out = out; r.lse = lse; r.B = B; r.T = T; r.H = m.H; r.N = m.C; r.M = M;
    c->tape.push_back(r);
    add_consumer(c, qkv, (int)c->tape.size() - 1);
    c->tensors[out].producer = (int)c->tape.size() - 1;
    return out;
}

// Cross entropy, forward and backward fused: the logits are replaced by their
// gradient in the same pass, so the logits tensor's gradient is its own buffer.
static void op_xent(tt_ctx* c, int z, const int32_t* targets, int V) {
    const tt_gpt2_config& m = c->cfg;
    const bool bf = m.dtype != TT_FP32;  // 16-bit storage (bf16 or half)
    const int M = (int)c->tensors[z].rows, ld = (int)c->tensors[z].cols;
    c->row_loss_dev = (float*)arena_alloc(c, (size_t)M * 4);
    c->loss_dev = (float*)arena_alloc(c, 4);
    ProfScope ps(c, PK_XENT, 0.0, 2.0 * M * ld * esize(m.dtype) + 8.0 * M);
    if (!c->oom)
        launch_xent(launch_of(c), bf, c->tensors[z].data, targets, c->row_loss_dev, c->loss_dev, M, V,
                    ld, 1.0f / (float)M, c->loss_scale_dev);
    Record r;
    r.kind = R_XENT;
    r.in = z; r.M = M; r.N = V; r.idx = targets;
    c->tape.push_back(r);
    add_consumer(c, z, (int)c->tape.size() - 1);
    c->tensors[z].grad = c->tensors[z].data;
}

// ------------------------------------------------------------------ backward
static bool first_write(tt_ctx* c, const float* p) {
    return c->grad_written.insert(p).second;
}

// gradient buffer of tensor t for writing: returns (pointer, accumulate?)
static void* grad_for_write(tt_ctx* c, int t, bool* accumulate) {
    TapeTensor& x = c->tensors[t];
    if (x.grad) { *accumulate = true; return x.grad; }
    const size_t es = esize(c->cfg.dtype);
    x.grad = arena_alloc(c, (size_t)(x.rows * x.cols) * es);
    *accumulate = false;
    return x.grad;
}

static tt_status backward_record(tt_ctx* c, int idx) {
    const Record& r = c->tape[idx];
    const tt_gpt2_config& m = c->cfg;
    const bool bf = m.dtype != TT_FP32;  // 16-bit storage (bf16 or half)
    Launch L = launch_of(c);
    switch (r.kind) {
    case R_XENT:
        return TT_OK;  // fused into the forward pass
    case R_LINEAR: {
        TapeTensor& y = c->tensors[r.out];
        if (!y.grad) return TT_OK;
        if (r.gelu && !y.grad_is_pre)
            return fail(c, TT_ERR, "tape: GELU output gradient was not produced by a linear input gradient");
        const void* dy = y.grad;  // for a GELU layer this is already d/d(pre)
        // residual input: the gradient passes through unchanged
        if (r.res >= 0) {
            TapeTensor& rt = c->tensors[r.res];
            if (rt.grad) return fail(c, TT_ERR, "tape: residual gradient already allocated");
            rt.grad = y.grad;
        }
        // input gradient dx = dy W (fused with GELU' when the input came from a GELU layer)
        {
            TapeTensor& xt = c->tensors[r.in];
            bool acc = false;
            Record* prod = xt.producer >= 0 ? &c->tape[xt.producer] : nullptr;
            const bool through_gelu = prod && prod->kind == R_LINEAR && prod->gelu && xt.consumers == 1;
            void* dx = grad_for_write(c, r.in, &acc);
            // Through the GELU, dx is the gradient of the GELU layer's
            // pre-activation, whose column sums are that layer's bias gradient:
            // the GEMM's epilogue forms them per 32-row slice (or, on paths
            // without that epilogue, one column-sum pass follows)
            float* cpart = nullptr;
            bool cdone = false;
            const size_t cmark = c->off;
            if (through_gelu && prod->db) {
                if (!first_write(c, prod->db)) return fail(c, TT_ERR, "tape: bias used twice");
                prod->db_fused = true;
                const size_t a = (size_t)gemm_colsum_rows(r.M) * r.K, b = colsum_scratch_floats(r.M, r.K);
                cpart = (float*)arena_alloc(c, (a > b ? a : b) * 4);
            }
            if (!c->oom) {
                GemmArgs g;
                g.A = dy; g.lda = r.N; g.a_kmajor = true;
                g.B = r.W; g.ldb = r.K; g.b_kmajor = false;
                g.M = r.M; g.N = r.K; g.K = r.N;
                g.k_valid = r.b_rows ? r.b_rows : 0;  // tied head: rows of wte beyond V are zero
                g.in_bf16 = bf;
                g.in_f16 = m.dtype == TT_FP16;
                g.D = dx; g.ldd = r.K; g.d_f32 = !bf;
                g.accumulate = acc;
                if (through_gelu) { g.epi = EPI_DGELU; g.aux = prod->pre; }
                g.colsum_part = cpart;
                g.colsum_done = &cdone;
                if (!run_gemm(c, g, PK_GEMM_DX)) return fail(c, TT_ERR_CUDA, "linear dx GEMM failed");
            }
            if (cpart) {
                ProfScope ps(c, PK_COLSUM, 0.0, cdone ? 4.0 * gemm_colsum_rows(r.M) * r.K
                                                      : (double)r.M * r.K * esize(m.dtype) + 4.0 * r.K);
                if (!c->oom) {
                    if (cdone) launch_sum_rows(L, cpart, gemm_colsum_rows(r.M), r.K, r.K, prod->db, nullptr,
                                               c->accum_params);
                    else launch_colsum(L, bf, dx, r.M, r.K, prod->db, cpart, c->accum_params);
                }
                c->off = cmark;
            }
            if (through_gelu) xt.grad_is_pre = true;
        }
        // weight and bias gradients (fp32, first write overwrites unless the step accumulates)
        {
            const bool accW = !first_write(c, r.dW) || c->accum_params;
            GemmArgs g;
            g.A = dy; g.lda = r.N; g.a_kmajor = false;
            g.B = c->tensors[r.in].data; g.ldb = r.K; g.b_kmajor = false;
            g.M = r.n_store ? std::min(r.n_store, r.b_rows ? r.b_rows : r.N) : r.N;
            g.a_rows = g.M;
            g.N = r.K; g.K = r.M;
            g.in_bf16 = bf;
            g.in_f16 = m.dtype == TT_FP16;
            g.D = r.dW; g.ldd = r.K; g.d_f32 = true;
            g.accumulate = accW;
            if (!c->oom && !run_gemm(c, g, PK_GEMM_DW)) return fail(c, TT_ERR_CUDA, "linear dW GEMM failed");
            if (r.db && !r.db_fused) {
                if (!first_write(c, r.db)) return fail(c, TT_ERR, "tape: bias used twice");
                size_t mark = c->off;
                float* s = (float*)arena_alloc(c, colsum_scratch_floats(r.M, r.N) * 4);
                ProfScope ps(c, PK_COLSUM, 0.0, (double)r.M * r.N * esize(m.dtype) + 4.0 * r.N);
                if (!c->oom) launch_colsum(L, bf, dy, r.M, r.N, r.db, s, c->accum_params);
                c->off = mark;
            }
        }
        return TT_OK;
    }
    case R_LN: {
        TapeTensor& y = c->tensors[r.out];
        if (!y.grad) return TT_OK;
        bool acc = false;
        void* dx = grad_for_write(c, r.in, &acc);
        if (!first_write(c, r.dW) || !first_write(c, r.db))
            return fail(c, TT_ERR, "tape: LayerNorm parameters used twice");
        // The input is complete once this LayerNorm has added its share when
        // this LayerNorm is its first consumer (reverse order: its last).  If
        // the input is the output of a linear layer with a bias, that bias's
        // gradient is the column sum of the finished gradient: the kernel
        // forms it on the way (no second pass over the gradient).
        Record* prod = nullptr;
        {
            const TapeTensor& xt = c->tensors[r.in];
            if (xt.first_consumer == idx && xt.producer >= 0) {
                Record& p = c->tape[xt.producer];
                if (p.kind == R_LINEAR && p.db && !p.gelu && p.out == r.in) prod = &p;
            }
        }
        size_t mark = c->off;
        float* s = (float*)arena_alloc(c, layernorm_bwd_scratch_floats(r.M, r.N) * 4);
        ProfScope ps(c, PK_LN_BWD, 0.0, (acc ? 4.0 : 3.0) * r.M * r.N * esize(m.dtype) + 8.0 * r.M);
        if (prod) {
            if (!first_write(c, prod->db)) return fail(c, TT_ERR, "tape: bias used twice");
            prod->db_fused = true;
        }
        if (!c->oom)
            launch_layernorm_bwd(L, bf, c->tensors[r.in].data, r.W, r.mean, r.rstd, y.grad, dx, r.dW, r.db, r.M,
                                 r.N, acc, s, c->accum_params, prod ? prod->db : nullptr);
        c->off = mark;
        return TT_OK;
    }
    case R_ATTN: {
        TapeTensor& y = c->tensors[r.out];
        if (!y.grad) return TT_OK;
        bool acc = false;
        void* dqkv = grad_for_write(c, r.in, &acc);
        if (acc) return fail(c, TT_ERR, "tape: attention input gradient already allocated");
        // qkv is the output of the qkv linear layer and attention its only
        // consumer: that layer's bias gradient, the column sums of dqkv, is
        // formed by the attention backward itself
        Record* prod = nullptr;
        {
            const TapeTensor& xt = c->tensors[r.in];
            if (xt.consumers == 1 && xt.producer >= 0) {
                Record& p = c->tape[xt.producer];
                if (p.kind == R_LINEAR && p.db && !p.gelu && p.out == r.in) prod = &p;
            }
        }
        if (prod) {
            if (!first_write(c, prod->db)) return fail(c, TT_ERR, "tape: bias used twice");
            prod->db_fused = true;
        }
        size_t mark = c->off;
        float* s = (float*)arena_alloc(c, attention_bwd_scratch_floats(r.B, r.T, r.N, r.H) * 4);
        // recompute QK^T, then dV, dP, dQ, dK: five products over the causal pairs
        const double pairs = (double)r.B * r.H * r.T * (r.T + 1) / 2.0;
        ProfScope ps(c, PK_ATTN_BWD, 10.0 * pairs * (r.N / r.H),
                     (3.0 + 2.0 + 3.0) * r.M * r.N * esize(m.dtype) + 4.0 * r.B * r.H * r.T);
        if (!c->oom)
            launch_attention_bwd(L, bf, c->tensors[r.in].data, y.data, r.lse, y.grad, dqkv, r.B, r.T,
                                 r.N, r.H, s, prod ? prod->db : nullptr, c->accum_params);
        c->off = mark;
        return TT_OK;
    }
    case R_EMBED: {
        TapeTensor& y = c->tensors[r.out];
        if (!y.grad) return TT_OK;
        if (first_write(c, r.dW) && !c->accum_params && !c->dry) {
            if (cudaMemsetAsync(r.dW, 0, (size_t)r.V * r.N * 4, c->stream) != cudaSuccess)
                return fail(c, TT_ERR_CUDA, "memset failed");
        }
        if (!first_write(c, r.dwpe)) return fail(c, TT_ERR, "tape: position table used twice");
        size_t mark = c->off;
        void* s = arena_alloc(c, embed_bwd_scratch_bytes(r.B * r.T, r.N));
        ProfScope ps(c, PK_EMBED_BWD, 0.0,
                     (double)r.B * r.T * r.N * (esize(m.dtype) + 8.0) + 4.0 * r.maxT * r.N);
        if (!c->oom)
            launch_embed_bwd(L, bf, y.grad, r.idx, r.dW, r.dwpe, r.B, r.T, r.N, r.V, r.maxT, s,
                             c->accum_params);
        c->off = mark;
        return TT_OK;
    }
    }
    return TT_OK;
}

static tt_status tape_backward(tt_ctx* c) {
    for (int i = (int)c->tape.size() - 1; i >= 0; i--) {
        tt_status s = backward_record(c, i);
        if (s != TT_OK) return s;
    }
    return TT_OK;
}

// ------------------------------------------------------------------ layout
static bool cfg_ok(const tt_gpt2_config* m) {
    if (!m || m->L < 0 || m->C <= 0 || m->H <= 0 || m->V <= 1 || m->maxT <= 0) return false;
    if (m->C % m->H || m->C % 64 || m->C > 1024 || m->V >= 65535 * 16) return false;
    if (m->dtype != TT_FP32 && m->dtype != TT_BF16 && m->dtype != TT_FP16) return false;
    const int hd = m->C / m->H;
    if (hd != 16 && hd != 32 && hd != 64) return false;
    if (m->dtype == TT_BF16 && hd != 64) return false;
    return true;
}

static int padded_vocab(int V) { return ((V + 127) / 128) * 128; }

struct Offsets {
    size_t wte, wpe, layers, per_layer, lnfw, lnfb, total;
    size_t sub[12];
};

static Offsets offsets_of(const tt_gpt2_config* m) {
    Offsets o{};
    const size_t C = (size_t)m->C;
    const size_t sizes[12] = {C, C, 3 * C * C, 3 * C, C * C, C, C, C, 4 * C * C, 4 * C, 4 * C * C, C};
    o.wte = 0;
    o.wpe = (size_t)m->V * C;
    o.layers = o.wpe + (size_t)m->maxT * C;
    size_t at = 0;
    for (int i = 0; i < 12; i++) { o.sub[i] = at; at += sizes[i]; }
    o.per_layer = at;
    o.lnfw = o.layers + (size_t)m->L * at;
    o.lnfb = o.lnfw + C;
    o.total = o.lnfb + C;
    return o;
}

// ------------------------------------------------------------------ the step
// The model's forward on the tape (tinytorch 三.6): returns the logits tensor
// [B*T, Vp].  grads may be NULL (no backward will follow); qkv, when given,
// receives each layer's qkv tensor.
static int gpt2_forward(tt_ctx* c, const void* params, float* grads, const int32_t* tok, int B, int T,
                        std::vector<int>* qkv_of_layer = nullptr) {
    const tt_gpt2_config& m = c->cfg;
    const size_t es = esize(m.dtype);
    const Offsets o = offsets_of(&m);
    auto P = [&](size_t off) -> const void* { return (const char*)params + off * es; };
    auto G = [&](size_t off) -> float* { return grads ? grads + off : nullptr; };
    const int C = m.C;
    const int Vp = padded_vocab(m.V);

    int x = op_embed(c, P(o.wte), P(o.wpe), G(o.wte), G(o.wpe), tok, B, T);
    for (int l = 0; l < m.L; l++) {
        const size_t base = o.layers + (size_t)l * o.per_layer;
        auto PL = [&](int i) { return P(base + o.sub[i]); };
        auto GL = [&](int i) { return G(base + o.sub[i]); };
        int h = op_layernorm(c, x, PL(0), PL(1), GL(0), GL(1));
        int qkv = op_linear(c, h, PL(2), PL(3), GL(2), GL(3), 3 * C, -1, false);
        if (qkv_of_layer) qkv_of_layer->push_back(qkv);
        int a = op_attention(c, qkv, B, T);
        int x1 = op_linear(c, a, PL(4), PL(5), GL(4), GL(5), C, x, false);
        int h2 = op_layernorm(c, x1, PL(6), PL(7), GL(6), GL(7));
        int g = op_linear(c, h2, PL(8), PL(9), GL(8), GL(9), 4 * C, -1, true);
        x = op_linear(c, g, PL(10), PL(11), GL(10), GL(11), C, x1, false);
    }
    int hf = op_layernorm(c, x, P(o.lnfw), P(o.lnfb), G(o.lnfw), G(o.lnfb));
    // tied LM head: logits[M, Vp] = hf wte^T; wte rows >= V read as zero
    return op_linear(c, hf, P(o.wte), nullptr, G(o.wte), nullptr, Vp, -1, false, m.V, Vp);
}

static tt_status gpt2_forward_backward(tt_ctx* c, const void* params, float* grads,
                                       const int32_t* tok, const int32_t* tgt, int B, int T) {
    int z = gpt2_forward(c, params, grads, tok, B, T);
    op_xent(c, z, tgt, c->cfg.V);
    if (c->oom) return TT_ERR_ARENA_OOM;
    return tape_backward(c);
}

// ------------------------------------------------------------------ greedy generation
// Prefill: the forward over the prompt, whose qkv tensors fill the key/value
// cache, and the greedy token after the prompt.  Then one decode step per new
// token: the newest token through every layer (its key and value appended to
// the cache, its query against keys 0..pos) and the greedy choice from its
// logits.  Tokens live in a device buffer [B, Tp + n_new]; nothing returns to
// the host until the end.  The decode kernels read the position from device
// memory and the step advances it, so every step launches the same kernels
// with the same arguments: the first step runs eagerly and the rest replay it
// as a CUDA graph.
static tt_status gpt2_generate(tt_ctx* c, const void* params, const int32_t* prompt_dev, int B, int Tp, int n_new,
                               int32_t* tokbuf) {
    const tt_gpt2_config& m = c->cfg;
    const bool bf = m.dtype == TT_BF16;
    const size_t es = esize(m.dtype);
    const Offsets o = offsets_of(&m);
    auto P = [&](size_t off) -> const void* { return (const char*)params + off * es; };
    const int C = m.C, Vp = padded_vocab(m.V), Ttot = Tp + n_new;
    const int max_keys = Ttot - 1;  // keys seen by the last decode step
    Launch L = launch_of(c);
    // the cache: per layer [B, maxT, 2C]
    const size_t layer_cache = (size_t)B * m.maxT * 2 * C * es;
    char* cache = (char*)arena_alloc(c, layer_cache * (size_t)m.L);
    int* pos_dev = (int*)arena_alloc(c, sizeof(int));
    int* counters = (int*)arena_alloc(c, (size_t)B * m.H * sizeof(int));
    float* part = (float*)arena_alloc(c, decode_attn_scratch_floats(B, m.H, max_keys) * sizeof(float));
    const int nct = skinny_pick_ctas(m.V);
    auto* keys = (unsigned long long*)arena_alloc(c, (size_t)B * nct * sizeof(unsigned long long));
    // one set of decode-step tensors, reused by every layer and step
    auto buf = [&](int cols) { return arena_alloc(c, (size_t)B * cols * es); };
    void* xa = buf(C);
    void* xb = buf(C);
    void* h = buf(C);
    void* qkv = buf(3 * C);
    void* att = buf(C);
    void* x1 = buf(C);
    void* u = buf(4 * C);
    void* g = buf(4 * C);
    void* zl = buf(Vp);
    float* mean = (float*)arena_alloc(c, (size_t)B * 4);
    float* rstd = (float*)arena_alloc(c, (size_t)B * 4);
    // prefill
    std::vector<int> qkv_ids;
    int z = gpt2_forward(c, params, nullptr, prompt_dev, B, Tp, &qkv_ids);
    if (c->oom) return TT_ERR_ARENA_OOM;
    for (int l = 0; l < m.L; l++)
        if (!launch_kv_fill(L, bf, c->tensors[qkv_ids[l]].data, cache + layer_cache * l, B, Tp, C, 0, m.maxT))
            return fail(c, TT_ERR_ARG, "generate: sequence longer than maxT");
    launch_argmax(L, bf, (const char*)c->tensors[z].data + (size_t)(Tp - 1) * Vp * es, (long long)Tp * Vp, B, m.V,
                  tokbuf, Ttot, Tp, nullptr);
    const int n_steps = n_new - 1;
    if (n_steps <= 0) return TT_OK;
    if (!L.dry && cudaMemsetAsync(counters, 0, (size_t)B * m.H * sizeof(int), c->stream) != cudaSuccess)
        return fail(c, TT_ERR_CUDA, "generate: counter reset failed");
    launch_set_int(L, pos_dev, Tp);

    // one decode step: the token at *pos_dev gives the one at *pos_dev + 1
    const size_t mark = c->off;
    auto step = [&]() -> tt_status {
        c->off = mark;
        Launch S = launch_of(c);
        S.pdl = true;
        auto linear = [&](const void* in, int K, const void* W, const void* bias, int N, void* out, const void* res,
                          void* pre) -> bool {
            // a few rows: the weight-streaming skinny GEMM
            if (launch_gemm_skinny(S, bf, in, W, bias, res, out, pre, B, N, K, N, N, pre != nullptr, nullptr))
                return true;
            GemmArgs ga;
            ga.A = in; ga.lda = K; ga.a_kmajor = true;
            ga.B = W; ga.ldb = K; ga.b_kmajor = true;
            ga.M = B; ga.N = N; ga.K = K;
            ga.in_bf16 = bf;
            ga.D = out; ga.ldd = N; ga.d_f32 = !bf;
            ga.epi = pre ? EPI_GELU : EPI_STORE;
            ga.bias = bias;
            ga.residual = res;
            ga.aux = pre;
            return run_gemm(c, ga, PK_GEMM_FWD);
        };
        // LayerNorm then a linear layer: one launch when the skinny GEMM takes the LayerNorm
        auto ln_linear = [&](const void* xin, const void* lw, const void* lb, const void* W, const void* bias, int N,
                             void* out, void* pre) -> bool {
            if (bf && launch_gemm_skinny(S, bf, xin, W, bias, nullptr, out, pre, B, N, C, N, N, pre != nullptr,
                                         nullptr, lw, lb))
                return true;
            launch_layernorm_fwd(S, bf, xin, lw, lb, h, mean, rstd, B, C);
            return linear(h, C, W, bias, N, out, nullptr, pre);
        };
        void* x = xa;
        void* x2 = xb;
        launch_embed_at(S, bf, P(o.wte), P(o.wpe), tokbuf, Ttot, pos_dev, x, B, C, m.V);
        for (int l = 0; l < m.L; l++) {
            const size_t base = o.layers + (size_t)l * o.per_layer;
            auto PL = [&](int i) { return P(base + o.sub[i]); };
            if (!ln_linear(x, PL(0), PL(1), PL(2), PL(3), 3 * C, qkv, nullptr)) return fail(c, TT_ERR_CUDA, "generate: GEMM");
            if (!launch_decode_attn(S, bf, qkv, cache + layer_cache * l, att, B, m.H, C, pos_dev, max_keys, m.maxT,
                                    part, counters))
                return fail(c, TT_ERR_ARG, "generate: attention shape not supported");
            if (!linear(att, C, PL(4), PL(5), C, x1, x, nullptr)) return fail(c, TT_ERR_CUDA, "generate: GEMM");
            if (!ln_linear(x1, PL(6), PL(7), PL(8), PL(9), 4 * C, g, u)) return fail(c, TT_ERR_CUDA, "generate: GEMM");
            if (!linear(g, 4 * C, PL(10), PL(11), C, x2, x1, nullptr)) return fail(c, TT_ERR_CUDA, "generate: GEMM");
            std::swap(x, x2);
        }
        // final LayerNorm (its own launch: folded into the LM head it would be
        // redone by each of that GEMM's thousands of CTAs), then the tied LM head
        // over the V real rows of wte, which also advances the position
        launch_layernorm_fwd(S, bf, x, P(o.lnfw), P(o.lnfb), h, mean, rstd, B, C);
        if (bf && launch_gemm_skinny_pick(S, h, P(o.wte), B, m.V, C, keys, pos_dev)) {
            launch_pick(S, keys, nct, B, tokbuf, Ttot, pos_dev);
            return TT_OK;
        }
        if (!launch_gemm_skinny(S, bf, h, P(o.wte), nullptr, nullptr, zl, nullptr, B, m.V, C, Vp, m.V, false,
                                pos_dev)) {
            GemmArgs ga;
            ga.A = h; ga.lda = C; ga.a_kmajor = true;
            ga.B = P(o.wte); ga.ldb = C; ga.b_kmajor = true;
            ga.M = B; ga.N = Vp; ga.K = C;
            ga.b_rows = m.V;
            ga.in_bf16 = bf;
            ga.D = zl; ga.ldd = Vp; ga.d_f32 = !bf;
            if (!run_gemm(c, ga, PK_GEMM_FWD)) return fail(c, TT_ERR_CUDA, "generate: LM head GEMM");
            launch_add_int(S, pos_dev, 1);
        }
        launch_argmax(S, bf, zl, Vp, B, m.V, tokbuf, Ttot, 0, pos_dev);
        return TT_OK;
    };

    tt_status st = step();
    if (st != TT_OK || c->oom || L.dry || n_steps == 1) return c->oom ? TT_ERR_ARENA_OOM : st;
    // capture the step once (its kernels go to a private stream while it is
    // recorded) and replay it for the remaining positions
    int done = 1;
    cudaStream_t cap = nullptr;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) == cudaSuccess) {
        cudaStream_t own = c->stream;
        const uint64_t n0 = c->launches;
        c->stream = cap;
        if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
            st = step();
            if (cudaStreamEndCapture(cap, &graph) != cudaSuccess) graph = nullptr;
        }
        c->stream = own;
        const uint64_t nodes = c->launches - n0;
        c->launches = n0;
        if (st != TT_OK) {
            if (graph) cudaGraphDestroy(graph);
            cudaStreamDestroy(cap);
            return st;
        }
        if (graph && cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess) {
            for (; done < n_steps; done++) {
                if (cudaGraphLaunch(exec, c->stream) != cudaSuccess) break;
                c->launches += nodes;
            }
        }
        cudaGetLastError();  // a failed capture leaves the eager steps below
        if (exec) {
            cudaStreamSynchronize(c->stream);
            cudaGraphExecDestroy(exec);
        }
        if (graph) cudaGraphDestroy(graph);
        cudaStreamDestroy(cap);
    } else {
        cudaGetLastError();
    }
    for (; done < n_steps; done++) {
        st = step();
        if (st != TT_OK) return st;
    }
    return TT_OK;
}

static void begin_step(tt_ctx* c) {
    c->tensors.clear();
    c->tape.clear();
    c->grad_written.clear();
    c->oom = false;
}

static bool is_host_pointer(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeUnregistered;
}

// ------------------------------------------------------------------ C ABI
extern "C" {

tt_status tt_ctx_create(size_t arena_bytes, tt_ctx** out) {
    if (!out) return TT_ERR_ARG;
    *out = nullptr;
    if (arena_bytes == 0) return TT_ERR_ARG;
    tt_ctx* c = new tt_ctx();
    c->gepoch = next_graph_epoch();
    c->cap = arena_bytes + ARENA_HEADER;
    if (cudaGetDevice(&c->device) != cudaSuccess) { delete c; return TT_ERR_CUDA; }
    cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (cudaMalloc((void**)&c->arena, c->cap) != cudaSuccess) {
        cudaGetLastError();
        delete c;
        return TT_ERR_CUDA;
    }
    if (cudaMemset(c->arena, 0, ARENA_HEADER) != cudaSuccess) {
        cudaFree(c->arena);
        delete c;
        return TT_ERR_CUDA;
    }
    *out = c;
    return TT_OK;
}

// The handle's small host shell is kept (poisoned) rather than freed, so that
// a later call through a stale handle is detected instead of reading freed memory.
void tt_ctx_destroy(tt_ctx* c) {
    if (!live(c)) return;
    c->magic = TT_DEAD;
    if (c->capturing) {
        cudaGraph_t g = nullptr;
        cudaStreamEndCapture(c->cap_stream, &g);
        if (g) cudaGraphDestroy(g);
        c->stream = c->saved_stream;
        c->capturing = false;
    }
    cudaStreamSynchronize(c->stream);
    if (c->recording) cudaGraphExecDestroy(c->recording);
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
    c->recording = nullptr;
    c->cap_stream = nullptr;
    cudaGetLastError();
    cudaFree(c->arena);
    c->arena = nullptr;
    c->cap = 0;
    std::vector<TapeTensor>().swap(c->tensors);
    std::vector<Record>().swap(c->tape);
    std::unordered_set<const float*>().swap(c->grad_written);
    std::string().swap(c->err);
    for (ProfEntry& e : c->prof) { cudaEventDestroy(e.e0); cudaEventDestroy(e.e1); }
    for (cudaEvent_t e : c->event_pool) cudaEventDestroy(e);
    std::vector<ProfEntry>().swap(c->prof);
    std::vector<cudaEvent_t>().swap(c->event_pool);
}

tt_status tt_ctx_set_stream(tt_ctx* c, void* stream) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    c->stream = (cudaStream_t)stream;
    return TT_OK;
}

tt_status tt_ctx_set_model(tt_ctx* c, const tt_gpt2_config* m) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (!cfg_ok(m)) return fail(c, TT_ERR_ARG, "invalid model config");
    c->cfg = *m;
    c->has_model = true;
    return TT_OK;
}

tt_status tt_ctx_set_gemm_backend(tt_ctx* c, int backend) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (backend < 0 || backend > 2) return fail(c, TT_ERR_ARG, "backend must be 0, 1 or 2");
    c->gemm_backend = backend;
    return TT_OK;
}

tt_status tt_ctx_set_wait_limit(tt_ctx* c, long long cycles) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    c->wait_cycles = cycles > 0 ? cycles : 4000000000LL;
    return TT_OK;
}

tt_status tt_ctx_reset(tt_ctx* c) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (c->capturing) return fail(c, TT_ERR_STATE, "reset while recording");
    if (c->recording) {  // freed once any replay in flight completes
        cudaGraphExecDestroy(c->recording);
        c->recording = nullptr;
    }
    c->off = ARENA_HEADER;
    begin_step(c);
    c->loss_dev = c->row_loss_dev = nullptr;
    c->gnodes.clear();
    c->gepoch = next_graph_epoch();
    if (cudaMemsetAsync(c->arena, 0, FLAG_COUNT * sizeof(int), c->stream) != cudaSuccess)
        return fail(c, TT_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(cudaGetLastError()));
    return TT_OK;
}

tt_status tt_ctx_sync(tt_ctx* c) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (c->capturing) return fail(c, TT_ERR_STATE, "sync while recording");
    int flags[FLAG_COUNT];
    if (cudaMemcpyAsync(flags, c->arena, sizeof flags, cudaMemcpyDeviceToHost, c->stream) != cudaSuccess ||
        cudaStreamSynchronize(c->stream) != cudaSuccess)
        return fail(c, TT_ERR_CUDA, "sync: %s", cudaGetErrorString(cudaGetLastError()));
    if (flags[FLAG_TIMEOUT])
        return fail(c, TT_ERR_TIMEOUT, "a device-side wait timed out (site 0x%x)", (unsigned)flags[FLAG_SITE]);
    if (flags[FLAG_BAD_TOKEN]) return fail(c, TT_ERR_ARG, "token id out of range");
    if (flags[FLAG_NONFINITE]) return fail(c, TT_ERR_NONFINITE, "non-finite loss");
    return TT_OK;
}

tt_status tt_ctx_set_profiling(tt_ctx* c, int on) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    c->profiling = on != 0;
    return TT_OK;
}

int tt_ctx_profile_read(tt_ctx* c, tt_op_profile* rows, int max_rows) {
    if (!live(c)) return TT_ERR_STALE;
    if (cudaStreamSynchronize(c->stream) != cudaSuccess) {
        fail(c, TT_ERR_CUDA, "profile: %s", cudaGetErrorString(cudaGetLastError()));
        return TT_ERR_CUDA;
    }
    tt_op_profile agg[PK_COUNT];
    memset(agg, 0, sizeof agg);
    for (const ProfEntry& e : c->prof) {
        float ms = 0.0f;
        cudaEventElapsedTime(&ms, e.e0, e.e1);
        tt_op_profile& a = agg[e.kind];
        a.calls++;
        a.ms += ms;
        a.flops += e.flops;
        a.bytes += e.bytes;
        c->event_pool.push_back(e.e0);
        c->event_pool.push_back(e.e1);
    }
    c->prof.clear();
    int n = 0;
    for (int k = 0; k < PK_COUNT; k++) {
        if (!agg[k].calls) continue;
        if (rows && n < max_rows) {
            rows[n] = agg[k];
            snprintf(rows[n].name, sizeof rows[n].name, "%s", PROF_NAMES[k]);
        }
        n++;
    }
    cudaGetLastError();
    return rows ? std::min(n, max_rows) : n;
}

size_t tt_ctx_arena_capacity(const tt_ctx* c) { return live(c) ? c->cap - ARENA_HEADER : 0; }
size_t tt_ctx_arena_used(const tt_ctx* c) { return live(c) ? c->off - ARENA_HEADER : 0; }
size_t tt_ctx_arena_high_water(const tt_ctx* c) { return live(c) ? c->high - ARENA_HEADER : 0; }
uint64_t tt_ctx_launch_count(const tt_ctx* c) { return live(c) ? c->launches : 0; }

const char* tt_last_error(const tt_ctx* c) {
    if (!c) return "NULL context";
    if (!live(c)) return "stale context";
    return c->err.c_str();
}

size_t tt_gpt2_num_params(const tt_gpt2_config* m) {
    if (!cfg_ok(m)) return 0;
    return offsets_of(m).total;
}

tt_status tt_gpt2_param_offset(const tt_gpt2_config* m, int layer, int which, size_t* off,
                               size_t* numel) {
    if (!cfg_ok(m) || !off || !numel) return TT_ERR_ARG;
    const Offsets o = offsets_of(m);
    const size_t C = (size_t)m->C;
    switch (which) {
    case 0: *off = o.wte; *numel = (size_t)m->V * C; return TT_OK;
    case 1: *off = o.wpe; *numel = (size_t)m->maxT * C; return TT_OK;
    case 14: *off = o.lnfw; *numel = C; return TT_OK;
    case 15: *off = o.lnfb; *numel = C; return TT_OK;
    default: break;
    }
    if (which < 2 || which > 13 || layer < 0 || layer >= m->L) return TT_ERR_ARG;
    const int i = which - 2;
    *off = o.layers + (size_t)layer * o.per_layer + o.sub[i];
    *numel = (i + 1 < 12 ? o.sub[i + 1] : o.per_layer) - o.sub[i];
    return TT_OK;
}

size_t tt_gpt2_arena_bytes(const tt_gpt2_config* m, int B, int T) {
    if (!cfg_ok(m) || B <= 0 || T <= 0 || T > m->maxT) return 0;
    tt_ctx c;
    c.cap = (size_t)-1 / 2;
    c.cfg = *m;
    c.has_model = true;
    c.dry = true;
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
        c.num_sms = sms;
    else
        cudaGetLastError();
    const size_t M = (size_t)B * T;
    arena_alloc(&c, M * 4);  // staged tokens (host inputs)
    arena_alloc(&c, M * 4);  // staged targets
    gpt2_forward_backward(&c, (const void*)(uintptr_t)0x1000, (float*)(uintptr_t)0x1000,
                          (const int32_t*)(uintptr_t)0x1000, (const int32_t*)(uintptr_t)0x1000, B, T);
    c.magic = TT_DEAD;
    return c.high - ARENA_HEADER;
}

tt_status tt_gpt2_step(tt_ctx* c, const void* params, float* grads, const int32_t* tokens,
                       const int32_t* targets, int B, int T, float* loss) {
    return tt_gpt2_step_ex(c, params, grads, tokens, targets, B, T, 0, nullptr, loss);
}

tt_status tt_gpt2_step_ex(tt_ctx* c, const void* params, float* grads, const int32_t* tokens,
                          const int32_t* targets, int B, int T, int flags, const float* loss_scale, float* loss) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (c->capturing) return fail(c, TT_ERR_STATE, "GPT-2 calls cannot be recorded");
    if (!c->has_model) return fail(c, TT_ERR_STATE, "tt_ctx_set_model was not called");
    if (!params || !grads || !tokens || !targets)
        return fail(c, TT_ERR_ARG, "NULL parameter, gradient or token pointer");
    if (B <= 0 || T <= 0 || T > c->cfg.maxT)
        return fail(c, TT_ERR_ARG, "bad batch shape B=%d T=%d (maxT=%d)", B, T, c->cfg.maxT);
    const size_t M = (size_t)B * T;
    // exact plan first: nothing is launched if it does not fit
    {
        const size_t need = tt_gpt2_arena_bytes(&c->cfg, B, T);
        const size_t at = (c->off + ARENA_ALIGN - 1) & ~(ARENA_ALIGN - 1);
        if (need == 0 || at + need > c->cap)
            return fail(c, TT_ERR_ARENA_OOM, "arena too small: step needs %zu bytes, %zu free", need,
                        c->cap > at ? c->cap - at : (size_t)0);
    }
    begin_step(c);
    // host token buffers are staged into the arena
    const int32_t* tok = tokens;
    const int32_t* tgt = targets;
    int32_t* st_tok = (int32_t*)arena_alloc(c, M * 4);
    int32_t* st_tgt = (int32_t*)arena_alloc(c, M * 4);
    if (is_host_pointer(tokens)) {
        if (cudaMemcpyAsync(st_tok, tokens, M * 4, cudaMemcpyHostToDevice, c->stream) != cudaSuccess)
            return fail(c, TT_ERR_CUDA, "token copy failed");
        tok = st_tok;
    }
    if (is_host_pointer(targets)) {
        if (cudaMemcpyAsync(st_tgt, targets, M * 4, cudaMemcpyHostToDevice, c->stream) != cudaSuccess)
            return fail(c, TT_ERR_CUDA, "target copy failed");
        tgt = st_tgt;
    }
    if (flags & ~TT_STEP_ACCUMULATE) return fail(c, TT_ERR_ARG, "unknown step flags 0x%x", (unsigned)flags);
    c->accum_params = (flags & TT_STEP_ACCUMULATE) != 0;
    c->loss_scale_dev = loss_scale;
    tt_status s = gpt2_forward_backward(c, params, grads, tok, tgt, B, T);
    c->accum_params = false;
    c->loss_scale_dev = nullptr;
    if (s != TT_OK) {
        if (s == TT_ERR_ARENA_OOM) return fail(c, s, "arena exhausted during the step");
        return s;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(c, TT_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    if (loss) {
        if (cudaMemcpyAsync(loss, c->loss_dev, 4, cudaMemcpyDeviceToHost, c->stream) != cudaSuccess)
            return fail(c, TT_ERR_CUDA, "loss copy failed");
        return tt_ctx_sync(c);
    }
    return TT_OK;
}

// Token inputs may be host or device buffers; host ones are staged into the arena.
static const int32_t* stage_tokens(tt_ctx* c, const int32_t* tokens, size_t n, tt_status* st) {
    int32_t* dst = (int32_t*)arena_alloc(c, n * 4);
    *st = TT_OK;
    if (c->oom || c->dry || !is_host_pointer(tokens)) return c->dry ? dst : tokens;
    if (cudaMemcpyAsync(dst, tokens, n * 4, cudaMemcpyHostToDevice, c->stream) != cudaSuccess) {
        *st = fail(c, TT_ERR_CUDA, "token copy failed");
        return nullptr;
    }
    return dst;
}

tt_status tt_gpt2_eval(tt_ctx* c, const void* params, const int32_t* tokens, const int32_t* targets, int B, int T,
                       float* loss) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (c->capturing) return fail(c, TT_ERR_STATE, "GPT-2 calls cannot be recorded");
    if (!c->has_model) return fail(c, TT_ERR_STATE, "tt_ctx_set_model was not called");
    if (!params || !tokens || !targets) return fail(c, TT_ERR_ARG, "NULL parameter or token pointer");
    if (B <= 0 || T <= 0 || T > c->cfg.maxT)
        return fail(c, TT_ERR_ARG, "bad batch shape B=%d T=%d (maxT=%d)", B, T, c->cfg.maxT);
    {
        const size_t need = tt_gpt2_arena_bytes(&c->cfg, B, T);
        const size_t at = (c->off + ARENA_ALIGN - 1) & ~(ARENA_ALIGN - 1);
        if (need == 0 || at + need > c->cap)
            return fail(c, TT_ERR_ARENA_OOM, "arena too small: evaluation needs %zu bytes, %zu free", need,
                        c->cap > at ? c->cap - at : (size_t)0);
    }
    begin_step(c);
    const size_t M = (size_t)B * T;
    tt_status st;
    const int32_t* tok = stage_tokens(c, tokens, M, &st);
    if (st != TT_OK) return st;
    const int32_t* tgt = stage_tokens(c, targets, M, &st);
    if (st != TT_OK) return st;
    int z = gpt2_forward(c, params, nullptr, tok, B, T);
    op_xent(c, z, tgt, c->cfg.V);
    if (c->oom) return fail(c, TT_ERR_ARENA_OOM, "arena exhausted during evaluation");
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(c, TT_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    if (loss) {
        if (cudaMemcpyAsync(loss, c->loss_dev, 4, cudaMemcpyDeviceToHost, c->stream) != cudaSuccess)
            return fail(c, TT_ERR_CUDA, "loss copy failed");
        return tt_ctx_sync(c);
    }
    return TT_OK;
}

size_t tt_gpt2_generate_arena_bytes(const tt_gpt2_config* m, int B, int T_prompt, int n_new) {
    if (!cfg_ok(m) || m->dtype == TT_FP16 || B <= 0 || T_prompt <= 0 || n_new < 0 || T_prompt + n_new > m->maxT)
        return 0;
    tt_ctx c;
    c.cap = (size_t)-1 / 2;
    c.cfg = *m;
    c.has_model = true;
    c.dry = true;
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
        c.num_sms = sms;
    else
        cudaGetLastError();
    arena_alloc(&c, (size_t)B * T_prompt * 4);              // staged prompt
    arena_alloc(&c, (size_t)B * (T_prompt + n_new) * 4);    // token buffer
    if (n_new > 0)
        gpt2_generate(&c, (const void*)(uintptr_t)0x1000, (const int32_t*)(uintptr_t)0x1000, B, T_prompt, n_new,
                      (int32_t*)(uintptr_t)0x1000);
    c.magic = TT_DEAD;
    return c.high - ARENA_HEADER;
}

tt_status tt_gpt2_generate(tt_ctx* c, const void* params, const int32_t* prompt, int B, int T_prompt, int n_new,
                           int32_t* out) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (c->capturing) return fail(c, TT_ERR_STATE, "GPT-2 calls cannot be recorded");
    if (!c->has_model) return fail(c, TT_ERR_STATE, "tt_ctx_set_model was not called");
    if (c->cfg.dtype == TT_FP16) return fail(c, TT_ERR_ARG, "generation takes a TT_FP32 or TT_BF16 model");
    if (!params || !prompt || !out) return fail(c, TT_ERR_ARG, "NULL parameter, prompt or output pointer");
    if (B <= 0 || T_prompt <= 0 || n_new < 0 || T_prompt + n_new > c->cfg.maxT)
        return fail(c, TT_ERR_ARG, "bad generation shape B=%d prompt=%d new=%d (maxT=%d)", B, T_prompt, n_new,
                    c->cfg.maxT);
    {
        const size_t need = tt_gpt2_generate_arena_bytes(&c->cfg, B, T_prompt, n_new);
        const size_t at = (c->off + ARENA_ALIGN - 1) & ~(ARENA_ALIGN - 1);
        if (need == 0 || at + need > c->cap)
            return fail(c, TT_ERR_ARENA_OOM, "arena too small: generation needs %zu bytes, %zu free", need,
                        c->cap > at ? c->cap - at : (size_t)0);
    }
    begin_step(c);
    const int Ttot = T_prompt + n_new;
    tt_status st;
    const int32_t* pr = stage_tokens(c, prompt, (size_t)B * T_prompt, &st);
    if (st != TT_OK) return st;
    int32_t* tokbuf = (int32_t*)arena_alloc(c, (size_t)B * Ttot * 4);
    if (c->oom) return fail(c, TT_ERR_ARENA_OOM, "arena exhausted during generation");
    // the prompt opens each row of the token buffer
    if (cudaMemcpy2DAsync(tokbuf, (size_t)Ttot * 4, pr, (size_t)T_prompt * 4, (size_t)T_prompt * 4, (size_t)B,
                          cudaMemcpyDeviceToDevice, c->stream) != cudaSuccess)
        return fail(c, TT_ERR_CUDA, "prompt copy failed");
    if (n_new > 0) {
        st = gpt2_generate(c, params, pr, B, T_prompt, n_new, tokbuf);
        if (st != TT_OK) return st == TT_ERR_ARENA_OOM ? fail(c, st, "arena exhausted during generation") : st;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(c, TT_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    if (cudaMemcpyAsync(out, tokbuf, (size_t)B * Ttot * 4, cudaMemcpyDefault, c->stream) != cudaSuccess)
        return fail(c, TT_ERR_CUDA, "token copy failed");
    return tt_ctx_sync(c);
}

tt_status tt_ctx_loss_device(const tt_ctx* c, const float** mean_loss, const float** row_losses) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (!c->loss_dev) return TT_ERR_STATE;
    if (mean_loss) *mean_loss = c->loss_dev;
    if (row_losses) *row_losses = c->row_loss_dev;
    return TT_OK;
}

tt_status tt_ctx_copy_row_losses(tt_ctx* c, float* dst, size_t n) {
    if (!c || !dst) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (!c->row_loss_dev) return fail(c, TT_ERR_STATE, "no step since the last reset");
    if (!c->tensors.empty() && n > (size_t)c->tensors[0].rows)
        return fail(c, TT_ERR_ARG, "n exceeds B*T");
    if (cudaMemcpyAsync(dst, c->row_loss_dev, n * 4, cudaMemcpyDefault, c->stream) != cudaSuccess ||
        cudaStreamSynchronize(c->stream) != cudaSuccess)
        return fail(c, TT_ERR_CUDA, "row loss copy: %s", cudaGetErrorString(cudaGetLastError()));
    return TT_OK;
}

tt_status tt_adamw(tt_ctx* c, float* master, void* params_lowp, const float* grads, float* m,
                   float* v, size_t n, float lr, float beta1, float beta2, float eps,
                   float weight_decay, int step) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (!master || !grads || !m || !v || step < 1)
        return fail(c, TT_ERR_ARG, "adamw: NULL pointer or step < 1");
    if (((uintptr_t)master | (uintptr_t)grads | (uintptr_t)m | (uintptr_t)v) & 15)
        return fail(c, TT_ERR_ARG, "adamw: pointers must be 16-byte aligned");
    if (params_lowp && ((uintptr_t)params_lowp & 7))
        return fail(c, TT_ERR_ARG, "adamw: 16-bit copy must be 8-byte aligned");
    ProfScope ps(c, PK_ADAMW, 0.0, (double)n * (28.0 + (params_lowp ? 2.0 : 0.0)));
    launch_adamw(launch_of(c), master, params_lowp, grads, m, v, n, lr, beta1, beta2,
                 eps, weight_decay, step);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(c, TT_ERR_CUDA, "adamw: %s", cudaGetErrorString(e));
    return TT_OK;
}

tt_status tt_cast_f32_to_bf16(tt_ctx* c, const float* src, void* dst, size_t n) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (!src || !dst) return fail(c, TT_ERR_ARG, "cast: NULL pointer");
    launch_cast_bf16(launch_of(c), src, (__nv_bfloat16*)dst, n);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(c, TT_ERR_CUDA, "cast: %s", cudaGetErrorString(e));
    return TT_OK;
}

tt_status tt_cast_f32_to_f16(tt_ctx* c, const float* src, void* dst, size_t n) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (!src || !dst) return fail(c, TT_ERR_ARG, "cast: NULL pointer");
    launch_cast_f16(launch_of(c), src, (__half*)dst, n);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(c, TT_ERR_CUDA, "cast: %s", cudaGetErrorString(e));
    return TT_OK;
}

// ------------------------------------------------------------------ op-level ABI
#define TT_OP_PROLOGUE()                                  \
    if (!c) return TT_ERR_ARG;                            \
    if (!live(c)) return TT_ERR_STALE;                    \
    if (dtype != TT_FP32 && dtype != TT_BF16) return fail(c, TT_ERR_ARG, "bad dtype");

static tt_status op_epilogue(tt_ctx* c, const char* what) {
    if (c->oom) { c->oom = false; return fail(c, TT_ERR_ARENA_OOM, "%s: scratch does not fit", what); }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(c, TT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return TT_OK;
}

tt_status tt_op_linear_fwd(tt_ctx* c, tt_dtype dtype, const void* x, const void* W, const void* b,
                           const void* residual, void* y, void* pre, int M, int K, int N, int gelu) {
    TT_OP_PROLOGUE();
    if (!x || !W || !y || M <= 0 || K <= 0 || N <= 0 || (gelu && !pre))
        return fail(c, TT_ERR_ARG, "linear_fwd: bad arguments");
    GemmArgs g;
    g.A = x; g.lda = K; g.a_kmajor = true;
    g.B = W; g.ldb = K; g.b_kmajor = true;
    g.M = M; g.N = N; g.K = K;
    g.in_bf16 = dtype == TT_BF16;
    g.D = y; g.ldd = N; g.d_f32 = dtype == TT_FP32;
    g.epi = gelu ? EPI_GELU : EPI_STORE;
    g.bias = b; g.residual = residual; g.aux = gelu ? pre : nullptr;
    c->oom = false;
    if (!run_gemm(c, g, PK_GEMM_FWD)) return fail(c, TT_ERR_CUDA, "linear_fwd: launch failed");
    return op_epilogue(c, "linear_fwd");
}

tt_status tt_op_linear_bwd_dx(tt_ctx* c, tt_dtype dtype, const void* dy, const void* W,
                              const void* pre, void* dx, int M, int K, int N, int accumulate) {
    TT_OP_PROLOGUE();
    if (!dy || !W || !dx || M <= 0 || K <= 0 || N <= 0)
        return fail(c, TT_ERR_ARG, "linear_bwd_dx: bad arguments");
    GemmArgs g;
    g.A = dy; g.lda = N; g.a_kmajor = true;
    g.B = W; g.ldb = K; g.b_kmajor = false;
    g.M = M; g.N = K; g.K = N;
    g.in_bf16 = dtype == TT_BF16;
    g.D = dx; g.ldd = K; g.d_f32 = dtype == TT_FP32;
    g.accumulate = accumulate != 0;
    if (pre) { g.epi = EPI_DGELU; g.aux = const_cast<void*>(pre); }
    c->oom = false;
    if (!run_gemm(c, g, PK_GEMM_DX)) return fail(c, TT_ERR_CUDA, "linear_bwd_dx: launch failed");
    return op_epilogue(c, "linear_bwd_dx");
}

tt_status tt_op_linear_bwd_dw(tt_ctx* c, tt_dtype dtype, const void* dy, const void* x, float* dW,
                              float* db, int M, int K, int N) {
    TT_OP_PROLOGUE();
    if (!dy || !x || !dW || M <= 0 || K <= 0 || N <= 0)
        return fail(c, TT_ERR_ARG, "linear_bwd_dw: bad arguments");
    const bool bf = dtype == TT_BF16;
    GemmArgs g;
    g.A = dy; g.lda = N; g.a_kmajor = false;
    g.B = x; g.ldb = K; g.b_kmajor = false;
    g.M = N; g.N = K; g.K = M;
    g.in_bf16 = bf;
    g.D = dW; g.ldd = K; g.d_f32 = true;
    c->oom = false;
    if (!run_gemm(c, g, PK_GEMM_DW)) return fail(c, TT_ERR_CUDA, "linear_bwd_dw: launch failed");
    if (db) {
        size_t mark = c->off;
        float* s = (float*)arena_alloc(c, colsum_scratch_floats(M, N) * 4);
        if (!c->oom) launch_colsum(op_launch(c), bf, dy, M, N, db, s);
        c->off = mark;
    }
    return op_epilogue(c, "linear_bwd_dw");
}

tt_status tt_op_attention_fwd(tt_ctx* c, tt_dtype dtype, const void* qkv, void* y, float* lse, int B,
                              int T, int C, int H) {
    TT_OP_PROLOGUE();
    if (!qkv || !y || !lse || B <= 0 || T <= 0 || H <= 0 || C % H) return fail(c, TT_ERR_ARG, "attention_fwd: bad arguments");
    const int hd = C / H;
    if (hd != 16 && hd != 32 && hd != 64) return fail(c, TT_ERR_ARG, "attention: head dim must be 16, 32 or 64");
    {
        const double pairs = (double)B * H * T * (T + 1) / 2.0;
        ProfScope ps(c, PK_ATTN_FWD, 4.0 * pairs * hd, 4.0 * B * T * C * (dtype == TT_BF16 ? 2 : 4));
        launch_attention_fwd(op_launch(c), dtype == TT_BF16, qkv, y, lse, B, T, C, H);
    }
    return op_epilogue(c, "attention_fwd");
}

tt_status tt_op_attention_bwd(tt_ctx* c, tt_dtype dtype, const void* qkv, const void* y,
                              const float* lse, const void* dy, void* dqkv, int B, int T, int C,
                              int H) {
    TT_OP_PROLOGUE();
    if (!qkv || !y || !lse || !dy || !dqkv || B <= 0 || T <= 0 || H <= 0 || C % H)
        return fail(c, TT_ERR_ARG, "attention_bwd: bad arguments");
    const int hd = C / H;
    if (hd != 16 && hd != 32 && hd != 64) return fail(c, TT_ERR_ARG, "attention: head dim must be 16, 32 or 64");
    c->oom = false;
    size_t mark = c->off;
    float* s = (float*)arena_alloc(c, attention_bwd_scratch_floats(B, T, C, H) * 4);
    if (!c->oom) {
        const double pairs = (double)B * H * T * (T + 1) / 2.0;
        ProfScope ps(c, PK_ATTN_BWD, 10.0 * pairs * hd, 8.0 * B * T * C * (dtype == TT_BF16 ? 2 : 4));
        launch_attention_bwd(op_launch(c), dtype == TT_BF16, qkv, y, lse, dy, dqkv, B, T, C, H, s);
    }
    c->off = mark;
    return op_epilogue(c, "attention_bwd");
}

tt_status tt_op_layernorm_fwd(tt_ctx* c, tt_dtype dtype, const void* x, const void* w, const void* b,
                              void* y, float* mean, float* rstd, int M, int C) {
    TT_OP_PROLOGUE();
    if (!x || !w || !b || !y || !mean || !rstd || M <= 0 || C <= 0 || C % 32 || C > 1024)
        return fail(c, TT_ERR_ARG, "layernorm_fwd: bad arguments");
    {
        ProfScope ps(c, PK_LN_FWD, 0.0, 2.0 * M * C * (dtype == TT_BF16 ? 2 : 4) + 8.0 * M);
        launch_layernorm_fwd(op_launch(c), dtype == TT_BF16, x, w, b, y, mean, rstd, M, C);
    }
    return op_epilogue(c, "layernorm_fwd");
}

tt_status tt_op_layernorm_bwd(tt_ctx* c, tt_dtype dtype, const void* x, const void* w,
                              const float* mean, const float* rstd, const void* dy, void* dx,
                              float* dw, float* db, int M, int C, int accumulate) {
    TT_OP_PROLOGUE();
    if (!x || !w || !mean || !rstd || !dy || !dx || M <= 0 || C <= 0 || C % 32 || C > 1024)
        return fail(c, TT_ERR_ARG, "layernorm_bwd: bad arguments");
    c->oom = false;
    size_t mark = c->off;
    float* s = (float*)arena_alloc(c, layernorm_bwd_scratch_floats(M, C) * 4);
    if (!c->oom) {
        ProfScope ps(c, PK_LN_BWD, 0.0, (accumulate ? 4.0 : 3.0) * M * C * (dtype == TT_BF16 ? 2 : 4) + 8.0 * M);
        launch_layernorm_bwd(op_launch(c), dtype == TT_BF16, x, w, mean, rstd, dy, dx, dw, db, M, C,
                             accumulate != 0, s);
    }
    c->off = mark;
    return op_epilogue(c, "layernorm_bwd");
}

tt_status tt_op_xent(tt_ctx* c, tt_dtype dtype, void* logits, const int32_t* targets,
                     float* row_loss, float* mean_loss, int M, int V, int ld, float dscale) {
    TT_OP_PROLOGUE();
    if (!logits || !targets || !row_loss || M <= 0 || V <= 0 || ld < V)
        return fail(c, TT_ERR_ARG, "xent: bad arguments");
    {
        ProfScope ps(c, PK_XENT, 0.0, 2.0 * M * ld * (dtype == TT_BF16 ? 2 : 4) + 8.0 * M);
        launch_xent(op_launch(c), dtype == TT_BF16, logits, targets, row_loss, mean_loss, M, V, ld, dscale);
    }
    return op_epilogue(c, "xent");
}

tt_status tt_op_embed_fwd(tt_ctx* c, tt_dtype dtype, const void* wte, const void* wpe,
                          const int32_t* tokens, void* x, int B, int T, int C, int V) {
    TT_OP_PROLOGUE();
    if (!wte || !wpe || !tokens || !x || B <= 0 || T <= 0 || C <= 0 || V <= 0)
        return fail(c, TT_ERR_ARG, "embed_fwd: bad arguments");
    launch_embed_fwd(op_launch(c), dtype == TT_BF16, wte, wpe, tokens, x, B, T, C, V);
    return op_epilogue(c, "embed_fwd");
}

tt_status tt_op_embed_bwd(tt_ctx* c, tt_dtype dtype, const void* dx, const int32_t* tokens,
                          float* dwte, float* dwpe, int B, int T, int C, int V, int maxT) {
    TT_OP_PROLOGUE();
    if (!dx || !tokens || !dwte || !dwpe || B <= 0 || T <= 0 || T > maxT || C <= 0 || C > 1024 ||
        V <= 0 || V >= 65535 * 16)
        return fail(c, TT_ERR_ARG, "embed_bwd: bad arguments");
    c->oom = false;
    size_t mark = c->off;
    void* s = arena_alloc(c, embed_bwd_scratch_bytes(B * T, C));
    if (!c->oom) {
        ProfScope ps(c, PK_EMBED_BWD, 0.0, (double)B * T * C * ((dtype == TT_BF16 ? 2 : 4) + 8.0) + 4.0 * maxT * C);
        launch_embed_bwd(op_launch(c), dtype == TT_BF16, dx, tokens, dwte, dwpe, B, T, C, V, maxT, s);
    }
    c->off = mark;
    return op_epilogue(c, "embed_bwd");
}

// ------------------------------------------------------------------ generic tensor graph
static constexpr int G_IDX_BITS = 20;

static int g_index(const tt_ctx* c, tt_node h) {
    if (h < 0) return -1;
    const uint32_t ep = ((uint32_t)h >> G_IDX_BITS) & 0x7FF;
    const int idx = h & ((1 << G_IDX_BITS) - 1);
    if (ep != c->gepoch || idx >= (int)c->gnodes.size()) return -1;
    return idx;
}

static tt_node g_handle(const tt_ctx* c, int idx) { return (tt_node)((c->gepoch << G_IDX_BITS) | (uint32_t)idx); }

#define G_CTX()                                  \
    if (!c) return TT_ERR_ARG;                   \
    if (!live(c)) return TT_ERR_STALE

static tt_node g_new(tt_ctx* c, int op, int type, int ndim, const int* shape, int in0, int in1) {
    if (c->capturing) return fail(c, TT_ERR_STATE, "graph: nodes cannot be made while recording");
    if ((int)c->gnodes.size() >= (1 << G_IDX_BITS)) return fail(c, TT_ERR_ARG, "graph: too many nodes");
    GNode g;
    g.op = op;
    g.type = type;
    g.ndim = ndim;
    long long n = 1;
    for (int i = 0; i < ndim; i++) {
        if (shape[i] <= 0 || n > (1ll << 40) / shape[i]) return fail(c, TT_ERR_ARG, "graph: bad shape");
        g.shape[i] = shape[i];
        n *= shape[i];
    }
    g.n = n;
    g.in0 = in0;
    g.in1 = in1;
    const size_t mark = c->off;
    c->oom = false;
    g.data = arena_alloc(c, (size_t)n * 4);
    if (type == TT_NODE_F32) g.grad = (float*)arena_alloc(c, (size_t)n * 4);
    if (c->oom) {
        c->off = mark;
        c->oom = false;
        return fail(c, TT_ERR_ARENA_OOM, "graph: the arena cannot hold a node of %lld elements", n);
    }
    if (cudaMemsetAsync(g.data, 0, (size_t)n * 4, c->stream) != cudaSuccess ||
        (g.grad && cudaMemsetAsync(g.grad, 0, (size_t)n * 4, c->stream) != cudaSuccess))
        return fail(c, TT_ERR_CUDA, "graph: %s", cudaGetErrorString(cudaGetLastError()));
    if (in0 >= 0) c->gnodes[in0].uses++;
    if (in1 >= 0) c->gnodes[in1].uses++;
    c->gnodes.push_back(g);
    return g_handle(c, (int)c->gnodes.size() - 1);
}

static int g_rows(const GNode& g) { return (int)(g.n / g.shape[g.ndim - 1]); }
static int g_cols(const GNode& g) { return g.shape[g.ndim - 1]; }
static float* g_f(const GNode& g) { return (float*)g.data; }

// run node i's forward
static void g_forward_one(tt_ctx* c, int i) {
    const Launch L = launch_of(c);
    const GNode& g = c->gnodes[i];
    const GNode* a = g.in0 >= 0 ? &c->gnodes[g.in0] : nullptr;
    const GNode* b = g.in1 >= 0 ? &c->gnodes[g.in1] : nullptr;
    switch (g.op) {
    case G_MATMUL: {
        const int M = a->shape[0], K = a->shape[1], N = b->shape[1];
        launch_g_matmul(L, g_f(*a), K, 1, g_f(*b), N, 1, g_f(g), M, N, K, false);
        break;
    }
    case G_ADD: launch_g_add(L, g_f(*a), g_f(*b), g_f(g), g.n, 0); break;
    case G_ADD_ROW: launch_g_add(L, g_f(*a), g_f(*b), g_f(g), g.n, (int)b->n); break;
    case G_MUL: launch_g_mul(L, g_f(*a), g_f(*b), g_f(g), g.n); break;
    case G_GELU: launch_g_gelu(L, g_f(*a), g_f(g), g.n); break;
    case G_SOFTMAX: launch_g_softmax(L, g_f(*a), g_f(g), g_rows(*a), g_cols(*a)); break;
    case G_XENT: launch_g_xent(L, g_f(*a), (const int32_t*)b->data, g_rows(*a), g_cols(*a), g_f(g)); break;
    default: break;
    }
}

// nodes that n depends on (n included), as a mark per node
static std::vector<char> g_ancestors(const tt_ctx* c, int n) {
    std::vector<char> need(c->gnodes.size(), 0);
    need[n] = 1;
    for (int i = n; i >= 0; i--) {  // inputs have smaller indices than their consumers
        if (!need[i]) continue;
        const GNode& g = c->gnodes[i];
        if (g.in0 >= 0) need[g.in0] = 1;
        if (g.in1 >= 0) need[g.in1] = 1;
    }
    return need;
}

static tt_status g_done(tt_ctx* c, const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(c, TT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return TT_OK;
}

tt_node tt_node_new(tt_ctx* c, int ndim, const int* shape, tt_node_type type) {
    G_CTX();
    if (ndim < 1 || ndim > 4 || !shape || (type != TT_NODE_F32 && type != TT_NODE_I32))
        return fail(c, TT_ERR_ARG, "node_new: ndim must be 1..4 with a shape and a known type");
    return g_new(c, G_LEAF, type, ndim, shape, -1, -1);
}

static int g_input(tt_ctx* c, tt_node h, const char* what, bool f32) {
    const int i = g_index(c, h);
    if (i < 0) {
        fail(c, TT_ERR_STALE, "%s: stale or foreign node handle %d", what, (int)h);
        return -1;
    }
    if (f32 && c->gnodes[i].type != TT_NODE_F32) {
        fail(c, TT_ERR_ARG, "%s: input %d is not float32", what, (int)h);
        return -2;
    }
    return i;
}

#define G_IN(var, h, what, f32)                        \
    const int var = g_input(c, h, what, f32);         \
    if (var < 0) return var == -1 ? TT_ERR_STALE : TT_ERR_ARG

tt_node tt_node_matmul(tt_ctx* c, tt_node ha, tt_node hb) {
    G_CTX();
    G_IN(a, ha, "matmul", true);
    G_IN(b, hb, "matmul", true);
    const GNode &A = c->gnodes[a], &B = c->gnodes[b];
    if (A.ndim != 2 || B.ndim != 2 || A.shape[1] != B.shape[0])
        return fail(c, TT_ERR_ARG, "matmul: needs A [M,K] and B [K,N]");
    const int shp[2] = {A.shape[0], B.shape[1]};
    return g_new(c, G_MATMUL, TT_NODE_F32, 2, shp, a, b);
}

tt_node tt_node_add(tt_ctx* c, tt_node ha, tt_node hb) {
    G_CTX();
    G_IN(a, ha, "add", true);
    G_IN(b, hb, "add", true);
    const GNode &A = c->gnodes[a], &B = c->gnodes[b];
    bool same = A.ndim == B.ndim;
    for (int i = 0; same && i < A.ndim; i++) same = A.shape[i] == B.shape[i];
    const bool row = !same && B.ndim == 1 && B.shape[0] == g_cols(A);
    if (!same && !row) return fail(c, TT_ERR_ARG, "add: b must have a's shape or be a row of a's last dimension");
    int shp[4];
    for (int i = 0; i < A.ndim; i++) shp[i] = A.shape[i];
    return g_new(c, same ? G_ADD : G_ADD_ROW, TT_NODE_F32, A.ndim, shp, a, b);
}

tt_node tt_node_mul(tt_ctx* c, tt_node ha, tt_node hb) {
    G_CTX();
    G_IN(a, ha, "mul", true);
    G_IN(b, hb, "mul", true);
    const GNode &A = c->gnodes[a], &B = c->gnodes[b];
    bool same = A.ndim == B.ndim;
    for (int i = 0; same && i < A.ndim; i++) same = A.shape[i] == B.shape[i];
    if (!same) return fail(c, TT_ERR_ARG, "mul: shapes differ");
    int shp[4];
    for (int i = 0; i < A.ndim; i++) shp[i] = A.shape[i];
    return g_new(c, G_MUL, TT_NODE_F32, A.ndim, shp, a, b);
}

static tt_node g_unary(tt_ctx* c, tt_node ha, int op, const char* what) {
    G_IN(a, ha, what, true);
    const GNode& A = c->gnodes[a];
    int shp[4];
    for (int i = 0; i < A.ndim; i++) shp[i] = A.shape[i];
    return g_new(c, op, TT_NODE_F32, A.ndim, shp, a, -1);
}

tt_node tt_node_gelu(tt_ctx* c, tt_node a) {
    G_CTX();
    return g_unary(c, a, G_GELU, "gelu");
}

tt_node tt_node_softmax(tt_ctx* c, tt_node a) {
    G_CTX();
    return g_unary(c, a, G_SOFTMAX, "softmax");
}

tt_node tt_node_cross_entropy(tt_ctx* c, tt_node hp, tt_node hy) {
    G_CTX();
    G_IN(p, hp, "cross_entropy", true);
    G_IN(y, hy, "cross_entropy", false);
    const GNode &P = c->gnodes[p], &Y = c->gnodes[y];
    if (Y.type != TT_NODE_I32 || Y.n != g_rows(P))
        return fail(c, TT_ERR_ARG, "cross_entropy: labels must be int32 with one per row of p");
    const int one = 1;
    return g_new(c, G_XENT, TT_NODE_F32, 1, &one, p, y);
}

tt_status tt_node_forward(tt_ctx* c, tt_node h) {
    G_CTX();
    G_IN(n, h, "forward", false);
    const std::vector<char> need = g_ancestors(c, n);
    for (int i = 0; i <= n; i++)
        if (need[i] && c->gnodes[i].op != G_LEAF) g_forward_one(c, i);
    return g_done(c, "forward");
}

// zero the gradients of the marked nodes (leaves only if with_leaves), a few
// dozen buffers per launch
static void g_zero_grads(tt_ctx* c, const std::vector<char>& need, int upto, bool with_leaves) {
    const Launch L = launch_of(c);
    GZeroList l{};
    for (int i = 0; i <= upto; i++) {
        const GNode& g = c->gnodes[i];
        if (!need[i] || !g.grad || (!with_leaves && g.op == G_LEAF)) continue;
        l.p[l.count] = g.grad;
        l.n[l.count] = g.n;
        if (++l.count == G_ZERO_MAX) {
            launch_g_zero_many(L, l);
            l.count = 0;
        }
    }
    launch_g_zero_many(L, l);
}

tt_status tt_node_zero_grad(tt_ctx* c, tt_node h) {
    G_CTX();
    G_IN(n, h, "zero_grad", false);
    g_zero_grads(c, g_ancestors(c, n), n, true);
    return g_done(c, "zero_grad");
}

tt_status tt_node_backward(tt_ctx* c, tt_node h) {
    G_CTX();
    G_IN(n, h, "backward", true);
    const Launch L = launch_of(c);
    const std::vector<char> need = g_ancestors(c, n);
    g_zero_grads(c, need, n - 1, false);
    launch_g_fill(L, c->gnodes[n].grad, c->gnodes[n].n, 1.0f);
    std::vector<char> done(c->gnodes.size(), 0);  // a softmax whose gradient its cross entropy formed
    for (int i = n; i >= 0; i--) {
        if (!need[i] || done[i]) continue;
        const GNode& g = c->gnodes[i];
        if (g.op == G_LEAF) continue;
        GNode* a = g.in0 >= 0 ? &c->gnodes[g.in0] : nullptr;
        GNode* b = g.in1 >= 0 ? &c->gnodes[g.in1] : nullptr;
        switch (g.op) {
        case G_MATMUL: {
            const int M = a->shape[0], K = a->shape[1], N = b->shape[1];
            // dA += dC B^T: (m, k) <- sum_n dC[m, n] B[k, n]
            launch_g_matmul(L, g.grad, N, 1, g_f(*b), 1, N, a->grad, M, K, N, true);
            // dB += A^T dC: (k, n) <- sum_m A[m, k] dC[m, n]
            launch_g_matmul(L, g_f(*a), 1, K, g.grad, N, 1, b->grad, K, N, M, true);
            break;
        }
        case G_ADD:
            launch_g_acc(L, a->grad, g.grad, g.n);
            launch_g_acc(L, b->grad, g.grad, g.n);
            break;
        case G_ADD_ROW:
            launch_g_acc(L, a->grad, g.grad, g.n);
            launch_g_colsum_acc(L, g.grad, g_rows(g), g_cols(g), b->grad);
            break;
        case G_MUL:
            launch_g_mul_bwd(L, g.grad, g_f(*a), g_f(*b), a->grad, b->grad, g.n);
            break;
        case G_GELU: launch_g_gelu_bwd(L, g.grad, g_f(*a), a->grad, g.n); break;
        case G_SOFTMAX: launch_g_softmax_bwd(L, g_f(g), g.grad, a->grad, g_rows(g), g_cols(g)); break;
        case G_XENT: {
            const int rows = g_rows(*a), cols = g_cols(*a);
            if (a->op == G_SOFTMAX && a->uses == 1) {
                // the pair's gradient directly: (p - onehot) / R into the logits
                GNode& z = c->gnodes[a->in0];
                launch_g_softmax_xent_bwd(L, g_f(*a), (const int32_t*)b->data, g.grad, rows, cols, z.grad);
                done[g.in0] = 1;
            } else {
                launch_g_xent_bwd(L, g_f(*a), (const int32_t*)b->data, g.grad, rows, cols, a->grad);
            }
            break;
        }
        default: break;
        }
    }
    return g_done(c, "backward");
}

static bool is_device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

tt_status tt_node_fill(tt_ctx* c, tt_node h, const void* src, size_t count) {
    G_CTX();
    G_IN(n, h, "fill", false);
    const GNode& g = c->gnodes[n];
    if (!src || count != (size_t)g.n) return fail(c, TT_ERR_ARG, "fill: %zu values for %lld elements", count, g.n);
    const cudaMemcpyKind k = is_device_ptr(src) ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    if (c->capturing && k == cudaMemcpyHostToDevice)
        return fail(c, TT_ERR_STATE, "fill from host memory while recording");
    if (cudaMemcpyAsync(g.data, src, count * 4, k, c->stream) != cudaSuccess)
        return fail(c, TT_ERR_CUDA, "fill: %s", cudaGetErrorString(cudaGetLastError()));
    if (k == cudaMemcpyHostToDevice && cudaStreamSynchronize(c->stream) != cudaSuccess)  // src may be reused
        return fail(c, TT_ERR_CUDA, "fill: %s", cudaGetErrorString(cudaGetLastError()));
    return TT_OK;
}

tt_status tt_node_read(tt_ctx* c, tt_node h, int grad, void* dst, size_t count) {
    G_CTX();
    G_IN(n, h, "read", false);
    const GNode& g = c->gnodes[n];
    if (!dst || count != (size_t)g.n) return fail(c, TT_ERR_ARG, "read: %zu values for %lld elements", count, g.n);
    const void* s = grad ? (const void*)g.grad : g.data;
    if (!s) return fail(c, TT_ERR_ARG, "read: an int32 node has no gradient");
    if (c->capturing) return fail(c, TT_ERR_STATE, "read while recording");
    if (cudaMemcpyAsync(dst, s, count * 4, cudaMemcpyDefault, c->stream) != cudaSuccess)
        return fail(c, TT_ERR_CUDA, "read: %s", cudaGetErrorString(cudaGetLastError()));
    return tt_ctx_sync(c);
}

tt_status tt_node_info(tt_ctx* c, tt_node h, int* ndim, int* shape, void** data, float** grad) {
    G_CTX();
    G_IN(n, h, "info", false);
    const GNode& g = c->gnodes[n];
    if (ndim) *ndim = g.ndim;
    if (shape)
        for (int i = 0; i < 4; i++) shape[i] = g.shape[i];
    if (data) *data = g.data;
    if (grad) *grad = g.grad;
    return TT_OK;
}

tt_status tt_node_sgd(tt_ctx* c, const tt_node* params, int n_params, float lr) {
    G_CTX();
    if (n_params < 0 || (n_params > 0 && !params)) return fail(c, TT_ERR_ARG, "sgd: bad parameter list");
    const Launch L = launch_of(c);
    for (int k = 0; k < n_params; k++) {
        G_IN(i, params[k], "sgd", true);
        const GNode& g = c->gnodes[i];
        launch_g_sgd(L, g_f(g), g.grad, g.n, lr);
    }
    return g_done(c, "sgd");
}

tt_status tt_capture_begin(tt_ctx* c) {
    G_CTX();
    if (c->capturing) return fail(c, TT_ERR_STATE, "a recording is already open");
    if (!c->cap_stream && cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking) != cudaSuccess)
        return fail(c, TT_ERR_CUDA, "capture: %s", cudaGetErrorString(cudaGetLastError()));
    // the recording is replayed on the context's stream, after whatever is queued there then
    if (cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
        return fail(c, TT_ERR_CUDA, "capture: %s", cudaGetErrorString(cudaGetLastError()));
    c->saved_stream = c->stream;
    c->stream = c->cap_stream;
    c->capturing = true;
    c->cap_launches0 = c->launches;
    return TT_OK;
}

tt_status tt_capture_end(tt_ctx* c) {
    G_CTX();
    if (!c->capturing) return fail(c, TT_ERR_STATE, "no open recording");
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(c->cap_stream, &g);
    c->stream = c->saved_stream;
    c->capturing = false;
    const uint64_t nodes = c->launches - c->cap_launches0;
    c->launches = c->cap_launches0;  // recorded, not run
    if (c->recording) {
        cudaGraphExecDestroy(c->recording);
        c->recording = nullptr;
    }
    if (e != cudaSuccess || !g) {
        if (g) cudaGraphDestroy(g);
        cudaGetLastError();
        return fail(c, TT_ERR_CUDA, "capture: %s", cudaGetErrorString(e));
    }
    const cudaError_t ei = cudaGraphInstantiate(&c->recording, g, 0);
    cudaGraphDestroy(g);
    if (ei != cudaSuccess) {
        c->recording = nullptr;
        cudaGetLastError();
        return fail(c, TT_ERR_CUDA, "capture: %s", cudaGetErrorString(ei));
    }
    c->rec_launches = nodes;
    return TT_OK;
}

tt_status tt_replay(tt_ctx* c, int times) {
    G_CTX();
    if (c->capturing || !c->recording) return fail(c, TT_ERR_STATE, "nothing recorded to replay");
    if (times < 0) return fail(c, TT_ERR_ARG, "replay: times < 0");
    for (int i = 0; i < times; i++) {
        if (cudaGraphLaunch(c->recording, c->stream) != cudaSuccess)
            return fail(c, TT_ERR_CUDA, "replay: %s", cudaGetErrorString(cudaGetLastError()));
        c->launches += c->rec_launches;
    }
    return TT_OK;
}

// ------------------------------------------------------------------ clipping and loss scaling
tt_status tt_grad_stats(tt_ctx* c, const float* grads, size_t n, const float* loss_scale, float* stats) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (!grads || !stats || n == 0) return fail(c, TT_ERR_ARG, "grad_stats: NULL pointer or n == 0");
    const Launch L = launch_of(c);
    const size_t mark = c->off;
    c->oom = false;
    double* s = (double*)arena_alloc(c, grad_stats_scratch_doubles(L) * sizeof(double));
    if (c->oom) {
        c->off = mark;
        c->oom = false;
        return fail(c, TT_ERR_ARENA_OOM, "grad_stats: no arena room for %zu partial sums", grad_stats_scratch_doubles(L));
    }
    launch_grad_stats(L, grads, n, loss_scale, stats, s);
    c->off = mark;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(c, TT_ERR_CUDA, "grad_stats: %s", cudaGetErrorString(e));
    return TT_OK;
}

tt_status tt_adamw_ex(tt_ctx* c, float* master, void* params_lowp, const float* grads, float* m, float* v, size_t n,
                      float lr, float beta1, float beta2, float eps, float weight_decay, int* step,
                      const float* stats, float max_norm, const float* loss_scale) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (!master || !grads || !m || !v || !step) return fail(c, TT_ERR_ARG, "adamw_ex: NULL pointer");
    if (max_norm > 0.0f && !stats) return fail(c, TT_ERR_ARG, "adamw_ex: clipping needs the gradient statistics");
    if (((uintptr_t)master | (uintptr_t)grads | (uintptr_t)m | (uintptr_t)v) & 15)
        return fail(c, TT_ERR_ARG, "adamw_ex: buffers must be 16-byte aligned");
    launch_adamw_ex(launch_of(c), master, params_lowp, grads, m, v, n, lr, beta1, beta2, eps,
                    weight_decay, step, stats, max_norm, loss_scale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(c, TT_ERR_CUDA, "adamw_ex: %s", cudaGetErrorString(e));
    return TT_OK;
}

tt_status tt_loss_scale_update(tt_ctx* c, float* loss_scale, int* clean_steps, const float* stats, int window,
                               float growth, float backoff) {
    if (!c) return TT_ERR_ARG;
    if (!live(c)) return TT_ERR_STALE;
    if (!loss_scale || !clean_steps || !stats || window < 1 || !(growth >= 1.0f) || !(backoff > 0.0f && backoff < 1.0f))
        return fail(c, TT_ERR_ARG, "loss_scale_update: bad arguments");
    launch_loss_scale_update(launch_of(c), loss_scale, clean_steps, stats, window, growth, backoff);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(c, TT_ERR_CUDA, "loss_scale_update: %s", cudaGetErrorString(e));
    return TT_OK;
}

}  // extern "C"

// kernels.cu -- memory-bound kernels of the GPT-2 step (embedding, LayerNorm,
// fused cross entropy, column sums, AdamW) and the SIMT contraction kernels
// (fp32-mode GEMM and attention, also the fallback for shapes the tensor-core
// kernels do not take).  All reductions run in a fixed order: no floating-point
// atomics anywhere, so every result is bitwise reproducible run to run.
#include "tt_internal.h"

#include <math.h>

namespace tt {

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ float ld(const float* p, long long i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, long long i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float ld(const __half* p, long long i) { return __half2float(p[i]); }
__device__ __forceinline__ void st(float* p, long long i, float v) { p[i] = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, long long i, float v) { p[i] = __float2bfloat16_rn(v); }
__device__ __forceinline__ void st(__half* p, long long i, float v) { p[i] = __float2half_rn(v); }

// four floats rounded to nearest even into elements 4i..4i+3 of a 16-bit copy (one 8-byte store)
__device__ __forceinline__ void st_low4(__nv_bfloat16* p, size_t i, float4 v) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&lo);
    packed.y = *reinterpret_cast<const uint32_t*>(&hi);
    reinterpret_cast<uint2*>(p)[i] = packed;
}
__device__ __forceinline__ void st_low4(__half* p, size_t i, float4 v) {
    const __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&lo);
    packed.y = *reinterpret_cast<const uint32_t*>(&hi);
    reinterpret_cast<uint2*>(p)[i] = packed;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

static inline unsigned blocks_for(long long n, int threads) {
    long long b = (n + threads - 1) / threads;
    return (unsigned)(b < 1 ? 1 : b);
}

// GELU, tanh form: g(u) = 0.5 u (1 + tanh(k (u + a u^3))), k = sqrt(2/pi), a = 0.044715.
__device__ __forceinline__ float gelu_f(float u) {
    const float k = 0.7978845608028654f, a = 0.044715f;
    return 0.5f * u * (1.0f + tanhf(k * (u + a * u * u * u)));
}
// its exact derivative
__device__ __forceinline__ float dgelu_f(float u) {
    const float k = 0.7978845608028654f, a = 0.044715f;
    float tau = tanhf(k * (u + a * u * u * u));
    return 0.5f * (1.0f + tau) + 0.5f * u * (1.0f - tau * tau) * k * (1.0f + 3.0f * a * u * u);
}

// ================================================================== embedding
template <typename T>
__global__ void k_embed_fwd(const T* __restrict__ wte, const T* __restrict__ wpe,
                            const int32_t* __restrict__ tok, T* __restrict__ x,
                            int T_, int C, int V, long long total, int* flags) {
    pdl_enter();
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    long long m = i / C;
    int c = (int)(i - m * C);
    int t = (int)(m % T_);
    int id = tok[m];
    float v = 0.0f;
    if (id < 0 || id >= V) {
        if (c == 0) atomicOr(&flags[FLAG_BAD_TOKEN], 1);
    } else {
        v = ld(wte, (long long)id * C + c) + ld(wpe, (long long)t * C + c);
    }
    st(x, i, v);
}

void launch_embed_fwd(const Launch& L, bool bf16, const void* wte, const void* wpe,
                      const int32_t* tok, void* x, int B, int T, int C, int V) {
    if (L.dry) return;
    long long total = (long long)B * T * C;
    L.count();
    if (bf16 && L.f16)
        launch_k(L, k_embed_fwd<__half>, dim3(blocks_for(total, 256)), dim3(256), 0, 
            (const __half*)wte, (const __half*)wpe, tok, (__half*)x, T, C, V,
            total, L.flags);
    else if (bf16)
        launch_k(L, k_embed_fwd<__nv_bfloat16>, dim3(blocks_for(total, 256)), dim3(256), 0, 
            (const __nv_bfloat16*)wte, (const __nv_bfloat16*)wpe, tok, (__nv_bfloat16*)x, T, C, V,
            total, L.flags);
    else
        launch_k(L, k_embed_fwd<float>, dim3(blocks_for(total, 256)), dim3(256), 0, 
            (const float*)wte, (const float*)wpe, tok, (float*)x, T, C, V, total, L.flags);
}

// Stable LSD radix sort of positions by token id, 8-bit digits, across the
// whole GPU.  Each pass is three launches over tiles of RS_TILE consecutive
// elements: per-tile digit counts; one exclusive scan of the counts in
// digit-major, tile-minor order; a scatter in which every element's place is
// its digit's scanned base for the tile plus its rank among the tile's
// earlier elements of the same digit -- so equal keys keep input (position)
// order, and the result is the same however the hardware schedules it.
// Pass 0 reads the token ids themselves (an id outside [0, V) gets key V and
// sorts last); the values are the positions.
constexpr int RS_THREADS = 256;
constexpr int RS_ROUNDS = 4;
constexpr int RS_TILE = RS_THREADS * RS_ROUNDS;
constexpr int RS_BINS = 256;

__device__ __forceinline__ int rs_key(const int32_t* __restrict__ in, int from_tok, int V, int i) {
    const int k = in[i];
    return from_tok ? ((k < 0 || k >= V) ? V : k) : k;
}

__global__ void __launch_bounds__(RS_THREADS)
k_rs_hist(const int32_t* __restrict__ in, int from_tok, int V, int M, int shift, int G, int* __restrict__ hist) {
    pdl_enter();
    __shared__ int s_h[RS_BINS];
    s_h[threadIdx.x] = 0;
    __syncthreads();
    const long long i0 = (long long)blockIdx.x * RS_TILE;
#pragma unroll
    for (int r = 0; r < RS_ROUNDS; r++) {
        const long long i = i0 + r * RS_THREADS + threadIdx.x;
        if (i < M) atomicAdd(&s_h[(rs_key(in, from_tok, V, (int)i) >> shift) & (RS_BINS - 1)], 1);
    }
    __syncthreads();
    hist[(long long)threadIdx.x * G + blockIdx.x] = s_h[threadIdx.x];
}

// exclusive scan of n ints in place, one block of 1024 threads: thread t
// takes a contiguous run of ceil(n/1024) entries
__global__ void __launch_bounds__(1024) k_rs_scan(int* __restrict__ a, int n) {
    pdl_enter();
    __shared__ int s_w[32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int per = (n + 1023) / 1024;
    const int lo = min(n, t * per), hi = min(n, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; i++) sum += a[i];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = s_w[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += v;
        }
        s_w[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    int run = incl - sum + (warp > 0 ? s_w[warp - 1] : 0);
    for (int i = lo; i < hi; i++) {
        const int v = a[i];
        a[i] = run;
        run += v;
    }
}

__global__ void __launch_bounds__(RS_THREADS)
k_rs_scatter(const int32_t* __restrict__ kin, const int32_t* __restrict__ vin, int from_tok, int V, int M,
             int shift, int G, const int* __restrict__ scan, int32_t* __restrict__ kout,
             int32_t* __restrict__ vout) {
    pdl_enter();
    __shared__ int s_base[RS_BINS];
    __shared__ int s_wc[RS_THREADS / 32][RS_BINS];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    s_base[t] = scan[(long long)t * G + blockIdx.x];
    const long long i0 = (long long)blockIdx.x * RS_TILE;
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll 1
    for (int r = 0; r < RS_ROUNDS; r++) {
#pragma unroll
        for (int w = 0; w < RS_THREADS / 32; w++) s_wc[w][t] = 0;
        const long long i = i0 + r * RS_THREADS + t;  // index order = round, warp, lane
        const bool ok = i < M;
        const int key = ok ? rs_key(kin, from_tok, V, (int)i) : 0;
        const int val = ok ? (from_tok ? (int)i : vin[i]) : 0;
        const int d = ok ? (key >> shift) & (RS_BINS - 1) : RS_BINS;
        __syncthreads();
        const unsigned same = __match_any_sync(0xffffffffu, d);
        const int rank = __popc(same & lt);
        if (ok && rank == 0) s_wc[warp][d] = __popc(same);
        __syncthreads();
        if (ok) {
            int pos = s_base[d] + rank;
            for (int w = 0; w < warp; w++) pos += s_wc[w][d];
            kout[pos] = key;
            vout[pos] = val;
        }
        __syncthreads();
        int add = 0;
#pragma unroll
        for (int w = 0; w < RS_THREADS / 32; w++) add += s_wc[w][t];
        s_base[t] += add;  // the tile's later rounds come after this one
    }
}

static int rs_tiles(int M) { return (M + RS_TILE - 1) / RS_TILE; }

// One block per sorted index; the block at the start of a run of equal
// token ids sums that run's rows of dx in increasing position order and adds
// the sum to dwte[id].
template <typename T>
__global__ void k_embed_segsum(const T* __restrict__ dx, const int32_t* __restrict__ keys,
                               const int32_t* __restrict__ vals, int M, int C, int V,
                               float* __restrict__ dwte) {
    pdl_enter();
    const int i = blockIdx.x;
    const int key = keys[i];
    if (key >= V) return;
    if (i > 0 && keys[i - 1] == key) return;
    constexpr int MAXC = 8;  // columns per thread: C <= 8 * blockDim.x
    float acc[MAXC];
#pragma unroll
    for (int j = 0; j < MAXC; j++) acc[j] = 0.0f;
    for (int r = i; r < M && keys[r] == key; r++) {
        const long long row = (long long)vals[r] * C;
#pragma unroll
        for (int j = 0; j < MAXC; j++) {
            int c = threadIdx.x + j * blockDim.x;
            if (c < C) acc[j] += ld(dx, row + c);
        }
    }
#pragma unroll
    for (int j = 0; j < MAXC; j++) {
        int c = threadIdx.x + j * blockDim.x;
        if (c < C) dwte[(long long)key * C + c] += acc[j];
    }
}

template <typename T>
__global__ void k_embed_wpe(const T* __restrict__ dx, int B, int T_, int C, int maxT,
                            float* __restrict__ dwpe, int acc) {
    pdl_enter();
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)maxT * C) return;
    int t = (int)(i / C), c = (int)(i % C);
    float s = 0.0f;
    if (t < T_)
        for (int b = 0; b < B; b++) s += ld(dx, ((long long)b * T_ + t) * C + c);
    dwpe[i] = acc ? dwpe[i] + s : s;
}

// scratch: keys/values A and B [M] each, the digit counts [256 x tiles], then
// the chunk partial sums of the segmented reduction
static size_t rs_ints(int M) { return (size_t)4 * M + (size_t)RS_BINS * rs_tiles(M); }

size_t embed_bwd_scratch_bytes(int M, int C) {
    return ((rs_ints(M) * sizeof(int32_t) + 255) & ~(size_t)255) +
           embed_chunk_scratch_floats(M, C) * sizeof(float);
}

void launch_embed_bwd(const Launch& L, bool bf16, const void* dx, const int32_t* tok,
                      float* dwte, float* dwpe, int B, int T, int C, int V, int maxT,
                      void* scratch, bool acc_params) {
    if (L.dry) return;
    const int M = B * T;
    int32_t* s = (int32_t*)scratch;
    int bits = 1;
    while ((1 << bits) <= V) bits++;  // keys take values 0..V
    const int passes = (bits + 7) / 8;
    const int G = rs_tiles(M);
    int32_t *kA = s, *vA = s + M, *kB = s + 2 * M, *vB = s + 3 * M;
    int* hist = s + 4 * (size_t)M;
    // the last pass must write buffer A
    int32_t* ko = (passes & 1) ? kA : kB;
    int32_t* vo = (passes & 1) ? vA : vB;
    const int32_t *ki = tok, *vi = nullptr;
    for (int p = 0; p < passes; p++) {
        const int from_tok = p == 0;
        L.count();
        launch_k(L, k_rs_hist, dim3(G), dim3(RS_THREADS), 0, ki, from_tok, V, M, 8 * p, G, hist);
        L.count();
        launch_k(L, k_rs_scan, dim3(1), dim3(1024), 0, hist, RS_BINS * G);
        L.count();
        launch_k(L, k_rs_scatter, dim3(G), dim3(RS_THREADS), 0, ki, vi, from_tok, V, M, 8 * p, G, hist, ko, vo);
        ki = ko; vi = vo;
        ko = (ko == kA) ? kB : kA;
        vo = (vo == vA) ? vB : vA;
    }
    float* chunk_scratch = (float*)((char*)scratch + ((rs_ints(M) * sizeof(int32_t) + 255) & ~(size_t)255));
    if (!launch_embed_chunks(L, bf16, dx, s, s + M, M, C, V, dwte, chunk_scratch)) {
        int threads = (C + 7) / 8;
        threads = ((threads + 31) / 32) * 32;
        L.count();
        if (bf16 && L.f16)
            launch_k(L, k_embed_segsum<__half>, dim3(M), dim3(threads), 0, 
                (const __half*)dx, s, s + M, M, C, V, dwte);
        else if (bf16)
            launch_k(L, k_embed_segsum<__nv_bfloat16>, dim3(M), dim3(threads), 0, 
                (const __nv_bfloat16*)dx, s, s + M, M, C, V, dwte);
        else
            launch_k(L, k_embed_segsum<float>, dim3(M), dim3(threads), 0, (const float*)dx, s, s + M, M, C, V, dwte);
    }
    long long n = (long long)maxT * C;
    L.count();
    if (bf16 && L.f16)
        launch_k(L, k_embed_wpe<__half>, dim3(blocks_for(n, 256)), dim3(256), 0, 
            (const __half*)dx, B, T, C, maxT, dwpe, acc_params ? 1 : 0);
    else if (bf16)
        launch_k(L, k_embed_wpe<__nv_bfloat16>, dim3(blocks_for(n, 256)), dim3(256), 0, 
            (const __nv_bfloat16*)dx, B, T, C, maxT, dwpe, acc_params ? 1 : 0);
    else
        launch_k(L, k_embed_wpe<float>, dim3(blocks_for(n, 256)), dim3(256), 0, (const float*)dx, B, T, C,
                                                                     maxT, dwpe, acc_params ? 1 : 0);
}

// ================================================================== layernorm
// One warp per row; the row lives in registers (C <= 1024: 32 values a lane).
constexpr int LN_MAXV = 32;

template <typename T>
__global__ void k_layernorm_fwd(const T* __restrict__ x, const T* __restrict__ w,
                                const T* __restrict__ b, T* __restrict__ y,
                                float* __restrict__ mean, float* __restrict__ rstd, int M, int C) {
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= M) return;
    const int n = C >> 5;
    const T* xr = x + row * C;
    float v[LN_MAXV];
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < LN_MAXV; i++)
        if (i < n) { v[i] = ld(xr, lane + 32 * i); s += v[i]; }
    const float mu = warp_sum(s) / C;
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < LN_MAXV; i++)
        if (i < n) { float d = v[i] - mu; q += d * d; }
    const float var = warp_sum(q) / C;
    const float rs = rsqrtf(var + 1e-5f);
    T* yr = y + row * C;
#pragma unroll
    for (int i = 0; i < LN_MAXV; i++)
        if (i < n) {
            int c = lane + 32 * i;
            st(yr, c, (v[i] - mu) * rs * ld(w, c) + ld(b, c));
        }
    if (lane == 0) { mean[row] = mu; rstd[row] = rs; }
}

void launch_layernorm_fwd(const Launch& L, bool bf16, const void* x, const void* w,
                          const void* b, void* y, float* mean, float* rstd, int M, int C) {
    if (L.dry) return;
    if (bf16 && launch_ln_fwd_bf16(L, x, w, b, y, mean, rstd, M, C)) return;
    const int warps = 8;
    L.count();
    if (bf16 && L.f16)
        k_layernorm_fwd<__half><<<blocks_for(M, warps), warps * 32, 0, L.stream>>>(
            (const __half*)x, (const __half*)w, (const __half*)b,
            (__half*)y, mean, rstd, M, C);
    else if (bf16)
        k_layernorm_fwd<__nv_bfloat16><<<blocks_for(M, warps), warps * 32, 0, L.stream>>>(
            (const __nv_bfloat16*)x, (const __nv_bfloat16*)w, (const __nv_bfloat16*)b,
            (__nv_bfloat16*)y, mean, rstd, M, C);
    else
        k_layernorm_fwd<float><<<blocks_for(M, warps), warps * 32, 0, L.stream>>>(
            (const float*)x, (const float*)w, (const float*)b, (float*)y, mean, rstd, M, C);
}

// Backward.  Each block owns LN_ROWS consecutive rows; each of its warps walks
// rows warp, warp+8, ... and keeps per-lane partial dw/db in registers; the
// block then combines its warps in warp order and writes one partial row;
// k_sum_partials adds the block partials in block order.
constexpr int LN_BWD_WARPS = 8;
constexpr int LN_ROWS = 64;

template <typename T>
__global__ void k_layernorm_bwd(const T* __restrict__ x, const T* __restrict__ w,
                                const float* __restrict__ mean, const float* __restrict__ rstd,
                                const T* __restrict__ dy, T* __restrict__ dx,
                                float* __restrict__ part, int M, int C, int accumulate) {
    extern __shared__ float s_part[];  // [LN_BWD_WARPS][2*C]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = C >> 5;
    float wv[LN_MAXV], pw[LN_MAXV], pb[LN_MAXV];
#pragma unroll
    for (int i = 0; i < LN_MAXV; i++)
        if (i < n) { wv[i] = ld(w, lane + 32 * i); pw[i] = 0.0f; pb[i] = 0.0f; }
    const long long r0 = (long long)blockIdx.x * LN_ROWS;
    for (int rr = warp; rr < LN_ROWS; rr += LN_BWD_WARPS) {
        const long long row = r0 + rr;
        if (row >= M) break;
        const T* xr = x + row * C;
        const T* dyr = dy + row * C;
        const float mu = mean[row], rs = rstd[row];
        float xh[LN_MAXV], g[LN_MAXV];
        float sg = 0.0f, sgx = 0.0f;
#pragma unroll
        for (int i = 0; i < LN_MAXV; i++)
            if (i < n) {
                int c = lane + 32 * i;
                float d = ld(dyr, c);
                xh[i] = (ld(xr, c) - mu) * rs;
                g[i] = d * wv[i];
                sg += g[i];
                sgx += g[i] * xh[i];
                pw[i] += d * xh[i];
                pb[i] += d;
            }
        const float mg = warp_sum(sg) / C, mgx = warp_sum(sgx) / C;
        T* dxr = dx + row * C;
#pragma unroll
        for (int i = 0; i < LN_MAXV; i++)
            if (i < n) {
                int c = lane + 32 * i;
                float v = rs * (g[i] - mg - xh[i] * mgx);
                if (accumulate) v += ld(dxr, c);
                st(dxr, c, v);
            }
    }
#pragma unroll
    for (int i = 0; i < LN_MAXV; i++)
        if (i < n) {
            s_part[warp * 2 * C + lane + 32 * i] = pw[i];
            s_part[warp * 2 * C + C + lane + 32 * i] = pb[i];
        }
    __syncthreads();
    for (int c = threadIdx.x; c < 2 * C; c += blockDim.x) {
        float s = 0.0f;
        for (int k = 0; k < LN_BWD_WARPS; k++) s += s_part[k * 2 * C + c];
        part[(long long)blockIdx.x * 2 * C + c] = s;
    }
}

// out_a[c] = sum_b part[b][c], out_b[c] = sum_b part[b][C + c] (b in order)
__global__ void k_sum_partials(const float* __restrict__ part, int nblk, int C,
                               float* __restrict__ out_a, float* __restrict__ out_b, int acc) {
    int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= 2 * C) return;
    float s = 0.0f;
    for (int b = 0; b < nblk; b++) s += part[(long long)b * 2 * C + c];
    if (c < C) { if (out_a) out_a[c] = acc ? out_a[c] + s : s; }
    else if (out_b) out_b[c - C] = acc ? out_b[c - C] + s : s;
}

size_t layernorm_bwd_scratch_floats(int M, int C) {
    size_t a = (size_t)((M + LN_ROWS - 1) / LN_ROWS) * 2 * C + 64;
    size_t b = ln_bwd_bf16_scratch_floats(C);
    size_t c = colsum_scratch_floats(M, C);
    return a > b ? (a > c ? a : c) : (b > c ? b : c);
}

void launch_layernorm_bwd(const Launch& L, bool bf16, const void* x, const void* w,
                          const float* mean, const float* rstd, const void* dy, void* dx,
                          float* dw, float* db, int M, int C, bool accumulate, float* scratch,
                          bool acc_params, float* dres) {
    if (bf16 && launch_ln_bwd_bf16(L, x, w, mean, rstd, dy, dx, dw, db, M, C, accumulate, scratch, acc_params,
                                   dres))
        return;
    if (L.dry) return;
    const int nblk = (M + LN_ROWS - 1) / LN_ROWS;
    const size_t smem = (size_t)LN_BWD_WARPS * 2 * C * sizeof(float);
    static PerDevice attr;
    attr.once([] {
        const int max_smem = LN_BWD_WARPS * 2 * 1024 * (int)sizeof(float);
        cudaFuncSetAttribute(k_layernorm_bwd<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        cudaFuncSetAttribute(k_layernorm_bwd<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             max_smem);
        cudaFuncSetAttribute(k_layernorm_bwd<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        return true;
    });
    L.count();
    if (bf16 && L.f16)
        k_layernorm_bwd<__half><<<nblk, LN_BWD_WARPS * 32, smem, L.stream>>>(
            (const __half*)x, (const __half*)w, mean, rstd,
            (const __half*)dy, (__half*)dx, scratch, M, C, accumulate ? 1 : 0);
    else if (bf16)
        k_layernorm_bwd<__nv_bfloat16><<<nblk, LN_BWD_WARPS * 32, smem, L.stream>>>(
            (const __nv_bfloat16*)x, (const __nv_bfloat16*)w, mean, rstd,
            (const __nv_bfloat16*)dy, (__nv_bfloat16*)dx, scratch, M, C, accumulate ? 1 : 0);
    else
        k_layernorm_bwd<float><<<nblk, LN_BWD_WARPS * 32, smem, L.stream>>>(
            (const float*)x, (const float*)w, mean, rstd, (const float*)dy, (float*)dx, scratch,
            M, C, accumulate ? 1 : 0);
    L.count();
    k_sum_partials<<<blocks_for(2 * C, 256), 256, 0, L.stream>>>(scratch, nblk, C, dw, db, acc_params ? 1 : 0);
    // the column sums of the finished dx, in a second pass (the scratch is free
    // again once the partials above are summed: stream order)
    if (dres) launch_colsum(L, bf16, dx, M, C, dres, scratch, acc_params);
}

// ================================================================== cross entropy
// One block per row.  Pass 1: per-thread online (max, sum of exp), combined
// across the block; pass 2 overwrites the logits with the gradient.
constexpr int XENT_THREADS = 512;

__device__ __forceinline__ void online_merge(float& m, float& s, float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) { m = m2; s = s2; return; }
    if (m2 > m) { s = s * expf(m - m2) + s2; m = m2; }
    else s += s2 * expf(m2 - m);
}

template <typename T>
__global__ void __launch_bounds__(XENT_THREADS)
k_xent(T* __restrict__ z, const int32_t* __restrict__ targets, float* __restrict__ row_loss,
       int V, int ld_, float dscale, const float* __restrict__ scale_dev, int* flags) {
    __shared__ float s_m[XENT_THREADS / 32], s_s[XENT_THREADS / 32];
    if (scale_dev) dscale *= *scale_dev;
    __shared__ float s_lse;
    const long long row = blockIdx.x;
    T* zr = z + row * (long long)ld_;
    float m = -INFINITY, s = 0.0f;
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
        float x = ld(zr, v);
        if (x > m) { s = (m == -INFINITY ? 0.0f : s * expf(m - x)) + 1.0f; m = x; }
        else s += expf(x - m);
    }
    // warp combine
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        online_merge(m, s, m2, s2);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) { s_m[warp] = m; s_s[warp] = s; }
    __syncthreads();
    if (threadIdx.x == 0) {
        float M_ = s_m[0], S_ = s_s[0];
        for (int k = 1; k < (int)(blockDim.x >> 5); k++) online_merge(M_, S_, s_m[k], s_s[k]);
        s_lse = M_ + logf(S_);
    }
    __syncthreads();
    const float lse = s_lse;
    const int tgt = targets[row];
    const bool ok = tgt >= 0 && tgt < V;
    if (threadIdx.x == 0) {
        if (!ok) { atomicOr(&flags[FLAG_BAD_TOKEN], 1); row_loss[row] = 0.0f; }
        else row_loss[row] = lse - ld(zr, tgt);
    }
    __syncthreads();  // z[tgt] is read above before it is overwritten below
    for (int v = threadIdx.x; v < ld_; v += blockDim.x) {
        float g = 0.0f;
        if (v < V) {
            g = expf(ld(zr, v) - lse);
            if (v == tgt) g -= 1.0f;
            g *= dscale;
        }
        st(zr, v, g);
    }
}

// mean over rows in a fixed order (one block, per-thread strided partials,
// combined in thread order)
__global__ void k_mean_loss(const float* __restrict__ row_loss, int M, float* __restrict__ out,
                            int* flags) {
    pdl_enter();
    __shared__ float s_p[1024];
    float s = 0.0f;
    for (int i = threadIdx.x; i < M; i += blockDim.x) s += row_loss[i];
    s_p[threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int k = 0; k < (int)blockDim.x; k++) t += s_p[k];
        t /= (float)M;
        out[0] = t;
        if (!isfinite(t)) atomicOr(&flags[FLAG_NONFINITE], 1);
    }
}

void launch_xent(const Launch& L, bool bf16, void* logits, const int32_t* targets,
                 float* row_loss, float* mean_loss, int M, int V, int ld_, float dscale,
                 const float* scale_dev) {
    if (L.dry) return;
    if (bf16 && launch_xent_bf16(L, logits, targets, row_loss, M, V, ld_, dscale, scale_dev)) {
        if (mean_loss) {
            L.count();
            launch_k(L, k_mean_loss, dim3(1), dim3(1024), 0, row_loss, M, mean_loss, L.flags);
        }
        return;
    }
    L.count();
    if (bf16 && L.f16)
        k_xent<__half><<<M, XENT_THREADS, 0, L.stream>>>(
            (__half*)logits, targets, row_loss, V, ld_, dscale, scale_dev, L.flags);
    else if (bf16)
        k_xent<__nv_bfloat16><<<M, XENT_THREADS, 0, L.stream>>>(
            (__nv_bfloat16*)logits, targets, row_loss, V, ld_, dscale, scale_dev, L.flags);
    else
        k_xent<float><<<M, XENT_THREADS, 0, L.stream>>>((float*)logits, targets, row_loss, V, ld_,
                                                        dscale, scale_dev, L.flags);
    if (mean_loss) {
        L.count();
        launch_k(L, k_mean_loss, dim3(1), dim3(1024), 0, row_loss, M, mean_loss, L.flags);
    }
}

// ================================================================== column sums
constexpr int COLSUM_ROWS = 256;

template <typename T>
__global__ void k_colsum_part(const T* __restrict__ x, int M, int N, float* __restrict__ part) {
    int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    long long r0 = (long long)blockIdx.y * COLSUM_ROWS;
    long long r1 = min((long long)M, r0 + COLSUM_ROWS);
    float s = 0.0f;
    for (long long r = r0; r < r1; r++) s += ld(x, r * N + n);
    part[(long long)blockIdx.y * N + n] = s;
}

__global__ void k_colsum_final(const float* __restrict__ part, int nchunk, int N,
                               float* __restrict__ out, int acc) {
    int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    float s = 0.0f;
    for (int c = 0; c < nchunk; c++) s += part[(long long)c * N + n];
    out[n] = acc ? out[n] + s : s;
}

size_t colsum_scratch_floats(int M, int N) {
    return (size_t)((M + COLSUM_ROWS - 1) / COLSUM_ROWS) * N + 64;
}

void launch_colsum(const Launch& L, bool bf16, const void* x, int M, int N, float* out,
                   float* scratch, bool acc) {
    if (L.dry) return;
    int nchunk = (M + COLSUM_ROWS - 1) / COLSUM_ROWS;
    if (bf16 && launch_colsum_bf16(L, x, M, N, scratch)) {
        launch_sum_rows(L, scratch, nchunk, N, N, out, nullptr, acc);
        return;
    }
    dim3 grid(blocks_for(N, 128), nchunk);
    L.count();
    if (bf16 && L.f16)
        k_colsum_part<__half><<<grid, 128, 0, L.stream>>>((const __half*)x, M, N, scratch);
    else if (bf16)
        k_colsum_part<__nv_bfloat16><<<grid, 128, 0, L.stream>>>((const __nv_bfloat16*)x, M, N, scratch);
    else
        k_colsum_part<float><<<grid, 128, 0, L.stream>>>((const float*)x, M, N, scratch);
    L.count();
    k_colsum_final<<<blocks_for(N, 256), 256, 0, L.stream>>>(scratch, nchunk, N, out, acc ? 1 : 0);
}

// ================================================================== AdamW
// Flat, grid-stride, four elements per thread per iteration (128-bit loads).
template <typename LT>
__global__ void k_adamw(float* __restrict__ p, LT* __restrict__ lowp,
                        const float* __restrict__ g, float* __restrict__ m, float* __restrict__ v,
                        size_t n, float lr, float b1, float b2, float eps, float wd, float c1,
                        float c2) {
    pdl_enter();
    const size_t n4 = n / 4;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 pp = reinterpret_cast<const float4*>(p)[i];
        float4 gg = reinterpret_cast<const float4*>(g)[i];
        float4 mm = reinterpret_cast<const float4*>(m)[i];
        float4 vv = reinterpret_cast<const float4*>(v)[i];
        float* pe = &pp.x; float* ge = &gg.x; float* me = &mm.x; float* ve = &vv.x;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            me[j] = b1 * me[j] + (1.0f - b1) * ge[j];
            ve[j] = b2 * ve[j] + (1.0f - b2) * ge[j] * ge[j];
            float mh = me[j] / c1;
            float vh = ve[j] / c2;
            pe[j] -= lr * (mh / (sqrtf(vh) + eps) + wd * pe[j]);
        }
        reinterpret_cast<float4*>(p)[i] = pp;
        reinterpret_cast<float4*>(m)[i] = mm;
        reinterpret_cast<float4*>(v)[i] = vv;
        if (lowp) st_low4(lowp, i, pp);
    }
    // tail (n not a multiple of 4)
    for (size_t i = n4 * 4 + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        float mm = b1 * m[i] + (1.0f - b1) * g[i];
        float vv = b2 * v[i] + (1.0f - b2) * g[i] * g[i];
        m[i] = mm;
        v[i] = vv;
        float pp = p[i] - lr * ((mm / c1) / (sqrtf(vv / c2) + eps) + wd * p[i]);
        p[i] = pp;
        if (lowp) st(lowp, (long long)i, pp);
    }
}

void launch_adamw(const Launch& L, float* master, void* lowp, const float* g, float* m,
                  float* v, size_t n, float lr, float b1, float b2, float eps, float wd, int step) {
    if (L.dry || n == 0) return;
    float c1 = (float)(1.0 - pow((double)b1, step));
    float c2 = (float)(1.0 - pow((double)b2, step));
    long long want = (long long)((n / 4 + 255) / 256);
    int grid = (int)(want < (long long)L.num_sms * 8 ? (want < 1 ? 1 : want) : (long long)L.num_sms * 8);
    L.count();
    if (L.f16)
        launch_k(L, k_adamw<__half>, dim3(grid), dim3(256), 0, master, (__half*)lowp, g, m, v, n, lr, b1, b2, eps, wd, c1, c2);
    else
        launch_k(L, k_adamw<__nv_bfloat16>, dim3(grid), dim3(256), 0, master, (__nv_bfloat16*)lowp, g, m, v, n, lr, b1, b2, eps, wd, c1, c2);
}

template <typename T>
__global__ void k_cast_low(const float* __restrict__ s, T* __restrict__ d, size_t n) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) st(d, (long long)i, s[i]);
}

static int cast_grid(const Launch& L, size_t n) {
    long long want = (long long)((n + 255) / 256);
    return (int)(want < (long long)L.num_sms * 8 ? want : (long long)L.num_sms * 8);
}

void launch_cast_bf16(const Launch& L, const float* src, __nv_bfloat16* dst, size_t n) {
    if (L.dry || n == 0) return;
    L.count();
    k_cast_low<<<cast_grid(L, n), 256, 0, L.stream>>>(src, dst, n);
}

void launch_cast_f16(const Launch& L, const float* src, __half* dst, size_t n) {
    if (L.dry || n == 0) return;
    L.count();
    k_cast_low<<<cast_grid(L, n), 256, 0, L.stream>>>(src, dst, n);
}

// ================================================================== SIMT GEMM
// 64x64 output tile, 256 threads, 4x4 outputs per thread, K-step 16; operands
// are read through the generic (K-major / MN-major) indexing of GemmArgs and
// converted to fp32 in shared memory.  Used in fp32 mode and as the fallback.
constexpr int SG_T = 64, SG_K = 16;

template <typename TI, typename TO>
__global__ void __launch_bounds__(256)
k_gemm_simt(GemmArgs g) {
    __shared__ float sA[SG_K][SG_T + 4];
    __shared__ float sB[SG_K][SG_T + 4];
    const TI* A = (const TI*)g.A;
    const TI* Bm = (const TI*)g.B;
    const int m0 = blockIdx.y * SG_T, n0 = blockIdx.x * SG_T;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int a_rows = g.a_rows ? g.a_rows : g.M;
    const int b_rows = g.b_rows ? g.b_rows : g.N;
    const int kval = g.k_valid ? g.k_valid : g.K;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = 0.0f;
    for (int k0 = 0; k0 < g.K; k0 += SG_K) {
        for (int e = threadIdx.x; e < SG_T * SG_K; e += 256) {
            int r, kk;
            if (g.a_kmajor) { r = e / SG_K; kk = e % SG_K; } else { kk = e / SG_T; r = e % SG_T; }
            int m = m0 + r, k = k0 + kk;
            float va = 0.0f;
            if (m < a_rows && m < g.M && k < kval)
                va = ld(A, g.a_kmajor ? (long long)m * g.lda + k : (long long)k * g.lda + m);
            sA[kk][r] = va;
            if (g.b_kmajor) { r = e / SG_K; kk = e % SG_K; } else { kk = e / SG_T; r = e % SG_T; }
            int n = n0 + r;
            k = k0 + kk;
            float vb = 0.0f;
            if (n < b_rows && n < g.N && k < kval)
                vb = ld(Bm, g.b_kmajor ? (long long)n * g.ldb + k : (long long)k * g.ldb + n);
            sB[kk][r] = vb;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SG_K; kk++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = sA[kk][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; j++) b[j] = sB[kk][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] += a[i] * b[j];
        }
        __syncthreads();
    }
    TO* D = (TO*)g.D;
    const TI* bias = (const TI*)g.bias;
    const TO* res = (const TO*)g.residual;
    TO* aux = (TO*)g.aux;
    const int nst = g.n_store ? g.n_store : g.N;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        int m = m0 + ty + 16 * i;
        if (m >= g.M) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            int n = n0 + tx + 16 * j;
            if (n >= g.N || n >= nst) continue;
            long long o = (long long)m * g.ldd + n;
            float v = acc[i][j];
            if (bias) v += ld(bias, n);
            if (g.epi == EPI_GELU) {
                st(aux, o, v);
                v = gelu_f(v);
            } else if (g.epi == EPI_DGELU) {
                v *= dgelu_f(ld(aux, o));
            }
            if (res) v += ld(res, o);
            if (g.accumulate) v += ld(D, o);
            st(D, o, v);
        }
    }
}

void gemm_simt_launch(const Launch& L, const GemmArgs& g) {
    if (L.dry) return;
    dim3 grid((g.N + SG_T - 1) / SG_T, (g.M + SG_T - 1) / SG_T);
    L.count();
    if (g.in_bf16 && g.in_f16) {
        if (g.d_f32) k_gemm_simt<__half, float><<<grid, 256, 0, L.stream>>>(g);
        else k_gemm_simt<__half, __half><<<grid, 256, 0, L.stream>>>(g);
    } else if (g.in_bf16) {
        if (g.d_f32) k_gemm_simt<__nv_bfloat16, float><<<grid, 256, 0, L.stream>>>(g);
        else k_gemm_simt<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, L.stream>>>(g);
    } else {
        k_gemm_simt<float, float><<<grid, 256, 0, L.stream>>>(g);
    }
}

// ================================================================== SIMT attention
// One thread per query row (forward, dq) or key row (dk, dv); one block per
// (batch, head).  Rows of the other side are read in lockstep by the lanes of
// a warp (same address: broadcast).  Sums run in increasing position order.
template <typename T, int HD>
__global__ void k_attn_fwd_simt(const T* __restrict__ qkv, T* __restrict__ y,
                                float* __restrict__ lse, int T_, int C, int H) {
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const long long ld3 = 3LL * C;
    const float scale = rsqrtf((float)HD);
    for (int t = threadIdx.x; t < T_; t += blockDim.x) {
        const T* qr = qkv + ((long long)b * T_ + t) * ld3 + h * HD;
        float q[HD], acc[HD];
#pragma unroll
        for (int i = 0; i < HD; i++) { q[i] = ld(qr, i) * scale; acc[i] = 0.0f; }
        float mx = -INFINITY, l = 0.0f;
        for (int s = 0; s <= t; s++) {
            const T* kr = qkv + ((long long)b * T_ + s) * ld3 + C + h * HD;
            const T* vr = kr + C;
            float sc = 0.0f;
#pragma unroll
            for (int i = 0; i < HD; i++) sc += q[i] * ld(kr, i);
            float mn = fmaxf(mx, sc);
            float corr = expf(mx - mn);  // mx = -inf at s = 0 gives 0
            float p = expf(sc - mn);
            l = l * corr + p;
#pragma unroll
            for (int i = 0; i < HD; i++) acc[i] = acc[i] * corr + p * ld(vr, i);
            mx = mn;
        }
        T* yr = y + ((long long)b * T_ + t) * C + h * HD;
        const float inv = 1.0f / l;
#pragma unroll
        for (int i = 0; i < HD; i++) st(yr, i, acc[i] * inv);
        lse[((long long)b * H + h) * T_ + t] = mx + logf(l);
    }
}

// D[b,h,t] = sum_i dy[t,i] * y[t,i]
template <typename T, int HD>
__global__ void k_attn_bwd_delta(const T* __restrict__ y, const T* __restrict__ dy,
                                 float* __restrict__ Dlt, int B, int T_, int C, int H) {
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)B * H * T_) return;
    int t = (int)(i % T_);
    int h = (int)((i / T_) % H);
    int b = (int)(i / ((long long)T_ * H));
    long long o = ((long long)b * T_ + t) * C + h * HD;
    float s = 0.0f;
#pragma unroll
    for (int d = 0; d < HD; d++) s += ld(dy, o + d) * ld(y, o + d);
    Dlt[i] = s;
}

template <typename T, int HD>
__global__ void k_attn_bwd_dq_simt(const T* __restrict__ qkv, const float* __restrict__ lse,
                                   const float* __restrict__ Dlt, const T* __restrict__ dy,
                                   T* __restrict__ dqkv, int T_, int C, int H) {
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const long long ld3 = 3LL * C;
    const float scale = rsqrtf((float)HD);
    for (int t = threadIdx.x; t < T_; t += blockDim.x) {
        const T* qr = qkv + ((long long)b * T_ + t) * ld3 + h * HD;
        const T* dyr = dy + ((long long)b * T_ + t) * C + h * HD;
        float q[HD], g[HD], dq[HD];
#pragma unroll
        for (int i = 0; i < HD; i++) { q[i] = ld(qr, i) * scale; g[i] = ld(dyr, i); dq[i] = 0.0f; }
        const long long bh = ((long long)b * H + h) * T_;
        const float L_ = lse[bh + t], Dt = Dlt[bh + t];
        for (int s = 0; s <= t; s++) {
            const T* kr = qkv + ((long long)b * T_ + s) * ld3 + C + h * HD;
            const T* vr = kr + C;
            float sc = 0.0f, dp = 0.0f;
#pragma unroll
            for (int i = 0; i < HD; i++) { sc += q[i] * ld(kr, i); dp += g[i] * ld(vr, i); }
            float p = expf(sc - L_);
            float ds = p * (dp - Dt);
#pragma unroll
            for (int i = 0; i < HD; i++) dq[i] += ds * ld(kr, i);
        }
        T* o = dqkv + ((long long)b * T_ + t) * ld3 + h * HD;
#pragma unroll
        for (int i = 0; i < HD; i++) st(o, i, dq[i] * scale);
    }
}

template <typename T, int HD>
__global__ void k_attn_bwd_dkv_simt(const T* __restrict__ qkv, const float* __restrict__ lse,
                                    const float* __restrict__ Dlt, const T* __restrict__ dy,
                                    T* __restrict__ dqkv, int T_, int C, int H) {
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const long long ld3 = 3LL * C;
    const float scale = rsqrtf((float)HD);
    for (int s = threadIdx.x; s < T_; s += blockDim.x) {
        const T* kr = qkv + ((long long)b * T_ + s) * ld3 + C + h * HD;
        const T* vr = kr + C;
        float k[HD], v[HD], dk[HD], dv[HD];
#pragma unroll
        for (int i = 0; i < HD; i++) { k[i] = ld(kr, i); v[i] = ld(vr, i); dk[i] = 0.0f; dv[i] = 0.0f; }
        const long long bh = ((long long)b * H + h) * T_;
        for (int t = s; t < T_; t++) {
            const T* qr = qkv + ((long long)b * T_ + t) * ld3 + h * HD;
            const T* dyr = dy + ((long long)b * T_ + t) * C + h * HD;
            float sc = 0.0f, dp = 0.0f;
#pragma unroll
            for (int i = 0; i < HD; i++) { sc += ld(qr, i) * k[i]; dp += ld(dyr, i) * v[i]; }
            float p = expf(sc * scale - lse[bh + t]);
            float ds = p * (dp - Dlt[bh + t]);
#pragma unroll
            for (int i = 0; i < HD; i++) {
                dv[i] += p * ld(dyr, i);
                dk[i] += ds * ld(qr, i);
            }
        }
        T* o = dqkv + ((long long)b * T_ + s) * ld3 + C + h * HD;
#pragma unroll
        for (int i = 0; i < HD; i++) { st(o, i, dk[i] * scale); st(o + C, i, dv[i]); }
    }
}

// D = rowsum(dO o O) [B, H, T], then the qkv bias-gradient partials: one row
// of 3C per (sequence, 128-row tile) for the tensor-core kernels, or the
// column-sum partials of the generic pass, whichever is larger
static size_t attn_d_floats(int B, int T, int H) { return ((size_t)B * H * T + 63) / 64 * 64; }
size_t attention_bwd_scratch_floats(int B, int T, int C, int H) {
    const size_t tiles = (size_t)B * ((T + 127) / 128) * 3 * C;
    const size_t cs = colsum_scratch_floats(B * T, 3 * C);
    return attn_d_floats(B, T, H) + (tiles > cs ? tiles : cs) + 64;
}

template <typename T, int HD>
static void attn_fwd_simt(const Launch& L, const void* qkv, void* y, float* lse, int B, int T_,
                          int C, int H) {
    int threads = T_ < 128 ? ((T_ + 31) / 32) * 32 : 128;
    L.count();
    k_attn_fwd_simt<T, HD><<<B * H, threads, 0, L.stream>>>((const T*)qkv, (T*)y, lse, T_, C, H);
}

template <typename T, int HD>
static void attn_bwd_simt(const Launch& L, const void* qkv, const void* y, const float* lse,
                          const void* dy, void* dqkv, int B, int T_, int C, int H, float* Dlt) {
    long long n = (long long)B * H * T_;
    L.count();
    k_attn_bwd_delta<T, HD><<<blocks_for(n, 256), 256, 0, L.stream>>>((const T*)y, (const T*)dy,
                                                                      Dlt, B, T_, C, H);
    int threads = T_ < 128 ? ((T_ + 31) / 32) * 32 : 128;
    L.count();
    k_attn_bwd_dq_simt<T, HD><<<B * H, threads, 0, L.stream>>>((const T*)qkv, lse, Dlt,
                                                               (const T*)dy, (T*)dqkv, T_, C, H);
    L.count();
    k_attn_bwd_dkv_simt<T, HD><<<B * H, threads, 0, L.stream>>>((const T*)qkv, lse, Dlt,
                                                                (const T*)dy, (T*)dqkv, T_, C, H);
}

#define TT_HD_DISPATCH(hd, FN, ...)                                             \
    do {                                                                        \
        if (bf16 && L.f16) {                                                    \
            if (hd == 16) FN<__half, 16>(__VA_ARGS__);                          \
            else if (hd == 32) FN<__half, 32>(__VA_ARGS__);                     \
            else FN<__half, 64>(__VA_ARGS__);                                   \
        } else if (bf16) {                                                      \
            if (hd == 16) FN<__nv_bfloat16, 16>(__VA_ARGS__);                   \
            else if (hd == 32) FN<__nv_bfloat16, 32>(__VA_ARGS__);              \
            else FN<__nv_bfloat16, 64>(__VA_ARGS__);                            \
        } else {                                                                \
            if (hd == 16) FN<float, 16>(__VA_ARGS__);                           \
            else if (hd == 32) FN<float, 32>(__VA_ARGS__);                      \
            else FN<float, 64>(__VA_ARGS__);                                    \
        }                                                                       \
    } while (0)

void launch_attention_fwd(const Launch& L, bool bf16, const void* qkv, void* y, float* lse,
                          int B, int T, int C, int H) {
    if (L.dry) return;
    const bool bf_only = bf16 && !L.f16;  // the mma.sync attention kernels are bf16 only
    // the tensor-core kernels take bf16 or half (L.f16)
    if (attention_tc_eligible(bf16, C, H) && launch_attention_fwd_tc(L, qkv, y, lse, B, T, C, H)) return;
    if (attention_mma_eligible(bf_only, C, H)) {
        launch_attention_fwd_mma(L, qkv, y, lse, B, T, C, H);
        return;
    }
    const int hd = C / H;
    TT_HD_DISPATCH(hd, attn_fwd_simt, L, qkv, y, lse, B, T, C, H);
}

void launch_attention_bwd(const Launch& L, bool bf16, const void* qkv, const void* y,
                          const float* lse, const void* dy, void* dqkv, int B, int T, int C,
                          int H, float* scratch, float* dbias, bool acc_bias) {
    if (L.dry) return;
    const bool bf_only = bf16 && !L.f16;
    float* bpart = scratch + attn_d_floats(B, T, H);
    if (attention_tc_eligible(bf16, C, H) &&
        launch_attention_bwd_tc(L, qkv, y, lse, dy, dqkv, B, T, C, H, scratch, dbias ? bpart : nullptr)) {
        if (dbias) launch_sum_rows(L, bpart, B * ((T + 127) / 128), 3 * C, 3 * C, dbias, nullptr, acc_bias);
        return;
    }
    if (attention_mma_eligible(bf_only, C, H)) {
        launch_attention_bwd_mma(L, qkv, y, lse, dy, dqkv, B, T, C, H, scratch);
    } else {
        const int hd = C / H;
        TT_HD_DISPATCH(hd, attn_bwd_simt, L, qkv, y, lse, dy, dqkv, B, T, C, H, scratch);
    }
    // the bias gradient of the qkv layer: column sums of dqkv, a second pass
    if (dbias) launch_colsum(L, bf16, dqkv, B * T, 3 * C, dbias, bpart, acc_bias);
}

}  // namespace tt

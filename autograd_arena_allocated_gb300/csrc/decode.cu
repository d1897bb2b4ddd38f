// decode.cu -- the kernels of autoregressive decoding with a key/value cache
// (the Forge page, 性能瓶颈与未来路线图: each new token's query is dotted with
// the cached keys of the earlier positions instead of recomputing them).
//
//   k_kv_fill      keys and values of a qkv tensor into the cache
//   k_embed_at     x[b] = wte[token(b, pos)] + wpe[pos]
//   k_decode_attn  one query per sequence against its cached keys 0..pos
//   k_argmax       greedy choice over the vocabulary (lowest index on ties)
//
// The cache holds, per layer, [B, maxT, 2C]: the key row then the value row of
// each position, in the storage type of the step.  Every reduction is in a
// fixed order, so decoding is deterministic.
#include "tt_internal.h"

#include <algorithm>

namespace tt {
namespace {

template <typename T> __device__ __forceinline__ float ld_f(const T* p);
template <> __device__ __forceinline__ float ld_f<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ T st_f(float v);
template <> __device__ __forceinline__ float st_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 st_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// cache[b][t0 + t][0 : 2C] = qkv[b*T + t][C : 3C]
template <typename T>
__global__ void k_kv_fill(const T* __restrict__ qkv, T* __restrict__ cache, int B, int Tn, int C, int t0,
                          int maxT) {
    const long long n = (long long)B * Tn * 2 * C;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(i % (2 * C));
        const long long r = i / (2 * C);
        const int t = (int)(r % Tn), b = (int)(r / Tn);
        cache[((long long)b * maxT + t0 + t) * 2 * C + c] = qkv[r * 3 * C + C + c];
    }
}

template <typename T>
__global__ void k_embed_at(const T* __restrict__ wte, const T* __restrict__ wpe, const int32_t* __restrict__ tok,
                           int ld_tok, int pos, T* __restrict__ x, int B, int C, int V, int* flags) {
    const int b = blockIdx.x;
    int id = tok[(long long)b * ld_tok + pos];
    if (id < 0 || id >= V) {
        if (threadIdx.x == 0) atomicOr(&flags[FLAG_BAD_TOKEN], 1);
        id = 0;
    }
    for (int c = threadIdx.x; c < C; c += blockDim.x)
        x[(long long)b * C + c] = st_f<T>(ld_f(wte + (long long)id * C + c) + ld_f(wpe + (long long)pos * C + c));
}

// One CTA (128 threads) per (b, h): the query (head dimension D <= 64) of the
// sequence's newest position against keys 0..pos.  Scores go to shared
// memory, then the max and the sum in a fixed order, then thread d of each
// half adds p_k v_k[d] over its half of the keys, and the halves are added.
constexpr int DA_THREADS = 128;
constexpr int DA_MAXT = 1024;

template <typename T>
__global__ void __launch_bounds__(DA_THREADS)
k_decode_attn(const T* __restrict__ qkv, const T* __restrict__ cache, T* __restrict__ y, int H, int C, int pos,
              int maxT, float scale) {
    __shared__ float s_p[DA_MAXT];
    __shared__ float s_q[64];
    __shared__ float s_red[DA_THREADS / 32];
    __shared__ float s_half[64];
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const int D = C / H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nk = pos + 1;
    if (tid < D) s_q[tid] = ld_f(qkv + (long long)b * 3 * C + h * D + tid);
    __syncthreads();
    const T* kb = cache + (long long)b * maxT * 2 * C + h * D;  // key k at kb + k * 2C
    float mx = -INFINITY;
    for (int k = tid; k < nk; k += DA_THREADS) {
        const T* kr = kb + (long long)k * 2 * C;
        float s = 0.0f;
        for (int d = 0; d < D; d++) s = fmaf(s_q[d], ld_f(kr + d), s);
        s *= scale;
        s_p[k] = s;
        mx = fmaxf(mx, s);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_red[warp] = mx;
    __syncthreads();
    mx = s_red[0];
#pragma unroll
    for (int w = 1; w < DA_THREADS / 32; w++) mx = fmaxf(mx, s_red[w]);
    __syncthreads();
    float sum = 0.0f;
    for (int k = tid; k < nk; k += DA_THREADS) {
        const float p = expf(s_p[k] - mx);
        s_p[k] = p;
        sum += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) s_red[warp] = sum;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < DA_THREADS / 32; w++) tot += s_red[w];
    // y[d] = sum_k p_k v_k[d] / tot: thread (half, d) takes keys half, half + 2, ...
    const int d = tid & 63, half = tid >> 6;
    float acc = 0.0f;
    if (d < D) {
        const T* vb = kb + C + d;
        for (int k = half; k < nk; k += 2) acc = fmaf(s_p[k], ld_f(vb + (long long)k * 2 * C), acc);
    }
    if (half == 1 && d < D) s_half[d] = acc;
    __syncthreads();
    if (half == 0 && d < D) y[(long long)b * C + h * D + d] = st_f<T>((acc + s_half[d]) / tot);
}

// Greedy choice per row: the first index of the largest of z[0 .. V-1].
constexpr int AM_THREADS = 512;

template <typename T>
__global__ void __launch_bounds__(AM_THREADS)
k_argmax(const T* __restrict__ z, long long row_stride, int V, int32_t* __restrict__ out, int ld_out, int col) {
    __shared__ float s_v[AM_THREADS / 32];
    __shared__ int s_i[AM_THREADS / 32];
    const int b = blockIdx.x;
    const T* zr = z + (long long)b * row_stride;
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = threadIdx.x; i < V; i += AM_THREADS) {
        const float v = ld_f(zr + i);
        if (v > best) { best = v; bi = i; }  // i increases: the first maximum is kept
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) { s_v[warp] = best; s_i[warp] = bi; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < AM_THREADS / 32; w++)
            if (s_v[w] > best || (s_v[w] == best && s_i[w] < bi)) { best = s_v[w]; bi = s_i[w]; }
        out[(long long)b * ld_out + col] = bi == 0x7fffffff ? 0 : bi;
    }
}

// Skinny GEMM for decode steps (M <= 16 rows): D[m, n] = sum_k A[m, k] W[n, k]
// (+ bias[n]) then GELU (keeping the pre-activation) or + residual[m, n].  The
// weights dominate the bytes: one warp per output column n streams W's row
// with 16-byte loads and dots it with all M rows of A (read through L1), then
// each of the M sums is reduced across the warp in a fixed order.
constexpr int SK_MMAX = 16;
constexpr int SK_WARPS = 8;

template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
    __device__ static void load(const __nv_bfloat16* p, float* f) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};
template <> struct Vec8<float> {
    __device__ static void load(const float* p, float* f) {
        const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
};

__device__ __forceinline__ float gelu_tanh_f(float u) {
    const float k = 0.7978845608028654f, a = 0.044715f;
    return 0.5f * u * (1.0f + tanhf(k * (u + a * u * u * u)));
}

template <typename T>
__global__ void __launch_bounds__(SK_WARPS * 32)
k_gemm_skinny(const T* __restrict__ A, const T* __restrict__ W, const T* __restrict__ bias,
              const T* __restrict__ res, T* __restrict__ D, T* __restrict__ pre, int M, int N, int K, int ldd,
              int n_store, int gelu) {
    const int lane = threadIdx.x & 31;
    for (int n = blockIdx.x * SK_WARPS + (threadIdx.x >> 5); n < N; n += gridDim.x * SK_WARPS) {
        float acc[SK_MMAX];
#pragma unroll
        for (int m = 0; m < SK_MMAX; m++) acc[m] = 0.0f;
        const T* wr = W + (long long)n * K;
        for (int k = lane * 8; k < K; k += 32 * 8) {
            float w[8];
            Vec8<T>::load(wr + k, w);
#pragma unroll
            for (int m = 0; m < SK_MMAX; m++) {
                if (m < M) {
                    float a[8];
                    Vec8<T>::load(A + (long long)m * K + k, a);
#pragma unroll
                    for (int e = 0; e < 8; e++) acc[m] = fmaf(a[e], w[e], acc[m]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < SK_MMAX; m++) {
            if (m < M) {
                float v = acc[m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[m] = v;
            }
        }
        if (lane == 0 && n < n_store) {
            const float bv = bias ? ld_f(bias + n) : 0.0f;
            for (int m = 0; m < M; m++) {
                float v = acc[m] + bv;
                const long long o = (long long)m * ldd + n;
                if (gelu) {
                    pre[o] = st_f<T>(v);
                    v = gelu_tanh_f(ld_f(pre + o));  // from the stored pre-activation, as the backward sees it
                } else if (res) {
                    v += ld_f(res + o);
                }
                D[o] = st_f<T>(v);
            }
        }
    }
}

static unsigned grid_for(long long n, int threads) {
    long long g = (n + threads - 1) / threads;
    return (unsigned)(g < 1 ? 1 : (g > 65535 ? 65535 : g));
}

}  // namespace

bool launch_kv_fill(const Launch& L, bool bf16, const void* qkv, void* cache, int B, int Tn, int C, int t0,
                    int maxT) {
    if (t0 < 0 || t0 + Tn > maxT) return false;
    if (L.dry) return true;
    L.count();
    const unsigned g = grid_for((long long)B * Tn * 2 * C, 256);
    if (bf16)
        k_kv_fill<__nv_bfloat16><<<g, 256, 0, L.stream>>>((const __nv_bfloat16*)qkv, (__nv_bfloat16*)cache, B, Tn,
                                                          C, t0, maxT);
    else
        k_kv_fill<float><<<g, 256, 0, L.stream>>>((const float*)qkv, (float*)cache, B, Tn, C, t0, maxT);
    return true;
}

void launch_embed_at(const Launch& L, bool bf16, const void* wte, const void* wpe, const int32_t* tok,
                     int ld_tok, int pos, void* x, int B, int C, int V) {
    if (L.dry) return;
    L.count();
    if (bf16)
        k_embed_at<__nv_bfloat16><<<B, 256, 0, L.stream>>>((const __nv_bfloat16*)wte, (const __nv_bfloat16*)wpe,
                                                           tok, ld_tok, pos, (__nv_bfloat16*)x, B, C, V, L.flags);
    else
        k_embed_at<float><<<B, 256, 0, L.stream>>>((const float*)wte, (const float*)wpe, tok, ld_tok, pos,
                                                   (float*)x, B, C, V, L.flags);
}

bool launch_decode_attn(const Launch& L, bool bf16, const void* qkv, const void* cache, void* y, int B, int H,
                        int C, int pos, int maxT) {
    if (C % H || C / H > 64 || pos + 1 > DA_MAXT || pos >= maxT) return false;
    if (L.dry) return true;
    L.count();
    const float scale = 1.0f / sqrtf((float)(C / H));
    if (bf16)
        k_decode_attn<__nv_bfloat16><<<B * H, DA_THREADS, 0, L.stream>>>(
            (const __nv_bfloat16*)qkv, (const __nv_bfloat16*)cache, (__nv_bfloat16*)y, H, C, pos, maxT, scale);
    else
        k_decode_attn<float><<<B * H, DA_THREADS, 0, L.stream>>>((const float*)qkv, (const float*)cache, (float*)y,
                                                                 H, C, pos, maxT, scale);
    return true;
}

bool launch_gemm_skinny(const Launch& L, bool bf16, const void* A, const void* W, const void* bias, const void* res,
                        void* D, void* pre, int M, int N, int K, int ldd, int n_store, bool gelu) {
    const size_t es = bf16 ? 2 : 4;
    if (M < 1 || M > SK_MMAX || K % 8 || ((uintptr_t)A & 15) || ((uintptr_t)W & 15) || ((K * es) & 15)) return false;
    if (L.dry) return true;
    L.count();
    const unsigned grid = (unsigned)std::min<long long>((N + SK_WARPS - 1) / SK_WARPS, 65535);
    if (bf16)
        k_gemm_skinny<__nv_bfloat16><<<grid, SK_WARPS * 32, 0, L.stream>>>(
            (const __nv_bfloat16*)A, (const __nv_bfloat16*)W, (const __nv_bfloat16*)bias, (const __nv_bfloat16*)res,
            (__nv_bfloat16*)D, (__nv_bfloat16*)pre, M, N, K, ldd, n_store, gelu ? 1 : 0);
    else
        k_gemm_skinny<float><<<grid, SK_WARPS * 32, 0, L.stream>>>((const float*)A, (const float*)W, (const float*)bias,
                                                                   (const float*)res, (float*)D, (float*)pre, M, N, K,
                                                                   ldd, n_store, gelu ? 1 : 0);
    return true;
}

void launch_argmax(const Launch& L, bool bf16, const void* z, long long row_stride, int rows, int V, int32_t* out,
                   int ld_out, int col) {
    if (L.dry) return;
    L.count();
    if (bf16)
        k_argmax<__nv_bfloat16><<<rows, AM_THREADS, 0, L.stream>>>((const __nv_bfloat16*)z, row_stride, V, out,
                                                                   ld_out, col);
    else
        k_argmax<float><<<rows, AM_THREADS, 0, L.stream>>>((const float*)z, row_stride, V, out, ld_out, col);
}

}  // namespace tt

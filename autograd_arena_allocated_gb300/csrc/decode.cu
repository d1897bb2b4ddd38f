// decode.cu -- the kernels of autoregressive decoding with a key/value cache
// (the Forge page, 性能瓶颈与未来路线图: each new token's query is dotted with
// the cached keys of the earlier positions instead of recomputing them).
//
//   k_kv_fill          keys and values of a prompt's qkv tensor into the cache
//   k_embed_at         x[b] = wte[token(b, pos)] + wpe[pos]
//   k_decode_attn      one query per sequence against its cached keys 0..pos,
//                      split over CTAs of 128 keys; the newest key and value
//                      join the cache on the way
//   k_gemm_skinny_mma  bf16 linear layers of a decode step (M <= 16 rows) on
//                      the tensor cores, weights streamed once
//   k_gemm_skinny      the same in fp32 with FMAs
//   k_pick / k_argmax  greedy choice (lowest index on ties)
//
// The newest position lives in device memory (pos_dev) and the step's last
// linear layer advances it, so one captured decode step replays for every
// position.  Within a step the kernels use programmatic dependent launch:
// each lets the next one start at its own entry, and each waits for its
// predecessor's results (griddepcontrol.wait) before it reads them; the
// skinny GEMM issues its weight loads, which nothing in the step writes,
// before that wait.  The cache holds, per layer, [B, maxT, 2C]: the key row then the
// value row of each position, in the storage type of the step.  Every
// reduction is in a fixed order, so decoding is deterministic.
#include "tt_internal.h"

#include <algorithm>
#include <utility>

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

// eight consecutive elements as floats (16 bytes of bf16, 32 of fp32; aligned)
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

__global__ void k_set_int(int* p, int v) { *p = v; }
__global__ void k_add_int(int* p, int v) { *p += v; }

template <typename T>
__global__ void k_embed_at(const T* __restrict__ wte, const T* __restrict__ wpe, const int32_t* __restrict__ tok,
                           int ld_tok, const int* __restrict__ pos_dev, T* __restrict__ x, int B, int C, int V,
                           int* flags) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x, pos = *pos_dev;
    int id = tok[(long long)b * ld_tok + pos];
    if (id < 0 || id >= V) {
        if (threadIdx.x == 0) atomicOr(&flags[FLAG_BAD_TOKEN], 1);
        id = 0;
    }
    for (int c = threadIdx.x; c < C; c += blockDim.x)
        x[(long long)b * C + c] = st_f<T>(ld_f(wte + (long long)id * C + c) + ld_f(wpe + (long long)pos * C + c));
}

// ---------------------------------------------------------------- attention
// CTA (b, h, s) takes keys [128 s, 128 s + 128) of the nk = pos + 1 keys.
// 256 threads: lane j of each group of eight holds head elements 8j..8j+7,
// and the 32 groups take one key each per 32.  Scores, then this split's max
// m_s and sum l_s = sum exp(score - m_s), then o_s = sum exp(score - m_s) v.
// With one split the CTA writes y = o_s / l_s.  Otherwise each split stores
// (m_s, l_s, o_s) and the CTA that finishes last (a counter per (b, h), reset
// by that CTA) combines the splits in split order:
//   y = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s,   M = max_s m_s.
constexpr int DA_THREADS = 256;
constexpr int DA_KEYS = 128;     // keys per CTA
constexpr int DA_DMAX = 64;      // head dimension bound
constexpr int DA_PART = DA_DMAX + 2;

template <typename T>
__global__ void __launch_bounds__(DA_THREADS)
k_decode_attn(const T* __restrict__ qkv, T* __restrict__ cache, T* __restrict__ y, int H, int C,
              const int* __restrict__ pos_dev, int maxT, int S, float scale, float* __restrict__ part,
              int* __restrict__ counter) {
    __shared__ float s_p[DA_KEYS];
    __shared__ float s_acc[32][DA_DMAX];
    __shared__ float s_red[DA_THREADS / 32];
    __shared__ int s_last;
    pdl_trigger();
    pdl_wait();
    const int bh = blockIdx.x / S, s = blockIdx.x % S;
    const int b = bh / H, h = bh % H;
    const int D = C / H;
    const int pos = *pos_dev, nk = pos + 1;
    const int k_lo = s * DA_KEYS;
    if (k_lo >= nk) return;  // an empty split: not counted below
    const int k_hi = min(k_lo + DA_KEYS, nk);
    const int n_split = (nk + DA_KEYS - 1) / DA_KEYS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = lane & 7, grp = warp * 4 + (lane >> 3);
    const bool act = j * 8 < D;
    const T* qrow = qkv + (long long)b * 3 * C;
    T* crow = cache + (long long)b * maxT * 2 * C;
    // the newest key and value join the cache (read from qkv below)
    if (k_hi == nk && tid < D) {
        crow[(long long)pos * 2 * C + h * D + tid] = qrow[C + h * D + tid];
        crow[(long long)pos * 2 * C + C + h * D + tid] = qrow[2 * C + h * D + tid];
    }
    auto key_row = [&](int k) -> const T* {
        return k == pos ? qrow + C + h * D : crow + (long long)k * 2 * C + h * D;
    };
    float q[8];
    if (act) Vec8<T>::load(qrow + h * D + 8 * j, q);
    else {
#pragma unroll
        for (int e = 0; e < 8; e++) q[e] = 0.0f;
    }
    // scores: key k_lo + 32 u + grp
    float kv[4][8];
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int k = k_lo + 32 * u + grp;
        if (act && k < k_hi) Vec8<T>::load(key_row(k) + 8 * j, kv[u]);
        else {
#pragma unroll
            for (int e = 0; e < 8; e++) kv[u][e] = 0.0f;
        }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < 4; u++) {
        float d = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; e++) d = fmaf(q[e], kv[u][e], d);
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        const int k = k_lo + 32 * u + grp;
        if (k < k_hi) {
            d *= scale;
            if (j == 0) s_p[k - k_lo] = d;
            mx = fmaxf(mx, d);
        }
    }
    // the value rows, loaded while the softmax statistics are reduced
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int k = k_lo + 32 * u + grp;
        if (act && k < k_hi) Vec8<T>::load(key_row(k) + C + 8 * j, kv[u]);
        else {
#pragma unroll
            for (int e = 0; e < 8; e++) kv[u][e] = 0.0f;
        }
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
    if (tid < k_hi - k_lo) {
        const float p = expf(s_p[tid] - mx);
        s_p[tid] = p;
        sum = p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) s_red[warp] = sum;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < DA_THREADS / 32; w++) tot += s_red[w];
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; e++) acc[e] = 0.0f;
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int k = k_lo + 32 * u + grp;
        if (k < k_hi) {
            const float p = s_p[k - k_lo];
#pragma unroll
            for (int e = 0; e < 8; e++) acc[e] = fmaf(p, kv[u][e], acc[e]);
        }
    }
    if (act) {
#pragma unroll
        for (int e = 0; e < 8; e++) s_acc[grp][8 * j + e] = acc[e];
    }
    __syncthreads();
    float o = 0.0f;
    if (tid < D) {
        for (int g = 0; g < 32; g++) o += s_acc[g][tid];
    }
    T* yr = y + (long long)b * C + h * D;
    if (n_split == 1) {
        if (tid < D) yr[tid] = st_f<T>(o / tot);
        return;
    }
    float* pp = part + ((long long)bh * S + s) * DA_PART;
    if (tid < D) pp[2 + tid] = o;
    if (tid == 0) { pp[0] = mx; pp[1] = tot; }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&counter[bh], 1) == n_split - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float* pb = part + (long long)bh * S * DA_PART;
    float M = -INFINITY;
    for (int t = 0; t < n_split; t++) M = fmaxf(M, __ldcg(pb + t * DA_PART));
    if (tid < D) {
        float num = 0.0f, den = 0.0f;
        for (int t = 0; t < n_split; t++) {
            const float w = expf(__ldcg(pb + t * DA_PART) - M);
            den = fmaf(w, __ldcg(pb + t * DA_PART + 1), den);
            num = fmaf(w, __ldcg(pb + t * DA_PART + 2 + tid), num);
        }
        yr[tid] = st_f<T>(num / den);
    }
    if (tid == 0) counter[bh] = 0;
}

// ---------------------------------------------------------------- greedy choice
// Order-preserving key of (value, index): larger values first, then smaller
// indices, so the largest key is the first maximum.  -0 counts as +0.
__device__ __forceinline__ unsigned long long pick_key(float v, int n) {
    uint32_t u = __float_as_uint(v);
    if ((u & 0x7FFFFFFFu) == 0) u = 0;
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)n);
}

// tok[b][pos] = index of the largest key among the nct partial keys of row b
__global__ void __launch_bounds__(256)
k_pick(const unsigned long long* __restrict__ keys, int nct, int32_t* __restrict__ tok, int ld_tok,
       const int* __restrict__ pos_dev) {
    __shared__ unsigned long long s_k[8];
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    unsigned long long best = 0;
    for (int i = threadIdx.x; i < nct; i += 256) best = max(best, keys[(long long)b * nct + i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
    if ((threadIdx.x & 31) == 0) s_k[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < 8; w++) best = max(best, s_k[w]);
        tok[(long long)b * ld_tok + *pos_dev] = best ? (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull)) : 0;
    }
}

// Greedy choice per row over stored logits: the first index of the largest of
// z[0 .. V-1], written to out[b][col] (col from col_dev when that is given).
constexpr int AM_THREADS = 512;

template <typename T>
__global__ void __launch_bounds__(AM_THREADS)
k_argmax(const T* __restrict__ z, long long row_stride, int V, int32_t* __restrict__ out, int ld_out, int col,
         const int* __restrict__ col_dev) {
    __shared__ float s_v[AM_THREADS / 32];
    __shared__ int s_i[AM_THREADS / 32];
    pdl_trigger();
    pdl_wait();
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
        out[(long long)b * ld_out + (col_dev ? *col_dev : col)] = bi == 0x7fffffff ? 0 : bi;
    }
}

// ---------------------------------------------------------------- skinny GEMMs
// D[m, n] = sum_k A[m, k] W[n, k] (+ bias[n]) then GELU (keeping the
// pre-activation) or + residual[m, n], for M <= 16 rows: the weights dominate
// the bytes and are streamed once.
//
// bf16: the tensor cores, one mma.sync m16n8k16 per 16 output columns x 8 rows
// x 16 k, with W as the 16-row operand and A^T as the 8-column one.  A dot
// product may take its k terms in any order as long as both operands agree,
// so each thread loads 16 contiguous bytes (8 k) of its W rows and of its A
// row and feeds them to two mma k-steps: step s takes the thread's k pairs 2s
// and 2s+1 where the instruction expects the pairs at k = 2q and 2q+8.  A CTA
// owns 16 output columns; its 8 warps split K in chunks of 32 (chunk c to warp
// c mod 8) and the partial sums meet in shared memory in warp order.
//
// With ln_w/ln_b the rows of A are first put through LayerNorm (the
// arithmetic of the step's LayerNorm kernel, rounded to bf16) into shared
// memory by the CTA itself, after its first weight loads are in flight: the
// decode step then needs no separate LayerNorm launch.
constexpr int SK_MMAX = 16;
constexpr int SKM_WARPS = 8;
constexpr int SKM_TN = 16;
constexpr int SKM_UNR = 4;
constexpr int SKM_LN_KMAX = 1024;  // LayerNorm rows live in registers: 4 x 8 values a lane

__device__ __forceinline__ float sk_wsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ uint4 sk_pack8(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// shared-memory row stride of the normalised rows, in 16-byte units: K + 32
// elements, so that rows r and r + 1 start 64 bytes apart modulo 128
__host__ __device__ __forceinline__ int sk_ln_stride(int K) { return (K + 32) / 8; }

__device__ __forceinline__ void mma_16816(float* d, const uint32_t a0, const uint32_t a1, const uint32_t a2,
                                          const uint32_t a3, const uint32_t b0, const uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int MT>  // row tiles of 8
__global__ void __launch_bounds__(SKM_WARPS * 32)
k_gemm_skinny_mma(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ W,
                  const __nv_bfloat16* __restrict__ bias, const __nv_bfloat16* __restrict__ res,
                  __nv_bfloat16* __restrict__ D, __nv_bfloat16* __restrict__ pre, int M, int N, int K, int ldd,
                  int n_store, int gelu, unsigned long long* __restrict__ pick, int* __restrict__ advance,
                  const __nv_bfloat16* __restrict__ ln_w, const __nv_bfloat16* __restrict__ ln_b) {
    __shared__ float s_part[SKM_WARPS][MT * 128];  // [warp][t*128 + row*16 + col]
    extern __shared__ uint4 s_xn[];                // normalised rows [MT*8][sk_ln_stride(K)] (with ln_w)
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int n0 = blockIdx.x * SKM_TN;
    const int nch = K / 32;
    const bool ra = n0 + g < N, rb = n0 + g + 8 < N;
    const uint4* wa = reinterpret_cast<const uint4*>(W + (long long)(ra ? n0 + g : 0) * K + q * 8);
    const uint4* wb = reinterpret_cast<const uint4*>(W + (long long)(rb ? n0 + g + 8 : 0) * K + q * 8);
    const uint4* xa[MT];
    bool xv[MT];
#pragma unroll
    for (int t = 0; t < MT; t++) {
        xv[t] = t * 8 + g < M;
        xa[t] = reinterpret_cast<const uint4*>(A + (long long)(xv[t] ? t * 8 + g : 0) * K + q * 8);
    }
    float acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; t++) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    uint4 va[SKM_UNR], vb[SKM_UNR];
    auto load_w = [&](int c0) {
#pragma unroll
        for (int u = 0; u < SKM_UNR; u++) {
            const int c = c0 + u * SKM_WARPS;  // chunk: 32 k = 4 uint4 per row
            const bool in = c < nch;
            va[u] = (in && ra) ? __ldcs(wa + c * 4) : zero;
            vb[u] = (in && rb) ? __ldcs(wb + c * 4) : zero;
        }
    };
    load_w(warp);
    pdl_wait();  // A, the residual and the outputs belong to the kernels before
    const int xs = sk_ln_stride(K);
    if (ln_w) {
        // warp w normalises rows w, w + 8 (rows >= M are zero)
        const int nvec = K >> 3;
        for (int r = warp; r < MT * 8; r += SKM_WARPS) {
            uint4* dst = s_xn + r * xs;
            if (r >= M) {
                for (int vi = lane; vi < nvec; vi += 32) dst[vi] = zero;
                continue;
            }
            const uint4* xr = reinterpret_cast<const uint4*>(A + (long long)r * K);
            float v[4][8];
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int vi = lane + 32 * i;
                if (vi < nvec) {
                    const uint4 u4 = xr[vi];
                    const uint32_t wv[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        v[i][2 * e] = __uint_as_float(wv[e] << 16);
                        v[i][2 * e + 1] = __uint_as_float(wv[e] & 0xFFFF0000u);
                    }
#pragma unroll
                    for (int e = 0; e < 8; e++) s += v[i][e];
                }
            }
            const float mu = sk_wsum(s) / K;
            float q2 = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; i++)
                if (lane + 32 * i < nvec)
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const float d = v[i][e] - mu;
                        q2 += d * d;
                    }
            const float rs = rsqrtf(sk_wsum(q2) / K + 1e-5f);
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int vi = lane + 32 * i;
                if (vi < nvec) {
                    const uint4 w4 = reinterpret_cast<const uint4*>(ln_w)[vi];
                    const uint4 b4 = reinterpret_cast<const uint4*>(ln_b)[vi];
                    const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w}, bw[4] = {b4.x, b4.y, b4.z, b4.w};
                    float o[8];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        o[2 * e] = (v[i][2 * e] - mu) * rs * __uint_as_float(ww[e] << 16) +
                                   __uint_as_float(bw[e] << 16);
                        o[2 * e + 1] = (v[i][2 * e + 1] - mu) * rs * __uint_as_float(ww[e] & 0xFFFF0000u) +
                                       __uint_as_float(bw[e] & 0xFFFF0000u);
                    }
                    dst[vi] = sk_pack8(o);
                }
            }
        }
        __syncthreads();
    }
    for (int c0 = warp; c0 < nch; c0 += SKM_WARPS * SKM_UNR) {
        uint4 vx[SKM_UNR][MT];
#pragma unroll
        for (int u = 0; u < SKM_UNR; u++) {
            const int c = c0 + u * SKM_WARPS;
            const bool in = c < nch;
#pragma unroll
            for (int t = 0; t < MT; t++) {
                if (ln_w) vx[u][t] = in ? s_xn[(t * 8 + g) * xs + c * 4 + q] : zero;
                else vx[u][t] = (in && xv[t]) ? __ldg(xa[t] + c * 4) : zero;
            }
        }
#pragma unroll
        for (int u = 0; u < SKM_UNR; u++) {
#pragma unroll
            for (int t = 0; t < MT; t++) {
                mma_16816(acc[t], va[u].x, vb[u].x, va[u].y, vb[u].y, vx[u][t].x, vx[u][t].y);
                mma_16816(acc[t], va[u].z, vb[u].z, va[u].w, vb[u].w, vx[u][t].z, vx[u][t].w);
            }
        }
        if (c0 + SKM_WARPS * SKM_UNR < nch) load_w(c0 + SKM_WARPS * SKM_UNR);
    }
    // accumulator (i, j) of the 16 x 8 tile: column n0 + i, row t*8 + j, with
    // i = g (+8 for entries 2, 3) and j = 2q (+1 for entries 1, 3)
#pragma unroll
    for (int t = 0; t < MT; t++) {
        float* sp = s_part[warp] + t * 128;
        sp[(2 * q) * 16 + g] = acc[t][0];
        sp[(2 * q + 1) * 16 + g] = acc[t][1];
        sp[(2 * q) * 16 + g + 8] = acc[t][2];
        sp[(2 * q + 1) * 16 + g + 8] = acc[t][3];
    }
    __syncthreads();
    if (advance && blockIdx.x == 0 && threadIdx.x == 0) *advance += 1;
    for (int idx = threadIdx.x; idx < MT * 128; idx += SKM_WARPS * 32) {  // 16 consecutive threads: one row
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < SKM_WARPS; w++) v += s_part[w][idx];
        const int m = (idx >> 7) * 8 + ((idx >> 4) & 7), n = n0 + (idx & 15);
        if (bias && n < N) v += __bfloat162float(bias[n]);
        if (pick) {  // the whole warp takes this branch: MT*128 is a multiple of 32
            unsigned long long key = (m < M && n < n_store) ? pick_key(__bfloat162float(__float2bfloat16_rn(v)), n) : 0ull;
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
            if ((idx & 15) == 0 && m < M) pick[(long long)m * gridDim.x + blockIdx.x] = key;
            continue;
        }
        if (m >= M || n >= n_store) continue;
        const long long o = (long long)m * ldd + n;
        if (gelu) {
            pre[o] = __float2bfloat16_rn(v);
            v = gelu_tanh_f(v);
        } else if (res) {
            v += __bfloat162float(res[o]);
        }
        D[o] = __float2bfloat16_rn(v);
    }
}

// fp32: one warp per output column n streams W's row with 16-byte loads and
// dots it with all M rows of A (read through L1); each of the M sums is
// reduced across the warp in a fixed order.
constexpr int SK_WARPS = 8;

template <typename T>
__global__ void __launch_bounds__(SK_WARPS * 32)
k_gemm_skinny(const T* __restrict__ A, const T* __restrict__ W, const T* __restrict__ bias,
              const T* __restrict__ res, T* __restrict__ D, T* __restrict__ pre, int M, int N, int K, int ldd,
              int n_store, int gelu, int* __restrict__ advance) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    if (advance && blockIdx.x == 0 && threadIdx.x == 0) *advance += 1;
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
                    v = gelu_tanh_f(v);
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

void launch_set_int(const Launch& L, int* p, int v) {
    if (L.dry) return;
    L.count();
    k_set_int<<<1, 1, 0, L.stream>>>(p, v);
}

void launch_add_int(const Launch& L, int* p, int v) {
    if (L.dry) return;
    L.count();
    k_add_int<<<1, 1, 0, L.stream>>>(p, v);
}

void launch_embed_at(const Launch& L, bool bf16, const void* wte, const void* wpe, const int32_t* tok,
                     int ld_tok, const int* pos_dev, void* x, int B, int C, int V) {
    if (L.dry) return;
    L.count();
    if (bf16)
        launch_k(L, k_embed_at<__nv_bfloat16>, B, 256, 0, (const __nv_bfloat16*)wte, (const __nv_bfloat16*)wpe, tok,
                 ld_tok, pos_dev, (__nv_bfloat16*)x, B, C, V, L.flags);
    else
        launch_k(L, k_embed_at<float>, B, 256, 0, (const float*)wte, (const float*)wpe, tok, ld_tok, pos_dev,
                 (float*)x, B, C, V, L.flags);
}

int decode_attn_splits(int max_keys) { return (max_keys + DA_KEYS - 1) / DA_KEYS; }

size_t decode_attn_scratch_floats(int B, int H, int max_keys) {
    return (size_t)B * H * decode_attn_splits(max_keys) * DA_PART;
}

bool launch_decode_attn(const Launch& L, bool bf16, const void* qkv, void* cache, void* y, int B, int H, int C,
                        const int* pos_dev, int max_keys, int maxT, float* part, int* counters) {
    const size_t es = bf16 ? 2 : 4;
    if (C % H || C / H > DA_DMAX || (C / H) % 8 || ((size_t)(C / H) * es) % 16 || max_keys < 1 || max_keys > maxT)
        return false;
    if (L.dry) return true;
    L.count();
    const int S = decode_attn_splits(max_keys);
    const float scale = 1.0f / sqrtf((float)(C / H));
    const unsigned grid = (unsigned)(B * H * S);
    if (bf16)
        launch_k(L, k_decode_attn<__nv_bfloat16>, grid, DA_THREADS, 0, (const __nv_bfloat16*)qkv,
                 (__nv_bfloat16*)cache, (__nv_bfloat16*)y, H, C, pos_dev, maxT, S, scale, part, counters);
    else
        launch_k(L, k_decode_attn<float>, grid, DA_THREADS, 0, (const float*)qkv, (float*)cache, (float*)y, H, C,
                 pos_dev, maxT, S, scale, part, counters);
    return true;
}

static bool ln_ok(const void* ln_w, const void* ln_b, int K) {
    if (!ln_w) return true;
    return ln_b && K <= SKM_LN_KMAX && !((uintptr_t)ln_w & 15) && !((uintptr_t)ln_b & 15);
}

static size_t ln_smem(const void* ln_w, int M, int K) {
    return ln_w ? (size_t)(M <= 8 ? 8 : 16) * sk_ln_stride(K) * 16 : 0;
}

bool launch_gemm_skinny(const Launch& L, bool bf16, const void* A, const void* W, const void* bias, const void* res,
                        void* D, void* pre, int M, int N, int K, int ldd, int n_store, bool gelu, int* advance,
                        const void* ln_w, const void* ln_b) {
    const size_t es = bf16 ? 2 : 4;
    if (M < 1 || M > SK_MMAX || K % 32 || ((uintptr_t)A & 15) || ((uintptr_t)W & 15) || ((K * es) & 15)) return false;
    if (ln_w && (!bf16 || !ln_ok(ln_w, ln_b, K))) return false;
    if (L.dry) return true;
    L.count();
    if (bf16) {
        const long long grid = (N + SKM_TN - 1) / SKM_TN;
        if (grid > 0x7fffffff) return false;
        const size_t smem = ln_smem(ln_w, M, K);
#define SKM(MT_)                                                                                               \
    launch_k(L, k_gemm_skinny_mma<MT_>, (unsigned)grid, SKM_WARPS * 32, smem, (const __nv_bfloat16*)A,          \
             (const __nv_bfloat16*)W, (const __nv_bfloat16*)bias, (const __nv_bfloat16*)res, (__nv_bfloat16*)D, \
             (__nv_bfloat16*)pre, M, N, K, ldd, n_store, gelu ? 1 : 0, (unsigned long long*)nullptr, advance,  \
             (const __nv_bfloat16*)ln_w, (const __nv_bfloat16*)ln_b)
        if (M <= 8) SKM(1); else SKM(2);
#undef SKM
        return true;
    }
    const unsigned grid = (unsigned)std::min<long long>((N + SK_WARPS - 1) / SK_WARPS, 65535);
    launch_k(L, k_gemm_skinny<float>, grid, SK_WARPS * 32, 0, (const float*)A, (const float*)W, (const float*)bias,
             (const float*)res, (float*)D, (float*)pre, M, N, K, ldd, n_store, gelu ? 1 : 0, advance);
    return true;
}

int skinny_pick_ctas(int N) { return (N + SKM_TN - 1) / SKM_TN; }

bool launch_gemm_skinny_pick(const Launch& L, const void* A, const void* W, int M, int N, int K,
                             unsigned long long* keys, int* advance, const void* ln_w, const void* ln_b) {
    if (M < 1 || M > SK_MMAX || K % 32 || ((uintptr_t)A & 15) || ((uintptr_t)W & 15)) return false;
    if (!ln_ok(ln_w, ln_b, K)) return false;
    if (L.dry) return true;
    L.count();
    const unsigned grid = (unsigned)skinny_pick_ctas(N);
    const size_t smem = ln_smem(ln_w, M, K);
#define SKP(MT_)                                                                                                \
    launch_k(L, k_gemm_skinny_mma<MT_>, grid, SKM_WARPS * 32, smem, (const __nv_bfloat16*)A,                     \
             (const __nv_bfloat16*)W, (const __nv_bfloat16*)nullptr, (const __nv_bfloat16*)nullptr,              \
             (__nv_bfloat16*)nullptr, (__nv_bfloat16*)nullptr, M, N, K, 0, N, 0, keys, advance,                  \
             (const __nv_bfloat16*)ln_w, (const __nv_bfloat16*)ln_b)
    if (M <= 8) SKP(1); else SKP(2);
#undef SKP
    return true;
}

void launch_pick(const Launch& L, const unsigned long long* keys, int nct, int rows, int32_t* tok, int ld_tok,
                 const int* pos_dev) {
    if (L.dry) return;
    L.count();
    launch_k(L, k_pick, rows, 256, 0, keys, nct, tok, ld_tok, pos_dev);
}

void launch_argmax(const Launch& L, bool bf16, const void* z, long long row_stride, int rows, int V, int32_t* out,
                   int ld_out, int col, const int* col_dev) {
    if (L.dry) return;
    L.count();
    if (bf16)
        launch_k(L, k_argmax<__nv_bfloat16>, rows, AM_THREADS, 0, (const __nv_bfloat16*)z, row_stride, V, out, ld_out,
                 col, col_dev);
    else
        launch_k(L, k_argmax<float>, rows, AM_THREADS, 0, (const float*)z, row_stride, V, out, ld_out, col, col_dev);
}

}  // namespace tt

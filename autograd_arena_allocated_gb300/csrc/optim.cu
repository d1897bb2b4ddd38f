// optim.cu -- the update-side variants of the training step, decided on the
// device: global gradient statistics (for clipping and overflow detection),
// AdamW on the clipped, unscaled gradient with the step skipped on overflow,
// and the dynamic loss scale (the dl-scratch page, 3.2 and 3.4).
#include "tt_internal.h"

#include <algorithm>

namespace tt {
namespace {

constexpr int GS_THREADS = 256;

// part[b] = sum of (g_i / s)^2 over the elements block b takes: float4 i of
// the n/4 goes to the thread i mod (gridDim * blockDim) in grid-stride order,
// four strides per round with four loads in flight (one partial sum each,
// added in order at the end), the tail to block 0.  Per-thread float sums,
// combined within the block in a fixed order.
__global__ void __launch_bounds__(GS_THREADS)
k_grad_sq_part(const float* __restrict__ g, size_t n, const float* __restrict__ scale_dev, double* __restrict__ part) {
    __shared__ float s_w[GS_THREADS / 32];
    const float inv = scale_dev ? 1.0f / *scale_dev : 1.0f;
    const size_t n4 = n / 4, stride = (size_t)gridDim.x * blockDim.x;
    const float4* g4 = reinterpret_cast<const float4*>(g);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    auto add = [&](float& s, const float4 v) {
        const float a = v.x * inv, b = v.y * inv, c = v.z * inv, d = v.w * inv;
        s = fmaf(a, a, s);
        s = fmaf(b, b, s);
        s = fmaf(c, c, s);
        s = fmaf(d, d, s);
    };
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n4; i += 4 * stride) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; u++) v[u] = __ldcs(g4 + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; u++) add(acc[u], v[u]);
    }
    for (int u = 0; i < n4; i += stride, u++) add(acc[u & 3], __ldcs(g4 + i));
    float s = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    if (blockIdx.x == 0)
        for (size_t i = n4 * 4 + threadIdx.x; i < n; i += blockDim.x) {
            const float a = g[i] * inv;
            s = fmaf(a, a, s);
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < GS_THREADS / 32; w++) t += (double)s_w[w];
        part[blockIdx.x] = t;
    }
}

// stats[0] = sqrt(sum of the partials, in block order), stats[1] = not finite
__global__ void k_grad_sq_final(const double* __restrict__ part, int nblk, float* __restrict__ stats) {
    if (threadIdx.x != 0) return;
    double t = 0.0;
    for (int b = 0; b < nblk; b++) t += part[b];
    const bool ok = isfinite(t);
    stats[0] = ok ? (float)sqrt(t) : INFINITY;
    stats[1] = ok ? 0.0f : 1.0f;
}

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
__device__ __forceinline__ void st_low(__nv_bfloat16* p, size_t i, float v) { p[i] = __float2bfloat16_rn(v); }
__device__ __forceinline__ void st_low(__half* p, size_t i, float v) { p[i] = __float2half_rn(v); }

// AdamW on g * k; the whole update is skipped when stats[1] != 0.  LT: the
// 16-bit type of the parameter copy (bf16 or half)
template <typename LT>
__global__ void __launch_bounds__(256)
k_adamw_ex(float* __restrict__ p, LT* __restrict__ lowp, const float* __restrict__ g,
           float* __restrict__ m, float* __restrict__ v, size_t n, float lr, float b1, float b2, float eps, float wd,
           const int* __restrict__ step, const float* __restrict__ stats, float max_norm,
           const float* __restrict__ scale_dev) {
    if (stats && stats[1] != 0.0f) return;
    float k = scale_dev ? 1.0f / *scale_dev : 1.0f;
    if (max_norm > 0.0f) k *= fminf(1.0f, max_norm / (stats[0] + 1e-6f));
    const int t = *step + 1;
    const float c1 = (float)(1.0 - pow((double)b1, t));
    const float c2 = (float)(1.0 - pow((double)b2, t));
    const size_t n4 = n / 4, stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 pp = reinterpret_cast<const float4*>(p)[i];
        const float4 gg = reinterpret_cast<const float4*>(g)[i];
        float4 mm = reinterpret_cast<const float4*>(m)[i];
        float4 vv = reinterpret_cast<const float4*>(v)[i];
        float* pe = &pp.x;
        const float* ge = &gg.x;
        float* me = &mm.x;
        float* ve = &vv.x;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float gj = ge[j] * k;
            me[j] = b1 * me[j] + (1.0f - b1) * gj;
            ve[j] = b2 * ve[j] + (1.0f - b2) * gj * gj;
            pe[j] -= lr * ((me[j] / c1) / (sqrtf(ve[j] / c2) + eps) + wd * pe[j]);
        }
        reinterpret_cast<float4*>(p)[i] = pp;
        reinterpret_cast<float4*>(m)[i] = mm;
        reinterpret_cast<float4*>(v)[i] = vv;
        if (lowp) st_low4(lowp, i, pp);
    }
    for (size_t i = n4 * 4 + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float gi = g[i] * k;
        const float mi = b1 * m[i] + (1.0f - b1) * gi;
        const float vi = b2 * v[i] + (1.0f - b2) * gi * gi;
        m[i] = mi;
        v[i] = vi;
        const float pi = p[i] - lr * ((mi / c1) / (sqrtf(vi / c2) + eps) + wd * p[i]);
        p[i] = pi;
        if (lowp) st_low(lowp, i, pi);
    }
}

// after the update: the step count advances unless the update was skipped
__global__ void k_step_advance(int* step, const float* stats) {
    if (!(stats && stats[1] != 0.0f)) *step += 1;
}

__global__ void k_loss_scale_update(float* scale, int* clean, const float* stats, int window, float growth,
                                    float backoff) {
    if (stats[1] != 0.0f) {
        *scale *= backoff;
        *clean = 0;
    } else if (++*clean >= window) {
        *scale *= growth;
        *clean = 0;
    }
}

int gs_blocks(const Launch& L) { return L.num_sms * 4; }

}  // namespace

size_t grad_stats_scratch_doubles(const Launch& L) { return (size_t)gs_blocks(L); }

void launch_grad_stats(const Launch& L, const float* g, size_t n, const float* scale_dev, float* stats,
                       double* scratch) {
    if (L.dry) return;
    const int G = gs_blocks(L);
    L.count();
    k_grad_sq_part<<<G, GS_THREADS, 0, L.stream>>>(g, n, scale_dev, scratch);
    L.count();
    k_grad_sq_final<<<1, 32, 0, L.stream>>>(scratch, G, stats);
}

void launch_adamw_ex(const Launch& L, float* master, void* lowp, const float* g, float* m, float* v,
                     size_t n, float lr, float b1, float b2, float eps, float wd, int* step, const float* stats,
                     float max_norm, const float* scale_dev) {
    if (L.dry) return;
    if (n > 0) {
        const long long want = (long long)((n / 4 + 255) / 256);
        const int grid = (int)std::max<long long>(1, std::min<long long>(want, (long long)L.num_sms * 8));
        L.count();
        if (L.f16)
            k_adamw_ex<<<grid, 256, 0, L.stream>>>(master, (__half*)lowp, g, m, v, n, lr, b1, b2, eps, wd, step,
                                                   stats, max_norm, scale_dev);
        else
            k_adamw_ex<<<grid, 256, 0, L.stream>>>(master, (__nv_bfloat16*)lowp, g, m, v, n, lr, b1, b2, eps, wd,
                                                   step, stats, max_norm, scale_dev);
    }
    L.count();
    k_step_advance<<<1, 1, 0, L.stream>>>(step, stats);
}

void launch_loss_scale_update(const Launch& L, float* scale, int* clean, const float* stats, int window,
                              float growth, float backoff) {
    if (L.dry) return;
    L.count();
    k_loss_scale_update<<<1, 1, 0, L.stream>>>(scale, clean, stats, window, growth, backoff);
}

}  // namespace tt

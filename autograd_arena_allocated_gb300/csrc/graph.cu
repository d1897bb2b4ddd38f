// graph.cu -- kernels of the generic tensor graph (tt_graph.h): the ops of
// the tinytorch page's library API (三.3 MatMul, 三.4 GELU, 三.5 Softmax and
// CrossEntropy, the bias add and the SGD update of its 八.5 example) in fp32,
// forward and backward.  Tensors here are small (a classifier's batch), so
// these are plain SIMT kernels; every sum is taken in a fixed order.
#include "tt_internal.h"

#include <algorithm>

namespace tt {
namespace {

constexpr int G_TILE = 32;

// C[i, j] (+)= sum_k X(i, k) Y(k, j) with X(i, k) = X[i*xi + k*xk] and
// Y(k, j) = Y[k*yk + j*yj]: one kernel for C = A B and for the two products
// of its backward (dA = dC B^T, dB = A^T dC).  32 x 32 output tile per CTA,
// k in chunks of 32 through shared memory, in increasing order.
__global__ void __launch_bounds__(256)
k_g_matmul(const float* __restrict__ X, long long xi, long long xk, const float* __restrict__ Y, long long yk,
           long long yj, float* __restrict__ C, int M, int N, int K, int accumulate) {
    __shared__ float sx[G_TILE][G_TILE + 1];
    __shared__ float sy[G_TILE][G_TILE + 1];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const int i0 = blockIdx.y * G_TILE, j0 = blockIdx.x * G_TILE;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int k0 = 0; k0 < K; k0 += G_TILE) {
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const int row = ty + 8 * r;  // tile row
            const int i = i0 + row, kx = k0 + tx;
            sx[row][tx] = (i < M && kx < K) ? X[i * xi + kx * xk] : 0.0f;
            const int ky = k0 + row, j = j0 + tx;
            sy[row][tx] = (ky < K && j < N) ? Y[ky * yk + j * yj] : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < G_TILE; k++) {
            const float y = sy[k][tx];
#pragma unroll
            for (int r = 0; r < 4; r++) acc[r] = fmaf(sx[ty + 8 * r][k], y, acc[r]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < 4; r++) {
        const int i = i0 + ty + 8 * r, j = j0 + tx;
        if (i < M && j < N) {
            float* c = C + (long long)i * N + j;
            *c = accumulate ? *c + acc[r] : acc[r];
        }
    }
}

// c = a + b, b either of a's shape (bcols == 0) or a row of bcols added to every row
__global__ void k_g_add(const float* __restrict__ a, const float* __restrict__ b, float* __restrict__ c, long long n,
                        int bcols) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        c[i] = a[i] + b[bcols ? i % bcols : i];
}

__global__ void k_g_mul(const float* __restrict__ a, const float* __restrict__ b, float* __restrict__ c, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        c[i] = a[i] * b[i];
}

__device__ __forceinline__ float g_gelu(float u) {
    const float k = 0.7978845608028654f, a = 0.044715f;
    return 0.5f * u * (1.0f + tanhf(k * (u + a * u * u * u)));
}
__device__ __forceinline__ float g_dgelu(float u) {
    const float k = 0.7978845608028654f, a = 0.044715f;
    const float t = tanhf(k * (u + a * u * u * u));
    return 0.5f * (1.0f + t) + 0.5f * u * (1.0f - t * t) * k * (1.0f + 3.0f * a * u * u);
}

__global__ void k_g_gelu(const float* __restrict__ a, float* __restrict__ c, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        c[i] = g_gelu(a[i]);
}

// one warp per row; the row maximum first, then the sum of exponentials
__global__ void k_g_softmax(const float* __restrict__ z, float* __restrict__ p, int rows, int cols) {
    const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (r >= rows) return;
    const float* zr = z + (long long)r * cols;
    float* pr = p + (long long)r * cols;
    float mx = -INFINITY;
    for (int c = lane; c < cols; c += 32) mx = fmaxf(mx, zr[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float s = 0.0f;
    for (int c = lane; c < cols; c += 32) {
        const float e = expf(zr[c] - mx);
        pr[c] = e;
        s += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv = 1.0f / s;
    for (int c = lane; c < cols; c += 32) pr[c] *= inv;
}

// loss[0] = -(1/R) sum_r ln p[r, y_r]; one CTA of 256 threads
__global__ void __launch_bounds__(256)
k_g_xent(const float* __restrict__ p, const int32_t* __restrict__ y, int rows, int cols, float* __restrict__ loss,
         int* flags) {
    __shared__ float s_w[8];
    float s = 0.0f;
    for (int r = threadIdx.x; r < rows; r += 256) {
        const int t = y[r];
        if (t < 0 || t >= cols) {
            atomicOr(&flags[FLAG_BAD_TOKEN], 1);
            continue;
        }
        s -= logf(p[(long long)r * cols + t]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int w = 0; w < 8; w++) t += s_w[w];
        loss[0] = t / (float)rows;
    }
}

// ---------------------------------------------------------------- backward
__global__ void k_g_fill(float* __restrict__ d, long long n, float v) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        d[i] = v;
}

// d += s (the gradient of an add reaching an input of the same shape)
__global__ void k_g_acc(float* __restrict__ d, const float* __restrict__ s, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        d[i] += s[i];
}

// db[c] += sum_r dC[r, c], rows in increasing order
__global__ void k_g_colsum_acc(const float* __restrict__ dC, int rows, int cols, float* __restrict__ db) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= cols) return;
    float s = 0.0f;
    for (int r = 0; r < rows; r++) s += dC[(long long)r * cols + c];
    db[c] += s;
}

// ga += dc * b and gb += dc * a (either may be null; they may be one buffer)
__global__ void k_g_mul_bwd(const float* __restrict__ dc, const float* a, const float* b, float* ga, float* gb,
                            long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const float g = dc[i], av = a[i], bv = b[i];
        if (ga) ga[i] += g * bv;
        if (gb) gb[i] += g * av;
    }
}

__global__ void k_g_gelu_bwd(const float* __restrict__ dc, const float* __restrict__ a, float* __restrict__ ga,
                             long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        ga[i] += dc[i] * g_dgelu(a[i]);
}

// dz += p o (dp - <p, dp>) per row; one warp per row
__global__ void k_g_softmax_bwd(const float* __restrict__ p, const float* __restrict__ dp, float* __restrict__ dz,
                                int rows, int cols) {
    const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (r >= rows) return;
    const float* pr = p + (long long)r * cols;
    const float* dr = dp + (long long)r * cols;
    float s = 0.0f;
    for (int c = lane; c < cols; c += 32) s = fmaf(pr[c], dr[c], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    for (int c = lane; c < cols; c += 32) dz[(long long)r * cols + c] += pr[c] * (dr[c] - s);
}

// dp[r, y_r] += -dloss / (R p[r, y_r]); dloss read from the loss node's gradient
__global__ void k_g_xent_bwd(const float* __restrict__ p, const int32_t* __restrict__ y,
                             const float* __restrict__ dloss, int rows, int cols, float* __restrict__ dp) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const int t = y[r];
    if (t < 0 || t >= cols) return;
    const long long o = (long long)r * cols + t;
    dp[o] += -dloss[0] / ((float)rows * p[o]);
}

// the softmax + cross entropy pair: dz[r, c] += dloss (p[r, c] - [c == y_r]) / R
__global__ void k_g_softmax_xent_bwd(const float* __restrict__ p, const int32_t* __restrict__ y,
                                     const float* __restrict__ dloss, int rows, int cols, float* __restrict__ dz) {
    const long long n = (long long)rows * cols;
    const float sc = dloss[0] / (float)rows;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(i / cols), c = (int)(i % cols);
        dz[i] += sc * (p[i] - (c == y[r] ? 1.0f : 0.0f));
    }
}

// zero up to G_ZERO_MAX buffers in one launch: blockIdx.y picks the buffer
__global__ void k_g_zero_many(GZeroList l) {
    const int e = blockIdx.y;
    float* d = l.p[e];
    const long long n = l.n[e];
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        d[i] = 0.0f;
}

__global__ void k_g_sgd(float* __restrict__ w, const float* __restrict__ g, long long n, float lr) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        w[i] -= lr * g[i];
}

unsigned g_grid(long long n, int threads, int sms) {
    const long long want = (n + threads - 1) / threads;
    return (unsigned)std::max<long long>(1, std::min<long long>(want, (long long)sms * 8));
}

}  // namespace

void launch_g_matmul(const Launch& L, const float* X, long long xi, long long xk, const float* Y, long long yk,
                     long long yj, float* C, int M, int N, int K, bool accumulate) {
    if (L.dry || M <= 0 || N <= 0) return;
    L.count();
    const dim3 grid((N + G_TILE - 1) / G_TILE, (M + G_TILE - 1) / G_TILE);
    k_g_matmul<<<grid, 256, 0, L.stream>>>(X, xi, xk, Y, yk, yj, C, M, N, K, accumulate ? 1 : 0);
}

#define G_EW(launch_, ...)                                                           \
    if (L.dry || n <= 0) return;                                                     \
    L.count();                                                                       \
    launch_<<<g_grid(n, 256, L.num_sms), 256, 0, L.stream>>>(__VA_ARGS__)

void launch_g_add(const Launch& L, const float* a, const float* b, float* c, long long n, int bcols) {
    G_EW(k_g_add, a, b, c, n, bcols);
}
void launch_g_mul(const Launch& L, const float* a, const float* b, float* c, long long n) { G_EW(k_g_mul, a, b, c, n); }
void launch_g_gelu(const Launch& L, const float* a, float* c, long long n) { G_EW(k_g_gelu, a, c, n); }
void launch_g_fill(const Launch& L, float* d, long long n, float v) { G_EW(k_g_fill, d, n, v); }
void launch_g_acc(const Launch& L, float* d, const float* s, long long n) { G_EW(k_g_acc, d, s, n); }
void launch_g_mul_bwd(const Launch& L, const float* dc, const float* a, const float* b, float* ga, float* gb,
                      long long n) {
    G_EW(k_g_mul_bwd, dc, a, b, ga, gb, n);
}
void launch_g_gelu_bwd(const Launch& L, const float* dc, const float* a, float* ga, long long n) {
    G_EW(k_g_gelu_bwd, dc, a, ga, n);
}
void launch_g_sgd(const Launch& L, float* w, const float* g, long long n, float lr) { G_EW(k_g_sgd, w, g, n, lr); }
void launch_g_softmax_xent_bwd(const Launch& L, const float* p, const int32_t* y, const float* dloss, int rows,
                               int cols, float* dz) {
    const long long n = (long long)rows * cols;
    G_EW(k_g_softmax_xent_bwd, p, y, dloss, rows, cols, dz);
}
#undef G_EW

void launch_g_zero_many(const Launch& L, const GZeroList& l) {
    if (L.dry || l.count <= 0) return;
    L.count();
    long long mx = 1;
    for (int i = 0; i < l.count; i++) mx = std::max(mx, l.n[i]);
    const dim3 grid((unsigned)std::min<long long>((mx + 255) / 256, 64), (unsigned)l.count);
    k_g_zero_many<<<grid, 256, 0, L.stream>>>(l);
}

void launch_g_softmax(const Launch& L, const float* z, float* p, int rows, int cols) {
    if (L.dry || rows <= 0) return;
    L.count();
    k_g_softmax<<<(rows + 7) / 8, 256, 0, L.stream>>>(z, p, rows, cols);
}
void launch_g_softmax_bwd(const Launch& L, const float* p, const float* dp, float* dz, int rows, int cols) {
    if (L.dry || rows <= 0) return;
    L.count();
    k_g_softmax_bwd<<<(rows + 7) / 8, 256, 0, L.stream>>>(p, dp, dz, rows, cols);
}
void launch_g_xent(const Launch& L, const float* p, const int32_t* y, int rows, int cols, float* loss) {
    if (L.dry) return;
    L.count();
    k_g_xent<<<1, 256, 0, L.stream>>>(p, y, rows, cols, loss, L.flags);
}
void launch_g_xent_bwd(const Launch& L, const float* p, const int32_t* y, const float* dloss, int rows, int cols,
                       float* dp) {
    if (L.dry || rows <= 0) return;
    L.count();
    k_g_xent_bwd<<<(rows + 255) / 256, 256, 0, L.stream>>>(p, y, dloss, rows, cols, dp);
}
void launch_g_colsum_acc(const Launch& L, const float* dC, int rows, int cols, float* db) {
    if (L.dry || cols <= 0) return;
    L.count();
    k_g_colsum_acc<<<(cols + 255) / 256, 256, 0, L.stream>>>(dC, rows, cols, db);
}

}  // namespace tt

// attn_mma.cu -- causal self-attention on the tensor cores (bf16 in, fp32
// accumulate), head dim 64, flash-style: scores never leave the SM.
//
// Forward: one CTA (4 warps) per 64 queries of one (batch, head); each warp
// owns 16 query rows.  Key/value tiles of 64 rows stream through shared
// memory (cp.async, double buffered); S = Q K^T and O += P V use
// mma.sync.m16n8k16; the softmax is online (running max and sum in fp32,
// base-2 exponentials); the log-sum-exp of every row is saved.
//
// Backward, deterministic (no atomics), recomputing P from the saved
// log-sum-exp: D = rowsum(dO * O) first, then
//   dK/dV kernel: one CTA per 64 keys, looping over the query blocks at or
//                 after it: dV += P^T dO, dK += dS^T Q;
//   dQ kernel:    one CTA per 64 queries, looping over the key blocks at or
//                 before it: dQ += dS K;
// with dS = P o (dP - D), dP = dO V^T, all sums in a fixed order.
//
// Shared tiles are 64 x 64 bf16 (128-byte rows) with the 16-byte chunks of
// row r XOR-swizzled by (r mod 8), so ldmatrix reads are conflict free.
#include "tt_internal.h"

#include <math.h>

namespace tt {
namespace fa {

constexpr int D = 64;        // head dim
constexpr int BQ = 64;       // queries per CTA
constexpr int BKV = 64;      // keys per tile
constexpr int THREADS = 128; // 4 warps x 16 rows
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// byte offset of element (row, col) in a swizzled 64x64 bf16 tile (col % 8 == 0)
__device__ __forceinline__ uint32_t tile_off(int row, int col) {
    return (uint32_t)((row * 8 + ((col >> 3) ^ (row & 7))) * 16);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 64 rows x 64 bf16 from global rows [row0, row0+64) (rows >= nvalid read as zero)
__device__ __forceinline__ void load_tile(uint32_t s, const bf16* g, long long ld, int row0,
                                          int nvalid) {
    for (int i = threadIdx.x; i < 64 * 8; i += THREADS) {
        const int r = i >> 3, c = i & 7;
        const bool ok = row0 + r < nvalid;
        const bf16* src = ok ? g + (long long)(row0 + r) * ld + c * 8 : g;
        cp_async16(s + tile_off(r, c * 8), src, ok);
    }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// c += a(16x16, row) * b(16x8, col)
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// A fragments (16 rows x 64 cols) of a swizzled tile, rows row0..row0+15
__device__ __forceinline__ void load_a_frags(uint32_t s, int row0, uint32_t (&f)[4][4]) {
    const int lane = threadIdx.x & 31;
    const int r = row0 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int ks = 0; ks < 4; ks++) {
        const int c = ks * 16 + 8 * (lane >> 4);
        ldsm_x4(s + tile_off(r, c), f[ks][0], f[ks][1], f[ks][2], f[ks][3]);
    }
}

// acc[16 x 64] += A[16 x 64 (k)] * B^T where B is a swizzled tile holding the
// n dimension in rows and k in columns (e.g. K for S = Q K^T)
__device__ __forceinline__ void mma_abT(float (&acc)[8][4], const uint32_t (&a)[4][4], uint32_t s) {
    const int lane = threadIdx.x & 31;
    const int i = lane >> 3, j = lane & 7;
#pragma unroll
    for (int ks = 0; ks < 4; ks++) {
#pragma unroll
        for (int np = 0; np < 4; np++) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(s + tile_off(np * 16 + j + 8 * (i >> 1), ks * 16 + 8 * (i & 1)), b0, b1, b2, b3);
            mma16816(acc[2 * np], a[ks], b0, b1);
            mma16816(acc[2 * np + 1], a[ks], b2, b3);
        }
    }
}

// acc[16 x 64] += P[16 x 64 (k)] * B where B is a swizzled tile holding k in
// rows and n in columns (e.g. V for O = P V); P given as A fragments
__device__ __forceinline__ void mma_ab(float (&acc)[8][4], const uint32_t (&p)[4][4], uint32_t s) {
    const int lane = threadIdx.x & 31;
    const int i = lane >> 3, j = lane & 7;
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
#pragma unroll
        for (int dp = 0; dp < 4; dp++) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(s + tile_off(kk * 16 + j + 8 * (i & 1), dp * 16 + 8 * (i >> 1)), b0, b1, b2, b3);
            mma16816(acc[2 * dp], p[kk], b0, b1);
            mma16816(acc[2 * dp + 1], p[kk], b2, b3);
        }
    }
}

// accumulator layout (16 x 64, 8 n-tiles) -> bf16 A fragments
__device__ __forceinline__ void acc_to_a(const float (&s)[8][4], uint32_t (&p)[4][4]) {
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
        p[kk][0] = pack2(s[2 * kk][0], s[2 * kk][1]);
        p[kk][1] = pack2(s[2 * kk][2], s[2 * kk][3]);
        p[kk][2] = pack2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        p[kk][3] = pack2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
    }
}

__device__ __forceinline__ void zero(float (&a)[8][4]) {
#pragma unroll
    for (int n = 0; n < 8; n++)
#pragma unroll
        for (int k = 0; k < 4; k++) a[n][k] = 0.0f;
}

// ------------------------------------------------------------------ forward
__global__ void __launch_bounds__(THREADS)
k_fwd(const bf16* __restrict__ qkv, bf16* __restrict__ y, float* __restrict__ lse, int T, int C,
      int H, float scale) {
    __shared__ __align__(128) uint8_t sQ[BQ * D * 2];
    __shared__ __align__(128) uint8_t sK[2][BKV * D * 2];
    __shared__ __align__(128) uint8_t sV[2][BKV * D * 2];
    const int nqb = gridDim.x;
    const int qb = nqb - 1 - blockIdx.x;  // heaviest blocks first
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    const long long ld3 = 3LL * C;
    const bf16* base = qkv + (long long)b * T * ld3 + (long long)h * D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const float sl2 = scale * LOG2E;

    load_tile(smem_u32(sQ), base, ld3, qb * BQ, T);
    load_tile(smem_u32(sK[0]), base + C, ld3, 0, T);
    load_tile(smem_u32(sV[0]), base + 2 * C, ld3, 0, T);
    cp_commit();

    uint32_t qf[4][4];
    float o[8][4];
    zero(o);
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    const int qrow0 = qb * BQ + warp * 16 + g;  // this thread's rows: qrow0, qrow0 + 8

    for (int kb = 0; kb <= qb; kb++) {
        const int buf = kb & 1;
        if (kb < qb) {
            load_tile(smem_u32(sK[buf ^ 1]), base + C, ld3, (kb + 1) * BKV, T);
            load_tile(smem_u32(sV[buf ^ 1]), base + 2 * C, ld3, (kb + 1) * BKV, T);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        if (kb == 0) load_a_frags(smem_u32(sQ), warp * 16, qf);

        float s[8][4];
        zero(s);
        mma_abT(s, qf, smem_u32(sK[buf]));
        // scale (base 2), causal mask on the diagonal block
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < 8; n++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                float v = s[n][e] * sl2;
                if (kb == qb) {
                    const int key = kb * BKV + n * 8 + 2 * t4 + (e & 1);
                    const int q = qrow0 + ((e >> 1) ? 8 : 0);
                    if (key > q) v = -INFINITY;
                }
                s[n][e] = v;
            }
            mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
            mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float c0 = exp2f(m0 - n0), c1 = exp2f(m1 - n1);
        m0 = n0;
        m1 = n1;
        float r0 = 0.0f, r1 = 0.0f;
#pragma unroll
        for (int n = 0; n < 8; n++) {
            s[n][0] = exp2f(s[n][0] - n0);
            s[n][1] = exp2f(s[n][1] - n0);
            s[n][2] = exp2f(s[n][2] - n1);
            s[n][3] = exp2f(s[n][3] - n1);
            r0 += s[n][0] + s[n][1];
            r1 += s[n][2] + s[n][3];
            o[n][0] *= c0;
            o[n][1] *= c0;
            o[n][2] *= c1;
            o[n][3] *= c1;
        }
        l0 = l0 * c0 + r0;
        l1 = l1 * c1 + r1;
        uint32_t pa[4][4];
        acc_to_a(s, pa);
        mma_ab(o, pa, smem_u32(sV[buf]));
        __syncthreads();  // the buffer is refilled next iteration
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float i0 = 1.0f / l0, i1 = 1.0f / l1;
    const long long ybase = (long long)b * T * C + (long long)h * D;
#pragma unroll
    for (int half = 0; half < 2; half++) {
        const int q = qrow0 + 8 * half;
        if (q >= T) continue;
        const float inv = half ? i1 : i0;
        uint32_t* yr = reinterpret_cast<uint32_t*>(y + ybase + (long long)q * C);
#pragma unroll
        for (int n = 0; n < 8; n++) yr[n * 4 + t4] = pack2(o[n][2 * half] * inv, o[n][2 * half + 1] * inv);
        if (t4 == 0)
            lse[((long long)b * H + h) * T + q] = ((half ? m1 : m0) + log2f(half ? l1 : l0)) * LN2;
    }
}

// ------------------------------------------------------------------ backward
// D[b,h,t] = sum_d dO[t,d] * O[t,d]  (one warp per row, 2 values per lane)
__global__ void k_delta(const bf16* __restrict__ y, const bf16* __restrict__ dy,
                        float* __restrict__ Dlt, int B, int T, int C, int H) {
    const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= (long long)B * H * T) return;
    const int t = (int)(row % T);
    const int h = (int)((row / T) % H);
    const int b = (int)(row / ((long long)T * H));
    const long long o = ((long long)b * T + t) * C + (long long)h * D + 2 * lane;
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(y + o);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(dy + o);
    float s = __low2float(a) * __low2float(d) + __high2float(a) * __high2float(d);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) s += __shfl_xor_sync(0xffffffffu, s, k);
    if (lane == 0) Dlt[row] = s;
}

// one CTA per 64 keys: dK, dV
__global__ void __launch_bounds__(THREADS)
k_bwd_dkdv(const bf16* __restrict__ qkv, const bf16* __restrict__ dy, const float* __restrict__ lse,
           const float* __restrict__ Dlt, bf16* __restrict__ dqkv, int T, int C, int H, float scale) {
    __shared__ __align__(128) uint8_t sK[BKV * D * 2];
    __shared__ __align__(128) uint8_t sV[BKV * D * 2];
    __shared__ __align__(128) uint8_t sQ[2][BQ * D * 2];
    __shared__ __align__(128) uint8_t sO[2][BQ * D * 2];  // dO tiles
    __shared__ float sL[2][BQ], sD[2][BQ];
    const int nkb = gridDim.x;
    const int kb = blockIdx.x;  // lightest first is fine: work ~ (nkb - kb)
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    const long long ld3 = 3LL * C;
    const bf16* base = qkv + (long long)b * T * ld3 + (long long)h * D;
    const bf16* dbase = dy + (long long)b * T * C + (long long)h * D;
    const float* lrow = lse + ((long long)b * H + h) * T;
    const float* drow = Dlt + ((long long)b * H + h) * T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const float sl2 = scale * LOG2E;
    (void)nkb;

    load_tile(smem_u32(sK), base + C, ld3, kb * BKV, T);
    load_tile(smem_u32(sV), base + 2 * C, ld3, kb * BKV, T);
    const int nqb = (T + BQ - 1) / BQ;
    auto load_q = [&](int qb, int buf) {
        load_tile(smem_u32(sQ[buf]), base, ld3, qb * BQ, T);
        load_tile(smem_u32(sO[buf]), dbase, C, qb * BQ, T);
        for (int i = threadIdx.x; i < BQ; i += THREADS) {
            const int q = qb * BQ + i;
            sL[buf][i] = q < T ? lrow[q] * LOG2E : INFINITY;  // padding rows get P = 0
            sD[buf][i] = q < T ? drow[q] : 0.0f;
        }
    };
    load_q(kb, 0);
    cp_commit();

    uint32_t kf[4][4], vf[4][4];
    float dk[8][4], dv[8][4];
    zero(dk);
    zero(dv);
    const int key0 = kb * BKV + warp * 16 + g;  // this thread's keys: key0, key0 + 8

    for (int qb = kb; qb < nqb; qb++) {
        const int buf = (qb - kb) & 1;
        if (qb + 1 < nqb) load_q(qb + 1, buf ^ 1);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        if (qb == kb) {
            load_a_frags(smem_u32(sK), warp * 16, kf);
            load_a_frags(smem_u32(sV), warp * 16, vf);
        }
        // S^T = K Q^T  (16 keys x 64 queries)
        float st[8][4];
        zero(st);
        mma_abT(st, kf, smem_u32(sQ[buf]));
        // P^T = exp2(S^T * scale*log2e - lse*log2e), masked where query < key
#pragma unroll
        for (int n = 0; n < 8; n++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int qi = n * 8 + 2 * t4 + (e & 1);
                const int key = key0 + ((e >> 1) ? 8 : 0);
                const int q = qb * BQ + qi;
                float p = exp2f(st[n][e] * sl2 - sL[buf][qi]);
                if (q < key) p = 0.0f;
                st[n][e] = p;
            }
        }
        uint32_t pa[4][4];
        acc_to_a(st, pa);
        mma_ab(dv, pa, smem_u32(sO[buf]));  // dV += P^T dO
        // dP^T = V dO^T
        float dpt[8][4];
        zero(dpt);
        mma_abT(dpt, vf, smem_u32(sO[buf]));
        // dS^T = P^T o (dP^T - D)
#pragma unroll
        for (int n = 0; n < 8; n++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int qi = n * 8 + 2 * t4 + (e & 1);
                dpt[n][e] = st[n][e] * (dpt[n][e] - sD[buf][qi]);
            }
        }
        uint32_t da[4][4];
        acc_to_a(dpt, da);
        mma_ab(dk, da, smem_u32(sQ[buf]));  // dK += dS^T Q
        __syncthreads();
    }
    bf16* out = dqkv + (long long)b * T * ld3 + (long long)h * D;
#pragma unroll
    for (int half = 0; half < 2; half++) {
        const int key = key0 + 8 * half;
        if (key >= T) continue;
        uint32_t* dkr = reinterpret_cast<uint32_t*>(out + (long long)key * ld3 + C);
        uint32_t* dvr = reinterpret_cast<uint32_t*>(out + (long long)key * ld3 + 2 * C);
#pragma unroll
        for (int n = 0; n < 8; n++) {
            dkr[n * 4 + t4] = pack2(dk[n][2 * half] * scale, dk[n][2 * half + 1] * scale);
            dvr[n * 4 + t4] = pack2(dv[n][2 * half], dv[n][2 * half + 1]);
        }
    }
}

// one CTA per 64 queries: dQ
__global__ void __launch_bounds__(THREADS)
k_bwd_dq(const bf16* __restrict__ qkv, const bf16* __restrict__ dy, const float* __restrict__ lse,
         const float* __restrict__ Dlt, bf16* __restrict__ dqkv, int T, int C, int H, float scale) {
    __shared__ __align__(128) uint8_t sQ[BQ * D * 2];
    __shared__ __align__(128) uint8_t sO[BQ * D * 2];
    __shared__ __align__(128) uint8_t sK[2][BKV * D * 2];
    __shared__ __align__(128) uint8_t sV[2][BKV * D * 2];
    const int nqb = gridDim.x;
    const int qb = nqb - 1 - blockIdx.x;
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    const long long ld3 = 3LL * C;
    const bf16* base = qkv + (long long)b * T * ld3 + (long long)h * D;
    const bf16* dbase = dy + (long long)b * T * C + (long long)h * D;
    const float* lrow = lse + ((long long)b * H + h) * T;
    const float* drow = Dlt + ((long long)b * H + h) * T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const float sl2 = scale * LOG2E;

    load_tile(smem_u32(sQ), base, ld3, qb * BQ, T);
    load_tile(smem_u32(sO), dbase, C, qb * BQ, T);
    load_tile(smem_u32(sK[0]), base + C, ld3, 0, T);
    load_tile(smem_u32(sV[0]), base + 2 * C, ld3, 0, T);
    cp_commit();

    const int qrow0 = qb * BQ + warp * 16 + g;
    float L0 = 0.0f, L1 = 0.0f, D0 = 0.0f, D1 = 0.0f;
    if (qrow0 < T) { L0 = lrow[qrow0] * LOG2E; D0 = drow[qrow0]; }
    if (qrow0 + 8 < T) { L1 = lrow[qrow0 + 8] * LOG2E; D1 = drow[qrow0 + 8]; }

    uint32_t qf[4][4], of[4][4];
    float dq[8][4];
    zero(dq);
    for (int kb = 0; kb <= qb; kb++) {
        const int buf = kb & 1;
        if (kb < qb) {
            load_tile(smem_u32(sK[buf ^ 1]), base + C, ld3, (kb + 1) * BKV, T);
            load_tile(smem_u32(sV[buf ^ 1]), base + 2 * C, ld3, (kb + 1) * BKV, T);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        if (kb == 0) {
            load_a_frags(smem_u32(sQ), warp * 16, qf);
            load_a_frags(smem_u32(sO), warp * 16, of);
        }
        float s[8][4];
        zero(s);
        mma_abT(s, qf, smem_u32(sK[buf]));
        float dp[8][4];
        zero(dp);
        mma_abT(dp, of, smem_u32(sV[buf]));  // dP = dO V^T
#pragma unroll
        for (int n = 0; n < 8; n++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int key = kb * BKV + n * 8 + 2 * t4 + (e & 1);
                const int q = qrow0 + ((e >> 1) ? 8 : 0);
                float p = exp2f(s[n][e] * sl2 - ((e >> 1) ? L1 : L0));
                if (key > q || q >= T) p = 0.0f;
                s[n][e] = p * (dp[n][e] - ((e >> 1) ? D1 : D0));  // dS
            }
        }
        uint32_t da[4][4];
        acc_to_a(s, da);
        mma_ab(dq, da, smem_u32(sK[buf]));  // dQ += dS K
        __syncthreads();
    }
    bf16* out = dqkv + (long long)b * T * ld3 + (long long)h * D;
#pragma unroll
    for (int half = 0; half < 2; half++) {
        const int q = qrow0 + 8 * half;
        if (q >= T) continue;
        uint32_t* r = reinterpret_cast<uint32_t*>(out + (long long)q * ld3);
#pragma unroll
        for (int n = 0; n < 8; n++) r[n * 4 + t4] = pack2(dq[n][2 * half] * scale, dq[n][2 * half + 1] * scale);
    }
}

}  // namespace fa

bool attention_mma_eligible(bool bf16, int C, int H) {
    return bf16 && H > 0 && C % H == 0 && C / H == fa::D && (3 * C) % 8 == 0;
}

void launch_attention_fwd_mma(const Launch& L, const void* qkv, void* y, float* lse, int B, int T,
                              int C, int H) {
    if (L.dry) return;
    dim3 grid((T + fa::BQ - 1) / fa::BQ, B * H);
    L.count();
    fa::k_fwd<<<grid, fa::THREADS, 0, L.stream>>>((const fa::bf16*)qkv, (fa::bf16*)y, lse, T, C, H,
                                                  1.0f / sqrtf((float)fa::D));
}

void launch_attention_bwd_mma(const Launch& L, const void* qkv, const void* y, const float* lse,
                              const void* dy, void* dqkv, int B, int T, int C, int H,
                              float* scratch) {
    if (L.dry) return;
    const long long rows = (long long)B * H * T;
    L.count();
    fa::k_delta<<<(unsigned)((rows + 7) / 8), 256, 0, L.stream>>>((const fa::bf16*)y,
                                                                 (const fa::bf16*)dy, scratch, B, T,
                                                                 C, H);
    dim3 grid((T + fa::BQ - 1) / fa::BQ, B * H);
    const float scale = 1.0f / sqrtf((float)fa::D);
    L.count();
    fa::k_bwd_dkdv<<<grid, fa::THREADS, 0, L.stream>>>((const fa::bf16*)qkv, (const fa::bf16*)dy, lse,
                                                       scratch, (fa::bf16*)dqkv, T, C, H, scale);
    L.count();
    fa::k_bwd_dq<<<grid, fa::THREADS, 0, L.stream>>>((const fa::bf16*)qkv, (const fa::bf16*)dy, lse,
                                                     scratch, (fa::bf16*)dqkv, T, C, H, scale);
}

}  // namespace tt

// attn_tc.cu -- causal self-attention on the 5th-generation tensor cores
// (tcgen05, bf16 in, fp32 accumulate in tensor memory), head dim 64.
//
// Forward, one CTA per (batch, head, 128-query tile), 192 threads:
//   warp 0      TMA: the Q tile once, K and V tiles of 128 keys (K double
//               buffered) from the packed [B*T, 3C] qkv buffer
//   warp 1      TMEM allocation and the MMAs: S = Q K^T (M=128, N=128, K=64)
//               into TMEM, then O_j = P_j V_j (M=128, N=64, K=128)
//   warps 2..5  one thread per query row: reads its row of S from TMEM,
//               applies the causal mask, keeps the running max and sum (base-2
//               exponentials), writes P_j as bf16 into shared memory in the
//               128-byte-swizzled K-major layout the MMA reads, and folds
//               O_j into an fp32 accumulator in registers, rescaled whenever
//               the running max moves.  Finally y = O / l and the row's
//               log-sum-exp are written.
// About 97 KB of shared memory and 256 TMEM columns per CTA: two CTAs share
// an SM, so one CTA's softmax overlaps the other's MMAs.  Every wait is
// bounded (FLAG_TIMEOUT), as in the GEMM.
#include "tt_internal.h"
#include "tc_ptx.cuh"

#include <math.h>

namespace tt {
namespace fa5 {

using namespace tc;
typedef __nv_bfloat16 bf16;

constexpr int D = 64;
constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int THREADS = 192;
constexpr int TILE = 128 * 128;  // 128 rows x 128 bytes
constexpr uint32_t TMEM_COLS = 256;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// forward shared-memory map (offsets from a 1024-aligned base)
constexpr int F_Q = 0;
constexpr int F_K = F_Q + TILE;      // 2 stages
constexpr int F_V = F_K + 2 * TILE;  // 1 stage
constexpr int F_P = F_V + TILE;      // 2 swizzle atoms (keys 0-63, 64-127)
constexpr int F_BAR = F_P + 2 * TILE;
constexpr int F_SMEM = F_BAR + 256 + 1024;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return (uint8_t*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

// Store 32 bf16 values (keys k0..k0+31 of row r) into a K-major, 128-byte
// swizzled operand made of 64-key atoms of [128 rows x 128 B].
__device__ __forceinline__ void store_row32(uint8_t* base, int r, int k0, const uint32_t (&w)[16]) {
    uint8_t* atom = base + (k0 >> 6) * TILE + r * 128;
    const int c0 = (k0 & 63) >> 3;  // first 16-byte chunk
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int phys = (c0 + i) ^ (r & 7);
        *reinterpret_cast<uint4*>(atom + phys * 16) = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
}

// 2^x by the single hardware instruction (relative error ~2^-22; inputs here
// are at most 0, results feed bf16 operands or fp32 sums)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// backward kernels: warps 0 (TMA) and 1 (MMA) plus 8 elementwise warps; warp
// w handles TMEM lanes 32*(w%4).. and column half (w-2)/4 of its rows
constexpr int THREADS_B = 320;

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------ forward
__global__ void __launch_bounds__(THREADS)
k_attn_fwd_tc(const __grid_constant__ CUtensorMap tm, bf16* __restrict__ y, float* __restrict__ lse,
              int T, int C, int H, int* flags) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint64_t* bars = (uint64_t*)(sm + F_BAR);
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;   // [2]
    uint64_t* k_empty = bars + 3;  // [2]
    uint64_t* v_full = bars + 5;
    uint64_t* v_empty = bars + 6;
    uint64_t* s_full = bars + 7;
    uint64_t* s_free = bars + 8;
    uint64_t* p_full = bars + 9;
    uint64_t* o_full = bars + 10;
    uint32_t* tmem_holder = (uint32_t*)(bars + 11);
    volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

    const int nqt = gridDim.x;
    const int qt = nqt - 1 - (int)blockIdx.x;  // longest rows first
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    const int nkv = qt + 1;
    const int row0 = b * T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(&k_full[0], 1);
        mbar_init(&k_full[1], 1);
        mbar_init(&k_empty[0], 1);
        mbar_init(&k_empty[1], 1);
        mbar_init(v_full, 1);
        mbar_init(v_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, 128);
        mbar_init(p_full, 128);
        mbar_init(o_full, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm) : "memory");
    }
    if (warp == 1) tmem_alloc(tmem_holder, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            const int xq = h * D, xk = C + h * D, xv = 2 * C + h * D;
            mbar_expect_tx(q_full, TILE);
            tma_load_2d(smem_u32(sm + F_Q), &tm, q_full, xq, row0 + qt * BQ);
            int issued_k = 0, issued_v = 0;
            bool ok = true;
            for (int j = 0; j < nkv && ok; j++) {
                const int st = j & 1;
                if (!mbar_wait(&k_empty[st], ((j >> 1) & 1) ^ 1, abort_flag, flags)) { ok = false; break; }
                mbar_expect_tx(&k_full[st], TILE);
                tma_load_2d(smem_u32(sm + F_K + st * TILE), &tm, &k_full[st], xk, row0 + j * BKV);
                ++issued_k;
                if (!mbar_wait(v_empty, (j & 1) ^ 1, abort_flag, flags)) { ok = false; break; }
                mbar_expect_tx(v_full, TILE);
                tma_load_2d(smem_u32(sm + F_V), &tm, v_full, xv, row0 + j * BKV);
                ++issued_v;
            }
            if (!ok) {  // let issued copies land before the CTA exits
                const long long t0 = clock64();
                while (!mbar_try_wait(q_full, 0) && clock64() - t0 < WAIT_CYCLES) {}
                for (int j = (issued_k > 2 ? issued_k - 2 : 0); j < issued_k; j++)
                    while (!mbar_try_wait(&k_full[j & 1], (j >> 1) & 1) && clock64() - t0 < 2 * WAIT_CYCLES) {}
                if (issued_v > 0)
                    while (!mbar_try_wait(v_full, (issued_v - 1) & 1) && clock64() - t0 < 3 * WAIT_CYCLES) {}
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(BQ, BKV, false, false);
            constexpr uint32_t ID_O = idesc_bf16(BQ, D, false, true);
            const uint32_t sq = smem_u32(sm + F_Q), sp = smem_u32(sm + F_P), sv = smem_u32(sm + F_V);
            bool ok = mbar_wait(q_full, 0, abort_flag, flags);
            for (int j = 0; j < nkv && ok; j++) {
                const int st = j & 1;
                if (!mbar_wait(&k_full[st], (j >> 1) & 1, abort_flag, flags)) break;
                if (!mbar_wait(s_free, (j & 1) ^ 1, abort_flag, flags)) break;
                tc_fence_after();
                const uint32_t sk = smem_u32(sm + F_K + st * TILE);
#pragma unroll
                for (int k = 0; k < D / 16; k++)
                    umma_bf16(tmem, sdesc(sq + 32 * k, 16, 1024), sdesc(sk + 32 * k, 16, 1024), ID_S,
                              k > 0 ? 1u : 0u);
                umma_commit(s_full);
                umma_commit(&k_empty[st]);
                if (!mbar_wait(p_full, j & 1, abort_flag, flags)) break;
                if (!mbar_wait(v_full, j & 1, abort_flag, flags)) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BKV / 16; k++)
                    umma_bf16(tmem + BKV, sdesc(sp + (k >> 2) * TILE + (k & 3) * 32, 16, 1024),
                              sdesc(sv + k * 2048, TILE, 1024), ID_O, k > 0 ? 1u : 0u);
                umma_commit(o_full);
                umma_commit(v_empty);
            }
        }
    } else {
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int q = qt * BQ + r;
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        const float sl2 = 0.125f * LOG2E;  // 1/sqrt(64) in base-2 units
        float m = -INFINITY, l = 0.0f, corr_prev = 1.0f;
        float o[D];
#pragma unroll
        for (int d = 0; d < D; d++) o[d] = 0.0f;
        bool ok = true;
        for (int j = 0; j < nkv; j++) {
            if (!mbar_wait(s_full, j & 1, abort_flag, flags)) { ok = false; break; }
            tc_fence_after();
            const bool diag = (j == qt);
            const int kq = q - j * BKV;  // keys with column index > kq are masked (diagonal block)
            // pass 1: row max of the raw scores (the scale is positive)
            float mx = -INFINITY;
#pragma unroll 1
            for (int c = 0; c < 4; c++) {
                uint32_t w[32];
                tmem_ld32(tl + c * 32, w);
                if (!diag) {
#pragma unroll
                    for (int e = 0; e < 32; e++) mx = fmaxf(mx, __uint_as_float(w[e]));
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e++)
                        if (c * 32 + e <= kq) mx = fmaxf(mx, __uint_as_float(w[e]));
                }
            }
            const float mn = fmaxf(m, mx * sl2);
            const float corr = ex2(m - mn);
            m = mn;
            // fold O_{j-1} (its MMA has finished reading P once o_full flips)
            if (j > 0) {
                if (!mbar_wait(o_full, (j - 1) & 1, abort_flag, flags)) { ok = false; break; }
                tc_fence_after();
                uint32_t w[32];
                tmem_ld32(tl + BKV, w);
#pragma unroll
                for (int d = 0; d < 32; d++) o[d] = fmaf(o[d], corr_prev, __uint_as_float(w[d]));
                tmem_ld32(tl + BKV + 32, w);
#pragma unroll
                for (int d = 0; d < 32; d++) o[32 + d] = fmaf(o[32 + d], corr_prev, __uint_as_float(w[d]));
            }
            corr_prev = corr;
            // pass 2: P = 2^(s*scale - m) as bf16 into shared memory
            float rs = 0.0f;
#pragma unroll 1
            for (int c = 0; c < 4; c++) {
                uint32_t w[32], pk[16];
                tmem_ld32(tl + c * 32, w);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float p0 = ex2(fmaf(__uint_as_float(w[e]), sl2, -m));
                    float p1 = ex2(fmaf(__uint_as_float(w[e + 1]), sl2, -m));
                    if (diag) {
                        if (c * 32 + e > kq) p0 = 0.0f;
                        if (c * 32 + e + 1 > kq) p1 = 0.0f;
                    }
                    rs += p0 + p1;
                    pk[e >> 1] = pack_bf2(p0, p1);
                }
                store_row32(sm + F_P, r, c * 32, pk);
            }
            l = fmaf(l, corr, rs);
            tc_fence_before();
            mbar_arrive(s_free);
            fence_proxy_async_smem();
            mbar_arrive(p_full);
        }
        if (ok && mbar_wait(o_full, (nkv - 1) & 1, abort_flag, flags)) {
            tc_fence_after();
            uint32_t w[32];
            tmem_ld32(tl + BKV, w);
#pragma unroll
            for (int d = 0; d < 32; d++) o[d] = fmaf(o[d], corr_prev, __uint_as_float(w[d]));
            tmem_ld32(tl + BKV + 32, w);
#pragma unroll
            for (int d = 0; d < 32; d++) o[32 + d] = fmaf(o[32 + d], corr_prev, __uint_as_float(w[d]));
            if (q < T) {
                const float inv = 1.0f / l;
                uint4* yr = reinterpret_cast<uint4*>(y + (long long)(row0 + q) * C + h * D);
#pragma unroll
                for (int i = 0; i < 8; i++)
                    yr[i] = make_uint4(pack_bf2(o[8 * i] * inv, o[8 * i + 1] * inv),
                                       pack_bf2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                       pack_bf2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                       pack_bf2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
                lse[((long long)b * H + h) * T + q] = (m + log2f(l)) * LN2;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------ backward
// dQ kernel shared-memory map.  One CTA per (batch, head, 128-query tile):
//   S = Q K_j^T and dP = dO V_j^T into TMEM; query-row threads form
//   dS = P o (dP - D) (P from the saved log-sum-exp) as bf16 in shared
//   memory; dQ += dS K_j accumulates in TMEM (K_j read as an MN-major B).
// The row threads first compute D = rowsum(dO o O) for their query and store
// it for the dK/dV kernel, which runs after this one.
constexpr int Q_Q = 0;
constexpr int Q_O = Q_Q + TILE;       // dO tile
constexpr int Q_K = Q_O + TILE;       // 2 stages
constexpr int Q_V = Q_K + 2 * TILE;   // 2 stages
constexpr int Q_S = Q_V + 2 * TILE;   // dS, 2 atoms
constexpr int Q_BAR = Q_S + 2 * TILE;
constexpr int Q_SMEM = Q_BAR + 256 + 1024;
constexpr uint32_t BWD_TMEM_COLS = 512;

__global__ void __launch_bounds__(THREADS_B, 1)
k_attn_bwd_dq_tc(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmo,
                 const bf16* __restrict__ y, const float* __restrict__ lse, float* __restrict__ Dlt,
                 bf16* __restrict__ dqkv, int T, int C, int H, int* flags) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint64_t* bars = (uint64_t*)(sm + Q_BAR);
    uint64_t* qo_full = bars + 0;
    uint64_t* kv_full = bars + 1;   // [2]
    uint64_t* kv_empty = bars + 3;  // [2]
    uint64_t* s_full = bars + 5;
    uint64_t* s_free = bars + 6;
    uint64_t* ds_full = bars + 7;
    uint64_t* ds_free = bars + 8;
    uint64_t* acc_full = bars + 9;
    uint32_t* tmem_holder = (uint32_t*)(bars + 10);
    volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

    const int nqt = gridDim.x;
    const int qt = nqt - 1 - (int)blockIdx.x;
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    const int nkv = qt + 1;
    const int row0 = b * T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(qo_full, 1);
        mbar_init(&kv_full[0], 1);
        mbar_init(&kv_full[1], 1);
        mbar_init(&kv_empty[0], 1);
        mbar_init(&kv_empty[1], 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, 256);
        mbar_init(ds_full, 256);
        mbar_init(ds_free, 1);
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(tmem_holder, BWD_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            const int xq = h * D, xk = C + h * D, xv = 2 * C + h * D;
            mbar_expect_tx(qo_full, 2 * TILE);
            tma_load_2d(smem_u32(sm + Q_Q), &tmq, qo_full, xq, row0 + qt * BQ);
            tma_load_2d(smem_u32(sm + Q_O), &tmo, qo_full, h * D, row0 + qt * BQ);
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < nkv; j++) {
                const int st = j & 1;
                if (!mbar_wait(&kv_empty[st], ((j >> 1) & 1) ^ 1, abort_flag, flags)) { ok = false; break; }
                mbar_expect_tx(&kv_full[st], 2 * TILE);
                tma_load_2d(smem_u32(sm + Q_K + st * TILE), &tmq, &kv_full[st], xk, row0 + j * BKV);
                tma_load_2d(smem_u32(sm + Q_V + st * TILE), &tmq, &kv_full[st], xv, row0 + j * BKV);
                ++issued;
            }
            if (!ok) {
                const long long t0 = clock64();
                while (!mbar_try_wait(qo_full, 0) && clock64() - t0 < WAIT_CYCLES) {}
                for (int j = (issued > 2 ? issued - 2 : 0); j < issued; j++)
                    while (!mbar_try_wait(&kv_full[j & 1], (j >> 1) & 1) && clock64() - t0 < 2 * WAIT_CYCLES) {}
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(BQ, BKV, false, false);
            constexpr uint32_t ID_Q = idesc_bf16(BQ, D, false, true);
            const uint32_t sq = smem_u32(sm + Q_Q), so = smem_u32(sm + Q_O), sds = smem_u32(sm + Q_S);
            bool ok = mbar_wait(qo_full, 0, abort_flag, flags);
            for (int j = 0; j < nkv && ok; j++) {
                const int st = j & 1;
                if (!mbar_wait(&kv_full[st], (j >> 1) & 1, abort_flag, flags)) { ok = false; break; }
                if (!mbar_wait(s_free, (j & 1) ^ 1, abort_flag, flags)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sk = smem_u32(sm + Q_K + st * TILE), sv = smem_u32(sm + Q_V + st * TILE);
#pragma unroll
                for (int k = 0; k < D / 16; k++)
                    umma_bf16(tmem, sdesc(sq + 32 * k, 16, 1024), sdesc(sk + 32 * k, 16, 1024), ID_S, k > 0);
#pragma unroll
                for (int k = 0; k < D / 16; k++)
                    umma_bf16(tmem + BKV, sdesc(so + 32 * k, 16, 1024), sdesc(sv + 32 * k, 16, 1024), ID_S,
                              k > 0);
                umma_commit(s_full);
                if (!mbar_wait(ds_full, j & 1, abort_flag, flags)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BKV / 16; k++)
                    umma_bf16(tmem + 2 * BKV, sdesc(sds + (k >> 2) * TILE + (k & 3) * 32, 16, 1024),
                              sdesc(sk + k * 2048, TILE, 1024), ID_Q, (j > 0 || k > 0) ? 1u : 0u);
                umma_commit(&kv_empty[st]);
                umma_commit(ds_free);
            }
            if (ok) umma_commit(acc_full);
        }
    } else {
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        const int q = qt * BQ + r;
        const bool qv = q < T;
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        const float sl2 = 0.125f * LOG2E;
        const long long bh = (long long)b * H + h;
        // D = rowsum(dO o O) for this query (dO row from the swizzled tile)
        if (!mbar_wait(qo_full, 0, abort_flag, flags)) goto rows_done;
        {
            float Dq = 0.0f;
            const uint8_t* orow = sm + Q_O + r * 128;
            const uint4* yr = reinterpret_cast<const uint4*>(y + (long long)(row0 + (qv ? q : 0)) * C + h * D);
#pragma unroll
            for (int c = 0; c < 8; c++) {
                const uint4 a = *reinterpret_cast<const uint4*>(orow + ((c ^ (r & 7)) * 16));
                const uint4 bb = yr[c];
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    Dq = fmaf(__uint_as_float(aw[i] << 16), __uint_as_float(bw[i] << 16), Dq);
                    Dq = fmaf(__uint_as_float(aw[i] & 0xFFFF0000u), __uint_as_float(bw[i] & 0xFFFF0000u), Dq);
                }
            }
            if (!qv) Dq = 0.0f;
            if (qv && half == 0) Dlt[bh * T + q] = Dq;
            const float Lq = qv ? lse[bh * T + q] * LOG2E : 0.0f;
            for (int j = 0; j < nkv; j++) {
                if (!mbar_wait(s_full, j & 1, abort_flag, flags)) goto rows_done;
                if (!mbar_wait(ds_free, (j & 1) ^ 1, abort_flag, flags)) goto rows_done;
                tc_fence_after();
                const bool diag = (j == qt);
                const int kq = q - j * BKV;  // key columns > kq are masked on the diagonal
#pragma unroll 1
                for (int c = 2 * half; c < 2 * half + 2; c++) {
                    uint32_t sw[32], pw[32], pk[16];
                    tmem_ld32(tl + c * 32, sw);
                    tmem_ld32(tl + BKV + c * 32, pw);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float d0 = ex2(fmaf(__uint_as_float(sw[e]), sl2, -Lq)) * (__uint_as_float(pw[e]) - Dq);
                        float d1 = ex2(fmaf(__uint_as_float(sw[e + 1]), sl2, -Lq)) * (__uint_as_float(pw[e + 1]) - Dq);
                        if (diag) {
                            if (c * 32 + e > kq) d0 = 0.0f;
                            if (c * 32 + e + 1 > kq) d1 = 0.0f;
                        }
                        pk[e >> 1] = pack_bf2(qv ? d0 : 0.0f, qv ? d1 : 0.0f);
                    }
                    store_row32(sm + Q_S, r, c * 32, pk);
                }
                tc_fence_before();
                mbar_arrive(s_free);
                fence_proxy_async_smem();
                mbar_arrive(ds_full);
            }
            if (!mbar_wait(acc_full, 0, abort_flag, flags)) goto rows_done;
            tc_fence_after();
            {
                uint32_t w0[32];
                tmem_ld32(tl + 2 * BKV + 32 * half, w0);
                if (qv) {
                    uint4* o = reinterpret_cast<uint4*>(dqkv + (long long)(row0 + q) * 3 * C + h * D + 32 * half);
                    const float sc = 0.125f;
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        o[i] = make_uint4(pack_bf2(__uint_as_float(w0[8 * i]) * sc, __uint_as_float(w0[8 * i + 1]) * sc),
                                          pack_bf2(__uint_as_float(w0[8 * i + 2]) * sc, __uint_as_float(w0[8 * i + 3]) * sc),
                                          pack_bf2(__uint_as_float(w0[8 * i + 4]) * sc, __uint_as_float(w0[8 * i + 5]) * sc),
                                          pack_bf2(__uint_as_float(w0[8 * i + 6]) * sc, __uint_as_float(w0[8 * i + 7]) * sc));
                }
            }
        }
    rows_done:;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, BWD_TMEM_COLS);
}

// dK/dV kernel shared-memory map.  One CTA per (batch, head, 128-key tile),
// looping over the query tiles at or after it:
//   S^T = K Q_j^T and dP^T = V dO_j^T into TMEM; key-row threads form P^T
//   and dS^T = P^T o (dP^T - D) as bf16 in shared memory; dV += P^T dO_j and
//   dK += dS^T Q_j accumulate in TMEM (Q_j and dO_j read as MN-major B).
constexpr int K_K = 0;
constexpr int K_V = K_K + TILE;
constexpr int K_Q = K_V + TILE;        // 2 stages
constexpr int K_O = K_Q + 2 * TILE;    // 2 stages
constexpr int K_P = K_O + 2 * TILE;    // P^T, 2 atoms
constexpr int K_S = K_P + 2 * TILE;    // dS^T, 2 atoms
constexpr int K_BAR = K_S + 2 * TILE;
constexpr int K_SMEM = K_BAR + 256 + 1024;

__global__ void __launch_bounds__(THREADS_B, 1)
k_attn_bwd_dkdv_tc(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmo,
                   const float* __restrict__ lse, const float* __restrict__ Dlt,
                   bf16* __restrict__ dqkv, int T, int C, int H, int* flags) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint64_t* bars = (uint64_t*)(sm + K_BAR);
    uint64_t* kv_full = bars + 0;
    uint64_t* qo_full = bars + 1;   // [2]
    uint64_t* qo_empty = bars + 3;  // [2]
    uint64_t* st_full = bars + 5;
    uint64_t* st_free = bars + 6;
    uint64_t* ps_full = bars + 7;
    uint64_t* ps_free = bars + 8;
    uint64_t* acc_full = bars + 9;
    uint32_t* tmem_holder = (uint32_t*)(bars + 10);
    volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

    const int nt = gridDim.x;
    const int kt = (int)blockIdx.x;   // key tile; tile kt loops over nt - kt query tiles
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    const int row0 = b * T;
    const int nq = nt - kt;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(&qo_full[0], 1);
        mbar_init(&qo_full[1], 1);
        mbar_init(&qo_empty[0], 1);
        mbar_init(&qo_empty[1], 1);
        mbar_init(st_full, 1);
        mbar_init(st_free, 256);
        mbar_init(ps_full, 256);
        mbar_init(ps_free, 1);
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(tmem_holder, BWD_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            const int xq = h * D, xk = C + h * D, xv = 2 * C + h * D;
            mbar_expect_tx(kv_full, 2 * TILE);
            tma_load_2d(smem_u32(sm + K_K), &tmq, kv_full, xk, row0 + kt * BKV);
            tma_load_2d(smem_u32(sm + K_V), &tmq, kv_full, xv, row0 + kt * BKV);
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < nq; i++) {
                const int st = i & 1, j = kt + i;
                if (!mbar_wait(&qo_empty[st], ((i >> 1) & 1) ^ 1, abort_flag, flags)) { ok = false; break; }
                mbar_expect_tx(&qo_full[st], 2 * TILE);
                tma_load_2d(smem_u32(sm + K_Q + st * TILE), &tmq, &qo_full[st], xq, row0 + j * BQ);
                tma_load_2d(smem_u32(sm + K_O + st * TILE), &tmo, &qo_full[st], h * D, row0 + j * BQ);
                ++issued;
            }
            if (!ok) {
                const long long t0 = clock64();
                while (!mbar_try_wait(kv_full, 0) && clock64() - t0 < WAIT_CYCLES) {}
                for (int i = (issued > 2 ? issued - 2 : 0); i < issued; i++)
                    while (!mbar_try_wait(&qo_full[i & 1], (i >> 1) & 1) && clock64() - t0 < 2 * WAIT_CYCLES) {}
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_bf16(BKV, BQ, false, false);
            constexpr uint32_t ID_A = idesc_bf16(BKV, D, false, true);
            const uint32_t sk = smem_u32(sm + K_K), sv = smem_u32(sm + K_V);
            const uint32_t sp = smem_u32(sm + K_P), sds = smem_u32(sm + K_S);
            bool ok = mbar_wait(kv_full, 0, abort_flag, flags);
            for (int i = 0; i < nq && ok; i++) {
                const int st = i & 1;
                if (!mbar_wait(&qo_full[st], (i >> 1) & 1, abort_flag, flags)) { ok = false; break; }
                if (!mbar_wait(st_free, (i & 1) ^ 1, abort_flag, flags)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sq = smem_u32(sm + K_Q + st * TILE), so = smem_u32(sm + K_O + st * TILE);
#pragma unroll
                for (int k = 0; k < D / 16; k++)
                    umma_bf16(tmem, sdesc(sk + 32 * k, 16, 1024), sdesc(sq + 32 * k, 16, 1024), ID_S, k > 0);
#pragma unroll
                for (int k = 0; k < D / 16; k++)
                    umma_bf16(tmem + BQ, sdesc(sv + 32 * k, 16, 1024), sdesc(so + 32 * k, 16, 1024), ID_S,
                              k > 0);
                umma_commit(st_full);
                if (!mbar_wait(ps_full, i & 1, abort_flag, flags)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BQ / 16; k++) {
                    const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
                    umma_bf16(tmem + 2 * BQ, sdesc(sp + (k >> 2) * TILE + (k & 3) * 32, 16, 1024),
                              sdesc(so + k * 2048, TILE, 1024), ID_A, acc);
                    umma_bf16(tmem + 2 * BQ + D, sdesc(sds + (k >> 2) * TILE + (k & 3) * 32, 16, 1024),
                              sdesc(sq + k * 2048, TILE, 1024), ID_A, acc);
                }
                umma_commit(&qo_empty[st]);
                umma_commit(ps_free);
            }
            if (ok) umma_commit(acc_full);
        }
    } else {
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        const int key = kt * BKV + r;
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        const float sl2 = 0.125f * LOG2E;
        const long long bh = (long long)b * H + h;
        const float* lrow = lse + bh * T;
        const float* drow = Dlt + bh * T;
        for (int i = 0; i < nq; i++) {
            const int j = kt + i;
            if (!mbar_wait(st_full, i & 1, abort_flag, flags)) break;
            if (!mbar_wait(ps_free, (i & 1) ^ 1, abort_flag, flags)) break;
            tc_fence_after();
            const bool diag = (i == 0);
#pragma unroll 1
            for (int c = 2 * half; c < 2 * half + 2; c++) {
                // the chunk's 32 queries: lane l fetches query q0 + l, then broadcasts
                const int q0 = j * BQ + c * 32;
                const bool lv = q0 + lane < T;
                const float Ll = lv ? __ldg(lrow + q0 + lane) * LOG2E : INFINITY;
                const float Dl = lv ? __ldg(drow + q0 + lane) : 0.0f;
                uint32_t sw[32], dw[32], pk[16], dk[16];
                tmem_ld32(tl + c * 32, sw);
                tmem_ld32(tl + BQ + c * 32, dw);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float L0 = __shfl_sync(0xffffffffu, Ll, e), L1 = __shfl_sync(0xffffffffu, Ll, e + 1);
                    const float D0 = __shfl_sync(0xffffffffu, Dl, e), D1 = __shfl_sync(0xffffffffu, Dl, e + 1);
                    float p0 = ex2(fmaf(__uint_as_float(sw[e]), sl2, -L0));
                    float p1 = ex2(fmaf(__uint_as_float(sw[e + 1]), sl2, -L1));
                    if (diag) {
                        if (q0 + e < key) p0 = 0.0f;
                        if (q0 + e + 1 < key) p1 = 0.0f;
                    }
                    pk[e >> 1] = pack_bf2(p0, p1);
                    dk[e >> 1] = pack_bf2(p0 * (__uint_as_float(dw[e]) - D0), p1 * (__uint_as_float(dw[e + 1]) - D1));
                }
                store_row32(sm + K_P, r, c * 32, pk);
                store_row32(sm + K_S, r, c * 32, dk);
            }
            tc_fence_before();
            mbar_arrive(st_free);
            fence_proxy_async_smem();
            mbar_arrive(ps_full);
        }
        if (mbar_wait(acc_full, 0, abort_flag, flags)) {
            tc_fence_after();
            // half 0 writes dV, half 1 writes dK (scaled by 1/sqrt(64))
            uint32_t w0[32], w1[32];
            tmem_ld32(tl + 2 * BQ + D * half, w0);
            tmem_ld32(tl + 2 * BQ + D * half + 32, w1);
            if (key < T) {
                const float sc = half ? 0.125f : 1.0f;
                uint4* o = reinterpret_cast<uint4*>(dqkv + (long long)(row0 + key) * 3 * C + (half ? C : 2 * C) + h * D);
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    o[i] = make_uint4(pack_bf2(__uint_as_float(w0[8 * i]) * sc, __uint_as_float(w0[8 * i + 1]) * sc),
                                      pack_bf2(__uint_as_float(w0[8 * i + 2]) * sc, __uint_as_float(w0[8 * i + 3]) * sc),
                                      pack_bf2(__uint_as_float(w0[8 * i + 4]) * sc, __uint_as_float(w0[8 * i + 5]) * sc),
                                      pack_bf2(__uint_as_float(w0[8 * i + 6]) * sc, __uint_as_float(w0[8 * i + 7]) * sc));
                    o[4 + i] = make_uint4(pack_bf2(__uint_as_float(w1[8 * i]) * sc, __uint_as_float(w1[8 * i + 1]) * sc),
                                          pack_bf2(__uint_as_float(w1[8 * i + 2]) * sc, __uint_as_float(w1[8 * i + 3]) * sc),
                                          pack_bf2(__uint_as_float(w1[8 * i + 4]) * sc, __uint_as_float(w1[8 * i + 5]) * sc),
                                          pack_bf2(__uint_as_float(w1[8 * i + 6]) * sc, __uint_as_float(w1[8 * i + 7]) * sc));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, BWD_TMEM_COLS);
}

}  // namespace fa5

bool attention_tc_eligible(bool bf16, int C, int H) {
    return bf16 && H > 0 && C % H == 0 && C / H == fa5::D && C % 8 == 0;
}

bool launch_attention_fwd_tc(const Launch& L, const void* qkv, void* y, float* lse, int B, int T,
                             int C, int H) {
    if (L.dry) return true;
    CUtensorMap tm;
    if (!tc::make_tmap_bf16(&tm, qkv, 3LL * C, (long long)B * T, 3LL * C, fa5::D, fa5::BQ)) return false;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(fa5::k_attn_fwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 fa5::F_SMEM) != cudaSuccess)
            return false;
        attr = true;
    }
    dim3 grid((T + fa5::BQ - 1) / fa5::BQ, B * H);
    L.count();
    fa5::k_attn_fwd_tc<<<grid, fa5::THREADS, fa5::F_SMEM, L.stream>>>(tm, (fa5::bf16*)y, lse, T, C, H,
                                                                     L.flags);
    return true;
}

}  // namespace tt

namespace tt {

bool launch_attention_bwd_tc(const Launch& L, const void* qkv, const void* y, const float* lse,
                             const void* dy, void* dqkv, int B, int T, int C, int H, float* Dlt) {
    if (L.dry) return true;
    CUtensorMap tmq, tmo;
    if (!tc::make_tmap_bf16(&tmq, qkv, 3LL * C, (long long)B * T, 3LL * C, fa5::D, fa5::BQ)) return false;
    if (!tc::make_tmap_bf16(&tmo, dy, (long long)C, (long long)B * T, (long long)C, fa5::D, fa5::BQ)) return false;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(fa5::k_attn_bwd_dq_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 fa5::Q_SMEM) != cudaSuccess ||
            cudaFuncSetAttribute(fa5::k_attn_bwd_dkdv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 fa5::K_SMEM) != cudaSuccess)
            return false;
        attr = true;
    }
    dim3 grid((T + fa5::BQ - 1) / fa5::BQ, B * H);
    L.count();
    fa5::k_attn_bwd_dq_tc<<<grid, fa5::THREADS_B, fa5::Q_SMEM, L.stream>>>(
        tmq, tmo, (const fa5::bf16*)y, lse, Dlt, (fa5::bf16*)dqkv, T, C, H, L.flags);
    L.count();
    fa5::k_attn_bwd_dkdv_tc<<<grid, fa5::THREADS_B, fa5::K_SMEM, L.stream>>>(
        tmq, tmo, lse, Dlt, (fa5::bf16*)dqkv, T, C, H, L.flags);
    return true;
}

}  // namespace tt

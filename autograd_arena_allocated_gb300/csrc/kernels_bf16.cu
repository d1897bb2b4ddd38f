// kernels_bf16.cu -- the memory-bound kernels of the bf16 step, written for
// HBM bandwidth: 16-byte vector loads and stores (8 bf16), rows held in
// registers between passes, grids sized from the SM count, and every
// reduction in a fixed order (no floating-point atomics).
//   LayerNorm forward / backward  (one warp per row)
//   fused cross entropy           (one 512-thread CTA per row, three passes, one exponential per logit)
//   column sums (bias gradients)  (8 columns per thread)
//   embedding-gradient scatter    (fixed 64-row chunks of the token-sorted
//                                  positions, then chunk partials in order)
#include "tt_internal.h"

#include <math.h>
#include <type_traits>
#include <algorithm>

namespace tt {

typedef __nv_bfloat16 bf16;

// Eight 16-bit values of a 16-byte vector as floats, and back (round to
// nearest even): bf16, or IEEE half when F16 (the fp16 mixed-precision step).
template <bool F16 = false>
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        if constexpr (F16) {
            f[2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xFFFFu)));
            f[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
        } else {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
}

template <bool F16 = false>
__device__ __forceinline__ uint32_t pk2(float a, float b) {
    if constexpr (F16) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

template <bool F16 = false>
__device__ __forceinline__ uint4 pack8(const float* f) {
    return make_uint4(pk2<F16>(f[0], f[1]), pk2<F16>(f[2], f[3]), pk2<F16>(f[4], f[5]), pk2<F16>(f[6], f[7]));
}

__device__ __forceinline__ float wsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ================================================================== LayerNorm
constexpr int LNV_WARPS = 8;

template <int NV, bool F16>
__global__ void __launch_bounds__(LNV_WARPS * 32)
k_ln_fwd_bf16(const bf16* __restrict__ x, const bf16* __restrict__ w, const bf16* __restrict__ b,
              bf16* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd, int M, int C) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * LNV_WARPS + (threadIdx.x >> 5);
    if (row >= M) return;
    const int nvec = C >> 3;
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * C);
    float v[NV][8];
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int vi = lane + 32 * i;
        if (vi < nvec) {
            unpack8<F16>(xr[vi], v[i]);
#pragma unroll
            for (int e = 0; e < 8; e++) s += v[i][e];
        }
    }
    const float mu = wsum(s) / C;
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < NV; i++)
        if (lane + 32 * i < nvec)
#pragma unroll
            for (int e = 0; e < 8; e++) { const float d = v[i][e] - mu; q += d * d; }
    const float rs = rsqrtf(wsum(q) / C + 1e-5f);
    uint4* yr = reinterpret_cast<uint4*>(y + row * C);
    const uint4* wr = reinterpret_cast<const uint4*>(w);
    const uint4* br = reinterpret_cast<const uint4*>(b);
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int vi = lane + 32 * i;
        if (vi < nvec) {
            float wf[8], bfv[8], o[8];
            unpack8<F16>(wr[vi], wf);
            unpack8<F16>(br[vi], bfv);
#pragma unroll
            for (int e = 0; e < 8; e++) o[e] = (v[i][e] - mu) * rs * wf[e] + bfv[e];
            yr[vi] = pack8<F16>(o);
        }
    }
    if (lane == 0) { mean[row] = mu; rstd[row] = rs; }
}

// Backward: a fixed grid of G blocks; warp j of block g takes rows
// g*8 + j, + 8G, + 16G, ...  Lane l owns columns 8(l + 32i) .. +7, so it keeps
// the dw/db partial sums of those columns (and gamma) in registers across its
// rows; at the end the block adds its warps' partials in warp order through
// shared memory and writes one partial row, and k_sum_rows adds the G block
// rows in block order (no atomics anywhere).
//
// With RES, the column sums of the finished dx (after the accumulation into
// the residual stream's gradient) are kept as a third partial: this
// LayerNorm's input is a residual-stream tensor whose gradient is complete
// once this kernel has added its share, and that tensor is the output of a
// linear layer, whose bias gradient is exactly these column sums.
// Rows reach shared memory by cp.async (16 bytes per lane, each lane copying
// exactly the vectors it later reads), LN_DEPTH(NV) rows ahead of the row the
// warp works on, so that a warp keeps several rows of loads in flight while it
// reduces one; both passes read the row from shared memory.
__host__ __device__ constexpr int ln_depth(int nv) { return nv <= 3 ? 3 : 2; }
// per warp: the row slots, reused at the end for the warp's partials
__host__ __device__ constexpr size_t ln_bwd_warp_bytes(int C, int nv, int np) {
    return (size_t)ln_depth(nv) * 3 * C * 2 > (size_t)np * C * 4 ? (size_t)ln_depth(nv) * 3 * C * 2
                                                                 : (size_t)np * C * 4;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int NV, bool RES, bool F16>
__global__ void __launch_bounds__(LNV_WARPS * 32, 2)
k_ln_bwd_bf16(const bf16* __restrict__ x, const bf16* __restrict__ w, const float* __restrict__ mean,
              const float* __restrict__ rstd, const bf16* __restrict__ dy, bf16* __restrict__ dx,
              float* __restrict__ part, int M, int C, int accumulate) {
    pdl_enter();
    constexpr int NP = RES ? 3 : 2;
    constexpr int DEPTH = ln_depth(NV);
    extern __shared__ __align__(16) uint8_t s_dyn[];  // [LNV_WARPS][ln_bwd_warp_bytes]
    __shared__ uint4 s_gamma[128];        // gamma, 8 values per entry (C <= 1024)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nvec = C >> 3;
    const float inv_c = 1.0f / (float)C;
    const size_t wbytes = ln_bwd_warp_bytes(C, NV, NP);
    uint8_t* wbase = s_dyn + warp * wbytes;
    // slot d of this warp: x | dy | old dx, C values each
    auto slot = [&](int d, int k) { return reinterpret_cast<uint4*>(wbase + ((size_t)d * 3 + k) * C * 2); };
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) s_gamma[v] = reinterpret_cast<const uint4*>(w)[v];
    float aw[NV][8], ab[NV][8], ar[RES ? NV : 1][8];
#pragma unroll
    for (int i = 0; i < NV; i++)
#pragma unroll
        for (int e = 0; e < 8; e++) { aw[i][e] = 0.0f; ab[i][e] = 0.0f; if (RES) ar[RES ? i : 0][e] = 0.0f; }
    __syncthreads();
    const long long stride = (long long)gridDim.x * LNV_WARPS;
    const long long row0 = (long long)blockIdx.x * LNV_WARPS + warp;
    auto issue = [&](long long row, int d) {
        if (row < M) {
#pragma unroll
            for (int i = 0; i < NV; i++) {
                const int vi = lane + 32 * i;
                if (vi < nvec) {
                    cp_async16(slot(d, 0) + vi, reinterpret_cast<const uint4*>(x + row * C) + vi);
                    cp_async16(slot(d, 1) + vi, reinterpret_cast<const uint4*>(dy + row * C) + vi);
                    if (accumulate) cp_async16(slot(d, 2) + vi, reinterpret_cast<const uint4*>(dx + row * C) + vi);
                }
            }
        }
        cp_async_commit();  // a group per row, empty past the end, so the waits count evenly
    };
#pragma unroll
    for (int d = 0; d < DEPTH - 1; d++) issue(row0 + d * stride, d);
    float mu_n = 0.0f, rs_n = 0.0f;
    if (row0 < M) { mu_n = mean[row0]; rs_n = rstd[row0]; }
    int k = 0;
    for (long long row = row0; row < M; row += stride, k++) {
        issue(row + (DEPTH - 1) * stride, (k + DEPTH - 1) % DEPTH);
        const float mu = mu_n, rs = rs_n;
        if (row + stride < M) { mu_n = mean[row + stride]; rs_n = rstd[row + stride]; }  // one row ahead
        cp_async_wait<DEPTH - 1>();  // this row's group has landed
        const int d = k % DEPTH;
        const uint4* sx = slot(d, 0);
        const uint4* sd = slot(d, 1);
        const uint4* so = slot(d, 2);
        uint4* xo = reinterpret_cast<uint4*>(dx + row * C);
        // pass 1: the two row sums, and this row's dw/db contributions
        float sg = 0.0f, sgx = 0.0f;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int vi = lane + 32 * i;
            if (vi < nvec) {
                float xf[8], df[8], wf[8];
                unpack8<F16>(sx[vi], xf);
                unpack8<F16>(sd[vi], df);
                unpack8<F16>(s_gamma[vi], wf);
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const float xh = (xf[e] - mu) * rs;
                    const float g = df[e] * wf[e];
                    sg += g;
                    sgx += g * xh;
                    aw[i][e] = fmaf(df[e], xh, aw[i][e]);
                    ab[i][e] += df[e];
                }
            }
        }
        const float mg = wsum(sg) * inv_c, mgx = wsum(sgx) * inv_c;
        // pass 2: dx
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int vi = lane + 32 * i;
            if (vi < nvec) {
                float xf[8], df[8], wf[8], o[8];
                unpack8<F16>(sx[vi], xf);
                unpack8<F16>(sd[vi], df);
                unpack8<F16>(s_gamma[vi], wf);
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const float xh = (xf[e] - mu) * rs;
                    o[e] = rs * (df[e] * wf[e] - mg - xh * mgx);
                }
                if (accumulate) {
                    float old[8];
                    unpack8<F16>(so[vi], old);
#pragma unroll
                    for (int e = 0; e < 8; e++) o[e] += old[e];
                }
                if (RES) {
#pragma unroll
                    for (int e = 0; e < 8; e++) ar[RES ? i : 0][e] += o[e];
                }
                xo[vi] = pack8<F16>(o);
            }
        }
    }
    cp_async_wait<0>();  // the empty trailing groups
    // the block's partials: warps in warp order (each warp over its own row slots)
    float* pw = reinterpret_cast<float*>(wbase);
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int vi = lane + 32 * i;
        if (vi < nvec) {
            float4* dwp = reinterpret_cast<float4*>(pw + vi * 8);
            float4* dbp = reinterpret_cast<float4*>(pw + C + vi * 8);
            dwp[0] = make_float4(aw[i][0], aw[i][1], aw[i][2], aw[i][3]);
            dwp[1] = make_float4(aw[i][4], aw[i][5], aw[i][6], aw[i][7]);
            dbp[0] = make_float4(ab[i][0], ab[i][1], ab[i][2], ab[i][3]);
            dbp[1] = make_float4(ab[i][4], ab[i][5], ab[i][6], ab[i][7]);
            if (RES) {
                const int ri = RES ? i : 0;
                float4* drp = reinterpret_cast<float4*>(pw + 2 * C + vi * 8);
                drp[0] = make_float4(ar[ri][0], ar[ri][1], ar[ri][2], ar[ri][3]);
                drp[1] = make_float4(ar[ri][4], ar[ri][5], ar[ri][6], ar[ri][7]);
            }
        }
    }
    __syncthreads();
    for (int c = threadIdx.x; c < NP * C; c += blockDim.x) {
        float s = 0.0f;
#pragma unroll
        for (int kk = 0; kk < LNV_WARPS; kk++)
            s += reinterpret_cast<const float*>(s_dyn + kk * wbytes)[c];
        part[(long long)blockIdx.x * NP * C + c] = s;
    }
}

// out[c] = sum_g part[g][c] over the G partial rows, in a fixed order: block
// = 32 columns x SR_WARPS warps; warp w adds rows w, w+SR_WARPS, ... (eight
// loads in flight); the warp sums are then added in warp order.  The G rows
// are few (a few hundred at most), so the kernel is latency bound: many warps
// keep the number of dependent load rounds per warp at one or two.  (Used for
// the LayerNorm dw/db (and dres) partials, with out_a taking columns [0, C),
// out_b columns [C, 2C) and out_c columns [2C, 3C), and for bias sums.)
constexpr int SR_WARPS = 32;

__global__ void __launch_bounds__(SR_WARPS * 32)
k_sum_rows(const float* __restrict__ part, int G, int ncols, int split, float* __restrict__ out_a,
           float* __restrict__ out_b, float* __restrict__ out_c, int acc) {
    pdl_enter();
    __shared__ float sm[SR_WARPS][33];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float s = 0.0f;
    if (c < ncols) {
        int g = warp;
        for (; g + 7 * SR_WARPS < G; g += 8 * SR_WARPS) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; u++) v[u] = part[(long long)(g + SR_WARPS * u) * ncols + c];
#pragma unroll
            for (int u = 0; u < 8; u++) s += v[u];
        }
        for (; g < G; g += SR_WARPS) s += part[(long long)g * ncols + c];
    }
    sm[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && c < ncols) {
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < SR_WARPS; w++) t += sm[w][lane];
        if (c < split) { if (out_a) out_a[c] = acc ? out_a[c] + t : t; }
        else if (c < 2 * split) { if (out_b) out_b[c - split] = acc ? out_b[c - split] + t : t; }
        else if (out_c) out_c[c - 2 * split] = acc ? out_c[c - 2 * split] + t : t;
    }
}

void launch_sum_rows(const Launch& L, const float* part, int G, int ncols, int split, float* out_a,
                     float* out_b, bool acc, float* out_c) {
    if (L.dry) return;
    L.count();
    launch_k(L, k_sum_rows, dim3((ncols + 31) / 32), dim3(SR_WARPS * 32), 0, part, G, ncols, split, out_a, out_b, out_c,
                                                                  acc ? 1 : 0);
}

constexpr int LN_BWD_MAX_BLOCKS = 1024;

// G = the blocks that are resident at once (SMs x blocks per SM), so that
// every block runs its rows in one wave; fewer when M is small.
template <int NV, bool RES>
static int ln_bwd_blocks(const Launch& L, int M) {
    static PerDevice per_sm;
    const int b = per_sm.value([] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_ln_bwd_bf16<NV, RES, false>, LNV_WARPS * 32,
                                                          LNV_WARPS * ln_bwd_warp_bytes(NV * 256, NV, RES ? 3 : 2)) !=
                cudaSuccess || n < 1) {
            cudaGetLastError();
            n = 1;
        }
        return n;
    });
    int g = b * (L.num_sms > 0 ? L.num_sms : 148);
    if (g > LN_BWD_MAX_BLOCKS) g = LN_BWD_MAX_BLOCKS;
    const int need = (M + LNV_WARPS - 1) / LNV_WARPS;
    return need < g ? need : g;
}

size_t ln_bwd_bf16_scratch_floats(int C) { return (size_t)LN_BWD_MAX_BLOCKS * 3 * C + 64; }

bool launch_ln_fwd_bf16(const Launch& L, const void* x, const void* w, const void* b, void* y,
                        float* mean, float* rstd, int M, int C) {
    if (C % 8 || C > 1024) return false;
    if (L.dry) return true;
    const unsigned grid = (unsigned)((M + LNV_WARPS - 1) / LNV_WARPS);
    const int nv = (C / 8 + 31) / 32;
    L.count();
#define LNF(NV, F) launch_k(L, k_ln_fwd_bf16<NV, F>, dim3(grid), dim3(LNV_WARPS * 32), 0,  \
        (const bf16*)x, (const bf16*)w, (const bf16*)b, (bf16*)y, mean, rstd, M, C)
    if (L.f16) {
        if (nv == 1) LNF(1, true); else if (nv == 2) LNF(2, true); else if (nv == 3) LNF(3, true); else LNF(4, true);
    } else {
        if (nv == 1) LNF(1, false); else if (nv == 2) LNF(2, false); else if (nv == 3) LNF(3, false); else LNF(4, false);
    }
#undef LNF
    return true;
}

bool launch_ln_bwd_bf16(const Launch& L, const void* x, const void* w, const float* mean,
                        const float* rstd, const void* dy, void* dx, float* dw, float* db, int M,
                        int C, bool accumulate, float* scratch, bool acc_params, float* dres) {
    if (C % 8 || C > 1024) return false;
    if (L.dry) return true;
    const int nv = (C / 8 + 31) / 32;
    const int np = dres ? 3 : 2;
    const size_t smem = LNV_WARPS * ln_bwd_warp_bytes(C, nv, np);
    static PerDevice attr;
    attr.once([] {
        // the largest any C <= 1024 needs
        int mx2 = 0, mx3 = 0;
        for (int c = 8; c <= 1024; c += 8) {
            const int v = (c / 8 + 31) / 32;
            mx2 = std::max(mx2, (int)(LNV_WARPS * ln_bwd_warp_bytes(c, v, 2)));
            mx3 = std::max(mx3, (int)(LNV_WARPS * ln_bwd_warp_bytes(c, v, 3)));
        }
#define LNA(NV, F)                                                                                        \
        cudaFuncSetAttribute(k_ln_bwd_bf16<NV, false, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx2); \
        cudaFuncSetAttribute(k_ln_bwd_bf16<NV, true, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx3)
        LNA(1, false); LNA(2, false); LNA(3, false); LNA(4, false);
        LNA(1, true); LNA(2, true); LNA(3, true); LNA(4, true);
#undef LNA
        return true;
    });
    L.count();
    int G = 0;
#define LNB(NV, RES, F) G = ln_bwd_blocks<NV, RES>(L, M); \
    launch_k(L, k_ln_bwd_bf16<NV, RES, F>, dim3(G), dim3(LNV_WARPS * 32), smem,  \
        (const bf16*)x, (const bf16*)w, mean, rstd, (const bf16*)dy, (bf16*)dx, scratch, M, C, \
        accumulate ? 1 : 0)
#define LNB_NV(RES, F) \
    if (nv == 1) { LNB(1, RES, F); } else if (nv == 2) { LNB(2, RES, F); } else if (nv == 3) { LNB(3, RES, F); } else { LNB(4, RES, F); }
    if (L.f16) {
        if (dres) { LNB_NV(true, true) } else { LNB_NV(false, true) }
    } else {
        if (dres) { LNB_NV(true, false) } else { LNB_NV(false, false) }
    }
#undef LNB_NV
#undef LNB
    L.count();
    launch_k(L, k_sum_rows, dim3((np * C + 31) / 32), dim3(SR_WARPS * 32), 0, scratch, G, np * C, C, dw, db, dres,
                                                                   acc_params ? 1 : 0);
    return true;
}

// ================================================================== cross entropy
constexpr float XV_LOG2E = 1.4426950408889634f;

// One CTA per row, three passes over the row (the first from HBM, the others
// from L2): (1) the row max, on packed bf16 pairs; (2) e = 2^((z - max) log2 e),
// summed, and written over z as bf16; (3) the gradient e * dscale / sum, written
// in place.  Each logit costs one exponential (the special-function pipe, not
// HBM, bounded the kernel when the gradient pass took a second one); the
// extra rounding of e to bf16 keeps the gradient within 2^-8 of its exact
// value.  Few registers, so several rows are in flight per SM; exponentials
// use the single hardware instruction ex2.approx (relative error ~2^-22).
constexpr int XS_THREADS = 512;

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <bool F16>
__global__ void __launch_bounds__(XS_THREADS)
k_xent_bf16(bf16* __restrict__ z, const int32_t* __restrict__ targets, float* __restrict__ row_loss,
            int V, int ld, float dscale, const float* __restrict__ scale_dev, int* flags) {
    pdl_enter();
    __shared__ float sm[XS_THREADS / 32];
    if (scale_dev) dscale *= *scale_dev;
    const long long row = blockIdx.x;
    uint4* zr = reinterpret_cast<uint4*>(z + row * (long long)ld);
    const int nvec = ld >> 3;
    const int vfull = V >> 3;  // vectors whose 8 columns are all < V
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // pass 1: max
    // the max on packed pairs of the storage type (exact in any order)
    using P2 = typename std::conditional<F16, __half2, __nv_bfloat162>::type;
    P2 m2;
    if constexpr (F16) m2 = __floats2half2_rn(-INFINITY, -INFINITY);
    else m2 = __floats2bfloat162_rn(-INFINITY, -INFINITY);
    float mx = -INFINITY;
    for (int vi = threadIdx.x; vi < nvec; vi += XS_THREADS) {
        const uint4 u = zr[vi];
        if (vi < vfull) {
            m2 = __hmax2(m2, *reinterpret_cast<const P2*>(&u.x));
            m2 = __hmax2(m2, *reinterpret_cast<const P2*>(&u.y));
            m2 = __hmax2(m2, *reinterpret_cast<const P2*>(&u.z));
            m2 = __hmax2(m2, *reinterpret_cast<const P2*>(&u.w));
        } else {
            float f[8];
            unpack8<F16>(u, f);
#pragma unroll
            for (int e = 0; e < 8; e++)
                if (vi * 8 + e < V) mx = fmaxf(mx, f[e]);
        }
    }
    mx = fmaxf(mx, fmaxf(__low2float(m2), __high2float(m2)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) sm[warp] = mx;
    __syncthreads();
    mx = sm[0];
#pragma unroll
    for (int k = 1; k < XS_THREADS / 32; k++) mx = fmaxf(mx, sm[k]);
    const float ml = mx * XV_LOG2E;
    const int tgt = targets[row];
    const bool ok = tgt >= 0 && tgt < V;
    const int tv = ok ? (tgt >> 3) : -1;
    // pass 2: e = 2^((z - max) log2 e), summed, and kept in place of z (bf16)
    // so that the gradient pass needs no second exponential
    float s = 0.0f, ztgt = 0.0f;
    for (int vi = threadIdx.x; vi < nvec; vi += XS_THREADS) {
        float f[8], ex[8];
        unpack8<F16>(zr[vi], f);
        if (vi == tv) ztgt = f[tgt & 7];
        if (vi < vfull) {
#pragma unroll
            for (int e = 0; e < 8; e++) {
                ex[e] = ex2f(fmaf(f[e], XV_LOG2E, -ml));
                s += ex[e];
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; e++) {
                ex[e] = (vi * 8 + e < V) ? ex2f(fmaf(f[e], XV_LOG2E, -ml)) : 0.0f;
                s += ex[e];
            }
        }
        zr[vi] = pack8<F16>(ex);
    }
    s = wsum(s);
    __syncthreads();  // everyone has read sm[] above
    if (lane == 0) sm[warp] = s;
    __syncthreads();
    float S_ = 0.0f;
#pragma unroll
    for (int k = 0; k < XS_THREADS / 32; k++) S_ += sm[k];  // same order in every thread
    const float lse = mx + logf(S_);
    if (!ok && threadIdx.x == 0) {
        atomicOr(&flags[FLAG_BAD_TOKEN], 1);
        row_loss[row] = 0.0f;
    }
    // pass 3: gradient, in place: softmax = e / S (pad columns hold e = 0)
    const float k = dscale / S_;
    for (int vi = threadIdx.x; vi < nvec; vi += XS_THREADS) {
        float ex[8], o[8];
        unpack8<F16>(zr[vi], ex);
#pragma unroll
        for (int e = 0; e < 8; e++) o[e] = ex[e] * k;
        if (vi == tv) {
            row_loss[row] = lse - ztgt;
            o[tgt & 7] -= dscale;
        }
        zr[vi] = pack8<F16>(o);
    }
}

bool launch_xent_bf16(const Launch& L, void* logits, const int32_t* targets, float* row_loss, int M,
                      int V, int ld, float dscale, const float* scale_dev) {
    if (ld % 8 || ((uintptr_t)logits & 15) || ld < 2048) return false;
    if (L.dry) return true;
    L.count();
    if (L.f16)
        launch_k(L, k_xent_bf16<true>, dim3(M), dim3(XS_THREADS), 0, (bf16*)logits, targets, row_loss, V, ld, dscale,
                                                           scale_dev, L.flags);
    else
        launch_k(L, k_xent_bf16<false>, dim3(M), dim3(XS_THREADS), 0, (bf16*)logits, targets, row_loss, V, ld, dscale,
                                                            scale_dev, L.flags);
    return true;
}

// ================================================================== column sums
constexpr int CS_ROWS = 256;  // rows per partial (the same chunking as the generic kernel)

// block: 32 lanes x 8 columns = 256 columns, 8 warps split the 256 rows of
// one partial (warp w takes rows w, w+8, ...); warps combine in warp order
template <bool F16>
__global__ void __launch_bounds__(256)
k_colsum_bf16(const bf16* __restrict__ x, int M, int N, float* __restrict__ part) {
    pdl_enter();
    __shared__ float sm[8][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n8 = blockIdx.x * 256 + lane * 8;
    const long long r0 = (long long)blockIdx.y * CS_ROWS;
    const long long r1 = min((long long)M, r0 + CS_ROWS);
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (n8 < N) {
        // rows r0 + warp + 8j in increasing j; 8 loads in flight per thread
        constexpr int U = 8;
        long long r = r0 + warp;
        for (; r + 8 * (U - 1) < r1; r += 8 * U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; u++) v[u] = *reinterpret_cast<const uint4*>(x + (r + 8 * u) * N + n8);
#pragma unroll
            for (int u = 0; u < U; u++) {
                float f[8];
                unpack8<F16>(v[u], f);
#pragma unroll
                for (int e = 0; e < 8; e++) acc[e] += f[e];
            }
        }
        for (; r < r1; r += 8) {
            float f[8];
            unpack8<F16>(*reinterpret_cast<const uint4*>(x + r * N + n8), f);
#pragma unroll
            for (int e = 0; e < 8; e++) acc[e] += f[e];
        }
    }
#pragma unroll
    for (int e = 0; e < 8; e++) sm[warp][lane * 8 + e] = acc[e];
    __syncthreads();
    const int col = blockIdx.x * 256 + threadIdx.x;
    if (col < N) {
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; w++) t += sm[w][threadIdx.x];
        part[(long long)blockIdx.y * N + col] = t;
    }
}

bool launch_colsum_bf16(const Launch& L, const void* x, int M, int N, float* part) {
    if (N % 8 || ((uintptr_t)x & 15) || ((uintptr_t)part & 15)) return false;
    if (L.dry) return true;
    dim3 grid((N + 255) / 256, (M + CS_ROWS - 1) / CS_ROWS);
    L.count();
    if (L.f16) launch_k(L, k_colsum_bf16<true>, dim3(grid), dim3(256), 0, (const bf16*)x, M, N, part);
    else launch_k(L, k_colsum_bf16<false>, dim3(grid), dim3(256), 0, (const bf16*)x, M, N, part);
    return true;
}

// ================================================================== embedding gradient
// After the stable sort, positions with equal token id form runs.  Chunk c
// (sorted indices [64c, 64c+64)) sums each run piece it holds in sorted order:
// a run wholly inside the chunk goes straight to dwte; the piece of a run
// that began in an earlier chunk goes to first[c]; the piece of a run that
// continues into the next chunk goes to last[c].  The chunk where such a run
// begins then adds last[c] + first[c+1] + ... in chunk order.
constexpr int EB_CHUNK = 64;

template <typename T>
__device__ __forceinline__ void load8(const T* p, float* f);
template <>
__device__ __forceinline__ void load8<bf16>(const bf16* p, float* f) {
    unpack8(*reinterpret_cast<const uint4*>(p), f);
}
template <>
__device__ __forceinline__ void load8<__half>(const __half* p, float* f) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float* f) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ void store8(float* p, const float* f) {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

__device__ __forceinline__ void add8(float* p, const float* f) {
    float4 a = reinterpret_cast<float4*>(p)[0], b = reinterpret_cast<float4*>(p)[1];
    a.x += f[0]; a.y += f[1]; a.z += f[2]; a.w += f[3];
    b.x += f[4]; b.y += f[5]; b.z += f[6]; b.w += f[7];
    reinterpret_cast<float4*>(p)[0] = a;
    reinterpret_cast<float4*>(p)[1] = b;
}

// thread t owns columns [8t, 8t+8)
template <typename T>
__global__ void k_embed_chunks(const T* __restrict__ dx, const int32_t* __restrict__ keys,
                               const int32_t* __restrict__ vals, int M, int C, int V,
                               float* __restrict__ dwte, float* __restrict__ first,
                               float* __restrict__ last) {
    pdl_enter();
    const int c = blockIdx.x;
    const int col = threadIdx.x * 8;
    if (col >= C) return;
    const int i0 = c * EB_CHUNK, i1 = min(M, i0 + EB_CHUNK);
    const bool continues_in = i0 > 0 && keys[i0 - 1] == keys[i0];
    const bool continues_out = i1 < M && keys[i1] == keys[i1 - 1];
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int run_key = keys[i0], run_start = i0;
    for (int i = i0; i <= i1; i++) {
        const int k = i < i1 ? keys[i] : -1;
        if (k != run_key) {
            // close the run piece [run_start, i)
            if (run_key < V) {
                const bool began_before = run_start == i0 && continues_in;
                const bool goes_on = i == i1 && continues_out;
                if (began_before) store8(first + (long long)c * C + col, acc);
                else if (goes_on) store8(last + (long long)c * C + col, acc);
                else add8(dwte + (long long)run_key * C + col, acc);
            }
#pragma unroll
            for (int e = 0; e < 8; e++) acc[e] = 0.0f;
            run_key = k;
            run_start = i;
            if (i == i1) break;
        }
        if (k < V) {
            float f[8];
            load8(dx + (long long)vals[i] * C + col, f);
#pragma unroll
            for (int e = 0; e < 8; e++) acc[e] += f[e];
        }
    }
}

template <typename T>
__global__ void k_embed_gather(const int32_t* __restrict__ keys, int M, int C, int V,
                               float* __restrict__ dwte, const float* __restrict__ first,
                               const float* __restrict__ last) {
    pdl_enter();
    const int c = blockIdx.x;
    const int col = threadIdx.x * 8;
    if (col >= C) return;
    const int i0 = c * EB_CHUNK, i1 = min(M, i0 + EB_CHUNK);
    if (!(i1 < M && keys[i1] == keys[i1 - 1])) return;  // last run does not continue
    const int key = keys[i1 - 1];
    if (key >= V) return;
    // owner only if the run begins in this chunk
    if (keys[i0] == key && i0 > 0 && keys[i0 - 1] == key) return;
    float acc[8], f[8];
    const float* p = last + (long long)c * C + col;
#pragma unroll
    for (int e = 0; e < 8; e++) acc[e] = p[e];
    for (int cc = c + 1; cc * EB_CHUNK < M; cc++) {
        const float* q = first + (long long)cc * C + col;
#pragma unroll
        for (int e = 0; e < 8; e++) f[e] = q[e];
#pragma unroll
        for (int e = 0; e < 8; e++) acc[e] += f[e];
        const int j1 = min(M, (cc + 1) * EB_CHUNK);
        if (!(j1 < M && keys[j1] == key)) break;  // the run ends in chunk cc
    }
    add8(dwte + (long long)key * C + col, acc);
}

size_t embed_chunk_scratch_floats(int M, int C) {
    return (size_t)2 * ((M + EB_CHUNK - 1) / EB_CHUNK) * C + 64;
}

bool launch_embed_chunks(const Launch& L, bool is_bf16, const void* dx, const int32_t* keys,
                         const int32_t* vals, int M, int C, int V, float* dwte, float* scratch) {
    if (C % 8 || C > 8 * 1024) return false;
    if (L.dry) return true;
    const int nchunk = (M + EB_CHUNK - 1) / EB_CHUNK;
    float* first = scratch;
    float* last = scratch + (size_t)nchunk * C;
    const int threads = ((C / 8 + 31) / 32) * 32;
    L.count();
    if (is_bf16 && L.f16)
        launch_k(L, k_embed_chunks<__half>, dim3(nchunk), dim3(threads), 0, (const __half*)dx, keys, vals, M, C, V,
                                                                 dwte, first, last);
    else if (is_bf16)
        launch_k(L, k_embed_chunks<bf16>, dim3(nchunk), dim3(threads), 0, (const bf16*)dx, keys, vals, M, C, V,
                                                               dwte, first, last);
    else
        launch_k(L, k_embed_chunks<float>, dim3(nchunk), dim3(threads), 0, (const float*)dx, keys, vals, M, C, V,
                                                                dwte, first, last);
    L.count();
    launch_k(L, k_embed_gather<float>, dim3(nchunk), dim3(threads), 0, keys, M, C, V, dwte, first, last);
    return true;
}

}  // namespace tt

// attn_tc.cu -- causal self-attention on the 5th-generation tensor cores
// (tcgen05, bf16 in, fp32 accumulate in tensor memory), head dim 64.
//
// Every kernel streams 64-wide blocks of the other sequence past a
// 128-row tile, so that the score block (128 x 64 fp32) needs only 64 TMEM
// columns and several CTAs fit on one SM; each CTA has 192 threads:
//   warp 0      TMA (128-byte-swizzled tiles straight from the packed
//               [B*T, 3C] qkv buffer and the [B*T, C] output gradient)
//   warp 1      TMEM allocation and the MMAs (one elected lane)
//   warps 2..5  one thread per tile row: reads its row of the score block
//               from TMEM, does the elementwise work in fp32, and writes the
//               bf16 operand of the next MMA into shared memory in the
//               128-byte-swizzled K-major layout the MMA reads.
//
// In every kernel the MMA warp issues the next block's score MMAs as soon as
// the row threads have copied the current scores from TMEM to registers, and
// the row threads compute the next MMA operand in registers before they wait
// for its shared-memory buffer, so the tensor pipe and the elementwise work
// overlap instead of taking turns.
//
// Forward (one CTA per 128 queries, 3 CTAs/SM): S = Q K_j^T; online softmax
//   in base 2; P_j to shared memory (two buffers); O += P_j V_j accumulates in
//   TMEM (V read as an MN-major operand), rescaled in place only when the row
//   max grows by more than 2^8; finally y = O / l and the row's log-sum-exp.
// Backward, deterministic (no atomics):
//   dQ kernel (one CTA per 128 queries, 2 CTAs/SM): D = rowsum(dO o O);
//     S = Q K_j^T, dP = dO V_j^T; dS = P o (dP - D) with P from the saved
//     log-sum-exp (two dS buffers); dQ += dS K_j accumulates in TMEM.
//   dK/dV kernel (one CTA per 128 keys, 2 CTAs/SM): S^T = K Q_j^T,
//     dP^T = V dO_j^T; P^T and dS^T; dV += P^T dO_j, dK += dS^T Q_j in TMEM
//     (Q_j and dO_j, loaded K-major, are read again as MN-major operands).
// Every wait is bounded (FLAG_TIMEOUT), as in the GEMM.
#include "tt_internal.h"
#include "tc_ptx.cuh"

#include <math.h>

namespace tt {
namespace fa5 {

using namespace tc;
typedef __nv_bfloat16 bf16;

constexpr int D = 64;
constexpr int BQ = 128;  // rows of the CTA's tile
constexpr int BN = 64;   // width of the streamed blocks
constexpr int THREADS = 192;
constexpr int T128 = 128 * 128;  // 128 rows x 128 bytes
constexpr int T64 = 64 * 128;    // 64 rows x 128 bytes
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float SL2 = 0.125f * LOG2E;  // 1/sqrt(64), base-2 units

// Grid (band, tiles, bands): blockIdx.x is a (batch, head) pair within a band
// of BAND pairs, y the tile (heaviest first), z the band.  The hardware hands
// CTAs out x fastest, so a band's pairs go out together, every pair's heaviest
// tile first: the short tiles fill the gaps at the band's end while the next
// band starts, and the operands of a band's pairs (256 KB a pair, read by all
// its tiles) stay in L2 while it runs, so each kernel reads them from DRAM
// about once.  Slots past the last pair return at once.
constexpr int BAND = 64;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return (uint8_t*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

// 2^x by the single hardware instruction (relative error ~2^-22)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 32 bf16 values (columns k0..k0+31, k0 in {0, 32}) of row r of a K-major,
// 128-byte-swizzled [128 rows x 64 columns] operand (16-byte chunk c of row r
// at c ^ (r mod 8)).  Rows of 32 consecutive lanes: conflict-free.
__device__ __forceinline__ void store_row32(uint8_t* base, int r, int k0, const uint32_t (&w)[16]) {
    uint8_t* row = base + r * 128;
    const int c0 = k0 >> 3;
#pragma unroll
    for (int i = 0; i < 4; i++)
        *reinterpret_cast<uint4*>(row + (((c0 + i) ^ (r & 7)) << 4)) =
            make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

template <bool F16>
__device__ __forceinline__ void store_out64(bf16* dst, const float* v, float scale) {
    uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 8; i++)
        o[i] = make_uint4(pack2<F16>(v[8 * i] * scale, v[8 * i + 1] * scale),
                          pack2<F16>(v[8 * i + 2] * scale, v[8 * i + 3] * scale),
                          pack2<F16>(v[8 * i + 4] * scale, v[8 * i + 5] * scale),
                          pack2<F16>(v[8 * i + 6] * scale, v[8 * i + 7] * scale));
}

__device__ __forceinline__ void init_done() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ================================================================== forward
// The softmax warps never wait for the P.V product of the previous block in
// the common case: P is double-buffered in shared memory (buffer j & 1, with
// its own full / consumed barriers), the exponentials of block j are
// computed in registers while P_{j-1} V_{j-1} runs, and the warps wait for
// the previous product only when the row maximum forces a rescale of O.
constexpr int F_Q = 0;
constexpr int F_K = F_Q + T128;     // 2 stages
constexpr int F_V = F_K + 2 * T64;  // 1 stage
constexpr int F_P = F_V + T64;      // P: 2 x [128 x 64] bf16
constexpr int F_BAR = F_P + 2 * T128;
constexpr int F_SMEM = F_BAR + 256 + 1024;
constexpr uint32_t F_TMEM = 128;    // S: cols 0..63, O: 64..127

template <bool F16>
__global__ void __launch_bounds__(THREADS, 3)
k_attn_fwd_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              bf16* __restrict__ y, float* __restrict__ lse, int T, int C, int H, int nbh, int* flags,
              long long wl) {
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
    uint64_t* p_full = bars + 9;   // [2]: P buffer written
    uint64_t* o_full = bars + 11;  // [2]: P.V of a block in buffer s done (buffer s consumed)
    uint64_t* drain = bars + 13;   // MMAs issued before an abort are done
    uint32_t* tmem_holder = (uint32_t*)(bars + 14);
    volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

    const int bh = (int)(blockIdx.z * gridDim.x + blockIdx.x);
    if (bh >= nbh) return;  // the last band's unused slots (uniform over the CTA, before any setup)
    const int nqt = gridDim.y;
    const int qt = nqt - 1 - (int)blockIdx.y;  // longest rows first within the band
    const int b = bh / H, h = bh % H;
    const int nkv = min(2 * qt + 2, (T + BN - 1) / BN);
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
        mbar_init(&p_full[0], 128);
        mbar_init(&p_full[1], 128);
        mbar_init(&o_full[0], 1);
        mbar_init(&o_full[1], 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        init_done();
    }
    if (warp == 1) tmem_alloc(tmem_holder, F_TMEM);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    pdl_enter();  // the set-up above overlaps the previous kernel's end; global memory only from here

    if (warp == 0) {
        if (lane == 0) {
            const int xq = h * D, xk = C + h * D, xv = 2 * C + h * D;
            mbar_expect_tx(q_full, T128);
            tma_load_2d(smem_u32(sm + F_Q), &tq, q_full, xq, row0 + qt * BQ);
            // K runs two blocks ahead of V: K_{j+2} needs only S_j done, while
            // V_{j+1} has to wait for P_j V_j (V has one buffer)
            int issued_k = 0, issued_v = 0;
            bool ok = true;
            auto load_k = [&](int j) -> bool {
                const int st = j & 1;
                if (!mbar_wait(&k_empty[st], ((j >> 1) & 1) ^ 1, abort_flag, flags, 0x100 + 1, wl)) return false;
                mbar_expect_tx(&k_full[st], T64);
                tma_load_2d(smem_u32(sm + F_K + st * T64), &tk, &k_full[st], xk, row0 + j * BN);
                ++issued_k;
                return true;
            };
            ok = load_k(0) && (nkv < 2 || load_k(1));
            for (int j = 0; j < nkv && ok; j++) {
                if (!mbar_wait(v_empty, (j & 1) ^ 1, abort_flag, flags, 0x100 + 2, wl)) { ok = false; break; }
                mbar_expect_tx(v_full, T64);
                tma_load_2d(smem_u32(sm + F_V), &tk, v_full, xv, row0 + j * BN);
                ++issued_v;
                if (j + 2 < nkv && !load_k(j + 2)) { ok = false; break; }
            }
            if (!ok) {  // let issued copies land before the CTA exits
                mbar_drain(q_full, 0);
                for (int j = (issued_k > 2 ? issued_k - 2 : 0); j < issued_k; j++)
                    mbar_drain(&k_full[j & 1], (j >> 1) & 1);
                if (issued_v > 0) mbar_drain(v_full, (issued_v - 1) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID = idesc16<F16>(BQ, BN, false, false);
            constexpr uint32_t ID_O = idesc16<F16>(BQ, D, false, true);
            const uint32_t sq = smem_u32(sm + F_Q), sv = smem_u32(sm + F_V);
            bool ok = mbar_wait(q_full, 0, abort_flag, flags, 0x100 + 3, wl);
            bool issued = false;
            // S_{j+1} is issued as soon as the row threads hold S_j in registers,
            // so that it overlaps the softmax of block j
            auto issue_s = [&](int j) -> bool {
                const int st = j & 1;
                if (!mbar_wait(&k_full[st], (j >> 1) & 1, abort_flag, flags, 0x100 + 4, wl)) return false;
                if (!mbar_wait(s_free, (j & 1) ^ 1, abort_flag, flags, 0x100 + 5, wl)) return false;
                tc_fence_after();
                const uint32_t sk = smem_u32(sm + F_K + st * T64);
#pragma unroll
                for (int k = 0; k < D / 16; k++)
                    umma_bf16(tmem, sdesc(sq + 32 * k, 16, 1024), sdesc(sk + 32 * k, 16, 1024), ID, k > 0);
                issued = true;
                umma_commit(s_full);
                umma_commit(&k_empty[st]);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; j < nkv && ok; j++) {
                if (j + 1 < nkv && !issue_s(j + 1)) { ok = false; break; }
                const int pb = j & 1;
                if (!mbar_wait(&p_full[pb], (j >> 1) & 1, abort_flag, flags, 0x100 + 6, wl)) { ok = false; break; }
                if (!mbar_wait(v_full, j & 1, abort_flag, flags, 0x100 + 7, wl)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sp = smem_u32(sm + F_P + pb * T128);
#pragma unroll
                for (int k = 0; k < BN / 16; k++)
                    umma_bf16(tmem + BN, sdesc(sp + 32 * k, 16, 1024), sdesc(sv + k * 2048, T64, 1024), ID_O,
                              (j > 0 || k > 0) ? 1u : 0u);
                umma_commit(&o_full[pb]);
                umma_commit(v_empty);
            }
            if (!ok && issued) {  // the MMAs already issued finish before tensor memory is freed
                umma_commit(drain);
                mbar_drain(drain, 0);
            }
        }
    } else {
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int q = qt * BQ + r;
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        // P is taken relative to a reference max m that is raised -- and O, l
        // rescaled in place -- only when some row of the warp exceeds it by
        // more than 8 (P <= 2^8 otherwise); the decision is a warp vote since
        // the TMEM loads and stores of O are warp-collective
        float m = -INFINITY, l = 0.0f;
        bool ok = true;
        for (int j = 0; j < nkv; j++) {
            if (!mbar_wait_warp(s_full, j & 1, abort_flag, flags, 0x100 + 8, wl)) { ok = false; break; }
            tc_fence_after();
            const bool diag = (j >= 2 * qt);
            const int kq = q - j * BN;  // on the diagonal, key columns > kq are masked
            uint32_t w0[32], w1[32];
            tmem_ld32x2(tl, w0, tl + 32, w1);
            tc_fence_before();
            mbar_arrive(s_free);  // S is in registers: the next S may be computed
            // row max over four independent chains (max is exact in any order)
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (!diag) {
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    mq[0] = fmaxf(mq[0], __uint_as_float(w0[e]));
                    mq[1] = fmaxf(mq[1], __uint_as_float(w0[e + 1]));
                    mq[2] = fmaxf(mq[2], __uint_as_float(w1[e]));
                    mq[3] = fmaxf(mq[3], __uint_as_float(w1[e + 1]));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    if (e <= kq) mq[0] = fmaxf(mq[0], __uint_as_float(w0[e]));
                    if (e + 1 <= kq) mq[1] = fmaxf(mq[1], __uint_as_float(w0[e + 1]));
                    if (32 + e <= kq) mq[2] = fmaxf(mq[2], __uint_as_float(w1[e]));
                    if (33 + e <= kq) mq[3] = fmaxf(mq[3], __uint_as_float(w1[e + 1]));
                }
            }
            const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            const float mn = fmaxf(m, mx * SL2);
            const bool rescale = j > 0 && __any_sync(0xffffffffu, mn > m + 8.0f);
            const float m_old = m;
            if (j == 0 || rescale) m = mn;
            const int pb = j & 1;
            // buffer pb was last read by P_{j-2} V_{j-2} (long done, as a rule)
            if (j >= 2 && !mbar_wait_warp(&o_full[pb], ((j - 2) >> 1) & 1, abort_flag, flags, 0x100 + 9, wl)) {
                ok = false;
                break;
            }
            // P = 2^(s*scale - m) as bf16, each 32-column half straight to shared memory
            uint8_t* pbuf = sm + F_P + pb * T128;
            // (packed fp32x2 scale-and-subtract and sums: two lanes per instruction;
            // the sums in two independent packed chains)
            float2 rsa = make_float2(0.0f, 0.0f), rsb = make_float2(0.0f, 0.0f);
            const float2 sl2 = make_float2(SL2, SL2), nm = make_float2(-m, -m);
#pragma unroll
            for (int c = 0; c < 2; c++) {
                const uint32_t(&w)[32] = c ? w1 : w0;
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(w[e]), __uint_as_float(w[e + 1])), sl2, nm);
                    float2 p = make_float2(ex2(x.x), ex2(x.y));
                    if (diag) {
                        if (32 * c + e > kq) p.x = 0.0f;
                        if (32 * c + e + 1 > kq) p.y = 0.0f;
                    }
                    if (e & 2) rsb = __fadd2_rn(rsb, p);
                    else rsa = __fadd2_rn(rsa, p);
                    pk[e >> 1] = pack2<F16>(p.x, p.y);
                }
                store_row32(pbuf, r, 32 * c, pk);
            }
            const float rs = (rsa.x + rsb.x) + (rsa.y + rsb.y);
            if (rescale) {
                // O must hold P_{j-1} V_{j-1} before it is scaled
                if (!mbar_wait_warp(&o_full[pb ^ 1], ((j - 1) >> 1) & 1, abort_flag, flags, 0x100 + 10, wl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float corr = ex2(m_old - m);
                uint32_t v[32];
                tmem_ld32(tl + BN, v);
#pragma unroll
                for (int d = 0; d < 32; d++) v[d] = __float_as_uint(__uint_as_float(v[d]) * corr);
                tmem_st32(tl + BN, v);
                tmem_ld32(tl + BN + 32, v);
#pragma unroll
                for (int d = 0; d < 32; d++) v[d] = __float_as_uint(__uint_as_float(v[d]) * corr);
                tmem_st32(tl + BN + 32, v);
                tmem_st_wait();
                l *= corr;
            }
            l += rs;
            tc_fence_before();  // orders the TMEM stores of a rescale before the next MMA
            fence_proxy_async_smem();
            mbar_arrive(&p_full[pb]);
        }
        const int jl = nkv - 1;
        if (ok && mbar_wait_warp(&o_full[jl & 1], (jl >> 1) & 1, abort_flag, flags, 0x100 + 11, wl)) {
            tc_fence_after();
            float o[D];
            uint32_t v[32];
            tmem_ld32(tl + BN, v);
#pragma unroll
            for (int d = 0; d < 32; d++) o[d] = __uint_as_float(v[d]);
            tmem_ld32(tl + BN + 32, v);
#pragma unroll
            for (int d = 0; d < 32; d++) o[32 + d] = __uint_as_float(v[d]);
            if (q < T) {
                store_out64<F16>(y + (long long)(row0 + q) * C + h * D, o, 1.0f / l);
                lse[((long long)b * H + h) * T + q] = (m + log2f(l)) * LN2;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, F_TMEM);
}

// ================================================================== backward
// Both backward kernels run 320 threads: warp 0 loads by TMA, warp 1 owns the
// tensor memory and issues the MMAs, and warps 2..9 are the row warps.  Two
// row warps share each 32-lane quarter of tensor memory (quarter = warp & 3)
// and split the streamed block's 64 columns: half (warp - 2) >> 2 takes
// columns [32 half, 32 half + 32).  Each thread therefore owns one row and
// 32 columns of the score block.
//
// The bf16 operand that the row threads produce (dS in the dQ kernel, P^T and
// dS^T in the dK/dV kernel) is written into tensor memory over the scores it
// was computed from -- half h writes the 16 columns [32 h, 32 h + 16) of its
// own 32 -- and the next MMAs read it from there as their A operand, so the
// N = 64 products read only their B operand from shared memory.  The next
// block's score MMAs overwrite those columns; they are issued after the MMAs
// that read them, and one thread's tcgen05.mma operations run in issue order.
constexpr int BW_THREADS = 320;
constexpr int BW_ROWS = 256;  // row threads

// tensor-memory column of the A operand for K step k (16 elements) of a
// 64-wide bf16 operand written as two 16-column halves 32 columns apart
__device__ __forceinline__ uint32_t split_a_col(int k) { return (uint32_t)(8 * k + (k >= 2 ? 16 : 0)); }

template <bool F16>
__device__ __forceinline__ void store_out32(bf16* dst, const uint32_t (&w)[32], float scale) {
    uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; i++)
        o[i] = make_uint4(pack2<F16>(__uint_as_float(w[8 * i]) * scale, __uint_as_float(w[8 * i + 1]) * scale),
                          pack2<F16>(__uint_as_float(w[8 * i + 2]) * scale, __uint_as_float(w[8 * i + 3]) * scale),
                          pack2<F16>(__uint_as_float(w[8 * i + 4]) * scale, __uint_as_float(w[8 * i + 5]) * scale),
                          pack2<F16>(__uint_as_float(w[8 * i + 6]) * scale, __uint_as_float(w[8 * i + 7]) * scale));
}

// One arrival per warp: every lane has passed its own fences (the caller's
// tcgen05.fence / fence.proxy.async) before lane 0 arrives for the warp.
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// Named barrier for the 256 row threads only.
__device__ __forceinline__ void rows_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// The tile's column sums of one 32-column output half: each warp's 32 rows by
// warp_colsum32, then the four quarter warps of the half in quarter order
// (cs: [2 halves][4 quarters][32] floats of shared memory).  Reached by all
// 256 row threads; `v` holds zeros for rows that are not valid.
__device__ __forceinline__ void tile_colsum(float (&v)[32], float* cs, float* dst, int half, int quarter, int lane) {
    cs[(half * 4 + quarter) * 32 + lane] = warp_colsum32(v, lane);
    rows_sync();
    if (quarter == 0 && dst)
        dst[lane] = cs[(half * 4) * 32 + lane] + cs[(half * 4 + 1) * 32 + lane] + cs[(half * 4 + 2) * 32 + lane] +
                    cs[(half * 4 + 3) * 32 + lane];
    rows_sync();
}

// ------------------------------------------------------------------ dQ
// One CTA per 128 queries (2 CTAs per SM).  S = Q K_j^T and dP = dO V_j^T
// (Q and dO are A operands read from shared memory); the row threads form
// dS = P o (dP - D), P from the saved log-sum-exp, into one of two bf16
// buffers in tensor memory; dQ += dS K_j accumulates in tensor memory.
// D = rowsum(dO o O) is computed here and saved for the dK/dV kernel.
//
// A tcgen05.mma costs its issuing thread tens of cycles, about twice the
// tensor time of an N = 64 product, so the MMA thread is the critical
// resource: the dQ MMAs of block j - 1 are issued after S_j and dP_j, while
// the row threads work on block j, and dS is double-buffered so that block
// j's dS never overwrites the operand of block j - 1's dQ MMAs.
constexpr int Q_Q = 0;
constexpr int Q_O = Q_Q + T128;          // dO tile
constexpr int Q_KST = 3;                 // K stages: K_j is read by S_j and by dQ_j
constexpr int Q_K = Q_O + T128;
constexpr int Q_V = Q_K + Q_KST * T64;   // 2 stages: V_j is free once dP_j is done
constexpr int Q_DP = Q_V + 2 * T64;      // D partials [2 halves][128 rows]
constexpr int Q_CS = Q_DP + 2 * 128 * 4; // column sums [2 halves][4 quarters][32]
constexpr int Q_BAR = Q_CS + 2 * 4 * 32 * 4;
constexpr int Q_SMEM = Q_BAR + 256 + 1024;
constexpr uint32_t Q_TMEM = 256;         // S 0..63, dP 64..127, dS[2] 128..191, dQ 192..255
constexpr uint32_t Q_TS = 0, Q_TP = 64, Q_TDS = 128, Q_TACC = 192;

template <bool F16>
__global__ void __launch_bounds__(BW_THREADS, 2)
k_attn_bwd_dq_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap to, const bf16* __restrict__ y,
                 const float* __restrict__ lse, float* __restrict__ Dlt, bf16* __restrict__ dqkv,
                 float* __restrict__ bpart, int T, int C, int H, int nbh, int* flags, long long wl) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint64_t* bars = (uint64_t*)(sm + Q_BAR);
    uint64_t* qo_full = bars + 0;
    uint64_t* k_full = bars + 1;    // [3]
    uint64_t* k_empty = bars + 4;   // [3]
    uint64_t* v_full = bars + 7;    // [2]
    uint64_t* v_empty = bars + 9;   // [2]
    uint64_t* s_full = bars + 11;   // S_j, dP_j (and every earlier MMA) done
    uint64_t* ds_full = bars + 12;  // block j's S, dP read and its dS written
    uint64_t* acc_full = bars + 13;
    uint64_t* drain = bars + 14;    // MMAs issued before an abort are done
    uint32_t* tmem_holder = (uint32_t*)(bars + 15);
    volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

    const int bh = (int)(blockIdx.z * gridDim.x + blockIdx.x);
    if (bh >= nbh) return;
    const int nqt = gridDim.y;
    const int qt = nqt - 1 - (int)blockIdx.y;  // longest rows first within the band
    const int b = bh / H, h = bh % H;
    const int nkv = min(2 * qt + 2, (T + BN - 1) / BN);
    const int row0 = b * T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(qo_full, 1);
        for (int i = 0; i < Q_KST; i++) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(ds_full, BW_ROWS / 32);
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        init_done();
    }
    if (warp == 1) tmem_alloc(tmem_holder, Q_TMEM);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    pdl_enter();  // the set-up above overlaps the previous kernel's end; global memory only from here

    if (warp == 0) {
        if (lane == 0) {
            const int xq = h * D, xk = C + h * D, xv = 2 * C + h * D;
            mbar_expect_tx(qo_full, 2 * T128);
            tma_load_2d(smem_u32(sm + Q_Q), &tq, qo_full, xq, row0 + qt * BQ);
            tma_load_2d(smem_u32(sm + Q_O), &to, qo_full, h * D, row0 + qt * BQ);
            int issued_k = 0, issued_v = 0;
            bool ok = true;
            for (int j = 0; j < nkv; j++) {
                const int ks = j % Q_KST, kr = j / Q_KST;
                if (!mbar_wait(&k_empty[ks], (kr & 1) ^ 1, abort_flag, flags, 0x200 + 1, wl)) { ok = false; break; }
                mbar_expect_tx(&k_full[ks], T64);
                tma_load_2d(smem_u32(sm + Q_K + ks * T64), &tk, &k_full[ks], xk, row0 + j * BN);
                ++issued_k;
                const int vs = j & 1;
                if (!mbar_wait(&v_empty[vs], ((j >> 1) & 1) ^ 1, abort_flag, flags, 0x200 + 10, wl)) { ok = false; break; }
                mbar_expect_tx(&v_full[vs], T64);
                tma_load_2d(smem_u32(sm + Q_V + vs * T64), &tk, &v_full[vs], xv, row0 + j * BN);
                ++issued_v;
            }
            if (!ok) {  // let issued copies land before the CTA exits
                mbar_drain(qo_full, 0);
                for (int j = (issued_k > Q_KST ? issued_k - Q_KST : 0); j < issued_k; j++)
                    mbar_drain(&k_full[j % Q_KST], (j / Q_KST) & 1);
                for (int j = (issued_v > 2 ? issued_v - 2 : 0); j < issued_v; j++)
                    mbar_drain(&v_full[j & 1], (j >> 1) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID = idesc16<F16>(BQ, BN, false, false);
            constexpr uint32_t ID_Q = idesc16<F16>(BQ, D, false, true);
            const uint32_t sq = smem_u32(sm + Q_Q), so = smem_u32(sm + Q_O);
            bool ok = mbar_wait(qo_full, 0, abort_flag, flags, 0x200 + 2, wl);
            bool issued = false;
            // dQ += dS_j K_j: dS from tensor-memory buffer j & 1, K_j read MN-major
            auto issue_dq = [&](int j) {
                const uint32_t sk = smem_u32(sm + Q_K + (j % Q_KST) * T64);
                const uint32_t ta = tmem + Q_TDS + 32 * (j & 1);
#pragma unroll
                for (int k = 0; k < BN / 16; k++)
                    umma_bf16_ts(tmem + Q_TACC, ta + 8 * k, sdesc(sk + k * 2048, T64, 1024), ID_Q,
                                 (j > 0 || k > 0) ? 1u : 0u);
                umma_commit(&k_empty[j % Q_KST]);
            };
            for (int j = 0; j < nkv && ok; j++) {
                const int ks = j % Q_KST, vs = j & 1;
                if (!mbar_wait(&k_full[ks], (j / Q_KST) & 1, abort_flag, flags, 0x200 + 3, wl)) { ok = false; break; }
                if (!mbar_wait(&v_full[vs], (j >> 1) & 1, abort_flag, flags, 0x200 + 11, wl)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sk = smem_u32(sm + Q_K + ks * T64), sv = smem_u32(sm + Q_V + vs * T64);
                // S_j and dP_j: two independent chains, interleaved
#pragma unroll
                for (int k = 0; k < D / 16; k++) {
                    umma_bf16(tmem + Q_TS, sdesc(sq + 32 * k, 16, 1024), sdesc(sk + 32 * k, 16, 1024), ID, k > 0);
                    umma_bf16(tmem + Q_TP, sdesc(so + 32 * k, 16, 1024), sdesc(sv + 32 * k, 16, 1024), ID, k > 0);
                }
                issued = true;
                umma_commit(s_full);
                umma_commit(&v_empty[vs]);  // V_j is no longer needed
                if (j > 0) issue_dq(j - 1);  // overlaps the row threads' work on block j
                if (!mbar_wait(ds_full, j & 1, abort_flag, flags, 0x200 + 5, wl)) { ok = false; break; }
                tc_fence_after();
            }
            if (ok) {
                issue_dq(nkv - 1);
                umma_commit(acc_full);
            } else if (issued) {  // the MMAs already issued finish before tensor memory is freed
                umma_commit(drain);
                mbar_drain(drain, 0);
            }
        }
    } else {
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        const int q = qt * BQ + r;
        const bool qv = q < T;
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        const long long bhl = (long long)b * H + h;
        float* dpart = reinterpret_cast<float*>(sm + Q_DP);
        bool ok = mbar_wait_warp(qo_full, 0, abort_flag, flags, 0x200 + 6, wl);
        // This thread's half of D = rowsum(dO o O) (16-byte chunks 4 half ..
        // 4 half + 3 of the swizzled dO row); the two halves meet in shared memory.
        float Dq = 0.0f;
        if (ok) {
            const uint8_t* orow = sm + Q_O + r * 128;
            float part = 0.0f;
            if (qv) {
                const uint4* yr = reinterpret_cast<const uint4*>(y + (long long)(row0 + q) * C + h * D + 32 * half);
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const uint4 a = *reinterpret_cast<const uint4*>(orow + (((4 * half + c) ^ (r & 7)) << 4));
                    const uint4 bb = yr[c];
                    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
                    const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        part = fmaf(lo16<F16>(aw[i]), lo16<F16>(bw[i]), part);
                        part = fmaf(hi16<F16>(aw[i]), hi16<F16>(bw[i]), part);
                    }
                }
            }
            dpart[half * 128 + r] = part;
        }
        rows_sync();
        if (ok) {
            Dq = dpart[r] + dpart[128 + r];  // the two halves in a fixed order
            if (qv && half == 0) Dlt[bhl * T + q] = Dq;
        }
        const float Lq = qv ? lse[bhl * T + q] * LOG2E : 0.0f;
        for (int j = 0; j < nkv && ok; j++) {
            if (!mbar_wait_warp(s_full, j & 1, abort_flag, flags, 0x200 + 7, wl)) { ok = false; break; }
            tc_fence_after();
            const bool diag = (j >= 2 * qt);
            const int kq = q - j * BN - 32 * half;  // on the diagonal, this half's columns > kq are masked
            uint32_t sw[32], pw[32];
            tmem_ld32x2(tl + Q_TS + 32 * half, sw, tl + Q_TP + 32 * half, pw);
            // dS = P o (dP - D), packed bf16
            // (packed fp32x2: the same roundings as the scalar fma, sub and mul)
            uint32_t pk[16];
            const float2 sl2 = make_float2(SL2, SL2), nl = make_float2(-Lq, -Lq), nd = make_float2(-Dq, -Dq);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const float2 x = __ffma2_rn(make_float2(__uint_as_float(sw[e]), __uint_as_float(sw[e + 1])), sl2, nl);
                const float2 dd = __fadd2_rn(make_float2(__uint_as_float(pw[e]), __uint_as_float(pw[e + 1])), nd);
                float2 d = __fmul2_rn(make_float2(ex2(x.x), ex2(x.y)), dd);
                if (diag) {
                    if (e > kq) d.x = 0.0f;
                    if (e + 1 > kq) d.y = 0.0f;
                }
                pk[e >> 1] = pack2<F16>(qv ? d.x : 0.0f, qv ? d.y : 0.0f);
            }
            tmem_st16(tl + Q_TDS + 32 * (j & 1) + 16 * half, pk);
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(ds_full, lane);
        }
        float cv[32];
#pragma unroll
        for (int d = 0; d < 32; d++) cv[d] = 0.0f;
        if (ok && mbar_wait_warp(acc_full, 0, abort_flag, flags, 0x200 + 9, wl)) {
            tc_fence_after();
            uint32_t w[32];
            tmem_ld32(tl + Q_TACC + 32 * half, w);
            if (qv) {
                store_out32<F16>(dqkv + (long long)(row0 + q) * 3 * C + h * D + 32 * half, w, 0.125f);
#pragma unroll
                for (int d = 0; d < 32; d++) cv[d] = __uint_as_float(w[d]) * 0.125f;
            }
        }
        if (bpart)  // the qkv bias gradient's partial: this tile's column sums of dQ
            tile_colsum(cv, reinterpret_cast<float*>(sm + Q_CS),
                        bpart + ((long long)b * nqt + qt) * 3 * C + h * D + 32 * half, half, quarter, lane);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, Q_TMEM);
}

// ------------------------------------------------------------------ dK, dV
// One CTA per 128 keys (2 CTAs per SM), streaming the query blocks at and
// after the diagonal: S^T = K Q_j^T and dP^T = V dO_j^T (K and V as A operands
// from shared memory), then P^T and dS^T into tensor memory, and
// dV += P^T dO_j, dK += dS^T Q_j (Q_j and dO_j read again as MN-major
// operands) accumulate in tensor memory.
constexpr int K_K = 0;
constexpr int K_V = K_K + T128;
constexpr int K_ST = 3;                  // Q / dO block stages
constexpr int K_Q = K_V + T128;
constexpr int K_O = K_Q + K_ST * T64;
constexpr int K_LD = K_O + K_ST * T64;   // per row warp: log-sum-exp and D of its 32 queries
constexpr int K_CS = K_LD + 8 * 64 * 4;  // column sums [2 halves][4 quarters][32]
constexpr int K_BAR = K_CS + 2 * 4 * 32 * 4;
constexpr int K_SMEM = K_BAR + 256 + 1024;
constexpr uint32_t K_TMEM = 256;         // S^T 0..63, dP^T 64..127, dV 128..191, dK 192..255
constexpr uint32_t K_TS = 0, K_TP = 64, K_TV = 128, K_TK = 192;

template <bool F16>
__global__ void __launch_bounds__(BW_THREADS, 2)
k_attn_bwd_dkdv_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap to, const float* __restrict__ lse,
                   const float* __restrict__ Dlt, bf16* __restrict__ dqkv, float* __restrict__ bpart, int T,
                   int C, int H, int nbh, int* flags, long long wl) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint64_t* bars = (uint64_t*)(sm + K_BAR);
    uint64_t* kv_full = bars + 0;
    uint64_t* qo_full = bars + 1;   // [3]
    uint64_t* qo_empty = bars + 4;  // [3]
    uint64_t* st_full = bars + 7;   // S^T_i, dP^T_i (and every earlier MMA) done
    uint64_t* ps_full = bars + 8;   // P^T_i, dS^T_i written to tensor memory
    uint64_t* acc_full = bars + 9;
    uint64_t* drain = bars + 10;
    uint32_t* tmem_holder = (uint32_t*)(bars + 11);
    volatile int* abort_flag = (volatile int*)(tmem_holder + 1);

    const int bh = (int)(blockIdx.z * gridDim.x + blockIdx.x);
    if (bh >= nbh) return;
    const int kt = (int)blockIdx.y;  // key tile; low tiles see the most query blocks
    const int b = bh / H, h = bh % H;
    const int row0 = b * T;
    const int nqb = (T + BN - 1) / BN;
    const int j0 = 2 * kt;
    const int nq = nqb - j0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int i = 0; i < K_ST; i++) {
            mbar_init(&qo_full[i], 1);
            mbar_init(&qo_empty[i], 1);
        }
        mbar_init(st_full, 1);
        mbar_init(ps_full, BW_ROWS / 32);
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        init_done();
    }
    if (warp == 1) tmem_alloc(tmem_holder, K_TMEM);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    pdl_enter();  // the set-up above overlaps the previous kernel's end; global memory only from here

    if (warp == 0) {
        if (lane == 0) {
            const int xq = h * D, xk = C + h * D, xv = 2 * C + h * D;
            mbar_expect_tx(kv_full, 2 * T128);
            tma_load_2d(smem_u32(sm + K_K), &tq, kv_full, xk, row0 + kt * BQ);
            tma_load_2d(smem_u32(sm + K_V), &tq, kv_full, xv, row0 + kt * BQ);
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < nq; i++) {
                const int st = i % K_ST, j = j0 + i;
                if (!mbar_wait(&qo_empty[st], ((i / K_ST) & 1) ^ 1, abort_flag, flags, 0x300 + 1, wl)) { ok = false; break; }
                mbar_expect_tx(&qo_full[st], 2 * T64);
                tma_load_2d(smem_u32(sm + K_Q + st * T64), &tk, &qo_full[st], xq, row0 + j * BN);
                tma_load_2d(smem_u32(sm + K_O + st * T64), &to, &qo_full[st], h * D, row0 + j * BN);
                ++issued;
            }
            if (!ok) {
                mbar_drain(kv_full, 0);
                for (int i = (issued > K_ST ? issued - K_ST : 0); i < issued; i++)
                    mbar_drain(&qo_full[i % K_ST], (i / K_ST) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID = idesc16<F16>(BQ, BN, false, false);
            constexpr uint32_t ID_A = idesc16<F16>(BQ, D, false, true);
            const uint32_t sk = smem_u32(sm + K_K), sv = smem_u32(sm + K_V);
            bool ok = mbar_wait(kv_full, 0, abort_flag, flags, 0x300 + 2, wl);
            bool issued = false;
            for (int i = 0; i < nq && ok; i++) {
                const int st = i % K_ST;
                if (!mbar_wait(&qo_full[st], (i / K_ST) & 1, abort_flag, flags, 0x300 + 3, wl)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sq = smem_u32(sm + K_Q + st * T64), so = smem_u32(sm + K_O + st * T64);
                // S^T_i and dP^T_i (two independent chains, interleaved); they
                // overwrite P^T_{i-1} and dS^T_{i-1}, read by MMAs issued before
#pragma unroll
                for (int k = 0; k < D / 16; k++) {
                    umma_bf16(tmem + K_TS, sdesc(sk + 32 * k, 16, 1024), sdesc(sq + 32 * k, 16, 1024), ID, k > 0);
                    umma_bf16(tmem + K_TP, sdesc(sv + 32 * k, 16, 1024), sdesc(so + 32 * k, 16, 1024), ID, k > 0);
                }
                issued = true;
                umma_commit(st_full);
                if (!mbar_wait(ps_full, i & 1, abort_flag, flags, 0x300 + 5, wl)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BN / 16; k++) {
                    const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
                    umma_bf16_ts(tmem + K_TV, tmem + K_TS + split_a_col(k), sdesc(so + k * 2048, T64, 1024), ID_A, acc);
                    umma_bf16_ts(tmem + K_TK, tmem + K_TP + split_a_col(k), sdesc(sq + k * 2048, T64, 1024), ID_A, acc);
                }
                umma_commit(&qo_empty[st]);
            }
            if (ok) umma_commit(acc_full);
            else if (issued) {
                umma_commit(drain);
                mbar_drain(drain, 0);
            }
        }
    } else {
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        const int key = kt * BQ + r;
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        const long long bhl = (long long)b * H + h;
        const float* lrow = lse + bhl * T;
        const float* drow = Dlt + bhl * T;
        bool ok = true;
        // The log-sum-exp (base 2) and D of this warp's 32 queries of block i
        // are fetched one block ahead (lane l: query 64 (j0 + i) + 32 half + l),
        // then placed in this warp's slice of shared memory, from which every
        // lane reads them as broadcasts.
        float* sl = reinterpret_cast<float*>(sm + K_LD) + (warp - 2) * 64;  // [32 L | 32 D]
        float Ln, Dn;
        auto fetch = [&](int i) {
            const int qq = (j0 + i) * BN + 32 * half + lane;
            Ln = qq < T ? __ldg(lrow + qq) * LOG2E : INFINITY;
            Dn = qq < T ? __ldg(drow + qq) : 0.0f;
        };
        fetch(0);
        for (int i = 0; i < nq; i++) {
            const int j = j0 + i;
            __syncwarp();  // the previous block's reads of the slice are done
            sl[lane] = -Ln;  // negated: the packed fma and add below take them as addends
            sl[32 + lane] = -Dn;
            __syncwarp();
            if (i + 1 < nq) fetch(i + 1);
            if (!mbar_wait_warp(st_full, i & 1, abort_flag, flags, 0x300 + 6, wl)) { ok = false; break; }
            tc_fence_after();
            const bool diag = (i < 2);  // query blocks that overlap this key tile
            const int q0 = j * BN + 32 * half;
            uint32_t sw[32], dw[32];
            tmem_ld32x2(tl + K_TS + 32 * half, sw, tl + K_TP + 32 * half, dw);
            uint32_t pk[16], dk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                // -L and -D from the slice; packed fp32x2 with the scalar
                // operations' roundings
                const float2 L2 = *reinterpret_cast<const float2*>(sl + e);
                const float2 D2 = *reinterpret_cast<const float2*>(sl + 32 + e);
                const float2 x = __ffma2_rn(make_float2(__uint_as_float(sw[e]), __uint_as_float(sw[e + 1])),
                                            make_float2(SL2, SL2), L2);
                float2 p = make_float2(ex2(x.x), ex2(x.y));
                if (diag) {
                    if (q0 + e < key) p.x = 0.0f;
                    if (q0 + e + 1 < key) p.y = 0.0f;
                }
                pk[e >> 1] = pack2<F16>(p.x, p.y);
                const float2 d =
                    __fmul2_rn(p, __fadd2_rn(make_float2(__uint_as_float(dw[e]), __uint_as_float(dw[e + 1])), D2));
                dk[e >> 1] = pack2<F16>(d.x, d.y);
            }
            tmem_st16(tl + K_TS + 32 * half, pk);
            tmem_st16(tl + K_TP + 32 * half, dk);
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(ps_full, lane);
        }
        const bool got = ok && mbar_wait_warp(acc_full, 0, abort_flag, flags, 0x300 + 8, wl);
        if (got) tc_fence_after();
        bf16* base = dqkv + (long long)(row0 + key) * 3 * C + h * D + 32 * half;
        // the qkv bias gradient's partials: this tile's column sums of dV, then dK
        float* brow = bpart ? bpart + ((long long)b * gridDim.y + kt) * 3 * C + h * D + 32 * half : nullptr;
#pragma unroll 1
        for (int which = 0; which < 2; which++) {  // 0: dV, 1: dK (times 1/sqrt(64))
            const float scale = which ? 0.125f : 1.0f;
            float v[32];
#pragma unroll
            for (int d = 0; d < 32; d++) v[d] = 0.0f;
            if (got) {
                uint32_t w[32];
                tmem_ld32(tl + (which ? K_TK : K_TV) + 32 * half, w);
                if (key < T) {
                    store_out32<F16>(base + (which ? C : 2 * C), w, scale);
#pragma unroll
                    for (int d = 0; d < 32; d++) v[d] = __uint_as_float(w[d]) * scale;
                }
            }
            if (brow) tile_colsum(v, reinterpret_cast<float*>(sm + K_CS), brow + (which ? C : 2 * C), half, quarter, lane);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, K_TMEM);
}

}  // namespace fa5

// bf16 or IEEE-half storage (the caller says which through Launch::f16)
bool attention_tc_eligible(bool bf16, int C, int H) {
    return bf16 && H > 0 && C % H == 0 && C / H == fa5::D && C % 8 == 0;
}

template <bool F16>
static bool attn_set_smem() {
    static PerDevice done;
    return done.once([] {
        return cudaFuncSetAttribute(fa5::k_attn_fwd_tc<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    fa5::F_SMEM) == cudaSuccess &&
               cudaFuncSetAttribute(fa5::k_attn_bwd_dq_tc<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    fa5::Q_SMEM) == cudaSuccess &&
               cudaFuncSetAttribute(fa5::k_attn_bwd_dkdv_tc<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    fa5::K_SMEM) == cudaSuccess;
    });
}

static dim3 attn_grid(int bh, int tiles) {
    const int band = bh < fa5::BAND ? bh : fa5::BAND;
    return dim3((unsigned)band, (unsigned)tiles, (unsigned)((bh + band - 1) / band));
}

template <bool F16>
static bool attn_fwd_tc(const Launch& L, const void* qkv, void* y, float* lse, int B, int T, int C, int H) {
    CUtensorMap tq, tk;
    if (!tc::make_tmap_bf16(&tq, qkv, 3LL * C, (long long)B * T, 3LL * C, fa5::D, fa5::BQ)) return false;
    if (!tc::make_tmap_bf16(&tk, qkv, 3LL * C, (long long)B * T, 3LL * C, fa5::D, fa5::BN)) return false;
    if (!attn_set_smem<F16>()) return false;
    const dim3 grid = attn_grid(B * H, (T + fa5::BQ - 1) / fa5::BQ);
    L.count();
    launch_k(L, fa5::k_attn_fwd_tc<F16>, dim3(grid), dim3(fa5::THREADS), fa5::F_SMEM, tq, tk, (fa5::bf16*)y, lse, T, C, H,
                                                                          B * H, L.flags, L.wait_cycles);
    return true;
}

template <bool F16>
static bool attn_bwd_tc(const Launch& L, const void* qkv, const void* y, const float* lse, const void* dy,
                        void* dqkv, int B, int T, int C, int H, float* Dlt, float* bpart) {
    // the maps only move 16-bit elements (no conversion), for bf16 and half alike
    CUtensorMap tq, tk, to128, to64;
    if (!tc::make_tmap_bf16(&tq, qkv, 3LL * C, (long long)B * T, 3LL * C, fa5::D, fa5::BQ)) return false;
    if (!tc::make_tmap_bf16(&tk, qkv, 3LL * C, (long long)B * T, 3LL * C, fa5::D, fa5::BN)) return false;
    if (!tc::make_tmap_bf16(&to128, dy, (long long)C, (long long)B * T, (long long)C, fa5::D, fa5::BQ))
        return false;
    if (!tc::make_tmap_bf16(&to64, dy, (long long)C, (long long)B * T, (long long)C, fa5::D, fa5::BN))
        return false;
    if (!attn_set_smem<F16>()) return false;
    const dim3 grid = attn_grid(B * H, (T + fa5::BQ - 1) / fa5::BQ);
    L.count();
    launch_k(L, fa5::k_attn_bwd_dq_tc<F16>, dim3(grid), dim3(fa5::BW_THREADS), fa5::Q_SMEM, 
        tq, tk, to128, (const fa5::bf16*)y, lse, Dlt, (fa5::bf16*)dqkv, bpart, T, C, H, B * H, L.flags,
        L.wait_cycles);
    L.count();
    launch_k(L, fa5::k_attn_bwd_dkdv_tc<F16>, dim3(grid), dim3(fa5::BW_THREADS), fa5::K_SMEM, 
        tq, tk, to64, lse, Dlt, (fa5::bf16*)dqkv, bpart, T, C, H, B * H, L.flags, L.wait_cycles);
    return true;
}

bool launch_attention_fwd_tc(const Launch& L, const void* qkv, void* y, float* lse, int B, int T,
                             int C, int H) {
    if (L.dry) return true;
    return L.f16 ? attn_fwd_tc<true>(L, qkv, y, lse, B, T, C, H) : attn_fwd_tc<false>(L, qkv, y, lse, B, T, C, H);
}

bool launch_attention_bwd_tc(const Launch& L, const void* qkv, const void* y, const float* lse,
                             const void* dy, void* dqkv, int B, int T, int C, int H, float* Dlt,
                             float* bpart) {
    if (L.dry) return true;
    return L.f16 ? attn_bwd_tc<true>(L, qkv, y, lse, dy, dqkv, B, T, C, H, Dlt, bpart)
                 : attn_bwd_tc<false>(L, qkv, y, lse, dy, dqkv, B, T, C, H, Dlt, bpart);
}

}  // namespace tt

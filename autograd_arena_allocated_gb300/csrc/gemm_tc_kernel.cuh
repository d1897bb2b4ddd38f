// gemm_tc_kernel.cuh -- the tcgen05 GEMM kernel template and its launch, shared
// by gemm_tc.cu (bf16 operands) and gemm_tc_f16.cu (IEEE-half operands).
// The design is described at the top of gemm_tc.cu.
#pragma once
#include "tt_internal.h"
#include "tc_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace tt {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 bf16 = 128 bytes = one 128B-swizzle row
constexpr int UMMA_K = 16;
constexpr int THREADS = 320;
constexpr int EPI_WARPS = 8;
constexpr int MN_BOX = 64;                  // MN extent of one MN-major TMA box
constexpr int MN_BOX_BYTES = MN_BOX * BK * 2;  // 8 KB: 64 k-rows x 128 bytes

template <int BN, bool PAIR = false>
struct Cfg {
    static constexpr int STAGES = (PAIR || BN < 192) ? 6 : 4;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;  // this CTA's part of the B tile
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = (2 * BN <= 256) ? 256 : 512;  // two accumulators, power of two
    static constexpr int BAR_BYTES = 1024;                 // barriers, padded to keep staging aligned
    static constexpr int STAGING_BYTES = EPI_WARPS * 2 * 2048;  // 2 x [32 rows x 64 B] per epilogue warp
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + STAGING_BYTES + 1024;
};

struct Params {
    int M, N, K;
    int m_tiles, n_tiles, tiles;
    int n_fast;  // tile order: n-tiles fastest (B stays in L2, A streams once) or m-tiles fastest
    int kb_total, kb_per_split, splits, units;
    void* D;
    long long ldd;
    int d_f32, n_store, epi, accumulate;
    const __nv_bfloat16* bias;
    const __nv_bfloat16* residual;
    __nv_bfloat16* aux;
    float* ws;  // split-K partials [splits][M][N]
    int* flags;
    int tma_store;  // bf16 outputs leave through shared memory and TMA stores
    int ext_tma;    // the extra epilogue operand (GELU' input or residual) arrives by TMA loads
    int cl;         // pair form: CTA pairs take M tiles 2i, 2i + 1
    int pair_units; // pair form: ceil(m_tiles / 2) * n_tiles * splits
    float* colsum;  // ext_tma path: column sums of each 32-row slice of the result, [M/32][N]
    long long wait_limit;  // bounded-wait limit (clock64 cycles)
};

// tanh by the hardware approximation (max relative error about 2^-11, far
// below the bf16 rounding of the epilogue's outputs)
__device__ __forceinline__ float tanh_hw(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The epilogue's elementwise work on pairs of values, in the packed fp32x2
// instructions of sm_100 and later (one instruction for both lanes, each
// lane rounded as the scalar instruction would): half the issue slots of the
// scalar form, which is what bounds the epilogue warps.
__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }

// GELU, tanh form: 0.5 u (1 + tanh(w)), w = k u (1 + a u^2)
__device__ __forceinline__ float2 gelu_tanh2(float2 u) {
    const float2 s = __fmul2_rn(u, u);
    const float2 w = __fmul2_rn(__fmul2_rn(f2(0.7978845608028654f), u), __ffma2_rn(f2(0.044715f), s, f2(1.0f)));
    const float2 t = make_float2(tanh_hw(w.x), tanh_hw(w.y));
    const float2 hu = __fmul2_rn(f2(0.5f), u);
    return __ffma2_rn(hu, t, hu);
}
// its derivative: 0.5 (1 + tau + k u (1 + 3 a u^2) (1 - tau^2)), tau = tanh(w);
// written with the signs folded into constants, (-r)(tau^2 - 1) = r (1 - tau^2)
__device__ __forceinline__ float2 dgelu_tanh2(float2 u) {
    const float2 s = __fmul2_rn(u, u);
    const float2 ku = __fmul2_rn(f2(0.7978845608028654f), u);
    const float2 w = __fmul2_rn(ku, __ffma2_rn(f2(0.044715f), s, f2(1.0f)));
    const float2 t = make_float2(tanh_hw(w.x), tanh_hw(w.y));
    const float2 nr = __fmul2_rn(ku, __ffma2_rn(f2(-3.0f * 0.044715f), s, f2(-1.0f)));
    const float2 y = __ffma2_rn(nr, __ffma2_rn(t, t, f2(-1.0f)), t);
    return __ffma2_rn(f2(0.5f), y, f2(0.5f));
}
__device__ __forceinline__ void add32(float* v, const float* w) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float2 r = __fadd2_rn(make_float2(v[j], v[j + 1]), make_float2(w[j], w[j + 1]));
        v[j] = r.x;
        v[j + 1] = r.y;
    }
}
__device__ __forceinline__ void gelu32(float* v) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float2 r = gelu_tanh2(make_float2(v[j], v[j + 1]));
        v[j] = r.x;
        v[j + 1] = r.y;
    }
}
// v *= gelu'(u)
__device__ __forceinline__ void mul_dgelu32(float* v, const float* u) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float2 r = __fmul2_rn(make_float2(v[j], v[j + 1]), dgelu_tanh2(make_float2(u[j], u[j + 1])));
        v[j] = r.x;
        v[j + 1] = r.y;
    }
}

// One warp's 32 x 32 bf16 staging tile (row = lane, 64 bytes per row) in the
// layout of a TMA SWIZZLE_64B box: the 16-byte chunk c of row r sits at
// c ^ ((r >> 1) & 3).  Row writes from the 32 lanes are bank-conflict free.
template <bool F16>
__device__ __forceinline__ void stage_row32(uint8_t* buf, int r, const float* v) {
    uint8_t* rowp = buf + r * 64;
#pragma unroll
    for (int c = 0; c < 4; c++) {
        uint4 w;
        w.x = pack2<F16>(v[8 * c + 0], v[8 * c + 1]);
        w.y = pack2<F16>(v[8 * c + 2], v[8 * c + 3]);
        w.z = pack2<F16>(v[8 * c + 4], v[8 * c + 5]);
        w.w = pack2<F16>(v[8 * c + 6], v[8 * c + 7]);
        *reinterpret_cast<uint4*>(rowp + ((c ^ ((r >> 1) & 3)) << 4)) = w;
    }
}

// Row r of a [32 rows x 32 bf16] buffer in the same 64-byte-swizzled layout
// (as a TMA load with SWIZZLE_64B leaves it), as floats.
template <bool F16>
__device__ __forceinline__ void load_row32(const uint8_t* buf, int r, float* v) {
    const uint8_t* rowp = buf + r * 64;
#pragma unroll
    for (int c = 0; c < 4; c++) {
        const uint4 w = *reinterpret_cast<const uint4*>(rowp + ((c ^ ((r >> 1) & 3)) << 4));
        v[8 * c + 0] = lo16<F16>(w.x); v[8 * c + 1] = hi16<F16>(w.x);
        v[8 * c + 2] = lo16<F16>(w.y); v[8 * c + 3] = hi16<F16>(w.y);
        v[8 * c + 4] = lo16<F16>(w.z); v[8 * c + 5] = hi16<F16>(w.z);
        v[8 * c + 6] = lo16<F16>(w.w); v[8 * c + 7] = hi16<F16>(w.w);
    }
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     (uint64_t)map),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Load 32 consecutive 16-bit values (64 bytes) as floats; vector path when aligned.
template <bool F16>
__device__ __forceinline__ void load32_16(const void* p, int valid, bool vec, float* v) {
    if (vec && valid >= 32) {
        const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            uint4 w = q[i];
            v[8 * i + 0] = lo16<F16>(w.x); v[8 * i + 1] = hi16<F16>(w.x);
            v[8 * i + 2] = lo16<F16>(w.y); v[8 * i + 3] = hi16<F16>(w.y);
            v[8 * i + 4] = lo16<F16>(w.z); v[8 * i + 5] = hi16<F16>(w.z);
            v[8 * i + 6] = lo16<F16>(w.w); v[8 * i + 7] = hi16<F16>(w.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; j++) v[j] = (j < valid) ? ld16<F16>(p, j) : 0.0f;
    }
}

template <bool F16>
__device__ __forceinline__ void store32_16(void* p, int valid, bool vec, const float* v) {
    if (vec && valid >= 32) {
        uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            uint4 w;
            w.x = pack2<F16>(v[8 * i + 0], v[8 * i + 1]);
            w.y = pack2<F16>(v[8 * i + 2], v[8 * i + 3]);
            w.z = pack2<F16>(v[8 * i + 4], v[8 * i + 5]);
            w.w = pack2<F16>(v[8 * i + 6], v[8 * i + 7]);
            q[i] = w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; j++)
            if (j < valid) st16<F16>(p, j, v[j]);
    }
}

__device__ __forceinline__ void store32_f32(float* p, int valid, bool vec, const float* v) {
    if (vec && valid >= 32) {
        float4* q = reinterpret_cast<float4*>(p);
#pragma unroll
        for (int i = 0; i < 8; i++) q[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
#pragma unroll
        for (int j = 0; j < 32; j++)
            if (j < valid) p[j] = v[j];
    }
}

__device__ __forceinline__ int tile_m(const Params& p, int t) { return p.n_fast ? t / p.n_tiles : t % p.m_tiles; }
__device__ __forceinline__ int tile_n(const Params& p, int t) { return p.n_fast ? t % p.n_tiles : t / p.m_tiles; }

// The units (tile, split) this CTA takes: it = first, first + step, ... < count.
// In the pair form a unit is a pair of M tiles and the CTA of rank r takes M
// tile 2 * pair + r; with an odd number of M tiles the last pair's second
// tile lies wholly past M (its loads read zeros, its rows are not written;
// only the weight-gradient form, whose output is written row by row, pairs
// an odd count).
struct UnitIter {
    int first, step, count, rank;
};
__device__ __forceinline__ UnitIter unit_iter(const Params& p) {
    if (p.cl) return {(int)blockIdx.x >> 1, (int)gridDim.x >> 1, p.pair_units, (int)blockIdx.x & 1};
    return {(int)blockIdx.x, (int)gridDim.x, p.units, 0};
}
// unit it -> first row m0, first column n0 and split
__device__ __forceinline__ void unit_mn(const Params& p, int it, int rank, int bn, int* m0, int* n0, int* split) {
    const int t = it / p.splits;
    *split = it - t * p.splits;
    int m, n;
    if (!p.cl) {
        m = tile_m(p, t);
        n = tile_n(p, t);
    } else {
        const int mpt = (p.m_tiles + 1) >> 1;
        const int mp = p.n_fast ? t / p.n_tiles : t % mpt;
        n = p.n_fast ? t % p.n_tiles : t / mpt;
        m = 2 * mp + rank;
    }
    *m0 = m * BM;
    *n0 = n * bn;
}

// the shared::cluster address of the same variable in the leader CTA (rank 0)
__device__ __forceinline__ uint32_t leader_addr(const void* p) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(0u));
    return r;
}
// TMA load into this CTA's shared memory, completing on an mbarrier of
// either CTA of the pair (bar: shared::cluster address)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrives on the barrier at this offset in both CTAs of the pair once the
// leader's MMAs issued so far have finished
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)3)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ the kernel
template <int BN, bool A_MN, bool B_MN, bool PAIR, bool F16>
__global__ void __launch_bounds__(THREADS, 1)
k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
          const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmX,
          const Params p) {
    using CF = Cfg<BN, PAIR>;
    constexpr int S = CF::STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzle atoms
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* tiles = smem;
    uint64_t* full = (uint64_t*)(smem + S * CF::STAGE_BYTES);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;   // [2]
    uint64_t* tempty = tfull + 2;  // [2]
    uint32_t* tmem_base_holder = (uint32_t*)(tempty + 2);
    volatile int* abort_flag = (volatile int*)(tmem_base_holder + 1);
    // two per epilogue warp: the extra operand's tile has landed in staging buffer 0 / 1
    uint64_t* ebar = (uint64_t*)(smem + S * CF::STAGE_BYTES + 512);
    uint64_t* drain = ebar + 2 * EPI_WARPS;  // MMAs issued before an abort are done

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(&tfull[a], 1);
            // pair: both CTAs' epilogues release the leader's accumulator
            mbar_init(&tempty[a], (PAIR ? 2 : 1) * EPI_WARPS * 32);
        }
        for (int e = 0; e < 2 * EPI_WARPS; e++) mbar_init(&ebar[e], 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
        if (p.tma_store) {
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmD) : "memory");
            if (p.epi == EPI_GELU || p.ext_tma) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmX) : "memory");
        }
    }
    if (warp == 1) {
        if (PAIR) {  // one warp of each CTA of the pair, collectively
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_base_holder)),
                         "r"((uint32_t)CF::TMEM_COLS));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_base_holder)),
                         "r"((uint32_t)CF::TMEM_COLS));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_base_holder;
    if (PAIR) cluster_sync_all();  // the peer's barriers exist before any copy or commit reaches them
    // everything above touches only this CTA's (and its peer's) shared and
    // tensor memory: it overlaps the previous kernel's end under a dependent
    // launch; global memory is read and written only after this wait
    pdl_enter();
    const UnitIter U = unit_iter(p);
    const bool leader = U.rank == 0;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int it = U.first; it < U.count && ok; it += U.step) {
                int split, m0, n0;
                unit_mn(p, it, U.rank, BN, &m0, &n0, &split);
                const int kb0 = split * p.kb_per_split;
                const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.flags, 0x400 + 1, p.wait_limit)) { ok = false; break; }
                    const uint32_t sa = smem_u32(tiles + stage * CF::STAGE_BYTES);
                    const uint32_t sb = sa + CF::A_BYTES;
                    const int k0 = kb * BK;
                    if (PAIR) {
                        // own A tile and own half of B; both CTAs' bytes land on the leader's barrier
                        if (leader) mbar_expect_tx(&full[stage], 2 * CF::STAGE_BYTES);
                        const uint32_t fb = leader_addr(&full[stage]);
                        if (!A_MN) {
                            tma_load_2d_pair(sa, &tmA, fb, k0, m0);
                        } else {
#pragma unroll
                            for (int j = 0; j < BM / MN_BOX; j++)
                                tma_load_2d_pair(sa + j * MN_BOX_BYTES, &tmA, fb, m0 + j * MN_BOX, k0);
                        }
                        if (!B_MN) {
                            tma_load_2d_pair(sb, &tmB, fb, k0, n0 + U.rank * (BN / 2));
                        } else {
                            constexpr int HB = BN / MN_BOX / 2;
#pragma unroll
                            for (int j = 0; j < HB; j++)
                                tma_load_2d_pair(sb + j * MN_BOX_BYTES, &tmB, fb, n0 + (U.rank * HB + j) * MN_BOX, k0);
                        }
                        ++issued;
                        if (++stage == S) { stage = 0; phase ^= 1; }
                        continue;
                    }
                    mbar_expect_tx(&full[stage], CF::STAGE_BYTES);
                    if (!A_MN) {
                        tma_load_2d(sa, &tmA, &full[stage], k0, m0);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / MN_BOX; j++)
                            tma_load_2d(sa + j * MN_BOX_BYTES, &tmA, &full[stage], m0 + j * MN_BOX, k0);
                    }
                    if (!B_MN) {
                        tma_load_2d(sb, &tmB, &full[stage], k0, n0);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / MN_BOX; j++)
                            tma_load_2d(sb + j * MN_BOX_BYTES, &tmB, &full[stage], n0 + j * MN_BOX, k0);
                    }
                    ++issued;
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
            if (ok && PAIR) {
                // the leader's releases of the last stages have arrived before
                // this CTA's barriers go away
                for (int i = 0; i < S && ok; i++) {
                    ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.flags, 0x400 + 7, p.wait_limit);
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && !PAIR) {
                // let the copies already issued land before the CTA exits (in
                // the pair form they complete on the leader's barriers, which
                // this CTA cannot watch; the closing cluster barrier waits)
                long long back = issued < S ? issued : S;
                int st = stage;
                uint32_t ph = phase;
                for (long long i = 0; i < back; i++) {
                    if (st == 0) { st = S - 1; ph ^= 1; } else { --st; }
                    const long long t0 = clock64();
                    while (!mbar_try_wait(&full[st], ph) && clock64() - t0 < WAIT_CYCLES) {}
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && leader) {  // pair form: the leader issues for both CTAs
            constexpr uint32_t IDESC = idesc16<F16>(PAIR ? 2 * BM : BM, BN, A_MN, B_MN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int it = U.first; it < U.count && ok; it += U.step) {
                int split, m0_, n0_;
                unit_mn(p, it, U.rank, BN, &m0_, &n0_, &split);
                const int kb0 = split * p.kb_per_split;
                const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, p.flags, 0x400 + 2, p.wait_limit)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.flags, 0x400 + 3, p.wait_limit)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(tiles + stage * CF::STAGE_BYTES);
                    const uint32_t sb = sa + CF::A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; k++) {
                        uint64_t ad, bd;
                        if (!A_MN) ad = sdesc(sa + k * (UMMA_K * 2), 16, 1024);
                        else ad = sdesc(sa + k * (UMMA_K / 8) * 1024, MN_BOX_BYTES, 1024);
                        if (!B_MN) bd = sdesc(sb + k * (UMMA_K * 2), 16, 1024);
                        else bd = sdesc(sb + k * (UMMA_K / 8) * 1024, MN_BOX_BYTES, 1024);
                        if (PAIR) umma_bf16_pair(d_tmem, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                        else umma_bf16(d_tmem, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    if (PAIR) umma_commit_pair(&empty[stage]);  // both CTAs' slots free once these MMAs finish
                    else umma_commit(&empty[stage]);
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                if (PAIR) umma_commit_pair(&tfull[acc]);  // accumulator complete, in both CTAs
                else umma_commit(&tfull[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            if (!ok) {  // the MMAs already issued finish before tensor memory is freed
                if (PAIR) umma_commit_pair(drain);
                else umma_commit(drain);
                mbar_drain(drain, 0);
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        constexpr int CHUNKS = BN / 32 / 2;  // 32-column chunks per half
        int acc = 0;
        uint32_t acc_phase = 0;
        const bool d_vec = p.d_f32 ? ((p.ldd & 3) == 0) : ((p.ldd & 7) == 0);
        // vector accesses also need 16-byte aligned base pointers
        const bool aux_vec = d_vec && ((uintptr_t)p.aux & 15) == 0;
        const bool res_vec = d_vec && ((uintptr_t)p.residual & 15) == 0;
        const bool out_vec = d_vec && ((uintptr_t)p.D & 15) == 0;
        uint8_t* stg = smem + S * CF::STAGE_BYTES + CF::BAR_BYTES + (warp - 2) * 2 * 2048;
        int sbuf = 0;
        if (p.ext_tma) {
            // bf16 result through shared memory and TMA stores, with the extra
            // operand (GELU' input, or residual) of each 32 x 32 chunk TMA-loaded
            // into the warp's staging buffer one chunk ahead.  A thread reads its
            // row, writes its result row over it, and lane 0 stores the buffer.
            // Every chunk is valid here (n_store is a multiple of BN).
            const int ew = warp - 2;
            uint64_t* eb = ebar + 2 * ew;
            uint32_t eph = 0u, pending = 0u;  // bit b: phase of ebar b / a load into buffer b in flight
            const int y_off = quarter * 32;
            auto issue_ext = [&](int b, int n, int y) {
                if (lane == 0) {
                    mbar_expect_tx(&eb[b], 2048);
                    tma_load_2d(smem_u32(stg + b * 2048), &tmX, &eb[b], n, y);
                }
                pending |= 1u << b;
            };
            int k = 0;  // chunk counter of this warp; buffer k & 1
            if (U.first < U.count) {
                int sp0, mf, nf;
                unit_mn(p, U.first, U.rank, BN, &mf, &nf, &sp0);
                issue_ext(0, nf + half * CHUNKS * 32, mf + y_off);
            }
            bool ok = true;
            for (int it = U.first; it < U.count && ok; it += U.step) {
                int split_, m0, n0;
                unit_mn(p, it, U.rank, BN, &m0, &n0, &split_);
                if (!mbar_wait_warp(&tfull[acc], acc_phase, abort_flag, p.flags, 0x400 + 4, p.wait_limit)) break;
                tc_fence_after();
#pragma unroll 1
                for (int i = 0; i < CHUNKS; i++, k++) {
                    const int c = half * CHUNKS + i;
                    const int n = n0 + c * 32;
                    const int b = k & 1;
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + c * 32), r);
                    // the next chunk's operand goes to the other buffer once that
                    // buffer's last store has been read out
                    int nn = -1, ny = 0;
                    if (i + 1 < CHUNKS) {
                        nn = n + 32;
                        ny = m0 + y_off;
                    } else if (it + U.step < U.count) {
                        int sp2, m2, n2;
                        unit_mn(p, it + U.step, U.rank, BN, &m2, &n2, &sp2);
                        nn = n2 + half * CHUNKS * 32;
                        ny = m2 + y_off;
                    }
                    if (nn >= 0) {
                        if (lane == 0) bulk_wait_read<0>();
                        __syncwarp();
                        issue_ext(b ^ 1, nn, ny);
                    }
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[j]);
                    if (p.bias) {
                        float bb[32];
                        load32_16<F16>(p.bias + n, 32, true, bb);
                        add32(v, bb);
                    }
                    if (!mbar_wait_warp(&eb[b], (eph >> b) & 1u, abort_flag, p.flags, 0x400 + 5, p.wait_limit)) { ok = false; break; }
                    eph ^= 1u << b;
                    pending &= ~(1u << b);
                    float e[32];
                    load_row32<F16>(stg + b * 2048, lane, e);
                    if (p.epi == EPI_DGELU) mul_dgelu32(v, e);
                    else add32(v, e);
                    stage_row32<F16>(stg + b * 2048, lane, v);
                    if (p.colsum) {
                        // this chunk's 32 rows summed per column (rows past M
                        // hold zeros: their A rows were read as zero)
                        const float cs = warp_colsum32(v, lane);
                        p.colsum[(long long)((m0 + y_off) >> 5) * p.N + n + lane] = cs;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmD, smem_u32(stg + b * 2048), n, m0 + y_off);
                        bulk_commit();
                    }
                }
                tc_fence_before();
                if (leader) mbar_arrive(&tempty[acc]);
                else mbar_arrive_cluster(leader_addr(&tempty[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            // a load still in flight must land before the CTA's shared memory
            // goes away (also after an abort: no abort check here)
            for (int b = 0; b < 2; b++)
                if ((pending >> b) & 1u) mbar_drain(&eb[b], (eph >> b) & 1u);
        }
        for (int it = U.first; it < U.count && !p.ext_tma; it += U.step) {
            int split, m0, n0;
            unit_mn(p, it, U.rank, BN, &m0, &n0, &split);
            if (!mbar_wait_warp(&tfull[acc], acc_phase, abort_flag, p.flags, 0x400 + 4, p.wait_limit)) break;
            tc_fence_after();
            const int m = m0 + row;
            const bool row_ok = m < p.M;
#pragma unroll 1
            for (int c = half * CHUNKS; c < (half + 1) * CHUNKS; c++) {
                uint32_t r[32];
                __syncwarp();
                tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + c * 32), r);
                const int n = n0 + c * 32;
                const int valid = min(32, p.n_store - n);
                if (valid <= 0) continue;  // uniform across the warp
                if (p.tma_store) {
                    // bf16 result through shared memory and TMA; rows >= M and
                    // columns >= n_store are clipped by the tensor map
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[j]);
                    const long long o = (long long)m * p.ldd + n;
                    if (p.bias) {
                        float b[32];
                        load32_16<F16>(p.bias + n, valid, true, b);
                        add32(v, b);
                    }
                    const bool gelu = p.epi == EPI_GELU;
                    if (lane == 0) {
                        if (gelu) bulk_wait_read<0>(); else bulk_wait_read<1>();
                    }
                    __syncwarp();
                    if (gelu) {
                        stage_row32<F16>(stg, lane, v);  // pre-activation
                        gelu32(v);
                    } else if (p.epi == EPI_DGELU) {
                        float u_[32];
                        if (row_ok) load32_16<F16>(p.aux + o, valid, aux_vec, u_);
                        else {
#pragma unroll
                            for (int j = 0; j < 32; j++) u_[j] = 0.0f;
                        }
                        mul_dgelu32(v, u_);
                    }
                    if (p.residual && row_ok) {
                        float rr[32];
                        load32_16<F16>(p.residual + o, valid, res_vec, rr);
                        add32(v, rr);
                    }
                    uint8_t* dbuf = gelu ? stg + 2048 : stg + sbuf * 2048;
                    stage_row32<F16>(dbuf, lane, v);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int y = m0 + quarter * 32;
                        if (gelu) tma_store_2d(&tmX, smem_u32(stg), n, y);
                        tma_store_2d(&tmD, smem_u32(dbuf), n, y);
                        bulk_commit();
                    }
                    sbuf ^= 1;
                    continue;
                }
                if (!row_ok) continue;
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[j]);
                if (p.splits > 1) {
                    float* w = p.ws + ((long long)split * p.M + m) * p.N + n;
                    store32_f32(w, valid, (p.N & 3) == 0, v);
                    continue;
                }
                const long long o = (long long)m * p.ldd + n;
                if (p.d_f32) {
                    float* d = (float*)p.D + o;
                    if (p.accumulate) {
#pragma unroll
                        for (int j = 0; j < 32; j++)
                            if (j < valid) v[j] += d[j];
                    }
                    store32_f32(d, valid, out_vec, v);
                    continue;
                }
                if (p.bias) {
                    float b[32];
                    load32_16<F16>(p.bias + n, valid, true, b);
                    add32(v, b);
                }
                if (p.epi == EPI_GELU) {
                    store32_16<F16>(p.aux + o, valid, aux_vec, v);
                    gelu32(v);
                } else if (p.epi == EPI_DGELU) {
                    float u_[32];
                    load32_16<F16>(p.aux + o, valid, aux_vec, u_);
                    mul_dgelu32(v, u_);
                }
                if (p.residual) {
                    float rr[32];
                    load32_16<F16>(p.residual + o, valid, res_vec, rr);
                    add32(v, rr);
                }
                uint16_t* d = (uint16_t*)p.D + o;
                if (p.accumulate) {
                    float old[32];
                    load32_16<F16>(d, valid, out_vec, old);
                    add32(v, old);
                }
                store32_16<F16>(d, valid, out_vec, v);
            }
            tc_fence_before();
            if (leader) mbar_arrive(&tempty[acc]);
            else mbar_arrive_cluster(leader_addr(&tempty[acc]));
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        if (p.tma_store && lane == 0) bulk_wait_all();  // staged stores done before exit
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (PAIR) cluster_sync_all();  // neither CTA leaves while the other may still signal it
    if (warp == 1) {
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"((uint32_t)CF::TMEM_COLS));
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"((uint32_t)CF::TMEM_COLS));
    }
}

struct Plan {
    int BN;
    Params p;
    int grid;
};

// Launch of one instantiation (the dynamic shared-memory limit set once per
// device); the pair form as clusters of two CTAs.
template <int BN, bool A_MN, bool B_MN, bool PAIR, bool F16>
bool launch_tc(const Launch& L, const Plan& pl, const CUtensorMap& ma, const CUtensorMap& mb,
               const CUtensorMap& md, const CUtensorMap& mx) {
    auto kern = k_gemm_tc<BN, A_MN, B_MN, PAIR, F16>;
    constexpr int smem = Cfg<BN, PAIR>::SMEM_BYTES;
    static PerDevice attr;  // one flag per instantiation and device
    if (!attr.once([&] {
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess;
        })) {
        cudaGetLastError();
        return false;
    }
    L.count();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute at[2];
    int na = 0;
    if (PAIR) {
        at[na].id = cudaLaunchAttributeClusterDimension;
        at[na].val.clusterDim.x = 2;
        at[na].val.clusterDim.y = 1;
        at[na].val.clusterDim.z = 1;
        ++na;
    }
    if (L.pdl) {  // the kernel waits for its predecessor before any global access
        at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = at;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, md, mx, pl.p) == cudaSuccess;
}

// The IEEE-half instantiations (gemm_tc_f16.cu): the same dispatch over
// (BN, operand forms, pair form).
bool launch_tc_f16(int BN, bool a_mn, bool b_mn, bool pair, const Launch& L, const Plan& pl,
                   const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md, const CUtensorMap& mx);

}  // namespace tc
}  // namespace tt

// gemm_tc.cu -- the dense contractions of the step on the 5th-generation
// tensor cores: tcgen05.mma (bf16 or half in, fp32 accumulate in tensor memory),
// operands staged by TMA (cp.async.bulk.tensor, 128-byte swizzle) through an
// mbarrier ring, accumulators read back with tcgen05.ld for a fused epilogue.
//
// Persistent, warp-specialised CTA (320 threads, one CTA per SM):
//   warp 0      TMA producer (one elected lane)
//   warp 1      TMEM allocator + MMA issuer (one elected lane)
//   warps 2..9  epilogue: TMEM -> registers -> bias / GELU / GELU' /
//               residual -> global.  Warp w reads TMEM lanes 32*(w%4)..+31;
//               warps 2..5 take the left half of the tile's columns, 6..9
//               the right half.
// The accumulator is double-buffered in TMEM (2 x BN fp32 columns), so the
// epilogue of tile i overlaps the main loop of tile i+1.
//
// Operand forms (the three GEMMs of a linear layer):
//   FWD y = x W^T   : A K-major, B K-major
//   DX  dx = dy W   : A K-major, B MN-major
//   DW  dW = dy^T x : A MN-major, B MN-major, split over tokens (K) with a
//                     fixed-order reduction when the output has few tiles.
//
// Pair form (PAIR): the two CTAs of a cluster take the M tiles 2i and 2i + 1
// of the same N tile as one 256 x BN tile of tcgen05.mma.cta_group::2, issued
// by the even CTA (the leader).  Each CTA's shared memory holds its own A
// tile and one half of the B tile, so per SM the operand bytes written by TMA
// and read by the tensor cores fall by a third at BN = 256: a single-CTA
// 128 x 256 tile needs more shared-memory bandwidth (A and B read by the MMA
// plus the TMA writes) than an SM has.  Both CTAs' loads complete on the
// leader's full barrier; the leader's commits arrive on both CTAs' empty and
// accumulator-full barriers; both CTAs' epilogues release the leader's
// accumulator.
//
// Every mbarrier wait is bounded (about two seconds of clock cycles); on
// expiry the kernel raises FLAG_TIMEOUT, stops all roles, lets in-flight TMA
// copies land, frees its tensor memory and returns.
//
// The kernel template and its launch live in gemm_tc_kernel.cuh, templated on
// the 16-bit operand format: this file instantiates bf16, gemm_tc_f16.cu IEEE
// half (the fp16 mixed-precision step).
#include "gemm_tc_kernel.cuh"

#include <cudaTypedefs.h>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace tt {
namespace tc {

// D[m, n] (+)= sum_s ws[s][m][n] in split order (fp32 output, n < n_store)
__global__ void k_splitk_reduce(const float* __restrict__ ws, int splits, int M, int N, int n_store,
                                float* __restrict__ D, long long ldd, int accumulate) {
    pdl_enter();
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    long long total = (long long)M * n_store;
    if (i >= total) return;
    int m = (int)(i / n_store), n = (int)(i % n_store);
    float s = 0.0f;
    for (int k = 0; k < splits; k++) s += ws[((long long)k * M + m) * N + n];
    float* d = D + (long long)m * ldd + n;
    *d = accumulate ? *d + s : s;
}

// The same, four consecutive outputs per thread (16-byte loads and stores;
// needs N, n_store and ldd multiples of 4 and 16-byte aligned ws and D), the
// loads of up to eight splits in flight before their adds, in split order.
__global__ void k_splitk_reduce4(const float* __restrict__ ws, int splits, int M, int N, int n_store,
                                 float* __restrict__ D, long long ldd, int accumulate) {
    pdl_enter();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int nq = n_store >> 2;
    if (i >= (long long)M * nq) return;
    const int m = (int)(i / nq), n = 4 * (int)(i % nq);
    const long long plane = (long long)M * N;
    const float4* src = reinterpret_cast<const float4*>(ws + (long long)m * N + n);
    const long long step = plane >> 2;  // one split, in float4 units
    float4 s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int k0 = 0; k0 < splits; k0 += 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; u++)
            if (k0 + u < splits) v[u] = src[(k0 + u) * step];
#pragma unroll
        for (int u = 0; u < 8; u++)
            if (k0 + u < splits) { s.x += v[u].x; s.y += v[u].y; s.z += v[u].z; s.w += v[u].w; }
    }
    float4* d = reinterpret_cast<float4*>(D + (long long)m * ldd + n);
    if (accumulate) {
        const float4 o = *d;
        s.x = o.x + s.x; s.y = o.y + s.y; s.z = o.z + s.z; s.w = o.w + s.w;
    }
    *d = s;
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    });
    return fn;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, long long inner, long long outer,
                    long long pitch, int box_inner, int box_outer);

// 2-D bf16 map: inner extent, outer extent, row pitch in elements, box.
static bool make_map(CUtensorMap* map, const void* base, long long inner, long long outer,
                     long long pitch, int box_inner, int box_outer,
                     CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)(pitch * 2)};
    cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, long long inner, long long outer,
                    long long pitch, int box_inner, int box_outer) {
    return make_map(map, base, inner, outer, pitch, box_inner, box_outer);
}

static Plan plan_for(const Launch& L, const GemmArgs& g, int BN) {
    Plan pl{};
    pl.BN = BN;
    Params& p = pl.p;
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.m_tiles = (g.M + BM - 1) / BM;
    p.n_tiles = (g.N + pl.BN - 1) / pl.BN;
    p.tiles = p.m_tiles * p.n_tiles;
    // Tile order.  With n fastest, the CTAs running at the same time share A's
    // row blocks, so A is read from DRAM once and B is re-read, wave after wave,
    // from L2; with m fastest it is the other way round.  The larger operand is
    // the one to stream once: A when M >= N (A holds M x K elements, B N x K).
    p.n_fast = (g.M >= g.N) ? 1 : 0;
    p.kb_total = (g.K + BK - 1) / BK;
    p.splits = 1;
    const int sms = L.num_sms > 0 ? L.num_sms : 148;
    if (!g.a_kmajor && !g.b_kmajor && p.tiles < sms) {
        // DW form: few output tiles, long contraction over tokens
        int s = sms / p.tiles;
        int max_s = p.kb_total / 4;  // at least 4 k-blocks per split
        if (s > max_s) s = max_s;
        if (s < 1) s = 1;
        p.splits = s;
    }
    p.kb_per_split = (p.kb_total + p.splits - 1) / p.splits;
    p.splits = (p.kb_total + p.kb_per_split - 1) / p.kb_per_split;  // no empty split
    p.units = p.tiles * p.splits;
    pl.grid = p.units < sms ? p.units : sms;
    return pl;
}

static Plan finish_plan(const Launch& L, const GemmArgs& g, Plan pl) {
    Params& p = pl.p;
    p.D = g.D;
    p.ldd = g.ldd;
    p.d_f32 = g.d_f32 ? 1 : 0;
    p.n_store = g.n_store ? g.n_store : g.N;
    p.epi = g.epi;
    p.accumulate = g.accumulate ? 1 : 0;
    p.bias = (const __nv_bfloat16*)g.bias;
    p.residual = (const __nv_bfloat16*)g.residual;
    p.aux = (__nv_bfloat16*)g.aux;
    p.ws = nullptr;
    p.flags = L.flags;
    return pl;
}

// The pair form of the kernel (see its description) is on unless
// TT_GEMM_PAIR=0 is in the environment.
static bool pair_disabled() {
    static const bool off = [] {
        const char* e = getenv("TT_GEMM_PAIR");
        return e && e[0] == '0';
    }();
    return off;
}

// Tile width: 128 for narrow outputs, else 256.  Without the pair form, the
// weight-gradient form (both operands MN-major, few output tiles, split K)
// may take 192 instead when that needs clearly fewer tile-times (waves of the
// persistent grid x width x k-blocks per unit): its tiles then fill more of
// the SMs (for the [2304, 768] QKV weight, 144 units instead of 108).  N = 192
// MMAs run at a lower rate per FLOP than N = 256, which outweighs the better
// wave fill of the other forms; and a 192-wide B tile does not split into the
// pair form's halves, so with pairs the width stays 256.
static Plan make_plan(const Launch& L, const GemmArgs& g) {
    if (g.N <= 128) return finish_plan(L, g, plan_for(L, g, 128));
    if (g.a_kmajor || g.b_kmajor || !pair_disabled()) return finish_plan(L, g, plan_for(L, g, 256));
    const int sms = L.num_sms > 0 ? L.num_sms : 148;
    Plan best{};
    double best_cost = 0.0;
    for (int bn : {256, 192}) {
        Plan c = plan_for(L, g, bn);
        const double waves = (double)((c.p.units + sms - 1) / sms);
        const double cost = waves * bn * (double)c.p.kb_per_split;
        if (bn == 256 || cost < 0.92 * best_cost) {  // 192 must win clearly
            best = c;
            best_cost = cost;
        }
    }
    return finish_plan(L, g, best);
}


}  // namespace tc

bool gemm_tc_eligible(const GemmArgs& g) {
    if (!g.in_bf16 || g.M <= 0 || g.N <= 0 || g.K <= 0) return false;  // 16-bit operands (bf16 or half)
    if (g.a_kmajor && g.b_kmajor && g.d_f32) return false;     // forward form writes bf16
    if (!g.a_kmajor && g.b_kmajor) return false;               // form not used by the step
    if (!g.a_kmajor && !(g.d_f32 && g.epi == EPI_STORE && !g.bias && !g.residual)) return false;
    if ((g.lda % 8) || (g.ldb % 8)) return false;              // 16-byte TMA pitches
    if (((uintptr_t)g.A & 15) || ((uintptr_t)g.B & 15)) return false;
    if (g.bias && ((uintptr_t)g.bias & 15)) return false;
    if (!tc::encode_fn()) return false;
    return true;
}

size_t gemm_tc_workspace_floats(const Launch& L, const GemmArgs& g) {
    tc::Plan pl = tc::make_plan(L, g);
    return pl.p.splits > 1 ? (size_t)pl.p.splits * g.M * g.N : 0;
}

// Clusters of two that can be resident at once for the pair form of an
// instantiation (0: not available).
template <int BN, bool A_MN, bool B_MN>
static int active_pairs(const Launch& L) {
    static PerDevice pairs;  // one value per instantiation and device
    return pairs.value([&]() -> int {
        auto kern = tc::k_gemm_tc<BN, A_MN, B_MN, true, false>;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (L.num_sms / 2));
        cfg.blockDim = dim3(tc::THREADS);
        cfg.dynamicSmemBytes = tc::Cfg<BN, true>::SMEM_BYTES;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::Cfg<BN, true>::SMEM_BYTES) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&n, (void*)kern, &cfg) != cudaSuccess)
            n = 0;
        cudaGetLastError();
        return n;
    });
}

// Whether the pair form applies: an even number of M tiles, B splitting into
// two equal halves, resident pairs available, and not switched off
// (TT_GEMM_PAIR=0 in the environment).
template <int BN, bool A_MN, bool B_MN>
static bool use_pair(const Launch& L, tc::Plan& pl) {
    if (tc::pair_disabled() || L.no_pair || pl.p.units < 2) return false;
    // an odd M-tile count only where the output is written row by row
    if ((pl.p.m_tiles & 1) && !(A_MN && B_MN)) return false;
    if (B_MN && ((BN / tc::MN_BOX) & 1)) return false;
    const int pairs = active_pairs<BN, A_MN, B_MN>(L);
    if (pairs <= 0) return false;
    const int want = ((pl.p.m_tiles + 1) / 2) * pl.p.n_tiles * pl.p.splits;
    pl.p.cl = 1;
    pl.p.pair_units = want;
    pl.grid = 2 * (want < pairs ? want : pairs);
    return true;
}

// every column of the result is stored (the column sums then cover all N)
static bool ns_all(const GemmArgs& g) { return g.n_store == 0 || g.n_store == g.N; }

bool gemm_tc_launch(const Launch& L, const GemmArgs& g, float* workspace, size_t workspace_floats) {
    if (!gemm_tc_eligible(g)) return false;
    tc::Plan pl = tc::make_plan(L, g);
    if (pl.p.splits > 1) {
        if (!workspace || workspace_floats < (size_t)pl.p.splits * g.M * g.N) return false;
        pl.p.ws = workspace;
    }
    if (L.dry) return true;
    const bool a_mn = !g.a_kmajor, b_mn = !g.b_kmajor;
    const int a_rows = g.a_rows ? g.a_rows : g.M;
    const int b_rows = g.b_rows ? g.b_rows : g.N;
    const int kval = g.k_valid ? g.k_valid : g.K;
    pl.p.cl = 0;
    if (pl.BN == 256) {
        if (!a_mn && !b_mn) use_pair<256, false, false>(L, pl);
        else if (!a_mn) use_pair<256, false, true>(L, pl);
        else use_pair<256, true, true>(L, pl);
    } else if (pl.BN == 128) {
        if (!a_mn && !b_mn) use_pair<128, false, false>(L, pl);
        else if (!a_mn) use_pair<128, false, true>(L, pl);
        else use_pair<128, true, true>(L, pl);
    }
    CUtensorMap ma, mb;
    bool ok;
    if (!a_mn) ok = tc::make_map(&ma, g.A, kval, a_rows, g.lda, tc::BK, tc::BM);
    else ok = tc::make_map(&ma, g.A, a_rows, kval, g.lda, tc::MN_BOX, tc::BK);
    if (!ok) return false;
    // in the pair form each CTA loads half of a K-major B tile
    if (!b_mn) ok = tc::make_map(&mb, g.B, kval, b_rows, g.ldb, tc::BK, pl.p.cl ? pl.BN / 2 : pl.BN);
    else ok = tc::make_map(&mb, g.B, b_rows, kval, g.ldb, tc::MN_BOX, tc::BK);
    if (!ok) return false;
    // bf16 outputs: TMA stores (box 32 x 32, 64-byte swizzle) when the rows allow
    CUtensorMap md, mx;
    memset(&md, 0, sizeof md);
    memset(&mx, 0, sizeof mx);
    pl.p.tma_store = 0;
    if (!g.d_f32 && !g.accumulate && (g.ldd % 8) == 0 && ((uintptr_t)g.D & 15) == 0 &&
        (g.epi != EPI_GELU || ((uintptr_t)g.aux & 15) == 0)) {
        const int ns = g.n_store ? g.n_store : g.N;
        bool ok2 = tc::make_map(&md, g.D, ns, g.M, g.ldd, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
        if (ok2 && g.epi == EPI_GELU)
            ok2 = tc::make_map(&mx, g.aux, ns, g.M, g.ldd, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
        pl.p.tma_store = ok2 ? 1 : 0;
        // the extra operand of the GELU' or residual epilogue by TMA loads, same
        // box and layout as the stores (needs whole chunks: n_store % BN == 0)
        const void* ext = g.epi == EPI_DGELU ? g.aux : (g.epi == EPI_STORE ? g.residual : nullptr);
        if (ok2 && ext && (ns % pl.BN) == 0 && ((uintptr_t)ext & 15) == 0 &&
            tc::make_map(&mx, ext, ns, g.M, g.ldd, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
            pl.p.ext_tma = 1;
    }
    pl.p.colsum = nullptr;
    pl.p.wait_limit = L.wait_cycles;
    if (g.colsum_part && pl.p.ext_tma && ns_all(g)) pl.p.colsum = g.colsum_part;
    bool launched;
    const bool pr = pl.p.cl != 0;
#define TC(BN_, AM_, BM_)                                                        \
    (pr ? tc::launch_tc<BN_, AM_, BM_, true, false>(L, pl, ma, mb, md, mx)         \
        : tc::launch_tc<BN_, AM_, BM_, false, false>(L, pl, ma, mb, md, mx))
    if (g.in_f16) {
        launched = tc::launch_tc_f16(pl.BN, a_mn, b_mn, pr, L, pl, ma, mb, md, mx);
    } else if (pl.BN == 256) {
        if (!a_mn && !b_mn) launched = TC(256, false, false);
        else if (!a_mn) launched = TC(256, false, true);
        else launched = TC(256, true, true);
    } else if (pl.BN == 192) {  // weight-gradient form only, never paired
        launched = (a_mn && b_mn && !pr) && tc::launch_tc<192, true, true, false, false>(L, pl, ma, mb, md, mx);
    } else {
        if (!a_mn && !b_mn) launched = TC(128, false, false);
        else if (!a_mn) launched = TC(128, false, true);
        else launched = TC(128, true, true);
    }
#undef TC
    if (!launched) return false;
    if (pl.p.colsum && g.colsum_done) *g.colsum_done = true;
    if (pl.p.splits > 1) {
        const bool vec = (g.N % 4) == 0 && (pl.p.n_store % 4) == 0 && (g.ldd % 4) == 0 &&
                         ((uintptr_t)workspace & 15) == 0 && ((uintptr_t)g.D & 15) == 0;
        L.count();
        if (vec) {
            const long long total = (long long)g.M * (pl.p.n_store / 4);
            launch_k(L, tc::k_splitk_reduce4, dim3((unsigned)((total + 255) / 256)), dim3(256), 0, 
                workspace, pl.p.splits, g.M, g.N, pl.p.n_store, (float*)g.D, g.ldd, g.accumulate ? 1 : 0);
        } else {
            const long long total = (long long)g.M * pl.p.n_store;
            launch_k(L, tc::k_splitk_reduce, dim3((unsigned)((total + 255) / 256)), dim3(256), 0, 
                workspace, pl.p.splits, g.M, g.N, pl.p.n_store, (float*)g.D, g.ldd, g.accumulate ? 1 : 0);
        }
    }
    return true;
}

}  // namespace tt

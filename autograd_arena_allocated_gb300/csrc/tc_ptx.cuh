// tc_ptx.cuh -- inline-PTX building blocks for the sm_103a tensor-core kernels:
// mbarriers (with bounded waits), TMA tile loads, tcgen05 MMA / commit /
// TMEM loads and the shared-memory and instruction descriptors.
#pragma once

#include <cuda.h>
#include <stdint.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tt_internal.h"

namespace tt {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: true when the phase with the given parity has completed;
// false if another role aborted or the limit passed (then FLAG_TIMEOUT and
// FLAG_SITE).  The limit (clock64 cycles) is a kernel argument taken from the
// context; WAIT_CYCLES is the default.  A failing try_wait returns after a
// couple of hundred cycles, and the abort flags and the clock are looked at
// every 64 polls -- every poll when the limit is below SHORT_WAIT, so that a
// wait that is not complete within a few hundred cycles of its start runs
// out (the form a test uses to make a wait run out).
constexpr long long WAIT_CYCLES = 4000000000LL;  // ~2 s at 2 GHz
constexpr long long SHORT_WAIT = 1000000LL;

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* flags, int site = 0, long long limit = WAIT_CYCLES) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    const uint32_t mask = limit < SHORT_WAIT ? 0u : 63u;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & mask) == 0) {
            if (*abort_flag) return false;
            // another CTA (or an earlier kernel) gave up: stop at once
            if (((volatile int*)flags)[FLAG_TIMEOUT]) {
                *abort_flag = 1;
                return false;
            }
            if (clock64() - t0 > limit) {
                atomicCAS(&flags[FLAG_SITE], 0, site);
                atomicOr(&flags[FLAG_TIMEOUT], 1);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// The same wait taken by all 32 lanes of a warp, with a warp-uniform result:
// the warp-collective tcgen05.ld/st that follow it must run converged, so no
// lane may leave the loop that issues them alone.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                               int* flags, int site = 0, long long limit = WAIT_CYCLES) {
    const bool ok = mbar_wait(bar, parity, abort_flag, flags, site, limit);
    return __all_sync(0xffffffffu, ok);
}

// Spins until the phase completes or the fixed landing bound (WAIT_CYCLES,
// whatever the context's limit) passes, with no abort check: used only to let
// copies and MMAs already issued finish before a CTA that gave up frees the
// shared or tensor memory they write.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity) && clock64() - t0 < WAIT_CYCLES) {}
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// The same MMA with A read from tensor memory: A's M rows are TMEM lanes
// and each 32-bit column holds two consecutive K elements (the lower K index
// in the low half), so one K=16 step reads 8 columns starting at a_tmem.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Two 32-column loads with one wait: both loads are in flight together.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t (&a)[32], uint32_t tb, uint32_t (&b)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
        : "r"(ta), "r"(tb)
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (all >> 4), version 1, 128-byte swizzle.
//   K-major tile  (rows of 128 B, 8-row atoms): LBO unused (16), SBO = 1024
//   MN-major tile (k-rows of 64 MN elements):   LBO = distance between 64-wide
//                                               MN blocks, SBO = 1024 (8 k-rows)
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B,
// operand majors, N >> 3 and M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}


// 16-bit storage: bf16, or IEEE half when F16 (the fp16 mixed-precision
// step); every sum stays fp32.  lo16 / hi16 unpack the element in the low /
// high half of a 32-bit word, pack2 rounds two floats to nearest even.
template <bool F16>
__device__ __forceinline__ float lo16(uint32_t u) {
    if constexpr (F16) return __half2float(__ushort_as_half((unsigned short)(u & 0xFFFFu)));
    else return __uint_as_float(u << 16);
}
template <bool F16>
__device__ __forceinline__ float hi16(uint32_t u) {
    if constexpr (F16) return __half2float(__ushort_as_half((unsigned short)(u >> 16)));
    else return __uint_as_float(u & 0xFFFF0000u);
}
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (F16) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}
template <bool F16>
__device__ __forceinline__ float ld16(const void* p, int j) {
    if constexpr (F16) return __half2float(reinterpret_cast<const __half*>(p)[j]);
    else return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[j]);
}
template <bool F16>
__device__ __forceinline__ void st16(void* p, int j, float v) {
    if constexpr (F16) reinterpret_cast<__half*>(p)[j] = __float2half_rn(v);
    else reinterpret_cast<__nv_bfloat16*>(p)[j] = __float2bfloat16_rn(v);
}
// the MMA instruction descriptor for 16-bit operands of either format
template <bool F16>
__host__ __device__ constexpr uint32_t idesc16(int M, int N, bool a_mn, bool b_mn) {
    return F16 ? (idesc_bf16(M, N, a_mn, b_mn) & ~((7u << 7) | (7u << 10))) : idesc_bf16(M, N, a_mn, b_mn);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// 16 consecutive 32-bit columns of this warp's 32 lanes
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Column sums of a 32 x 32 block held one row per lane (v: the lane's 32
// columns; overwritten): after a butterfly that halves the columns each lane
// keeps at each step, lane l holds the sum over the 32 rows of column l.  The
// order of the additions is fixed, so the result is deterministic.
__device__ __forceinline__ float warp_colsum32(float (&v)[32], int lane) {
#pragma unroll
    for (int s = 16; s >= 2; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; i += 2) {  // two columns per packed fp32x2 add
            float2 send, keep;
            send.x = up ? v[i] : v[i + s];
            send.y = up ? v[i + 1] : v[i + s + 1];
            keep.x = up ? v[i + s] : v[i];
            keep.y = up ? v[i + s + 1] : v[i + 1];
            const float2 got = make_float2(__shfl_xor_sync(0xffffffffu, send.x, s),
                                           __shfl_xor_sync(0xffffffffu, send.y, s));
            const float2 r = __fadd2_rn(keep, got);
            v[i] = r.x;
            v[i + 1] = r.y;
        }
    }
    const bool up = (lane & 1) != 0;
    return (up ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, up ? v[0] : v[1], 1);
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* holder, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(holder)),
                 "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// Host: a 2-D bf16 TMA map with 128-byte swizzle (inner extent, outer extent,
// row pitch in elements, box); false if the driver entry point is missing.
bool make_tmap_bf16(CUtensorMap* map, const void* base, long long inner, long long outer,
                    long long pitch, int box_inner, int box_outer);

}  // namespace tc
}  // namespace tt

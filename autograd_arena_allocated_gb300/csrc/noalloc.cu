// noalloc.cu -- tt_linear_bwd_dw_noalloc: the weight-gradient GEMM for
// callers that cannot allocate device memory.
//
// Its scratch (split-K partial sums and bias-gradient partial sums) lives in
// one fixed file-scope device array instead of a context arena, so the call
// needs no tt_ctx and performs no allocation of any kind.  Every GPU that
// loads this library holds the array (TT_NOALLOC_SCRATCH_BYTES) until the
// process exits.
//
// Layout of the array: [256 B device flags][split-K partials][bias partials].
#include "tt_internal.h"

#include <mutex>

namespace {

constexpr size_t kFlagBytes = 256;
constexpr size_t kSplitFloats = TT_NOALLOC_SPLIT_FLOATS;
constexpr size_t kBiasFloats = TT_NOALLOC_BIAS_FLOATS;
static_assert(kFlagBytes + 4 * (kSplitFloats + kBiasFloats) == TT_NOALLOC_SCRATCH_BYTES,
              "scratch layout");

// The scratch.  In host code this name is only a host-side stand-in for the
// symbol: kernels are given the device address that cudaGetSymbolAddress
// returns for the current device.
static __device__ __align__(256) unsigned char g_scratch[TT_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_addr[tt::kMaxDevices] = {};
int g_sms[tt::kMaxDevices] = {};

// Set-up, once per device, with that device current: look up (and cache) the
// device address of g_scratch and the device's SM count.
tt_status scratch_for_current_device(void** addr, int* sms) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= tt::kMaxDevices) {
        cudaGetLastError();
        return TT_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return TT_ERR_CUDA;
        }
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return TT_ERR_CUDA;
        }
        g_addr[dev] = p;
        g_sms[dev] = n;
    }
    *addr = g_addr[dev];
    *sms = g_sms[dev];
    return TT_OK;
}

}  // namespace

extern "C" tt_status tt_linear_bwd_dw_noalloc(void* stream, const void* dy, const void* x, float* dW,
                                              float* db, int M, int K, int N) {
    if (!dy || !x || !dW || M <= 0 || K <= 0 || N <= 0) return TT_ERR_ARG;
    // bias-gradient partial sums: one row of N floats per 256 tokens
    if (db && (size_t)((M + 255) / 256) * (size_t)N > kBiasFloats) return TT_ERR_ARG;

    tt::GemmArgs g;
    g.A = dy; g.lda = N; g.a_kmajor = false;
    g.B = x; g.ldb = K; g.b_kmajor = false;
    g.M = N; g.N = K; g.K = M;
    g.in_bf16 = true;
    g.D = dW; g.ldd = K; g.d_f32 = true;
    if (!tt::gemm_tc_eligible(g)) return TT_ERR_ARG;

    void* base = nullptr;
    int sms = 0;
    tt_status s = scratch_for_current_device(&base, &sms);
    if (s != TT_OK) return s;

    tt::Launch L;
    L.stream = (cudaStream_t)stream;
    L.flags = (int*)base;
    L.num_sms = sms;
    float* split_ws = (float*)((char*)base + kFlagBytes);
    float* bias_ws = split_ws + kSplitFloats;
    const size_t ws = tt::gemm_tc_workspace_floats(L, g);
    if (ws > kSplitFloats) return TT_ERR_ARG;  // only on GPUs with more than 192 SMs

    // The flags must start at zero.  Nothing else needs clearing: every
    // scratch element this call reads is written earlier in the same call.
    if (cudaMemsetAsync(L.flags, 0, kFlagBytes, L.stream) != cudaSuccess) {
        cudaGetLastError();
        return TT_ERR_CUDA;
    }
    if (!tt::gemm_tc_launch(L, g, ws ? split_ws : nullptr, ws)) return TT_ERR_CUDA;
    if (db) tt::launch_colsum(L, true, dy, M, N, db, bias_ws);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

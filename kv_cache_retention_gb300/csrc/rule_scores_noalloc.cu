// kvsel_rule_scores_noalloc: the rule-score call without any device allocation.
//
// kvsel_rule_scores takes its scratch (the [L][Hq][N] logits, the per-chunk
// (max, sum) pairs and the per-head log-sum-exps) from the context workspace,
// which grows with cudaMalloc/cudaFree.  Some callers cannot let a library do
// that: serving engines that hand almost all device memory to their own KV
// page pool at start-up and route every other allocation through their own
// allocator, code that records a CUDA graph (allocation is not allowed inside
// stream capture), and latency-critical loops that cannot afford the implicit
// device synchronisation of cudaFree.  This variant runs the same kernels on a
// fixed scratch array that is part of the library image instead.
//
// The array below is a host-side symbol in host code; the kernels must be given
// its device address, which cudaGetSymbolAddress returns once per device (with
// that device current) and which is cached here.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "kvsel_internal.h"

namespace {

constexpr size_t kScratchBytes = 64ull << 20;  // 64 MiB, held by every GPU that loads the library
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
void* scratch_address(int device, cudaError_t* err) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[device]) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (*err != cudaSuccess) return nullptr;
        g_scratch_addr[device] = p;
    }
    *err = cudaSuccess;
    return g_scratch_addr[device];
}

int fail(kvsel_ctx* ctx, int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(ctx->err, sizeof ctx->err, fmt, ap);
    va_end(ap);
    return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int kvsel_rule_scores_noalloc(kvsel_ctx* ctx, const void* k_pool, int k_dtype, const int32_t* slot_map,
                                         int n_slots, int L, int Hq, int Hkv, int N, int D, int64_t layer_stride,
                                         int64_t slot_stride, const float* M, int pi, int q_s, int q_e, float* rule,
                                         void* stream) {
    if (!ctx) return KVSEL_ERR_INVALID_ARG;
    ctx->err[0] = 0;
    cudaError_t e = cudaSetDevice(ctx->device);
    if (e != cudaSuccess) return fail(ctx, KVSEL_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(e));
    // the same argument rules as kvsel_rule_scores
    if (!k_pool || !M || !rule) return fail(ctx, KVSEL_ERR_INVALID_ARG, "rule_scores_noalloc: null pointer");
    if (k_dtype != KVSEL_F32 && k_dtype != KVSEL_BF16)
        return fail(ctx, KVSEL_ERR_INVALID_ARG, "rule_scores_noalloc: bad dtype");
    if (L <= 0 || Hq <= 0 || Hkv <= 0 || N < 0 || n_slots < 0)
        return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_noalloc: bad sizes");
    if (Hq % Hkv) return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_noalloc: Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
    if (Hq / Hkv > 8) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "rule_scores_noalloc: group size Hq/Hkv=%d > 8", Hq / Hkv);
    if (!(D == 16 || D == 32 || D == 64 || D == 128 || D == 256))
        return fail(ctx, KVSEL_ERR_UNSUPPORTED, "rule_scores_noalloc: D=%d unsupported", D);
    if ((int64_t)Hkv * D > 4096) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "rule_scores_noalloc: Hkv*D > 4096");
    if (pi < 0 || pi > N || q_s < 0 || q_s > q_e || q_e > N)
        return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_noalloc: forced ranges outside [0,N]");
    if (!slot_map && n_slots < N)
        return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_noalloc: identity slot map needs n_slots >= N");
    if (slot_stride < (int64_t)Hkv * D || layer_stride < 0)
        return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_noalloc: slot_stride < Hkv*D");
    if (L > 1 && layer_stride < (int64_t)n_slots * slot_stride)
        return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_noalloc: layers overlap");
    const int64_t es = k_dtype == KVSEL_BF16 ? 2 : 4;
    if (!aligned16(k_pool) || (layer_stride * es) % 16 || (slot_stride * es) % 16 || !aligned16(M) ||
        !aligned16(rule))
        return fail(ctx, KVSEL_ERR_ALIGN, "rule_scores_noalloc: pool, strides, M and rule must be 16-byte aligned");
    const size_t need = rule_scores_workspace(ctx, L, Hq, N);
    if (need > kScratchBytes)
        return fail(ctx, KVSEL_ERR_UNSUPPORTED,
                    "rule_scores_noalloc: this size needs %zu bytes of scratch but the fixed scratch holds %zu "
                    "(4*L*Hq*N must stay below ~64 MiB); use kvsel_rule_scores",
                    need, kScratchBytes);
    if (ctx->device < 0 || ctx->device >= kMaxDevices)
        return fail(ctx, KVSEL_ERR_UNSUPPORTED, "rule_scores_noalloc: device %d beyond %d", ctx->device, kMaxDevices);
    if (N == 0) return KVSEL_OK;
    void* ws = scratch_address(ctx->device, &e);
    if (!ws) return fail(ctx, KVSEL_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    // Every scratch word the kernels read is written earlier in the same call, so
    // nothing has to be cleared between calls.
    e = launch_rule_scores(ctx, k_pool, k_dtype, slot_map, n_slots, L, Hq, Hkv, N, D, layer_stride, slot_stride, M, pi,
                           q_s, q_e, rule, ws, (cudaStream_t)stream);
    return e == cudaSuccess ? KVSEL_OK
                            : fail(ctx, KVSEL_ERR_CUDA, "rule_scores_noalloc launch: %s", cudaGetErrorString(e));
}

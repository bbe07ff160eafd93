// kvsel_rule_scores_noalloc: the rule-score call without any device allocation.
//
// kvsel_rule_scores takes its scratch (the [L][Hq][N] logits, the per-chunk
// (max, sum) pairs and the per-head log-sum-exps) from the context workspace,
// which grows with cudaMalloc/cudaFree.  Some callers cannot let a library do
// that: serving engines that hand almost all device memory to their own KV
// page pool at start-up and route every other allocation through their own
// allocator, and latency-critical loops that cannot afford the implicit device
// synchronisation of cudaFree.  This variant runs the same kernels on a fixed
// scratch array that is part of the library image instead.
//
// In host code the array below names a host-side stand-in, not device memory:
// the kernels must be given its device address, which cudaGetSymbolAddress
// returns with the context's device current.  The address is looked up on the
// first call with a context and kept in that context, so a context created
// after a device reset looks it up again.
#include <cstdint>

#include "kvsel_internal.h"

namespace {

constexpr size_t kScratchBytes = 64ull << 20;  // 64 MiB, held by every GPU that loads the library

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

}  // namespace

extern "C" int kvsel_rule_scores_noalloc(kvsel_ctx* ctx, const void* k_pool, int k_dtype, const int32_t* slot_map,
                                         int n_slots, int L, int Hq, int Hkv, int N, int D, int64_t layer_stride,
                                         int64_t slot_stride, const float* M, int pi, int q_s, int q_e, float* rule,
                                         void* stream) {
    const kvsel_trace trace_("kvsel_rule_scores_noalloc");
    int rc = kvsel_enter(ctx);  // also makes the context's device current
    if (rc) return rc;
    rc = kvsel_check_rule_scores_args(ctx, "rule_scores_noalloc", k_pool, k_dtype, slot_map, n_slots, L, Hq, Hkv, N,
                                      D, layer_stride, slot_stride, M, pi, q_s, q_e, rule);
    if (rc) return rc;
    const size_t need = rule_scores_workspace(ctx, L, Hq, N);
    if (need > kScratchBytes)
        return kvsel_fail(ctx, KVSEL_ERR_UNSUPPORTED,
                          "rule_scores_noalloc: this size needs %zu bytes of scratch but the fixed scratch holds %zu "
                          "(4*L*Hq*N must stay below ~64 MiB); use kvsel_rule_scores",
                          need, kScratchBytes);
    if (N == 0) return KVSEL_OK;
    if (!ctx->noalloc_scratch) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return kvsel_cuda_fail(ctx, e, "rule_scores_noalloc: cudaGetSymbolAddress");
        ctx->noalloc_scratch = p;
    }
    // Every scratch word the kernels read is written earlier in the same call, so
    // nothing has to be cleared between calls.
    cudaError_t e = launch_rule_scores(ctx, k_pool, k_dtype, slot_map, n_slots, L, Hq, Hkv, N, D, layer_stride,
                                       slot_stride, M, pi, q_s, q_e, rule, ctx->noalloc_scratch, (cudaStream_t)stream);
    return e == cudaSuccess ? KVSEL_OK : kvsel_cuda_fail(ctx, e, "rule_scores_noalloc launch");
}

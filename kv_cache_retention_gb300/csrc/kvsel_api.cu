// libkvsel C ABI: context management and host-side validation of every call.
// Each entry point checks its arguments completely before launching anything,
// so a rejected call leaves every buffer untouched (see include/kvsel.h).
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "kvsel_internal.h"

#define KVSEL_VERSION 100  // 0.1.0

namespace {

int vfail(kvsel_ctx* ctx, int code, const char* fmt, va_list ap) {
    if (ctx) vsnprintf(ctx->err, sizeof ctx->err, fmt, ap);
    return code;
}

int fail(kvsel_ctx* ctx, int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    const int rc = vfail(ctx, code, fmt, ap);
    va_end(ap);
    return rc;
}

int cuda_fail(kvsel_ctx* ctx, cudaError_t e, const char* what) {
    return fail(ctx, KVSEL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2_head_dim(int D) { return D == 16 || D == 32 || D == 64 || D == 128 || D == 256; }

// |[0,pi) U [q_s,q_e)|
int64_t forced_count(int pi, int q_s, int q_e) {
    int64_t overlap = 0;
    int64_t lo = q_s, hi = q_e < pi ? q_e : pi;
    if (hi > lo) overlap = hi - lo;
    return (int64_t)pi + (q_e - q_s) - overlap;
}

// Entry guard: context present, device current, error string cleared.
int enter(kvsel_ctx* ctx) {
    if (!ctx) return KVSEL_ERR_INVALID_ARG;
    ctx->err[0] = 0;
    cudaError_t e = cudaSetDevice(ctx->device);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaSetDevice");
    return KVSEL_OK;
}

int launched(kvsel_ctx* ctx, cudaError_t e, const char* what) {
    return e == cudaSuccess ? KVSEL_OK : cuda_fail(ctx, e, what);
}

}  // namespace

int kvsel_enter(kvsel_ctx* ctx) { return enter(ctx); }

int kvsel_fail(kvsel_ctx* ctx, int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    const int rc = vfail(ctx, code, fmt, ap);
    va_end(ap);
    return rc;
}

int kvsel_cuda_fail(kvsel_ctx* ctx, cudaError_t e, const char* what) { return cuda_fail(ctx, e, what); }

int kvsel_check_rule_scores_args(kvsel_ctx* ctx, const char* who, const void* k_pool, int k_dtype,
                                 const int32_t* slot_map, int n_slots, int L, int Hq, int Hkv, int N, int D,
                                 int64_t layer_stride, int64_t slot_stride, const float* M, int pi, int q_s, int q_e,
                                 const float* rule) {
    if (!k_pool || !M || !rule) return fail(ctx, KVSEL_ERR_INVALID_ARG, "%s: null pointer", who);
    if (k_dtype != KVSEL_F32 && k_dtype != KVSEL_BF16) return fail(ctx, KVSEL_ERR_INVALID_ARG, "%s: bad dtype", who);
    if (L <= 0 || Hq <= 0 || Hkv <= 0 || N < 0 || n_slots < 0) return fail(ctx, KVSEL_ERR_SHAPE, "%s: bad sizes", who);
    if (Hq % Hkv) return fail(ctx, KVSEL_ERR_SHAPE, "%s: Hq=%d not a multiple of Hkv=%d", who, Hq, Hkv);
    if (Hq / Hkv > 8) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "%s: group size Hq/Hkv=%d > 8", who, Hq / Hkv);
    if (!pow2_head_dim(D)) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "%s: D=%d unsupported", who, D);
    if ((int64_t)Hkv * D > 4096) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "%s: Hkv*D > 4096", who);
    if (pi < 0 || pi > N || q_s < 0 || q_s > q_e || q_e > N)
        return fail(ctx, KVSEL_ERR_SHAPE, "%s: forced ranges outside [0,N]", who);
    if (!slot_map && n_slots < N) return fail(ctx, KVSEL_ERR_SHAPE, "%s: identity slot map needs n_slots >= N", who);
    if (slot_stride < (int64_t)Hkv * D || layer_stride < 0)
        return fail(ctx, KVSEL_ERR_SHAPE, "%s: slot_stride < Hkv*D", who);
    if (L > 1 && layer_stride < (int64_t)n_slots * slot_stride)
        return fail(ctx, KVSEL_ERR_SHAPE, "%s: layers overlap", who);
    const int64_t es = k_dtype == KVSEL_BF16 ? 2 : 4;
    if (!aligned16(k_pool) || (layer_stride * es) % 16 || (slot_stride * es) % 16 || !aligned16(M) || !aligned16(rule))
        return fail(ctx, KVSEL_ERR_ALIGN, "%s: pool, strides, M and rule must be 16-byte aligned", who);
    return KVSEL_OK;
}

void* kvsel_workspace(kvsel_ctx* ctx, size_t bytes) {
    if (bytes == 0) bytes = 256;
    if (bytes <= ctx->ws_bytes) return ctx->ws;
    if (ctx->ws) {
        cudaFree(ctx->ws);  // implicit device synchronisation: no launch still uses it
        ctx->ws = nullptr;
        ctx->ws_bytes = 0;
    }
    size_t want = (bytes + (1u << 20) - 1) & ~((size_t)(1u << 20) - 1);
    if (cudaMalloc(&ctx->ws, want) != cudaSuccess) {
        ctx->ws = nullptr;
        return nullptr;
    }
    ctx->ws_bytes = want;
    return ctx->ws;
}

const kvsel_ctx::RopeTab* kvsel_rope_tables(kvsel_ctx* ctx, int D, double base, cudaStream_t s) {
    for (int i = 0; i < ctx->n_rope; ++i)
        if (ctx->rope[i].D == D && ctx->rope[i].base == base) return &ctx->rope[i];
    int slot = ctx->n_rope < 8 ? ctx->n_rope : 7;  // keep at most 8; recycle the last
    kvsel_ctx::RopeTab& t = ctx->rope[slot];
    auto release = [&t]() {
        cudaFree(t.lo);
        cudaFree(t.hi);
        cudaFree(t.lodf);
        cudaFree(t.hidf);
        t.lo = t.hi = nullptr;
        t.lodf = t.hidf = nullptr;
        t.D = 0;
    };
    if (t.lo) release();
    size_t half = (size_t)D / 2;
    if (cudaMalloc(&t.lo, sizeof(float2) * half * KVSEL_ROPE_LO) != cudaSuccess ||
        cudaMalloc(&t.hi, sizeof(float2) * half * KVSEL_ROPE_HI) != cudaSuccess ||
        cudaMalloc(&t.lodf, sizeof(float4) * half * KVSEL_ROPE_LO) != cudaSuccess ||
        cudaMalloc(&t.hidf, sizeof(float4) * half * KVSEL_ROPE_HI) != cudaSuccess) {
        release();
        return nullptr;
    }
    if (launch_rope_tables(t.lo, t.hi, t.lodf, t.hidf, D, base, s) != cudaSuccess) {
        release();
        return nullptr;
    }
    t.D = D;
    t.base = base;
    if (slot == ctx->n_rope) ++ctx->n_rope;
    return &t;
}

extern "C" {

int kvsel_version(void) { return KVSEL_VERSION; }

int kvsel_ctx_create(int device, kvsel_ctx** out) {
    if (!out) return KVSEL_ERR_INVALID_ARG;
    *out = nullptr;
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) return KVSEL_ERR_INVALID_ARG;
    if (cudaSetDevice(device) != cudaSuccess) return KVSEL_ERR_CUDA;
    kvsel_ctx* ctx = new (std::nothrow) kvsel_ctx();
    if (!ctx) return KVSEL_ERR_CUDA;
    ctx->device = device;
    if (cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaMalloc(&ctx->dev_err, sizeof(unsigned)) != cudaSuccess ||
        cudaMemset(ctx->dev_err, 0, sizeof(unsigned)) != cudaSuccess) {
        if (ctx->dev_err) cudaFree(ctx->dev_err);
        delete ctx;
        return KVSEL_ERR_CUDA;
    }
    *out = ctx;
    return KVSEL_OK;
}

int kvsel_ctx_destroy(kvsel_ctx* ctx) {
    if (!ctx) return KVSEL_OK;
    cudaSetDevice(ctx->device);
    cudaDeviceSynchronize();
    kvsel_stager_release(ctx);
    if (ctx->ws) cudaFree(ctx->ws);
    if (ctx->dev_err) cudaFree(ctx->dev_err);
    for (int i = 0; i < ctx->n_rope; ++i) {
        cudaFree(ctx->rope[i].lo);
        cudaFree(ctx->rope[i].hi);
        cudaFree(ctx->rope[i].lodf);
        cudaFree(ctx->rope[i].hidf);
    }
    delete ctx;
    return KVSEL_OK;
}

const char* kvsel_last_error_string(const kvsel_ctx* ctx) { return ctx ? ctx->err : "null context"; }

int kvsel_check_device(kvsel_ctx* ctx, void* stream) {
    const kvsel_trace trace_("kvsel_check_device");
    int rc = enter(ctx);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
    unsigned word = 0;
    e = cudaMemcpy(&word, ctx->dev_err, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "read device error word");
    if (!word) return KVSEL_OK;
    cudaMemset(ctx->dev_err, 0, sizeof(unsigned));
    if (word & KVSEL_DEV_TIMEOUT) return fail(ctx, KVSEL_ERR_TIMEOUT, "a bounded device wait gave up (tensor-core pipeline)");
    return fail(ctx, KVSEL_ERR_DEVICE_CHECK, "device check failed:%s%s%s%s%s%s",
                (word & KVSEL_DEV_BAD_SLOT) ? " slot out of range" : "",
                (word & KVSEL_DEV_BAD_POSITION) ? " position out of range" : "",
                (word & KVSEL_DEV_BAD_BLOCK) ? " source block or cursor id out of range" : "",
                (word & KVSEL_DEV_BAD_PAGE) ? " page out of range" : "",
                (word & KVSEL_DEV_BAD_SET) ? " working set not ascending or page held twice" : "",
                (word & KVSEL_DEV_POOL_FULL) ? " too few free pages" : "");
}

int kvsel_memory_update(kvsel_ctx* ctx, const void* q_rows, int q_dtype, int L, int Hq, int R, int D,
                        float lambda, int first_turn, int norm_mode, float* M, float* A, void* stream) {
    const kvsel_trace trace_("kvsel_memory_update");
    int rc = enter(ctx);
    if (rc) return rc;
    if (!q_rows || !M) return fail(ctx, KVSEL_ERR_INVALID_ARG, "memory_update: null q_rows or M");
    if (q_dtype != KVSEL_F32 && q_dtype != KVSEL_BF16) return fail(ctx, KVSEL_ERR_INVALID_ARG, "memory_update: bad dtype");
    if (norm_mode != 0 && norm_mode != 1) return fail(ctx, KVSEL_ERR_INVALID_ARG, "memory_update: norm_mode must be 0 or 1");
    if (norm_mode == 1 && !A) return fail(ctx, KVSEL_ERR_INVALID_ARG, "memory_update: norm_mode 1 needs A");
    if (L <= 0 || Hq <= 0 || R <= 0 || D <= 0) return fail(ctx, KVSEL_ERR_SHAPE, "memory_update: sizes must be positive");
    if (D > 1024 || D % (q_dtype == KVSEL_BF16 ? 8 : 4)) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "memory_update: D=%d unsupported", D);
    if (!(lambda >= 0.0f) || lambda != lambda) return fail(ctx, KVSEL_ERR_INVALID_ARG, "memory_update: lambda must be >= 0");
    if (!aligned16(q_rows) || !aligned16(M) || (A && !aligned16(A))) return fail(ctx, KVSEL_ERR_ALIGN, "memory_update: pointers must be 16-byte aligned");
    return launched(ctx, launch_memory_update(q_rows, q_dtype, L, Hq, R, D, lambda, first_turn, norm_mode, M, A, (cudaStream_t)stream), "memory_update launch");
}

int kvsel_memory_update_batch(kvsel_ctx* ctx, int q_dtype, int L, int Hq, int D, int norm_mode,
                              const kvsel_memory_session* sessions, int S, void* stream) {
    const kvsel_trace trace_("kvsel_memory_update_batch");
    int rc = enter(ctx);
    if (rc) return rc;
    if (S < 0 || S > 65535 || (S > 0 && !sessions)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "memory_update_batch: bad session table");
    if (q_dtype != KVSEL_F32 && q_dtype != KVSEL_BF16) return fail(ctx, KVSEL_ERR_INVALID_ARG, "memory_update_batch: bad dtype");
    if (norm_mode != 0 && norm_mode != 1) return fail(ctx, KVSEL_ERR_INVALID_ARG, "memory_update_batch: norm_mode must be 0 or 1");
    if (L <= 0 || Hq <= 0 || D <= 0) return fail(ctx, KVSEL_ERR_SHAPE, "memory_update_batch: sizes must be positive");
    if (D > 1024 || D % (q_dtype == KVSEL_BF16 ? 8 : 4)) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "memory_update_batch: D=%d unsupported", D);
    for (int i = 0; i < S; ++i) {
        const kvsel_memory_session& x = sessions[i];
        if (!x.q_rows || !x.M) return fail(ctx, KVSEL_ERR_INVALID_ARG, "memory_update_batch: session %d: null q_rows or M", i);
        if (norm_mode == 1 && !x.A) return fail(ctx, KVSEL_ERR_INVALID_ARG, "memory_update_batch: session %d: norm_mode 1 needs A", i);
        if (x.R <= 0) return fail(ctx, KVSEL_ERR_SHAPE, "memory_update_batch: session %d: R must be positive", i);
        if (!(x.lambda >= 0.0f)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "memory_update_batch: session %d: lambda must be >= 0", i);
        if (!aligned16(x.q_rows) || !aligned16(x.M) || (x.A && !aligned16(x.A)))
            return fail(ctx, KVSEL_ERR_ALIGN, "memory_update_batch: session %d: pointers must be 16-byte aligned", i);
    }
    if (S == 0) return KVSEL_OK;
    void* ws = kvsel_workspace(ctx, memory_update_batch_workspace(S));
    if (!ws) return fail(ctx, KVSEL_ERR_CUDA, "memory_update_batch: workspace allocation failed");
    return launched(ctx, launch_memory_update_batch(q_dtype, L, Hq, D, norm_mode, sessions, S, ws, (cudaStream_t)stream),
                    "memory_update_batch launch");
}

int kvsel_rule_scores(kvsel_ctx* ctx, const void* k_pool, int k_dtype, const int32_t* slot_map, int n_slots,
                      int L, int Hq, int Hkv, int N, int D, int64_t layer_stride, int64_t slot_stride,
                      const float* M, int pi, int q_s, int q_e, float* rule, void* stream) {
    const kvsel_trace trace_("kvsel_rule_scores");
    int rc = enter(ctx);
    if (rc) return rc;
    rc = kvsel_check_rule_scores_args(ctx, "rule_scores", k_pool, k_dtype, slot_map, n_slots, L, Hq, Hkv, N, D,
                                      layer_stride, slot_stride, M, pi, q_s, q_e, rule);
    if (rc) return rc;
    if (N == 0) return KVSEL_OK;
    void* ws = kvsel_workspace(ctx, rule_scores_workspace(ctx, L, Hq, N));
    if (!ws) return fail(ctx, KVSEL_ERR_CUDA, "rule_scores: workspace allocation failed");
    return launched(ctx, launch_rule_scores(ctx, k_pool, k_dtype, slot_map, n_slots, L, Hq, Hkv, N, D, layer_stride,
                                            slot_stride, M, pi, q_s, q_e, rule, ws, (cudaStream_t)stream),
                    "rule_scores launch");
}

int kvsel_topk_retain(kvsel_ctx* ctx, const float* score, int N, int pi, int q_s, int q_e, int C, uint8_t* keep,
                      int32_t* keep_idx, int* n_keep_host, void* stream) {
    const kvsel_trace trace_("kvsel_topk_retain");
    int rc = enter(ctx);
    if (rc) return rc;
    if (!score || (!keep && !keep_idx)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "topk_retain: null score or no output");
    if (N < 0 || C < 0) return fail(ctx, KVSEL_ERR_SHAPE, "topk_retain: negative N or C");
    if (pi < 0 || pi > N || q_s < 0 || q_s > q_e || q_e > N) return fail(ctx, KVSEL_ERR_SHAPE, "topk_retain: forced ranges outside [0,N]");
    int64_t nF = forced_count(pi, q_s, q_e);
    int64_t nH = N - nF;
    int64_t cstar = C - nF > 0 ? C - nF : 0;
    int64_t need = cstar < nH ? cstar : nH;
    if (n_keep_host) *n_keep_host = (int)(nF + need);
    if (N == 0) return KVSEL_OK;
    void* ws = nullptr;
    if (const size_t wb = topk_workspace(N)) {
        if (!(ws = kvsel_workspace(ctx, wb))) return fail(ctx, KVSEL_ERR_CUDA, "topk_retain: workspace allocation failed");
    }
    return launched(ctx, launch_topk(score, N, pi, q_s, q_e, (int)need, (int)nH, keep, keep_idx, ws, (cudaStream_t)stream),
                    "topk_retain launch");
}

int kvsel_topk_retain_batch(kvsel_ctx* ctx, const kvsel_topk_session* sessions, int S, int* n_keep_host,
                            void* stream) {
    const kvsel_trace trace_("kvsel_topk_retain_batch");
    int rc = enter(ctx);
    if (rc) return rc;
    if (S < 0 || (S > 0 && !sessions)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "topk_retain_batch: bad session table");
    std::vector<int> need((size_t)S), n_cand((size_t)S);
    int max_N = 0;
    for (int i = 0; i < S; ++i) {
        const kvsel_topk_session& x = sessions[i];
        if (!x.rule || (!x.keep && !x.keep_idx)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "topk_retain_batch: session %d: null score or no output", i);
        if (x.N < 0 || x.C < 0) return fail(ctx, KVSEL_ERR_SHAPE, "topk_retain_batch: session %d: negative N or C", i);
        if (x.pi < 0 || x.pi > x.N || x.q_s < 0 || x.q_s > x.q_e || x.q_e > x.N)
            return fail(ctx, KVSEL_ERR_SHAPE, "topk_retain_batch: session %d: forced ranges outside [0,N]", i);
        const int64_t nF = forced_count(x.pi, x.q_s, x.q_e), nH = x.N - nF;
        const int64_t cstar = x.C - nF > 0 ? x.C - nF : 0;
        need[i] = (int)(cstar < nH ? cstar : nH);
        n_cand[i] = (int)nH;
        if (x.N > max_N) max_N = x.N;
        if (n_keep_host) n_keep_host[i] = (int)(nF + need[i]);
    }
    if (S == 0) return KVSEL_OK;
    void* ws = kvsel_workspace(ctx, topk_batch_workspace(S, max_N));
    if (!ws) return fail(ctx, KVSEL_ERR_CUDA, "topk_retain_batch: workspace allocation failed");
    return launched(ctx, launch_topk_batch(sessions, need.data(), n_cand.data(), S, ws, (cudaStream_t)stream),
                    "topk_retain_batch launch");
}

int kvsel_rule_scores_batch(kvsel_ctx* ctx, const void* k_pool, int k_dtype, int n_slots, int L, int Hq, int Hkv,
                            int D, int64_t layer_stride, int64_t slot_stride, const kvsel_rule_session* sessions,
                            int S, void* stream) {
    const kvsel_trace trace_("kvsel_rule_scores_batch");
    int rc = enter(ctx);
    if (rc) return rc;
    if (!k_pool || (S > 0 && !sessions)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "rule_scores_batch: null pointer");
    if (S < 0 || S > 65535) return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_batch: S=%d outside [0, 65535]", S);
    if (k_dtype != KVSEL_F32 && k_dtype != KVSEL_BF16) return fail(ctx, KVSEL_ERR_INVALID_ARG, "rule_scores_batch: bad dtype");
    if (L <= 0 || Hq <= 0 || Hkv <= 0 || n_slots < 0) return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_batch: bad sizes");
    if (Hq % Hkv) return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_batch: Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
    if (Hq / Hkv > 8) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "rule_scores_batch: group size Hq/Hkv=%d > 8", Hq / Hkv);
    if (!pow2_head_dim(D)) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "rule_scores_batch: D=%d unsupported", D);
    if ((int64_t)Hkv * D > 4096) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "rule_scores_batch: Hkv*D > 4096");
    if (slot_stride < (int64_t)Hkv * D || layer_stride < 0) return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_batch: slot_stride < Hkv*D");
    if (L > 1 && layer_stride < (int64_t)n_slots * slot_stride) return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_batch: layers overlap");
    size_t es = k_dtype == KVSEL_BF16 ? 2 : 4;
    if (!aligned16(k_pool) || (layer_stride * es) % 16 || (slot_stride * es) % 16)
        return fail(ctx, KVSEL_ERR_ALIGN, "rule_scores_batch: pool and strides must be 16-byte aligned");
    for (int i = 0; i < S; ++i) {
        const kvsel_rule_session& x = sessions[i];
        if (x.N < 0) return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_batch: session %d: negative N", i);
        if (x.N > 0 && (!x.M || !x.rule)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "rule_scores_batch: session %d: null pointer", i);
        if (x.pi < 0 || x.pi > x.N || x.q_s < 0 || x.q_s > x.q_e || x.q_e > x.N)
            return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_batch: session %d: forced ranges outside [0,N]", i);
        if (!x.slot_map && n_slots < x.N) return fail(ctx, KVSEL_ERR_SHAPE, "rule_scores_batch: session %d: identity slot map needs n_slots >= N", i);
        if (x.N > 0 && (!aligned16(x.M) || !aligned16(x.rule)))
            return fail(ctx, KVSEL_ERR_ALIGN, "rule_scores_batch: session %d: M and rule must be 16-byte aligned", i);
    }
    if (S == 0) return KVSEL_OK;
    void* ws = kvsel_workspace(ctx, rule_scores_batch_workspace(L, Hq, sessions, S));
    if (!ws) return fail(ctx, KVSEL_ERR_CUDA, "rule_scores_batch: workspace allocation failed");
    return launched(ctx, launch_rule_scores_batch(ctx, k_pool, k_dtype, n_slots, L, Hq, Hkv, D, layer_stride, slot_stride,
                                                  sessions, S, ws, (cudaStream_t)stream),
                    "rule_scores_batch launch");
}

int kvsel_redirect_slots(kvsel_ctx* ctx, const int32_t* slot_in, const uint8_t* keep, int N, int32_t dead_slot,
                         int32_t* slot_out, void* stream) {
    const kvsel_trace trace_("kvsel_redirect_slots");
    int rc = enter(ctx);
    if (rc) return rc;
    if (!slot_in || !keep || !slot_out) return fail(ctx, KVSEL_ERR_INVALID_ARG, "redirect_slots: null pointer");
    if (N < 0) return fail(ctx, KVSEL_ERR_SHAPE, "redirect_slots: negative N");
    if (N == 0) return KVSEL_OK;
    return launched(ctx, launch_redirect(slot_in, keep, N, dead_slot, slot_out, (cudaStream_t)stream), "redirect_slots launch");
}

int kvsel_span_keep(kvsel_ctx* ctx, const int32_t* span_start, const int32_t* span_end, int n_cursors,
                    const int32_t* del_ids, int n_del, const uint8_t* keep_in, int N, uint8_t* keep_out, void* stream) {
    const kvsel_trace trace_("kvsel_span_keep");
    int rc = enter(ctx);
    if (rc) return rc;
    if (N < 0 || n_cursors < 0 || n_del < 0) return fail(ctx, KVSEL_ERR_SHAPE, "span_keep: negative size");
    if (!keep_out || (n_del > 0 && !del_ids) || (n_cursors > 0 && (!span_start || !span_end)))
        return fail(ctx, KVSEL_ERR_INVALID_ARG, "span_keep: null pointer");
    if (N == 0) return KVSEL_OK;
    return launched(ctx, launch_span_keep(span_start, span_end, n_cursors, del_ids, n_del, keep_in, N, keep_out,
                                          ctx->dev_err, (cudaStream_t)stream),
                    "span_keep launch");
}

int kvsel_index_to_fp8(kvsel_ctx* ctx, const void* index, int64_t rows, int D, uint8_t* codes, int8_t* exps,
                       void* stream) {
    const kvsel_trace trace_("kvsel_index_to_fp8");
    int rc = enter(ctx);
    if (rc) return rc;
    if (rows < 0) return fail(ctx, KVSEL_ERR_SHAPE, "index_to_fp8: negative row count");
    if (D != 64 && D != 128 && D != 256) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "index_to_fp8: D=%d unsupported", D);
    if (rows == 0) return KVSEL_OK;
    if (!index || !codes || !exps) return fail(ctx, KVSEL_ERR_INVALID_ARG, "index_to_fp8: null pointer");
    if (!aligned16(index) || (reinterpret_cast<uintptr_t>(codes) & 3u))
        return fail(ctx, KVSEL_ERR_ALIGN, "index_to_fp8: index must be 16-byte and codes 4-byte aligned");
    return launched(ctx, launch_index_to_fp8(ctx, index, rows, D, codes, exps, (cudaStream_t)stream),
                    "index_to_fp8 launch");
}

int kvsel_index_from_fp8(kvsel_ctx* ctx, const uint8_t* codes, const int8_t* exps, int64_t rows, int D, void* index,
                         void* stream) {
    const kvsel_trace trace_("kvsel_index_from_fp8");
    int rc = enter(ctx);
    if (rc) return rc;
    if (rows < 0) return fail(ctx, KVSEL_ERR_SHAPE, "index_from_fp8: negative row count");
    if (D != 64 && D != 128 && D != 256) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "index_from_fp8: D=%d unsupported", D);
    if (rows == 0) return KVSEL_OK;
    if (!index || !codes || !exps) return fail(ctx, KVSEL_ERR_INVALID_ARG, "index_from_fp8: null pointer");
    if (!aligned16(index) || (reinterpret_cast<uintptr_t>(codes) & 3u))
        return fail(ctx, KVSEL_ERR_ALIGN, "index_from_fp8: index must be 16-byte and codes 4-byte aligned");
    return launched(ctx, launch_index_from_fp8(ctx, codes, exps, rows, D, index, (cudaStream_t)stream),
                    "index_from_fp8 launch");
}

int kvsel_meank_build(kvsel_ctx* ctx, const void* k_src, int L, int Hkv, int T, int D, int block, int first_block,
                      const int32_t* src_pos, double rope_base, int rope_style, void* index, int Bcap, void* stream) {
    const kvsel_trace trace_("kvsel_meank_build");
    int rc = enter(ctx);
    if (rc) return rc;
    if (!k_src || !index) return fail(ctx, KVSEL_ERR_INVALID_ARG, "meank_build: null pointer");
    if (L <= 0 || Hkv <= 0 || T < 0 || block <= 0 || first_block < 0 || Bcap <= 0) return fail(ctx, KVSEL_ERR_SHAPE, "meank_build: bad sizes");
    if (!pow2_head_dim(D)) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "meank_build: D=%d unsupported", D);
    int64_t nb = ((int64_t)T + block - 1) / block;
    if (first_block + nb > Bcap) return fail(ctx, KVSEL_ERR_SHAPE, "meank_build: blocks [%d,%lld) exceed Bcap=%d", first_block, (long long)(first_block + nb), Bcap);
    if (src_pos && (rope_style != KVSEL_ROPE_NEOX && rope_style != KVSEL_ROPE_INTERLEAVED)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "meank_build: bad rope_style");
    if (src_pos && !(rope_base > 1.0)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "meank_build: rope_base must be > 1");
    if (!aligned16(k_src) || !aligned16(index)) return fail(ctx, KVSEL_ERR_ALIGN, "meank_build: pointers must be 16-byte aligned");
    if (T == 0) return KVSEL_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const kvsel_ctx::RopeTab* tab = nullptr;
    if (src_pos) {
        tab = kvsel_rope_tables(ctx, D, rope_base, s);
        if (!tab) return fail(ctx, KVSEL_ERR_CUDA, "meank_build: rope table allocation failed");
    }
    return launched(ctx, launch_meank(k_src, L, Hkv, T, D, block, first_block, src_pos, tab, rope_style, index, Bcap,
                                      ctx->dev_err, s),
                    "meank_build launch");
}

// kvsel_block_scores with the bounded waits' limit and the give-up test hook as arguments.
static int block_scores_call(kvsel_ctx* ctx, const void* q, const void* index, int L, int Hq, int Hkv, int M, int D,
                      int n_blocks, int Bcap, int n_sink, int n_recent, float* R, float* R_partial, void* stream,
                      uint64_t wait_ns, int stuck) {
    int rc = enter(ctx);
    if (rc) return rc;
    if (!q || !index || !R) return fail(ctx, KVSEL_ERR_INVALID_ARG, "block_scores: null pointer");
    if (L <= 0 || Hq <= 0 || Hkv <= 0 || M <= 0 || n_blocks < 0 || Bcap < n_blocks || n_sink < 0 || n_recent < 0)
        return fail(ctx, KVSEL_ERR_SHAPE, "block_scores: bad sizes");
    if (Hq % Hkv) return fail(ctx, KVSEL_ERR_SHAPE, "block_scores: Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
    if (D != 128) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "block_scores: D=%d unsupported (128 only)", D);
    if (!aligned16(q) || !aligned16(index) || !aligned16(R) || (R_partial && !aligned16(R_partial)))
        return fail(ctx, KVSEL_ERR_ALIGN, "block_scores: pointers must be 16-byte aligned");
    if (n_blocks == 0) return KVSEL_OK;
    void* ws = kvsel_workspace(ctx, block_scores_workspace(L, Hq, Hkv, M, n_blocks));
    if (!ws) return fail(ctx, KVSEL_ERR_CUDA, "block_scores: workspace allocation failed");
    return launched(ctx, launch_block_scores(ctx, q, index, L, Hq, Hkv, M, D, n_blocks, Bcap, n_sink, n_recent, R,
                                             R_partial, ws, (cudaStream_t)stream, wait_ns, stuck),
                    "block_scores launch");
}

int kvsel_block_scores(kvsel_ctx* ctx, const void* q, const void* index, int L, int Hq, int Hkv, int M, int D,
                       int n_blocks, int Bcap, int n_sink, int n_recent, float* R, float* R_partial, void* stream) {
    const kvsel_trace trace_("kvsel_block_scores");
    return block_scores_call(ctx, q, index, L, Hq, Hkv, M, D, n_blocks, Bcap, n_sink, n_recent, R, R_partial, stream,
                             KVSEL_BLOCK_WAIT_NS, 0);
}

// Test entry (not part of the public header): kvsel_block_scores in which the row
// pass's first MMA issuer of every CTA waits on a barrier that nothing completes,
// with every bounded wait of the row pass limited to wait_ns.  That wait gives up while copies and
// MMAs are in flight, so the call exercises the tensor-core kernel's give-up path:
// flag KVSEL_ERR_TIMEOUT in the device error word, drain its own copies and MMAs
// (bounded waits), free TMEM and return.  R holds no meaningful values afterwards;
// kvsel_check_device reports KVSEL_ERR_TIMEOUT.
int kvsel_test_block_scores_give_up(kvsel_ctx* ctx, const void* q, const void* index, int L, int Hq, int Hkv, int M,
                                    int D, int n_blocks, int Bcap, int n_sink, int n_recent, float* R,
                                    uint64_t wait_ns, void* stream) {
    const kvsel_trace trace_("kvsel_test_block_scores_give_up");
    if (wait_ns == 0 || wait_ns > KVSEL_BLOCK_WAIT_NS)
        return fail(ctx, KVSEL_ERR_INVALID_ARG, "test_block_scores_give_up: wait_ns must be in (0, 1 s]");
    return block_scores_call(ctx, q, index, L, Hq, Hkv, M, D, n_blocks, Bcap, n_sink, n_recent, R, nullptr, stream,
                             wait_ns, 1);
}

int kvsel_select_blocks(kvsel_ctx* ctx, const float* R, int n_blocks, int n_sink, int n_recent, int k, int32_t* ids,
                        int* n_sel_host, void* stream) {
    const kvsel_trace trace_("kvsel_select_blocks");
    int rc = enter(ctx);
    if (rc) return rc;
    if (!R || !ids) return fail(ctx, KVSEL_ERR_INVALID_ARG, "select_blocks: null pointer");
    if (n_blocks < 0 || n_sink < 0 || n_recent < 0 || k < 0) return fail(ctx, KVSEL_ERR_SHAPE, "select_blocks: negative size");
    int S = n_sink < n_blocks ? n_sink : n_blocks;
    int q_s = n_blocks - n_recent > 0 ? n_blocks - n_recent : 0;
    int64_t nF = forced_count(S, q_s, n_blocks);
    int64_t nC = n_blocks - nF;
    int64_t need = k < nC ? k : nC;
    if (n_sel_host) *n_sel_host = (int)(nF + need);
    if (n_blocks == 0) return KVSEL_OK;
    void* ws = nullptr;
    if (const size_t wb = topk_workspace(n_blocks)) {
        if (!(ws = kvsel_workspace(ctx, wb))) return fail(ctx, KVSEL_ERR_CUDA, "select_blocks: workspace allocation failed");
    }
    return launched(ctx, launch_topk(R, n_blocks, S, q_s, n_blocks, (int)need, (int)nC, nullptr, ids, ws, (cudaStream_t)stream),
                    "select_blocks launch");
}

int kvsel_rerope_scatter(kvsel_ctx* ctx, const void* k_src, int64_t src_layer_stride, int64_t src_head_stride,
                         int src_tokens, const int32_t* src_block, const int32_t* dst_page, const int32_t* dst_pos0,
                         int n, int L, int Hkv, int D, int page, double rope_base, int rope_style, void* pool, int P,
                         void* stream) {
    const kvsel_trace trace_("kvsel_rerope_scatter");
    int rc = enter(ctx);
    if (rc) return rc;
    if (!k_src || !src_block || !dst_page || !dst_pos0 || !pool) return fail(ctx, KVSEL_ERR_INVALID_ARG, "rerope_scatter: null pointer");
    if (n < 0 || L <= 0 || Hkv <= 0 || page <= 0 || P <= 0 || src_tokens < 0) return fail(ctx, KVSEL_ERR_SHAPE, "rerope_scatter: bad sizes");
    if (!pow2_head_dim(D)) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "rerope_scatter: D=%d unsupported", D);
    if ((int64_t)page * D > 16384) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "rerope_scatter: page*D=%lld > 16384", (long long)page * D);
    if (rope_style != KVSEL_ROPE_NEOX && rope_style != KVSEL_ROPE_INTERLEAVED) return fail(ctx, KVSEL_ERR_INVALID_ARG, "rerope_scatter: bad rope_style");
    if (!(rope_base > 1.0)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "rerope_scatter: rope_base must be > 1");
    if (src_head_stride < (int64_t)src_tokens * D || src_layer_stride < 0) return fail(ctx, KVSEL_ERR_SHAPE, "rerope_scatter: head stride < src_tokens*D");
    if (!aligned16(k_src) || !aligned16(pool) || (src_layer_stride * 2) % 16 || (src_head_stride * 2) % 16)
        return fail(ctx, KVSEL_ERR_ALIGN, "rerope_scatter: pointers and strides must be 16-byte aligned");
    if (n == 0) return KVSEL_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const kvsel_ctx::RopeTab* tab = kvsel_rope_tables(ctx, D, rope_base, s);
    if (!tab) return fail(ctx, KVSEL_ERR_CUDA, "rerope_scatter: rope table allocation failed");
    return launched(ctx, launch_rerope(k_src, src_layer_stride, src_head_stride, src_tokens, src_block, dst_page, dst_pos0,
                                       n, nullptr, L, Hkv, D, page, tab, rope_style, pool, nullptr, nullptr, P,
                                       ctx->dev_err, s),
                    "rerope_scatter launch");
}

int kvsel_workset_diff(kvsel_ctx* ctx, const int32_t* prev_ids, const int32_t* prev_pages, int n_prev,
                       const int32_t* new_ids, int n_new, int P, int page, int32_t* new_pages, int32_t* shift,
                       int32_t* in_rank, int32_t* in_page, int32_t* mv_rank, int32_t* mv_shift, int32_t* out_page,
                       int32_t* counts, void* stream) {
    const kvsel_trace trace_("kvsel_workset_diff");
    int rc = enter(ctx);
    if (rc) return rc;
    if (n_prev < 0 || n_new < 0 || P <= 0 || page <= 0) return fail(ctx, KVSEL_ERR_SHAPE, "workset_diff: bad sizes");
    if (P > (1 << 20)) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "workset_diff: P=%d > 2^20 pages", P);
    if (n_prev > P || n_new > P) return fail(ctx, KVSEL_ERR_SHAPE, "workset_diff: a working set larger than the pool");
    if ((int64_t)P * page >= KVSEL_MAX_POS) return fail(ctx, KVSEL_ERR_SHAPE, "workset_diff: P*page must stay below 2^24 positions");
    if ((n_prev > 0 && (!prev_ids || !prev_pages || !out_page)) ||
        (n_new > 0 && (!new_ids || !new_pages || !shift || !in_rank || !in_page || !mv_rank || !mv_shift)) || !counts)
        return fail(ctx, KVSEL_ERR_INVALID_ARG, "workset_diff: null pointer");
    return launched(ctx, launch_workset_diff(prev_ids, prev_pages, n_prev, new_ids, n_new, P, page, new_pages, shift,
                                             in_rank, in_page, mv_rank, mv_shift, out_page, counts, ctx->dev_err,
                                             (cudaStream_t)stream),
                    "workset_diff launch");
}

int kvsel_restore_blocks(kvsel_ctx* ctx, const void* k_src, const void* v_src, int64_t src_layer_stride,
                         int64_t src_head_stride, int src_tokens, const int32_t* src_block, const int32_t* dst_page,
                         const int32_t* dst_pos0, int n, const int32_t* n_dev, int L, int Hkv, int D, int page,
                         double rope_base, int rope_style, void* k_pool, void* v_pool, int P, void* stream) {
    const kvsel_trace trace_("kvsel_restore_blocks");
    int rc = enter(ctx);
    if (rc) return rc;
    if (!k_src || !v_src || !src_block || !dst_page || !dst_pos0 || !k_pool || !v_pool)
        return fail(ctx, KVSEL_ERR_INVALID_ARG, "restore_blocks: null pointer");
    if (n < 0 || L <= 0 || Hkv <= 0 || page <= 0 || P <= 0 || src_tokens < 0) return fail(ctx, KVSEL_ERR_SHAPE, "restore_blocks: bad sizes");
    if (!pow2_head_dim(D)) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "restore_blocks: D=%d unsupported", D);
    if ((int64_t)page * D > 16384) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "restore_blocks: page*D=%lld > 16384", (long long)page * D);
    if (rope_style != KVSEL_ROPE_NEOX && rope_style != KVSEL_ROPE_INTERLEAVED) return fail(ctx, KVSEL_ERR_INVALID_ARG, "restore_blocks: bad rope_style");
    if (!(rope_base > 1.0)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "restore_blocks: rope_base must be > 1");
    if (src_head_stride < (int64_t)src_tokens * D || src_layer_stride < 0) return fail(ctx, KVSEL_ERR_SHAPE, "restore_blocks: head stride < src_tokens*D");
    if (!aligned16(k_src) || !aligned16(v_src) || !aligned16(k_pool) || !aligned16(v_pool) || (src_layer_stride * 2) % 16 ||
        (src_head_stride * 2) % 16)
        return fail(ctx, KVSEL_ERR_ALIGN, "restore_blocks: pointers and strides must be 16-byte aligned");
    if (n == 0) return KVSEL_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const kvsel_ctx::RopeTab* tab = kvsel_rope_tables(ctx, D, rope_base, s);
    if (!tab) return fail(ctx, KVSEL_ERR_CUDA, "restore_blocks: rope table allocation failed");
    return launched(ctx, launch_rerope(k_src, src_layer_stride, src_head_stride, src_tokens, src_block, dst_page, dst_pos0,
                                       n, n_dev, L, Hkv, D, page, tab, rope_style, k_pool, v_src, v_pool, P,
                                       ctx->dev_err, s),
                    "restore_blocks launch");
}

int kvsel_rerope_shift(kvsel_ctx* ctx, void* pool, int P, const int32_t* pages, const int32_t* shifts, int n,
                       const int32_t* n_dev, int L, int Hkv, int D, int page, double rope_base, int rope_style,
                       void* stream) {
    const kvsel_trace trace_("kvsel_rerope_shift");
    int rc = enter(ctx);
    if (rc) return rc;
    if (!pool || !pages || !shifts) return fail(ctx, KVSEL_ERR_INVALID_ARG, "rerope_shift: null pointer");
    if (n < 0 || L <= 0 || Hkv <= 0 || page <= 0 || P <= 0) return fail(ctx, KVSEL_ERR_SHAPE, "rerope_shift: bad sizes");
    if (!pow2_head_dim(D)) return fail(ctx, KVSEL_ERR_UNSUPPORTED, "rerope_shift: D=%d unsupported", D);
    if (rope_style != KVSEL_ROPE_NEOX && rope_style != KVSEL_ROPE_INTERLEAVED) return fail(ctx, KVSEL_ERR_INVALID_ARG, "rerope_shift: bad rope_style");
    if (!(rope_base > 1.0)) return fail(ctx, KVSEL_ERR_INVALID_ARG, "rerope_shift: rope_base must be > 1");
    if (!aligned16(pool)) return fail(ctx, KVSEL_ERR_ALIGN, "rerope_shift: pool must be 16-byte aligned");
    if (n == 0) return KVSEL_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const kvsel_ctx::RopeTab* tab = kvsel_rope_tables(ctx, D, rope_base, s);
    if (!tab) return fail(ctx, KVSEL_ERR_CUDA, "rerope_shift: rope table allocation failed");
    return launched(ctx, launch_shift(pool, P, pages, shifts, n, n_dev, L, Hkv, D, page, tab, rope_style, ctx->dev_err, s),
                    "rerope_shift launch");
}

}  // extern "C"

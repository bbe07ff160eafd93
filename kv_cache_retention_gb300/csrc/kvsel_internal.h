// Internal declarations shared by the libkvsel translation units (not part of
// the public ABI; see include/kvsel.h for the calls and their contracts).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#include "../../include/kvsel.h"

struct kvsel_ctx {
    int device = 0;
    int num_sms = 0;
    // Scratch workspace; grows on demand (see kvsel.h "Scratch").
    void* ws = nullptr;
    size_t ws_bytes = 0;
    // Device error word: kernels OR kvsel_devcheck bits into it on bad data.
    unsigned* dev_err = nullptr;
    // RoPE angle tables, one per (D, base): split-position cos/sin pairs, in
    // fp32 for the fast path and as double-floats for outputs that nearly cancel.
    struct RopeTab {
        int D = 0;
        double base = 0.0;
        float2* lo = nullptr;     // [KVSEL_ROPE_LO][D/2]: angle lo * theta_i
        float2* hi = nullptr;     // [KVSEL_ROPE_HI][D/2]: angle hi * LO * theta_i
        float4* lodf = nullptr;   // the same angles as double-floats (cos hi, cos lo, sin hi, sin lo)
        float4* hidf = nullptr;
    };
    RopeTab rope[8];
    int n_rope = 0;
    // Host -> device staging of kvsel_stage_restore: two slots of a pinned and a
    // device buffer, and a copy stream; grown on demand, freed with the context.
    struct Stager {
        struct Slot {
            void* host = nullptr;
            void* dev = nullptr;
            cudaEvent_t copied = nullptr;    // the slot's last copy has left the host buffer
            cudaEvent_t consumed = nullptr;  // the slot's last kernel has read the device buffer
        } slot[2];
        cudaStream_t copy_stream = nullptr;
        size_t capacity = 0;
    } stager;
    // Device address of the fixed scratch array of kvsel_rule_scores_noalloc on
    // this context's device, looked up by that call's first use on the context.
    void* noalloc_scratch = nullptr;
    char err[512] = {0};
};

// Device error-word bits.
enum kvsel_devcheck : unsigned {
    KVSEL_DEV_BAD_SLOT = 1u << 0,
    KVSEL_DEV_BAD_POSITION = 1u << 1,
    KVSEL_DEV_BAD_BLOCK = 1u << 2,
    KVSEL_DEV_BAD_PAGE = 1u << 3,
    KVSEL_DEV_BAD_SET = 1u << 4,   // a working set not ascending, or a page held twice
    KVSEL_DEV_POOL_FULL = 1u << 5, // fewer free pages than incoming blocks
    KVSEL_DEV_TIMEOUT = 1u << 8,  // a bounded wait inside a kernel gave up
};

// Positions p are split as p = hi * KVSEL_ROPE_LO + lo; both tables in fp64 -> fp32.
#define KVSEL_ROPE_LO_BITS 10
#define KVSEL_ROPE_LO (1 << KVSEL_ROPE_LO_BITS)
#define KVSEL_ROPE_HI (1 << 14)
#define KVSEL_MAX_POS (KVSEL_ROPE_LO * KVSEL_ROPE_HI)  // 2^24

// NVTX range around one C-ABI call, named after the call, for profilers and
// tracers.  Off unless the environment variable KVSEL_NVTX is set to 1 when the
// library first checks it; then every kvsel_* call that launches work pushes a
// range on entry and pops it on return.
inline bool kvsel_nvtx_on() {
    static const bool on = [] {
        const char* v = getenv("KVSEL_NVTX");
        return v && v[0] == '1' && v[1] == 0;
    }();
    return on;
}
struct kvsel_trace {
    const bool on;
    explicit kvsel_trace(const char* name) : on(kvsel_nvtx_on()) {
        if (on) nvtxRangePushA(name);
    }
    ~kvsel_trace() {
        if (on) nvtxRangePop();
    }
    kvsel_trace(const kvsel_trace&) = delete;
    kvsel_trace& operator=(const kvsel_trace&) = delete;
};

// Error helpers shared by the translation units that implement calls:
// entry guard, formatted failure (sets the context's error string), CUDA failure.
int kvsel_enter(kvsel_ctx* ctx);
int kvsel_fail(kvsel_ctx* ctx, int code, const char* fmt, ...);
int kvsel_cuda_fail(kvsel_ctx* ctx, cudaError_t e, const char* what);
// The argument rules of kvsel_rule_scores (shared by its no-allocation variant);
// KVSEL_OK or the failure code, with `who` leading the error string.
int kvsel_check_rule_scores_args(kvsel_ctx* ctx, const char* who, const void* k_pool, int k_dtype,
                                 const int32_t* slot_map, int n_slots, int L, int Hq, int Hkv, int N, int D,
                                 int64_t layer_stride, int64_t slot_stride, const float* M, int pi, int q_s, int q_e,
                                 const float* rule);
// Frees the staging buffers, events and copy stream of kvsel_stage_restore.
void kvsel_stager_release(kvsel_ctx* ctx);

// Returns a pointer into the context workspace of at least `bytes` (256-byte
// aligned), growing it if needed; nullptr on allocation failure.
void* kvsel_workspace(kvsel_ctx* ctx, size_t bytes);
// Finds or builds the RoPE tables for (D, base); nullptr on failure.
const kvsel_ctx::RopeTab* kvsel_rope_tables(kvsel_ctx* ctx, int D, double base, cudaStream_t s);

// ---- launchers (return cudaGetLastError() of their launches) ---------------

size_t memory_update_batch_workspace(int S);
cudaError_t launch_memory_update_batch(int dtype, int L, int Hq, int D, int norm_mode, const kvsel_memory_session* sess,
                                       int S, void* ws, cudaStream_t s);
cudaError_t launch_memory_update(const void* q, int dtype, int L, int Hq, int R, int D, float lambda,
                                 int first_turn, int norm_mode, float* M, float* A, cudaStream_t s);

size_t rule_scores_batch_workspace(int L, int Hq, const kvsel_rule_session* sess, int S);
cudaError_t launch_rule_scores_batch(kvsel_ctx* ctx, const void* k_pool, int dtype, int n_slots, int L, int Hq,
                                     int Hkv, int D, int64_t layer_stride, int64_t slot_stride,
                                     const kvsel_rule_session* sess, int S, void* ws, cudaStream_t s);
cudaError_t launch_rule_scores(kvsel_ctx* ctx, const void* k_pool, int dtype, const int32_t* slot_map,
                               int n_slots, int L, int Hq, int Hkv, int N, int D, int64_t layer_stride,
                               int64_t slot_stride, const float* M, int pi, int q_s, int q_e,
                               float* rule, void* ws, cudaStream_t s);
size_t rule_scores_workspace(kvsel_ctx* ctx, int L, int Hq, int N);

// need: how many of the non-forced positions to keep by score (0..|H|).
// Workspace of the grid-wide selection for sessions longer than one cluster holds (0 below).
size_t topk_workspace(int N);
size_t topk_batch_workspace(int S, int max_N);
cudaError_t launch_topk_batch(const kvsel_topk_session* sess, const int* need, const int* n_cand, int S, void* ws,
                              cudaStream_t s);
cudaError_t launch_topk(const float* score, int N, int pi, int q_s, int q_e, int need, int n_cand,
                        uint8_t* keep, int32_t* keep_idx, void* ws, cudaStream_t s);

cudaError_t launch_redirect(const int32_t* slot_in, const uint8_t* keep, int N, int32_t dead,
                            int32_t* slot_out, cudaStream_t s);

cudaError_t launch_rope_tables(float2* lo, float2* hi, float4* lodf, float4* hidf, int D, double base,
                               cudaStream_t s);

cudaError_t launch_meank(const void* k_src, int L, int Hkv, int T, int D, int block, int first_block,
                         const int32_t* src_pos, const kvsel_ctx::RopeTab* tab, int rope_style,
                         void* index, int Bcap, unsigned* dev_err, cudaStream_t s);

cudaError_t launch_rerope(const void* k_src, int64_t sls, int64_t shs, int src_tokens, const int32_t* src_block,
                          const int32_t* dst_page, const int32_t* dst_pos0, int n, const int32_t* n_dev, int L,
                          int Hkv, int D, int page, const kvsel_ctx::RopeTab* tab, int rope_style, void* pool,
                          const void* v_src, void* v_pool, int P, unsigned* dev_err, cudaStream_t s);
cudaError_t launch_shift(void* pool, int P, const int32_t* pages, const int32_t* shifts, int n, const int32_t* n_dev,
                         int L, int Hkv, int D, int page, const kvsel_ctx::RopeTab* tab, int rope_style,
                         unsigned* dev_err, cudaStream_t s);
cudaError_t launch_index_to_fp8(const kvsel_ctx* ctx, const void* index, int64_t rows, int D, uint8_t* codes,
                                int8_t* exps, cudaStream_t s);
cudaError_t launch_index_from_fp8(const kvsel_ctx* ctx, const uint8_t* codes, const int8_t* exps, int64_t rows, int D,
                                  void* index, cudaStream_t s);
cudaError_t launch_span_keep(const int32_t* span_start, const int32_t* span_end, int n_cursors, const int32_t* del_ids,
                             int n_del, const uint8_t* keep_in, int N, uint8_t* keep_out, unsigned* dev_err,
                             cudaStream_t s);
cudaError_t launch_workset_diff(const int32_t* prev_ids, const int32_t* prev_pages, int n_prev,
                                const int32_t* new_ids, int n_new, int P, int page, int32_t* new_pages,
                                int32_t* shift, int32_t* in_rank, int32_t* in_page, int32_t* mv_rank,
                                int32_t* mv_shift, int32_t* out_page, int32_t* counts, unsigned* dev_err,
                                cudaStream_t s);

// wait_ns: how long a bounded wait inside the tensor-core kernels waits before it
// gives up (KVSEL_BLOCK_WAIT_NS in normal calls); stuck: test hook, see
// kvsel_test_block_scores_give_up.
constexpr uint64_t KVSEL_BLOCK_WAIT_NS = 1000000000ull;
cudaError_t launch_block_scores(kvsel_ctx* ctx, const void* q, const void* index, int L, int Hq, int Hkv,
                                int M, int D, int n_blocks, int Bcap, int n_sink, int n_recent, float* R,
                                float* R_partial, void* ws, cudaStream_t s, uint64_t wait_ns = KVSEL_BLOCK_WAIT_NS,
                                int stuck = 0);
size_t block_scores_workspace(int L, int Hq, int Hkv, int M, int n_blocks);
// The driver's cuTensorMapEncodeTiled (looked up once), or nullptr.
PFN_cuTensorMapEncodeTiled_v12000 kvsel_tmap_encoder();

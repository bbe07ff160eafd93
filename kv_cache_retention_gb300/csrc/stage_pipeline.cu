// KVMEM packed and pipelined rematerialisation (section "engineering: tiered
// movement, page-table aliasing and position-consistent rebuild"): the blocks
// to restore lie scattered in a host repository; they are gathered into one
// contiguous pinned buffer per batch, moved host -> device in one copy per
// batch, and re-RoPE'd / scattered into the page pool on the GPU, with the CPU
// gather, the copy and the GPU work of adjacent batches overlapped.
//
// Per batch (two slots, alternating):
//   host   wait until the slot's previous copy has left the pinned buffer, then
//          gather the batch's K rows, V rows and entry arrays into it (a few
//          threads, one contiguous page of rows per memcpy)
//   copy   on the context's copy stream, after the slot's previous kernel has
//          finished reading the device buffer: one cudaMemcpyAsync
//   GPU    on the caller's stream, after the copy: the restore kernel (K re-RoPE
//          + V copy) reading the device buffer
// The call returns once every batch is gathered and queued; the GPU work stays
// asynchronous on the caller's stream.
//
// Direct path: when both repositories are pinned and mapped (the runtime gives
// a device pointer for them), the GPU reaches host memory itself -- over
// NVLink-C2C on a Grace host -- and the restore kernel gathers, re-rotates and
// scatters straight from it: no CPU gather, no staging copy.  Only the three
// entry arrays go through the pinned slot, which the kernel reads in place.
#include <algorithm>
#include <cstring>
#include <thread>
#include <vector>

#include "kvsel_internal.h"

namespace {

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// Byte layout of one batch of nb blocks in a slot (host and device alike):
// K [L][Hkv][nb*page][D] bf16, V likewise, then src_block, dst_page, dst_pos0.
struct BatchLayout {
    size_t k_off, v_off, sb_off, dp_off, d0_off, bytes;
    BatchLayout(int nb, int L, int Hkv, int D, int page) {
        const size_t kv = (size_t)L * Hkv * nb * page * D * 2;
        k_off = 0;
        v_off = up(kv);
        sb_off = v_off + up(kv);
        dp_off = sb_off + up((size_t)nb * 4);
        d0_off = dp_off + up((size_t)nb * 4);
        bytes = d0_off + up((size_t)nb * 4);
    }
};

}  // namespace

void kvsel_stager_release(kvsel_ctx* ctx) {
    auto& st = ctx->stager;
    for (auto& s : st.slot) {
        if (s.host) cudaFreeHost(s.host);
        if (s.dev) cudaFree(s.dev);
        if (s.copied) cudaEventDestroy(s.copied);
        if (s.consumed) cudaEventDestroy(s.consumed);
        s = kvsel_ctx::Stager::Slot();
    }
    if (st.copy_stream) cudaStreamDestroy(st.copy_stream);
    st.copy_stream = nullptr;
    st.capacity = 0;
}

// Make both slots hold at least `bytes`; waits for any queued use of the old buffers.
static cudaError_t stager_reserve(kvsel_ctx* ctx, size_t bytes) {
    auto& st = ctx->stager;
    cudaError_t e;
    if (!st.copy_stream && (e = cudaStreamCreateWithFlags(&st.copy_stream, cudaStreamNonBlocking)) != cudaSuccess)
        return e;
    for (auto& s : st.slot) {
        if (!s.copied && (e = cudaEventCreateWithFlags(&s.copied, cudaEventDisableTiming)) != cudaSuccess) return e;
        if (!s.consumed && (e = cudaEventCreateWithFlags(&s.consumed, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    if (st.capacity >= bytes) return cudaSuccess;
    for (auto& s : st.slot) {
        // the old buffers may still be read by a queued copy or kernel
        cudaEventSynchronize(s.copied);
        cudaEventSynchronize(s.consumed);
        if (s.host) cudaFreeHost(s.host);
        if (s.dev) cudaFree(s.dev);
        s.host = nullptr;
        s.dev = nullptr;
        if ((e = cudaHostAlloc(&s.host, bytes, cudaHostAllocDefault)) != cudaSuccess) return e;
        if ((e = cudaMalloc(&s.dev, bytes)) != cudaSuccess) return e;
    }
    st.capacity = bytes;
    return cudaSuccess;
}

int kvsel_stage_restore(kvsel_ctx* ctx, const void* host_k, const void* host_v, int64_t host_layer_stride,
                        int64_t host_head_stride, int host_tokens, const int32_t* blocks, const int32_t* dst_page,
                        const int32_t* dst_pos0, int n, int L, int Hkv, int D, int page, double rope_base,
                        int rope_style, void* k_pool, void* v_pool, int P, int chunk_blocks, int gather_threads,
                        int mode, void* stream) {
    const kvsel_trace trace_("kvsel_stage_restore");
    int rc = kvsel_enter(ctx);
    if (rc) return rc;
    if (!host_k || !host_v || !blocks || !dst_page || !dst_pos0 || !k_pool || !v_pool)
        return kvsel_fail(ctx, KVSEL_ERR_INVALID_ARG, "stage_restore: null pointer");
    if (n < 0 || L <= 0 || Hkv <= 0 || page <= 0 || P <= 0 || host_tokens < 0 || chunk_blocks <= 0)
        return kvsel_fail(ctx, KVSEL_ERR_SHAPE, "stage_restore: bad sizes");
    if (D != 16 && D != 32 && D != 64 && D != 128 && D != 256)
        return kvsel_fail(ctx, KVSEL_ERR_UNSUPPORTED, "stage_restore: D=%d unsupported", D);
    if ((int64_t)page * D > 16384) return kvsel_fail(ctx, KVSEL_ERR_UNSUPPORTED, "stage_restore: page*D > 16384");
    if (rope_style != KVSEL_ROPE_NEOX && rope_style != KVSEL_ROPE_INTERLEAVED)
        return kvsel_fail(ctx, KVSEL_ERR_INVALID_ARG, "stage_restore: bad rope_style");
    if (!(rope_base > 1.0)) return kvsel_fail(ctx, KVSEL_ERR_INVALID_ARG, "stage_restore: rope_base must be > 1");
    if (host_head_stride < (int64_t)host_tokens * D || host_layer_stride < 0)
        return kvsel_fail(ctx, KVSEL_ERR_SHAPE, "stage_restore: head stride < host_tokens*D");
    if (((uintptr_t)k_pool | (uintptr_t)v_pool) % 16) return kvsel_fail(ctx, KVSEL_ERR_ALIGN, "stage_restore: pools must be 16-byte aligned");
    // the entries are host data: check them all before any work
    const int n_host_blocks = host_tokens / page;
    for (int i = 0; i < n; ++i) {
        if (blocks[i] < 0 || blocks[i] >= n_host_blocks)
            return kvsel_fail(ctx, KVSEL_ERR_SHAPE, "stage_restore: block %d of entry %d outside the repository", blocks[i], i);
        if (dst_page[i] < 0 || dst_page[i] >= P) return kvsel_fail(ctx, KVSEL_ERR_SHAPE, "stage_restore: page %d outside the pool", dst_page[i]);
        if (dst_pos0[i] < 0 || (int64_t)dst_pos0[i] + page > KVSEL_MAX_POS)
            return kvsel_fail(ctx, KVSEL_ERR_SHAPE, "stage_restore: position %d outside [0, 2^24)", dst_pos0[i]);
    }
    if (mode < KVSEL_STAGE_AUTO || mode > KVSEL_STAGE_DIRECT) return kvsel_fail(ctx, KVSEL_ERR_INVALID_ARG, "stage_restore: bad mode");
    if (n == 0) return KVSEL_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const kvsel_ctx::RopeTab* tab = kvsel_rope_tables(ctx, D, rope_base, s);
    if (!tab) return kvsel_fail(ctx, KVSEL_ERR_CUDA, "stage_restore: rope table allocation failed");
    cudaError_t e;

    // direct path: both repositories mapped into the device address space
    void* dk = nullptr;
    void* dv = nullptr;
    if (mode != KVSEL_STAGE_PACKED) {
        cudaPointerAttributes ak{}, av{};
        const bool mapped = cudaPointerGetAttributes(&ak, host_k) == cudaSuccess &&
                            cudaPointerGetAttributes(&av, host_v) == cudaSuccess && ak.type == cudaMemoryTypeHost &&
                            av.type == cudaMemoryTypeHost && ak.devicePointer && av.devicePointer;
        cudaGetLastError();  // a pageable pointer may leave an error behind
        if (mapped) {
            dk = ak.devicePointer;
            dv = av.devicePointer;
        } else if (mode == KVSEL_STAGE_DIRECT) {
            return kvsel_fail(ctx, KVSEL_ERR_INVALID_ARG, "stage_restore: direct mode needs pinned, mapped repositories");
        }
    }
    if (dk) {
        const size_t arr = up((size_t)n * 4);
        if ((e = stager_reserve(ctx, 3 * arr)) != cudaSuccess) return kvsel_cuda_fail(ctx, e, "stage_restore: staging buffers");
        auto& sl = ctx->stager.slot[0];
        // the slot's earlier readers are done before its entry arrays are rewritten
        if ((e = cudaEventSynchronize(sl.copied)) != cudaSuccess || (e = cudaEventSynchronize(sl.consumed)) != cudaSuccess)
            return kvsel_cuda_fail(ctx, e, "stage_restore: wait slot");
        char* h = static_cast<char*>(sl.host);
        std::memcpy(h, blocks, (size_t)n * 4);
        std::memcpy(h + arr, dst_page, (size_t)n * 4);
        std::memcpy(h + 2 * arr, dst_pos0, (size_t)n * 4);
        void* hd = nullptr;
        if ((e = cudaHostGetDevicePointer(&hd, sl.host, 0)) != cudaSuccess)
            return kvsel_cuda_fail(ctx, e, "stage_restore: map entry arrays");
        const char* ent = static_cast<const char*>(hd);
        e = launch_rerope(dk, host_layer_stride, host_head_stride, host_tokens, reinterpret_cast<const int32_t*>(ent),
                          reinterpret_cast<const int32_t*>(ent + arr), reinterpret_cast<const int32_t*>(ent + 2 * arr), n,
                          nullptr, L, Hkv, D, page, tab, rope_style, k_pool, dv, v_pool, P, ctx->dev_err, s);
        if (e != cudaSuccess) return kvsel_cuda_fail(ctx, e, "stage_restore: direct restore launch");
        if ((e = cudaEventRecord(sl.consumed, s)) != cudaSuccess) return kvsel_cuda_fail(ctx, e, "stage_restore: record");
        return KVSEL_OK;
    }

    // packed, pipelined path
    const int cb = std::min(chunk_blocks, n);
    e = stager_reserve(ctx, BatchLayout(cb, L, Hkv, D, page).bytes);
    if (e != cudaSuccess) return kvsel_cuda_fail(ctx, e, "stage_restore: staging buffers");
    auto& st = ctx->stager;
    const int threads = std::max(1, std::min(gather_threads, 64));
    const size_t row_bytes = (size_t)page * D * 2;  // one block's tokens of one (layer, head)
    const char* hk = static_cast<const char*>(host_k);
    const char* hv = static_cast<const char*>(host_v);

    for (int c0 = 0, batch = 0; c0 < n; c0 += cb, ++batch) {
        const int nb = std::min(cb, n - c0);
        auto& sl = st.slot[batch & 1];
        const BatchLayout lay(nb, L, Hkv, D, page);
        // the pinned buffer is free once the slot's previous copy has completed
        if ((e = cudaEventSynchronize(sl.copied)) != cudaSuccess) return kvsel_cuda_fail(ctx, e, "stage_restore: wait copy");
        char* h = static_cast<char*>(sl.host);
        // gather: work item w = (kind, l, g, i) copies one page of rows
        const int64_t items = 2LL * L * Hkv * nb;
        auto gather = [&](int tid) {
            for (int64_t w = tid; w < items; w += threads) {
                const int i = (int)(w % nb);
                const int64_t lg = (w / nb) % ((int64_t)L * Hkv);
                const int kind = (int)(w / ((int64_t)nb * L * Hkv));
                const int l = (int)(lg / Hkv), g = (int)(lg % Hkv);
                const char* src = (kind ? hv : hk) +
                                  2 * ((int64_t)l * host_layer_stride + (int64_t)g * host_head_stride +
                                       (int64_t)blocks[c0 + i] * page * D);
                char* dst = h + (kind ? lay.v_off : lay.k_off) + ((lg * nb + i) * row_bytes);
                std::memcpy(dst, src, row_bytes);
            }
        };
        if (threads == 1) {
            gather(0);
        } else {
            std::vector<std::thread> pool;
            pool.reserve(threads - 1);
            for (int t = 1; t < threads; ++t) pool.emplace_back(gather, t);
            gather(0);
            for (auto& th : pool) th.join();
        }
        int32_t* sb = reinterpret_cast<int32_t*>(h + lay.sb_off);
        for (int i = 0; i < nb; ++i) sb[i] = i;
        std::memcpy(h + lay.dp_off, dst_page + c0, (size_t)nb * 4);
        std::memcpy(h + lay.d0_off, dst_pos0 + c0, (size_t)nb * 4);
        // copy: after the slot's previous kernel is done with the device buffer
        if ((e = cudaStreamWaitEvent(st.copy_stream, sl.consumed, 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(sl.dev, sl.host, lay.bytes, cudaMemcpyHostToDevice, st.copy_stream)) != cudaSuccess ||
            (e = cudaEventRecord(sl.copied, st.copy_stream)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(s, sl.copied, 0)) != cudaSuccess)
            return kvsel_cuda_fail(ctx, e, "stage_restore: copy");
        // GPU: re-RoPE K, copy V, from the device buffer into the pool
        char* d = static_cast<char*>(sl.dev);
        const int64_t tokens = (int64_t)nb * page;
        e = launch_rerope(d + lay.k_off, (int64_t)Hkv * tokens * D, tokens * D, (int)tokens,
                          reinterpret_cast<const int32_t*>(d + lay.sb_off), reinterpret_cast<const int32_t*>(d + lay.dp_off),
                          reinterpret_cast<const int32_t*>(d + lay.d0_off), nb, nullptr, L, Hkv, D, page, tab, rope_style,
                          k_pool, d + lay.v_off, v_pool, P, ctx->dev_err, s);
        if (e != cudaSuccess) return kvsel_cuda_fail(ctx, e, "stage_restore: restore launch");
        if ((e = cudaEventRecord(sl.consumed, s)) != cudaSuccess) return kvsel_cuda_fail(ctx, e, "stage_restore: record");
    }
    return KVSEL_OK;
}

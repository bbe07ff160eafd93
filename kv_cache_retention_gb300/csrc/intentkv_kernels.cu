// IntentKV kernels: QueryMemory update (Sec. 3.2, Eq. 2), rule scores
// (Sec. 3.2, Eq. 3-4) and the dead-slot redirect of the layout layer.
//
// Rule scores run in three launches so that K is read from HBM exactly once:
//   1. rule_logits: one sweep over the K rows of every (layer, kv head,
//      candidate token).  A warp task is 64 tokens of one (layer, kv head);
//      lane t owns tokens t and t + 32 and loads their rows straight from the
//      pool (through the slot map) in 32-byte pieces, two pieces per token in
//      flight in a register ring that runs on into the next task.  Each piece
//      is multiplied against the G = Hq/Hkv query heads that share the kv head
//      (GQA reuse, packed fp32x2 FMA, M broadcast from the warp's slice of
//      shared memory).  Logits, pre-scaled into the exp2 domain, are stored
//      coalesced along tokens, and each lane keeps an online (max, sum
//      2^(z-max)) per head, merged across the warp once per run of one (layer,
//      kv head); one pair per (l, h, 64-token chunk) goes to global memory.
//   2. rule_lse: merges the chunk partials into log2-sum-exp per (l,h).
//   3. rule_accum: rule[j] = sum_{l,h} 2^(z - lse), a token-parallel pass over
//      the logits (coalesced along j), reduced across warps in a fixed order.
#include <cuda_bf16.h>

#include <vector>

#include "kvsel_internal.h"

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

// L2 policy that keeps the written logits resident until the accumulate pass reads them.
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void store_f32_hint(float* ptr, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(pol) : "memory");
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Merge two (max, sum) pairs of an exp2-domain log-sum-exp.
__device__ __forceinline__ float2 lse_merge(float2 a, float2 b) {
    float m = fmaxf(a.x, b.x);
    if (m == -INFINITY) return make_float2(-INFINITY, 0.f);
    return make_float2(m, a.y * exp2f(a.x - m) + b.y * exp2f(b.x - m));
}

__device__ __forceinline__ bool is_forced(int j, int pi, int q_s, int q_e) {
    return j < pi || (j >= q_s && j < q_e);
}

// ---------------------------------------------------------------------------
// QueryMemory (Eq. 2)
// ---------------------------------------------------------------------------

// One turn of one session, for the batched launch (grid.y = session).
struct MemJob {
    const void* q;
    int R;
    float decay;
    int first_turn;
    float* M;
    float* A;
};

template <typename T>
__global__ void __launch_bounds__(256) memory_update_kernel(const T* __restrict__ q, int R, int D, float decay,
                                                            int first_turn, int norm_mode, float* __restrict__ M,
                                                            float* __restrict__ A, const MemJob* __restrict__ batch) {
    if (batch) {
        const MemJob& b = batch[blockIdx.y];
        q = static_cast<const T*>(b.q);
        R = b.R;
        decay = b.decay;
        first_turn = b.first_turn;
        M = b.M;
        A = b.A;
    }
    constexpr int VEC = 16 / sizeof(T);
    extern __shared__ float sm[];  // [rows_per_iter][D] partial sums, then U[D]
    __shared__ float red[32];
    const int head = blockIdx.x;
    const int chunks = D / VEC;
    const int rpi = blockDim.x / chunks;
    const int c = threadIdx.x % chunks, r0 = threadIdx.x / chunks;
    float acc[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) acc[k] = 0.f;
    if (r0 < rpi) {
        const T* base = q + (int64_t)head * R * D + (int64_t)c * VEC;
        auto add = [&](const uint4& raw) {
            if constexpr (sizeof(T) == 2) {
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float2 f = bf16x2_to_float2(w[k]);
                    acc[2 * k] += f.x;
                    acc[2 * k + 1] += f.y;
                }
            } else {
                acc[0] += __uint_as_float(raw.x);
                acc[1] += __uint_as_float(raw.y);
                acc[2] += __uint_as_float(raw.z);
                acc[3] += __uint_as_float(raw.w);
            }
        };
        // batches of kMemBatch 16-byte loads issued before any is summed: a head's rows are
        // one short stream per thread, so memory-level parallelism has to come from here
        constexpr int kMemBatch = 8;
        int r = r0;
        for (; r + (kMemBatch - 1) * rpi < R; r += kMemBatch * rpi) {
            uint4 raw[kMemBatch];
#pragma unroll
            for (int j = 0; j < kMemBatch; ++j) raw[j] = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)(r + j * rpi) * D));
#pragma unroll
            for (int j = 0; j < kMemBatch; ++j) add(raw[j]);
        }
        for (; r < R; r += rpi) add(__ldg(reinterpret_cast<const uint4*>(base + (int64_t)r * D)));
#pragma unroll
        for (int k = 0; k < VEC; ++k) sm[r0 * D + c * VEC + k] = acc[k];
    }
    __syncthreads();
    float* U = sm + rpi * D;
    float* state = norm_mode == 0 ? M : A;
    float sq = 0.f;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float e = 0.f;
        for (int r = 0; r < rpi; ++r) e += sm[r * D + d];
        e /= (float)R;
        float u = (first_turn ? 0.f : decay * state[(int64_t)head * D + d]) + e;
        if (norm_mode != 0) A[(int64_t)head * D + d] = u;
        U[d] = u;
        sq += u * u;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(kFull, sq, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sq;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float nrm = sqrtf(red[0]);
    for (int d = threadIdx.x; d < D; d += blockDim.x)
        M[(int64_t)head * D + d] = nrm > 0.f ? U[d] / nrm : 0.f;
}

// ---------------------------------------------------------------------------
// Rule scores, pass 1: logits and per-chunk (max, sum)
// ---------------------------------------------------------------------------

struct RuleArgs {
    const void* k_pool;
    const int32_t* slot_map;
    int n_slots;
    int L, Hq, Hkv, N, D;
    int64_t layer_stride, slot_stride;  // in elements
    const float* M;
    int pi, q_s, q_e;
    float scale;       // log2(e) / sqrt(D)
    int n_sub;         // 64-token sub-chunks per layer
    int R;             // sub-chunks per work item (so that Hkv*R tasks fill the block's warps)
    int n_items;       // L * ceil(n_sub / R)
    int items_per_block;
    float* z;          // [L][Hq][N]
    float2* part;      // [L][Hq][n_sub]
    float* lse2;       // [L][Hq]
    float* rule;       // [N] out
    unsigned* dev_err;
    bool aligned32;    // pool base, layer and slot strides are 32-byte aligned
};

#ifndef KVSEL_RULE_TPL
#define KVSEL_RULE_TPL 2
#endif
#ifndef KVSEL_RULE_MINB
#define KVSEL_RULE_MINB 2
#endif
#ifndef KVSEL_RULE_BATCH
#define KVSEL_RULE_BATCH 2
#endif
constexpr int kWarps = 8;                 // warps per block; a warp owns one kv head of an item's tokens
constexpr int kTPL = KVSEL_RULE_TPL;      // tokens per lane in a task
constexpr int kSub = 32 * kTPL;           // tokens per task: lane t takes tokens t, t + 32, ...

// 32 contiguous bytes: one 256-bit load when the address is 32-byte aligned
// (aligned32), else two 128-bit loads (the pool is only required to be 16-byte
// aligned).  An L2 miss fetches the surrounding 256 bytes, which the lane's
// next pieces of the same row use (1% faster at the 8B shape than 32-byte
// fetches).
__device__ __forceinline__ void ldg32(const void* p, uint32_t* r, bool aligned32) {
    if (aligned32) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                       "=r"(r[7])
                     : "l"(p));
    } else {
        asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "l"(p));
        asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "l"(static_cast<const char*>(p) + 16));
    }
}

// Lane-level online (max, sum 2^(z-max)) update.
__device__ __forceinline__ void stat_add(float z, float& m, float& s) {
    if (z > m) {
        s = s * fast_exp2(m - z) + 1.f;
        m = z;
    } else {
        s += fast_exp2(z - m);
    }
}

// Per-warp online (max, sum) statistics of one run: consecutive sub-chunks of
// one layer and one kv head.  Each lane keeps its own pair per query head of
// the group; a flush merges them across the warp and stores the result at the
// run's first sub-chunk, the run's other sub-chunks carrying (-inf, 0).
template <int G>
struct RunStats {
    float m[G], s[G];
    int sub0 = 0, g = -1, l = -1;

    __device__ __forceinline__ void flush(const RuleArgs& a, int lane) {
        if (g < 0) return;
#pragma unroll
        for (int i = 0; i < G; ++i) {
            float2 acc = make_float2(m[i], s[i]);
#pragma unroll
            for (int o = 16; o; o >>= 1)
                acc = lse_merge(acc, make_float2(__shfl_xor_sync(kFull, acc.x, o), __shfl_xor_sync(kFull, acc.y, o)));
            if (lane == 0) a.part[((int64_t)l * a.Hq + g * G + i) * a.n_sub + sub0] = acc;
        }
        g = -1;
    }

    // Enter sub-chunk `sub` of (layer ll, kv head gg): continue the run or start a new one.
    __device__ __forceinline__ void enter(const RuleArgs& a, int ll, int gg, int sub, int lane) {
        if (g != gg || l != ll) {
            flush(a, lane);
            g = gg;
            l = ll;
            sub0 = sub;
#pragma unroll
            for (int i = 0; i < G; ++i) {
                m[i] = -INFINITY;
                s[i] = 0.f;
            }
        } else if (lane < G) {
            a.part[((int64_t)l * a.Hq + g * G + lane) * a.n_sub + sub] = make_float2(-INFINITY, 0.f);
        }
    }
};

// The (layer, kv head, sub-chunk) tasks a warp takes within its block's items,
// in order; next() is false when the warp has none left.
struct TaskCursor {
    int item, t, l, g, sub;

    __device__ __forceinline__ bool next(const RuleArgs& a, int item1, int warp, int tasks, int per_layer) {
        if (warp >= tasks) return false;
        for (;;) {
            t += kWarps;
            if (t >= tasks) {
                t = warp;
                ++item;
            }
            if (item >= item1) return false;
            l = item / per_layer;
            g = t % a.Hkv;
            sub = (item % per_layer) * a.R + t / a.Hkv;
            if (sub < a.n_sub) return true;
        }
    }
};

// Slot-map entries of a task's tokens, lane t holding tokens t, t + 32, ...;
// -1 for tokens that are past N or forced (no row is read for them).  The
// values are only loaded here, and checked where they are used, so that the
// loads overlap the task before.
__device__ __forceinline__ void task_slots(const RuleArgs& a, int sub, int lane, int (&slot)[kTPL]) {
#pragma unroll
    for (int u = 0; u < kTPL; ++u) {
        const int j = sub * kSub + u * 32 + lane;
        slot[u] = -1;
        if (j < a.N && !is_forced(j, a.pi, a.q_s, a.q_e)) slot[u] = a.slot_map ? __ldg(a.slot_map + j) : j;
    }
}

// One warp task = (layer l, kv head g, 32*kTPL tokens): lane t owns tokens t,
// t+32, ... for all D dims of head g and all G query heads sharing it.  The
// warp keeps the G rows of M it needs in its own slice of shared memory, and
// every lane reads the same M entries, so the reads are broadcasts; K comes
// straight from the pool in 32-byte pieces.  A warp streams through its tasks
// without a block barrier: the last loads of a task already fetch the first
// pieces of the next one, whose slot-map entries were loaded a task ahead.
// BATCHED: one launch for many sessions; grid.y is the session, batch[s] its
// arguments, and CTAs past a session's last item find no task.
template <int G, bool BF16, bool BATCHED>
__global__ void __launch_bounds__(kWarps * 32, KVSEL_RULE_MINB)
    rule_logits_kernel(const __grid_constant__ RuleArgs a_in, const RuleArgs* __restrict__ batch) {
    const RuleArgs& a = BATCHED ? batch[blockIdx.y] : a_in;
    extern __shared__ __align__(16) float Msm[];  // [kWarps][G][D]
    constexpr int ES = BF16 ? 2 : 4;
    constexpr int DPP = 32 / ES;                  // dims per 32-byte piece
    constexpr int BATCH = KVSEL_RULE_BATCH;       // pieces per token in flight (rolling)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hq = a.Hq, D = a.D;
    float* Ms = Msm + warp * G * D;
    const int n_pieces = D / DPP;
    const bool stream = n_pieces % BATCH == 0;    // pieces of consecutive tasks line up in the ring
    const int tasks = a.Hkv * a.R;
    const int item1 = min(a.n_items, (blockIdx.x + 1) * a.items_per_block);
    const int per_layer = (a.n_sub + a.R - 1) / a.R;
    const uint64_t pol_z = policy_evict_last();

    TaskCursor cur{(int)blockIdx.x * a.items_per_block, warp - kWarps, 0, 0, 0};
    if (!cur.next(a, item1, warp, tasks, per_layer)) return;
    TaskCursor nxt = cur;
    bool have_nxt = nxt.next(a, item1, warp, tasks, per_layer);
    int slot_cur[kTPL], slot_nxt[kTPL];
    task_slots(a, cur.sub, lane, slot_cur);
    if (have_nxt) task_slots(a, nxt.sub, lane, slot_nxt);

    auto row_of = [&](const TaskCursor& tk, int slot) -> const char* {
        if (slot < 0 || slot >= a.n_slots) return nullptr;
        return reinterpret_cast<const char*>(a.k_pool) +
               ((size_t)tk.l * a.layer_stride + (size_t)slot * a.slot_stride + (size_t)tk.g * D) * ES;
    };
    const char* row[kTPL];
    uint32_t raw[kTPL][BATCH][8];
    auto load_first = [&]() {
#pragma unroll
        for (int u = 0; u < kTPL; ++u)
#pragma unroll
            for (int q = 0; q < BATCH; ++q) {
                if (row[u] && q < n_pieces) {
                    ldg32(row[u] + (size_t)q * 32, raw[u][q], a.aligned32);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) raw[u][q][k] = 0u;
                }
            }
    };
#pragma unroll
    for (int u = 0; u < kTPL; ++u) row[u] = row_of(cur, slot_cur[u]);
    load_first();

    RunStats<G> run;
    int m_l = -1, m_g = -1;
    for (;;) {
        run.enter(a, cur.l, cur.g, cur.sub, lane);
        if (m_l != cur.l || m_g != cur.g) {
            __syncwarp();
            const float4* src = reinterpret_cast<const float4*>(a.M + ((int64_t)cur.l * Hq + cur.g * G) * D);
            for (int idx = lane; idx < G * D / 4; idx += 32) reinterpret_cast<float4*>(Ms)[idx] = __ldg(src + idx);
            __syncwarp();
            m_l = cur.l;
            m_g = cur.g;
        }
        float2 acc[kTPL][G];
#pragma unroll
        for (int u = 0; u < kTPL; ++u)
#pragma unroll
            for (int i = 0; i < G; ++i) acc[u][i] = make_float2(0.f, 0.f);
        // Rolling prefetch: slot q of raw holds piece p0 + q; right after it is
        // consumed it is refilled with piece p0 + BATCH + q, of this task or,
        // past its last piece, of the next task.
        for (int p0 = 0; p0 < n_pieces; p0 += BATCH) {
#pragma unroll
            for (int q = 0; q < BATCH; ++q) {
                if (p0 + q >= n_pieces) break;
                const int d0 = (p0 + q) * DPP;
#pragma unroll
                for (int w = 0; w < 8; w += (BF16 ? 2 : 4)) {
                    // 4 dims of K for each of the lane's tokens
                    float2 k01[kTPL], k23[kTPL];
#pragma unroll
                    for (int u = 0; u < kTPL; ++u) {
                        if constexpr (BF16) {
                            k01[u] = bf16x2_to_float2(raw[u][q][w]);
                            k23[u] = bf16x2_to_float2(raw[u][q][w + 1]);
                        } else {
                            k01[u] = make_float2(__uint_as_float(raw[u][q][w]), __uint_as_float(raw[u][q][w + 1]));
                            k23[u] = make_float2(__uint_as_float(raw[u][q][w + 2]), __uint_as_float(raw[u][q][w + 3]));
                        }
                    }
                    const int d = d0 + (BF16 ? 2 * w : w);
#pragma unroll
                    for (int i = 0; i < G; ++i) {
                        const float4 m4 = *reinterpret_cast<const float4*>(&Ms[i * D + d]);
                        const float2 m01 = make_float2(m4.x, m4.y), m23 = make_float2(m4.z, m4.w);
#pragma unroll
                        for (int u = 0; u < kTPL; ++u) {
                            acc[u][i] = __ffma2_rn(m01, k01[u], acc[u][i]);
                            acc[u][i] = __ffma2_rn(m23, k23[u], acc[u][i]);
                        }
                    }
                }
                const int pn = p0 + BATCH + q;
                if (pn < n_pieces) {
#pragma unroll
                    for (int u = 0; u < kTPL; ++u)
                        if (row[u]) ldg32(row[u] + (size_t)pn * 32, raw[u][q], a.aligned32);
                } else if (stream && have_nxt) {
#pragma unroll
                    for (int u = 0; u < kTPL; ++u) {
                        const char* r2 = row_of(nxt, slot_nxt[u]);
                        if (r2) {
                            ldg32(r2 + (size_t)(pn - n_pieces) * 32, raw[u][q], a.aligned32);
                        } else {
#pragma unroll
                            for (int k = 0; k < 8; ++k) raw[u][q][k] = 0u;
                        }
                    }
                }
            }
        }
        // logits: coalesced along tokens; statistics per lane
#pragma unroll
        for (int u = 0; u < kTPL; ++u) {
            const int j = cur.sub * kSub + u * 32 + lane;
            if (j < a.N) {
                const bool cand = !is_forced(j, a.pi, a.q_s, a.q_e);
                if (cand && !row[u]) atomicOr(a.dev_err, (unsigned)KVSEL_DEV_BAD_SLOT);  // read as a zero row
#pragma unroll
                for (int i = 0; i < G; ++i) {
                    const float z = cand ? (acc[u][i].x + acc[u][i].y) * a.scale : -INFINITY;
                    store_f32_hint(a.z + ((int64_t)cur.l * Hq + cur.g * G + i) * a.N + j, z, pol_z);
                    if (cand) stat_add(z, run.m[i], run.s[i]);
                }
            }
        }
        if (!have_nxt) break;
        cur = nxt;
#pragma unroll
        for (int u = 0; u < kTPL; ++u) {
            slot_cur[u] = slot_nxt[u];
            row[u] = row_of(cur, slot_cur[u]);
        }
        have_nxt = nxt.next(a, item1, warp, tasks, per_layer);
        if (have_nxt) task_slots(a, nxt.sub, lane, slot_nxt);
        if (!stream) load_first();
    }
    run.flush(a, lane);
}

// ---------------------------------------------------------------------------
// Rule scores, pass 2 and 3
// ---------------------------------------------------------------------------

template <bool BATCHED>
__global__ void __launch_bounds__(256) rule_lse_kernel(const __grid_constant__ RuleArgs a_in,
                                                       const RuleArgs* __restrict__ batch, int rows) {
    const RuleArgs& a = BATCHED ? batch[blockIdx.y] : a_in;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= rows) return;
    const int n_chunks = a.n_sub;
    const float2* part = a.part;
    float2 acc = make_float2(-INFINITY, 0.f);
    for (int c = lane; c < n_chunks; c += 32) acc = lse_merge(acc, part[(int64_t)warp * n_chunks + c]);
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        float2 other = make_float2(__shfl_xor_sync(kFull, acc.x, o), __shfl_xor_sync(kFull, acc.y, o));
        acc = lse_merge(acc, other);
    }
    if (lane == 0) a.lse2[warp] = acc.y > 0.f ? acc.x + log2f(acc.y) : -INFINITY;
}

// Block = 8 warps x 32 tokens; warp w sums its share of the (l,h) rows for its
// lane's token; the 8 partial sums are added in warp order.
template <bool BATCHED>
__global__ void __launch_bounds__(256) rule_accum_kernel(const __grid_constant__ RuleArgs a_in,
                                                         const RuleArgs* __restrict__ batch, int rows) {
    const RuleArgs& a = BATCHED ? batch[blockIdx.y] : a_in;
    const int N = a.N;
    if (BATCHED && (int)blockIdx.x * 32 >= N) return;  // past this session's tokens
    const float* __restrict__ z = a.z;
    const float* __restrict__ lse2 = a.lse2;
    const int pi = a.pi, q_s = a.q_s, q_e = a.q_e;
    float* __restrict__ rule = a.rule;
    extern __shared__ float s_lse[];  // [rows]
    __shared__ float red[8][32];
    for (int r = threadIdx.x; r < rows; r += blockDim.x) s_lse[r] = lse2[r];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.x * 32 + lane;
    const int r0 = (int)((int64_t)rows * warp / 8), r1 = (int)((int64_t)rows * (warp + 1) / 8);
    float acc = 0.f;
    if (j < N) {
        const float* zp = z + j;
        int r = r0;
        for (; r + 8 <= r1; r += 8) {
            float t[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) t[u] = __ldcs(zp + (int64_t)(r + u) * N);
#pragma unroll
            for (int u = 0; u < 8; ++u) acc += exp2f(t[u] - s_lse[r + u]);
        }
        for (; r < r1; ++r) acc += exp2f(__ldcs(zp + (int64_t)r * N) - s_lse[r]);
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && j < N) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) sum += red[w][lane];
        rule[j] = is_forced(j, pi, q_s, q_e) ? 0.f : sum;
    }
}

__global__ void redirect_kernel(const int32_t* __restrict__ slot_in, const uint8_t* __restrict__ keep, int N,
                                int32_t dead, int32_t* slot_out) {
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < N; j += gridDim.x * blockDim.x)
        slot_out[j] = keep[j] ? slot_in[j] : dead;
}

// SideQuest cursor eviction ("SideQuest" page, method overview, Figure 1): the
// listed cursors' half-open spans [span_start, span_end) are cleared from a keep
// mask.  Each CTA holds the listed spans in shared memory (in chunks of kSpanChunk)
// and each thread tests its positions against all of them; keep_out may alias
// keep_in.  Ids outside the cursor table are ignored and flagged.
constexpr int kSpanChunk = 2048;

__global__ void __launch_bounds__(256) span_keep_kernel(const int32_t* __restrict__ span_start,
                                                        const int32_t* __restrict__ span_end, int n_cursors,
                                                        const int32_t* __restrict__ del_ids, int n_del,
                                                        const uint8_t* keep_in, int N, uint8_t* keep_out,
                                                        unsigned* dev_err) {
    __shared__ int2 spans[kSpanChunk];
    const int stride = gridDim.x * blockDim.x;
    const int j0 = blockIdx.x * blockDim.x + threadIdx.x;
    // positions of this thread: j0, j0 + stride, ... (at most kPer of them)
    constexpr int kPer = 8;
    bool keep[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int j = j0 + u * stride;
        keep[u] = j < N && (keep_in ? keep_in[j] != 0 : true);
    }
    for (int c0 = 0; c0 < n_del; c0 += kSpanChunk) {
        const int nc = min(kSpanChunk, n_del - c0);
        __syncthreads();
        for (int d = threadIdx.x; d < nc; d += blockDim.x) {
            const int c = __ldg(del_ids + c0 + d);
            int2 sp = make_int2(0, 0);  // empty span for an unknown id
            if (c >= 0 && c < n_cursors) {
                sp = make_int2(__ldg(span_start + c), __ldg(span_end + c));
            } else if (blockIdx.x == 0) {
                atomicOr(dev_err, (unsigned)KVSEL_DEV_BAD_BLOCK);
            }
            spans[d] = sp;
        }
        __syncthreads();
        for (int d = 0; d < nc; ++d) {
            const int2 sp = spans[d];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int j = j0 + u * stride;
                if (j >= sp.x && j < sp.y) keep[u] = false;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int j = j0 + u * stride;
        if (j < N) keep_out[j] = keep[u] ? 1 : 0;
    }
}

template <int G, bool BF16, bool BATCHED>
cudaError_t launch_logits(const RuleArgs& a, const RuleArgs* batch, dim3 grid, size_t smem, cudaStream_t s) {
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(rule_logits_kernel<G, BF16, BATCHED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    rule_logits_kernel<G, BF16, BATCHED><<<grid, kWarps * 32, smem, s>>>(a, batch);
    return cudaGetLastError();
}

template <bool BF16, bool BATCHED>
cudaError_t dispatch_logits(int G, const RuleArgs& a, const RuleArgs* batch, dim3 grid, size_t smem, cudaStream_t s) {
    switch (G) {
        case 1: return launch_logits<1, BF16, BATCHED>(a, batch, grid, smem, s);
        case 2: return launch_logits<2, BF16, BATCHED>(a, batch, grid, smem, s);
        case 3: return launch_logits<3, BF16, BATCHED>(a, batch, grid, smem, s);
        case 4: return launch_logits<4, BF16, BATCHED>(a, batch, grid, smem, s);
        case 5: return launch_logits<5, BF16, BATCHED>(a, batch, grid, smem, s);
        case 6: return launch_logits<6, BF16, BATCHED>(a, batch, grid, smem, s);
        case 7: return launch_logits<7, BF16, BATCHED>(a, batch, grid, smem, s);
        case 8: return launch_logits<8, BF16, BATCHED>(a, batch, grid, smem, s);
    }
    return cudaErrorInvalidValue;
}

int rule_chunks(int N) { return (N + kSub - 1) / kSub; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// Threads per QueryMemory block: 128 (a head per block, all heads resident at once on
// GB300, each thread with eight 16-byte loads in flight) unless a row has more
// 16-byte chunks than that.
int mu_threads(int chunks) { return chunks > 128 ? 256 : 128; }

cudaError_t launch_memory_update(const void* q, int dtype, int L, int Hq, int R, int D, float lambda, int first_turn,
                                 int norm_mode, float* M, float* A, cudaStream_t s) {
    const float decay = expf(-lambda);
    const int vec = dtype == KVSEL_BF16 ? 8 : 4;
    const int nt = mu_threads(D / vec);
    const int rpi = nt / (D / vec);
    const size_t smem = sizeof(float) * ((size_t)rpi * D + D);
    const int heads = L * Hq;
    if (dtype == KVSEL_BF16) {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(memory_update_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        memory_update_kernel<__nv_bfloat16><<<heads, nt, smem, s>>>(static_cast<const __nv_bfloat16*>(q), R, D, decay,
                                                                      first_turn, norm_mode, M, A, nullptr);
    } else {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(memory_update_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        memory_update_kernel<float><<<heads, nt, smem, s>>>(static_cast<const float*>(q), R, D, decay, first_turn,
                                                             norm_mode, M, A, nullptr);
    }
    return cudaGetLastError();
}

size_t memory_update_batch_workspace(int S) { return (size_t)S * sizeof(MemJob) + 256; }

cudaError_t launch_memory_update_batch(int dtype, int L, int Hq, int D, int norm_mode, const kvsel_memory_session* sess,
                                       int S, void* ws, cudaStream_t s) {
    std::vector<MemJob> jobs((size_t)S);
    for (int i = 0; i < S; ++i)
        jobs[i] = MemJob{sess[i].q_rows, sess[i].R, expf(-sess[i].lambda), sess[i].first_turn, sess[i].M, sess[i].A};
    MemJob* dev = static_cast<MemJob*>(ws);
    cudaError_t e = cudaMemcpyAsync(dev, jobs.data(), (size_t)S * sizeof(MemJob), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    const int vec = dtype == KVSEL_BF16 ? 8 : 4;
    const int nt = mu_threads(D / vec);
    const int rpi = nt / (D / vec);
    const size_t smem = sizeof(float) * ((size_t)rpi * D + D);
    const dim3 grid((unsigned)(L * Hq), (unsigned)S);
    if (dtype == KVSEL_BF16) {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(memory_update_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        memory_update_kernel<__nv_bfloat16><<<grid, nt, smem, s>>>(nullptr, 0, D, 0.f, 0, norm_mode, nullptr, nullptr, dev);
    } else {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(memory_update_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        memory_update_kernel<float><<<grid, nt, smem, s>>>(nullptr, 0, D, 0.f, 0, norm_mode, nullptr, nullptr, dev);
    }
    return cudaGetLastError();
}

size_t rule_scores_workspace(kvsel_ctx*, int L, int Hq, int N) {
    const size_t rows = (size_t)L * Hq;
    return align256(rows * N * sizeof(float)) + align256(rows * rule_chunks(N) * sizeof(float2)) +
           align256(rows * sizeof(float));
}

cudaError_t launch_rule_scores(kvsel_ctx* ctx, const void* k_pool, int dtype, const int32_t* slot_map, int n_slots,
                               int L, int Hq, int Hkv, int N, int D, int64_t layer_stride, int64_t slot_stride,
                               const float* M, int pi, int q_s, int q_e, float* rule, void* ws, cudaStream_t s) {
    const size_t rows = (size_t)L * Hq;
    char* w = static_cast<char*>(ws);
    RuleArgs a;
    a.k_pool = k_pool;
    a.slot_map = slot_map;
    a.n_slots = n_slots;
    a.L = L;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.N = N;
    a.D = D;
    a.layer_stride = layer_stride;
    a.slot_stride = slot_stride;
    a.M = M;
    a.pi = pi;
    a.q_s = q_s;
    a.q_e = q_e;
    a.scale = kLog2e / sqrtf((float)D);
    a.n_sub = rule_chunks(N);
    a.z = reinterpret_cast<float*>(w);
    w += align256(rows * N * sizeof(float));
    a.part = reinterpret_cast<float2*>(w);
    w += align256(rows * a.n_sub * sizeof(float2));
    a.lse2 = reinterpret_cast<float*>(w);
    a.rule = rule;
    a.dev_err = ctx->dev_err;
    {
        const int64_t es = dtype == KVSEL_BF16 ? 2 : 4;  // row offsets g*D*es are multiples of 32 for D >= 16
        a.aligned32 = reinterpret_cast<uintptr_t>(k_pool) % 32 == 0 && (layer_stride * es) % 32 == 0 &&
                      (slot_stride * es) % 32 == 0;
    }
    a.R = Hkv >= kWarps ? 1 : kWarps / Hkv;
    const int items_per_layer = (a.n_sub + a.R - 1) / a.R;
    a.n_items = L * items_per_layer;
    const int G = Hq / Hkv;
    const size_t smem = sizeof(float) * (size_t)kWarps * G * D;  // each warp's slice of M
    const int blocks_per_sm = KVSEL_RULE_MINB;
    const int grid_max = blocks_per_sm * ctx->num_sms;
    a.items_per_block = (a.n_items + grid_max - 1) / grid_max;
    const int grid = (a.n_items + a.items_per_block - 1) / a.items_per_block;
    cudaError_t e = dtype == KVSEL_BF16 ? dispatch_logits<true, false>(G, a, nullptr, dim3(grid), smem, s)
                                        : dispatch_logits<false, false>(G, a, nullptr, dim3(grid), smem, s);
    if (e != cudaSuccess) return e;
    rule_lse_kernel<false><<<(int)((rows * 32 + 255) / 256), 256, 0, s>>>(a, nullptr, (int)rows);
    const size_t smem3 = rows * sizeof(float);
    if (smem3 > 48 * 1024)
        cudaFuncSetAttribute(rule_accum_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem3);
    rule_accum_kernel<false><<<(N + 31) / 32, 256, smem3, s>>>(a, nullptr, (int)rows);
    return cudaGetLastError();
}

size_t rule_scores_batch_workspace(int L, int Hq, const kvsel_rule_session* sess, int S) {
    const size_t rows = (size_t)L * Hq;
    size_t b = align256((size_t)S * sizeof(RuleArgs));
    for (int i = 0; i < S; ++i) {
        const int N = sess[i].N;
        b += align256(rows * N * sizeof(float)) + align256(rows * rule_chunks(N) * sizeof(float2)) +
             align256(rows * sizeof(float));
    }
    return b;
}

cudaError_t launch_rule_scores_batch(kvsel_ctx* ctx, const void* k_pool, int dtype, int n_slots, int L, int Hq,
                                     int Hkv, int D, int64_t layer_stride, int64_t slot_stride,
                                     const kvsel_rule_session* sess, int S, void* ws, cudaStream_t s) {
    const size_t rows = (size_t)L * Hq;
    char* w = static_cast<char*>(ws);
    RuleArgs* dev_args = reinterpret_cast<RuleArgs*>(w);
    w += align256((size_t)S * sizeof(RuleArgs));
    const int64_t es = dtype == KVSEL_BF16 ? 2 : 4;
    const bool aligned32 = reinterpret_cast<uintptr_t>(k_pool) % 32 == 0 && (layer_stride * es) % 32 == 0 &&
                           (slot_stride * es) % 32 == 0;
    const int R = Hkv >= kWarps ? 1 : kWarps / Hkv;
    std::vector<RuleArgs> args((size_t)S);
    int64_t total_items = 0;
    int max_N = 0;
    for (int i = 0; i < S; ++i) {
        RuleArgs& a = args[i];
        a.k_pool = k_pool;
        a.slot_map = sess[i].slot_map;
        a.n_slots = n_slots;
        a.L = L;
        a.Hq = Hq;
        a.Hkv = Hkv;
        a.N = sess[i].N;
        a.D = D;
        a.layer_stride = layer_stride;
        a.slot_stride = slot_stride;
        a.M = sess[i].M;
        a.pi = sess[i].pi;
        a.q_s = sess[i].q_s;
        a.q_e = sess[i].q_e;
        a.scale = kLog2e / sqrtf((float)D);
        a.n_sub = rule_chunks(a.N);
        a.R = R;
        a.n_items = L * ((a.n_sub + R - 1) / R);
        a.z = reinterpret_cast<float*>(w);
        w += align256(rows * a.N * sizeof(float));
        a.part = reinterpret_cast<float2*>(w);
        w += align256(rows * a.n_sub * sizeof(float2));
        a.lse2 = reinterpret_cast<float*>(w);
        w += align256(rows * sizeof(float));
        a.rule = sess[i].rule;
        a.dev_err = ctx->dev_err;
        a.aligned32 = aligned32;
        total_items += a.n_items;
        max_N = a.N > max_N ? a.N : max_N;
    }
    // every CTA gets the same number of items, sized to fill the GPU once over all sessions: the
    // per-session ceilings must not add up to more CTAs than one wave holds, or a few SMs run a
    // second round while the rest idle
    const int64_t grid_max = (int64_t)KVSEL_RULE_MINB * ctx->num_sms;
    int ipb = (int)((total_items + grid_max - 1) / grid_max > 0 ? (total_items + grid_max - 1) / grid_max : 1);
    for (;; ++ipb) {
        int64_t ctas = 0;
        for (const auto& a : args) ctas += (a.n_items + ipb - 1) / ipb;
        if (ctas <= grid_max) break;
    }
    int gx = 1;
    for (auto& a : args) {
        a.items_per_block = ipb;
        const int g = (a.n_items + ipb - 1) / ipb;
        gx = g > gx ? g : gx;
    }
    cudaError_t e = cudaMemcpyAsync(dev_args, args.data(), (size_t)S * sizeof(RuleArgs), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    const int G = Hq / Hkv;
    const size_t smem = sizeof(float) * (size_t)kWarps * G * D;
    e = dtype == KVSEL_BF16 ? dispatch_logits<true, true>(G, args[0], dev_args, dim3(gx, S), smem, s)
                            : dispatch_logits<false, true>(G, args[0], dev_args, dim3(gx, S), smem, s);
    if (e != cudaSuccess) return e;
    rule_lse_kernel<true><<<dim3((unsigned)((rows * 32 + 255) / 256), S), 256, 0, s>>>(args[0], dev_args, (int)rows);
    const size_t smem3 = rows * sizeof(float);
    if (smem3 > 48 * 1024)
        cudaFuncSetAttribute(rule_accum_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem3);
    if (max_N > 0)
        rule_accum_kernel<true><<<dim3((max_N + 31) / 32, S), 256, smem3, s>>>(args[0], dev_args, (int)rows);
    return cudaGetLastError();
}

cudaError_t launch_span_keep(const int32_t* span_start, const int32_t* span_end, int n_cursors, const int32_t* del_ids,
                             int n_del, const uint8_t* keep_in, int N, uint8_t* keep_out, unsigned* dev_err,
                             cudaStream_t s) {
    // every position is covered: grid * 256 threads * 8 positions >= N
    const int grid = (N + 256 * 8 - 1) / (256 * 8);
    span_keep_kernel<<<grid, 256, 0, s>>>(span_start, span_end, n_cursors, del_ids, n_del, keep_in, N, keep_out, dev_err);
    return cudaGetLastError();
}

cudaError_t launch_redirect(const int32_t* slot_in, const uint8_t* keep, int N, int32_t dead, int32_t* slot_out,
                            cudaStream_t s) {
    int grid = (N + 255) / 256;
    if (grid > 4096) grid = 4096;
    redirect_kernel<<<grid, 256, 0, s>>>(slot_in, keep, N, dead, slot_out);
    return cudaGetLastError();
}

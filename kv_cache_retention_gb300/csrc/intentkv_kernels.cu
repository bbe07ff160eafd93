// IntentKV kernels: QueryMemory update (Sec. 3.2, Eq. 2), rule scores
// (Sec. 3.2, Eq. 3-4) and the dead-slot redirect of the layout layer.
//
// Rule scores run in three launches so that K is read from HBM exactly once:
//   1. rule_logits: one sweep over the K rows of every (layer, candidate
//      token).  Each 32-byte piece of a K row is loaded once into registers and
//      multiplied against the G = Hq/Hkv query heads that share its kv head
//      (GQA reuse), the per-head partial dot products are summed across the
//      D/16 lanes of the head with a halving shuffle exchange, and the logits
//      (pre-scaled into the exp2 domain) go through a shared-memory tile to
//      coalesced stores.  Each lane keeps an online (max, sum 2^(z-max)) per
//      head it owns; a block merges them per chunk of tokens.
//   2. rule_lse: merges the chunk partials into log2-sum-exp per (l,h).
//   3. rule_accum: rule[j] = sum_{l,h} 2^(z - lse), a token-parallel pass over
//      the logits (coalesced along j), reduced across warps in a fixed order.
#include <cuda_bf16.h>

#include "kvsel_internal.h"

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kRuleThreads = 256;
constexpr int kZTile = 64;       // tokens per shared-memory logit tile
constexpr int kChunkTiles = 2;   // tiles per work item (chunk = 128 tokens)
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 32 contiguous bytes, read-only path, not allocated in L1, evict-first in L2;
// one 256-bit load when the address is 32-byte aligned, else two 128-bit loads.
__device__ __forceinline__ void load32(const void* ptr, uint32_t* r, uint64_t pol, bool aligned32) {
    if (aligned32) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                       "=r"(r[7])
                     : "l"(ptr), "l"(pol));
    } else {
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.b32 {%0,%1,%2,%3}, [%4], %5;"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "l"(ptr), "l"(pol));
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.b32 {%0,%1,%2,%3}, [%4], %5;"
                     : "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "l"(static_cast<const char*>(ptr) + 16), "l"(pol));
    }
}

__device__ __forceinline__ void store_f32_hint(float* ptr, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(pol) : "memory");
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
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

template <typename T>
__global__ void __launch_bounds__(256) memory_update_kernel(const T* __restrict__ q, int R, int D, float decay,
                                                            int first_turn, int norm_mode, float* __restrict__ M,
                                                            float* __restrict__ A) {
    constexpr int VEC = 16 / sizeof(T);
    extern __shared__ float sm[];  // [rows_per_iter][D] partial sums, then U[D]
    __shared__ float red[32];
    const int head = blockIdx.x;
    const int chunks = D / VEC;
    const int rpi = 256 / chunks;
    const int c = threadIdx.x % chunks, r0 = threadIdx.x / chunks;
    float acc[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) acc[k] = 0.f;
    if (r0 < rpi) {
        const T* base = q + (int64_t)head * R * D + (int64_t)c * VEC;
        for (int r = r0; r < R; r += rpi) {
            uint4 raw = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)r * D));
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
        }
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
    int64_t layer_stride, slot_stride;
    const float* M;
    int pi, q_s, q_e;
    float scale;   // log2(e) / sqrt(D)
    int n_chunks;  // chunks per layer (chunk = kZTile * kChunkTiles tokens)
    float* z;      // [L][Hq][N]
    float2* part;  // [L][Hq][n_chunks]
    unsigned* dev_err;
    bool aligned32;  // pool base and strides allow 32-byte loads
};

__host__ __device__ constexpr int next_pow2(int g) { return g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8; }

// Thread layout: S = D/16 lanes per kv head (16 dims each), TT = Hkv*S lanes per
// token, P = 256/TT tokens per pass.  A lane owns (token slot tp, kv head g,
// dims [16s, 16s+16)) and keeps those dims of the G query heads' M in registers.
template <int G, bool BF16>
__global__ void __launch_bounds__(kRuleThreads, 2) rule_logits_kernel(const RuleArgs a) {
    constexpr int P2 = next_pow2(G);
    extern __shared__ float smem[];
    const int S = a.D >> 4;
    const int TT = a.Hkv * S;
    const int P = kRuleThreads / TT;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int tp = tid / TT;                 // token slot in a pass (>= P: idle)
    const int g = (tid % TT) / S;            // kv head
    const int s = tid % S;                   // 16-dim slice
    const bool active = tp < P;
    const int Hq = a.Hq;
    const int zpitch = Hq + 1;
    float* ztile = smem;                                  // [kZTile][Hq+1]
    float* red_m = ztile + kZTile * zpitch;               // [P][Hq]
    float* red_s = red_m + P * Hq;                        // [P][Hq]

    // after the shuffle exchange: values per lane, lanes sharing a value
    const int nv = P2 >= S ? P2 / S : 1;
    const int nshare = S > P2 ? S / P2 : 1;
    const bool writer = active && (s % nshare) == 0;

    const uint64_t pol_k = policy_evict_first();
    const uint64_t pol_z = policy_evict_last();
    const int chunk_len = kZTile * kChunkTiles;
    const int total_items = a.L * a.n_chunks;

    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int l = item / a.n_chunks;
        const int chunk = item % a.n_chunks;
        const int j_begin = chunk * chunk_len;
        const int j_end = min(a.N, j_begin + chunk_len);

        // M slice for the G query heads of kv head g, dims [16s, 16s+16)
        float m_reg[G][16];
#pragma unroll
        for (int i = 0; i < G; ++i) {
            const float* mp = a.M + ((int64_t)l * Hq + (int64_t)g * G + i) * a.D + 16 * s;
#pragma unroll
            for (int k = 0; k < 16; k += 4) {
                float4 v = active ? __ldg(reinterpret_cast<const float4*>(mp + k)) : make_float4(0, 0, 0, 0);
                m_reg[i][k] = v.x;
                m_reg[i][k + 1] = v.y;
                m_reg[i][k + 2] = v.z;
                m_reg[i][k + 3] = v.w;
            }
        }
        float run_m[P2 > 1 ? P2 : 1], run_s[P2 > 1 ? P2 : 1];
#pragma unroll
        for (int k = 0; k < P2; ++k) {
            run_m[k] = -INFINITY;
            run_s[k] = 0.f;
        }
        int my_base = 0;  // first local head index this lane holds after the exchange

        const char* layer_base = reinterpret_cast<const char*>(a.k_pool) +
                                 ((int64_t)l * a.layer_stride + (int64_t)g * a.D + 16 * s) * (BF16 ? 2 : 4);

        for (int t0 = j_begin; t0 < j_end; t0 += kZTile) {
            for (int pb = 0; pb < kZTile; pb += 2 * P) {
                uint32_t raw[2][BF16 ? 8 : 16];
                bool cand[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int tl = pb + u * P + tp;
                    const int j = t0 + tl;
                    cand[u] = active && tl < kZTile && j < j_end && !is_forced(j, a.pi, a.q_s, a.q_e);
#pragma unroll
                    for (int k = 0; k < (BF16 ? 8 : 16); ++k) raw[u][k] = 0u;
                    if (cand[u]) {
                        int64_t slot = a.slot_map ? (int64_t)__ldg(a.slot_map + j) : (int64_t)j;
                        if (slot < 0 || slot >= a.n_slots) {
                            atomicOr(a.dev_err, (unsigned)KVSEL_DEV_BAD_SLOT);
                        } else {
                            const char* p = layer_base + slot * a.slot_stride * (BF16 ? 2 : 4);
                            load32(p, &raw[u][0], pol_k, a.aligned32);
                            if constexpr (!BF16) load32(p + 32, &raw[u][8], pol_k, a.aligned32);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float x[16];
                    if constexpr (BF16) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            float2 f = bf16x2_to_float2(raw[u][k]);
                            x[2 * k] = f.x;
                            x[2 * k + 1] = f.y;
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) x[k] = __uint_as_float(raw[u][k]);
                    }
                    float v[P2];
#pragma unroll
                    for (int i = 0; i < P2; ++i) v[i] = 0.f;
#pragma unroll
                    for (int i = 0; i < G; ++i) {
                        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                        for (int k = 0; k < 16; k += 2)
                            acc = __ffma2_rn(make_float2(m_reg[i][k], m_reg[i][k + 1]), make_float2(x[k], x[k + 1]), acc);
                        v[i] = acc.x + acc.y;
                    }
                    // halving exchange across the S lanes of the head: at each level a
                    // lane keeps half of its values and receives the partner's copy of
                    // that half, so the per-lane shuffle count falls with the level.
                    int base = 0;
#pragma unroll
                    for (int lev = 0; lev < 5; ++lev) {
                        const int o = S >> (lev + 1);
                        if (o == 0) break;
                        const int cur = P2 >> lev;
                        if (cur > 1) {
                            const int half = cur >> 1;
                            const bool up = (lane & o) != 0;
#pragma unroll
                            for (int k = 0; k < (P2 >> (lev + 1) > 0 ? P2 >> (lev + 1) : 1); ++k) {
                                if (k < half) {
                                    float send = up ? v[k] : v[k + half];
                                    float keep = up ? v[k + half] : v[k];
                                    v[k] = keep + __shfl_xor_sync(kFull, send, o);
                                }
                            }
                            if (up) base += half;
                        } else {
                            v[0] += __shfl_xor_sync(kFull, v[0], o);
                        }
                    }
                    my_base = base;
                    const int tl = pb + u * P + tp;
                    if (writer && tl < kZTile && t0 + tl < j_end) {
#pragma unroll
                        for (int k = 0; k < P2; ++k) {
                            if (k < nv && base + k < G) {
                                const float zz = cand[u] ? v[k] * a.scale : -INFINITY;
                                ztile[tl * zpitch + g * G + base + k] = zz;
                                if (cand[u]) {
                                    if (zz > run_m[k]) {
                                        run_s[k] = run_s[k] * exp2f(run_m[k] - zz) + 1.f;
                                        run_m[k] = zz;
                                    } else {
                                        run_s[k] += exp2f(zz - run_m[k]);
                                    }
                                }
                            }
                        }
                    }
                }
            }
            __syncthreads();
            // coalesced store of the tile: rows h, tokens t0 .. t0+kZTile
            const int tile_n = min(kZTile, j_end - t0);
            for (int idx = tid; idx < Hq * kZTile; idx += kRuleThreads) {
                const int h = idx / kZTile, t = idx % kZTile;
                if (t < tile_n)
                    store_f32_hint(a.z + ((int64_t)l * Hq + h) * a.N + t0 + t, ztile[t * zpitch + h], pol_z);
            }
            __syncthreads();
        }
        // merge the lanes' running (max, sum) per head for this chunk
        if (writer) {
#pragma unroll
            for (int k = 0; k < P2; ++k) {
                if (k < nv && my_base + k < G) {
                    red_m[tp * Hq + g * G + my_base + k] = run_m[k];
                    red_s[tp * Hq + g * G + my_base + k] = run_s[k];
                }
            }
        }
        __syncthreads();
        for (int h = tid; h < Hq; h += kRuleThreads) {
            float2 acc = make_float2(-INFINITY, 0.f);
            for (int t = 0; t < P; ++t) acc = lse_merge(acc, make_float2(red_m[t * Hq + h], red_s[t * Hq + h]));
            a.part[((int64_t)l * Hq + h) * a.n_chunks + chunk] = acc;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Rule scores, pass 2 and 3
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) rule_lse_kernel(const float2* __restrict__ part, int rows, int n_chunks,
                                                       float* __restrict__ lse2) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= rows) return;
    float2 acc = make_float2(-INFINITY, 0.f);
    for (int c = lane; c < n_chunks; c += 32) acc = lse_merge(acc, part[(int64_t)warp * n_chunks + c]);
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        float2 other = make_float2(__shfl_xor_sync(kFull, acc.x, o), __shfl_xor_sync(kFull, acc.y, o));
        acc = lse_merge(acc, other);
    }
    if (lane == 0) lse2[warp] = acc.y > 0.f ? acc.x + log2f(acc.y) : -INFINITY;
}

// Block = 8 warps x 32 tokens; warp w sums its share of the (l,h) rows for its
// lane's token; the 8 partial sums are added in warp order.
__global__ void __launch_bounds__(256) rule_accum_kernel(const float* __restrict__ z, const float* __restrict__ lse2,
                                                         int rows, int N, int pi, int q_s, int q_e,
                                                         float* __restrict__ rule) {
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

template <int G, bool BF16>
cudaError_t launch_logits(const RuleArgs& a, int grid, size_t smem, cudaStream_t s) {
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(rule_logits_kernel<G, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    rule_logits_kernel<G, BF16><<<grid, kRuleThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <bool BF16>
cudaError_t dispatch_logits(int G, const RuleArgs& a, int grid, size_t smem, cudaStream_t s) {
    switch (G) {
        case 1: return launch_logits<1, BF16>(a, grid, smem, s);
        case 2: return launch_logits<2, BF16>(a, grid, smem, s);
        case 3: return launch_logits<3, BF16>(a, grid, smem, s);
        case 4: return launch_logits<4, BF16>(a, grid, smem, s);
        case 5: return launch_logits<5, BF16>(a, grid, smem, s);
        case 6: return launch_logits<6, BF16>(a, grid, smem, s);
        case 7: return launch_logits<7, BF16>(a, grid, smem, s);
        case 8: return launch_logits<8, BF16>(a, grid, smem, s);
    }
    return cudaErrorInvalidValue;
}

int rule_chunks(int N) {
    const int chunk_len = kZTile * kChunkTiles;
    return (N + chunk_len - 1) / chunk_len;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

cudaError_t launch_memory_update(const void* q, int dtype, int L, int Hq, int R, int D, float lambda, int first_turn,
                                 int norm_mode, float* M, float* A, cudaStream_t s) {
    const float decay = expf(-lambda);
    const int vec = dtype == KVSEL_BF16 ? 8 : 4;
    const int rpi = 256 / (D / vec);
    const size_t smem = sizeof(float) * ((size_t)rpi * D + D);
    const int heads = L * Hq;
    if (dtype == KVSEL_BF16) {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(memory_update_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        memory_update_kernel<__nv_bfloat16><<<heads, 256, smem, s>>>(static_cast<const __nv_bfloat16*>(q), R, D, decay,
                                                                      first_turn, norm_mode, M, A);
    } else {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(memory_update_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        memory_update_kernel<float><<<heads, 256, smem, s>>>(static_cast<const float*>(q), R, D, decay, first_turn,
                                                             norm_mode, M, A);
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
    a.n_chunks = rule_chunks(N);
    a.z = reinterpret_cast<float*>(w);
    w += align256(rows * N * sizeof(float));
    a.part = reinterpret_cast<float2*>(w);
    w += align256(rows * a.n_chunks * sizeof(float2));
    float* lse2 = reinterpret_cast<float*>(w);
    a.dev_err = ctx->dev_err;
    const int64_t es = dtype == KVSEL_BF16 ? 2 : 4;
    a.aligned32 = (reinterpret_cast<uintptr_t>(k_pool) % 32 == 0) && (layer_stride * es) % 32 == 0 &&
                  (slot_stride * es) % 32 == 0;

    const int G = Hq / Hkv;
    const int TT = Hkv * (D / 16);
    const int P = kRuleThreads / TT;
    const size_t smem = sizeof(float) * ((size_t)kZTile * (Hq + 1) + 2 * (size_t)P * Hq);
    const int items = L * a.n_chunks;
    const int grid = items < 2 * ctx->num_sms ? items : 2 * ctx->num_sms;
    cudaError_t e = dtype == KVSEL_BF16 ? dispatch_logits<true>(G, a, grid, smem, s)
                                        : dispatch_logits<false>(G, a, grid, smem, s);
    if (e != cudaSuccess) return e;
    rule_lse_kernel<<<(int)((rows * 32 + 255) / 256), 256, 0, s>>>(a.part, (int)rows, a.n_chunks, lse2);
    const size_t smem3 = rows * sizeof(float);
    if (smem3 > 48 * 1024)
        cudaFuncSetAttribute(rule_accum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem3);
    rule_accum_kernel<<<(N + 31) / 32, 256, smem3, s>>>(a.z, lse2, (int)rows, N, pi, q_s, q_e, rule);
    return cudaGetLastError();
}

cudaError_t launch_redirect(const int32_t* slot_in, const uint8_t* keep, int N, int32_t dead, int32_t* slot_out,
                            cudaStream_t s) {
    int grid = (N + 255) / 256;
    if (grid > 4096) grid = 4096;
    redirect_kernel<<<grid, 256, 0, s>>>(slot_in, keep, N, dead, slot_out);
    return cudaGetLastError();
}

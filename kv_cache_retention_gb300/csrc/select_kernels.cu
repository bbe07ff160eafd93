// Budgeted top-k with a forced set (IntentKV Sec. 3.1, Eq. 1), also used for
// the KVMEM working set (sink + recent blocks forced, top-R_b candidates).
//
// One 1024-thread block: four 8-bit radix passes over order-preserving
// uint32 keys find the need-th largest candidate key (the threshold); a final
// pass keeps every forced position, every candidate above the threshold, and
// the lowest-index candidates equal to it until `need` are taken; block-wide
// exclusive scans over per-thread contiguous index ranges write the kept
// indices in ascending order.  The keep set is therefore a pure function of
// the scores: ties resolve to the lower index, NaN ranks lowest, -0 == +0.
#include "kvsel_internal.h"

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ uint32_t score_key(float f) {
    if (f != f) return 0u;     // NaN: below every number
    if (f == 0.0f) f = 0.0f;   // -0 -> +0
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ bool is_forced(int j, int pi, int q_s, int q_e) {
    return j < pi || (j >= q_s && j < q_e);
}

// Exclusive prefix sum over the block, in thread order; returns the total too.
__device__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(kFull, wi, o);
            if (lane >= o) wi += t;
        }
        warp_sums[lane] = wi - w;  // exclusive
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    const int excl = warp_sums[warp] + incl - v;
    total = warp_sums[32];
    __syncthreads();
    return excl;
}

// need: candidates to keep by score; n_cand: |H|.  need == n_cand keeps all.
__global__ void __launch_bounds__(kThreads) topk_kernel(const float* __restrict__ score, int N, int pi, int q_s,
                                                        int q_e, int need, int n_cand, uint8_t* __restrict__ keep,
                                                        int32_t* __restrict__ keep_idx) {
    __shared__ uint32_t hist[kWarps][256];
    __shared__ uint32_t bins[256];
    __shared__ int warp_sums[33];
    __shared__ uint32_t s_prefix, s_remaining;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0, mask = 0, remaining = (uint32_t)need;
    const bool select = need > 0 && need < n_cand;

    if (select) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < kWarps * 256; i += kThreads) (&hist[0][0])[i] = 0;
            __syncthreads();
            for (int j = tid; j < N; j += kThreads) {
                if (is_forced(j, pi, q_s, q_e)) continue;
                const uint32_t k = score_key(__ldg(score + j));
                if ((k & mask) == prefix) atomicAdd(&hist[warp][(k >> shift) & 255u], 1u);
            }
            __syncthreads();
            for (int b = tid; b < 256; b += kThreads) {
                uint32_t c = 0;
                for (int w = 0; w < kWarps; ++w) c += hist[w][b];
                bins[b] = c;
            }
            __syncthreads();
            if (warp == 0) {
                // lane L covers digits 255-8L .. 248-8L (descending)
                uint32_t cnt[8], lsum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    cnt[i] = bins[255 - 8 * lane - i];
                    lsum += cnt[i];
                }
                uint32_t incl = lsum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    uint32_t t = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += t;
                }
                const uint32_t excl = incl - lsum;  // count of larger digits
                if (excl < remaining && remaining <= incl) {
                    uint32_t above = excl;
                    int digit = 255 - 8 * lane;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (above + cnt[i] >= remaining) {
                            digit = 255 - 8 * lane - i;
                            break;
                        }
                        above += cnt[i];
                    }
                    s_prefix = prefix | ((uint32_t)digit << shift);
                    s_remaining = remaining - above;
                }
            }
            __syncthreads();
            prefix = s_prefix;
            remaining = s_remaining;
            mask |= 255u << shift;
            __syncthreads();
        }
    }
    // prefix is now the threshold key; `remaining` candidates equal to it are kept.
    const uint32_t thr = prefix;
    const bool keep_all = need >= n_cand;
    const int seg = (N + kThreads - 1) / kThreads;
    const int j0 = min(N, tid * seg), j1 = min(N, j0 + seg);

    int ties = 0;
    if (select)
        for (int j = j0; j < j1; ++j)
            if (!is_forced(j, pi, q_s, q_e) && score_key(__ldg(score + j)) == thr) ++ties;
    int total;
    const int tie_base = block_exclusive_scan(ties, warp_sums, total);

    int kept = 0;
    {
        int tie_rank = tie_base;
        for (int j = j0; j < j1; ++j) {
            bool k;
            if (is_forced(j, pi, q_s, q_e) || keep_all) {
                k = true;
            } else if (!select) {
                k = false;
            } else {
                const uint32_t key = score_key(__ldg(score + j));
                k = key > thr || (key == thr && (uint32_t)(tie_rank++) < remaining);
            }
            kept += k;
        }
    }
    const int out_base = block_exclusive_scan(kept, warp_sums, total);
    int pos = out_base, tie_rank = tie_base;
    for (int j = j0; j < j1; ++j) {
        bool k;
        if (is_forced(j, pi, q_s, q_e) || keep_all) {
            k = true;
        } else if (!select) {
            k = false;
        } else {
            const uint32_t key = score_key(__ldg(score + j));
            k = key > thr || (key == thr && (uint32_t)(tie_rank++) < remaining);
        }
        if (keep) keep[j] = (uint8_t)k;
        if (k && keep_idx) keep_idx[pos] = j;
        pos += k;
    }
}

}  // namespace

cudaError_t launch_topk(const float* score, int N, int pi, int q_s, int q_e, int need, int n_cand, uint8_t* keep,
                        int32_t* keep_idx, cudaStream_t s) {
    topk_kernel<<<1, kThreads, 0, s>>>(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx);
    return cudaGetLastError();
}

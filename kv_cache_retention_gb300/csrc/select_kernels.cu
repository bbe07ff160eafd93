// Budgeted top-k with a forced set (IntentKV Sec. 3.1, Eq. 1), also used for
// the KVMEM working set (sink + recent blocks forced, top-R_b candidates).
//
// Four 8-bit radix passes over order-preserving uint32 keys find the need-th
// largest candidate key (the threshold); a final pass keeps every forced
// position, every candidate above the threshold, and the lowest-index
// candidates equal to it until `need` are taken; exclusive scans over
// per-thread contiguous index ranges write the kept indices in ascending order.
// The keep set is therefore a pure function of the scores: ties resolve to the
// lower index, NaN ranks lowest, -0 == +0.
//
// N <= 16384: one CTA, keys in registers.  N <= 131072: the same code on one
// cluster of 8 CTAs, histograms merged through distributed shared memory.  Larger
// N: one 1024-thread block re-reading the scores for each pass.
#include <cooperative_groups.h>

#include <vector>

#include "kvsel_internal.h"

namespace cg = cooperative_groups;

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

// ---------------------------------------------------------------------------
// Cluster variant: 8 CTAs x 1024 threads, each thread holding up to kKeys keys
// of a contiguous index range in registers (N <= 8 * 1024 * kKeys).  Each radix
// pass builds per-CTA histograms in shared memory; every CTA then sums the 8
// histograms through distributed shared memory and takes the same digit
// decision.  The ordered compaction uses block scans plus the lower-ranked
// CTAs' totals read through distributed shared memory.  Cluster barriers are
// hardware barriers: no thread spins.
// ---------------------------------------------------------------------------
constexpr int kCluster = 8;
constexpr int kKeys = 16;
constexpr int kClusterCap = kCluster * kThreads * kKeys;

// One selection of a batched launch.
struct TopkJob {
    const float* score;
    int N, pi, q_s, q_e, need, n_cand;
    uint8_t* keep;
    int32_t* keep_idx;
};

// The selection over a cluster of CL CTAs.  batch: NULL, or one TopkJob per
// cluster (cluster c = CTAs CL*c .. CL*c + CL - 1 takes batch[c]); the scalar
// arguments are then ignored.  CL = 1 is a plain (non-cluster) launch of one CTA
// per selection.
// Cluster barrier and distributed shared memory view; a lone CTA (CL = 1) uses a
// block barrier and its own shared memory.
template <int CL>
__device__ __forceinline__ void csync() {
    if constexpr (CL == 1)
        __syncthreads();
    else
        cg::this_cluster().sync();
}
template <int CL, typename T>
__device__ __forceinline__ T* cmap(T* p, int r) {
    if constexpr (CL == 1)
        return p;
    else
        return cg::this_cluster().map_shared_rank(p, r);
}

template <int CL>
__device__ __forceinline__ void topk_select(const float* __restrict__ score, int N, int pi, int q_s, int q_e, int need,
                                            int n_cand, uint8_t* __restrict__ keep, int32_t* __restrict__ keep_idx,
                                            const TopkJob* __restrict__ batch) {
    if (batch) {
        const TopkJob& b = batch[blockIdx.x / CL];
        score = b.score;
        N = b.N;
        pi = b.pi;
        q_s = b.q_s;
        q_e = b.q_e;
        need = b.need;
        n_cand = b.n_cand;
        keep = b.keep;
        keep_idx = b.keep_idx;
    }
    __shared__ uint32_t sub[8][256];        // per-warp-group sub-histograms
    __shared__ uint32_t hist[2][256];       // this CTA's histogram, double-buffered across passes
    __shared__ uint32_t tot[256];
    __shared__ int warp_sums[33];
    __shared__ int cta_tot[2];              // this CTA's (ties, kept) totals
    __shared__ uint32_t s_prefix, s_remaining;
    int rank = 0;
    if constexpr (CL > 1) rank = (int)cg::this_cluster().block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // contiguous ranges: CTA rank -> [cb, ce), thread -> [j0, j1)
    const int per_cta = (N + CL - 1) / CL;
    const int cb = min(N, rank * per_cta), ce = min(N, cb + per_cta);
    const int per_thr = (ce - cb + kThreads - 1) / kThreads;
    const int j0 = min(ce, cb + tid * per_thr), j1 = min(ce, j0 + per_thr);
    uint32_t key[kKeys];
    uint32_t cand_mask = 0;  // bit k: element j0+k is a candidate (not forced)
#pragma unroll
    for (int k = 0; k < kKeys; ++k) {
        const int j = j0 + k;
        key[k] = 0;
        if (j < j1) {
            key[k] = score_key(__ldg(score + j));
            if (!is_forced(j, pi, q_s, q_e)) cand_mask |= 1u << k;
        }
    }
    const bool select = need > 0 && need < n_cand;
    const bool keep_all = need >= n_cand;
    uint32_t prefix = 0, mask = 0, remaining = (uint32_t)need;
    if (select) {
        int buf = 0;
        for (int shift = 24; shift >= 0; shift -= 8, buf ^= 1) {
            for (int i = tid; i < 8 * 256; i += kThreads) (&sub[0][0])[i] = 0;
            __syncthreads();
#pragma unroll
            for (int k = 0; k < kKeys; ++k)
                if (((cand_mask >> k) & 1u) && (key[k] & mask) == prefix)
                    atomicAdd(&sub[warp & 7][(key[k] >> shift) & 255u], 1u);
            __syncthreads();
            if (tid < 256) {
                uint32_t c = 0;
#pragma unroll
                for (int w = 0; w < 8; ++w) c += sub[w][tid];
                hist[buf][tid] = c;
            }
            csync<CL>();  // every CTA's histogram is complete
            if (tid < 256) {
                uint32_t c = 0;
                for (int r = 0; r < CL; ++r) c += cmap<CL>(&hist[buf][0], r)[tid];
                tot[tid] = c;
            }
            __syncthreads();
            if (warp == 0) {
                uint32_t cnt[8], lsum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    cnt[i] = tot[255 - 8 * lane - i];
                    lsum += cnt[i];
                }
                uint32_t incl = lsum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    uint32_t t = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += t;
                }
                const uint32_t excl = incl - lsum;
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
        }
    }
    const uint32_t thr = prefix;

    // ties equal to the threshold, in global index order
    int ties = 0;
    if (select) {
#pragma unroll
        for (int k = 0; k < kKeys; ++k) ties += ((cand_mask >> k) & 1u) && key[k] == thr;
    }
    int total;
    int tie_base = block_exclusive_scan(ties, warp_sums, total);
    if (tid == 0) cta_tot[0] = total;
    csync<CL>();
    for (int r = 0; r < rank; ++r) tie_base += cmap<CL>(&cta_tot[0], r)[0];

    int kept = 0;
    uint32_t keep_bits = 0;
    {
        int tie_rank = tie_base;
#pragma unroll
        for (int k = 0; k < kKeys; ++k) {
            if (j0 + k >= j1) continue;
            bool kk;
            if (!((cand_mask >> k) & 1u) || keep_all) {
                kk = true;
            } else if (!select) {
                kk = false;
            } else {
                kk = key[k] > thr || (key[k] == thr && (uint32_t)(tie_rank++) < remaining);
            }
            keep_bits |= (uint32_t)kk << k;
            kept += kk;
        }
    }
    int out_base = block_exclusive_scan(kept, warp_sums, total);
    if (tid == 0) cta_tot[1] = total;
    csync<CL>();
    for (int r = 0; r < rank; ++r) out_base += cmap<CL>(&cta_tot[1], r)[0];
    int pos = out_base;
#pragma unroll
    for (int k = 0; k < kKeys; ++k) {
        if (j0 + k >= j1) continue;
        const bool kk = (keep_bits >> k) & 1u;
        if (keep) keep[j0 + k] = (uint8_t)kk;
        if (kk && keep_idx) keep_idx[pos] = j0 + k;
        pos += kk;
    }
    csync<CL>();  // no CTA leaves while another may still read its shared memory
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    topk_cluster_kernel(const float* __restrict__ score, int N, int pi, int q_s, int q_e, int need, int n_cand,
                        uint8_t* __restrict__ keep, int32_t* __restrict__ keep_idx, const TopkJob* __restrict__ batch) {
    topk_select<kCluster>(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx, batch);
}

// N <= kCtaCap: one CTA, no cluster launch and no cross-CTA barrier.
constexpr int kCtaCap = kThreads * kKeys;
__global__ void __launch_bounds__(kThreads)
    topk_cta_kernel(const float* __restrict__ score, int N, int pi, int q_s, int q_e, int need, int n_cand,
                    uint8_t* __restrict__ keep, int32_t* __restrict__ keep_idx, const TopkJob* __restrict__ batch) {
    topk_select<1>(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx, batch);
}

}  // namespace

cudaError_t launch_topk(const float* score, int N, int pi, int q_s, int q_e, int need, int n_cand, uint8_t* keep,
                        int32_t* keep_idx, cudaStream_t s) {
    if (N <= kCtaCap)
        topk_cta_kernel<<<1, kThreads, 0, s>>>(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx, nullptr);
    else if (N <= kClusterCap)
        topk_cluster_kernel<<<kCluster, kThreads, 0, s>>>(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx, nullptr);
    else
        topk_kernel<<<1, kThreads, 0, s>>>(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx);
    return cudaGetLastError();
}

size_t topk_batch_workspace(int S) { return (size_t)S * sizeof(TopkJob) + 256; }

// Sessions that fit one cluster share one launch (a cluster each, or a CTA each when
// every such session fits one CTA); larger ones take the single-CTA re-reading
// kernel one by one.  need / n_cand per session as kvsel_topk_retain.
cudaError_t launch_topk_batch(const kvsel_topk_session* sess, const int* need, const int* n_cand, int S, void* ws,
                              cudaStream_t s) {
    std::vector<TopkJob> jobs;
    jobs.reserve((size_t)S);
    for (int i = 0; i < S; ++i) {
        const kvsel_topk_session& x = sess[i];
        if (x.N == 0) continue;
        if (x.N > kClusterCap) {
            topk_kernel<<<1, kThreads, 0, s>>>(x.rule, x.N, x.pi, x.q_s, x.q_e, need[i], n_cand[i], x.keep, x.keep_idx);
            continue;
        }
        jobs.push_back(TopkJob{x.rule, x.N, x.pi, x.q_s, x.q_e, need[i], n_cand[i], x.keep, x.keep_idx});
    }
    if (!jobs.empty()) {
        TopkJob* dev = static_cast<TopkJob*>(ws);
        cudaError_t e = cudaMemcpyAsync(dev, jobs.data(), jobs.size() * sizeof(TopkJob), cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return e;
        bool small = true;
        for (const TopkJob& j : jobs) small = small && j.N <= kCtaCap;
        if (small)
            topk_cta_kernel<<<(unsigned)jobs.size(), kThreads, 0, s>>>(nullptr, 0, 0, 0, 0, 0, 0, nullptr, nullptr, dev);
        else
            topk_cluster_kernel<<<(unsigned)(kCluster * jobs.size()), kThreads, 0, s>>>(nullptr, 0, 0, 0, 0, 0, 0,
                                                                                       nullptr, nullptr, dev);
    }
    return cudaGetLastError();
}

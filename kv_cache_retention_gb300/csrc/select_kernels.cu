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
// N <= KVSEL_TOPK_CTA_MAX (8192; 16384 at most): one CTA, keys in registers.
// N <= 131072: the same code on one cluster of 8 CTAs, histograms merged through
// distributed shared memory; N <= 262144: a cluster of 16 (where the GPU can
// place one).  Larger N: the grid-wide variant below (several launches, a small
// workspace).
#include <cooperative_groups.h>

#include <vector>

#include "kvsel_internal.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 1024;
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

// Exclusive prefix sum over the block (any multiple of 32 threads up to 1024), in
// thread order; returns the total too.
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
        int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
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

// Sessions of up to 262144 positions: a cluster of 16 CTAs (a size the GPU allows
// only on request, and places only where a GPC has 16 SMs free).
constexpr int kCluster16 = 16;
constexpr int kCluster16Cap = kCluster16 * kThreads * kKeys;
__global__ void __cluster_dims__(kCluster16, 1, 1) __launch_bounds__(kThreads)
    topk_cluster16_kernel(const float* __restrict__ score, int N, int pi, int q_s, int q_e, int need, int n_cand,
                          uint8_t* __restrict__ keep, int32_t* __restrict__ keep_idx) {
    topk_select<kCluster16>(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx, nullptr);
}

// Whether a 16-CTA cluster of topk_cluster16_kernel can run on the current device
// (asked once per device).
bool cluster16_ok() {
    static int state[64] = {};  // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (state[dev] == 0) {
        int n = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kCluster16);
        cfg.blockDim = dim3(kThreads);
        bool ok = cudaFuncSetAttribute(topk_cluster16_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                      cudaSuccess &&
                  cudaOccupancyMaxActiveClusters(&n, topk_cluster16_kernel, &cfg) == cudaSuccess && n > 0;
        cudaGetLastError();  // a refused query leaves no error behind
        state[dev] = ok ? 1 : 2;
    }
    return state[dev] == 1;
}

// N <= kCtaCap: one CTA, no cluster launch and no cross-CTA barrier.  Above
// KVSEL_TOPK_CTA_MAX the cluster path is faster even where one CTA holds the keys.
#ifndef KVSEL_TOPK_CTA_MAX
#define KVSEL_TOPK_CTA_MAX 8192
#endif
constexpr int kCtaCap = KVSEL_TOPK_CTA_MAX < kThreads * kKeys ? KVSEL_TOPK_CTA_MAX : kThreads * kKeys;
__global__ void __launch_bounds__(kThreads)
    topk_cta_kernel(const float* __restrict__ score, int N, int pi, int q_s, int q_e, int need, int n_cand,
                    uint8_t* __restrict__ keep, int32_t* __restrict__ keep_idx, const TopkJob* __restrict__ batch) {
    topk_select<1>(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx, batch);
}


// ---------------------------------------------------------------------------
// Grid-wide variant for sessions too long for one cluster: the same selection in
// several launches.  Four radix passes each count, among the candidates whose key
// matches the digits chosen so far, the next 8-bit digit into a global histogram
// (per-block shared-memory histograms merged with atomics) and let one warp pick
// the digit.  Three launches then count, per block of 4096 positions, the
// candidates tied with the threshold and the positions kept outright, scan those
// counts in block order (ties go to the lower index), and write the keep mask
// and the ascending kept indices.  Only integer counts are combined, so the
// result does not depend on the order of the atomics.
// ---------------------------------------------------------------------------
struct GridTopkState {
    uint32_t hist[4][256];
    uint32_t prefix, remaining;
};
constexpr int kGridThreads = 256;
constexpr int kGridPer = 16;                           // positions per thread in the final launches
constexpr int kGridChunk = kGridThreads * kGridPer;    // positions per block in the final launches

__global__ void __launch_bounds__(kGridThreads) topk_grid_init(GridTopkState* st, int need) {
    for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x) (&st->hist[0][0])[i] = 0u;
    if (threadIdx.x == 0) {
        st->prefix = 0u;
        st->remaining = (uint32_t)need;
    }
}

__global__ void __launch_bounds__(kGridThreads) topk_grid_hist(const float* __restrict__ score, int N, int pi,
                                                                 int q_s, int q_e, GridTopkState* st, int pass) {
    __shared__ uint32_t h[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0u;
    __syncthreads();
    const int shift = 24 - 8 * pass;
    const uint32_t mask = pass == 0 ? 0u : 0xffffffffu << (shift + 8);  // the digits chosen so far
    const uint32_t prefix = st->prefix;
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < N; j += gridDim.x * blockDim.x) {
        if (is_forced(j, pi, q_s, q_e)) continue;
        const uint32_t k = score_key(__ldg(score + j));
        if ((k & mask) == prefix) atomicAdd(&h[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
        if (h[i]) atomicAdd(&st->hist[pass][i], h[i]);
}

// One warp: the digit at which the count of larger keys reaches `remaining`.
__global__ void topk_grid_digit(GridTopkState* st, int pass) {
    const int lane = threadIdx.x;
    const int shift = 24 - 8 * pass;
    const uint32_t remaining = st->remaining;
    uint32_t cnt[8], lsum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // lane L covers digits 255-8L .. 248-8L (descending)
        cnt[i] = st->hist[pass][255 - 8 * lane - i];
        lsum += cnt[i];
    }
    uint32_t incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
    }
    const uint32_t excl = incl - lsum;  // keys with a larger digit
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
        st->prefix |= (uint32_t)digit << shift;
        st->remaining = remaining - above;
    }
}

// Per position: kept outright (forced, every candidate when all are kept, or a key
// above the threshold) or tied with the threshold.  mode 0: no candidate is kept,
// 1: every candidate is, 2: the threshold in st decides.
__device__ __forceinline__ void grid_class(const float* __restrict__ score, int j, int pi, int q_s, int q_e, int mode,
                                           uint32_t thr, bool& sure, bool& tie) {
    if (is_forced(j, pi, q_s, q_e) || mode == 1) {
        sure = true;
        tie = false;
    } else if (mode == 0) {
        sure = tie = false;
    } else {
        const uint32_t k = score_key(__ldg(score + j));
        sure = k > thr;
        tie = k == thr;
    }
}

__device__ __forceinline__ int block_sum(int v, int* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
    __syncthreads();
    return t;
}

__global__ void __launch_bounds__(kGridThreads) topk_grid_count(const float* __restrict__ score, int N, int pi,
                                                                  int q_s, int q_e, int mode,
                                                                  const GridTopkState* st, int* ties, int* sure) {
    __shared__ int red[kGridThreads / 32];
    const uint32_t thr = mode == 2 ? st->prefix : 0u;
    const int j0 = blockIdx.x * kGridChunk + threadIdx.x * kGridPer, j1 = min(N, j0 + kGridPer);
    int nt = 0, ns = 0;
    for (int j = j0; j < j1; ++j) {
        bool s1, t1;
        grid_class(score, j, pi, q_s, q_e, mode, thr, s1, t1);
        ns += s1;
        nt += t1;
    }
    nt = block_sum(nt, red);
    ns = block_sum(ns, red);
    if (threadIdx.x == 0) {
        ties[blockIdx.x] = nt;
        sure[blockIdx.x] = ns;
    }
}

// One block: in block order, the ties before each block and the kept positions
// before each block (ties taken while `remaining` lasts).
__global__ void __launch_bounds__(1024) topk_grid_scan(const GridTopkState* st, int mode, int n_blocks,
                                                         const int* ties, const int* sure, int* tie_base,
                                                         int* out_base) {
    __shared__ int warp_sums[33];
    const int64_t remaining = mode == 2 ? (int64_t)st->remaining : 0;
    int carry_t = 0, carry_o = 0;
    for (int b0 = 0; b0 < n_blocks; b0 += 1024) {
        const int b = b0 + (int)threadIdx.x;
        const int t = b < n_blocks ? ties[b] : 0;
        int total_t;
        const int tb = carry_t + block_exclusive_scan(t, warp_sums, total_t);
        int64_t take = remaining - tb;
        take = take < 0 ? 0 : (take > t ? t : take);
        const int kept = (b < n_blocks ? sure[b] : 0) + (int)take;
        int total_o;
        const int ob = carry_o + block_exclusive_scan(kept, warp_sums, total_o);
        if (b < n_blocks) {
            tie_base[b] = tb;
            out_base[b] = ob;
        }
        carry_t += total_t;
        carry_o += total_o;
    }
}

__global__ void __launch_bounds__(kGridThreads) topk_grid_write(const float* __restrict__ score, int N, int pi,
                                                                  int q_s, int q_e, int mode,
                                                                  const GridTopkState* st, const int* tie_base,
                                                                  const int* out_base, uint8_t* __restrict__ keep,
                                                                  int32_t* __restrict__ keep_idx) {
    __shared__ int warp_sums[33];
    const uint32_t thr = mode == 2 ? st->prefix : 0u;
    const uint32_t remaining = mode == 2 ? st->remaining : 0u;
    const int j0 = blockIdx.x * kGridChunk + threadIdx.x * kGridPer, j1 = min(N, j0 + kGridPer);
    int nt = 0;
    for (int j = j0; j < j1; ++j) {
        bool s1, t1;
        grid_class(score, j, pi, q_s, q_e, mode, thr, s1, t1);
        nt += t1;
    }
    int total;
    int tie_rank = tie_base[blockIdx.x] + block_exclusive_scan(nt, warp_sums, total);
    int nk = 0;
    {
        int r = tie_rank;
        for (int j = j0; j < j1; ++j) {
            bool s1, t1;
            grid_class(score, j, pi, q_s, q_e, mode, thr, s1, t1);
            nk += s1 || (t1 && (uint32_t)(r++) < remaining);
        }
    }
    int pos = out_base[blockIdx.x] + block_exclusive_scan(nk, warp_sums, total);
    for (int j = j0; j < j1; ++j) {
        bool s1, t1;
        grid_class(score, j, pi, q_s, q_e, mode, thr, s1, t1);
        const bool k = s1 || (t1 && (uint32_t)(tie_rank++) < remaining);
        if (keep) keep[j] = (uint8_t)k;
        if (k && keep_idx) keep_idx[pos] = j;
        pos += k;
    }
}

size_t grid_workspace(int N) {
    const size_t nb = ((size_t)N + kGridChunk - 1) / kGridChunk;
    return ((sizeof(GridTopkState) + 255) & ~(size_t)255) + 4 * nb * sizeof(int) + 256;
}

cudaError_t launch_topk_grid(const float* score, int N, int pi, int q_s, int q_e, int need, int n_cand,
                             uint8_t* keep, int32_t* keep_idx, void* ws, cudaStream_t s) {
    GridTopkState* st = static_cast<GridTopkState*>(ws);
    const int nb = (N + kGridChunk - 1) / kGridChunk;
    int* ties = reinterpret_cast<int*>(static_cast<char*>(ws) + ((sizeof(GridTopkState) + 255) & ~(size_t)255));
    int* sure = ties + nb;
    int* tie_base = sure + nb;
    int* out_base = tie_base + nb;
    const int mode = need <= 0 ? 0 : (need >= n_cand ? 1 : 2);
    if (mode == 2) {
        topk_grid_init<<<1, kGridThreads, 0, s>>>(st, need);
        int hist_blocks = (N + kGridThreads * 8 - 1) / (kGridThreads * 8);
        hist_blocks = hist_blocks < 1024 ? hist_blocks : 1024;
        for (int pass = 0; pass < 4; ++pass) {
            topk_grid_hist<<<hist_blocks, kGridThreads, 0, s>>>(score, N, pi, q_s, q_e, st, pass);
            topk_grid_digit<<<1, 32, 0, s>>>(st, pass);
        }
    }
    topk_grid_count<<<nb, kGridThreads, 0, s>>>(score, N, pi, q_s, q_e, mode, st, ties, sure);
    topk_grid_scan<<<1, 1024, 0, s>>>(st, mode, nb, ties, sure, tie_base, out_base);
    topk_grid_write<<<nb, kGridThreads, 0, s>>>(score, N, pi, q_s, q_e, mode, st, tie_base, out_base, keep, keep_idx);
    return cudaGetLastError();
}

}  // namespace

// Above one 8-CTA cluster the grid-wide path may run (it does wherever the 16-CTA
// cluster cannot be placed), so its workspace is reserved for every such N.
size_t topk_workspace(int N) { return N > kClusterCap ? grid_workspace(N) : 0; }

cudaError_t launch_topk(const float* score, int N, int pi, int q_s, int q_e, int need, int n_cand, uint8_t* keep,
                        int32_t* keep_idx, void* ws, cudaStream_t s) {
    if (N <= kCtaCap)
        topk_cta_kernel<<<1, kThreads, 0, s>>>(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx, nullptr);
    else if (N <= kClusterCap)
        topk_cluster_kernel<<<kCluster, kThreads, 0, s>>>(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx, nullptr);
    else if (N <= kCluster16Cap && cluster16_ok())
        topk_cluster16_kernel<<<kCluster16, kThreads, 0, s>>>(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx);
    else
        return launch_topk_grid(score, N, pi, q_s, q_e, need, n_cand, keep, keep_idx, ws, s);
    return cudaGetLastError();
}

size_t topk_batch_workspace(int S, int max_N) {
    return (((size_t)S * sizeof(TopkJob) + 255) & ~(size_t)255) + topk_workspace(max_N);
}

// Sessions that fit one cluster share one launch (a cluster each, or a CTA each when
// every such session fits one CTA); larger ones take launch_topk's paths (16-CTA
// cluster or grid-wide) one by one.  need / n_cand per session as kvsel_topk_retain.
cudaError_t launch_topk_batch(const kvsel_topk_session* sess, const int* need, const int* n_cand, int S, void* ws,
                              cudaStream_t s) {
    std::vector<TopkJob> jobs;
    jobs.reserve((size_t)S);
    for (int i = 0; i < S; ++i) {
        const kvsel_topk_session& x = sess[i];
        if (x.N == 0) continue;
        if (x.N > kClusterCap) {  // one at a time, on the grid-wide path's share of the workspace
            void* gws = static_cast<char*>(ws) + (((size_t)S * sizeof(TopkJob) + 255) & ~(size_t)255);
            cudaError_t e = launch_topk(x.rule, x.N, x.pi, x.q_s, x.q_e, need[i], n_cand[i], x.keep, x.keep_idx, gws, s);
            if (e != cudaSuccess) return e;
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

// KVMEM differential working-set update (section "engineering: tiered
// movement, page-table aliasing and position-consistent rebuild"): of the new
// working set W_t only the blocks absent from the resident set G_{t-1} are
// moved in; retained blocks keep their page, and the pages of blocks that left
// are reused.  Integer work on a few thousand entries: one CTA.
//
//   retained  (in W_t and G_{t-1}): page kept; compact position moves by
//             shift = (new rank - old rank) * page
//   incoming  (in W_t only): the free pages of the pool -- every page not held
//             by a retained block -- in ascending page order, incoming blocks
//             in ascending block id
//   outgoing  (in G_{t-1} only): page released
// Both sets are ascending block ids; membership is a binary search in the other
// set; the ordered lists come from block-wide exclusive scans.
#include "kvsel_internal.h"

namespace {

constexpr int kThreads = 1024;
constexpr unsigned kFull = 0xffffffffu;

// Exclusive prefix sum over the CTA of one value per thread; *total gets the sum.
__device__ __forceinline__ int cta_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < n_warps ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += y;
        }
        if (lane < n_warps) warp_sums[lane] = w;
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    *total = warp_sums[n_warps - 1];
    __syncthreads();  // warp_sums is reused by the next scan
    return before;
}

// Index of id in the ascending array a[0..n), or -1.
__device__ __forceinline__ int find_sorted(const int32_t* __restrict__ a, int n, int id) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a + mid) < id)
            lo = mid + 1;
        else
            hi = mid;
    }
    return (lo < n && __ldg(a + lo) == id) ? lo : -1;
}

__global__ void __launch_bounds__(kThreads) workset_diff_kernel(
    const int32_t* __restrict__ prev_ids, const int32_t* __restrict__ prev_pages, int n_prev,
    const int32_t* __restrict__ new_ids, int n_new, int P, int page, int32_t* new_pages, int32_t* shift,
    int32_t* in_rank, int32_t* in_page, int32_t* mv_rank, int32_t* mv_shift, int32_t* out_page, int32_t* counts,
    unsigned* dev_err) {
    extern __shared__ uint32_t held[];  // one bit per pool page
    __shared__ int warp_sums[32];
    const int tid = threadIdx.x;
    const int words = (P + 31) >> 5;
    for (int w = tid; w < words; w += blockDim.x) held[w] = 0u;
    __syncthreads();

    // retained entries keep their page; a page named twice or out of the pool is an error
    unsigned err = 0;
    for (int r = tid; r < n_new; r += blockDim.x) {
        const int id = __ldg(new_ids + r);
        if (r > 0 && __ldg(new_ids + r - 1) >= id) err |= KVSEL_DEV_BAD_SET;
        const int q = find_sorted(prev_ids, n_prev, id);
        int pg = -1;
        if (q >= 0) {
            pg = __ldg(prev_pages + q);
            if (pg < 0 || pg >= P) {
                err |= KVSEL_DEV_BAD_PAGE;
                pg = -1;
            } else if (atomicOr(&held[pg >> 5], 1u << (pg & 31)) & (1u << (pg & 31))) {
                err |= KVSEL_DEV_BAD_SET;
            }
        }
        new_pages[r] = pg;
        shift[r] = pg >= 0 ? (r - q) * page : 0;
    }
    for (int q = tid + 1; q < n_prev; q += blockDim.x)
        if (__ldg(prev_ids + q - 1) >= __ldg(prev_ids + q)) err |= KVSEL_DEV_BAD_SET;
    if (err) atomicOr(dev_err, err);
    __syncthreads();

    // incoming and moved ranks, ascending
    int n_in = 0, n_mv = 0;
    for (int c0 = 0; c0 < n_new; c0 += blockDim.x) {
        const int r = c0 + tid;
        const int pg = r < n_new ? new_pages[r] : 0;
        const int sh = r < n_new ? shift[r] : 0;
        const int f_in = (r < n_new && pg < 0) ? 1 : 0, f_mv = (r < n_new && pg >= 0 && sh != 0) ? 1 : 0;
        int t_in, t_mv;
        const int p_in = cta_scan(f_in, warp_sums, &t_in);
        const int p_mv = cta_scan(f_mv, warp_sums, &t_mv);
        if (f_in) in_rank[n_in + p_in] = r;
        if (f_mv) {
            mv_rank[n_mv + p_mv] = r;
            mv_shift[n_mv + p_mv] = sh;
        }
        n_in += t_in;
        n_mv += t_mv;
    }
    // outgoing pages, ascending block id
    int n_out = 0;
    for (int c0 = 0; c0 < n_prev; c0 += blockDim.x) {
        const int q = c0 + tid;
        const int f = (q < n_prev && find_sorted(new_ids, n_new, __ldg(prev_ids + q)) < 0) ? 1 : 0;
        int t;
        const int pre = cta_scan(f, warp_sums, &t);
        if (f) out_page[n_out + pre] = __ldg(prev_pages + q);
        n_out += t;
    }
    __syncthreads();  // in_rank complete before it is read below

    // the f-th free page (ascending) goes to the f-th incoming rank
    int n_free = 0;
    for (int c0 = 0; c0 < words && n_free < n_in; c0 += blockDim.x) {
        const int w = c0 + tid;
        uint32_t bits = 0u;
        if (w < words) {
            bits = ~held[w];
            const int valid = P - w * 32;
            if (valid < 32) bits &= (1u << valid) - 1u;
        }
        int t;
        int f = n_free + cta_scan(__popc(bits), warp_sums, &t);
        while (bits && f < n_in) {
            const int b = __ffs(bits) - 1;
            const int pg = w * 32 + b;
            in_page[f] = pg;
            new_pages[in_rank[f]] = pg;
            ++f;
            bits &= bits - 1u;
        }
        n_free += t;
    }
    if (tid == 0) {
        if (n_free < n_in) atomicOr(dev_err, (unsigned)KVSEL_DEV_POOL_FULL);
        counts[0] = n_in;
        counts[1] = n_mv;
        counts[2] = n_out;
    }
}

}  // namespace

cudaError_t launch_workset_diff(const int32_t* prev_ids, const int32_t* prev_pages, int n_prev,
                                const int32_t* new_ids, int n_new, int P, int page, int32_t* new_pages,
                                int32_t* shift, int32_t* in_rank, int32_t* in_page, int32_t* mv_rank,
                                int32_t* mv_shift, int32_t* out_page, int32_t* counts, unsigned* dev_err,
                                cudaStream_t s) {
    const size_t smem = sizeof(uint32_t) * (size_t)((P + 31) / 32);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(workset_diff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    workset_diff_kernel<<<1, kThreads, smem, s>>>(prev_ids, prev_pages, n_prev, new_ids, n_new, P, page, new_pages,
                                                  shift, in_rank, in_page, mv_rank, mv_shift, out_page, counts,
                                                  dev_err);
    return cudaGetLastError();
}

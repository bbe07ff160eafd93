// KVMEM block relevance R_b on the 5th-generation tensor cores (tcgen05).
//
// Retrieval step of the KVMEM page: for every (layer l, query head h, query
// token m) a softmax over the candidate blocks b in C of q . kbar / sqrt(d);
// the probabilities are summed over query tokens and averaged over all
// layer-heads.
//
// For one (layer l, kv head g) the G = Hq/Hkv query heads' rows form one
// contiguous [G*M][128] bf16 matrix Q_lg and the index one [Bcap][128] matrix
// K_lg.  The logits S = Q_lg K_lg^T are never stored; two passes recompute them
// on the tensor cores, each reducing along the axis its epilogue threads own:
//   row pass:    A = 128 query rows (TMEM lanes), B = 256 candidate blocks per
//                tile; each lane keeps an online (max, sum 2^x) over its row
//                -> lse2[r] = log2 sum_{b in C} 2^(S[r,b] log2e/sqrt(d))
//   column pass: A = 128 candidate blocks (TMEM lanes), B = 256 query rows per
//                tile; each lane sums 2^(S[b,r] log2e/sqrt(d) - lse2[r]) over
//                all rows of the group -> mass[lg][b], complete per CTA
//   finalize:    R[b] = sum_lg mass[lg][b] / (L*Hq), in fixed (l,g) order.
//
// Kernel structure (one persistent CTA per SM, 576 threads):
//   warp 0      TMA producer: A tile per unit, B tiles through a 2-stage ring
//               (128-byte swizzled, K-major, no multicast)
//   warp 1      allocates 512 TMEM columns; lane 0 issues tcgen05.mma
//               (kind::f16, bf16 x bf16 -> fp32, M=128 N=256 K=16, 8 per tile)
//               into one of two 256-column accumulators and commits to
//               mbarriers that free the smem stage and hand the accumulator on
//   warps 2-17  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31; four column slices of 64), exp2 on the MUFU,
//               packed fp32 adds; the accumulator is handed back as soon as it
//               is in registers
// Every mbarrier wait is bounded (1 s of globaltimer); on a timeout the CTA
// flags KVSEL_ERR_TIMEOUT in the device error word, drains its own copies and
// MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "kvsel_internal.h"

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kD = 128;
constexpr int BM = 128;                         // A rows per unit = TMEM lanes
constexpr int BN = 256;                         // B rows per tile = accumulator columns
constexpr int kABytes = BM * kD * 2;            // 32 KB: two 64-column K blocks of 16 KB
constexpr int kBBytes = BN * kD * 2;            // 64 KB: two K blocks of 32 KB
constexpr int kNA = 2, kNB = 2, kNAcc = 2;
constexpr int kTmemCols = 512;
constexpr int kEpiWarps = 16;                   // 4 TMEM lane quarters x kSlices column slices
constexpr int kSlices = kEpiWarps / 4;
constexpr int kSliceCols = BN / kSlices;        // accumulator columns per epilogue thread and tile
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;
constexpr uint64_t kWaitNs = 1000000000ull;     // 1 s per wait
constexpr uint32_t kSuspendNs = 20000;          // try_wait may park the thread this long (woken on completion)

// instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, N=256, M=128
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

struct TcArgs {
    int mode;          // 0 row pass, 1 column pass
    int n_units;
    int units_per_lg;
    int n_bt;          // B tiles per unit
    int rows_g;        // G*M
    int rows_pad;      // rows_g rounded up to a multiple of 4 (row stride of lse2)
    int c0, c1;        // candidate blocks [c0, c1)
    int Bcap;
    int n_blocks;
    float scale;       // log2(e)/sqrt(D)
    float* lse2;       // [L*Hkv][rows_pad]; pad entries hold +inf
    float* mass;       // [L*Hkv][n_blocks]
    unsigned* err;
};

struct __align__(8) SmemTail {
    float colv[kNAcc][BN];        // column pass: lse2 of the tile's query rows (bulk-copied)
    float red[kSlices][BM][2];    // merge of the column slices at unit end
    uint64_t full_a[kNA], empty_a[kNA], full_b[kNB], empty_b[kNB], acc_full[kNAcc], acc_empty[kNAcc];
    uint64_t lse_full[kNAcc], lse_empty[kNAcc];  // column pass: colv ring, one slot per accumulator
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};
constexpr size_t kSmemBytes = (size_t)kNA * kABytes + (size_t)kNB * kBBytes + sizeof(SmemTail) + 1024;

// ---- PTX wrappers ----------------------------------------------------------

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(saddr(b)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase of parity `parity`.  Returns false if this or
// another role gave up (the CTA is then draining).
__device__ __noinline__ bool wait_phase(uint64_t* b, uint32_t parity, volatile int* abort_flag, unsigned* err) {
    if (mbar_test(b, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(b, parity)) return true;
        if ((i & 63) == 0) {
            if (*abort_flag) return false;
            if (gtimer() - t0 > kWaitNs) {
                *abort_flag = 1;
                atomicOr(err, (unsigned)KVSEL_DEV_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag: used to drain this thread's own
// copies and MMAs before the CTA frees TMEM and exits.
__device__ __noinline__ void drain_phase(uint64_t* b, uint32_t parity) {
    const uint64_t t0 = gtimer();
    while (!mbar_test(b, parity) && gtimer() - t0 < kWaitNs) {
    }
}

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            saddr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(saddr(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Plain bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     saddr(dst)),
                 "l"(src), "r"(bytes), "r"(saddr(bar))
                 : "memory");
}

// 2^x on the FMA pipe, for a share of the exponentials (the MUFU computes the
// rest): x = n + f with n = rint(x) (added to 1.5*2^23 and subtracted back),
// |f| <= 1/2; 2^f = e^(f ln 2) by its Taylor series to degree 5 (truncation
// below 3.4e-6 relative); 2^n goes into the exponent field.  x is clamped at
// -125, so x = -inf gives ~2e-38 instead of 0 (far below anything summed here).
__device__ __forceinline__ float2 exp2_fma(float2 x) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    constexpr float c1 = 0.693147182464599609375f, c2 = 0.2402265071868896484375f, c3 = 0.0555041097104549407958984375f,
                    c4 = 0.009618128649890422821044921875f, c5 = 0.001333355787210166454315185546875f;
    x = make_float2(fmaxf(x.x, -125.f), fmaxf(x.y, -125.f));
    const float2 t = __fadd2_rn(x, make_float2(kMagic, kMagic));
    const float2 n = __fadd2_rn(t, make_float2(-kMagic, -kMagic));
    const float2 f = __fadd2_rn(x, make_float2(-n.x, -n.y));
    float2 p = __ffma2_rn(make_float2(c5, c5), f, make_float2(c4, c4));
    p = __ffma2_rn(p, f, make_float2(c3, c3));
    p = __ffma2_rn(p, f, make_float2(c2, c2));
    p = __ffma2_rn(p, f, make_float2(c1, c1));
    p = __ffma2_rn(p, f, make_float2(1.f, 1.f));
    const int ex = (__float_as_int(t.x) - __float_as_int(kMagic)) << 23;
    const int ey = (__float_as_int(t.y) - __float_as_int(kMagic)) << 23;
    return make_float2(__int_as_float(__float_as_int(p.x) + ex), __int_as_float(__float_as_int(p.y) + ey));
}

// Exponentials of a pair: pairs with index < kPolyPairs (of 16 per 32-column
// chunk) go to the FMA pipe, the rest to the MUFU.
#ifndef KVSEL_POLY_PAIRS
#define KVSEL_POLY_PAIRS 0
#endif
constexpr int kPolyPairs = KVSEL_POLY_PAIRS;
__device__ __forceinline__ float2 exp2_pair(float2 x, int pair) {
    if (pair < kPolyPairs) return exp2_fma(x);
    return make_float2(ex2(x.x), ex2(x.y));
}

__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4)   // start address
           | ((uint64_t)1 << 16)                // leading byte offset (unused with 128B swizzle)
           | ((uint64_t)(1024 >> 4) << 32)      // stride byte offset: 8 rows x 128 B
           | ((uint64_t)1 << 46)                // descriptor version
           | ((uint64_t)2 << 61);               // 128-byte swizzle
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accum)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%"
        "19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }
// Barrier over the epilogue threads that also ANDs a flag across them, so that
// every epilogue thread takes the same continue / give-up decision.
__device__ __forceinline__ bool epi_bar_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kEpiThreads)
        : "memory");
    return r != 0;
}

// Column-pass accumulation of one slice: s2 += 2^(v*scale - lse[col]); with MASK,
// columns >= nvalid are skipped (their lse slots may hold stale data).
template <bool MASK>
__device__ __forceinline__ void col_accumulate(const float (&v)[kSliceCols / 32][32], const float* cv, float scale,
                                               int nvalid, float2 (&s2)[4]) {
    const float2 sc = make_float2(scale, scale);
#pragma unroll
    for (int c = 0; c < kSliceCols / 32; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(cv + c * 32 + i);
            float2 x0 = __ffma2_rn(make_float2(v[c][i], v[c][i + 1]), sc, make_float2(-l4.x, -l4.y));
            float2 x1 = __ffma2_rn(make_float2(v[c][i + 2], v[c][i + 3]), sc, make_float2(-l4.z, -l4.w));
            if (MASK) {
                const int col = c * 32 + i;
                if (col >= nvalid) x0.x = -INFINITY;
                if (col + 1 >= nvalid) x0.y = -INFINITY;
                if (col + 2 >= nvalid) x1.x = -INFINITY;
                if (col + 3 >= nvalid) x1.y = -INFINITY;
            }
            s2[(i >> 2) & 3] = __fadd2_rn(s2[(i >> 2) & 3], exp2_pair(x0, i >> 1));
            s2[((i >> 2) + 2) & 3] = __fadd2_rn(s2[((i >> 2) + 2) & 3], exp2_pair(x1, (i >> 1) + 1));
        }
}

// ---- the kernel -----------------------------------------------------------

__global__ void __launch_bounds__(kThreads, 1)
    block_scores_tc(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;                                   // [kNA][kABytes]
    uint8_t* sB = smem + kNA * kABytes;                   // [kNB][kBBytes]
    SmemTail& t = *reinterpret_cast<SmemTail*>(sB + kNB * kBBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &t.abort_flag;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNA; ++i) {
            mbar_init(&t.full_a[i], 1);
            mbar_init(&t.empty_a[i], 1);
        }
        for (int i = 0; i < kNB; ++i) {
            mbar_init(&t.full_b[i], 1);
            mbar_init(&t.empty_b[i], 1);
        }
        for (int i = 0; i < kNAcc; ++i) {
            mbar_init(&t.acc_full[i], 1);
            mbar_init(&t.acc_empty[i], kEpiWarps);  // one arrival per epilogue warp
            mbar_init(&t.lse_full[i], 1);
            mbar_init(&t.lse_empty[i], kEpiWarps);
        }
        mbar_init(&t.mma_done, 1);
        t.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapB)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&t.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = t.tmem_base;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            uint32_t a_it = 0, b_it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
                const int lg = u / a.units_per_lg, ta = u % a.units_per_lg;
                int ya, yb0;
                if (a.mode == 0) {
                    ya = lg * a.rows_g + ta * BM;
                    yb0 = lg * a.Bcap + a.c0;
                } else {
                    ya = lg * a.Bcap + a.c0 + ta * BM;
                    yb0 = lg * a.rows_g;
                }
                const int sa = a_it % kNA;
                if (!(ok = wait_phase(&t.empty_a[sa], ((a_it / kNA) & 1) ^ 1, abort_flag, a.err))) break;
                mbar_expect_tx(&t.full_a[sa], kABytes);
                tma_load_2d(&mapA, &t.full_a[sa], sA + sa * kABytes, 0, ya);
                tma_load_2d(&mapA, &t.full_a[sa], sA + sa * kABytes + kABytes / 2, 64, ya);
                ++a_it;
                for (int tb = 0; tb < a.n_bt; ++tb) {
                    const int sb = b_it % kNB;
                    if (!(ok = wait_phase(&t.empty_b[sb], ((b_it / kNB) & 1) ^ 1, abort_flag, a.err))) break;
                    mbar_expect_tx(&t.full_b[sb], kBBytes);
                    tma_load_2d(&mapB, &t.full_b[sb], sB + sb * kBBytes, 0, yb0 + tb * BN);
                    tma_load_2d(&mapB, &t.full_b[sb], sB + sb * kBBytes + kBBytes / 2, 64, yb0 + tb * BN);
                    if (a.mode == 1) {
                        // the log-sum-exps of this tile's query rows, one slot per accumulator
                        const int k = b_it % kNAcc;
                        if (!(ok = wait_phase(&t.lse_empty[k], ((b_it / kNAcc) & 1) ^ 1, abort_flag, a.err))) break;
                        const int r0 = tb * BN;
                        const uint32_t bytes = 4u * (uint32_t)min(BN, a.rows_pad - r0);
                        mbar_expect_tx(&t.lse_full[k], bytes);
                        bulk_copy(&t.colv[k][0], a.lse2 + (int64_t)lg * a.rows_pad + r0, bytes, &t.lse_full[k]);
                    }
                    ++b_it;
                }
            }
            // drain: wait until every copy this thread started has landed
            for (uint32_t i = (b_it > (uint32_t)kNB ? b_it - kNB : 0); i < b_it; ++i)
                drain_phase(&t.full_b[i % kNB], (i / kNB) & 1);
            for (uint32_t i = (a_it > (uint32_t)kNA ? a_it - kNA : 0); i < a_it; ++i)
                drain_phase(&t.full_a[i % kNA], (i / kNA) & 1);
            if (a.mode == 1)
                for (uint32_t i = (b_it > (uint32_t)kNAcc ? b_it - kNAcc : 0); i < b_it; ++i)
                    drain_phase(&t.lse_full[i % kNAcc], (i / kNAcc) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            uint32_t a_it = 0, b_it = 0, acc_it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
                const int sa = a_it % kNA;
                if (!(ok = wait_phase(&t.full_a[sa], (a_it / kNA) & 1, abort_flag, a.err))) break;
                tc_fence_after();
                const uint32_t a_base = saddr(sA + sa * kABytes);
                for (int tb = 0; tb < a.n_bt; ++tb) {
                    const int sb = b_it % kNB;
                    const int k = acc_it % kNAcc;
                    if (!(ok = wait_phase(&t.full_b[sb], (b_it / kNB) & 1, abort_flag, a.err))) break;
                    if (!(ok = wait_phase(&t.acc_empty[k], ((acc_it / kNAcc) & 1) ^ 1, abort_flag, a.err))) break;
                    tc_fence_after();
                    const uint32_t b_base = saddr(sB + sb * kBBytes);
                    const uint32_t d_tmem = tmem_base + (uint32_t)(k * BN);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint32_t off = (uint32_t)((kk & 3) * 32);
                        const uint64_t ad = sw128_desc(a_base + (kk >> 2) * (kABytes / 2) + off);
                        const uint64_t bd = sw128_desc(b_base + (kk >> 2) * (kBBytes / 2) + off);
                        umma_bf16(d_tmem, ad, bd, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&t.empty_b[sb]);
                    umma_commit(&t.acc_full[k]);
                    ++b_it;
                    ++acc_it;
                }
                if (ok) umma_commit(&t.empty_a[sa]);
                ++a_it;
            }
            // drain: every MMA issued by this thread completes before TMEM is freed
            umma_commit(&t.mma_done);
            drain_phase(&t.mma_done, 0);
        }
    } else {
        // ------------------------------ epilogue ------------------------------
        const int ew = warp - 2;                 // 0 .. kEpiWarps-1
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int slice = ew >> 2;               // column slice
        const int r_local = q * 32 + lane;       // TMEM lane = A row of the unit
        const int etid = ew * 32 + lane;
        uint32_t acc_it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
            const int lg = u / a.units_per_lg, ta = u % a.units_per_lg;
            float m_run = -INFINITY;
            float2 s2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                            make_float2(0.f, 0.f)};
            for (int tb = 0; tb < a.n_bt; ++tb) {
                const int k = acc_it % kNAcc;
                // a timed-out wait makes this thread skip its work; the epilogue warps
                // agree on giving up at the end of the unit
                if (ok) ok = wait_phase(&t.acc_full[k], (acc_it / kNAcc) & 1, abort_flag, a.err);
                if (ok && a.mode == 1) ok = wait_phase(&t.lse_full[k], (acc_it / kNAcc) & 1, abort_flag, a.err);
                ok = __all_sync(0xffffffffu, ok);  // warp-uniform: TMEM loads are warp-collective
                if (!ok) {
                    ++acc_it;
                    continue;
                }
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(k * BN + slice * kSliceCols);
                float v[kSliceCols / 32][32];
#pragma unroll
                for (int c = 0; c < kSliceCols / 32; ++c) tmem_ld32(taddr + 32 * c, v[c]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&t.acc_empty[k]);  // this warp's part of the accumulator is read
                if (a.mode == 0) {
                    // row pass: online (max, sum 2^x) over this slice's columns
                    const int col0 = a.c0 + tb * BN + slice * kSliceCols;  // block id of the slice's column 0
                    const int nvalid = a.c1 - col0;                        // columns >= nvalid are masked
                    if (nvalid < kSliceCols) {
#pragma unroll
                        for (int c = 0; c < kSliceCols / 32; ++c)
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (c * 32 + i >= nvalid) v[c][i] = -INFINITY;
                    }
                    float mx = -INFINITY;
#pragma unroll
                    for (int c = 0; c < kSliceCols / 32; ++c)
#pragma unroll
                        for (int i = 0; i < 32; i += 2) mx = max3(mx, v[c][i], v[c][i + 1]);
                    const float m_new = fmaxf(m_run, mx * a.scale);
                    if (m_new != -INFINITY) {
                        if (m_new > m_run) {
                            const float f = ex2(m_run - m_new);
#pragma unroll
                            for (int j = 0; j < 4; ++j) s2[j] = make_float2(s2[j].x * f, s2[j].y * f);
                            m_run = m_new;
                        }
                        const float2 sc = make_float2(a.scale, a.scale), nm = make_float2(-m_run, -m_run);
#pragma unroll
                        for (int c = 0; c < kSliceCols / 32; ++c)
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                const float2 x = __ffma2_rn(make_float2(v[c][i], v[c][i + 1]), sc, nm);
                                s2[(i >> 1) & 3] = __fadd2_rn(s2[(i >> 1) & 3], exp2_pair(x, i >> 1));
                            }
                    }
                } else {
                    // column pass: sum over this slice's query rows of 2^(x - lse2[row]);
                    // rows past the group (last tile only) contribute nothing
                    const int nvalid = a.rows_g - (tb * BN + slice * kSliceCols);
                    const float* cv = &t.colv[k][slice * kSliceCols];
                    if (nvalid >= kSliceCols)
                        col_accumulate<false>(v, cv, a.scale, nvalid, s2);
                    else
                        col_accumulate<true>(v, cv, a.scale, nvalid, s2);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&t.lse_empty[k]);  // colv slot k may be refilled
                }
                ++acc_it;
            }
            if (!(ok = epi_bar_and(ok))) break;
            // merge the column slices of each lane, in slice order
            const float s_part = (s2[0].x + s2[0].y) + (s2[1].x + s2[1].y) + (s2[2].x + s2[2].y) + (s2[3].x + s2[3].y);
            t.red[slice][r_local][0] = m_run;
            t.red[slice][r_local][1] = s_part;
            epi_bar();
            if (slice == 0) {
                if (a.mode == 0) {
                    const int row = ta * BM + r_local;
                    if (row >= a.rows_g && row < a.rows_pad) a.lse2[(int64_t)lg * a.rows_pad + row] = INFINITY;
                    if (row < a.rows_g) {
                        float m = -INFINITY;
#pragma unroll
                        for (int j = 0; j < kSlices; ++j) m = fmaxf(m, t.red[j][r_local][0]);
                        float sum = 0.f;
                        if (m != -INFINITY) {
#pragma unroll
                            for (int j = 0; j < kSlices; ++j) sum += t.red[j][r_local][1] * ex2(t.red[j][r_local][0] - m);
                        }
                        a.lse2[(int64_t)lg * a.rows_pad + row] = sum > 0.f ? m + __log2f(sum) : -INFINITY;
                    }
                } else {
                    const int b = a.c0 + ta * BM + r_local;
                    if (b < a.c1) {
                        float sum = 0.f;
#pragma unroll
                        for (int j = 0; j < kSlices; ++j) sum += t.red[j][r_local][1];
                        a.mass[(int64_t)lg * a.n_blocks + b] = sum;
                    }
                }
            }
            epi_bar();
        }
    }

    // all roles: TMEM is released once every MMA has completed (MMA lane drained above)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

// R[b] = sum_lg mass[lg][b] / (L*Hq) on C; zero outside C (also in mass).
__global__ void bs_finalize(const float* __restrict__ mass_in, float* mass, float* R, int LH, int n_blocks, int c0,
                            int c1, float inv) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= n_blocks) return;
    if (b < c0 || b >= c1) {
        R[b] = 0.f;
        for (int lg = 0; lg < LH; ++lg) mass[(int64_t)lg * n_blocks + b] = 0.f;
        return;
    }
    float acc = 0.f;
    for (int lg = 0; lg < LH; ++lg) acc += mass_in[(int64_t)lg * n_blocks + b];
    R[b] = acc * inv;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 [rows][128] view, box {64 columns, box_rows}, 128-byte swizzle, zero fill.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
    auto fn = encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t block_scores_workspace(int L, int Hq, int Hkv, int M, int n_blocks) {
    const size_t rows_pad = (((size_t)(Hq / Hkv) * M + 3) & ~(size_t)3);
    return align256((size_t)L * Hkv * rows_pad * sizeof(float)) + align256((size_t)L * Hkv * n_blocks * sizeof(float));
}

cudaError_t launch_block_scores(kvsel_ctx* ctx, const void* q, const void* index, int L, int Hq, int Hkv, int M, int D,
                                int n_blocks, int Bcap, int n_sink, int n_recent, float* R, float* R_partial, void* ws,
                                cudaStream_t s) {
    (void)D;
    const int G = Hq / Hkv;
    const int rows_g = G * M;
    const int c0 = n_sink < n_blocks ? n_sink : n_blocks;
    const int c1 = n_blocks - n_recent > c0 ? n_blocks - n_recent : c0;
    const int ncand = c1 - c0;
    const int LH = L * Hkv;
    char* w = static_cast<char*>(ws);
    float* lse2 = reinterpret_cast<float*>(w);
    const int rows_pad = (rows_g + 3) & ~3;
    w += align256((size_t)LH * rows_pad * sizeof(float));
    float* mass = R_partial ? R_partial : reinterpret_cast<float*>(w);

    if (ncand > 0) {
        CUtensorMap qA, qB, iA, iB;
        const uint64_t q_rows = (uint64_t)L * Hq * M, i_rows = (uint64_t)LH * Bcap;
        if (!make_map(&qA, q, q_rows, BM) || !make_map(&qB, q, q_rows, BN) || !make_map(&iA, index, i_rows, BM) ||
            !make_map(&iB, index, i_rows, BN))
            return cudaErrorInvalidValue;
        cudaError_t e = cudaFuncSetAttribute(block_scores_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        TcArgs a;
        a.rows_g = rows_g;
        a.rows_pad = rows_pad;
        a.c0 = c0;
        a.c1 = c1;
        a.Bcap = Bcap;
        a.n_blocks = n_blocks;
        a.scale = kLog2e / sqrtf((float)kD);
        a.lse2 = lse2;
        a.mass = mass;
        a.err = ctx->dev_err;
        // row pass
        a.mode = 0;
        a.units_per_lg = (rows_g + BM - 1) / BM;
        a.n_units = LH * a.units_per_lg;
        a.n_bt = (ncand + BN - 1) / BN;
        int grid = a.n_units < ctx->num_sms ? a.n_units : ctx->num_sms;
        block_scores_tc<<<grid, kThreads, kSmemBytes, s>>>(qA, iB, a);
        // column pass
        a.mode = 1;
        a.units_per_lg = (ncand + BM - 1) / BM;
        a.n_units = LH * a.units_per_lg;
        a.n_bt = (rows_g + BN - 1) / BN;
        grid = a.n_units < ctx->num_sms ? a.n_units : ctx->num_sms;
        block_scores_tc<<<grid, kThreads, kSmemBytes, s>>>(iA, qB, a);
    }
    bs_finalize<<<(n_blocks + 255) / 256, 256, 0, s>>>(mass, mass, R, LH, n_blocks, c0, c1,
                                                       1.0f / ((float)L * (float)Hq));
    return cudaGetLastError();
}

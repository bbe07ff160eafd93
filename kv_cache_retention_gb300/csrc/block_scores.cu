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
// on the tensor cores.  A unit holds a fixed operand of 256 rows (B, the
// accumulator columns) and streams the other operand 128 rows a tile (A, the
// TMEM lanes):
//   row pass:    a unit is (l,g, 256 query rows); tiles of 128 candidate blocks
//                stream.  A warp reads its 32 blocks x 64 query rows as two
//                16x256b loads, so a thread holds 4 blocks x 16 rows, and adds
//                2^(x - ref) into 16 per-row sums.  ref: one per warp, the
//                largest logit over the warp's 32 blocks x 64 rows of the unit's
//                first tile plus 16 (log2) of headroom.  At the end of the unit
//                the sums are added across the warp's lanes (butterfly) and
//                merged across the four lane quarters with their references
//                -> lse2[r] = log2 sum_{b in C} 2^(S[r,b] log2e/sqrt(d)), stored
//                negated, the row range padded to whole column-pass tiles with
//                -inf.  A row whose merged sum is below 2^-90 of its reference (its
//                largest logit lies more than 74 below the warp's) may have lost
//                terms to underflow; a sum that is not finite overflowed (a
//                logit more than about 134 above the reference's).  Either marks
//                the unit for
//   exact pass:  the row pass again on the marked units only (every other unit
//                is skipped by all roles), with one reference per (warp, row):
//                the row's largest logit over the warp's blocks of the first
//                tile plus 64, moved up by 64 when a sum passes 2^100.  It
//                overwrites the unit's lse2.
//   column pass: a unit is (l,g, 256 candidate blocks); tiles of 128 query rows
//                stream.  A thread holds 4 rows x 16 blocks; it adds
//                2^(x - lse2[r]) into 16 per-block sums.  -lse2 is loaded one
//                tile ahead, one lane per row, handed on by shuffles and used as
//                the fma's addend as it is (no bounds test: the padding reads
//                -inf).  At the end of the unit the sums are added across lanes
//                (butterfly) and across the four lane quarters -> mass[lg][b],
//                complete per CTA
//   finalize:    R[b] = sum_lg mass[lg][b] / (L*Hq), in fixed (l,g) order.
// Every pass completes each unit's results inside one CTA: no atomics, no
// partial results in global memory.
//
// Kernel structure (one persistent CTA per SM, 640 threads = 5 warpgroups):
//   warp 0      TMA producer: the unit's fixed tile (64 KB), then the streamed
//               tiles through a ring of 4 x 32 KB (128-byte swizzled, K-major,
//               no multicast)
//   warps 1, 2  allocate 512 TMEM columns (warp 1); lane 0 of each issues
//               tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, M=128 N=256 K=16,
//               8 per tile) for alternate tiles, each into its own 256-column
//               accumulator, and commits to mbarriers that free the smem stage
//               and hand the accumulator on
//   warp 3      idle (completes the first warpgroup)
//   warps 4-19  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31; four column slices of 64), release, a
//               non-blocking probe of the next tile's accumulator, exp2 on the
//               MUFU, packed fp32 arithmetic
// The first warpgroup gives registers back (setmaxnreg.dec to kRegsCtl) and the
// four epilogue warpgroups take them (setmaxnreg.inc to kRegsEpi): the launch
// allows 96 per thread, the epilogue's 64 accumulator values, 16 sums and
// addressing need more.
// Every mbarrier wait is bounded (1 s of globaltimer); on a timeout the CTA
// flags KVSEL_ERR_TIMEOUT in the device error word, drains its own copies and
// MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <type_traits>

#include "kvsel_internal.h"

namespace {

constexpr float kScale = (float)(1.4426950408889634 / 11.313708498984761);  // log2(e)/sqrt(128), logits to base 2
constexpr int kD = 128;
constexpr int BM = 128;                         // TMEM lanes = streamed rows per MMA
constexpr int kRowBytes = kD * 2;               // one bf16 row of 128 dims

constexpr int kNAcc = 2;                        // accumulator buffers

// Operand tiling of both passes: the fixed operand (B, 256 rows, the
// accumulator columns) is loaded once per unit, the streamed one (A, 128 rows,
// the TMEM lanes) once per tile through a ring of kNS stages.
//   row pass:    fixed = 256 query rows, streamed = 128 candidate blocks
//   column pass: fixed = 256 candidate blocks, streamed = 128 query rows
struct Tiling {
    static constexpr int kFRows = 256, kSRows = 128;
    static constexpr int kNF = 1, kNS = 4;
    static constexpr int kFBytes = kFRows * kRowBytes, kSBytes = kSRows * kRowBytes;
    static constexpr int kStageBytes = kNF * kFBytes + kNS * kSBytes;
    static_assert(kStageBytes == 192 * 1024, "operand buffers");
    static_assert(kNS >= kNAcc, "a stage ring at least as deep as the accumulator ring");
    // tile j is issued by MMA thread j % 2 and uses stage j % kNS: with kNS even every stage
    // belongs to one issuer, which then sees each of its barrier's phases in order (an issuer
    // skipping the other's phases could mistake an older phase for its own)
    static_assert(kNS % 2 == 0, "an even stage ring for the two MMA issuers");
};
constexpr int kMaxStages = 4;
// A tile's MMAs wait on one barrier of their operand stage, completed by the
// stage's copies and by the epilogue's release of the accumulator they
// overwrite (tile j's accumulator was last used by tile j - kNAcc).  That
// needs kNS >= kNAcc, so that a release never lands on a stage barrier whose
// previous phase is still open.
constexpr int kAccCols = 256;                   // TMEM columns per accumulator buffer
constexpr int kTmemCols = kNAcc * kAccCols;
constexpr int kEpiWarps = 16;                   // 4 TMEM lane quarters x kSlices column slices
constexpr int kSlices = kEpiWarps / 4;
constexpr int kSliceCols = kAccCols / kSlices;  // accumulator columns per epilogue thread and tile
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kIssuer2 = 2;                     // the second MMA-issuing warp
constexpr int kEpi0 = 4;                        // first epilogue warp (warps 0-3: one warpgroup)
static_assert(kNAcc == 2, "the two MMA issuers own one accumulator each");
static_assert(kEpiWarps == 16 && kEpi0 == 4, "one first warpgroup and four epilogue warpgroups");
constexpr int kThreads = 128 + kEpiThreads;
// Registers per thread after the first warpgroup's setmaxnreg.dec / the epilogue's .inc.
// Each SM sub-partition holds one first-group warp and four epilogue warps, so the
// split fits the launch's registers iff kRegsCtl + 4 * kRegsEpi <= 5 * (registers at
// launch); an .inc beyond that would wait forever.  Here it fits exactly
// (64 + 4 * 104 = 5 * 96), and the launcher checks the compiled kernel's count
// before any launch.
constexpr int kRegsCtl = 64, kRegsEpi = 104;
constexpr int kRegsLaunch = 96;  // registers per thread the launch of 640 threads allows
static_assert(kRegsCtl + 4 * kRegsEpi <= 5 * kRegsLaunch && kRegsLaunch * kThreads <= 65536, "register split");
static_assert(kRegsCtl % 8 == 0 && kRegsEpi % 8 == 0 && kRegsCtl >= 24 && kRegsEpi <= 256, "setmaxnreg values");
constexpr uint64_t kWaitNs = 1000000000ull;     // 1 s per wait
#ifndef KVSEL_SUSPEND_NS
#define KVSEL_SUSPEND_NS 20000
#endif
constexpr uint32_t kSuspendNs = KVSEL_SUSPEND_NS;  // try_wait may park the thread this long (woken on completion)

// instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M=128
__host__ __device__ constexpr uint32_t idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

struct TcArgs {
    int n_units;
    int units_per_lg;
    int n_it;          // streamed tiles per unit
    int rows_g;        // G*M
    int rows_pad;      // rows_g rounded up to a multiple of 128 (row stride of nlse2)
    int c0, c1;        // candidate blocks [c0, c1)
    int Bcap;
    int n_blocks;
    float* nlse2;      // [L*Hkv][rows_pad]: -lse2 of each query row; pad entries hold -inf
    float* mass;       // [L*Hkv][n_blocks]
    unsigned* err;
    int* redo;         // [row-pass units]: set by the row pass where the exact pass must redo the unit
    uint64_t wait_ns;  // give-up limit of a bounded wait
    int stuck;         // test hook: the row pass's first MMA issuer waits on a barrier nothing completes
};

// MODE 0: row pass, one reference per warp; MODE 2: the exact row pass over the
// units the row pass marked, one reference per (warp, row); MODE 1: column pass.
template <int MODE>
constexpr bool kRowPass = MODE != 1;

template <int MODE>
struct __align__(8) SmemTail {
    uint64_t full_f[2], empty_f[2], go[kMaxStages], empty_s[kMaxStages], acc_full[kNAcc];
    uint64_t mma_done;
    uint64_t never;    // no thread arrives on it (the give-up test hook waits here)
    uint32_t tmem_base;
    int abort_flag;
    // unit end: [slice][lane quarter][column] (reference, sum) pairs (row passes) or sums (column pass)
    float red[(kRowPass<MODE> ? 2 : 1) * kSlices * 4 * kSliceCols];
    // exact row pass: each epilogue warp's negated references of its 64 query rows
    float nref[MODE == 2 ? kEpiWarps * kSliceCols : 1];
};
// operand buffers + barriers + room to align the buffers to 1024 bytes
template <int MODE>
constexpr size_t smem_bytes() { return (size_t)Tiling::kStageBytes + sizeof(SmemTail<MODE>) + 1024; }
static_assert(smem_bytes<0>() <= 232448 && smem_bytes<1>() <= 232448 && smem_bytes<2>() <= 232448,
              "shared memory per CTA");

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
// Arrive from lane 0 of the warp only, as a predicated instruction (no branch).
__device__ __forceinline__ void mbar_arrive_lane0(uint64_t* b, int lane) {
    asm volatile("{\n .reg .pred p;\n setp.eq.s32 p, %1, 0;\n @p mbarrier.arrive.shared::cta.b64 _, [%0];\n}\n" ::"r"(
                     saddr(b)),
                 "r"(lane)
                 : "memory");
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
// Non-blocking: has the phase of parity `parity` completed?
__device__ __forceinline__ bool mbar_done(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(saddr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase of parity `parity`, giving up after limit_ns.
// Returns false if this or another role gave up (the CTA is then draining).
// Everything is inlined: a called function would be compiled for one register
// budget, and the kernel's warpgroups run under two (setmaxnreg).
__device__ __forceinline__ bool wait_phase_retry(uint64_t* b, uint32_t parity, volatile int* abort_flag, unsigned* err,
                                             uint64_t limit_ns) {
    const uint64_t t0 = gtimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(b, parity)) return true;
        if ((i & 63) == 0) {
            if (*abort_flag) return false;
            if (gtimer() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(err, (unsigned)KVSEL_DEV_TIMEOUT);
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool wait_phase(uint64_t* b, uint32_t parity, volatile int* abort_flag, unsigned* err,
                                           uint64_t limit_ns) {
    return mbar_test(b, parity) || wait_phase_retry(b, parity, abort_flag, err, limit_ns);
}

// Bounded wait that ignores the abort flag: used to drain this thread's own
// copies and MMAs before the CTA frees TMEM and exits.
__device__ __forceinline__ void drain_phase(uint64_t* b, uint32_t parity) {
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

__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4)   // start address
           | ((uint64_t)1 << 16)                // leading byte offset (unused with 128B swizzle)
           | ((uint64_t)(1024 >> 4) << 32)      // stride byte offset: 8 rows x 128 B
           | ((uint64_t)1 << 46)                // descriptor version
           | ((uint64_t)2 << 61);               // 128-byte swizzle
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc_v,
                                          uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc_v), "r"(accum)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 TMEM lanes x 8 repetitions of 256 bits.  Thread t receives, for repetition j,
// v[4j], v[4j+1] from lane t/4 and v[4j+2], v[4j+3] from lane t/4 + 8, both at
// columns 8j + 2(t%4) and 8j + 2(t%4) + 1.
__device__ __forceinline__ void tmem_ld16x256_8(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%"
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

// Barrier over the epilogue threads that ORs a flag across them.
__device__ __forceinline__ bool epi_bar_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kEpiThreads)
        : "memory");
    return r != 0;
}

// ---- epilogue helpers -----------------------------------------------------

// Column pass: adds 2^(v*scale - lse2) of one TMEM lane of a 16x256b load
// (e = 0: lane t/4, e = 1: lane t/4 + 8) into the thread's 8 packed column sums.
__device__ __forceinline__ void col_terms(const float (&v)[32], int e, float2 sc, float nlse, float2 (&cs)[8]) {
    const float2 nl = make_float2(nlse, nlse);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float2 x = __ffma2_rn(make_float2(v[4 * j + 2 * e], v[4 * j + 2 * e + 1]), sc, nl);
        cs[j] = __fadd2_rn(cs[j], make_float2(ex2(x.x), ex2(x.y)));
    }
}

// Row pass: adds 2^(v*scale - ref) of column pair j over the
// thread's four TMEM lanes (two 16x256b loads, each lanes t/4 and t/4 + 8) into
// that pair's packed sum; nr: the pair's negated references.
__device__ __forceinline__ void col_pair_terms(const float (&v0)[32], const float (&v1)[32], int j, float2 sc,
                                               float2 nr, float2& sum) {
    const float2 x0 = __ffma2_rn(make_float2(v0[4 * j], v0[4 * j + 1]), sc, nr);
    const float2 x1 = __ffma2_rn(make_float2(v0[4 * j + 2], v0[4 * j + 3]), sc, nr);
    const float2 x2 = __ffma2_rn(make_float2(v1[4 * j], v1[4 * j + 1]), sc, nr);
    const float2 x3 = __ffma2_rn(make_float2(v1[4 * j + 2], v1[4 * j + 3]), sc, nr);
    sum = __fadd2_rn(sum, make_float2(ex2(x0.x), ex2(x0.y)));
    sum = __fadd2_rn(sum, make_float2(ex2(x1.x), ex2(x1.y)));
    sum = __fadd2_rn(sum, make_float2(ex2(x2.x), ex2(x2.y)));
    sum = __fadd2_rn(sum, make_float2(ex2(x3.x), ex2(x3.y)));
}

// Largest of column pair j's values over the thread's four TMEM lanes (two loads).
__device__ __forceinline__ float2 col_max(const float (&v0)[32], const float (&v1)[32], int j) {
    return make_float2(fmaxf(max3(v0[4 * j], v0[4 * j + 2], v1[4 * j]), v1[4 * j + 2]),
                       fmaxf(max3(v0[4 * j + 1], v0[4 * j + 3], v1[4 * j + 1]), v1[4 * j + 3]));
}

// Merge of two (reference, sum) pairs of base-2 exponentials.
__device__ __forceinline__ float2 lse2_merge(float2 a, float2 b) {
    const float m = fmaxf(a.x, b.x);
    if (m == -INFINITY) return make_float2(-INFINITY, 0.f);
    return make_float2(m, a.y * ex2(a.x - m) + b.y * ex2(b.x - m));
}

// Column sums of a warp after the column pass: on entry lane t holds, for
// j = 0..7, the sums of columns 8j + 2(t%4) and 8j + 2(t%4) + 1 over its rows;
// the eight lanes with the same t%4 hold the same columns.  Three butterfly
// levels over lane bits 4, 3, 2, each keeping half of the values and sending
// the other half to the partner; on exit f[0], f[1] hold the sums over the
// warp's 32 rows of columns 2t and 2t + 1.
__device__ __forceinline__ void column_reduce(float (&f)[16], int lane) {
#pragma unroll
    for (int s = 16, n = 8; s >= 4; s >>= 1, n >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float keep = up ? f[n + i] : f[i];
            const float send = up ? f[i] : f[n + i];
            f[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
}

// ---- the kernel -----------------------------------------------------------

// MODE 0 / 2: row pass / exact row pass, MODE 1: column pass (operand roles in
// Tiling).  Either way one tile is one 128 x 256 accumulator: TMEM lanes = the
// streamed rows, columns = the unit's fixed rows.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    block_scores_tc(const __grid_constant__ CUtensorMap mapF, const __grid_constant__ CUtensorMap mapS, const TcArgs a) {
    using T = Tiling;
    if constexpr (MODE == 2) {
        // The row pass marks no unit on ordinary inputs: a CTA none of whose units is
        // marked leaves before it sets anything up (one parallel read of the marks).
        bool any = false;
        for (int u = blockIdx.x + threadIdx.x * gridDim.x; u < a.n_units; u += blockDim.x * gridDim.x)
            any |= a.redo[u] != 0;
        if (!__syncthreads_or(any)) return;
    }
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sF = smem;                                   // [kNF][kFBytes]
    uint8_t* sS = smem + T::kNF * T::kFBytes;             // [kNS][kSBytes]
    SmemTail<MODE>& t = *reinterpret_cast<SmemTail<MODE>*>(smem + T::kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &t.abort_flag;

    if (threadIdx.x == 0) {
        for (int i = 0; i < T::kNF; ++i) {
            mbar_init(&t.full_f[i], 1);
            mbar_init(&t.empty_f[i], 2);  // both MMA issuers are done with the unit
        }
        for (int i = 0; i < T::kNS; ++i) {
            mbar_init(&t.go[i], 1 + kEpiWarps);  // the stage's copies + the accumulator's release
            mbar_init(&t.empty_s[i], 1);
        }
        for (int i = 0; i < kNAcc; ++i) mbar_init(&t.acc_full[i], 1);
        mbar_init(&t.mma_done, 2);
        mbar_init(&t.never, 1);
        t.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapF)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapS)) : "memory");
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

    // The two register budgets: each branch below runs to the kernel's end on its own
    // (no code is shared after a setmaxnreg).
    if (warp < kEpi0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            uint32_t f_it = 0, s_it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
                if (MODE == 2 && !a.redo[u]) continue;  // every role skips the same units
                const int lg = u / a.units_per_lg, o = u % a.units_per_lg;
                const int fs = f_it % T::kNF;
                const int yf = MODE == 1 ? lg * a.Bcap + a.c0 + o * T::kFRows : lg * a.rows_g + o * T::kFRows;
                if (!(ok = wait_phase(&t.empty_f[fs], ((f_it / T::kNF) & 1) ^ 1, abort_flag, a.err, a.wait_ns))) break;
                mbar_expect_tx(&t.full_f[fs], T::kFBytes);
                tma_load_2d(&mapF, &t.full_f[fs], sF + fs * T::kFBytes, 0, yf);
                tma_load_2d(&mapF, &t.full_f[fs], sF + fs * T::kFBytes + T::kFBytes / 2, 64, yf);
                ++f_it;
                for (int i = 0; i < a.n_it; ++i) {
                    const int st = s_it % T::kNS;
                    const int ys = MODE == 1 ? lg * a.rows_g + i * T::kSRows : lg * a.Bcap + a.c0 + i * T::kSRows;
                    if (!(ok = wait_phase(&t.empty_s[st], ((s_it / T::kNS) & 1) ^ 1, abort_flag, a.err, a.wait_ns))) break;
                    mbar_expect_tx(&t.go[st], T::kSBytes);
                    tma_load_2d(&mapS, &t.go[st], sS + st * T::kSBytes, 0, ys);
                    tma_load_2d(&mapS, &t.go[st], sS + st * T::kSBytes + T::kSBytes / 2, 64, ys);
                    ++s_it;
                }
            }
            // drain: wait until every copy this thread started has landed
            for (uint32_t i = (s_it > (uint32_t)T::kNS ? s_it - T::kNS : 0); i < s_it; ++i)
                drain_phase(&t.go[i % T::kNS], (i / T::kNS) & 1);
            for (uint32_t i = (f_it > (uint32_t)T::kNF ? f_it - T::kNF : 0); i < f_it; ++i)
                drain_phase(&t.full_f[i % T::kNF], (i / T::kNF) & 1);
        }
    } else if (warp == 1 || warp == kIssuer2) {
        // ------------------------------ MMA issuers ------------------------------
        // Two threads on two SM sub-partitions issue alternate tiles (tile j uses
        // accumulator j % 2, so each issuer owns one).  One thread alone spent about
        // as long per tile as the MMAs take: its barrier and tcgen05 instructions
        // queue behind the epilogue's exp2 instructions on its sub-partition.
        if (lane == 0) {
            const uint32_t me = warp == 1 ? 0u : 1u;
            uint32_t f_it = 0, s_it = 0, acc_it = 0;
            bool ok = true;
            // test hook: a wait that can only give up, taken while the producer's
            // copies and the other issuer's MMAs are in flight
            if (MODE == 0 && a.stuck && me == 0) ok = wait_phase(&t.never, 0, abort_flag, a.err, a.wait_ns);
            for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
                if (MODE == 2 && !a.redo[u]) continue;
                const int fs = f_it % T::kNF;
                if (!(ok = wait_phase(&t.full_f[fs], (f_it / T::kNF) & 1, abort_flag, a.err, a.wait_ns))) break;
                tc_fence_after();
                const uint32_t f_base = saddr(sF + fs * T::kFBytes);
                for (int i = 0; i < a.n_it; ++i) {
                    const int st = s_it % T::kNS;
                    const int k = acc_it % kNAcc;
                    if ((acc_it & 1u) != me) {  // the other issuer's tile
                        ++s_it;
                        ++acc_it;
                        continue;
                    }
                    // one wait per tile: the stage's operand has landed and the epilogue has
                    // read the accumulator this tile overwrites
                    if (!(ok = wait_phase(&t.go[st], (s_it / T::kNS) & 1, abort_flag, a.err, a.wait_ns))) break;
                    tc_fence_after();
                    const uint32_t s_base = saddr(sS + st * T::kSBytes);
                    // A = the streamed 128-row operand, B = the unit's fixed 256 rows
                    const uint32_t a_base = s_base, b_base = f_base;
                    const uint32_t d_tmem = tmem_base + (uint32_t)(k * kAccCols);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint32_t off = (uint32_t)((kk & 3) * 32);
                        const uint64_t ad = sw128_desc(a_base + (kk >> 2) * (BM * 128) + off);
                        const uint64_t bd = sw128_desc(b_base + (kk >> 2) * (kAccCols * 128) + off);
                        umma_bf16(d_tmem, ad, bd, idesc(kAccCols), kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&t.empty_s[st]);
                    umma_commit(&t.acc_full[k]);
                    ++s_it;
                    ++acc_it;
                }
                if (ok) umma_commit(&t.empty_f[fs]);
                ++f_it;
            }
            // drain: every MMA issued by this thread completes before TMEM is freed
            umma_commit(&t.mma_done);
            drain_phase(&t.mma_done, 0);
        }
    }
    // first warpgroup's end: TMEM is released once every MMA has completed (the MMA
    // lanes drained above) and the epilogue has passed the same barrier
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
    return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    {
        // ------------------------------ epilogue ------------------------------
        const int ew = warp - kEpi0;             // 0 .. kEpiWarps-1
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int slice = ew >> 2;               // column slice
        const int r_local = q * 32 + lane;       // this lane's TMEM lane (column pass: a query row of the tile)
        const int etid = ew * 32 + lane;
        const float2 sc = make_float2(kScale, kScale);
        // the first kNAcc tiles find their accumulators free
        if (lane == 0)
            for (int j = 0; j < kNAcc; ++j) mbar_arrive(&t.go[j % T::kNS]);
        uint32_t acc_it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < a.n_units && ok; u += gridDim.x) {
            if (MODE == 2 && !a.redo[u]) continue;
            const int lg = u / a.units_per_lg, o = u % a.units_per_lg;
            const float* nlse_lg = a.nlse2 + (int64_t)lg * a.rows_pad;
            // the thread's 16 sums (row pass: per query row, column pass: per block)
            float2 cs[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) cs[j] = make_float2(0.f, 0.f);
            // column pass: -lse2 of this lane's row in the next tile (loaded ahead; every
            // tile's rows lie inside the padded row range)
            float nl_n = 0.f;
            if (MODE == 1) nl_n = __ldg(nlse_lg + r_local);
            // exact row pass: the warp's negated references of its 64 query rows, in
            // shared memory (set by the unit's first tile)
            float* const wref = t.nref + (MODE == 2 ? ew * kSliceCols : 0);
            // row pass: the warp's one negated reference (set by the unit's first tile)
            float wnr = 0.f;
            bool ready = false;  // this tile's accumulator was seen complete by the probe below
            const uint32_t taddr_q = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(slice * kSliceCols);
            // One tile, accumulator K = the tile's position in the accumulator ring; MASK:
            // the row pass's last tile, whose TMEM lanes past the candidate range are masked.
            auto tile = [&](auto kc, auto maskc, auto posc, int i) {
                constexpr int K = decltype(kc)::value;
                [[maybe_unused]] constexpr bool MASK = decltype(maskc)::value;
                // POS: acc_it % 4 when the caller knows it (barrier indices and parities are
                // then constants), else -1
                constexpr int POS = decltype(posc)::value;
                // After a timed-out wait a thread waits no more: its warp still runs the
                // remaining tiles' TMEM loads (always in range, and warp-collective) and
                // math on whatever the accumulator holds, and the epilogue warps agree on
                // giving up at the end of the unit.  No per-tile vote or branch: in the
                // column pass that alone cost a tenth of the tensor pipe's time.
                const uint32_t par = POS >= 0 ? (uint32_t)((POS >> 1) & 1) : (acc_it >> 1) & 1u;
                if (ok && !ready) ok = wait_phase(&t.acc_full[K], par, abort_flag, a.err, a.wait_ns);
                tc_fence_after();
                const uint32_t taddr = taddr_q + (uint32_t)(K * kAccCols);
                // releases accumulator K on the stage barrier of the tile kNAcc ahead
                uint64_t* release = POS >= 0 ? &t.go[(POS + kNAcc) % T::kNS] : &t.go[(acc_it + kNAcc) % T::kNS];
                const bool more = i + 1 < a.n_it;
                const uint32_t next_par = POS >= 0 ? (uint32_t)(((POS + 1) >> 1) & 1) : ((acc_it + 1) >> 1) & 1u;
                if constexpr (kRowPass<MODE>) {
                    // row passes: TMEM lanes are candidate blocks, columns query rows; a
                    // thread holds 4 blocks x 16 rows and sums each row
                    float v0[32], v1[32];
                    tmem_ld16x256_8(taddr, v0);
                    tmem_ld16x256_8(taddr + (16u << 16), v1);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_lane0(release, lane);
                    ready = more && mbar_done(&t.acc_full[1 - K], next_par);
                    if (MASK) {
                        // blocks past the candidate range (TMEM lanes q*32 + 16h + t/4 + 8e)
                        const int b0 = a.c0 + i * BM + q * 32 + (lane >> 2);
                        const bool ok00 = b0 < a.c1, ok01 = b0 + 8 < a.c1, ok10 = b0 + 16 < a.c1, ok11 = b0 + 24 < a.c1;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            if (!ok00) v0[4 * j] = v0[4 * j + 1] = -INFINITY;
                            if (!ok01) v0[4 * j + 2] = v0[4 * j + 3] = -INFINITY;
                            if (!ok10) v1[4 * j] = v1[4 * j + 1] = -INFINITY;
                            if (!ok11) v1[4 * j + 2] = v1[4 * j + 3] = -INFINITY;
                        }
                    }
                    if constexpr (MODE == 0) {
                        if (i == 0) {
                            // the reference: the largest logit over the warp's 32 blocks x 64
                            // rows of the unit's first tile, plus 16 (log2) of headroom; 0
                            // where the warp holds no candidate
                            float mx = -INFINITY;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float2 m = col_max(v0, v1, j);
                                mx = fmaxf(mx, fmaxf(m.x, m.y));
                            }
#pragma unroll
                            for (int o2 = 1; o2 <= 16; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
                            wnr = mx == -INFINITY ? 0.f : -(mx * kScale + 16.f);
                        }
                        const float2 nr = make_float2(wnr, wnr);
#pragma unroll
                        for (int j = 0; j < 8; ++j) col_pair_terms(v0, v1, j, sc, nr, cs[j]);
                    } else {
                        const int cq = 2 * (lane & 3);  // the thread's first column within each 8
                        if (i == 0) {
                            // references: each column's largest logit over the warp's 32 blocks of
                            // the unit's first tile, plus 64 (log2) of headroom; 0 where the warp
                            // holds no candidate
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                float2 m = col_max(v0, v1, j);
#pragma unroll
                                for (int o2 = 4; o2 <= 16; o2 <<= 1)
                                    m = make_float2(fmaxf(m.x, __shfl_xor_sync(0xffffffffu, m.x, o2)),
                                                    fmaxf(m.y, __shfl_xor_sync(0xffffffffu, m.y, o2)));
                                if (lane < 4)
                                    *reinterpret_cast<float2*>(wref + 8 * j + cq) =
                                        make_float2(m.x == -INFINITY ? 0.f : -(m.x * kScale + 64.f),
                                                    m.y == -INFINITY ? 0.f : -(m.y * kScale + 64.f));
                            }
                            __syncwarp();
                        }
                        // column pair by column pair, so that one pair's references are live at a time
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float2 nr = *reinterpret_cast<const float2*>(wref + 8 * j + cq);
                            col_pair_terms(v0, v1, j, sc, nr, cs[j]);
                        }
                        float big = fmaxf(max3(cs[0].x, cs[0].y, cs[1].x), max3(cs[1].y, cs[2].x, cs[2].y));
                        big = fmaxf(big, max3(cs[3].x, cs[3].y, cs[4].x));
                        big = fmaxf(big, max3(cs[4].y, cs[5].x, cs[5].y));
                        big = fmaxf(big, max3(cs[6].x, cs[6].y, fmaxf(cs[7].x, cs[7].y)));
                        if (__any_sync(0xffffffffu, !(big <= 0x1p100f))) {
                            // sums far above their references: move every reference of the warp
                            // up by 64 and scale the sums down to match
#pragma unroll
                            for (int j = 0; j < 8; ++j) cs[j] = make_float2(cs[j].x * 0x1p-64f, cs[j].y * 0x1p-64f);
                            if (lane < 4) {
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    float2* r = reinterpret_cast<float2*>(wref + 8 * j + cq);
                                    *r = make_float2(r->x - 64.f, r->y - 64.f);
                                }
                            }
                            __syncwarp();
                        }
                    }
                } else {
                    // column pass: pad rows read -inf and add nothing
                    const float nl = nl_n;
                    if (more) nl_n = __ldg(nlse_lg + (i + 1) * BM + r_local);
                    // the warp's 32 lanes in two halves of 16; each thread gets 4 rows x 16
                    // columns, so the whole slice is read before the accumulator is released
                    float v0[32], v1[32];
                    tmem_ld16x256_8(taddr, v0);
                    tmem_ld16x256_8(taddr + (16u << 16), v1);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_lane0(release, lane);
                    ready = more && mbar_done(&t.acc_full[1 - K], next_par);
                    // -lse2 of the thread's rows, from the lanes that loaded them
                    const int rl = lane >> 2;
                    col_terms(v0, 0, sc, __shfl_sync(0xffffffffu, nl, rl), cs);
                    col_terms(v0, 1, sc, __shfl_sync(0xffffffffu, nl, rl + 8), cs);
                    col_terms(v1, 0, sc, __shfl_sync(0xffffffffu, nl, rl + 16), cs);
                    col_terms(v1, 1, sc, __shfl_sync(0xffffffffu, nl, rl + 24), cs);
                }
            };
            using K0 = std::integral_constant<int, 0>;
            using K1 = std::integral_constant<int, 1>;
            using M0 = std::integral_constant<bool, false>;
            using M1 = std::integral_constant<bool, true>;
            // Tiles in fours (accumulators 0, 1, 0, 1 and the four stages' barriers, all
            // known at compile time) after at most three tiles that align the ring; the
            // row pass's ragged last tile (the only one past the candidate range) and the
            // remainder go one at a time.
            static_assert(T::kNS == 4 && kNAcc == 2, "four tiles cycle through the stages once");
            using PR = std::integral_constant<int, -1>;
            using P0 = std::integral_constant<int, 0>;
            using P1 = std::integral_constant<int, 1>;
            using P2 = std::integral_constant<int, 2>;
            using P3 = std::integral_constant<int, 3>;
            const int n_plain = kRowPass<MODE> ? a.n_it - 1 : a.n_it;
            int i = 0;
            auto one = [&](int ii) {
                const bool mask = kRowPass<MODE> && ii + 1 == a.n_it;
                if (acc_it & 1u) {
                    if (mask) tile(K1{}, M1{}, PR{}, ii); else tile(K1{}, M0{}, PR{}, ii);
                } else {
                    if (mask) tile(K0{}, M1{}, PR{}, ii); else tile(K0{}, M0{}, PR{}, ii);
                }
                ++acc_it;
            };
            for (; (acc_it & 3u) && i < n_plain; ++i) one(i);
            for (; i + 4 <= n_plain; i += 4) {
                tile(K0{}, M0{}, P0{}, i);
                ++acc_it;
                tile(K1{}, M0{}, P1{}, i + 1);
                ++acc_it;
                tile(K0{}, M0{}, P2{}, i + 2);
                ++acc_it;
                tile(K1{}, M0{}, P3{}, i + 3);
                ++acc_it;
            }
            for (; i < a.n_it; ++i) one(i);
            if (!(ok = epi_bar_and(ok))) break;
            bool redo = false;  // row pass: a row of the unit needs the exact pass
            if constexpr (kRowPass<MODE>) {
                // each query row's sum over the warp's blocks (one reference per warp and
                // column), then a (reference, sum) merge over the four lane quarters in
                // fixed order -> lse2 of the unit's 256 query rows
                float f[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    f[2 * j] = cs[j].x;
                    f[2 * j + 1] = cs[j].y;
                }
                column_reduce(f, lane);
                float2* red = reinterpret_cast<float2*>(t.red);  // [kSlices][4][kSliceCols]
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int col = 2 * lane + c;
                    const float ref = MODE == 0 ? -wnr : -wref[col];
                    red[(slice * 4 + q) * kSliceCols + col] = make_float2(f[c] > 0.f ? ref : -INFINITY, f[c]);
                }
                epi_bar();
                if (etid < kAccCols) {
                    const int sl = etid / kSliceCols, cc = etid % kSliceCols;
                    const float2* rc = red + sl * 4 * kSliceCols + cc;
                    const float2 m = lse2_merge(lse2_merge(lse2_merge(rc[0], rc[kSliceCols]), rc[2 * kSliceCols]),
                                                rc[3 * kSliceCols]);
                    const int row = o * T::kFRows + etid;
                    if (row < a.rows_g) {
                        a.nlse2[(int64_t)lg * a.rows_pad + row] = m.y > 0.f ? -(m.x + __log2f(m.y)) : INFINITY;
                        // every row has a candidate, so its sum is at least 2^-(74 + 16) of the
                        // reference unless its largest logit lies more than 74 below the warp's
                        redo = MODE == 0 && !(m.y >= 0x1p-90f && m.y <= 0x1p126f);
                    } else if (row < a.rows_pad) {
                        a.nlse2[(int64_t)lg * a.rows_pad + row] = -INFINITY;
                    }
                }
            } else {
                // sum each column over the warp's rows, then over the four lane quarters
                float f[16];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    f[2 * j] = cs[j].x;
                    f[2 * j + 1] = cs[j].y;
                }
                column_reduce(f, lane);
                float* red = t.red;  // [kSlices][4][kSliceCols]
                red[(slice * 4 + q) * kSliceCols + 2 * lane] = f[0];
                red[(slice * 4 + q) * kSliceCols + 2 * lane + 1] = f[1];
                epi_bar();
                if (etid < kAccCols) {
                    const int sl = etid / kSliceCols, cc = etid % kSliceCols;
                    const float* rc = red + sl * 4 * kSliceCols + cc;
                    const float sum = ((rc[0] + rc[kSliceCols]) + rc[2 * kSliceCols]) + rc[3 * kSliceCols];
                    const int b = a.c0 + o * kAccCols + etid;
                    if (b < a.c1) a.mass[(int64_t)lg * a.n_blocks + b] = sum;
                }
            }
            if (MODE == 0) {
                redo = epi_bar_or(redo);
                if (etid == 0) a.redo[u] = redo ? 1 : 0;
            } else {
                epi_bar();
            }
        }
    }

    // epilogue's end: the barrier the first warpgroup waits on before it frees TMEM
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// R[b] = sum_lg mass[lg][b] / (L*Hq) on C; zero outside C (also in mass).  A CTA
// takes 64 blocks; its four thread groups add a quarter of the (l,g) rows each, in
// ascending order, and the four partial sums are added in fixed order.
constexpr int kFinBlocks = 64, kFinParts = 4;
static_assert(kFinParts == 4, "the partial sums are added as ((p0 + p1) + p2) + p3");
__global__ void __launch_bounds__(kFinBlocks * kFinParts) bs_finalize(const float* __restrict__ mass_in, float* mass,
                                                                        float* R, int LH, int n_blocks, int c0, int c1,
                                                                        float inv) {
    __shared__ float part_sum[kFinParts][kFinBlocks];
    const int bl = threadIdx.x % kFinBlocks, part = threadIdx.x / kFinBlocks;
    const int b = blockIdx.x * kFinBlocks + bl;
    const bool in_range = b < n_blocks;
    const bool cand = in_range && b >= c0 && b < c1;
    const int lg0 = (int)((int64_t)LH * part / kFinParts), lg1 = (int)((int64_t)LH * (part + 1) / kFinParts);
    float acc = 0.f;
    if (cand) {
        for (int lg = lg0; lg < lg1; ++lg) acc += mass_in[(int64_t)lg * n_blocks + b];
    } else if (in_range) {
        for (int lg = lg0; lg < lg1; ++lg) mass[(int64_t)lg * n_blocks + b] = 0.f;
    }
    part_sum[part][bl] = acc;
    __syncthreads();
    if (part == 0 && in_range)
        R[b] = cand ? (((part_sum[0][bl] + part_sum[1][bl]) + part_sum[2][bl]) + part_sum[3][bl]) * inv : 0.f;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

PFN_cuTensorMapEncodeTiled_v12000 encoder() { return kvsel_tmap_encoder(); }

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

PFN_cuTensorMapEncodeTiled_v12000 kvsel_tmap_encoder() {
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

size_t block_scores_workspace(int L, int Hq, int Hkv, int M, int n_blocks) {
    const size_t rows_g = (size_t)(Hq / Hkv) * M;
    const size_t rows_pad = (rows_g + BM - 1) / BM * BM;
    const size_t units = (size_t)L * Hkv * ((rows_g + kAccCols - 1) / kAccCols);
    return align256((size_t)L * Hkv * rows_pad * sizeof(float)) + align256((size_t)L * Hkv * n_blocks * sizeof(float)) +
           align256(units * sizeof(int));
}

cudaError_t launch_block_scores(kvsel_ctx* ctx, const void* q, const void* index, int L, int Hq, int Hkv, int M, int D,
                                int n_blocks, int Bcap, int n_sink, int n_recent, float* R, float* R_partial, void* ws,
                                cudaStream_t s, uint64_t wait_ns, int stuck) {
    (void)D;
    const int G = Hq / Hkv;
    const int rows_g = G * M;
    const int c0 = n_sink < n_blocks ? n_sink : n_blocks;
    const int c1 = n_blocks - n_recent > c0 ? n_blocks - n_recent : c0;
    const int ncand = c1 - c0;
    const int LH = L * Hkv;
    char* w = static_cast<char*>(ws);
    float* nlse2 = reinterpret_cast<float*>(w);
    const int rows_pad = (rows_g + BM - 1) / BM * BM;  // whole column-pass tiles
    w += align256((size_t)LH * rows_pad * sizeof(float));
    float* mass_ws = reinterpret_cast<float*>(w);
    w += align256((size_t)LH * n_blocks * sizeof(float));
    int* redo = reinterpret_cast<int*>(w);
    float* mass = R_partial ? R_partial : mass_ws;

    if (ncand > 0) {
        // query rows and index rows as 2-D tensors, in boxes of 256 rows (the fixed
        // operand) and of 128 rows (the streamed one)
        CUtensorMap q256, q128, i256, i128;
        const uint64_t q_rows = (uint64_t)L * Hq * M, i_rows = (uint64_t)LH * Bcap;
        if (!make_map(&q256, q, q_rows, kAccCols) || !make_map(&q128, q, q_rows, BM) ||
            !make_map(&i256, index, i_rows, kAccCols) || !make_map(&i128, index, i_rows, BM))
            return cudaErrorInvalidValue;
        // the register split needs every pass compiled to exactly the launch's count
        for (const void* f : {(const void*)block_scores_tc<0>, (const void*)block_scores_tc<1>,
                              (const void*)block_scores_tc<2>}) {
            cudaFuncAttributes fa;
            const cudaError_t ea = cudaFuncGetAttributes(&fa, f);
            if (ea != cudaSuccess) return ea;
            if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
        }
        cudaError_t e = cudaFuncSetAttribute(block_scores_tc<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem_bytes<0>());
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(block_scores_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem_bytes<1>());
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(block_scores_tc<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem_bytes<2>());
        if (e != cudaSuccess) return e;
        TcArgs a;
        a.rows_g = rows_g;
        a.rows_pad = rows_pad;
        a.c0 = c0;
        a.c1 = c1;
        a.Bcap = Bcap;
        a.n_blocks = n_blocks;
        a.nlse2 = nlse2;
        a.mass = mass;
        a.err = ctx->dev_err;
        a.redo = redo;
        a.wait_ns = wait_ns;
        a.stuck = stuck;
        // row pass: a unit per 256 query rows, the candidate blocks streamed 128 at a
        // time; it writes lse2 of its rows
        a.units_per_lg = (rows_g + kAccCols - 1) / kAccCols;
        a.n_units = LH * a.units_per_lg;
        a.n_it = (ncand + BM - 1) / BM;
        int grid = a.n_units < ctx->num_sms ? a.n_units : ctx->num_sms;
        block_scores_tc<0><<<grid, kThreads, smem_bytes<0>(), s>>>(q256, i128, a);
        // exact pass: the units the row pass marked (none on ordinary inputs; then every
        // CTA only reads its units' marks)
        a.stuck = 0;  // the test hook and its wait limit apply to the row pass only
        a.wait_ns = KVSEL_BLOCK_WAIT_NS;
        block_scores_tc<2><<<grid, kThreads, smem_bytes<2>(), s>>>(q256, i128, a);
        // column pass: a unit per 256 candidate blocks, the query rows streamed 128 at a time
        a.units_per_lg = (ncand + kAccCols - 1) / kAccCols;
        a.n_units = LH * a.units_per_lg;
        a.n_it = (rows_g + BM - 1) / BM;
        grid = a.n_units < ctx->num_sms ? a.n_units : ctx->num_sms;
        block_scores_tc<1><<<grid, kThreads, smem_bytes<1>(), s>>>(i256, q128, a);
    }
    bs_finalize<<<(n_blocks + kFinBlocks - 1) / kFinBlocks, kFinBlocks * kFinParts, 0, s>>>(
        mass, mass, R, LH, n_blocks, c0, c1, 1.0f / ((float)L * (float)Hq));
    return cudaGetLastError();
}

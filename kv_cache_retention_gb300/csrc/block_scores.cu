// KVMEM block relevance R_b (retrieval step: per (layer, query head, query
// token) softmax over the candidate blocks of q . kbar / sqrt(d), summed over
// query tokens and averaged over layer-heads).
//
// For one (layer l, kv head g) the G = Hq/Hkv query heads' rows form one
// contiguous [G*M][D] matrix Q_lg and the index rows one [n_blocks][D] matrix
// K_lg.  The work is two passes over the logits S = Q_lg K_lg^T:
//   pass 1 (row pass):    lse2[r] = log2 sum_{b in C} 2^(S[r,b] * log2e/sqrt(D))
//   pass 2 (column pass): mass[lg][b] = sum_r 2^(S[r,b] * log2e/sqrt(D) - lse2[r])
//   pass 3:               R[b] = sum_lg mass[lg][b] / (L*Hq)   (fixed order)
// Both passes walk the whole logit matrix; nothing of size rows x blocks is
// ever stored.  Each pass reduces along the axis its threads own, so no
// cross-thread reduction of the big matrix is needed.
#include <cuda_bf16.h>

#include "kvsel_internal.h"

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kTile = 64;   // rows x cols per CTA tile (CUDA-core engine)
constexpr int kD = 128;

// Load a 64-row x 128 bf16 tile (rows row0.., clipped to [lo, hi)) transposed
// into fp32 shared memory as sm[d][row].
__device__ void load_tile_t(const __nv_bfloat16* __restrict__ base, int row0, int lo, int hi,
                            float (*sm)[kTile + 4]) {
    for (int idx = threadIdx.x; idx < kTile * (kD / 8); idx += blockDim.x) {
        const int r = idx / (kD / 8), c = idx % (kD / 8);
        const int row = row0 + r;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (row >= lo && row < hi) raw = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)row * kD + 8 * c));
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            sm[8 * c + 2 * k][r] = __uint_as_float(w[k] << 16);
            sm[8 * c + 2 * k + 1][r] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
}

// acc[i][j] = sum_d A[d][ty*4+i] * B[d][tx*4+j]
__device__ __forceinline__ void mma_tile(const float (*A)[kTile + 4], const float (*B)[kTile + 4], int ty, int tx,
                                         float (&acc)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 8
    for (int d = 0; d < kD; ++d) {
        const float4 a = *reinterpret_cast<const float4*>(&A[d][ty * 4]);
        const float4 b = *reinterpret_cast<const float4*>(&B[d][tx * 4]);
        const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
}

struct BSArgs {
    const __nv_bfloat16* q;      // [L][Hq][M][D]
    const __nv_bfloat16* index;  // [L][Hkv][Bcap][D]
    int L, Hq, Hkv, M, Bcap, n_blocks, c0, c1;
    float scale;                 // log2(e)/sqrt(D)
    float* lse2;                 // [L*Hq*M], row order of the [G*M] group matrices
    float* mass;                 // [L*Hkv][n_blocks]
    float* R;
};

// pass 1: grid (row tiles, L*Hkv); 256 threads as 16 x 16, 4x4 outputs each.
__global__ void __launch_bounds__(256) bs_rows_simt(const BSArgs a) {
    extern __shared__ float smem[];
    float (*Qs)[kTile + 4] = reinterpret_cast<float (*)[kTile + 4]>(smem);
    float (*Ks)[kTile + 4] = reinterpret_cast<float (*)[kTile + 4]>(smem + kD * (kTile + 4));
    const int lg = blockIdx.y;
    const int l = lg / a.Hkv, g = lg % a.Hkv;
    const int G = a.Hq / a.Hkv;
    const int rows = G * a.M;
    const int row0 = blockIdx.x * kTile;
    const __nv_bfloat16* Q = a.q + ((int64_t)l * a.Hq + (int64_t)g * G) * a.M * kD;
    const __nv_bfloat16* K = a.index + ((int64_t)l * a.Hkv + g) * a.Bcap * kD;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    load_tile_t(Q, row0, 0, rows, Qs);
    float m[4], s[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        s[i] = 0.f;
    }
    for (int col0 = a.c0; col0 < a.c1; col0 += kTile) {
        __syncthreads();
        load_tile_t(K, col0, a.c0, a.c1, Ks);
        __syncthreads();
        float acc[4][4];
        mma_tile(Qs, Ks, ty, tx, acc);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float v[4], tmax = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool ok = col0 + tx * 4 + j < a.c1;
                v[j] = ok ? acc[i][j] * a.scale : -INFINITY;
                tmax = fmaxf(tmax, v[j]);
            }
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, o));
            const float mn = fmaxf(m[i], tmax);
            float ts = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) ts += exp2f(v[j] - mn);
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) ts += __shfl_xor_sync(kFull, ts, o);
            s[i] = s[i] * exp2f(m[i] - mn) + ts;
            m[i] = mn;
        }
    }
    if (tx == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = row0 + ty * 4 + i;
            if (r < rows) a.lse2[((int64_t)l * a.Hq + (int64_t)g * G) * a.M + r] = m[i] + log2f(s[i]);
        }
    }
}

// pass 2: grid (candidate column tiles, L*Hkv).  Threads own 4 blocks x 4 rows.
__global__ void __launch_bounds__(256) bs_cols_simt(const BSArgs a) {
    extern __shared__ float smem[];
    float (*Ks)[kTile + 4] = reinterpret_cast<float (*)[kTile + 4]>(smem);
    float (*Qs)[kTile + 4] = reinterpret_cast<float (*)[kTile + 4]>(smem + kD * (kTile + 4));
    float* lse_s = smem + 2 * kD * (kTile + 4);
    const int lg = blockIdx.y;
    const int l = lg / a.Hkv, g = lg % a.Hkv;
    const int G = a.Hq / a.Hkv;
    const int rows = G * a.M;
    const int col0 = a.c0 + blockIdx.x * kTile;
    const __nv_bfloat16* Q = a.q + ((int64_t)l * a.Hq + (int64_t)g * G) * a.M * kD;
    const __nv_bfloat16* K = a.index + ((int64_t)l * a.Hkv + g) * a.Bcap * kD;
    const float* lse_lg = a.lse2 + ((int64_t)l * a.Hq + (int64_t)g * G) * a.M;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    load_tile_t(K, col0, a.c0, a.c1, Ks);
    float colsum[4] = {0.f, 0.f, 0.f, 0.f};
    for (int row0 = 0; row0 < rows; row0 += kTile) {
        __syncthreads();
        load_tile_t(Q, row0, 0, rows, Qs);
        for (int r = threadIdx.x; r < kTile; r += blockDim.x)
            lse_s[r] = row0 + r < rows ? lse_lg[row0 + r] : INFINITY;
        __syncthreads();
        float acc[4][4];
        mma_tile(Ks, Qs, ty, tx, acc);  // acc[i][j]: block ty*4+i, row tx*4+j
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) colsum[i] += exp2f(acc[i][j] * a.scale - lse_s[tx * 4 + j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float v = colsum[i];
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
        const int b = col0 + ty * 4 + i;
        if (tx == 0 && b < a.c1) a.mass[(int64_t)lg * a.n_blocks + b] = v;
    }
}

// pass 3: R[b] = sum_lg mass[lg][b] / (L*Hq) on C; zero outside C (also in mass).
__global__ void bs_finalize(const BSArgs a) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= a.n_blocks) return;
    const int LH = a.L * a.Hkv;
    if (b < a.c0 || b >= a.c1) {
        a.R[b] = 0.f;
        for (int lg = 0; lg < LH; ++lg) a.mass[(int64_t)lg * a.n_blocks + b] = 0.f;
        return;
    }
    float acc = 0.f;
    for (int lg = 0; lg < LH; ++lg) acc += a.mass[(int64_t)lg * a.n_blocks + b];
    a.R[b] = acc / ((float)a.L * (float)a.Hq);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t block_scores_workspace(int L, int Hq, int Hkv, int M, int n_blocks) {
    return align256((size_t)L * Hq * M * sizeof(float)) + align256((size_t)L * Hkv * n_blocks * sizeof(float));
}

cudaError_t launch_block_scores(kvsel_ctx* ctx, const void* q, const void* index, int L, int Hq, int Hkv, int M, int D,
                                int n_blocks, int Bcap, int n_sink, int n_recent, float* R, float* R_partial, void* ws,
                                cudaStream_t s) {
    (void)ctx;
    (void)D;
    BSArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.index = static_cast<const __nv_bfloat16*>(index);
    a.L = L;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.M = M;
    a.Bcap = Bcap;
    a.n_blocks = n_blocks;
    a.c0 = n_sink < n_blocks ? n_sink : n_blocks;
    a.c1 = n_blocks - n_recent > a.c0 ? n_blocks - n_recent : a.c0;
    a.scale = kLog2e / sqrtf(128.f);
    char* w = static_cast<char*>(ws);
    a.lse2 = reinterpret_cast<float*>(w);
    w += align256((size_t)L * Hq * M * sizeof(float));
    a.mass = R_partial ? R_partial : reinterpret_cast<float*>(w);
    a.R = R;
    const int G = Hq / Hkv;
    const int rows = G * M;
    const int ncand = a.c1 - a.c0;
    if (ncand > 0) {
        const size_t smem = sizeof(float) * 2 * kD * (kTile + 4);
        cudaFuncSetAttribute(bs_rows_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        bs_rows_simt<<<dim3((rows + kTile - 1) / kTile, L * Hkv), 256, smem, s>>>(a);
        const size_t smem2 = smem + sizeof(float) * kTile;
        cudaFuncSetAttribute(bs_cols_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
        bs_cols_simt<<<dim3((ncand + kTile - 1) / kTile, L * Hkv), 256, smem2, s>>>(a);
    }
    bs_finalize<<<(n_blocks + 255) / 256, 256, 0, s>>>(a);
    return cudaGetLastError();
}

// FP8 (E4M3) storage of the Mean-K index.
//
// KVMEM page, section "design and trade-offs" (one Mean-K vector per block,
// layer and kv head; 9.5 GiB of index for a 10M-token workspace) and its
// server runs, which keep the KV cache in FP8.  A row of D values is stored
// as D E4M3 codes and one power-of-two scale 2^e with e the smallest integer
// >= -100 for which max|x| <= 448 * 2^e; a value is code * 2^e, exact in bf16,
// so the block-score kernel consumes the expanded rows unchanged.
//
// Both kernels give a row to one warp, lane l owning D/32 consecutive values:
// a row moves as one coalesced warp access in each direction.  Rounding to
// E4M3 is the hardware conversion (round to nearest, ties to even); the
// scaling by 2^-e is exact, as is the expansion.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvsel_internal.h"

namespace {

constexpr int kRowsPerBlock = 8;  // warps per CTA

// 2^k as a float, k in [-126, 127]
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float((uint32_t)(127 + k) << 23); }

// e of a row from the bit pattern of its largest magnitude (a non-negative
// float): m = f * 2^x with f in [1/2, 1); 448 = 0.875 * 2^9, so e = x - 9 when
// f <= 0.875 and x - 8 otherwise; at least -100 (zero and tiny rows).
__device__ __forceinline__ int row_exp(uint32_t mbits) {
    const int field = (int)(mbits >> 23);
    if (field == 0) return -100;
    const int x = field - 126;
    const int e = (mbits & 0x7FFFFFu) <= 0x600000u ? x - 9 : x - 8;
    return e < -100 ? -100 : e;
}

// A lane's V values of row r (bf16 bits widened to float).
template <int V>
__device__ __forceinline__ void load_row(const uint16_t* __restrict__ idx, int64_t r, int lane, float (&x)[V]) {
    const uint16_t* src = idx + r * (32 * V) + lane * V;
    if constexpr (V == 4) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
        x[0] = __uint_as_float(w.x << 16);
        x[1] = __uint_as_float(w.x & 0xFFFF0000u);
        x[2] = __uint_as_float(w.y << 16);
        x[3] = __uint_as_float(w.y & 0xFFFF0000u);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) x[i] = __uint_as_float((uint32_t)__ldg(src + i) << 16);
    }
}

// Each warp takes kU rows at a time and issues all their loads before it
// works on any of them, so that several rows per warp are in flight (one row
// at a time reached 0.65 of the HBM copy rate, four reach 0.83 and 1.0; eight
// were slower again).
constexpr int kU = 4;

template <int V>  // values per lane: D / 32
__global__ void __launch_bounds__(32 * kRowsPerBlock) to_fp8_kernel(const uint16_t* __restrict__ idx, int64_t rows,
                                                                     uint8_t* __restrict__ codes,
                                                                     int8_t* __restrict__ exps) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * kRowsPerBlock;
    for (int64_t r0 = ((int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5)) * kU; r0 < rows; r0 += warps * kU) {
        float x[kU][V];
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (r0 + u < rows) load_row<V>(idx, r0 + u, lane, x[u]);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t r = r0 + u;
            if (r >= rows) break;  // warp-uniform
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < V; ++i) m = max(m, __float_as_uint(x[u][i]) & 0x7FFFFFFFu);
#pragma unroll
            for (int s = 16; s >= 1; s >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, s));
            const int e = row_exp(m);
            const float sc = exp2i(-e);
            uint8_t c[V];
#pragma unroll
            for (int i = 0; i < V; i += 2) {
                uint16_t pair;
                // the first source goes to the upper byte
                asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(x[u][i + 1] * sc), "f"(x[u][i] * sc));
                c[i] = (uint8_t)(pair & 0xFF);
                c[i + 1] = (uint8_t)(pair >> 8);
            }
            uint8_t* dst = codes + r * (32 * V) + lane * V;
            if constexpr (V == 4) {
                *reinterpret_cast<uint32_t*>(dst) =
                    (uint32_t)c[0] | ((uint32_t)c[1] << 8) | ((uint32_t)c[2] << 16) | ((uint32_t)c[3] << 24);
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) dst[i] = c[i];
            }
            if (lane == 0) exps[r] = (int8_t)e;
        }
    }
}

template <int V>
__global__ void __launch_bounds__(32 * kRowsPerBlock) from_fp8_kernel(const uint8_t* __restrict__ codes,
                                                                       const int8_t* __restrict__ exps, int64_t rows,
                                                                       uint16_t* __restrict__ idx) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * kRowsPerBlock;
    for (int64_t r0 = ((int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5)) * kU; r0 < rows; r0 += warps * kU) {
        uint8_t c[kU][V];
        int e[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t r = r0 + u;
            e[u] = 0;
            if (r >= rows) continue;
            e[u] = __ldg(exps + r);
            const uint8_t* src = codes + r * (32 * V) + lane * V;
            if constexpr (V == 4) {
                const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(src));
#pragma unroll
                for (int i = 0; i < 4; ++i) c[u][i] = (uint8_t)(w >> (8 * i));
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) c[u][i] = __ldg(src + i);
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t r = r0 + u;
            if (r >= rows) break;  // warp-uniform
            const float sc = exp2i(e[u]);
            uint16_t out[V];
#pragma unroll
            for (int i = 0; i < V; i += 2) {
                const uint16_t pair = (uint16_t)c[u][i] | ((uint16_t)c[u][i + 1] << 8);
                uint32_t h2;  // f16x2: the upper byte's value in the upper half
                asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
                const float lo = __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFF))) * sc;
                const float hi = __half2float(__ushort_as_half((uint16_t)(h2 >> 16))) * sc;
                out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
                out[i + 1] = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
            }
            uint16_t* dst = idx + r * (32 * V) + lane * V;
            if constexpr (V == 4) {
                *reinterpret_cast<uint2*>(dst) = make_uint2((uint32_t)out[0] | ((uint32_t)out[1] << 16),
                                                            (uint32_t)out[2] | ((uint32_t)out[3] << 16));
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) dst[i] = out[i];
            }
        }
    }
}

int grid_for(const kvsel_ctx* ctx, int64_t rows) {
    const int64_t want = (rows + kRowsPerBlock * kU - 1) / (kRowsPerBlock * kU);
    const int64_t cap = (int64_t)ctx->num_sms * 16;
    return (int)(want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_index_to_fp8(const kvsel_ctx* ctx, const void* index, int64_t rows, int D, uint8_t* codes,
                                int8_t* exps, cudaStream_t s) {
    const int g = grid_for(ctx, rows);
    const uint16_t* idx = static_cast<const uint16_t*>(index);
    switch (D) {
        case 64: to_fp8_kernel<2><<<g, 32 * kRowsPerBlock, 0, s>>>(idx, rows, codes, exps); break;
        case 128: to_fp8_kernel<4><<<g, 32 * kRowsPerBlock, 0, s>>>(idx, rows, codes, exps); break;
        case 256: to_fp8_kernel<8><<<g, 32 * kRowsPerBlock, 0, s>>>(idx, rows, codes, exps); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_index_from_fp8(const kvsel_ctx* ctx, const uint8_t* codes, const int8_t* exps, int64_t rows, int D,
                                  void* index, cudaStream_t s) {
    const int g = grid_for(ctx, rows);
    uint16_t* idx = static_cast<uint16_t*>(index);
    switch (D) {
        case 64: from_fp8_kernel<2><<<g, 32 * kRowsPerBlock, 0, s>>>(codes, exps, rows, idx); break;
        case 128: from_fp8_kernel<4><<<g, 32 * kRowsPerBlock, 0, s>>>(codes, exps, rows, idx); break;
        case 256: from_fp8_kernel<8><<<g, 32 * kRowsPerBlock, 0, s>>>(codes, exps, rows, idx); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// KVMEM elementwise kernels: the Mean-K index build (retrieval index: one mean
// of the position-free K rows per block, layer and kv head) and the
// position-consistent restore (re-RoPE of raw K at new compact positions,
// scattered into a paged pool).  Both are HBM-bound: every K byte is read once
// with 16-byte coalesced loads and every output byte written once.
//
// Rotation angles: position p < 2^24 is split as p = hi * 1024 + lo and the
// angle p * theta_i is rebuilt by the angle-addition formula from two tables
// of cos/sin computed in fp64 and stored in fp32, so that large positions keep
// ~1e-7 absolute accuracy (a plain fp32 product p * theta_i would not).
#include <cuda_bf16.h>

#include "kvsel_internal.h"

namespace {

constexpr unsigned kFull = 0xffffffffu;

__global__ void rope_tables_kernel(float2* __restrict__ lo, float2* __restrict__ hi, int D, double base) {
    const int half = D / 2;
    const int64_t total = (int64_t)(KVSEL_ROPE_LO + KVSEL_ROPE_HI) * half;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(idx % half);
        const int64_t row = idx / half;
        const double theta = pow(base, -2.0 * (double)i / (double)D);
        double s, c;
        if (row < KVSEL_ROPE_LO) {
            sincos((double)row * theta, &s, &c);
            lo[row * half + i] = make_float2((float)c, (float)s);
        } else {
            const int64_t r = row - KVSEL_ROPE_LO;
            sincos((double)(r * KVSEL_ROPE_LO) * theta, &s, &c);
            hi[r * half + i] = make_float2((float)c, (float)s);
        }
    }
}

// cos/sin of p * theta_i by angle addition of the hi and lo table entries.
__device__ __forceinline__ float2 rope_cs(const float2* __restrict__ tlo, const float2* __restrict__ thi, int half,
                                          int p, int i) {
    const float2 a = __ldg(thi + (int64_t)(p >> KVSEL_ROPE_LO_BITS) * half + i);
    const float2 b = __ldg(tlo + (int64_t)(p & (KVSEL_ROPE_LO - 1)) * half + i);
    return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.y, b.x, a.x * b.y));
}

__device__ __forceinline__ void unpack8(uint4 raw, float (&x)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Rotate the 8 dims [8c, 8c+8) a lane holds by position p (inverse: by -p).
// NeoX pairs (i, i+D/2) live in lanes c and c ^ (LR/2) of the same row; the
// interleaved pairs (2i, 2i+1) are inside the lane.  All lanes of the warp must
// call this (it shuffles).
__device__ __forceinline__ void rotate8(float (&x)[8], int c, int LR, int D, int p, bool inverse, int style,
                                        const float2* tlo, const float2* thi) {
    const int half = D / 2;
    if (style == KVSEL_ROPE_NEOX) {
        const bool a_side = c < (LR >> 1);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float y = __shfl_xor_sync(kFull, x[k], LR >> 1);
            const int i = (8 * c + k) & (half - 1);
            float2 cs = rope_cs(tlo, thi, half, p, i);
            const float s = inverse ? -cs.y : cs.y;
            x[k] = a_side ? fmaf(x[k], cs.x, -y * s) : fmaf(x[k], cs.x, y * s);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const int i = (8 * c + k) >> 1;
            float2 cs = rope_cs(tlo, thi, half, p, i);
            const float s = inverse ? -cs.y : cs.y;
            const float a = x[k], b = x[k + 1];
            x[k] = fmaf(a, cs.x, -b * s);
            x[k + 1] = fmaf(b, cs.x, a * s);
        }
    }
}

// One warp per (l, g, block).  LR = D/8 lanes cover a row; RI = 32/LR rows per step.
__global__ void __launch_bounds__(256) meank_kernel(const __nv_bfloat16* __restrict__ k_src, int T, int D, int block,
                                                    int first_block, int nb, int64_t n_warps,
                                                    const int32_t* __restrict__ src_pos, const float2* tlo,
                                                    const float2* thi, int style, __nv_bfloat16* __restrict__ index,
                                                    int Bcap, unsigned* dev_err) {
    const int64_t w = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
    if (w >= n_warps) return;  // whole warp leaves together
    const int lane = threadIdx.x & 31;
    const int b = (int)(w % nb);
    const int64_t lg = w / nb;
    const int t0 = b * block, t1 = min(T, t0 + block);
    const int LR = D >> 3, RI = 32 / LR;
    const int c = lane % LR, r0 = lane / LR;
    const __nv_bfloat16* rows = k_src + lg * (int64_t)T * D + 8 * c;
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
    if (!src_pos) {
#pragma unroll 4
        for (int t = t0 + r0; t < t1; t += RI) {
            float x[8];
            unpack8(__ldcs(reinterpret_cast<const uint4*>(rows + (int64_t)t * D)), x);
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] += x[k];
        }
    } else {
        for (int tb = t0; tb < t1; tb += RI) {  // uniform trip count: rotate8 shuffles
            const int t = tb + r0;
            const bool valid = t < t1;
            float x[8];
            int p = 0;
            if (valid) {
                unpack8(__ldcs(reinterpret_cast<const uint4*>(rows + (int64_t)t * D)), x);
                p = __ldg(src_pos + t);
                if (p < 0 || p >= KVSEL_MAX_POS) {
                    atomicOr(dev_err, (unsigned)KVSEL_DEV_BAD_POSITION);
                    p = 0;
                }
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) x[k] = 0.f;
            }
            rotate8(x, c, LR, D, p, true, style, tlo, thi);
            if (valid) {
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[k] += x[k];
            }
        }
    }
    for (int o = LR; o < 32; o <<= 1) {
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] += __shfl_xor_sync(kFull, acc[k], o);
    }
    if (r0 == 0) {
        const float cnt = (float)(t1 - t0);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = acc[k] / cnt;
        __nv_bfloat16* out = index + (lg * Bcap + first_block + b) * (int64_t)D + 8 * c;
        *reinterpret_cast<uint4*>(out) = pack8(acc);
    }
}

// One block per (entry i, group of kLayerGroup layers).  The block first fills
// a shared [page][D/2] table of (cos, sin) for positions dst_pos0[i] + t (the
// same for every layer and kv head), then moves the page: a lane owns one
// rotation pair of 16-byte chunks of a row -- chunks c and c + D/16, i.e. the
// NeoX halves (i, i + D/2) of 8 frequencies, or two chunks of interleaved
// pairs -- so no data crosses lanes.  Rows r = t*Hkv + g are contiguous in the
// destination page; each source row is contiguous too.
constexpr int kLayerGroup = 8;

// Incoming-block restore.  WITH_V also copies the block's V rows (V carries no
// position) to the same page of v_pool in the same pass.  n_dev, when given, is
// a device-side entry count: CTAs past it return at once, so a launch sized
// for the largest count needs no host round trip.
template <bool WITH_V>
__global__ void __launch_bounds__(256) rerope_kernel(const __nv_bfloat16* __restrict__ k_src, int64_t sls, int64_t shs,
                                                     int src_tokens, const int32_t* __restrict__ src_block,
                                                     const int32_t* __restrict__ dst_page,
                                                     const int32_t* __restrict__ dst_pos0, const int32_t* n_dev,
                                                     int L, int Hkv, int D, int page, const float2* tlo,
                                                     const float2* thi, int style, __nv_bfloat16* __restrict__ pool,
                                                     const __nv_bfloat16* __restrict__ v_src,
                                                     __nv_bfloat16* __restrict__ v_pool, int P, unsigned* dev_err) {
    if (n_dev && (int)blockIdx.x >= __ldg(n_dev)) return;
    extern __shared__ float2 cs[];  // [page][D/2]
    const int i = blockIdx.x;
    const int l0 = blockIdx.y * kLayerGroup, l1 = min(L, l0 + kLayerGroup);
    const int sb = __ldg(src_block + i), dp = __ldg(dst_page + i), p0 = __ldg(dst_pos0 + i);
    const bool ok_src = sb >= 0 && (int64_t)(sb + 1) * page <= src_tokens;
    const bool ok_dst = dp >= 0 && dp < P;
    const bool ok_pos = p0 >= 0 && (int64_t)p0 + page <= KVSEL_MAX_POS;
    if (!(ok_src && ok_dst && ok_pos)) {
        if (threadIdx.x == 0 && blockIdx.y == 0)
            atomicOr(dev_err, (ok_src ? 0u : (unsigned)KVSEL_DEV_BAD_BLOCK) | (ok_dst ? 0u : (unsigned)KVSEL_DEV_BAD_PAGE) |
                                  (ok_pos ? 0u : (unsigned)KVSEL_DEV_BAD_POSITION));
        return;  // whole block leaves together
    }
    const int half = D / 2;
    for (int idx = threadIdx.x; idx < page * half; idx += blockDim.x)
        cs[idx] = rope_cs(tlo, thi, half, p0 + idx / half, idx % half);
    __syncthreads();
    const int PR = D >> 4;              // chunk pairs per row
    const int total = page * Hkv * PR;
    for (int l = l0; l < l1; ++l) {
        const __nv_bfloat16* src_l = k_src + (int64_t)l * sls + (int64_t)sb * page * D;
        __nv_bfloat16* dst = pool + ((int64_t)l * P + dp) * (int64_t)page * Hkv * D;
        for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
            const int cp = idx % PR, r = idx / PR;
            const int t = r / Hkv, g = r % Hkv;
            const __nv_bfloat16* srow = src_l + (int64_t)g * shs + (int64_t)t * D;
            __nv_bfloat16* drow = dst + (int64_t)r * D;
            const float2* cst = cs + t * half;
            // NeoX: chunk cp holds dims 8cp.. (first half), chunk cp + PR holds dims 8cp + D/2..
            // interleaved: chunks cp and cp + PR each hold 4 adjacent pairs
            const int ca = cp, cb = cp + PR;
            float xa[8], xb[8];
            unpack8(__ldcs(reinterpret_cast<const uint4*>(srow + 8 * ca)), xa);
            unpack8(__ldcs(reinterpret_cast<const uint4*>(srow + 8 * cb)), xb);
            if (style == KVSEL_ROPE_NEOX) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 c = cst[8 * cp + k];
                    const float a = xa[k], b = xb[k];
                    xa[k] = fmaf(a, c.x, -b * c.y);
                    xb[k] = fmaf(b, c.x, a * c.y);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 8; k += 2) {
                    const float2 c1 = cst[4 * ca + k / 2], c2 = cst[4 * cb + k / 2];
                    const float a1 = xa[k], b1 = xa[k + 1], a2 = xb[k], b2 = xb[k + 1];
                    xa[k] = fmaf(a1, c1.x, -b1 * c1.y);
                    xa[k + 1] = fmaf(b1, c1.x, a1 * c1.y);
                    xb[k] = fmaf(a2, c2.x, -b2 * c2.y);
                    xb[k + 1] = fmaf(b2, c2.x, a2 * c2.y);
                }
            }
            __stcs(reinterpret_cast<uint4*>(drow + 8 * ca), pack8(xa));
            __stcs(reinterpret_cast<uint4*>(drow + 8 * cb), pack8(xb));
            if constexpr (WITH_V) {
                // V: the same two 16-byte chunks of the V row, copied as they are
                const __nv_bfloat16* vrow = v_src + (srow - k_src);
                __nv_bfloat16* vdst = v_pool + (drow - pool);
                __stcs(reinterpret_cast<uint4*>(vdst + 8 * ca), __ldcs(reinterpret_cast<const uint4*>(vrow + 8 * ca)));
                __stcs(reinterpret_cast<uint4*>(vdst + 8 * cb), __ldcs(reinterpret_cast<const uint4*>(vrow + 8 * cb)));
            }
        }
    }
}

// In-place move of retained blocks: every row of page pages[i] is turned by
// shifts[i] positions (negative: backwards), one rounding to bf16.  Grid: one
// CTA per (entry, group of kLayerGroup layers); the D/2 (cos, sin) pairs of the
// shift are computed once per CTA.
__global__ void __launch_bounds__(256) shift_kernel(__nv_bfloat16* __restrict__ pool, int P,
                                                    const int32_t* __restrict__ pages,
                                                    const int32_t* __restrict__ shifts, const int32_t* n_dev, int L,
                                                    int Hkv, int D, int page, const float2* tlo, const float2* thi,
                                                    int style, unsigned* dev_err) {
    __shared__ float2 cs[128];  // [D/2]
    if (n_dev && (int)blockIdx.x >= __ldg(n_dev)) return;
    const int i = blockIdx.x;
    const int l0 = blockIdx.y * kLayerGroup, l1 = min(L, l0 + kLayerGroup);
    const int pg = __ldg(pages + i), sh = __ldg(shifts + i);
    const int mag = sh < 0 ? -sh : sh;
    const bool ok_page = pg >= 0 && pg < P, ok_shift = mag < KVSEL_MAX_POS;
    if (!(ok_page && ok_shift)) {
        if (threadIdx.x == 0 && blockIdx.y == 0)
            atomicOr(dev_err, (ok_page ? 0u : (unsigned)KVSEL_DEV_BAD_PAGE) | (ok_shift ? 0u : (unsigned)KVSEL_DEV_BAD_POSITION));
        return;
    }
    const int half = D / 2;
    for (int idx = threadIdx.x; idx < half; idx += blockDim.x) {
        const float2 c = rope_cs(tlo, thi, half, mag, idx);
        cs[idx] = make_float2(c.x, sh < 0 ? -c.y : c.y);  // a backward turn negates the sine
    }
    __syncthreads();
    const int PR = D >> 4;
    const int total = page * Hkv * PR;
    for (int l = l0; l < l1; ++l) {
        __nv_bfloat16* base = pool + ((int64_t)l * P + pg) * (int64_t)page * Hkv * D;
        for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
            const int cp = idx % PR, r = idx / PR;
            __nv_bfloat16* row = base + (int64_t)r * D;
            const int ca = cp, cb = cp + PR;
            float xa[8], xb[8];
            unpack8(*reinterpret_cast<const uint4*>(row + 8 * ca), xa);
            unpack8(*reinterpret_cast<const uint4*>(row + 8 * cb), xb);
            if (style == KVSEL_ROPE_NEOX) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 c = cs[8 * cp + k];
                    const float a = xa[k], b = xb[k];
                    xa[k] = fmaf(a, c.x, -b * c.y);
                    xb[k] = fmaf(b, c.x, a * c.y);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 8; k += 2) {
                    const float2 c1 = cs[4 * ca + k / 2], c2 = cs[4 * cb + k / 2];
                    const float a1 = xa[k], b1 = xa[k + 1], a2 = xb[k], b2 = xb[k + 1];
                    xa[k] = fmaf(a1, c1.x, -b1 * c1.y);
                    xa[k + 1] = fmaf(b1, c1.x, a1 * c1.y);
                    xb[k] = fmaf(a2, c2.x, -b2 * c2.y);
                    xb[k + 1] = fmaf(b2, c2.x, a2 * c2.y);
                }
            }
            *reinterpret_cast<uint4*>(row + 8 * ca) = pack8(xa);
            *reinterpret_cast<uint4*>(row + 8 * cb) = pack8(xb);
        }
    }
}

}  // namespace

cudaError_t launch_rope_tables(float2* lo, float2* hi, int D, double base, cudaStream_t s) {
    const int64_t total = (int64_t)(KVSEL_ROPE_LO + KVSEL_ROPE_HI) * (D / 2);
    int grid = (int)((total + 255) / 256);
    if (grid > 8192) grid = 8192;
    rope_tables_kernel<<<grid, 256, 0, s>>>(lo, hi, D, base);
    return cudaGetLastError();
}

cudaError_t launch_meank(const void* k_src, int L, int Hkv, int T, int D, int block, int first_block,
                         const int32_t* src_pos, const kvsel_ctx::RopeTab* tab, int rope_style, void* index, int Bcap,
                         unsigned* dev_err, cudaStream_t s) {
    const int nb = (T + block - 1) / block;
    const int64_t n_warps = (int64_t)L * Hkv * nb;
    const int64_t grid = (n_warps + 7) / 8;
    meank_kernel<<<(unsigned)grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(k_src), T, D, block, first_block, nb,
                                                n_warps, src_pos, tab ? tab->lo : nullptr, tab ? tab->hi : nullptr,
                                                rope_style, static_cast<__nv_bfloat16*>(index), Bcap, dev_err);
    return cudaGetLastError();
}

cudaError_t launch_rerope(const void* k_src, int64_t sls, int64_t shs, int src_tokens, const int32_t* src_block,
                          const int32_t* dst_page, const int32_t* dst_pos0, int n, const int32_t* n_dev, int L,
                          int Hkv, int D, int page, const kvsel_ctx::RopeTab* tab, int rope_style, void* pool,
                          const void* v_src, void* v_pool, int P, unsigned* dev_err, cudaStream_t s) {
    const dim3 grid((unsigned)n, (unsigned)((L + kLayerGroup - 1) / kLayerGroup));
    const size_t smem = sizeof(float2) * (size_t)page * (D / 2);
    auto kern = v_src ? rerope_kernel<true> : rerope_kernel<false>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<grid, 256, smem, s>>>(static_cast<const __nv_bfloat16*>(k_src), sls, shs, src_tokens, src_block, dst_page,
                                 dst_pos0, n_dev, L, Hkv, D, page, tab->lo, tab->hi, rope_style,
                                 static_cast<__nv_bfloat16*>(pool), static_cast<const __nv_bfloat16*>(v_src),
                                 static_cast<__nv_bfloat16*>(v_pool), P, dev_err);
    return cudaGetLastError();
}

cudaError_t launch_shift(void* pool, int P, const int32_t* pages, const int32_t* shifts, int n, const int32_t* n_dev,
                         int L, int Hkv, int D, int page, const kvsel_ctx::RopeTab* tab, int rope_style,
                         unsigned* dev_err, cudaStream_t s) {
    const dim3 grid((unsigned)n, (unsigned)((L + kLayerGroup - 1) / kLayerGroup));
    shift_kernel<<<grid, 256, 0, s>>>(static_cast<__nv_bfloat16*>(pool), P, pages, shifts, n_dev, L, Hkv, D, page,
                                      tab->lo, tab->hi, rope_style, dev_err);
    return cudaGetLastError();
}

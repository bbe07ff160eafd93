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
//
// Turning a pair (a, b) in fp32 this way leaves an absolute error below
// 2^-20.5 * rho, rho = |(a, b)|.  That is under half a bf16 ulp of an output r
// as long as |r| >= 2^-11.5 * rho.  Outputs that nearly cancel (|r| below
// 2^-11 * max(|a|, |b|), about one pair in 1700) are turned again in
// double-float arithmetic (pairs of fp32 numbers, about 44 bits) from
// double-float copies of the same tables and rounded once to bf16, so every
// output lands within one bf16 ulp of the exactly rotated value rounded to bf16.
// Double-float rather than fp64: this GPU's fp64 pipe is narrow, and fp64 turns
// kept it a quarter busy in the scatter.
#include <cuda_bf16.h>

#include "kvsel_internal.h"

namespace {

constexpr unsigned kFull = 0xffffffffu;

// fp64 value v as a double-float (hi, lo): hi = v rounded to fp32, lo = the rest rounded to fp32.
__device__ __forceinline__ float2 split_df(double v) {
    const float h = (float)v;
    return make_float2(h, (float)(v - (double)h));
}

__global__ void rope_tables_kernel(float2* __restrict__ lo, float2* __restrict__ hi, float4* __restrict__ lodf,
                                   float4* __restrict__ hidf, int D, double base) {
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
            const float2 cd = split_df(c), sd = split_df(s);
            lodf[row * half + i] = make_float4(cd.x, cd.y, sd.x, sd.y);
        } else {
            const int64_t r = row - KVSEL_ROPE_LO;
            sincos((double)(r * KVSEL_ROPE_LO) * theta, &s, &c);
            hi[r * half + i] = make_float2((float)c, (float)s);
            const float2 cd = split_df(c), sd = split_df(s);
            hidf[r * half + i] = make_float4(cd.x, cd.y, sd.x, sd.y);
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

// Double-float arithmetic: a value held as the unevaluated sum hi + lo of two
// fp32 numbers.  Products take the exact remainder of the leading product from
// an fma; sums take the exact rounding error of the leading sum (Knuth's
// two-sum), so each operation keeps about 44 bits where fp32 keeps 24.  The
// explicitly rounded intrinsics keep the compiler from fusing a product into a
// later sum, which would break the error terms.
struct DF {
    float hi, lo;
};
__device__ __forceinline__ DF df_mul(DF x, DF y) {
    const float p = __fmul_rn(x.hi, y.hi);
    float e = fmaf(x.hi, y.hi, -p);
    e = fmaf(x.hi, y.lo, e);
    e = fmaf(x.lo, y.hi, e);
    return {p, e};
}
__device__ __forceinline__ DF df_mul(float x, DF y) {
    const float p = __fmul_rn(x, y.hi);
    float e = fmaf(x, y.hi, -p);
    e = fmaf(x, y.lo, e);
    return {p, e};
}
__device__ __forceinline__ DF df_add(DF x, DF y) {
    const float s = __fadd_rn(x.hi, y.hi);
    const float bb = __fsub_rn(s, x.hi);
    const float err = __fadd_rn(__fsub_rn(x.hi, __fsub_rn(s, bb)), __fsub_rn(y.hi, bb));
    const float lo = __fadd_rn(err, __fadd_rn(x.lo, y.lo));
    const float h = __fadd_rn(s, lo);
    return {h, __fsub_rn(lo, __fsub_rn(h, s))};
}
__device__ __forceinline__ DF df_neg(DF x) { return {-x.hi, -x.lo}; }

// Double-float turn of one rotation pair, elements ia and ib of a bf16 row read
// again from memory (the row is not overwritten before this runs), at position
// p and frequency f (sine negated when neg): cos and sin of p * theta_f by angle
// addition of the double-float table entries, then the rotation, each output
// rounded once to bf16 and returned as the exactly representable fp32 value.
// Out of line: it runs for about one pair in 1700, and an inlined copy would be
// predicated into every pass.
__device__ __noinline__ float2 turn_pair_df(const __nv_bfloat16* __restrict__ row, int ia, int ib,
                                            const float4* __restrict__ tlo, const float4* __restrict__ thi,
                                            int half, int p, int f, int neg) {
    const float a = __bfloat162float(row[ia]), b = __bfloat162float(row[ib]);
    const float4 u = __ldg(thi + (int64_t)(p >> KVSEL_ROPE_LO_BITS) * half + f);
    const float4 v = __ldg(tlo + (int64_t)(p & (KVSEL_ROPE_LO - 1)) * half + f);
    const DF cu = {u.x, u.y}, su = {u.z, u.w}, cv = {v.x, v.y}, sv = {v.z, v.w};
    const DF c = df_add(df_mul(cu, cv), df_neg(df_mul(su, sv)));
    DF s = df_add(df_mul(su, cv), df_mul(cu, sv));
    if (neg) s = df_neg(s);
    const DF ra = df_add(df_mul(a, c), df_neg(df_mul(b, s)));
    const DF rb = df_add(df_mul(b, c), df_mul(a, s));
    return make_float2(__bfloat162float(__float2bfloat16_rn(ra.hi)), __bfloat162float(__float2bfloat16_rn(rb.hi)));
}

// (cos, sin) tables in shared memory, one row of D/2 frequencies per position.
// Frequencies f of a row are grouped by eight (the ones a NeoX chunk pair uses):
// group g holds four float4 (c_f, c_f+1, s_f, s_f+1) for f = 8g, 8g+2, 8g+4, 8g+6
// and one float4 of padding, so that the eight groups a warp reads at once fall
// in different shared-memory banks, and the packed fp32x2 turn below finds its
// cosines and sines in register pairs.
constexpr int kQuadsPerGroup = 5;
__device__ __forceinline__ void cs_put(float4* row, int f, float c, float s) {
    float* q = reinterpret_cast<float*>(row + (f >> 3) * kQuadsPerGroup + ((f & 7) >> 1));
    q[f & 1] = c;
    q[2 + (f & 1)] = s;
}
__device__ __forceinline__ float2 cs_get(const float4* row, int f) {
    const float* q = reinterpret_cast<const float*>(row + (f >> 3) * kQuadsPerGroup + ((f & 7) >> 1));
    return make_float2(q[f & 1], q[2 + (f & 1)]);
}

// Records in `near` (bit k) whether pair k's fp32 turn (ra, rb) of (a, b) has an
// output below 2^-11 of its larger input.
__device__ __forceinline__ void mark_near(unsigned& near, int k, float a, float b, float ra, float rb) {
    near |= (fminf(fabsf(ra), fabsf(rb)) < fmaxf(fabsf(a), fabsf(b)) * 0x1p-11f ? 1u : 0u) << k;
}

// Turns again in double-float arithmetic the pairs marked in `near`, reading their inputs from `row`.
template <bool NEOX>
__device__ __forceinline__ void fix_near(unsigned near, float (&xa)[8], float (&xb)[8], int f0, int fa, int fb,
                                         const __nv_bfloat16* __restrict__ row, int ca, int cb,
                                         const float4* __restrict__ tlodf, const float4* __restrict__ thidf,
                                         int half, int p, bool neg) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if (near & (1u << k)) {
            float& a = NEOX ? xa[k] : (k < 4 ? xa[2 * k] : xb[2 * (k - 4)]);
            float& b = NEOX ? xb[k] : (k < 4 ? xa[2 * k + 1] : xb[2 * (k - 4) + 1]);
            const int ia = NEOX ? 8 * ca + k : (k < 4 ? 8 * ca + 2 * k : 8 * cb + 2 * (k - 4));
            const int ib = NEOX ? 8 * cb + k : ia + 1;
            const int f = NEOX ? f0 + k : (k < 4 ? fa + k : fb + k - 4);
            const float2 r = turn_pair_df(row, ia, ib, tlodf, thidf, half, p, f, neg ? 1 : 0);
            a = r.x;
            b = r.y;
        }
    }
}

// Turns the 8 rotation pairs held in two unpacked 16-byte chunks (chunks ca and
// cb of `row`) with the (cos, sin) table row `tq` of their position.  NeoX: pair
// k is (xa[k], xb[k]) at frequency f0 + k (f0 a multiple of 8), turned two pairs
// at a time in packed fp32x2; interleaved: pairs (xa[2k], xa[2k+1]) at fa + k and
// (xb[2k], xb[2k+1]) at fb + k.  A pair with an output below 2^-11 of its larger
// input is turned again in double-float arithmetic.
template <bool NEOX>
__device__ __forceinline__ void turn_chunks(float (&xa)[8], float (&xb)[8], const float4* __restrict__ tq, int f0,
                                            int fa, int fb, const __nv_bfloat16* __restrict__ row, int ca, int cb,
                                            const float4* __restrict__ tlodf, const float4* __restrict__ thidf,
                                            int half, int p, bool neg) {
    unsigned near = 0;
    if (NEOX) {
        const float4* grp = tq + (f0 >> 3) * kQuadsPerGroup;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 q = grp[j];
            const float2 c2 = make_float2(q.x, q.y), s2 = make_float2(q.z, q.w);
            const float2 a2 = make_float2(xa[2 * j], xa[2 * j + 1]), b2 = make_float2(xb[2 * j], xb[2 * j + 1]);
            const float2 ra2 = __ffma2_rn(a2, c2, __fmul2_rn(b2, make_float2(-s2.x, -s2.y)));
            const float2 rb2 = __ffma2_rn(b2, c2, __fmul2_rn(a2, s2));
            mark_near(near, 2 * j, a2.x, b2.x, ra2.x, rb2.x);
            mark_near(near, 2 * j + 1, a2.y, b2.y, ra2.y, rb2.y);
            xa[2 * j] = ra2.x;
            xa[2 * j + 1] = ra2.y;
            xb[2 * j] = rb2.x;
            xb[2 * j + 1] = rb2.y;
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float& a = k < 4 ? xa[2 * k] : xb[2 * (k - 4)];
            float& b = k < 4 ? xa[2 * k + 1] : xb[2 * (k - 4) + 1];
            const float2 c = cs_get(tq, k < 4 ? fa + k : fb + k - 4);
            const float ra = fmaf(a, c.x, -b * c.y);
            const float rb = fmaf(b, c.x, a * c.y);
            mark_near(near, k, a, b, ra, rb);
            a = ra;
            b = rb;
        }
    }
    if (__any_sync(__activemask(), near != 0))
        fix_near<NEOX>(near, xa, xb, f0, fa, fb, row, ca, cb, tlodf, thidf, half, p, neg);
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
constexpr int kLayerGroup = 16;
#ifndef KVSEL_REROPE_MINB
#define KVSEL_REROPE_MINB 4  // resident CTAs per SM the register budget allows (64 registers)
#endif

// Incoming-block restore.  WITH_V also copies the block's V rows (V carries no
// position) to the same page of v_pool in the same pass.  n_dev, when given, is
// a device-side entry count: CTAs past it return at once, so a launch sized
// for the largest count needs no host round trip.
template <bool WITH_V>
__global__ void __launch_bounds__(256, KVSEL_REROPE_MINB) rerope_kernel(const __nv_bfloat16* __restrict__ k_src, int64_t sls, int64_t shs,
                                                     int src_tokens, const int32_t* __restrict__ src_block,
                                                     const int32_t* __restrict__ dst_page,
                                                     const int32_t* __restrict__ dst_pos0, const int32_t* n_dev,
                                                     int L, int Hkv, int D, int page, const float2* tlo,
                                                     const float2* thi, const float4* tlodf, const float4* thidf,
                                                     int style, __nv_bfloat16* __restrict__ pool,
                                                     const __nv_bfloat16* __restrict__ v_src,
                                                     __nv_bfloat16* __restrict__ v_pool, int P, unsigned* dev_err) {
    if (n_dev && (int)blockIdx.x >= __ldg(n_dev)) return;
    extern __shared__ float4 cs[];  // [page][D/16 groups][kQuadsPerGroup]
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
    const int PR = D >> 4;              // chunk pairs per row = frequency groups of eight
    const int qrow = PR * kQuadsPerGroup;  // float4 per table row
    // A thread keeps one chunk pair cp of rows r0, r0 + dr, ... of every layer
    // (blockDim is a multiple of PR), and loads its next row's chunks before it
    // turns the current ones.
    const int rows = page * Hkv;
    const int cp = threadIdx.x & (PR - 1), r0 = threadIdx.x / PR;
    const int dr = blockDim.x / PR, dt = dr / Hkv, dg = dr % Hkv;
    const int t0 = r0 / Hkv, g0 = r0 % Hkv;
    // NeoX: chunk cp holds dims 8cp.. (first half), chunk cp + PR holds dims 8cp + D/2..
    // interleaved: chunks cp and cp + PR each hold 4 adjacent pairs
    const int ca = cp, cb = cp + PR;
    auto src_row = [&](int l, int t, int g) {
        return k_src + (int64_t)l * sls + (int64_t)sb * page * D + (int64_t)g * shs + (int64_t)t * D;
    };
    int l = l0, r = r0, t = t0, g = g0;
    const __nv_bfloat16* srow = src_row(l, t, g);
    // the first row's chunks are on their way while the table is built
    uint4 wa = make_uint4(0, 0, 0, 0), wb = wa;
    if (r0 < rows) {
        wa = __ldcs(reinterpret_cast<const uint4*>(srow + 8 * ca));
        wb = __ldcs(reinterpret_cast<const uint4*>(srow + 8 * cb));
    }
    for (int idx = threadIdx.x; idx < page * half; idx += blockDim.x) {
        const float2 c = rope_cs(tlo, thi, half, p0 + idx / half, idx % half);
        cs_put(cs + (idx / half) * qrow, idx % half, c.x, c.y);
    }
    __syncthreads();
    if (r0 >= rows) return;  // no barrier follows
    for (;;) {
        int ln = l, rn = r + dr, tn = t + dt, gn = g + dg;
        if (gn >= Hkv) {
            gn -= Hkv;
            ++tn;
        }
        if (rn >= rows) {
            ++ln;
            rn = r0;
            tn = t0;
            gn = g0;
        }
        const bool more = ln < l1;
        const __nv_bfloat16* snext = more ? src_row(ln, tn, gn) : srow;
        uint4 na = make_uint4(0, 0, 0, 0), nb = na;
        if (more) {
            na = __ldcs(reinterpret_cast<const uint4*>(snext + 8 * ca));
            nb = __ldcs(reinterpret_cast<const uint4*>(snext + 8 * cb));
        }
        __nv_bfloat16* drow = pool + (((int64_t)l * P + dp) * page * Hkv + r) * (int64_t)D;
        uint4 va, vb;
        const __nv_bfloat16* vrow = nullptr;
        if constexpr (WITH_V) {
            // V: the same two 16-byte chunks of the V row, copied as they are
            vrow = v_src + (srow - k_src);
            va = __ldcs(reinterpret_cast<const uint4*>(vrow + 8 * ca));
            vb = __ldcs(reinterpret_cast<const uint4*>(vrow + 8 * cb));
        }
        float xa[8], xb[8];
        unpack8(wa, xa);
        unpack8(wb, xb);
        const float4* cst = cs + t * qrow;
        if (style == KVSEL_ROPE_NEOX)
            turn_chunks<true>(xa, xb, cst, 8 * cp, 0, 0, srow, ca, cb, tlodf, thidf, half, p0 + t, false);
        else
            turn_chunks<false>(xa, xb, cst, 0, 4 * ca, 4 * cb, srow, ca, cb, tlodf, thidf, half, p0 + t, false);
        __stcs(reinterpret_cast<uint4*>(drow + 8 * ca), pack8(xa));
        __stcs(reinterpret_cast<uint4*>(drow + 8 * cb), pack8(xb));
        if constexpr (WITH_V) {
            __nv_bfloat16* vdst = v_pool + (drow - pool);
            __stcs(reinterpret_cast<uint4*>(vdst + 8 * ca), va);
            __stcs(reinterpret_cast<uint4*>(vdst + 8 * cb), vb);
        }
        if (!more) break;
        l = ln;
        r = rn;
        t = tn;
        g = gn;
        srow = snext;
        wa = na;
        wb = nb;
    }
}

// In-place move of retained blocks: every row of page pages[i] is turned by
// shifts[i] positions (negative: backwards), one rounding to bf16.  Grid: one
// CTA per (entry, group of kLayerGroup layers); the D/2 (cos, sin) pairs of the
// shift are computed once per CTA.
__global__ void __launch_bounds__(256, KVSEL_REROPE_MINB) shift_kernel(__nv_bfloat16* __restrict__ pool, int P,
                                                    const int32_t* __restrict__ pages,
                                                    const int32_t* __restrict__ shifts, const int32_t* n_dev, int L,
                                                    int Hkv, int D, int page, const float2* tlo, const float2* thi,
                                                    const float4* tlodf, const float4* thidf, int style,
                                                    unsigned* dev_err) {
    __shared__ float4 cs[16 * kQuadsPerGroup];  // one table row (D <= 256)
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
        cs_put(cs, idx, c.x, sh < 0 ? -c.y : c.y);  // a backward turn negates the sine
    }
    __syncthreads();
    const int PR = D >> 4;
    // as in rerope_kernel: a thread keeps one chunk pair of rows r0, r0 + dr, ...
    // of every layer and loads its next row before it turns the current one
    const int rows = page * Hkv;
    const int cp = threadIdx.x & (PR - 1), r0 = threadIdx.x / PR;
    if (r0 >= rows) return;  // no barrier follows
    const int dr = blockDim.x / PR;
    const int ca = cp, cb = cp + PR;
    auto row_of = [&](int l, int r) { return pool + (((int64_t)l * P + pg) * page * Hkv + r) * (int64_t)D; };
    int l = l0, r = r0;
    __nv_bfloat16* row = row_of(l, r);
    uint4 wa = *reinterpret_cast<const uint4*>(row + 8 * ca);
    uint4 wb = *reinterpret_cast<const uint4*>(row + 8 * cb);
    for (;;) {
        int ln = l, rn = r + dr;
        if (rn >= rows) {
            ++ln;
            rn = r0;
        }
        const bool more = ln < l1;
        __nv_bfloat16* rnext = more ? row_of(ln, rn) : row;
        uint4 na = make_uint4(0, 0, 0, 0), nb = na;
        if (more) {
            na = *reinterpret_cast<const uint4*>(rnext + 8 * ca);
            nb = *reinterpret_cast<const uint4*>(rnext + 8 * cb);
        }
        float xa[8], xb[8];
        unpack8(wa, xa);
        unpack8(wb, xb);
        if (style == KVSEL_ROPE_NEOX)
            turn_chunks<true>(xa, xb, cs, 8 * cp, 0, 0, row, ca, cb, tlodf, thidf, half, mag, sh < 0);
        else
            turn_chunks<false>(xa, xb, cs, 0, 4 * ca, 4 * cb, row, ca, cb, tlodf, thidf, half, mag, sh < 0);
        *reinterpret_cast<uint4*>(row + 8 * ca) = pack8(xa);
        *reinterpret_cast<uint4*>(row + 8 * cb) = pack8(xb);
        if (!more) break;
        l = ln;
        r = rn;
        row = rnext;
        wa = na;
        wb = nb;
    }
}

}  // namespace

cudaError_t launch_rope_tables(float2* lo, float2* hi, float4* lodf, float4* hidf, int D, double base,
                               cudaStream_t s) {
    const int64_t total = (int64_t)(KVSEL_ROPE_LO + KVSEL_ROPE_HI) * (D / 2);
    int grid = (int)((total + 255) / 256);
    if (grid > 8192) grid = 8192;
    rope_tables_kernel<<<grid, 256, 0, s>>>(lo, hi, lodf, hidf, D, base);
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
    const size_t smem = sizeof(float4) * (size_t)page * (D / 16) * kQuadsPerGroup;
    auto kern = v_src ? rerope_kernel<true> : rerope_kernel<false>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<grid, 256, smem, s>>>(static_cast<const __nv_bfloat16*>(k_src), sls, shs, src_tokens, src_block, dst_page,
                                 dst_pos0, n_dev, L, Hkv, D, page, tab->lo, tab->hi, tab->lodf, tab->hidf, rope_style,
                                 static_cast<__nv_bfloat16*>(pool), static_cast<const __nv_bfloat16*>(v_src),
                                 static_cast<__nv_bfloat16*>(v_pool), P, dev_err);
    return cudaGetLastError();
}

cudaError_t launch_shift(void* pool, int P, const int32_t* pages, const int32_t* shifts, int n, const int32_t* n_dev,
                         int L, int Hkv, int D, int page, const kvsel_ctx::RopeTab* tab, int rope_style,
                         unsigned* dev_err, cudaStream_t s) {
    const dim3 grid((unsigned)n, (unsigned)((L + kLayerGroup - 1) / kLayerGroup));
    shift_kernel<<<grid, 256, 0, s>>>(static_cast<__nv_bfloat16*>(pool), P, pages, shifts, n_dev, L, Hkv, D, page,
                                      tab->lo, tab->hi, tab->lodf, tab->hidf, rope_style, dev_err);
    return cudaGetLastError();
}

/*
 * kvsel oracle: a plain, slow, single-threaded fp64 CPU statement of what the
 * retention scoring / selection path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the package smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library: every conversion (bf16 <-> double), every rotation and every
 * reduction below is written out here on its own.
 *
 * Sources (titles and sections of the pages this restates):
 *   IntentKV  = "IntentKV: cross-turn intent-aware KV cache pruning for agent
 *               reasoning", Sec. 3.1 (Eq. 1) and
 *               Sec. 3.2 (Eq. 2, Eq. 3, Eq. 4), abstract (dead-slot redirect).
 *   KVMEM     = "KVMEM: virtualising million-token agent workspaces onto one
 *               laptop GPU", section "design and trade-offs: step-level
 *               attention trigger and Mean-K model-native retrieval"
 *               (Mean-K index, block score R_b, sink/recent/top selection) and
 *               section "engineering: tiered movement, page-table aliasing and
 *               position-consistent rebuild" (re-RoPE from raw K).
 *
 * Readings taken where the pages are silent are stated next to the code that
 * takes them.  Precision: every arithmetic step is fp64; bf16 inputs are
 * widened exactly; bf16 outputs are rounded once, to nearest-even, from the
 * fp64 result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

#define ORC_ROPE_NEOX 0        /* pairs (i, i + D/2), rotate-half          */
#define ORC_ROPE_INTERLEAVED 1 /* pairs (2i, 2i + 1)                        */

/* ------------------------------------------------------------------------ */
/* element conversion                                                        */
/* ------------------------------------------------------------------------ */

/* A bf16 value is the upper 16 bits of an IEEE binary32; widening is exact. */
static double orc_bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double orc_load(const void* base, int dtype, int64_t i) {
    if (dtype == ORC_F32) return (double)((const float*)base)[i];
    return orc_bf16_to_double(((const uint16_t*)base)[i]);
}

/*
 * Round a double to the nearest bf16 (ties to even), in one step.
 * bf16 keeps 8 significant bits and the binary32 exponent range, so the
 * spacing of representable values around x is 2^(E-7) with E the binary
 * exponent of x (clamped to -126 for subnormals).  x / spacing is exact in
 * double, rint() rounds it half-to-even, and the product is exact again.
 */
uint16_t orc_double_to_bf16(double x) {
    if (isnan(x)) return (uint16_t)0x7fc0;
    double ax = fabs(x);
    double r;
    if (ax == 0.0 || isinf(x)) {
        r = x;
    } else {
        int e;
        frexp(ax, &e);            /* ax = m * 2^e, m in [0.5, 1)  */
        int E = e - 1;            /* ax = 1.f * 2^E               */
        if (E < -126) E = -126;   /* subnormal spacing            */
        double q = ldexp(1.0, E - 7);
        r = rint(x / q) * q;
        /* largest finite bf16 is (2 - 2^-7) * 2^127 */
        if (fabs(r) > ldexp(2.0 - ldexp(1.0, -7), 127)) r = copysign(INFINITY, x);
    }
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

double orc_bf16_bits_to_double(uint16_t b) { return orc_bf16_to_double(b); }

/* ------------------------------------------------------------------------ */
/* RoPE (rotary position embedding)                                           */
/* ------------------------------------------------------------------------ */

/*
 * Rotate the D-vector x in place by position pos: pair (a, b) of frequency
 * index i turns by the angle pos * theta_i, theta_i = base^(-2i/D).
 * inverse != 0 turns by -pos * theta_i (removes the embedding).
 * NeoX pairing (a, b) = (i, i + D/2); interleaved pairing (2i, 2i + 1).
 *   x_a' = x_a cos - x_b sin,  x_b' = x_b cos + x_a sin.
 */
void orc_rope_rotate(double* x, int D, double pos, double base, int style, int inverse) {
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double theta = pow(base, -2.0 * (double)i / (double)D);
        double ang = pos * theta;
        if (inverse) ang = -ang;
        double c = cos(ang), s = sin(ang);
        int a = (style == ORC_ROPE_NEOX) ? i : 2 * i;
        int b = (style == ORC_ROPE_NEOX) ? i + half : 2 * i + 1;
        double xa = x[a], xb = x[b];
        x[a] = xa * c - xb * s;
        x[b] = xb * c + xa * s;
    }
}

/* ------------------------------------------------------------------------ */
/* IntentKV Eq. 2: QueryMemory                                               */
/* ------------------------------------------------------------------------ */

/*
 * One QueryMemory update for one turn (IntentKV Sec. 3.2, Eq. 2).
 *   E[l,h,:]  = (1/R) sum_r Q[l,h,r,:]      Enc(): mean of the actionable
 *                                           span's post-RoPE query rows
 *   norm_mode 0 (default; the page normalises M_t per head after every
 *   update, so the normalised state is what decays next turn):
 *               U = e^-lambda * M + E;  M <- U / ||U||
 *   norm_mode 1 (alternative reading): the raw geometric sum is carried,
 *               A <- e^-lambda * A + E;  M <- A / ||A||
 * first_turn != 0 takes the previous state as zero (M_0 = 0).
 * A zero vector U (or A) gives M = 0 for that (l,h).
 * q: [L][Hq][R][D] (f32 or bf16), M: [L][Hq][D], A: [L][Hq][D] (mode 1 only).
 */
void orc_memory_update(const void* q, int dtype, int L, int Hq, int R, int D,
                       double lambda, int first_turn, int norm_mode,
                       double* M, double* A) {
    double decay = exp(-lambda);
    double* E = (double*)malloc(sizeof(double) * (size_t)D);
    double* U = (double*)malloc(sizeof(double) * (size_t)D);
    for (int l = 0; l < L; ++l) {
        for (int h = 0; h < Hq; ++h) {
            int64_t head = (int64_t)l * Hq + h;
            for (int d = 0; d < D; ++d) E[d] = 0.0;
            for (int r = 0; r < R; ++r)
                for (int d = 0; d < D; ++d)
                    E[d] += orc_load(q, dtype, (head * R + r) * D + d);
            for (int d = 0; d < D; ++d) E[d] /= (double)R;

            double* state = (norm_mode == 0) ? (M + head * D) : (A + head * D);
            for (int d = 0; d < D; ++d)
                U[d] = (first_turn ? 0.0 : decay * state[d]) + E[d];
            if (norm_mode != 0)
                for (int d = 0; d < D; ++d) state[d] = U[d];

            double nrm2 = 0.0;
            for (int d = 0; d < D; ++d) nrm2 += U[d] * U[d];
            double nrm = sqrt(nrm2);
            for (int d = 0; d < D; ++d) M[head * D + d] = (nrm > 0.0) ? U[d] / nrm : 0.0;
        }
    }
    free(E);
    free(U);
}

/* ------------------------------------------------------------------------ */
/* IntentKV Eq. 3-4: rule scores                                             */
/* ------------------------------------------------------------------------ */

/* F = [0, pi) U [q_s, q_e)  (IntentKV Sec. 3.1) */
static int orc_forced(int j, int pi, int q_s, int q_e) {
    return (j < pi) || (j >= q_s && j < q_e);
}

/*
 * rule_j = sum_{l,h} a_{l,h,j},  a_{l,h,j} = softmax over i in H of
 * M[l,h] . K[l,g(h),i] / sqrt(D)      (IntentKV Eq. 3, Eq. 4)
 * GQA expansion: g(h) = floor(h / (Hq/Hkv)) (contiguous grouping; the page
 * says only that KV heads are expanded to Hq heads).
 * K row of token j, kv head g, layer l starts at element
 *   l*layer_stride + slot(j)*slot_stride + g*D,   slot(j) = slot_map[j] or j.
 * Candidates H = [0,N) \ F.  Positions in F get rule 0 and enter no
 * denominator (Eq. 4 sums over i in H only).  H empty -> rule == 0.
 */
void orc_rule_scores(const void* k_pool, int dtype, const int32_t* slot_map,
                     int L, int Hq, int Hkv, int N, int D,
                     int64_t layer_stride, int64_t slot_stride,
                     const double* M, int pi, int q_s, int q_e, double* rule) {
    int G = Hq / Hkv;
    double inv_sqrt_d = 1.0 / sqrt((double)D);
    double* z = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int j = 0; j < N; ++j) rule[j] = 0.0;
    for (int l = 0; l < L; ++l) {
        for (int h = 0; h < Hq; ++h) {
            int g = h / G;
            const double* m = M + ((int64_t)l * Hq + h) * D;
            double zmax = -INFINITY;
            int any = 0;
            for (int j = 0; j < N; ++j) {
                if (orc_forced(j, pi, q_s, q_e)) continue;
                int64_t slot = slot_map ? (int64_t)slot_map[j] : (int64_t)j;
                int64_t base = (int64_t)l * layer_stride + slot * slot_stride + (int64_t)g * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += m[d] * orc_load(k_pool, dtype, base + d);
                z[j] = dot * inv_sqrt_d;
                if (z[j] > zmax) zmax = z[j];
                any = 1;
            }
            if (!any) continue;
            double denom = 0.0;
            for (int j = 0; j < N; ++j)
                if (!orc_forced(j, pi, q_s, q_e)) denom += exp(z[j] - zmax);
            for (int j = 0; j < N; ++j)
                if (!orc_forced(j, pi, q_s, q_e)) rule[j] += exp(z[j] - zmax) / denom;
        }
    }
    free(z);
}

/* ------------------------------------------------------------------------ */
/* IntentKV Eq. 1: budgeted top-k with a forced set                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    double s;
    int j;
} orc_scored;

/* Order (-score, index): larger score first; equal scores keep the lower
 * index first (the page does not say; the reading is a stable tie-break).
 * A NaN score ranks below every number; -0 and +0 are equal. */
static int orc_cmp_scored(const void* pa, const void* pb) {
    const orc_scored* a = (const orc_scored*)pa;
    const orc_scored* b = (const orc_scored*)pb;
    int na = isnan(a->s), nb = isnan(b->s);
    if (na != nb) return na ? 1 : -1;
    if (!na) {
        if (a->s > b->s) return -1;
        if (a->s < b->s) return 1;
    }
    return (a->j < b->j) ? -1 : (a->j > b->j);
}

/*
 * K* = F U argtop_{C*} s_j over H,  C* = max(0, C - |F|)   (IntentKV Eq. 1)
 * keep[j] = 1 for kept positions; keep_idx (if not NULL) lists them in
 * ascending order; returns |K*| = |F| + min(C*, |H|).
 */
int orc_topk_retain(const double* score, int N, int pi, int q_s, int q_e, int C,
                    uint8_t* keep, int32_t* keep_idx) {
    int nF = 0;
    for (int j = 0; j < N; ++j) nF += orc_forced(j, pi, q_s, q_e);
    int cstar = C - nF;
    if (cstar < 0) cstar = 0;
    orc_scored* cand = (orc_scored*)malloc(sizeof(orc_scored) * (size_t)(N > 0 ? N : 1));
    int nH = 0;
    for (int j = 0; j < N; ++j) {
        keep[j] = (uint8_t)orc_forced(j, pi, q_s, q_e);
        if (!keep[j]) {
            cand[nH].s = score[j];
            cand[nH].j = j;
            ++nH;
        }
    }
    qsort(cand, (size_t)nH, sizeof(orc_scored), orc_cmp_scored);
    int take = cstar < nH ? cstar : nH;
    for (int t = 0; t < take; ++t) keep[cand[t].j] = 1;
    free(cand);
    int n = 0;
    for (int j = 0; j < N; ++j)
        if (keep[j]) {
            if (keep_idx) keep_idx[n] = j;
            ++n;
        }
    return n;
}

/* ------------------------------------------------------------------------ */
/* IntentKV layout layer: dead-slot redirect                                 */
/* ------------------------------------------------------------------------ */

/* Dropped positions are routed to the sentinel dead slot; kept positions keep
 * their slot (surviving rows never move). */
void orc_redirect_slots(const int32_t* slot_in, const uint8_t* keep, int N,
                        int32_t dead_slot, int32_t* slot_out) {
    for (int j = 0; j < N; ++j) slot_out[j] = keep[j] ? slot_in[j] : dead_slot;
}

/* ------------------------------------------------------------------------ */
/* KVMEM: Mean-K index                                                       */
/* ------------------------------------------------------------------------ */

/*
 * kbar[l,g,b,:] = mean over the tokens i of block b of Ktilde[l,g,i,:]
 * Ktilde is the position-free K: k_src itself, or, when src_pos is given, k_src
 * with the rotation of position src_pos[i] removed.  Block b of k_src covers
 * tokens [b*block, min((b+1)*block, T)) (a short last block is averaged over the
 * tokens it has) and lands in index block first_block + b.
 * k_src: bf16 [L][Hkv][T][D]; index: bf16 [L][Hkv][Bcap][D];
 * mean_out (optional): the fp64 means before rounding, [L][Hkv][n_blocks][D].
 */
void orc_meank_build(const uint16_t* k_src, int L, int Hkv, int T, int D, int block,
                     int first_block, const int32_t* src_pos, double rope_base,
                     int rope_style, uint16_t* index, int Bcap, double* mean_out) {
    int n_blocks = (T + block - 1) / block;
    double* row = (double*)malloc(sizeof(double) * (size_t)D);
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
    for (int l = 0; l < L; ++l)
        for (int g = 0; g < Hkv; ++g)
            for (int b = 0; b < n_blocks; ++b) {
                int t0 = b * block;
                int t1 = t0 + block < T ? t0 + block : T;
                for (int d = 0; d < D; ++d) acc[d] = 0.0;
                for (int t = t0; t < t1; ++t) {
                    int64_t base = (((int64_t)l * Hkv + g) * T + t) * D;
                    for (int d = 0; d < D; ++d) row[d] = orc_bf16_to_double(k_src[base + d]);
                    if (src_pos) orc_rope_rotate(row, D, (double)src_pos[t], rope_base, rope_style, 1);
                    for (int d = 0; d < D; ++d) acc[d] += row[d];
                }
                int64_t ob = (((int64_t)l * Hkv + g) * Bcap + (first_block + b)) * D;
                for (int d = 0; d < D; ++d) {
                    double mean = acc[d] / (double)(t1 - t0);
                    index[ob + d] = orc_double_to_bf16(mean);
                    if (mean_out) mean_out[(((int64_t)l * Hkv + g) * n_blocks + b) * D + d] = mean;
                }
            }
    free(row);
    free(acc);
}

/* ------------------------------------------------------------------------ */
/* KVMEM: block relevance R_b                                                */
/* ------------------------------------------------------------------------ */

/*
 * Unnormalised block mass of one (layer l, kv head g):
 *   part[b] = sum_{h in group g} sum_m softmax_{b' in C}( q[l,h,m] . kbar[l,g,b'] / sqrt(D) )_b
 * for b in the candidate set C = [n_sink, n_blocks - n_recent); part[b] = 0
 * outside C.  q: bf16 [L][Hq][M][D] (position-free queries); index: bf16
 * [L][Hkv][Bcap][D]; part: [n_blocks].
 */
void orc_block_mass(const uint16_t* q, const uint16_t* index, int L, int Hq, int Hkv,
                    int M, int D, int n_blocks, int Bcap, int n_sink, int n_recent,
                    int l, int g, double* part) {
    (void)L;
    int G = Hq / Hkv;
    int c0 = n_sink, c1 = n_blocks - n_recent;
    double inv_sqrt_d = 1.0 / sqrt((double)D);
    for (int b = 0; b < n_blocks; ++b) part[b] = 0.0;
    if (c1 <= c0) return;
    double* s = (double*)malloc(sizeof(double) * (size_t)n_blocks);
    double* qrow = (double*)malloc(sizeof(double) * (size_t)D);
    for (int h = g * G; h < (g + 1) * G; ++h) {
        for (int m = 0; m < M; ++m) {
            int64_t qb = (((int64_t)l * Hq + h) * M + m) * D;
            for (int d = 0; d < D; ++d) qrow[d] = orc_bf16_to_double(q[qb + d]);
            double smax = -INFINITY;
            for (int b = c0; b < c1; ++b) {
                int64_t kb = (((int64_t)l * Hkv + g) * Bcap + b) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += qrow[d] * orc_bf16_to_double(index[kb + d]);
                s[b] = dot * inv_sqrt_d;
                if (s[b] > smax) smax = s[b];
            }
            double denom = 0.0;
            for (int b = c0; b < c1; ++b) denom += exp(s[b] - smax);
            for (int b = c0; b < c1; ++b) part[b] += exp(s[b] - smax) / denom;
        }
    }
    free(s);
    free(qrow);
}

/*
 * R_b = (1 / (L*Hq)) sum_{l,h} sum_m p_{l,h,m,b}: the per-(l,h,m) softmax over
 * candidate blocks, summed over query tokens and averaged over all layer-heads
 * (KVMEM retrieval).  part_out (optional) receives every (l,g) mass row,
 * [L*Hkv][n_blocks]; the (l,g) rows are summed in ascending (l,g) order.
 */
void orc_block_scores(const uint16_t* q, const uint16_t* index, int L, int Hq, int Hkv,
                      int M, int D, int n_blocks, int Bcap, int n_sink, int n_recent,
                      double* R, double* part_out) {
    double* part = (double*)malloc(sizeof(double) * (size_t)(n_blocks > 0 ? n_blocks : 1));
    for (int b = 0; b < n_blocks; ++b) R[b] = 0.0;
    for (int l = 0; l < L; ++l)
        for (int g = 0; g < Hkv; ++g) {
            orc_block_mass(q, index, L, Hq, Hkv, M, D, n_blocks, Bcap, n_sink, n_recent, l, g, part);
            for (int b = 0; b < n_blocks; ++b) R[b] += part[b];
            if (part_out)
                memcpy(part_out + ((int64_t)l * Hkv + g) * n_blocks, part, sizeof(double) * (size_t)n_blocks);
        }
    for (int b = 0; b < n_blocks; ++b) R[b] /= (double)L * (double)Hq;
    free(part);
}

/* ------------------------------------------------------------------------ */
/* KVMEM: working-set selection                                              */
/* ------------------------------------------------------------------------ */

/*
 * W = [0, n_sink) U [n_blocks - n_recent, n_blocks) U top-k of R over the
 * candidates, ties to the lower block id; ids ascending.  Returns |W|.
 * This is Eq. 1's selection with the sink and recent blocks as forced set.
 */
int orc_select_blocks(const double* R, int n_blocks, int n_sink, int n_recent, int k,
                      int32_t* ids) {
    uint8_t* keep = (uint8_t*)malloc((size_t)(n_blocks > 0 ? n_blocks : 1));
    int n_forced = 0;
    for (int b = 0; b < n_blocks; ++b)
        n_forced += (b < n_sink) || (b >= n_blocks - n_recent);
    int n = orc_topk_retain(R, n_blocks, n_sink, n_blocks - n_recent, n_blocks, n_forced + k, keep, ids);
    free(keep);
    return n;
}

/* ------------------------------------------------------------------------ */
/* KVMEM: position-consistent restore (re-RoPE scatter)                       */
/* ------------------------------------------------------------------------ */

/*
 * For entry i and token t < page: the raw (position-free) row
 *   k_src[l*src_layer_stride + g*src_head_stride + (src_block[i]*page + t)*D + :]
 * is rotated to its new compact position dst_pos0[i] + t and written to
 *   pool[l][dst_page[i]][t][g][:]      (pool: bf16 [L][P][page][Hkv][D]).
 * Other pool pages are left untouched.
 */
void orc_rerope_scatter(const uint16_t* k_src, int64_t src_layer_stride, int64_t src_head_stride,
                        const int32_t* src_block, const int32_t* dst_page, const int32_t* dst_pos0,
                        int n, int L, int Hkv, int D, int page, double rope_base, int rope_style,
                        uint16_t* pool, int P) {
    double* row = (double*)malloc(sizeof(double) * (size_t)D);
    for (int i = 0; i < n; ++i)
        for (int l = 0; l < L; ++l)
            for (int t = 0; t < page; ++t)
                for (int g = 0; g < Hkv; ++g) {
                    int64_t sb = (int64_t)l * src_layer_stride + (int64_t)g * src_head_stride +
                                 ((int64_t)src_block[i] * page + t) * D;
                    for (int d = 0; d < D; ++d) row[d] = orc_bf16_to_double(k_src[sb + d]);
                    orc_rope_rotate(row, D, (double)(dst_pos0[i] + t), rope_base, rope_style, 0);
                    int64_t ob = ((((int64_t)l * P + dst_page[i]) * page + t) * Hkv + g) * D;
                    for (int d = 0; d < D; ++d) pool[ob + d] = orc_double_to_bf16(row[d]);
                }
    free(row);
}

/* ------------------------------------------------------------------------ */
/* KVMEM: differential working-set update                                    */
/* ------------------------------------------------------------------------ */

/*
 * KVMEM, section "engineering: tiered movement, page-table aliasing and
 * position-consistent rebuild": only blocks that are selected now (W_t) but
 * not resident in the GPU page pool (G_{t-1}) are moved in; the retained /
 * incoming / outgoing split follows the same set difference.
 *
 * Readings (the pages give no formula for the split or the page choice):
 *  - G_{t-1} is the previous working set: prev_ids[n_prev] ascending, block
 *    prev_ids[r] held in page prev_pages[r] at compact position r * page.
 *  - retained = W_t n G_{t-1} keep their page; incoming = W_t \ G_{t-1} take
 *    the free pages of the pool [0, P) -- every page not held by a retained
 *    block -- in ascending page order, incoming blocks in ascending block id;
 *    outgoing = G_{t-1} \ W_t release their pages.
 *  - the new working set new_ids[n_new] is ascending; block new_ids[r] sits at
 *    compact position r * page, so a retained block whose rank moved from r'
 *    to r must be turned by shift = (r - r') * page positions.
 * Outputs: new_pages[r]; shift[r] (0 for incoming); in_rank / in_page: the
 * incoming ranks ascending and their pages; mv_rank / mv_shift: retained ranks
 * with a non-zero shift; out_page: the released pages, ascending by block id;
 * counts[0..2] = (n_incoming, n_moved, n_outgoing).  Returns 0, or -1 when the
 * pool has too few free pages.
 */
int orc_workset_diff(const int32_t* prev_ids, const int32_t* prev_pages, int n_prev, const int32_t* new_ids,
                     int n_new, int P, int page, int32_t* new_pages, int32_t* shift, int32_t* in_rank,
                     int32_t* in_page, int32_t* mv_rank, int32_t* mv_shift, int32_t* out_page, int32_t* counts) {
    uint8_t* held = (uint8_t*)calloc((size_t)(P > 0 ? P : 1), 1);
    int n_in = 0, n_mv = 0, n_out = 0;
    /* retained entries: linear search of the previous set */
    for (int r = 0; r < n_new; ++r) {
        int found = -1;
        for (int q = 0; q < n_prev; ++q)
            if (prev_ids[q] == new_ids[r]) found = q;
        if (found >= 0) {
            new_pages[r] = prev_pages[found];
            shift[r] = (r - found) * page;
            held[prev_pages[found]] = 1;
            if (shift[r] != 0) {
                mv_rank[n_mv] = r;
                mv_shift[n_mv] = shift[r];
                ++n_mv;
            }
        } else {
            new_pages[r] = -1;
            shift[r] = 0;
        }
    }
    /* incoming entries take the free pages in ascending order */
    int next_free = 0;
    for (int r = 0; r < n_new; ++r) {
        if (new_pages[r] >= 0) continue;
        while (next_free < P && held[next_free]) ++next_free;
        if (next_free >= P) {
            free(held);
            return -1;
        }
        new_pages[r] = next_free;
        held[next_free] = 1;
        in_rank[n_in] = r;
        in_page[n_in] = next_free;
        ++n_in;
    }
    /* outgoing entries: previous blocks absent from the new set */
    for (int q = 0; q < n_prev; ++q) {
        int kept = 0;
        for (int r = 0; r < n_new; ++r)
            if (new_ids[r] == prev_ids[q]) kept = 1;
        if (!kept) out_page[n_out++] = prev_pages[q];
    }
    counts[0] = n_in;
    counts[1] = n_mv;
    counts[2] = n_out;
    free(held);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* KVMEM: restore of incoming blocks (re-RoPE'd K, copied V)                  */
/* ------------------------------------------------------------------------ */

/*
 * KVMEM, same section: K is rebuilt from the position-free raw K at the new
 * compact position; V carries no position and is copied as it is.  K is
 * exactly orc_rerope_scatter's output; for entry i and token t < page the V
 * row v_src[l*v_layer_stride + g*v_head_stride + (src_block[i]*page + t)*D + :]
 * is copied bit for bit to v_pool[l][dst_page[i]][t][g][:].
 */
void orc_restore_blocks(const uint16_t* k_src, const uint16_t* v_src, int64_t src_layer_stride,
                        int64_t src_head_stride, const int32_t* src_block, const int32_t* dst_page,
                        const int32_t* dst_pos0, int n, int L, int Hkv, int D, int page, double rope_base,
                        int rope_style, uint16_t* k_pool, uint16_t* v_pool, int P) {
    orc_rerope_scatter(k_src, src_layer_stride, src_head_stride, src_block, dst_page, dst_pos0, n, L, Hkv, D, page,
                       rope_base, rope_style, k_pool, P);
    for (int i = 0; i < n; ++i)
        for (int l = 0; l < L; ++l)
            for (int t = 0; t < page; ++t)
                for (int g = 0; g < Hkv; ++g) {
                    int64_t sb = (int64_t)l * src_layer_stride + (int64_t)g * src_head_stride +
                                 ((int64_t)src_block[i] * page + t) * D;
                    int64_t ob = ((((int64_t)l * P + dst_page[i]) * page + t) * Hkv + g) * D;
                    for (int d = 0; d < D; ++d) v_pool[ob + d] = v_src[sb + d];
                }
}

/* ------------------------------------------------------------------------ */
/* KVMEM: moving a retained block to its new compact position                */
/* ------------------------------------------------------------------------ */

/*
 * A retained block keeps its page (page-table aliasing) but its compact
 * position moves by shift[i] positions.  RoPE rotations by angles a and b
 * compose to the rotation by a + b, so the stored K (rotated to its old
 * position) is turned by shift[i] more positions in place: every row of
 * pool[l][pages[i]][t][g][:] becomes bf16(R(shift[i]) * row), one rounding.
 * A negative shift turns backwards.
 */
void orc_rerope_shift(uint16_t* pool, int P, const int32_t* pages, const int32_t* shifts, int n, int L, int Hkv,
                      int D, int page, double rope_base, int rope_style) {
    double* row = (double*)malloc(sizeof(double) * (size_t)D);
    for (int i = 0; i < n; ++i)
        for (int l = 0; l < L; ++l)
            for (int t = 0; t < page; ++t)
                for (int g = 0; g < Hkv; ++g) {
                    int64_t ob = ((((int64_t)l * P + pages[i]) * page + t) * Hkv + g) * D;
                    for (int d = 0; d < D; ++d) row[d] = orc_bf16_to_double(pool[ob + d]);
                    orc_rope_rotate(row, D, (double)shifts[i], rope_base, rope_style, 0);
                    for (int d = 0; d < D; ++d) pool[ob + d] = orc_double_to_bf16(row[d]);
                }
    free(row);
}

/* ------------------------------------------------------------------------ */
/* SideQuest: cursor-span eviction as a keep mask                            */
/* ------------------------------------------------------------------------ */

/*
 * "SideQuest" page, method overview and Figure 1: the auxiliary thread names
 * the cursors to delete ({del_cursors: [ids]}); the main thread then clears
 * those cursors' KV entries.  Cursor c spans positions [span_start[c],
 * span_end[c]) (readings: half-open spans, clipped to [0, N); spans may
 * overlap).  The result ANDs into an existing keep mask (keep_in, or all ones
 * when keep_in is NULL), so it composes with a retention policy and feeds the
 * dead-slot redirect:
 *   keep_out[j] = keep_in[j] && j lies in no span of a listed cursor.
 * Returns the number of listed ids outside [0, n_cursors) (they are ignored).
 */
int orc_span_keep(const int32_t* span_start, const int32_t* span_end, int n_cursors, const int32_t* del_ids,
                  int n_del, const uint8_t* keep_in, int N, uint8_t* keep_out) {
    int bad = 0;
    for (int j = 0; j < N; ++j) keep_out[j] = keep_in ? (keep_in[j] != 0) : 1;
    for (int d = 0; d < n_del; ++d) {
        int c = del_ids[d];
        if (c < 0 || c >= n_cursors) {
            ++bad;
            continue;
        }
        for (int j = span_start[c]; j < span_end[c]; ++j)
            if (j >= 0 && j < N) keep_out[j] = 0;
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* FP8 storage of the Mean-K index                                          */
/* ------------------------------------------------------------------------ */

/*
 * KVMEM page, section "design and trade-offs" (the per-block index and its
 * size: 9.5 GiB of index for a 10M-token workspace) and the server
 * experiments, which keep the KV cache in FP8.  Reading: an index row (one
 * Mean-K vector of D values for one (layer, kv head, block)) is stored as D
 * E4M3 codes and one power-of-two scale 2^e, the value being code * 2^e.
 *
 * E4M3, the OCP 8-bit floating-point format: a sign bit, 4 exponent bits with
 * bias 7 and 3 mantissa bits.  Exponent field 0 holds the subnormals m * 2^-9;
 * fields 1..15 hold (1 + m/8) * 2^(E-7), except E = 15, m = 7, which is NaN.
 * There is no infinity; the largest finite value is 1.75 * 2^8 = 448.
 */
double orc_e4m3_decode(unsigned code) {
    const unsigned E = (code >> 3) & 15u, m = code & 7u;
    if (E == 15u && m == 7u) return NAN;
    const double mag = E == 0 ? ldexp((double)m, -9) : ldexp((double)(8u + m), (int)E - 10);
    return (code & 0x80u) ? -mag : mag;
}

/* Nearest E4M3 value to y, ties to the even code (an even last mantissa bit);
 * |y| must not exceed 448.  The sign is kept, also for results of zero. */
unsigned orc_e4m3_encode(double y) {
    const unsigned sign = signbit(y) ? 0x80u : 0u;
    const double a = fabs(y);
    unsigned code;
    if (a < ldexp(1.0, -6)) {
        /* subnormal spacing 2^-9; k = 8 is the smallest normal, code 0x08 */
        code = (unsigned)nearbyint(a / ldexp(1.0, -9));
    } else {
        int ex;
        frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1): 2^(ex-1) <= a < 2^ex */
        int E = ex - 1;
        unsigned k = (unsigned)nearbyint(a / ldexp(1.0, E - 3)); /* 8 .. 16 */
        if (k == 16u) {
            k = 8u;
            ++E;
        }
        code = ((unsigned)(E + 7) << 3) | (k - 8u);
    }
    return sign | code;
}

/* Scale exponent of a row: the smallest e >= -100 with max|x| <= 448 * 2^e
 * (an all-zero row gets -100).  448 = 0.875 * 2^9. */
int orc_fp8_row_exp(const double* x, int D) {
    double mx = 0.0;
    for (int i = 0; i < D; ++i) mx = fmax(mx, fabs(x[i]));
    if (mx == 0.0) return -100;
    int ex;
    const double f = frexp(mx, &ex);
    const int e = f <= 0.875 ? ex - 9 : ex - 8;
    return e < -100 ? -100 : e;
}

void orc_index_to_fp8(const uint16_t* idx, int64_t rows, int D, uint8_t* codes, int8_t* exps) {
    double* x = (double*)malloc(sizeof(double) * (size_t)D);
    for (int64_t r = 0; r < rows; ++r) {
        for (int i = 0; i < D; ++i) x[i] = orc_bf16_bits_to_double(idx[r * D + i]);
        const int e = orc_fp8_row_exp(x, D);
        exps[r] = (int8_t)e;
        for (int i = 0; i < D; ++i) codes[r * D + i] = (uint8_t)orc_e4m3_encode(ldexp(x[i], -e));
    }
    free(x);
}

void orc_index_from_fp8(const uint8_t* codes, const int8_t* exps, int64_t rows, int D, uint16_t* idx) {
    for (int64_t r = 0; r < rows; ++r)
        for (int i = 0; i < D; ++i)
            idx[r * D + i] = orc_double_to_bf16(ldexp(orc_e4m3_decode(codes[r * D + i]), exps[r]));
}

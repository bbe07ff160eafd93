/*
 * kvsel.h: C ABI of libkvsel, query-driven KV-cache retention scoring and
 * selection on one NVIDIA GB300 GPU (sm_103a).
 *
 * Two methods share the library:
 *   IntentKV  ("IntentKV: cross-turn intent-aware KV cache pruning for agent
 *             reasoning"): QueryMemory (Sec. 3.2, Eq. 2), rule scores
 *             (Sec. 3.2, Eq. 3-4), budgeted top-C* retention with a forced set
 *             (Sec. 3.1, Eq. 1) and the dead-slot redirect of the layout layer
 *             (abstract; Sec. 3 overview).
 *   KVMEM     ("KVMEM: virtualising million-token agent workspaces onto one
 *             laptop GPU"): the Mean-K block index, the block relevance R_b and
 *             the sink + recent + top-R_b working set (section "design and
 *             trade-offs: step-level attention trigger and Mean-K model-native
 *             retrieval"), and the position-consistent restore that re-applies
 *             RoPE to raw K at new compact positions (section "engineering:
 *             tiered movement, page-table aliasing and position-consistent
 *             rebuild").
 *
 * Conventions shared by every call
 *   - Tensor pointers are DEVICE pointers on the context's device, owned by
 *     the caller; the library never frees or keeps them.  Arguments named
 *     *_host are host pointers.
 *   - Layouts are row-major with the innermost (head-dim) axis contiguous.
 *     bf16 tensors are passed as void* holding IEEE bfloat16 values.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and never synchronises the host.
 *   - Every call returns a kvsel_status.  Arguments are validated on the host
 *     before anything is launched; on an error nothing is launched, nothing is
 *     written, and kvsel_last_error_string() says why.  Calls never throw.
 *   - A context is not thread-safe: use one context per host thread, and do
 *     not let calls on one context overlap on different streams (they share
 *     the context's scratch workspace).
 *   - Scratch: calls that need temporary device memory take it from the
 *     context's workspace, which grows on first use at a larger size
 *     (cudaMalloc, synchronous).  Make one call at the largest size before
 *     capturing calls into a CUDA graph.
 */
#ifndef KVSEL_H_
#define KVSEL_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kvsel_ctx kvsel_ctx;

typedef enum {
    KVSEL_OK = 0,
    KVSEL_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad enum     */
    KVSEL_ERR_SHAPE = -2,       /* inconsistent sizes or ranges               */
    KVSEL_ERR_ALIGN = -3,       /* pointer or stride breaks 16-byte alignment */
    KVSEL_ERR_UNSUPPORTED = -4, /* valid but not supported (e.g. head dim)    */
    KVSEL_ERR_CUDA = -5,        /* a CUDA runtime call failed                 */
    KVSEL_ERR_TIMEOUT = -6,     /* a bounded device wait gave up              */
    KVSEL_ERR_DEVICE_CHECK = -7 /* a kernel found bad data (see below)        */
} kvsel_status;

typedef enum { KVSEL_F32 = 0, KVSEL_BF16 = 1 } kvsel_dtype;

/* RoPE pairing: NeoX / rotate-half pairs (i, i + D/2); interleaved (2i, 2i+1). */
typedef enum { KVSEL_ROPE_NEOX = 0, KVSEL_ROPE_INTERLEAVED = 1 } kvsel_rope_style;

/* How kvsel_stage_restore reaches the host repository (see there). */
typedef enum { KVSEL_STAGE_AUTO = 0, KVSEL_STAGE_PACKED = 1, KVSEL_STAGE_DIRECT = 2 } kvsel_stage_mode;

/* ------------------------------------------------------------------------ */
/* context                                                                   */
/* ------------------------------------------------------------------------ */

/* Create a context on CUDA device `device` (made current for the call). */
int kvsel_ctx_create(int device, kvsel_ctx** out);
/* Free the context's workspace and tables; waits for the device. NULL is ok. */
int kvsel_ctx_destroy(kvsel_ctx* ctx);
/* Detail of the last error on this context ("" if none); valid until the next call. */
const char* kvsel_last_error_string(const kvsel_ctx* ctx);
/* Synchronise `stream`, then read and clear the device error word that kernels
 * set when they meet bad data (a slot, block id or position out of range):
 * returns KVSEL_OK or KVSEL_ERR_DEVICE_CHECK. */
int kvsel_check_device(kvsel_ctx* ctx, void* stream);
/* Library version, major * 10000 + minor * 100 + patch. */
int kvsel_version(void);

/* ------------------------------------------------------------------------ */
/* IntentKV                                                                  */
/* ------------------------------------------------------------------------ */

/*
 * QueryMemory update for one turn (IntentKV Sec. 3.2, Eq. 2):
 *   E[l,h,:] = (1/R) sum_r q_rows[l,h,r,:]   (the actionable span's post-RoPE
 *                                             query rows; Enc = their mean)
 *   norm_mode 0: M <- normalise(e^-lambda * M + E)          (state = M)
 *   norm_mode 1: A <- e^-lambda * A + E;  M <- normalise(A) (state = A)
 * normalise() divides each (l,h) vector by its L2 norm over D; a zero vector
 * stays zero.  first_turn != 0 treats the previous state as zero.
 *   q_rows  [L][Hq][R][D], q_dtype F32 or BF16, 16-byte aligned
 *   M       [L][Hq][D] fp32, in/out (mode 0) or out (mode 1)
 *   A       [L][Hq][D] fp32 in/out, mode 1 only (NULL in mode 0)
 * Requires R >= 1, D % 8 == 0 (BF16) or D % 4 == 0 (F32), D <= 1024.
 */
int kvsel_memory_update(kvsel_ctx* ctx, const void* q_rows, int q_dtype, int L, int Hq, int R,
                        int D, float lambda, int first_turn, int norm_mode, float* M, float* A,
                        void* stream);

/*
 * Rule scores (IntentKV Sec. 3.2, Eq. 3-4):
 *   rule[j] = sum_{l<L, h<Hq} softmax_{i in H}( M[l,h] . K[l,g(h),i] / sqrt(D) )_j
 * for j in H = [0,N) \ F, F = [0,pi) U [q_s,q_e); rule[j] = 0 for j in F, and
 * no position of F enters a denominator.  g(h) = h / (Hq/Hkv).
 * K is read in place from a paged pool: the row of token j, kv head g, layer l
 * starts at element  l*layer_stride + slot(j)*slot_stride + g*D  of k_pool,
 * slot(j) = slot_map[j] (slot_map == NULL: slot(j) = j).  Rows of a slot hold
 * the Hkv heads back to back.
 *   k_pool   k_dtype F32 or BF16; base, layer_stride and slot_stride 16-byte
 *            aligned in bytes
 *   slot_map int32 [N] or NULL; slots of candidate positions must lie in
 *            [0, n_slots) (a slot outside is read as a zero row and sets the
 *            device error word, see kvsel_check_device)
 *   n_slots  rows per layer in the pool (>= N when slot_map == NULL)
 *   M        [L][Hq][D] fp32 (normalised QueryMemory)
 *   rule     [N] fp32 out
 * Requires Hq % Hkv == 0, Hq/Hkv <= 8, D in {16,32,64,128,256},
 * 0 <= pi <= N, 0 <= q_s <= q_e <= N.  Uses workspace: 4*L*Hq*N bytes + a little.
 */
int kvsel_rule_scores(kvsel_ctx* ctx, const void* k_pool, int k_dtype, const int32_t* slot_map,
                      int n_slots, int L, int Hq, int Hkv, int N, int D, int64_t layer_stride,
                      int64_t slot_stride, const float* M, int pi, int q_s, int q_e, float* rule,
                      void* stream);

/*
 * kvsel_rule_scores without any device allocation.  The pages have no
 * counterpart: this is a deployment variant for callers that cannot let a
 * library allocate device memory, such as serving engines that give nearly all
 * of the GPU to their own KV page pool and allocator, and latency-critical
 * loops that cannot take cudaFree's implicit device synchronisation.
 * Same arguments, rules and result as kvsel_rule_scores (the same kernels, so
 * bit-identical scores); the scratch it needs (4*L*Hq*N bytes plus a little)
 * comes from a fixed 64 MiB array inside the library, which every GPU that
 * loads the library holds until the process exits.  A size that needs more
 * returns KVSEL_ERR_UNSUPPORTED without launching.  The first call with a
 * context looks up the array's device address on the context's device (a
 * one-time set-up with that device current, kept in the context); make that
 * first call before any stream capture.  All calls share the one array and it
 * keeps the last call's contents (nothing in it needs clearing between calls):
 * calls that overlap on the GPU, on any stream or context of the process, race.
 */
int kvsel_rule_scores_noalloc(kvsel_ctx* ctx, const void* k_pool, int k_dtype, const int32_t* slot_map,
                              int n_slots, int L, int Hq, int Hkv, int N, int D, int64_t layer_stride,
                              int64_t slot_stride, const float* M, int pi, int q_s, int q_e,
                              float* rule, void* stream);

/*
 * Budgeted retention (IntentKV Sec. 3.1, Eq. 1):
 *   K* = F U (the C* largest scores of H),  C* = max(0, C - |F|)
 * Ties between equal scores go to the lower index; NaN ranks below every
 * number; -0 equals +0.  If N <= C every position is kept.
 *   score     [N] fp32
 *   keep      [N] uint8 out (1 = kept) or NULL
 *   keep_idx  [|K*|] int32 out, kept positions ascending, or NULL
 *   n_keep_host  host out: |K*| = |F| + min(C*, |H|) (closed form, no sync)
 * Uses no workspace for N <= 131072; above that the grid-wide selection may use
 * 4 KB + 16 bytes per 4096 positions of it.
 */
int kvsel_topk_retain(kvsel_ctx* ctx, const float* score, int N, int pi, int q_s, int q_e,
                      int C, uint8_t* keep, int32_t* keep_idx, int* n_keep_host, void* stream);

/*
 * Dead-slot redirect (IntentKV abstract; Sec. 3 overview, layout layer):
 *   slot_out[j] = keep[j] ? slot_in[j] : dead_slot
 * Kept rows never move.  slot_out may alias slot_in.  Int32 [N], uint8 [N].
 */
int kvsel_redirect_slots(kvsel_ctx* ctx, const int32_t* slot_in, const uint8_t* keep, int N,
                         int32_t dead_slot, int32_t* slot_out, void* stream);

/* ------------------------------------------------------------------------ */
/* KVMEM                                                                     */
/* ------------------------------------------------------------------------ */

/*
 * Mean-K index build (KVMEM retrieval index):
 *   index[l,g,first_block+b,:] = bf16( mean over tokens i of block b of Ktilde[l,g,i,:] )
 * Block b covers tokens [b*block, min((b+1)*block, T)) of k_src (a short last
 * block averages the tokens it has).  Ktilde = k_src when src_pos == NULL (raw,
 * position-free K), else k_src with the rotation of position src_pos[i]
 * removed (rope_base, rope_style).  Accumulation is fp32, the store rounds to
 * nearest even.  Index blocks outside [first_block, first_block + ceil(T/block))
 * are not touched.
 *   k_src   bf16 [L][Hkv][T][D], 16-byte aligned
 *   src_pos int32 [T] or NULL; positions in [0, 2^24)
 *   index   bf16 [L][Hkv][Bcap][D]
 * Requires D in {16,32,64,128,256}, block >= 1, first_block + ceil(T/block) <= Bcap.
 */
int kvsel_meank_build(kvsel_ctx* ctx, const void* k_src, int L, int Hkv, int T, int D, int block,
                      int first_block, const int32_t* src_pos, double rope_base, int rope_style,
                      void* index, int Bcap, void* stream);

/*
 * Block relevance (KVMEM retrieval):
 *   R[b] = 1/(L*Hq) * sum_{l,h,m} softmax_{b' in C}( q[l,h,m] . index[l,g(h),b'] / sqrt(D) )_b
 * C = [n_sink, n_blocks - n_recent): sink and recent blocks are always kept
 * and take no part in the softmax; R[b] = 0 outside C (and everywhere if C is
 * empty).  q holds position-free (pre-RoPE) query rows.
 *   q          bf16 [L][Hq][M][D]
 *   index      bf16 [L][Hkv][Bcap][D]
 *   R          [n_blocks] fp32 out
 *   R_partial  [L*Hkv][n_blocks] fp32 out or NULL: the unnormalised mass of
 *              each (l, g), sum over its Hq/Hkv heads and M query tokens
 * The dot products run on the tensor cores (bf16 in, fp32 accumulate), the
 * softmax in fp32.  Requires D == 128, Hq % Hkv == 0, n_blocks <= Bcap,
 * 16-byte aligned q and index.  Uses workspace: 4*L*Hkv*R bytes for the query
 * rows' log-sum-exps, R = Hq/Hkv*M rounded up to a multiple of 128, plus
 * 4*L*Hkv*n_blocks for the masses and 4 bytes per 256 query rows of each (l, g).
 */
int kvsel_block_scores(kvsel_ctx* ctx, const void* q, const void* index, int L, int Hq, int Hkv,
                       int M, int D, int n_blocks, int Bcap, int n_sink, int n_recent, float* R,
                       float* R_partial, void* stream);

/*
 * Working set (KVMEM retrieval):
 *   W = [0, n_sink) U [n_blocks - n_recent, n_blocks) U (the k largest R over C)
 * ties to the lower block id; ids ascending.  This is Eq. 1's selection with
 * the sink and recent blocks as the forced set.
 *   R         [n_blocks] fp32
 *   ids       [|W|] int32 out
 *   n_sel_host host out: |W| = |sink U recent| + min(k, |C|)
 * Workspace as kvsel_topk_retain with N = n_blocks.
 */
int kvsel_select_blocks(kvsel_ctx* ctx, const float* R, int n_blocks, int n_sink, int n_recent,
                        int k, int32_t* ids, int* n_sel_host, void* stream);

/*
 * Position-consistent restore (KVMEM, re-RoPE scatter): for entry i < n,
 * token t < page, layer l, kv head g, the raw position-free row
 *   k_src[l*src_layer_stride + g*src_head_stride + (src_block[i]*page + t)*D + :]
 * is rotated to position dst_pos0[i] + t and stored (bf16, nearest even) at
 *   pool[l][dst_page[i]][t][g][:]
 * Pool pages not named in dst_page are not touched; entries should name
 * distinct pages.
 *   k_src  bf16; strides in elements, 16-byte aligned in bytes; each head row
 *          holds src_tokens tokens
 *   src_block, dst_page, dst_pos0  int32 [n]; (src_block+1)*page <= src_tokens,
 *          dst_page < P, positions in [0, 2^24).  An entry breaking these is
 *          skipped and sets the device error word.
 *   pool   bf16 [L][P][page][Hkv][D]
 * Requires D in {16,32,64,128,256}, page*D <= 16384.
 */
int kvsel_rerope_scatter(kvsel_ctx* ctx, const void* k_src, int64_t src_layer_stride,
                         int64_t src_head_stride, int src_tokens, const int32_t* src_block,
                         const int32_t* dst_page, const int32_t* dst_pos0, int n, int L, int Hkv,
                         int D, int page, double rope_base, int rope_style, void* pool, int P,
                         void* stream);

/*
 * Many sessions per call.  A serving batch holds many agent sessions (the
 * pages' serving runs reach batches of 36) that share the model's shapes and
 * one paged K pool but differ in N, slot map, query memory, forced set and
 * budget.  The *_batch calls run the step of every session in one launch per
 * kernel (grid.y = session) and give, session by session, exactly what the
 * single-session call gives.  Session tables are host arrays; every pointer
 * inside them is a device pointer.
 */
typedef struct {
    const void* q_rows;      /* [L][Hq][R][D] post-RoPE query rows of the turn's span (q_dtype) */
    int R;                   /* rows of the span */
    float lambda;            /* decay rate */
    int first_turn;          /* 1: M = Enc(q)/|Enc(q)| (also IntentKV's query mode) */
    float* M;                /* [L][Hq][D] in/out */
    float* A;                /* [L][Hq][D] in/out for norm_mode 1, else NULL */
} kvsel_memory_session;

/*
 * kvsel_memory_update for S sessions in one launch (q_dtype, L, Hq, D and
 * norm_mode shared; each session checked as the single call checks it).
 */
int kvsel_memory_update_batch(kvsel_ctx* ctx, int q_dtype, int L, int Hq, int D, int norm_mode,
                              const kvsel_memory_session* sessions, int S, void* stream);

typedef struct {
    const int32_t* slot_map; /* [N] pool slot of each position, or NULL (identity) */
    int N;                   /* positions of this session */
    const float* M;          /* [L][Hq][D] query memory, 16-byte aligned */
    int pi, q_s, q_e;        /* forced set [0, pi) U [q_s, q_e) */
    float* rule;             /* [N] out, 16-byte aligned */
} kvsel_rule_session;

/*
 * kvsel_rule_scores for S sessions in one launch per kernel.  k_pool, dtype,
 * n_slots, strides and L, Hq, Hkv, D are shared, as in kvsel_rule_scores; each
 * session is checked as the single call checks it.  Uses workspace:
 * sum over sessions of (4*L*Hq*N + 8*L*Hq*ceil(N/64) + 4*L*Hq) bytes plus the
 * session table.  1 <= S <= 65535.
 */
int kvsel_rule_scores_batch(kvsel_ctx* ctx, const void* k_pool, int k_dtype, int n_slots, int L, int Hq,
                            int Hkv, int D, int64_t layer_stride, int64_t slot_stride,
                            const kvsel_rule_session* sessions, int S, void* stream);

typedef struct {
    const float* rule;       /* [N] scores */
    int N;
    int pi, q_s, q_e;        /* forced set [0, pi) U [q_s, q_e) */
    int C;                   /* budget */
    uint8_t* keep;           /* [N] out or NULL */
    int32_t* keep_idx;       /* [n_keep] out or NULL (not both NULL) */
} kvsel_topk_session;

/*
 * kvsel_topk_retain for S sessions.  Sessions of N <= 131072 share one launch:
 * one CTA each when every one of them has N <= 8192, else one thread-block
 * cluster each; larger sessions are selected one call each, on the paths (and
 * the workspace) of kvsel_topk_retain.  Results are
 * those of kvsel_topk_retain on each session.
 * n_keep_host: NULL or a host int array [S] receiving each session's |keep|.
 */
int kvsel_topk_retain_batch(kvsel_ctx* ctx, const kvsel_topk_session* sessions, int S, int* n_keep_host,
                            void* stream);

/*
 * Cursor-span eviction ("SideQuest" page, method overview and Figure 1): the
 * auxiliary thread lists the cursors whose KV entries the main thread clears.
 *   keep_out[j] = keep_in[j] (1 when keep_in is NULL) AND no listed cursor c has
 *                 span_start[c] <= j < span_end[c]
 * Spans are half-open and may overlap or run past [0, N); keep_out may alias
 * keep_in, so the call can clear spans from an IntentKV keep mask in place
 * before kvsel_redirect_slots.  Listed ids outside [0, n_cursors) are ignored
 * and set the device error word.
 *   span_start, span_end  int32 [n_cursors]; del_ids int32 [n_del]; masks u8 [N]
 */
int kvsel_span_keep(kvsel_ctx* ctx, const int32_t* span_start, const int32_t* span_end, int n_cursors,
                    const int32_t* del_ids, int n_del, const uint8_t* keep_in, int N, uint8_t* keep_out,
                    void* stream);

/*
 * FP8 storage of a Mean-K index (KVMEM page, section "design and trade-offs":
 * one Mean-K vector per block, layer and kv head, 9.5 GiB of index for a
 * 10M-token workspace; its server runs keep the KV cache in FP8).  A row of D
 * values (one (layer, kv head, block)) is stored as D E4M3 codes (OCP 8-bit
 * float: 4 exponent bits with bias 7, 3 mantissa bits, largest value 448) and
 * one scale exponent e, the smallest integer >= -100 with max|x| <= 448 * 2^e;
 * a stored value is code * 2^e.  Codes round to nearest, ties to the even
 * code.  Every stored value is exact in bf16, so kvsel_index_from_fp8's rows
 * feed kvsel_block_scores directly.  Half the index bytes, plus one byte a row.
 *   index  bf16 [rows][D] (16-byte aligned); codes u8 [rows][D] (4-byte
 *   aligned); exps i8 [rows].  D in {64, 128, 256}.  Inputs must be finite.
 */
int kvsel_index_to_fp8(kvsel_ctx* ctx, const void* index, int64_t rows, int D, uint8_t* codes, int8_t* exps,
                       void* stream);
int kvsel_index_from_fp8(kvsel_ctx* ctx, const uint8_t* codes, const int8_t* exps, int64_t rows, int D, void* index,
                         void* stream);

/*
 * Differential working-set update (KVMEM, section "engineering: tiered
 * movement, page-table aliasing and position-consistent rebuild"): of the new
 * working set W_t only the blocks that are not resident in the page pool are
 * moved in.  G_{t-1} is the previous working set prev_ids[n_prev] (ascending
 * block ids), block prev_ids[r] held in page prev_pages[r] at compact
 * position r*page; W_t is new_ids[n_new] (ascending), block new_ids[r] at
 * compact position r*page.
 *   retained (in both):   new_pages[r] = its old page; shift[r] = (r - old rank)*page
 *   incoming (new only):  new_pages[r] = the free pages of [0, P) -- every page
 *                         not held by a retained block -- in ascending order,
 *                         incoming blocks in ascending id; shift[r] = 0
 *   outgoing (prev only): its page is released
 * Outputs (device, int32): new_pages, shift [n_new]; in_rank, in_page [<= n_new]
 * (the incoming ranks ascending, their pages); mv_rank, mv_shift [<= n_new]
 * (retained ranks whose shift is non-zero); out_page [<= n_prev] (released
 * pages, ascending block id); counts[3] = (n_incoming, n_moved, n_outgoing).
 * Nothing is synchronised: counts stay on the device (see n_dev below).
 * Requires n_prev, n_new <= P <= 2^20 and P*page < 2^24.  A set that is not
 * strictly ascending, a previous page outside [0, P) or held twice, or a pool
 * with too few free pages sets the device error word (kvsel_check_device).
 */
int kvsel_workset_diff(kvsel_ctx* ctx, const int32_t* prev_ids, const int32_t* prev_pages, int n_prev,
                       const int32_t* new_ids, int n_new, int P, int page, int32_t* new_pages,
                       int32_t* shift, int32_t* in_rank, int32_t* in_page, int32_t* mv_rank,
                       int32_t* mv_shift, int32_t* out_page, int32_t* counts, void* stream);

/*
 * Restore of incoming blocks (same KVMEM section): K rebuilt from the raw,
 * position-free K at the new compact position, exactly as
 * kvsel_rerope_scatter; V, which carries no position, copied bit for bit.
 * v_src has k_src's layout and strides; v_pool has pool's layout.  For
 * entry i < n, token t < page, layer l, kv head g:
 *   k_pool[l][dst_page[i]][t][g][:] = bf16(RoPE(k_src row, dst_pos0[i] + t))
 *   v_pool[l][dst_page[i]][t][g][:] = v_src row
 * n_dev: NULL, or a device int32 count <= n: entries >= *n_dev are skipped, so
 * that a launch sized for n can follow kvsel_workset_diff without a host sync.
 * Checks, limits and errors as kvsel_rerope_scatter; both pools must be
 * 16-byte aligned.
 */
int kvsel_restore_blocks(kvsel_ctx* ctx, const void* k_src, const void* v_src, int64_t src_layer_stride,
                         int64_t src_head_stride, int src_tokens, const int32_t* src_block,
                         const int32_t* dst_page, const int32_t* dst_pos0, int n, const int32_t* n_dev,
                         int L, int Hkv, int D, int page, double rope_base, int rope_style, void* k_pool,
                         void* v_pool, int P, void* stream);

/*
 * Move retained blocks to their new compact positions in place (page-table
 * aliasing keeps the page; the K rows must follow the position): every row
 * pool[l][pages[i]][t][g][:] becomes bf16(R(shifts[i]) * row), the RoPE
 * rotation by shifts[i] positions (negative: backwards).  Rotations compose,
 * so a row rotated to position p lands on position p + shifts[i].
 *   pool    bf16 [L][P][page][Hkv][D], 16-byte aligned
 *   pages, shifts  int32 [n]; |shift| < 2^24, page < P, else the entry is
 *           skipped and the device error word is set
 *   n_dev   NULL or a device count <= n, as in kvsel_restore_blocks
 * Requires D in {16,32,64,128,256}.  Entries should name distinct pages.
 */
int kvsel_rerope_shift(kvsel_ctx* ctx, void* pool, int P, const int32_t* pages, const int32_t* shifts, int n,
                       const int32_t* n_dev, int L, int Hkv, int D, int page, double rope_base,
                       int rope_style, void* stream);

/*
 * Packed and pipelined rematerialisation (KVMEM, same section): restores n
 * blocks from a HOST repository into the GPU page pools, as
 * kvsel_restore_blocks would from device memory.  The blocks lie scattered in
 * the repository; each batch of chunk_blocks blocks is gathered by
 * gather_threads CPU threads into one contiguous pinned buffer, copied to the
 * device in one cudaMemcpyAsync on the context's copy stream, and restored by
 * the K re-RoPE + V copy kernel on `stream`.  Two buffer slots alternate, so
 * the gather of batch c+1, the copy of batch c and the kernel of batch c-1 run
 * at the same time.
 *   host_k, host_v  bf16 [L][Hkv][host_tokens][D] in host memory (pinned or
 *                   pageable), strides in elements; block b is tokens
 *                   [b*page, (b+1)*page)
 *   blocks, dst_page, dst_pos0  HOST int32 [n]: repository block, pool page and
 *                   first compact position of each entry; all are checked on
 *                   the host before any work (KVSEL_ERR_SHAPE)
 *   k_pool, v_pool  device bf16 [L][P][page][Hkv][D], 16-byte aligned
 * Blocks the host until every batch is gathered and queued (at most two
 * batches ahead of the GPU); the restore itself completes asynchronously on
 * `stream`.  The context owns the staging buffers (two slots of the largest
 * batch, pinned and device) and reuses them across calls.
 * mode:
 *   KVSEL_STAGE_AUTO    direct when both repositories are pinned and mapped
 *                       (cudaHostAlloc / cudaHostRegister), packed otherwise
 *   KVSEL_STAGE_PACKED  always the packed, pipelined path above
 *   KVSEL_STAGE_DIRECT  the restore kernel reads the mapped repositories in
 *                       place (on a Grace host over NVLink-C2C): no CPU gather,
 *                       no staging copy; KVSEL_ERR_INVALID_ARG if not mapped
 * Results are identical in every mode.
 */
int kvsel_stage_restore(kvsel_ctx* ctx, const void* host_k, const void* host_v, int64_t host_layer_stride,
                        int64_t host_head_stride, int host_tokens, const int32_t* blocks,
                        const int32_t* dst_page, const int32_t* dst_pos0, int n, int L, int Hkv, int D,
                        int page, double rope_base, int rope_style, void* k_pool, void* v_pool, int P,
                        int chunk_blocks, int gather_threads, int mode, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVSEL_H_ */

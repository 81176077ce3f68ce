/*
 * llsa.h -- C ABI of the GB300 (sm_103a) Log-linear Sparse Attention library.
 *
 * The method: "Trainable Log-linear Sparse Attention for Efficient Diffusion
 * Transformers" (arXiv 2512.16615), as described on its Pith review page
 * (pith.science/paper/2512.16615), sections "Core claim" and "What carries the
 * argument", and the referee report (Algorithm 1, Eq. (6), KV Reweighting,
 * Sec. 4.3 / Figure 4 on the sparse backward).
 *
 * Notation, per (batch b, head h) slice:
 *   N tokens, head dimension d, block size B, levels L = floor(log_B N - 1),
 *   n_l = N / B^l pooled tokens at level l (n_0 = N), T = n_1 query blocks
 *   (= fine key blocks), Top-K K, K_l = K clamped to level l's candidates,
 *   P = n_1 + ... + n_L pooled rows, L_e enrichment levels.
 *
 * Conventions shared by every call:
 *   - Memory. Every pointer is a DEVICE pointer owned by the caller, 16-byte
 *     aligned, to a contiguous row-major buffer. The library never allocates,
 *     frees or synchronises; scratch memory comes from the caller's workspace
 *     (`ws`, `ws_bytes`; size from llsa_workspace_bytes).
 *   - Streams. `stream` is a cudaStream_t passed as void*; every call only
 *     enqueues kernels on it and returns.
 *   - Layout. Token tensors are [batch, heads, N, d]; dtype LLSA_DTYPE_BF16
 *     (bf16 storage, fp32 accumulation) or LLSA_DTYPE_F32.
 *   - Errors. Calls return LLSA_OK (0) or a negative LLSA_ERR_* code and then
 *     enqueue nothing. Faults found on the device (a bounded wait that ran out,
 *     an index out of range) are recorded in a device status word that
 *     llsa_get_status reads. No C++ exception crosses this boundary.
 *   - Empty input (batch * heads == 0) is valid and enqueues nothing.
 */
#ifndef LLSA_H
#define LLSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LLSA_MAX_LEVELS 8

enum {
    LLSA_OK = 0,
    LLSA_ERR_INVALID_ARG = -1, /* NULL pointer, negative size, bad option */
    LLSA_ERR_SHAPE = -2,       /* N < B^2, N not divisible by B^L, d unsupported */
    LLSA_ERR_DTYPE = -3,       /* dtype not BF16 / F32 */
    LLSA_ERR_ALIGN = -4,       /* a pointer is not 16-byte aligned */
    LLSA_ERR_DEVICE = -5,      /* current device is not compute capability 10.3 */
    LLSA_ERR_WORKSPACE = -6,   /* ws NULL or smaller than llsa_workspace_bytes */
    LLSA_ERR_CUDA = -7,        /* a kernel launch failed */
    LLSA_ERR_UNSUPPORTED = -8, /* sizes beyond the kernels' limits (see each call) */
    LLSA_ERR_TIMEOUT = -9,     /* device status: a bounded wait gave up */
    LLSA_ERR_BAD_INDEX = -10   /* device status: an index outside its range */
};

enum { LLSA_DTYPE_BF16 = 0, LLSA_DTYPE_F32 = 1 };

/* Enrichment rule: which coarse tokens of level l join query block i's keys
 * ("Core claim": one coarse token from every level; the page does not say
 * which, so three readings are offered).
 * TOP1: the rank-1 selection of level l for i's level-l ancestor
 *       floor(i / B^(l-1));
 * ANCESTOR: that ancestor itself, the level-l token whose B^l tokens contain
 *       query block i;
 * ALLK: all K_l selections of level l for that ancestor (K_l tokens per
 *       level instead of one, each with weight B^l). */
enum { LLSA_ENRICH_TOP1 = 0, LLSA_ENRICH_ANCESTOR = 1, LLSA_ENRICH_ALLK = 2 };

/* Token order of q, k, v, o, dout, dq, dk and dv (referee comments on Sec. 5.1
 * and Figure 2, index reordering; the ordering is the one llsa_reorder
 * computes). LLSA_ORDER_TILE: the tokens are already in the hierarchical tile
 * order, so every block of B consecutive tokens is compact in the image.
 * LLSA_ORDER_RASTER: they are in the raster order of a square image of side
 * sqrt(N); pool, forward and backward read and write them in place of a
 * reordering pass, working in tile order inside. Needs B = 16 and a side of
 * 4^m (LLSA_ERR_SHAPE otherwise); llsa_fwd and llsa_bwd take it only on the
 * per-query-block tensor-core kernels (bf16, d in {64, 128} with K_1 in
 * {8, 16}, or d = 64 with K_1 = 32; one coarse token per level; the forward
 * needs no workspace then), else
 * LLSA_ERR_UNSUPPORTED. Everything that is not a token
 * tensor keeps the tile order: pyr, lse, sel_idx, coarse_idx, level_idx,
 * col_ptr and row_idx index blocks and tokens by tile position. */
enum { LLSA_ORDER_TILE = 0, LLSA_ORDER_RASTER = 1 };

enum { LLSA_OP_POOL = 0, LLSA_OP_SELECT = 1, LLSA_OP_FWD = 2, LLSA_OP_TRANSPOSE = 3, LLSA_OP_BWD = 4 };

typedef struct llsa_params {
    int batch, heads;   /* slices = batch * heads */
    int n;              /* N, tokens per slice */
    int d;              /* head dimension: multiple of 8, at most 256 */
    int block;          /* B >= 2 */
    int levels;         /* L; 0 selects floor(log_B N - 1); at most that value */
    int topk;           /* K >= 1 */
    int enrich_levels;  /* L_e; -1 selects L; 0 disables enrichment */
    int dtype;          /* LLSA_DTYPE_BF16 or LLSA_DTYPE_F32 */
    float scale;        /* softmax scale; 0 selects 1/sqrt(d) */
    int enrich_rule;    /* LLSA_ENRICH_TOP1, LLSA_ENRICH_ANCESTOR or LLSA_ENRICH_ALLK */
    int token_order;    /* LLSA_ORDER_TILE (0) or LLSA_ORDER_RASTER */
} llsa_params;

/* Sizes derived from the parameters. */
typedef struct llsa_sizes {
    int levels;                               /* L */
    int enrich_levels;                        /* L_e */
    int n_level[LLSA_MAX_LEVELS + 1];         /* n_0 .. n_L */
    int topk_level[LLSA_MAX_LEVELS + 1];      /* K_1 .. K_L (index 0 unused) */
    int row_offset[LLSA_MAX_LEVELS + 1];      /* first pyramid row of level l (index 0 unused) */
    int pyr_rows;                             /* P */
    int n_blocks;                             /* T = n_1 */
    int keys_per_query;                       /* K_1 * B + enrich_cols */
    long long slices;                         /* batch * heads */
    long long level_idx_offset[LLSA_MAX_LEVELS + 1]; /* int32 offset of level l >= 2 inside one slice of level_idx */
    long long level_idx_per_slice;            /* int32 entries per slice of level_idx */
    float scale;                              /* effective softmax scale */
    int coarse_cols;                          /* C: entries per row of coarse_idx (levels 1..L) */
    int enrich_cols;                          /* coarse keys per query: the columns of levels 1..L_e */
} llsa_sizes;

/* Derive sizes and validate the parameters (no device work). */
int llsa_get_sizes(const llsa_params *p, llsa_sizes *out);

/* Workspace each call needs, in bytes (0 when none); op is LLSA_OP_*.
 * Returns 0 also when the parameters are invalid (the call then fails). */
size_t llsa_workspace_bytes(const llsa_params *p, int op);

/* Hierarchical compression ("Core claim": Q, K, V mean-pooled over log-many
 * levels of contiguous B-token blocks).
 *   q, k, v : [batch, heads, N, d] in p->dtype.
 *   pyr     : output, fp32 [3][batch*heads][P][d]: the Q pyramid, then K, then V;
 *             level l of a slice occupies rows row_offset[l] .. +n_l, with
 *             P^(l)[j] = (1/B) sum_{c<B} P^(l-1)[jB + c], P^(0) = the input. */
int llsa_pool(const llsa_params *p, const void *q, const void *k, const void *v, float *pyr,
              void *ws, size_t ws_bytes, void *stream);

/* Hierarchical Top-K selection ("Core claim"; referee comment on Algorithm 1,
 * Eq. (6)). The coarsest level scores every pair of its n_L tokens; each finer
 * level l scores, for query token i, only the K_{l+1} * B children
 * {jB + c : j in I^(l+1)[floor(i/B)], c < B}. The score is the raw dot product
 * of pooled Q and pooled K in fp32; ties go to the lower index.
 *   pyr        : input from llsa_pool.
 *   sel_idx    : output int32 [batch*heads][T][K_1], I^(1), rows ascending.
 *   coarse_idx : output int32 [batch*heads][T][C] (C = coarse_cols): the
 *                enrichment tokens of query block i, level 1 first; one
 *                column per level (TOP1, ANCESTOR), or K_l columns holding
 *                I^(l)[floor(i / B^(l-1))] ascending (ALLK).
 *   level_idx  : output int32, I^(2) .. I^(L), each slice holding
 *                level_idx_per_slice entries, level l at level_idx_offset[l]
 *                as n_l rows of K_l ascending indices. May be NULL when L == 1.
 * Limits: at most 1024 candidates per query token at any level; ALLK at most
 * 64 coarse keys per query (enrich_cols). */
int llsa_select(const llsa_params *p, const float *pyr, int32_t *sel_idx, int32_t *coarse_idx,
                int32_t *level_idx, void *ws, size_t ws_bytes, void *stream);

/* Block-sparse attention with hierarchical KV enrichment ("Core claim").
 * For token t of query block i, the keys are the B tokens of each block in
 * sel_idx[i] plus, for each column c of coarse_idx[i] whose level l is at most
 * L_e, the pooled token K^(l)[coarse_idx[i][c]] with weight B^l (logit +
 * ln B^l, KV Reweighting); then
 *   lse_t = ln sum_x exp(s_tx),  o_t = sum_x exp(s_tx - lse_t) v_x,
 * with s_tx = scale * q_t . k_x (+ ln B^l for coarse keys).
 *   q, k, v    : [batch, heads, N, d] (p->dtype); pyr from llsa_pool.
 *   sel_idx    : int32 [batch*heads][T][K_1], entries in [0, T).
 *   coarse_idx : int32 [batch*heads][T][C], level-l entries in [0, n_l).
 *   o          : output [batch, heads, N, d] (p->dtype).
 *   lse        : output fp32 [batch, heads, N] (natural log).
 *   ws         : llsa_workspace_bytes(p, LLSA_OP_FWD) bytes, 16-byte aligned
 *                (0 bytes, ws may be NULL, where that is 0): the grouping of
 *                query blocks that share selected key blocks, which the
 *                grouped tensor-core forward gathers once per group. Too
 *                small a workspace: LLSA_ERR_WORKSPACE, nothing enqueued.
 * Where the grouped forward applies (bf16, B = 16, d = 64, K_1 in {4, 8, 16},
 * one enrichment column per level, L_e <= 3), the call groups the query blocks
 * first and then takes the grouped forward when the groups hold at least 4.5
 * query blocks on average, else the per-query-block one (decided on the
 * device; both agree within rounding; K_1 = 4 has only the grouped one). The
 * per-query-block tensor-core forward takes d in {64, 128} with K_1 in {8, 16},
 * and d = 64 with K_1 = 32; other shapes run on CUDA-core kernels.
 * A key block listed twice in a row of sel_idx counts once (the key set is
 * the union of the listed blocks). */
int llsa_fwd(const llsa_params *p, const void *q, const void *k, const void *v, const float *pyr,
             const int32_t *sel_idx, const int32_t *coarse_idx, void *o, float *lse,
             void *ws, size_t ws_bytes, void *stream);

/* Sparse index transpose ("What carries the argument": a CSR-to-CSC scan that
 * gives each key block its query blocks without a dense N x N mask).
 *   sel_idx : int32 [batch*heads][T][K_1] (rows need not be sorted; entries
 *             of a row must be distinct and in [0, T)).
 *   col_ptr : output int32 [batch*heads][T + 1]; col_ptr[j] is the exclusive
 *             prefix sum of the counts of columns < j (col_ptr[T] = T*K_1).
 *   row_idx : output int32 [batch*heads][T * K_1]; entries col_ptr[j] ..
 *             col_ptr[j+1]-1 list, ascending, every i with j in sel_idx[i].
 *   ws      : llsa_workspace_bytes(p, LLSA_OP_TRANSPOSE) bytes, 16-byte
 *             aligned (column counters; the one-kernel form leaves it unused).
 * Bit-exact and deterministic. An entry outside [0, T) is skipped and
 * reported through llsa_get_status (col_ptr[T] then counts the valid
 * entries). Too small a workspace: LLSA_ERR_WORKSPACE, nothing enqueued. */
int llsa_index_transpose(const llsa_params *p, const int32_t *sel_idx, int32_t *col_ptr, int32_t *row_idx,
                         void *ws, size_t ws_bytes, void *stream);

/* Sparse backward (referee report, Sec. 4.3 and Figure 4: the backward uses
 * only sparse indices), gradients of sum_t dO_t . o_t with the selection held
 * fixed. Fine keys get dk_x = scale sum dS q, dv_x = sum P dO through the
 * K-major CSC; every pooled key K^(l)[e] used by enrichment passes its gradient
 * to the B^l fine rows it averages, each receiving 1/B^l of it. Pooled Q gets
 * no gradient (it only feeds the Top-K).
 *   o, lse        : from llsa_fwd; dout: [batch, heads, N, d] (p->dtype).
 *   col_ptr, row_idx : from llsa_index_transpose of the same sel_idx.
 *   dq, dk, dv    : outputs [batch, heads, N, d] (p->dtype), overwritten. */
int llsa_bwd(const llsa_params *p, const void *q, const void *k, const void *v, const void *o,
             const float *lse, const void *dout, const float *pyr, const int32_t *sel_idx,
             const int32_t *coarse_idx, const int32_t *col_ptr, const int32_t *row_idx,
             void *dq, void *dk, void *dv, void *ws, size_t ws_bytes, void *stream);

/* Test hook; no counterpart in the paper. Sets how many polls a bounded
 * device wait of the tensor-core kernels makes before it gives up and records
 * LLSA_ERR_TIMEOUT in the status word (polls <= 0 restores the kernels' own
 * limit, about a second of polling), and test switches:
 *   LLSA_TEST_NO_COPIES        the kernels' copy warps issue no copies, so
 *                              every consumer's first wait runs out with no
 *                              copy or MMA in flight; the kernel then drains,
 *                              frees its tensor memory and exits, leaving its
 *                              outputs undefined (failure detection).
 *   LLSA_TEST_FORCE_GROUPED    llsa_fwd takes the grouped tensor-core forward
 *   LLSA_TEST_FORCE_PER_BLOCK  or the per-query-block one, whatever the
 *                              grouping found (normally the grouped forward
 *                              runs when its groups hold at least 4.5 query
 *                              blocks on average); results agree either way
 *                              within rounding.
 * Process-wide; applies to calls made after it; (0, 0) is the default state.
 * Host-side only, no device work. Unknown flag bits, or both FORCE bits:
 * LLSA_ERR_INVALID_ARG. */
#define LLSA_TEST_NO_COPIES 1
#define LLSA_TEST_FORCE_GROUPED 2
#define LLSA_TEST_FORCE_PER_BLOCK 4
int llsa_test_set_wait_limit(int polls, int flags);

/* Sparse index transpose for callers that cannot allocate device memory.
 * No counterpart in the paper: this is a deployment variant of
 * llsa_index_transpose for callers that may not call cudaMalloc or hand over a
 * workspace (an allocator-free runtime, a caller inside someone else's memory
 * pool or budget). Same inputs, outputs, layout and results as
 * llsa_index_transpose, without `ws`: its scratch -- one int32 counter per
 * fine key block per slice -- lives in a fixed device array of
 * LLSA_NOALLOC_TRANSPOSE_MAX_COUNTERS entries (4 MiB) that every GPU which
 * loads this library holds until the process exits.
 *   - Limit: batch * heads * T <= LLSA_NOALLOC_TRANSPOSE_MAX_COUNTERS, else
 *     LLSA_ERR_UNSUPPORTED and nothing is enqueued.
 *   - Allocation: none; no cudaMalloc, cudaFree or allocating library call.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture. The address is kept for the life of the
 *     process: after cudaDeviceReset of that device (or any other teardown of
 *     its primary context) the kept address is stale, so such a caller
 *     reloads the library before calling again. The device status word read
 *     by llsa_get_status is looked up and kept the same way.
 *   - Sharing: the multi-kernel form of the transpose (slices too large for
 *     the one-kernel form, or more slices than resident thread-block
 *     clusters) uses the array; every such call uses the same array. It is
 *     zeroed on the stream at the start of each call, so no earlier contents
 *     leak into a result, but such calls whose kernels overlap on the GPU
 *     (different streams, no ordering) race on it and give wrong results. */
#define LLSA_NOALLOC_TRANSPOSE_MAX_COUNTERS (1 << 20)
int llsa_index_transpose_noalloc(const llsa_params *p, const int32_t *sel_idx, int32_t *col_ptr, int32_t *row_idx,
                                 void *stream);

/* Exhaustive single-level selection, the reference for routing recall (the
 * referee's question of how much of the full fine-level Top-K the hierarchy
 * keeps): every level-1 query token scores all T level-1 key tokens with the
 * selection's score (raw pooled dot product, fp32) and keeps its
 * K_x = min(K, T) best; ties go to the lower index.
 *   pyr     : input from llsa_pool.
 *   sel_idx : output int32 [batch*heads][T][K_x], rows ascending.
 * Limits: K_x <= 64; d <= 256. */
int llsa_select_exhaustive(const llsa_params *p, const float *pyr, int32_t *sel_idx, void *stream);

/* Hierarchical tile order of the tokens of a square image (referee comments
 * on Sec. 5.1 and Figure 2, index reordering; the page gives no formula, the
 * reading is: with B = s^2 and an s^m x s^m raster image, every run of B^l
 * consecutive positions of the new order is an s^l x s^l square of pixels,
 * applied recursively; pixel (r, c) with base-s digits r_k, c_k goes to
 * position sum_k (r_k * s + c_k) * B^k).
 *   in, out  : [batch, heads, N, d] in p->dtype, distinct buffers (16-byte
 *              aligned); out receives in's rows in the new order (inverse = 0,
 *              raster -> tile order) or back (inverse = 1).
 *   height, width : the image, height * width == N, height == width == s^m.
 * Errors: LLSA_ERR_SHAPE unless B is a perfect square s^2 (s >= 2) and the
 * image is s^m x s^m; LLSA_ERR_INVALID_ARG for inverse not 0 / 1 or in == out. */
int llsa_reorder(const llsa_params *p, int height, int width, const void *in, void *out, int inverse, void *stream);

/* Reads (after synchronising `stream`) and clears the device status word of
 * the current device: LLSA_OK, LLSA_ERR_TIMEOUT or LLSA_ERR_BAD_INDEX. */
int llsa_get_status(void *stream, int *device_status);

/* Message for an LLSA_* code (static storage). */
const char *llsa_strerror(int code);

/* Number of kernels this library has launched in this process. */
unsigned long long llsa_launch_count(void);

/* Kernel timing: when enabled, every kernel launch is bracketed by CUDA events
 * on its stream. llsa_profile_read copies up to `cap` records (kernel name,
 * elapsed ms) of the launches since the last reset, synchronising on the
 * recorded events, and returns how many it wrote. */
int llsa_profile_enable(int on);
int llsa_profile_reset(void);
int llsa_profile_read(const char **names, float *ms, int cap);

/* Restricts the timing above to kernels whose name starts with `prefix` (the
 * names llsa_profile_read reports); NULL or "" times every kernel again. The
 * string is copied. Events recorded between kernels keep the GPU from
 * starting the next kernel while the one before drains, so a timed run that
 * needs one kernel's duration records only that kernel. Returns LLSA_OK. */
int llsa_profile_only(const char *prefix);

#ifdef __cplusplus
}
#endif

#endif /* LLSA_H */

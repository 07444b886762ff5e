/*
 * spin.h -- C ABI of the SPIN (Shadow Predictive Indexer) decode-time indexer step
 * for NVIDIA GB300 (sm_103a).
 *
 * Paper: "SPIN: Shadow Predictive Indexer for Sparse Attention" (arXiv 2610.09025).
 * Per request, per layer and per decode step the library
 *   1. predicts each 64-slot KV block's importance from two EMAs of past indexer scores
 *      (Eq. 1, Eq. 2) and selects the layer's block budget: forced sink and newest
 *      blocks, the top-ranked blocks and a random exploration share (Algorithm 1's
 *      budget, prediction and selection steps, §3.2 practical details, §3.2.1)
 *                                                          -> spin_select_blocks
 *   2. runs the indexer z[i] = sum_h w_h ReLU(q_h . k_{i,h}) over the slots of the
 *      selected blocks only, read through a paged block table (§2, Algorithm 1's scoring step)
 *                                                          -> spin_indexer_score
 *   3. takes the post-indexer top-K of the fresh scores (Algorithm 1's top-K step) -> spin_topk
 *   4. updates the vertical EMA V[i] and the diagonal EMA D[q-i] (Algorithm 1's EMA update)
 *                                                          -> spin_update_ema
 *   and, for speculative decoding (§3.2.2), unions the masks of several verifier rows
 *   (spin_select_blocks with rows > 1) and replays the EMA updates of the accepted
 *   prefix of rows once verification is known (spin_commit_mtp).
 *
 * Conventions (every entry point):
 *   - All pointers except `cfg`, `bytes` and those of the per-layer budget functions
 *     (host functions on host arrays) are DEVICE pointers owned by the caller; the
 *     library allocates nothing and keeps no state between calls (except the built-in
 *     scratch array of spin_select_blocks_noalloc, see there).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream): the host validates the configuration and sizes, then enqueues kernels.
 *     Kernels are launched with programmatic dependent launch allowed (PTX ISA:
 *     griddepcontrol): one may be scheduled while the previous kernel on the stream
 *     still runs, but it reads and writes memory only after that kernel has completed,
 *     so stream order holds exactly as for plain launches.
 *   - Host-side validation failures return an error code and enqueue nothing; the
 *     message is available from spin_last_error_string() (thread-local).
 *   - Values the host cannot see (N, q, block ids, page ids, accepted counts) are
 *     checked by the kernels: a bad value sets a bit in the caller's `*status`
 *     (atomicOr; may be NULL) and the affected request or block is skipped -- no
 *     out-of-range access and no trap.  Kernels that stage data through shared memory
 *     wait on mbarriers; every such wait is bounded (1 s of GPU global time), and a
 *     wait that runs out sets SPIN_STATUS_TIMEOUT, drains the kernel's own copies in
 *     flight, frees its tensor memory and returns.
 *
 * Layouts (R = n_req, MB = ceil(max_slots / 64), DL = max_slots + max_rows, rows <= max_rows):
 *   V        float  [R][max_slots]       vertical EMA per absolute slot i
 *   D        float  [R][DL]              diagonal EMA per relative offset q - i
 *   Vmax     float  [R][MB]              max of V over each block's 64 slots (kept exact)
 *   warm     int32  [R]                  0 after a reset: the next selection is dense
 *   n_slots  int32  [R]                  N, context length in KV slots (N <= max_slots)
 *   q_pos    int32  [R]                  query position of row 0 (row r sits at q + r)
 *   blocks   int32  [R][rows][MB]        per-row selection, ascending block ids
 *   n_blocks int32  [R][rows]
 *   list     int32  [R][MB], n_list [R]  a block list: a row-0 selection (rows == 1) or
 *                                        the union of the rows' selections
 *   q        [R][rows][n_heads][head_dim] in q_dtype (F32 or BF16)
 *   w        float  [R][rows][n_heads]
 *   k_pool   [n_pages][64][kv_heads][head_dim] in k_dtype (F32, BF16 or E4M3)
 *   k_scale  float  [n_pages][64]        per-slot dequantisation scale (E4M3 only)
 *   block_table int32 [R][bt_stride]     logical block j of request r -> page id
 *   scores   float  [R][rows][MB*64]     slot s of list entry k at k*64 + s; slots
 *                                        i >= N hold 0
 *   topk_idx int32  [R][rows][top_k]     ascending slot ids, -1 padded
 */
#ifndef SPIN_H
#define SPIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* spin_stream_t; /* a cudaStream_t */

typedef enum spin_status {
    SPIN_OK = 0,
    SPIN_ERR_INVALID_ARG = 1,      /* NULL pointer, value out of range */
    SPIN_ERR_SHAPE = 2,            /* inconsistent sizes (rows > max_rows, kv_heads, ...) */
    SPIN_ERR_CAPACITY = 3,         /* a size beyond what the kernels support */
    SPIN_ERR_UNSUPPORTED = 4,      /* dtype or score path not available for this shape */
    SPIN_ERR_CUDA = 5              /* a CUDA runtime call or a launch failed */
} spin_status_t;

/* Bits of the device status word. */
#define SPIN_STATUS_BAD_N        0x01u /* N < 0 or N > max_slots */
#define SPIN_STATUS_BAD_QPOS     0x02u /* q < N - 1 or q + rows - 1 >= max_slots + max_rows */
#define SPIN_STATUS_BAD_LIST     0x04u /* list count > MB or a listed block outside [0, ceil(N/64)) */
#define SPIN_STATUS_BAD_PAGE     0x08u /* block-table entry outside [0, n_pages) */
#define SPIN_STATUS_BAD_ACCEPTED 0x10u /* accepted outside [0, rows - 1] */
#define SPIN_STATUS_TIMEOUT      0x20u /* a bounded wait inside a kernel gave up */
#define SPIN_STATUS_BAD_RHO      0x40u /* budget override outside [0, 10000] */

typedef enum spin_dtype { SPIN_DTYPE_F32 = 0, SPIN_DTYPE_BF16 = 1, SPIN_DTYPE_E4M3 = 2 } spin_dtype_t;

/* Predicted slot score: Eq. 1's max(V[i], D[q-i]) (default) or the additive reading
 * V[i] + D[q-i]. */
typedef enum spin_combine { SPIN_COMBINE_MAX = 0, SPIN_COMBINE_SUM = 1 } spin_combine_t;

/* Block pooling of the predicted slot scores.  MAX is Eq. 2 (the method).  MEAN and TOP4 are
 * the pooling ablations of §4.6 ("Block reduction"), for diagnostics: the mean of the block's
 * slot predictions (slots i < N), or the mean of its (up to) four largest.  Their fp32 sums
 * have a fixed order -- MEAN: slots l and l + 32 first, then the 32 pair sums pairwise at
 * distance 16, 8, 4, 2, 1; TOP4: (t1 + t2) + (t3 + t4) in descending order -- divided
 * (correctly rounded) by the count.  SLOTS is §4.6's A0: the top_k slots with the largest
 * predicted score (equal scores: lower slot), then every block holding one, plus the sink and
 * newest blocks; no exploration and no block budget (a cold request or a budget of every
 * block still selects every block).  SLOTS needs a larger workspace (spin_workspace_size).
 * A2 is §4.6's A2 with max pooling, for one query row: the state is kept per block -- the
 * first ceil(max_slots/64) entries of a request's V hold the block-level vertical EMA Vb[j],
 * and D[o] the block-level diagonal EMA at the block offset o = floor(q/64) - j from the
 * query's block; spin_update_ema updates both with each scored block's max over its slots
 * i < N (t = fl((1-alpha) zb), fma(alpha, old, t)); the predicted block score is
 * max(Vb[j], Db[floor(q/64) - j]) (or their sum under SPIN_COMBINE_SUM); Vmax and the
 * slot-level entries are not used.  rows > 1 is rejected with SPIN_ERR_UNSUPPORTED. */
/* Exploration policy of the selection's exploration share (gamma).  RANDOM is §3.2.1 (the
 * method): Philox draws.  BLOCK_AGE is the block-age alternative of §4.6 ("Staleness
 * mitigation"), for diagnostics and one query row: the not yet selected blocks observed least
 * recently, i.e. with the smallest age (the decode step + 1 at which the block was last
 * scored, 0 = never), equal ages to the lower block.  It keeps a caller-owned age array
 * uint32 [R][MB] and needs spin_select_blocks_age / spin_update_ema_age. */
typedef enum spin_explore { SPIN_EXPLORE_RANDOM = 0, SPIN_EXPLORE_BLOCK_AGE = 1 } spin_explore_t;

typedef enum spin_pooling {
    SPIN_POOL_MAX = 0,
    SPIN_POOL_MEAN = 1,
    SPIN_POOL_TOP4 = 2,
    SPIN_POOL_SLOTS = 3,
    SPIN_POOL_A2 = 4
} spin_pooling_t;

/* Indexer-score kernel choice.  AUTO takes the tensor-core kernel when the key is shared
 * by all heads (kv_heads == 1) and the shape is supported, the streaming CUDA-core
 * kernel for per-head keys, and the generic kernel otherwise. */
typedef enum spin_score_path {
    SPIN_SCORE_AUTO = 0,
    SPIN_SCORE_GENERIC = 1,   /* any shape; slow; a cross-check */
    SPIN_SCORE_STREAM = 2,    /* per-head keys on CUDA cores, bulk-copy staged pages */
    SPIN_SCORE_TCGEN05 = 3    /* shared key on tcgen05 tensor cores (TMA + TMEM) */
} spin_score_path_t;

typedef struct spin_config {
    int32_t n_req;       /* R >= 1 */
    int32_t max_slots;   /* capacity of V per request, 1 .. 2^24 */
    int32_t max_rows;    /* verifier rows D leaves room for, 1 .. 8 */
    int32_t block;       /* b: must be 64 (one KV page of compressed slots) */
    int32_t n_heads;     /* n_h, 1 .. 128 */
    int32_t head_dim;    /* d, 1 .. 256 */
    int32_t kv_heads;    /* 1 (one key shared by all heads) or n_heads (a key per head) */
    int32_t q_dtype;     /* SPIN_DTYPE_F32 or SPIN_DTYPE_BF16 */
    int32_t k_dtype;     /* SPIN_DTYPE_F32, SPIN_DTYPE_BF16 or SPIN_DTYPE_E4M3 */
    int32_t top_k;       /* K, 1 .. 16384 */
    int32_t rho_bp;      /* target block sparsity rho in basis points, 0 .. 10000 */
    int32_t gamma_bp;    /* exploration share gamma in basis points, 0 .. 10000 */
    float alpha;         /* EMA decay, 0 .. 1 */
    int32_t combine;     /* spin_combine_t */
    uint64_t seed;       /* exploration key */
    int32_t score_path;  /* spin_score_path_t */
    int32_t pooling;     /* spin_pooling_t: MAX (Eq. 2, the method) or an ablation variant */
    int32_t explore;     /* spin_explore_t: RANDOM (the method) or BLOCK_AGE */
    int32_t reserved;    /* must be 0 */
} spin_config;

/* Zero V, D and Vmax and mark the request cold: the reset after prefill and at every
 * turn start (§3.2 practical details).  req < 0 resets every request. */
spin_status_t spin_init_state(const spin_config* cfg, float* V, float* D, float* Vmax,
                              int32_t* warm, int32_t req, spin_stream_t stream);

/* Block prediction and selection (Eq. 1, Eq. 2, Algorithm 1's prediction, budget and block top-m steps; §3.2 forced blocks;
 * §3.2.1 exploration; §3.2.2 union), for `rows` verifier rows of every request.
 *   B = ceil(N/64); m = min(B, max(ceil(K/64), ceil((10000 - rho) B / 10000)));
 *   forced F = {0, B-1}; e = min(floor(gamma m / 10000), m - |F|) (0 if m <= |F|);
 *   the m - |F| - e non-forced blocks with the largest S (S desc, j asc), then the e
 *   not-yet-selected blocks with the smallest exploration key (ties: lower j), where the
 *   output of Philox4x64-10(key = {seed, layer}, counter = {step, row, req, floor(j/8)})
 *   serves blocks 8 floor(j/8) .. +7: block j takes 32-bit half j % 8 of it, word by word,
 *   high half first.  A cold request selects every block.
 * rho_override: NULL, or a device int32 read by the kernel in place of cfg->rho_bp (a
 *   per-layer budget table entry that CUDA graphs can replay).
 * union_blocks/n_union: required when rows > 1 (ascending union of the rows), else may
 *   be NULL.  workspace: at least spin_workspace_size(cfg, rows) bytes, 256-byte aligned. */
spin_status_t spin_select_blocks(const spin_config* cfg, const float* V, const float* D,
                                 const float* Vmax, const int32_t* warm,
                                 const int32_t* n_slots, const int32_t* q_pos, int32_t rows,
                                 const int32_t* rho_override, uint64_t step, int32_t layer,
                                 int32_t* blocks, int32_t* n_blocks, int32_t* union_blocks,
                                 int32_t* n_union, void* workspace, size_t workspace_bytes,
                                 uint32_t* status, spin_stream_t stream);

/* spin_select_blocks with the decode step read from device memory: the kernels read the
 * uint64 *step_dev when they run, in place of `step`.  A CUDA graph that captures a step
 * once can then replay every later step, the caller advancing *step_dev in stream order
 * between replays (the other inputs -- V, D, N, q, the budget table -- are already device
 * memory).  Arguments, outputs and errors are otherwise those of spin_select_blocks;
 * step_dev must be non-NULL. */
spin_status_t spin_select_blocks_dstep(const spin_config* cfg, const float* V, const float* D,
                                       const float* Vmax, const int32_t* warm,
                                       const int32_t* n_slots, const int32_t* q_pos, int32_t rows,
                                       const int32_t* rho_override, const uint64_t* step_dev,
                                       int32_t layer, int32_t* blocks, int32_t* n_blocks,
                                       int32_t* union_blocks, int32_t* n_union, void* workspace,
                                       size_t workspace_bytes, uint32_t* status,
                                       spin_stream_t stream);

/* Layer stacks.  A model runs the indexer step in every layer, and a layer's selection for
 * decode step t needs only that layer's state after step t-1 -- not the layer's query -- so
 * the selections of all layers can be computed together at the start of a step
 * (§3.2 lets block prediction and the EMA update run off the layer's own critical path,
 * hidden behind other layers' work).  The _layers calls take n_layers layers whose
 * arrays are stacked along a new outermost dimension -- V [L][R][max_slots], D [L][R][DL],
 * Vmax [L][R][MB], warm [L][R], blocks [L][R][rows][MB], n_blocks [L][R][rows], union
 * [L][R][MB], n_union [L][R], scores [L][R][rows][MB*64], list [L][R][MB], n_list [L][R]
 * -- and do in one launch what n_layers single-layer calls on the slices l = 0 .. L-1
 * would do, with identical results.  n_slots, q_pos and accepted are per request, shared by
 * the layers.  1 <= n_layers <= 1024.
 *
 * spin_select_blocks_layers: layer l of the stack is model layer layer0 + l (the Philox
 *   key); rho_override is NULL or a device table of n_layers sparsities (a per-layer budget
 *   table); step_dev, if non-NULL, is read in place of `step` (as spin_select_blocks_dstep);
 *   workspace: n_layers * spin_workspace_size(cfg, rows) bytes, 256-byte aligned. */
spin_status_t spin_select_blocks_layers(const spin_config* cfg, int32_t n_layers, int32_t layer0,
                                        const float* V, const float* D, const float* Vmax,
                                        const int32_t* warm, const int32_t* n_slots,
                                        const int32_t* q_pos, int32_t rows,
                                        const int32_t* rho_override, uint64_t step,
                                        const uint64_t* step_dev, int32_t* blocks,
                                        int32_t* n_blocks, int32_t* union_blocks, int32_t* n_union,
                                        void* workspace, size_t workspace_bytes, uint32_t* status,
                                        spin_stream_t stream);
/* spin_update_ema of every layer of a stack (row-0 scores [L][R][1][MB*64]). */
spin_status_t spin_update_ema_layers(const spin_config* cfg, int32_t n_layers, float* V, float* D,
                                     float* Vmax, int32_t* warm, const float* scores,
                                     const int32_t* list, const int32_t* n_list,
                                     const int32_t* n_slots, const int32_t* q_pos, uint32_t* status,
                                     spin_stream_t stream);
/* spin_commit_mtp of every layer of a stack (scores [L][R][rows][MB*64], unions [L][R][MB]). */
spin_status_t spin_commit_mtp_layers(const spin_config* cfg, int32_t n_layers, float* V, float* D,
                                     float* Vmax, int32_t* warm, const float* scores, int32_t rows,
                                     const int32_t* union_blocks, const int32_t* n_union,
                                     const int32_t* n_slots, const int32_t* q_pos,
                                     const int32_t* accepted, uint32_t* status,
                                     spin_stream_t stream);

/* Allocation-free variant of spin_select_blocks (the paper has no counterpart: this is a
 * deployment convenience).  Some callers cannot allocate device memory for the workspace:
 * serving engines that reserve all device memory up front in their own pool and forbid
 * other allocations, plugin hosts that give the library no allocator, and latency-critical
 * loops that must not pay for an allocation.  This entry point takes the same arguments
 * minus the workspace and uses instead a scratch array that lives in the library itself
 * (a static device array of 8 MiB, held on every GPU that loads the library until the
 * process exits).  It calls no cudaMalloc/cudaFree and no allocating library routine.
 *   - Capacity: n_req * rows * ceil(max_slots/64) <= 1048576 (a block score and an
 *     exploration draw per block and row), and spin_workspace_size <= 8 MiB (which under
 *     SPIN_POOL_SLOTS holds a prediction per slot); larger configurations are rejected
 *     with SPIN_ERR_CAPACITY.
 *   - The first call on a device looks up the array's device address (with that device
 *     current) and caches it.  The cached address belongs to the device's current
 *     context: it does not survive cudaDeviceReset, after which this entry point must
 *     not be called again in the process.
 *   - Every call shares the one array, which keeps the last call's contents: calls that
 *     may overlap on the GPU (different streams, or different host threads, on one
 *     device) race on it and must be serialised by the caller.
 * Outputs are identical to spin_select_blocks. */
spin_status_t spin_select_blocks_noalloc(const spin_config* cfg, const float* V, const float* D,
                                         const float* Vmax, const int32_t* warm,
                                         const int32_t* n_slots, const int32_t* q_pos,
                                         int32_t rows, const int32_t* rho_override,
                                         uint64_t step, int32_t layer, int32_t* blocks,
                                         int32_t* n_blocks, int32_t* union_blocks,
                                         int32_t* n_union, uint32_t* status,
                                         spin_stream_t stream);

/* spin_select_blocks under SPIN_EXPLORE_BLOCK_AGE (rows = 1; rows > 1 is
 * SPIN_ERR_UNSUPPORTED): block_age uint32 [R][MB] (device, read) gives each block's age; the
 * exploration share goes to the not yet selected blocks with the smallest age, equal ages to
 * the lower block.  The other selection entry points, the MTP commit and the stacked calls
 * refuse BLOCK_AGE (SPIN_ERR_INVALID_ARG, or SPIN_ERR_UNSUPPORTED for rows > 1); a NULL
 * block_age is SPIN_ERR_INVALID_ARG, and so is an age array under SPIN_EXPLORE_RANDOM. */
spin_status_t spin_select_blocks_age(const spin_config* cfg, const float* V, const float* D,
                                     const float* Vmax, const int32_t* warm,
                                     const int32_t* n_slots, const int32_t* q_pos, int32_t rows,
                                     const int32_t* rho_override, uint64_t step, int32_t layer,
                                     const uint32_t* block_age, int32_t* blocks, int32_t* n_blocks,
                                     int32_t* union_blocks, int32_t* n_union, void* workspace,
                                     size_t workspace_bytes, uint32_t* status, spin_stream_t stream);

/* Indexer score (§2; Algorithm 1's scoring step) of every slot of every listed block for `rows`
 * query rows: z_r[i] = sum_h w[r][h] * ReLU(s_i * (q[r][h] . k[i][h'])), h' = h for
 * per-head keys and 0 for a shared key, s_i = k_scale (E4M3) or 1.  fp32 accumulation.
 * n_pages bounds the page ids of block_table (checked on the device). */
spin_status_t spin_indexer_score(const spin_config* cfg, const void* q, const float* w,
                                 const void* k_pool, const float* k_scale, int64_t n_pages,
                                 const int32_t* block_table, int64_t bt_stride,
                                 const int32_t* list, const int32_t* n_list,
                                 const int32_t* n_slots, int32_t rows, float* scores,
                                 uint32_t* status, spin_stream_t stream);

/* Optional work fused into spin_indexer_score_ex (zero-initialise, then set what is wanted). */
typedef struct spin_score_extras {
    /* Temporal top-K (see spin_topk_hinted): a hint buffer of at least topk_hint_bytes bytes
     * (spin_topk_hint_size).  The streaming and generic score kernels then compare every
     * fresh score with its row's threshold and append the live slots at or above it to the
     * hint, for the next spin_topk_hinted call on the same rows; the tensor-core kernel
     * leaves that to spin_topk_hinted.  NULL: nothing is collected. */
    void* topk_hint;
    size_t topk_hint_bytes;
} spin_score_extras;

/* spin_indexer_score with the work of `extras` (may be NULL) fused into its kernel.  Errors
 * as spin_indexer_score, plus SPIN_ERR_UNSUPPORTED when a hint is given for a shape without
 * a hinted top-K and SPIN_ERR_INVALID_ARG for a hint that is too small or not 256-byte
 * aligned. */
spin_status_t spin_indexer_score_ex(const spin_config* cfg, const void* q, const float* w,
                                    const void* k_pool, const float* k_scale, int64_t n_pages,
                                    const int32_t* block_table, int64_t bt_stride,
                                    const int32_t* list, const int32_t* n_list,
                                    const int32_t* n_slots, int32_t rows, float* scores,
                                    const spin_score_extras* extras, uint32_t* status,
                                    spin_stream_t stream);

/* Post-indexer top-K (Algorithm 1's top-K step) of every row over the scored slots i < N of
 * the list: the K largest z, equal z ordered by the lower slot id (-0 == +0); written
 * as ascending slot ids and padded with -1 when fewer than K slots were scored. */
spin_status_t spin_topk(const spin_config* cfg, const float* scores, const int32_t* list,
                        const int32_t* n_list, const int32_t* n_slots, int32_t rows,
                        int32_t* topk_idx, uint32_t* status, spin_stream_t stream);

/* Temporal top-K ("SPIN: Shadow Predictive Indexer for Sparse Attention", §5: the
 * Guess-Verify-Refine top-K exploits the correlation of consecutive decode steps).  The
 * result is exactly spin_topk's (same ties, same padding); the hint only makes it cheaper.
 *   - hint: caller-owned device memory of spin_topk_hint_size bytes, 256-byte aligned,
 *     holding per (request, row) a 64-byte record -- guess key, candidate count, rank margin,
 *     and counters of hit / miss / overflow / cold / exact steps as uint32 words 0..8 -- and
 *     then the candidate arrays.  Zero the records with spin_init_topk_hint before the first
 *     step and whenever spin_init_state resets a request.
 *   - A step is spin_indexer_score_ex with extras->topk_hint = hint, then spin_topk_hinted
 *     on the same scores, head weights w ([R][rows][n_heads], those the scores were computed
 *     with), list and rows with the same hint.  The live slots whose score is >= the row's
 *     threshold (the guess times this step's sum_h |w_h|) are the candidates, collected by
 *     the score kernel or, where it does not, by spin_topk_hinted in one pass.  If K
 *     to cap of them were found (cap = 8 K rounded up to a power of two, at least 4096, or
 *     4 K when 8 K candidates would not fit in shared memory beside the list), the
 *     top-K is selected among them; otherwise (no guess yet, too few, too many) the row is
 *     recomputed from its scores.  The score at rank K + margin divided by sum_h |w_h|
 *     becomes the next step's guess; the margin (initially sqrt(K cap) - K, within
 *     [K/8, cap/2 - K]) doubles after a miss and halves after an overflow.
 *   - Calling spin_indexer_score_ex twice with one hint without a spin_topk_hinted in
 *     between mixes two steps' candidates; the count then usually exceeds cap and the row is
 *     recomputed (still exact), unless fewer than cap were collected in total -- so do not.
 *   - Supported for top_k <= 2048 and at most 8192 blocks (ceil(max_slots/64)) when the
 *     candidates, a one-bit-per-slot bitmap and the list fit in 220 KB of shared memory; other
 *     shapes get SPIN_ERR_UNSUPPORTED from all three calls. */
spin_status_t spin_topk_hint_size(const spin_config* cfg, int32_t rows, size_t* bytes);
spin_status_t spin_init_topk_hint(const spin_config* cfg, int32_t rows, void* hint,
                                  size_t hint_bytes, int32_t req, spin_stream_t stream);
spin_status_t spin_topk_hinted(const spin_config* cfg, const float* scores, const float* w,
                               const int32_t* list, const int32_t* n_list,
                               const int32_t* n_slots, int32_t rows, int32_t* topk_idx, void* hint,
                               size_t hint_bytes, uint32_t* status, spin_stream_t stream);

/* EMA update (Algorithm 1's EMA update) from the row-0 scores of the list:
 *   t = fl((1 - alpha) z[i]);  V[i] = fma(alpha, V[i], t);  D[q-i] = fma(alpha, D[q-i], t)
 * for every listed slot i < N; Vmax of the listed blocks is refreshed and the request
 * is marked warm.  `scores` has the layout of a rows == 1 spin_indexer_score call. */
spin_status_t spin_update_ema(const spin_config* cfg, float* V, float* D, float* Vmax,
                              int32_t* warm, const float* scores, const int32_t* list,
                              const int32_t* n_list, const int32_t* n_slots,
                              const int32_t* q_pos, uint32_t* status, spin_stream_t stream);

/* Deferred MTP commit (§3.2.2): with a = accepted[req] drafts accepted, replay the
 * observations of rows 0..a in order (row r at query position q + r) with the update of
 * spin_update_ema; rows a+1.. are discarded.  `scores` is the rows-row output of
 * spin_indexer_score over the union list. */
spin_status_t spin_commit_mtp(const spin_config* cfg, float* V, float* D, float* Vmax,
                              int32_t* warm, const float* scores, int32_t rows,
                              const int32_t* union_blocks, const int32_t* n_union,
                              const int32_t* n_slots, const int32_t* q_pos,
                              const int32_t* accepted, uint32_t* status, spin_stream_t stream);

/* Per-layer block budgets ("Sparse Attention Still Has a Dense Problem", section "Per-layer
 * block budgets", Figures 5-6).  HOST functions on host pointers: they enqueue nothing and
 * need no GPU.  A dense probe step (sparsity 0) gives each layer's dense top-K; the miss
 * curve of a layer is the share of those slots that the selection at each budget would skip,
 * and the budgets minimise the worst layer's miss while the total kept fraction stays at
 * the target.  Budgets are kept fractions on a grid of n_points points,
 * p_g = g * 10000 / (n_points - 1) basis points; n_points - 1 must divide 10000.
 *
 * spin_miss_curve: one layer's curve over a batch, the mean of its requests' curves.
 *   S      float [n_req][s_stride]  the probe step's predicted block scores (the selection's
 *                                   ranking key), entries 0 .. nb[r]-1 used; no NaN
 *   nb     int32 [n_req]            blocks of each request's context, 1 .. s_stride
 *   topk   int32 [n_req][top_k]     the dense top-K slot ids of each request (-1 = none)
 *   miss   float [n_points] out     miss[g] = mean over requests of (dense top-K slots in
 *                                   blocks not selected at p_g) / (valid slots), where the
 *                                   selection at p_g is the budget rule's m blocks (sparsity
 *                                   10000 - p_g basis points): blocks 0 and nb-1, then the
 *                                   best m - f by S (equal S: lower block id); the random
 *                                   exploration share is not modelled.  Requests with no valid
 *                                   slot are left out; none left gives zeros.
 *   Errors: SPIN_ERR_INVALID_ARG (NULL pointer, bad sizes or grid, NaN score, a top-K id
 *   outside [-1, 64 * nb)); nothing is written then.
 *
 * spin_allocate_budgets: per-layer grid points from the layers' curves.
 *   miss       float [n_layers][n_points]  the curves (no NaN)
 *   target_g   the grid point of the global kept fraction: sum_l g_l = n_layers * target_g
 *   g_min      the lowest grid point a layer may take, 0 <= g_min <= target_g <= n_points - 1
 *   g_out      int32 [n_layers] out        each layer's grid point
 *   rho_bp_out int32 [n_layers] out or NULL: each layer's sparsity, 10000 - p_{g_l} (the value
 *              a device budget table hands to spin_select_blocks as rho_override)
 *   The worst layer's miss max_l miss[l][g_l] is the smallest any allocation with that total
 *   attains; each layer takes the fewest points reaching it, and the spare points go one at
 *   a time to the layer with the largest miss at its current point (equal misses: fewer
 *   points, then lower layer; a layer at the top of the grid takes none).
 *   Errors: SPIN_ERR_INVALID_ARG (NULL pointer, bad sizes or grid, NaN). */
spin_status_t spin_miss_curve(const float* S, int32_t n_req, int64_t s_stride, const int32_t* nb,
                              const int32_t* topk, int32_t top_k, int32_t n_points, float* miss);
spin_status_t spin_allocate_budgets(const float* miss, int32_t n_layers, int32_t n_points,
                                    int32_t target_g, int32_t g_min, int32_t* g_out,
                                    int32_t* rho_bp_out);

/* Self-test of the bounded wait the pipelined kernels use on their shared-memory stage
 * barriers (no counterpart in the paper: it checks the library's failure handling).  One
 * CTA waits on an mbarrier with a limit of limit_ns (0 < limit_ns <= 10 s) of GPU global time:
 *   mode 0: nobody arrives -- the wait must end at the limit;
 *   mode 1: the kernel's abort flag is raised first -- the wait must end at once;
 *   mode 2: a second warp arrives -- the wait must succeed.
 * A wait that gives up sets SPIN_STATUS_TIMEOUT in *status (device); *elapsed_ns (device)
 * receives the time the wait took. */
spin_status_t spin_selftest_wait(int32_t mode, uint64_t limit_ns, uint32_t* status,
                                 uint64_t* elapsed_ns, spin_stream_t stream);

/* spin_update_ema under SPIN_EXPLORE_BLOCK_AGE: also sets block_age[req][blk] = step + 1 for
 * every listed block inside the context (device, read-write; zero it at a reset).  The other
 * update entry points refuse BLOCK_AGE (SPIN_ERR_INVALID_ARG). */
spin_status_t spin_update_ema_age(const spin_config* cfg, float* V, float* D, float* Vmax,
                                  int32_t* warm, const float* scores, const int32_t* list,
                                  const int32_t* n_list, const int32_t* n_slots,
                                  const int32_t* q_pos, uint32_t* block_age, uint64_t step,
                                  uint32_t* status, spin_stream_t stream);

/* Bytes of device workspace spin_select_blocks needs for `rows` rows: block scores and
 * exploration draws (2 x 4 B per request, row and block), or under SPIN_POOL_SLOTS the slot
 * predictions, an identity block list and the top-K slots (4 B per request, row and slot,
 * and more); the stacked calls need n_layers times this. */
spin_status_t spin_workspace_size(const spin_config* cfg, int32_t rows, size_t* bytes);

/* Version string of the library ("spin-gb300 <major>.<minor>.<patch> sm_103a"). */
const char* spin_version(void);

/* Message of the last host-side error of the calling thread ("" if none). */
const char* spin_last_error_string(void);

#ifdef __cplusplus
}
#endif
#endif /* SPIN_H */

/*
 * spin_oracle.h -- plain, slow, single-threaded CPU oracle of the SPIN decode-time
 * indexer step.  TEST INFRASTRUCTURE ONLY: the tests, the package's smoke check and
 * the benchmark's CPU-baseline leg are the only callers.  It shares no code, header,
 * table or constant with the CUDA library, and the library never calls it.
 *
 * Source: "SPIN: Shadow Predictive Indexer for Sparse Attention" (arXiv 2610.09025),
 * §2 (indexer score), §3.2 (Eq. 1, Eq. 2, Algorithm 1 and its practical details),
 * §3.2.1 (exploration) and §3.2.2 (speculative decoding); the NVIDIA Research blog
 * "Sparse Attention Still Has a Dense Problem" (block size 64, 5 % exploration).
 *
 * Buffer layouts are the ones the C ABI uses (R = n_req, MB = ceil(max_slots/64)):
 *   V      float [R][max_slots]                 vertical EMA per absolute slot
 *   D      float [R][max_slots + max_rows]      diagonal EMA per relative offset q - i
 *   warm   int32 [R]                            0 right after a reset
 *   blocks int32 [R][rows][MB] + n_blocks [R][rows]   per-row selected blocks, ascending
 *   list   int32 [R][MB] + n_list [R]           a block list consumed by score/top-K/EMA
 *   scores float [R][rows][MB*64]               slot s of list entry k at k*64 + s
 *   topk   int32 [R][rows][top_k]               ascending slot ids, -1 padded
 *
 * Parity status of every function is stated in the header comment of spin_oracle.c.
 */
#ifndef SPIN_ORACLE_H
#define SPIN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_E4M3 = 2 };
enum { ORACLE_COMBINE_MAX = 0, ORACLE_COMBINE_SUM = 1 };
enum { ORACLE_POOL_MAX = 0, ORACLE_POOL_MEAN = 1, ORACLE_POOL_TOP4 = 2, ORACLE_POOL_SLOTS = 3, ORACLE_POOL_A2 = 4 };
enum { ORACLE_EXPLORE_RANDOM = 0, ORACLE_EXPLORE_AGE = 1 };

typedef struct oracle_cfg {
    int32_t n_req;      /* R */
    int32_t max_slots;  /* capacity of V per request */
    int32_t max_rows;   /* verifier rows the D array leaves room for */
    int32_t block;      /* b, must be 64 */
    int32_t n_heads;    /* n_h */
    int32_t head_dim;   /* d */
    int32_t kv_heads;   /* 1 (one key shared by all heads) or n_heads (a key per head) */
    int32_t q_dtype;    /* ORACLE_F32 or ORACLE_BF16 */
    int32_t k_dtype;    /* ORACLE_F32, ORACLE_BF16 or ORACLE_E4M3 */
    int32_t top_k;      /* K */
    int32_t rho_bp;     /* target block sparsity, basis points */
    int32_t gamma_bp;   /* exploration share, basis points */
    float alpha;        /* EMA decay */
    int32_t combine;    /* ORACLE_COMBINE_MAX (Eq. 1) or ORACLE_COMBINE_SUM */
    uint64_t seed;      /* exploration key */
    int32_t pooling;    /* ORACLE_POOL_MAX (Eq. 2), the MEAN / TOP4 ablations, the A0
                           ablation ORACLE_POOL_SLOTS or the A2 ablation ORACLE_POOL_A2
                           (§4.6); under A2 the first ceil(max_slots/64) entries of a
                           request's V hold the block-level vertical EMA and D[o] the
                           block-level diagonal EMA at block offset o (one query row) */
    int32_t explore;    /* ORACLE_EXPLORE_RANDOM (§3.2.1) or the block-age exploration of
                           §4.6 "Staleness mitigation" (ORACLE_EXPLORE_AGE, one query row) */
} oracle_cfg;

/* Philox4x64-10 block function (Salmon et al., SC'11). */
void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]);
/* Exploration draw of block j: high 32 bits of word 0 of Philox4x64-10 with
 * key = {seed, layer} and counter = {step, row, req, j}. */
uint32_t oracle_explore_key(uint64_t seed, int32_t layer, uint64_t step, int32_t row,
                            int32_t req, int64_t j);

/* Exact decoders of the stored number formats. */
double oracle_decode_e4m3(uint8_t code);
double oracle_decode_bf16(uint16_t bits);

/* Algorithm 1's budget step, rho in basis points. */
int64_t oracle_budget(int64_t n_blocks, int64_t top_k, int64_t block, int32_t rho_bp);
/* Exploration share of §3.2.1: floor(gamma*m), capped by the capacity m - f left
 * after the forced blocks; 0 when m <= f. */
int64_t oracle_explore_count(int64_t m, int64_t n_forced, int32_t gamma_bp);

/* Eq. 2 (Algorithm 1's pooling step) for one query row at position q: S[j], j < ceil(N/b). */
void oracle_block_scores(const oracle_cfg* cfg, const float* V_req, const float* D_req,
                         int64_t n_slots, int64_t q, float* S_out);

/* Block selection for every request and row (Algorithm 1's prediction, budget and block top-m steps plus forced
 * blocks, exploration and the multi-row union).  rho_bp < 0 uses cfg->rho_bp.
 * union_blocks / n_union may be NULL. Returns 0, or -1 on invalid input. */
int oracle_select_blocks(const oracle_cfg* cfg, const float* V, const float* D,
                         const int32_t* warm, const int32_t* n_slots, const int32_t* q_pos,
                         int32_t rows, int32_t rho_bp, uint64_t step, int32_t layer,
                         int32_t* blocks, int32_t* n_blocks,
                         int32_t* union_blocks, int32_t* n_union);
/* oracle_select_blocks with block-age exploration (§4.6 "Staleness mitigation"): the
 * exploration share goes to the not yet selected blocks observed least recently, i.e. with
 * the smallest age[req][j] (the decode step + 1 at which block j was last scored, 0 =
 * never), equal ages to the lower block. */
int oracle_select_blocks_age(const oracle_cfg* cfg, const float* V, const float* D,
                             const int32_t* warm, const int32_t* n_slots, const int32_t* q_pos,
                             int32_t rows, int32_t rho_bp, uint64_t step, int32_t layer,
                             const uint32_t* age, int32_t* blocks, int32_t* n_blocks,
                             int32_t* union_blocks, int32_t* n_union);
/* Record that the listed blocks were scored at decode step `step`: age[req][blk] = step + 1. */
int oracle_block_age_update(const oracle_cfg* cfg, uint32_t* age, const int32_t* list,
                            const int32_t* n_list, const int32_t* n_slots, uint64_t step);

/* Indexer score (Algorithm 1's scoring step) of every slot i < N of every listed block, for
 * `rows` query rows.  q: [R][rows][n_heads][d] in q_dtype; w: [R][rows][n_heads];
 * k_pool: [pages][64][kv_heads][d] in k_dtype; k_scale: [pages][64] (E4M3 only, else
 * NULL); block_table: [R][bt_stride].  Slots i >= N get score 0.  mags (nullable,
 * same layout as scores) receives sum_h |w_h| |s_i| sum_c |q_hc k_ihc| in double. */
int oracle_indexer_score(const oracle_cfg* cfg, const void* q, const float* w,
                         const void* k_pool, const float* k_scale, int64_t n_pages,
                         const int32_t* block_table, int64_t bt_stride,
                         const int32_t* list, const int32_t* n_list, const int32_t* n_slots,
                         int32_t rows, float* scores, double* mags);

/* Score of a single slot for `rows` rows of one request (q_req: [rows][n_heads][d],
 * w_req: [rows][n_heads], key: [kv_heads][d]). */
void oracle_score_slot(const oracle_cfg* cfg, const void* q_req, const float* w_req,
                       const void* key, float scale, int32_t rows, float* z_out,
                       double* mag_out);

/* Post-indexer top-K (Algorithm 1's top-K step) per request and row over the scored slots. */
int oracle_topk(const oracle_cfg* cfg, const float* scores, const int32_t* list,
                const int32_t* n_list, const int32_t* n_slots, int32_t rows,
                int32_t* topk_idx);

/* EMA update (Algorithm 1's EMA update) replayed for rows 0..a in order (§3.2.2);
 * accepted == NULL means a = 0 for every request (the single-row update). */
int oracle_replay_ema(const oracle_cfg* cfg, float* V, float* D, int32_t* warm,
                      const float* scores, int32_t rows, const int32_t* list,
                      const int32_t* n_list, const int32_t* n_slots, const int32_t* q_pos,
                      const int32_t* accepted);

/* Reset after prefill / at a turn start (§3.2 practical details): zero V and D and
 * mark the request cold.  req < 0 resets every request. */
void oracle_init_state(const oracle_cfg* cfg, float* V, float* D, int32_t* warm, int32_t req);

#ifdef __cplusplus
}
#endif
#endif

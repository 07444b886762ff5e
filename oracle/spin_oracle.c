/*
 * spin_oracle.c -- plain CPU oracle of the SPIN decode-time indexer step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, loads or calls this file;
 * only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It shares
 * no code with the CUDA path.  Single-threaded, no blocking, no fusion: every
 * function follows the steps of the method in the order the paper states them.
 *
 * Paper: "SPIN: Shadow Predictive Indexer for Sparse Attention" (arXiv 2610.09025).
 *
 * Precision: the EMA state is fp32 and its update is one fixed fp32 expression,
 * t = fl((1-alpha) * z), V = fma(alpha, V, t), because the state decides the block
 * masks, which must be identical on both sides.  Indexer scores are accumulated in
 * double over the exactly decoded inputs and rounded once to float.
 *
 * Pins (each checked by a CPU test against something other than this file):
 *   oracle_philox4x64_10 ...... numpy's Philox4x64-10 bit generator (library routine)
 *   oracle_decode_e4m3 ........ torch's float8_e4m3fn conversion, all 256 codes
 *   oracle_decode_bf16 ........ torch's bfloat16 conversion
 *   oracle_budget ............. hand-derived table of Algorithm 1's budget step (golden file)
 *   oracle_explore_count ...... hand-derived table (golden file) + invariants
 *   oracle_block_scores ....... numpy reductions in the degenerate cases D = -inf and
 *                               V = -inf, and brute force on tiny inputs; the MEAN and
 *                               TOP4 poolings: numpy's mean / sorted top four where the
 *                               fp32 sums are exact (small integers), constant blocks,
 *                               one-slot blocks, max >= top-4 mean >= mean
 *   oracle_select_blocks ...... |selection| = budget, forced blocks kept, top set
 *                               dominance, exploration uniformity (chi-square),
 *                               rho = 0 gives the dense selection
 *   oracle_indexer_score ...... numpy einsum brute force; integer-valued inputs exact;
 *                               signed scales: z(s) - z(-s) is the plain dot product
 *   oracle_topk ............... numpy lexsort brute force; rho = 0 equals dense top-K
 *   oracle_replay_ema ......... closed forms of the EMA recurrence and of the
 *                               prefix-valid replay; a = 0 equals the one-row update
 * Parity unpinned: none of the functions above; the realized sparsity and miss-rate
 * diagnostics on synthetic data have no published value to compare with.
 */
#include "spin_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------
 * Philox4x64-10, from "Parallel Random Numbers: As Easy as 1, 2, 3" (Salmon, Moraes,
 * Dror, Shaw, SC'11), §4: ten rounds of two 64x64->128 multiplies, the high halves
 * xored with the other counter words and the round key, with the Weyl key schedule
 * bumped between rounds.
 * ---------------------------------------------------------------------------- */
static const uint64_t PHILOX_M0 = 0xD2E7470EE14C6C93ULL;
static const uint64_t PHILOX_M1 = 0xCA5A826395121157ULL;
static const uint64_t PHILOX_W0 = 0x9E3779B97F4A7C15ULL; /* golden ratio */
static const uint64_t PHILOX_W1 = 0xBB67AE8584CAA73BULL; /* sqrt(3) - 1 */

static void mul_hi_lo(uint64_t a, uint64_t b, uint64_t* hi, uint64_t* lo) {
    unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
    *hi = (uint64_t)(p >> 64);
    *lo = (uint64_t)p;
}

void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
    uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t hi0, lo0, hi1, lo1;
        mul_hi_lo(PHILOX_M0, c0, &hi0, &lo0);
        mul_hi_lo(PHILOX_M1, c2, &hi1, &lo1);
        uint64_t n0 = hi1 ^ c1 ^ k0;
        uint64_t n1 = lo1;
        uint64_t n2 = hi0 ^ c3 ^ k1;
        uint64_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Exploration draw of block j: one Philox4x64-10 output (256 bits) serves the eight blocks
 * 8m .. 8m+7, counter {step, row, req, m}; block j takes 32-bit half (j mod 8) in order:
 * word (j mod 8)/2, its high half first. */
uint32_t oracle_explore_key(uint64_t seed, int32_t layer, uint64_t step, int32_t row,
                            int32_t req, int64_t j) {
    uint64_t ctr[4] = {step, (uint64_t)(uint32_t)row, (uint64_t)(uint32_t)req, (uint64_t)(j >> 3)};
    uint64_t key[2] = {seed, (uint64_t)(uint32_t)layer};
    uint64_t out[4];
    oracle_philox4x64_10(ctr, key, out);
    const int h = (int)(j & 7);
    const uint64_t w = out[h >> 1];
    return (h & 1) ? (uint32_t)(w & 0xFFFFFFFFu) : (uint32_t)(w >> 32);
}

/* ------------------------------------------------------------------------------
 * Number formats.
 * E4M3 (OCP 8-bit floating point specification): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); the pattern
 * S.1111.111 is NaN and there is no infinity.
 * bfloat16: the high 16 bits of an IEEE binary32.
 * ---------------------------------------------------------------------------- */
double oracle_decode_e4m3(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

double oracle_decode_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void* base, int32_t dtype, int64_t idx) {
    switch (dtype) {
        case ORACLE_F32: return (double)((const float*)base)[idx];
        case ORACLE_BF16: return oracle_decode_bf16(((const uint16_t*)base)[idx]);
        case ORACLE_E4M3: return oracle_decode_e4m3(((const uint8_t*)base)[idx]);
        default: return NAN;
    }
}

static int64_t elem_size(int32_t dtype) {
    return dtype == ORACLE_F32 ? 4 : (dtype == ORACLE_BF16 ? 2 : 1);
}

/* ------------------------------------------------------------------------------
 * Budget (Algorithm 1's budget step): m = min{B, max(ceil(K/b), ceil((1-rho) B))}, rho in
 * integer basis points so that the ceiling is exact.
 * ---------------------------------------------------------------------------- */
int64_t oracle_budget(int64_t n_blocks, int64_t top_k, int64_t block, int32_t rho_bp) {
    int64_t floor_k = (top_k + block - 1) / block;
    int64_t keep = ((int64_t)(10000 - rho_bp) * n_blocks + 9999) / 10000;
    int64_t m = floor_k > keep ? floor_k : keep;
    return m < n_blocks ? m : n_blocks;
}

/* §3.2.1: a fraction gamma of m_t is reserved for exploration; forced blocks count
 * toward m_t and the exploration budget is capped by the remaining capacity. */
int64_t oracle_explore_count(int64_t m, int64_t n_forced, int32_t gamma_bp) {
    if (m <= n_forced) return 0;
    int64_t e = ((int64_t)gamma_bp * m) / 10000;
    int64_t cap = m - n_forced;
    return e < cap ? e : cap;
}

/* ------------------------------------------------------------------------------
 * Eq. 1 and Eq. 2 (Algorithm 1's pooling step): predicted slot score max(V[i], D[q-i])
 * (or V[i] + D[q-i] in the additive mode), max-pooled over the slots i < N of each
 * block of b slots.
 * ---------------------------------------------------------------------------- */
static float predicted_slot_score(const oracle_cfg* cfg, const float* V_req,
                                  const float* D_req, int64_t q, int64_t i) {
    float v = V_req[i];
    float d = D_req[q - i];
    if (cfg->combine == ORACLE_COMBINE_SUM) return v + d;
    return v > d ? v : d;
}

/* §4.6 (block-reduction ablation): instead of Eq. 2's max, a block's score is the mean of
 * its slots' predictions (MEAN) or the mean of the (up to) four largest (TOP4).  The pages
 * give no precision; the sums are fp32 in a fixed order, the one the GPU kernel uses, so
 * that both sides rank blocks identically:
 *   MEAN: slot l and slot l + 32 of the block are added first (a slot at or beyond N adds
 *         nothing), then the 32 pair sums pairwise at distance 16, 8, 4, 2, 1 (each step
 *         replaces t[l] by t[l] + t[l ^ d]), and the sum is divided by the count of slots < N;
 *   TOP4: the largest values t1 >= t2 >= t3 >= t4 are added as (t1 + t2) + (t3 + t4) (with
 *         fewer slots: t1, t1 + t2, (t1 + t2) + t3) and divided by their count. */
static float pool_mean(const float* p, const int* valid) {
    float t[32], u[32];
    for (int l = 0; l < 32; ++l) t[l] = (valid[l] ? p[l] : 0.0f) + (valid[l + 32] ? p[l + 32] : 0.0f);
    for (int d = 16; d >= 1; d >>= 1) {
        for (int l = 0; l < 32; ++l) u[l] = t[l] + t[l ^ d];
        memcpy(t, u, sizeof t);
    }
    int count = 0;
    for (int l = 0; l < 64; ++l) count += valid[l] != 0;
    return t[0] / (float)count;
}

static float pool_top4(const float* p, const int* valid) {
    float top[4];
    int c = 0, used[64];
    for (int l = 0; l < 64; ++l) used[l] = !valid[l];
    for (; c < 4; ++c) {  /* the largest remaining value, each slot taken once */
        int best = -1;
        for (int l = 0; l < 64; ++l)
            if (!used[l] && (best < 0 || p[l] > p[best])) best = l;
        if (best < 0) break;
        used[best] = 1;
        top[c] = p[best];
    }
    float sum = top[0];
    if (c == 2) sum = top[0] + top[1];
    if (c == 3) sum = (top[0] + top[1]) + top[2];
    if (c == 4) sum = (top[0] + top[1]) + (top[2] + top[3]);
    return sum / (float)c;
}

/* §4.6, A2: block reduction before the predictor.  The state is kept per block: Vb[j] (the
 * request's V[j]) and Db[o] (the request's D[o]) at the block offset o = floor(q / 64) - j of
 * block j from the query's block, both EMAs of the block's pooled indexer score (its max over
 * the live slots).  A block's predicted score combines them as Eq. 1 combines V and D. */
static float a2_block_score(const oracle_cfg* cfg, const float* V_req, const float* D_req,
                            int64_t q, int64_t j) {
    float v = V_req[j];
    float d = D_req[q / cfg->block - j];
    if (cfg->combine == ORACLE_COMBINE_SUM) return v + d;
    return v > d ? v : d;
}

void oracle_block_scores(const oracle_cfg* cfg, const float* V_req, const float* D_req,
                         int64_t n_slots, int64_t q, float* S_out) {
    int64_t b = cfg->block;
    int64_t nb = (n_slots + b - 1) / b;
    for (int64_t j = 0; j < nb; ++j) {
        if (cfg->pooling == ORACLE_POOL_A2) {
            S_out[j] = a2_block_score(cfg, V_req, D_req, q, j);
            continue;
        }
        int64_t lo = j * b;
        int64_t hi = (j + 1) * b < n_slots ? (j + 1) * b : n_slots;
        if (cfg->pooling == ORACLE_POOL_MEAN || cfg->pooling == ORACLE_POOL_TOP4) {
            float p[64];
            int valid[64];
            for (int64_t l = 0; l < 64; ++l) {
                valid[l] = lo + l < hi;
                p[l] = valid[l] ? predicted_slot_score(cfg, V_req, D_req, q, lo + l) : 0.0f;
            }
            S_out[j] = cfg->pooling == ORACLE_POOL_MEAN ? pool_mean(p, valid) : pool_top4(p, valid);
            continue;
        }
        float s = predicted_slot_score(cfg, V_req, D_req, q, lo);
        for (int64_t i = lo + 1; i < hi; ++i) {
            float p = predicted_slot_score(cfg, V_req, D_req, q, i);
            if (p > s) s = p;
        }
        S_out[j] = s;
    }
}

/* Sorting helpers: block top-m by (S desc, j asc); exploration by (u asc, j asc);
 * slot top-K by (z desc, i asc).  C comparison treats -0 and +0 as equal. */
typedef struct { float s; int64_t j; } score_idx;
typedef struct { uint32_t u; int64_t j; } key_idx;

static int cmp_score_desc(const void* a, const void* b) {
    const score_idx* x = (const score_idx*)a;
    const score_idx* y = (const score_idx*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

static int cmp_key_asc(const void* a, const void* b) {
    const key_idx* x = (const key_idx*)a;
    const key_idx* y = (const key_idx*)b;
    if (x->u < y->u) return -1;
    if (x->u > y->u) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

static int cmp_i32_asc(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

static int64_t max_blocks_of(const oracle_cfg* cfg) {
    return ((int64_t)cfg->max_slots + cfg->block - 1) / cfg->block;
}

static int64_t d_len_of(const oracle_cfg* cfg) {
    return (int64_t)cfg->max_slots + cfg->max_rows;
}

static int request_ok(const oracle_cfg* cfg, int64_t n, int64_t q, int32_t rows) {
    if (n < 0 || n > cfg->max_slots) return 0;
    if (n > 0 && q < n - 1) return 0;
    if (q < 0 || q + rows - 1 >= d_len_of(cfg)) return 0;
    return 1;
}

/* One query row of one request: Algorithm 1's prediction, budget and block top-m steps, the forced sink and newest
 * blocks and the warm-up rule of §3.2, and random exploration of §3.2.1.  Writes a
 * 0/1 mask of B entries; returns the number of selected blocks. */
static int64_t select_row(const oracle_cfg* cfg, const float* V_req, const float* D_req,
                          int64_t n_slots, int64_t q, int warm, int32_t rho_bp,
                          uint64_t step, int32_t layer, int32_t row, int32_t req,
                          const uint32_t* age_req, unsigned char* mask) {
    int64_t b = cfg->block;
    int64_t nb = (n_slots + b - 1) / b;                      /* block count */
    memset(mask, 0, (size_t)(nb > 0 ? nb : 1));
    if (nb == 0) return 0;
    if (!warm) {                                             /* first step after a reset */
        memset(mask, 1, (size_t)nb);
        return nb;
    }
    if (cfg->pooling == ORACLE_POOL_SLOTS) {
        /* §4.6, A0: the K slots with the largest predicted scores (equal scores: lower slot),
         * then every block holding one of them, with the sink and newest blocks; no
         * exploration.  A budget of every block still selects every block. */
        if (oracle_budget(nb, cfg->top_k, b, rho_bp) >= nb) {
            memset(mask, 1, (size_t)nb);
            return nb;
        }
        score_idx* sl = (score_idx*)malloc(sizeof(score_idx) * (size_t)n_slots);
        for (int64_t i = 0; i < n_slots; ++i) {
            sl[i].s = predicted_slot_score(cfg, V_req, D_req, q, i);
            sl[i].j = i;
        }
        qsort(sl, (size_t)n_slots, sizeof(score_idx), cmp_score_desc);
        mask[0] = 1;
        mask[nb - 1] = 1;
        for (int64_t k = 0; k < cfg->top_k && k < n_slots; ++k) mask[sl[k].j / b] = 1;
        free(sl);
        int64_t cnt = 0;
        for (int64_t j = 0; j < nb; ++j) cnt += mask[j];
        return cnt;
    }
    float* S = (float*)malloc(sizeof(float) * (size_t)nb);  /* predict and pool */
    oracle_block_scores(cfg, V_req, D_req, n_slots, q, S);
    int64_t m = oracle_budget(nb, cfg->top_k, b, rho_bp);    /* budget */

    mask[0] = 1;                                             /* sink block */
    mask[nb - 1] = 1;                                        /* newest active block */
    int64_t f = nb > 1 ? 2 : 1;
    int64_t e = oracle_explore_count(m, f, cfg->gamma_bp);
    int64_t t = m > f ? m - f - e : 0;                       /* top-ranked share */

    /* block top-m over the blocks that are not forced */
    score_idx* cand = (score_idx*)malloc(sizeof(score_idx) * (size_t)nb);
    int64_t nc = 0;
    for (int64_t j = 0; j < nb; ++j)
        if (!mask[j]) { cand[nc].s = S[j]; cand[nc].j = j; ++nc; }
    qsort(cand, (size_t)nc, sizeof(score_idx), cmp_score_desc);
    for (int64_t k = 0; k < t && k < nc; ++k) mask[cand[k].j] = 1;

    /* exploration: e distinct blocks drawn uniformly from the ones not yet selected, as the
     * e smallest counter-based random keys; or (block age, §4.6) the e observed least
     * recently, as the e smallest ages */
    if (e > 0) {
        key_idx* ex = (key_idx*)malloc(sizeof(key_idx) * (size_t)nb);
        int64_t ne = 0;
        for (int64_t j = 0; j < nb; ++j)
            if (!mask[j]) {
                ex[ne].u = age_req ? age_req[j] : oracle_explore_key(cfg->seed, layer, step, row, req, j);
                ex[ne].j = j;
                ++ne;
            }
        qsort(ex, (size_t)ne, sizeof(key_idx), cmp_key_asc);
        for (int64_t k = 0; k < e && k < ne; ++k) mask[ex[k].j] = 1;
        free(ex);
    }
    free(cand);
    free(S);
    int64_t cnt = 0;
    for (int64_t j = 0; j < nb; ++j) cnt += mask[j];
    return cnt;
}

static int select_impl(const oracle_cfg* cfg, const float* V, const float* D,
                       const int32_t* warm, const int32_t* n_slots, const int32_t* q_pos,
                       int32_t rows, int32_t rho_bp, uint64_t step, int32_t layer,
                       const uint32_t* age, int32_t* blocks, int32_t* n_blocks,
                       int32_t* union_blocks, int32_t* n_union) {
    int64_t MB = max_blocks_of(cfg);
    int64_t DL = d_len_of(cfg);
    int bad = 0;
    if (rho_bp < 0) rho_bp = cfg->rho_bp;
    if (cfg->pooling == ORACLE_POOL_A2 && rows != 1) return -1;  /* A2: one query row */
    if ((cfg->explore == ORACLE_EXPLORE_AGE) != (age != NULL)) return -1;
    if (cfg->explore == ORACLE_EXPLORE_AGE && rows != 1) return -1;  /* block age: one row */
    unsigned char* mask = (unsigned char*)malloc((size_t)MB + 1);
    unsigned char* umask = (unsigned char*)malloc((size_t)MB + 1);
    for (int32_t req = 0; req < cfg->n_req; ++req) {
        int64_t n = n_slots[req];
        int64_t q = q_pos[req];
        memset(umask, 0, (size_t)MB + 1);
        int ok = request_ok(cfg, n, q, rows);
        if (!ok) bad = 1;
        int64_t nb = ok ? (n + cfg->block - 1) / cfg->block : 0;
        for (int32_t r = 0; r < rows; ++r) {
            int32_t* out = blocks + ((int64_t)req * rows + r) * MB;
            int64_t cnt = 0;
            if (ok) {
                select_row(cfg, V + (int64_t)req * cfg->max_slots, D + (int64_t)req * DL,
                           n, q + r, warm[req], rho_bp, step, layer, r, req,
                           age ? age + (int64_t)req * MB : NULL, mask);
                for (int64_t j = 0; j < nb; ++j)
                    if (mask[j]) { out[cnt++] = (int32_t)j; umask[j] = 1; }
            }
            n_blocks[(int64_t)req * rows + r] = (int32_t)cnt;
        }
        if (union_blocks && n_union) {
            int32_t* out = union_blocks + (int64_t)req * MB;
            int64_t cnt = 0;
            for (int64_t j = 0; j < nb; ++j)
                if (umask[j]) out[cnt++] = (int32_t)j;
            n_union[req] = (int32_t)cnt;
        }
    }
    free(mask);
    free(umask);
    return bad ? -1 : 0;
}

int oracle_select_blocks(const oracle_cfg* cfg, const float* V, const float* D,
                         const int32_t* warm, const int32_t* n_slots, const int32_t* q_pos,
                         int32_t rows, int32_t rho_bp, uint64_t step, int32_t layer,
                         int32_t* blocks, int32_t* n_blocks,
                         int32_t* union_blocks, int32_t* n_union) {
    return select_impl(cfg, V, D, warm, n_slots, q_pos, rows, rho_bp, step, layer, NULL, blocks, n_blocks,
                       union_blocks, n_union);
}

int oracle_select_blocks_age(const oracle_cfg* cfg, const float* V, const float* D,
                             const int32_t* warm, const int32_t* n_slots, const int32_t* q_pos,
                             int32_t rows, int32_t rho_bp, uint64_t step, int32_t layer,
                             const uint32_t* age, int32_t* blocks, int32_t* n_blocks,
                             int32_t* union_blocks, int32_t* n_union) {
    if (!age) return -1;
    return select_impl(cfg, V, D, warm, n_slots, q_pos, rows, rho_bp, step, layer, age, blocks, n_blocks,
                       union_blocks, n_union);
}

/* §4.6 "Staleness mitigation", block age: the listed blocks (those inside the context) were
 * observed at this decode step. */
int oracle_block_age_update(const oracle_cfg* cfg, uint32_t* age, const int32_t* list,
                            const int32_t* n_list, const int32_t* n_slots, uint64_t step) {
    int64_t MB = max_blocks_of(cfg);
    int bad = 0;
    for (int32_t req = 0; req < cfg->n_req; ++req) {
        int64_t n = n_slots[req], cnt = n_list[req];
        if (n < 0 || n > cfg->max_slots || cnt < 0 || cnt > MB) { bad = 1; continue; }
        int64_t nb = (n + cfg->block - 1) / cfg->block;
        for (int64_t k = 0; k < cnt; ++k) {
            int64_t blk = list[(int64_t)req * MB + k];
            if (blk < 0 || blk >= nb) { bad = 1; continue; }
            age[(int64_t)req * MB + blk] = (uint32_t)(step + 1);
        }
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------
 * Indexer score, §2: z_t[i] = sum_h w_h ReLU(q_{t,h} . k_{i,h}); with a per-slot
 * FP8 scale s_i the dot product is multiplied by s_i before the ReLU.  A shared key
 * (kv_heads == 1) is used by every head.
 * ---------------------------------------------------------------------------- */
static void score_slot_impl(const oracle_cfg* cfg, const void* q_req, const float* w_req,
                            const void* key, int64_t key_off, double scale, int32_t rows,
                            float* z_out, double* mag_out) {
    int64_t H = cfg->n_heads, d = cfg->head_dim;
    for (int32_t r = 0; r < rows; ++r) {
        double z = 0.0, mag = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            int64_t kh = cfg->kv_heads == 1 ? 0 : h;
            double dot = 0.0, adot = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                double qv = load_elem(q_req, cfg->q_dtype, ((int64_t)r * H + h) * d + c);
                double kv = load_elem(key, cfg->k_dtype, key_off + kh * d + c);
                dot += qv * kv;
                adot += fabs(qv * kv);
            }
            double x = scale * dot;
            double wh = (double)w_req[(int64_t)r * H + h];
            z += wh * (x > 0.0 ? x : 0.0);
            mag += fabs(wh) * fabs(scale) * adot;
        }
        z_out[r] = (float)z;
        if (mag_out) mag_out[r] = mag;
    }
}

void oracle_score_slot(const oracle_cfg* cfg, const void* q_req, const float* w_req,
                       const void* key, float scale, int32_t rows, float* z_out,
                       double* mag_out) {
    score_slot_impl(cfg, q_req, w_req, key, 0, (double)scale, rows, z_out, mag_out);
}

int oracle_indexer_score(const oracle_cfg* cfg, const void* q, const float* w,
                         const void* k_pool, const float* k_scale, int64_t n_pages,
                         const int32_t* block_table, int64_t bt_stride,
                         const int32_t* list, const int32_t* n_list, const int32_t* n_slots,
                         int32_t rows, float* scores, double* mags) {
    int64_t MB = max_blocks_of(cfg);
    int64_t b = cfg->block, H = cfg->n_heads, d = cfg->head_dim;
    int64_t slot_elems = (int64_t)cfg->kv_heads * d;
    int64_t q_elems = (int64_t)rows * H * d;
    int64_t qsz = elem_size(cfg->q_dtype);
    int bad = 0;
    float z[64];
    double mg[64];
    for (int32_t req = 0; req < cfg->n_req; ++req) {
        int64_t n = n_slots[req];
        int64_t cnt = n_list[req];
        if (n < 0 || n > cfg->max_slots || cnt < 0 || cnt > MB) { bad = 1; continue; }
        const void* q_req = (const char*)q + (int64_t)req * q_elems * qsz;
        const float* w_req = w + (int64_t)req * rows * H;
        for (int64_t k = 0; k < cnt; ++k) {
            int64_t blk = list[(int64_t)req * MB + k];
            int64_t page = (blk >= 0 && blk < MB) ? block_table[(int64_t)req * bt_stride + blk] : -1;
            int valid_page = page >= 0 && page < n_pages;
            if (!valid_page) bad = 1;
            for (int64_t s = 0; s < b; ++s) {
                int64_t i = blk * b + s;
                int scored = valid_page && i < n;
                if (scored) {
                    int64_t slot = page * b + s;
                    double scale = k_scale ? (double)k_scale[slot] : 1.0;
                    score_slot_impl(cfg, q_req, w_req, k_pool, slot * slot_elems, scale,
                                    rows, z, mg);
                }
                for (int32_t r = 0; r < rows; ++r) {
                    int64_t o = (((int64_t)req * rows + r) * MB + k) * b + s;
                    scores[o] = scored ? z[r] : 0.0f;
                    if (mags) mags[o] = scored ? mg[r] : 0.0;
                }
            }
        }
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------
 * Post-indexer top-K (Algorithm 1's top-K step) over the slots that were scored: the K
 * largest scores, equal scores ordered by the lower slot id; returned in ascending
 * slot order, padded with -1 when fewer than K slots were scored.
 * ---------------------------------------------------------------------------- */
int oracle_topk(const oracle_cfg* cfg, const float* scores, const int32_t* list,
                const int32_t* n_list, const int32_t* n_slots, int32_t rows,
                int32_t* topk_idx) {
    int64_t MB = max_blocks_of(cfg);
    int64_t b = cfg->block, K = cfg->top_k;
    int bad = 0;
    score_idx* cand = (score_idx*)malloc(sizeof(score_idx) * (size_t)(MB * b + 1));
    int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K + 1));
    for (int32_t req = 0; req < cfg->n_req; ++req) {
        int64_t n = n_slots[req];
        int64_t cnt = n_list[req];
        if (n < 0 || n > cfg->max_slots || cnt < 0 || cnt > MB) { bad = 1; cnt = 0; }
        for (int32_t r = 0; r < rows; ++r) {
            int64_t nc = 0;
            for (int64_t k = 0; k < cnt; ++k) {
                int64_t blk = list[(int64_t)req * MB + k];
                for (int64_t s = 0; s < b; ++s) {
                    int64_t i = blk * b + s;
                    if (i >= n) continue;
                    cand[nc].s = scores[(((int64_t)req * rows + r) * MB + k) * b + s];
                    cand[nc].j = i;
                    ++nc;
                }
            }
            qsort(cand, (size_t)nc, sizeof(score_idx), cmp_score_desc);
            int64_t take = nc < K ? nc : K;
            for (int64_t k = 0; k < take; ++k) sel[k] = (int32_t)cand[k].j;
            qsort(sel, (size_t)take, sizeof(int32_t), cmp_i32_asc);
            int32_t* out = topk_idx + ((int64_t)req * rows + r) * K;
            for (int64_t k = 0; k < K; ++k) out[k] = k < take ? sel[k] : -1;
        }
    }
    free(sel);
    free(cand);
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------
 * EMA update, Algorithm 1's EMA update: for every scored slot i,
 *   V[i] <- alpha V[i] + (1-alpha) z[i],   D[q-i] <- alpha D[q-i] + (1-alpha) z[i].
 * §3.2.2: with a accepted drafts the observations of rows 0..a are replayed in order
 * (row r at query position q + r); rows above a are discarded.
 * ---------------------------------------------------------------------------- */
int oracle_replay_ema(const oracle_cfg* cfg, float* V, float* D, int32_t* warm,
                      const float* scores, int32_t rows, const int32_t* list,
                      const int32_t* n_list, const int32_t* n_slots, const int32_t* q_pos,
                      const int32_t* accepted) {
    int64_t MB = max_blocks_of(cfg);
    int64_t DL = d_len_of(cfg);
    int64_t b = cfg->block;
    const float alpha = cfg->alpha;
    const float one_minus_alpha = 1.0f - alpha;
    int bad = 0;
    for (int32_t req = 0; req < cfg->n_req; ++req) {
        int64_t n = n_slots[req];
        int64_t q = q_pos[req];
        int64_t cnt = n_list[req];
        int64_t a = accepted ? accepted[req] : 0;
        if (!request_ok(cfg, n, q, rows) || cnt < 0 || cnt > MB || a < 0 || a >= rows) {
            bad = 1;
            continue;
        }
        float* V_req = V + (int64_t)req * cfg->max_slots;
        float* D_req = D + (int64_t)req * DL;
        if (cfg->pooling == ORACLE_POOL_A2) {
            /* §4.6, A2: one observation per scored block, its max over the live slots (one
             * query row) */
            if (rows != 1) { bad = 1; continue; }
            for (int64_t k = 0; k < cnt; ++k) {
                int64_t blk = list[(int64_t)req * MB + k];
                float zb = 0.0f;
                int seen = 0;
                for (int64_t s = 0; s < b; ++s) {
                    int64_t i = blk * b + s;
                    if (i >= n) continue;
                    float z = scores[((int64_t)req * MB + k) * b + s];
                    if (!seen || z > zb) zb = z;
                    seen = 1;
                }
                if (!seen) continue;
                float t = one_minus_alpha * zb;
                V_req[blk] = fmaf(alpha, V_req[blk], t);
                D_req[q / b - blk] = fmaf(alpha, D_req[q / b - blk], t);
            }
            warm[req] = 1;
            continue;
        }
        for (int64_t r = 0; r <= a; ++r) {
            for (int64_t k = 0; k < cnt; ++k) {
                int64_t blk = list[(int64_t)req * MB + k];
                for (int64_t s = 0; s < b; ++s) {
                    int64_t i = blk * b + s;
                    if (i >= n) continue;
                    float z = scores[(((int64_t)req * rows + r) * MB + k) * b + s];
                    float t = one_minus_alpha * z;
                    V_req[i] = fmaf(alpha, V_req[i], t);
                    D_req[q + r - i] = fmaf(alpha, D_req[q + r - i], t);
                }
            }
        }
        warm[req] = 1;
    }
    return bad ? -1 : 0;
}

void oracle_init_state(const oracle_cfg* cfg, float* V, float* D, int32_t* warm, int32_t req) {
    int64_t DL = d_len_of(cfg);
    for (int32_t r = 0; r < cfg->n_req; ++r) {
        if (req >= 0 && r != req) continue;
        memset(V + (int64_t)r * cfg->max_slots, 0, sizeof(float) * (size_t)cfg->max_slots);
        memset(D + (int64_t)r * DL, 0, sizeof(float) * (size_t)DL);
        warm[r] = 0;
    }
}

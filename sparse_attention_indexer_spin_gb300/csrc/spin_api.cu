// spin_api.cu -- the C ABI (include/spin.h): host-side validation and kernel dispatch.
//
// Every entry point validates what the host can see (configuration, sizes, pointers),
// records a message for spin_last_error_string() on failure, and otherwise enqueues the
// kernels on the caller's stream.  Nothing is allocated, nothing is synchronised.
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include <cmath>

#include "spin_common.cuh"
#include "spin_internal.h"

namespace spin {

static thread_local char g_err[512];

static spin_status_t fail(spin_status_t code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

static spin_status_t cuda_fail(cudaError_t e, const char* what) {
    return fail(SPIN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    return n;
}

static spin_status_t check_cfg(const spin_config* c) {
    g_err[0] = 0;
    if (!c) return fail(SPIN_ERR_INVALID_ARG, "cfg is NULL");
    if (c->block != kBlock) return fail(SPIN_ERR_INVALID_ARG, "block must be %d (got %d)", kBlock, c->block);
    if (c->n_req < 1 || c->n_req > 65535) return fail(SPIN_ERR_INVALID_ARG, "n_req %d outside [1, 65535]", c->n_req);
    if (c->max_slots < 1 || c->max_slots > (1 << 24))
        return fail(SPIN_ERR_CAPACITY, "max_slots %d outside [1, 2^24]", c->max_slots);
    if (c->max_rows < 1 || c->max_rows > kMaxRows)
        return fail(SPIN_ERR_INVALID_ARG, "max_rows %d outside [1, %d]", c->max_rows, kMaxRows);
    if (c->n_heads < 1 || c->n_heads > 128) return fail(SPIN_ERR_INVALID_ARG, "n_heads %d outside [1, 128]", c->n_heads);
    if (c->head_dim < 1 || c->head_dim > 256)
        return fail(SPIN_ERR_INVALID_ARG, "head_dim %d outside [1, 256]", c->head_dim);
    if (c->kv_heads != 1 && c->kv_heads != c->n_heads)
        return fail(SPIN_ERR_SHAPE, "kv_heads must be 1 or n_heads (got %d, n_heads %d)", c->kv_heads, c->n_heads);
    if (c->q_dtype != SPIN_DTYPE_F32 && c->q_dtype != SPIN_DTYPE_BF16)
        return fail(SPIN_ERR_UNSUPPORTED, "q_dtype %d: F32 or BF16 only", c->q_dtype);
    if (c->k_dtype != SPIN_DTYPE_F32 && c->k_dtype != SPIN_DTYPE_BF16 && c->k_dtype != SPIN_DTYPE_E4M3)
        return fail(SPIN_ERR_UNSUPPORTED, "k_dtype %d: F32, BF16 or E4M3 only", c->k_dtype);
    if (c->top_k < 1 || c->top_k > 16384) return fail(SPIN_ERR_INVALID_ARG, "top_k %d outside [1, 16384]", c->top_k);
    if (c->rho_bp < 0 || c->rho_bp > 10000) return fail(SPIN_ERR_INVALID_ARG, "rho_bp %d outside [0, 10000]", c->rho_bp);
    if (c->gamma_bp < 0 || c->gamma_bp > 10000)
        return fail(SPIN_ERR_INVALID_ARG, "gamma_bp %d outside [0, 10000]", c->gamma_bp);
    if (!(c->alpha >= 0.0f && c->alpha <= 1.0f)) return fail(SPIN_ERR_INVALID_ARG, "alpha outside [0, 1]");
    if (c->combine != SPIN_COMBINE_MAX && c->combine != SPIN_COMBINE_SUM)
        return fail(SPIN_ERR_INVALID_ARG, "combine %d unknown", c->combine);
    if (c->score_path < SPIN_SCORE_AUTO || c->score_path > SPIN_SCORE_TCGEN05)
        return fail(SPIN_ERR_INVALID_ARG, "score_path %d unknown", c->score_path);
    if (c->pooling < SPIN_POOL_MAX || c->pooling > SPIN_POOL_A2)
        return fail(SPIN_ERR_INVALID_ARG, "pooling %d unknown", c->pooling);
    if (c->explore < SPIN_EXPLORE_RANDOM || c->explore > SPIN_EXPLORE_BLOCK_AGE)
        return fail(SPIN_ERR_INVALID_ARG, "explore %d unknown", c->explore);
    if (c->reserved != 0) return fail(SPIN_ERR_INVALID_ARG, "reserved must be 0");
    return SPIN_OK;
}

static spin_status_t check_rows(const spin_config* c, int rows) {
    if (rows < 1 || rows > c->max_rows) return fail(SPIN_ERR_SHAPE, "rows %d outside [1, max_rows=%d]", rows, c->max_rows);
    if ((int64_t)c->n_req * rows > 65535) return fail(SPIN_ERR_CAPACITY, "n_req * rows above 65535");
    if (c->pooling == SPIN_POOL_A2 && rows > 1)
        return fail(SPIN_ERR_UNSUPPORTED, "the A2 ablation keeps block-level state for one query row");
    if (c->explore == SPIN_EXPLORE_BLOCK_AGE && rows > 1)
        return fail(SPIN_ERR_UNSUPPORTED, "block-age exploration keeps one age per block: one query row");
    return SPIN_OK;
}

static spin_status_t launched(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return SPIN_OK;
    return cuda_fail(e, what);
}

}  // namespace spin

using namespace spin;

extern "C" {

spin_status_t spin_init_state(const spin_config* cfg, float* V, float* D, float* Vmax, int32_t* warm, int32_t req,
                              spin_stream_t stream) {
    spin_status_t st = check_cfg(cfg);
    if (st) return st;
    if (!V || !D || !Vmax || !warm) return fail(SPIN_ERR_INVALID_ARG, "V, D, Vmax and warm must be non-NULL");
    if (req >= cfg->n_req) return fail(SPIN_ERR_INVALID_ARG, "req %d >= n_req %d", req, cfg->n_req);
    return launched(launch_init_state(*cfg, V, D, Vmax, warm, req, (cudaStream_t)stream), "spin_init_state");
}

spin_status_t spin_workspace_size(const spin_config* cfg, int32_t rows, size_t* bytes) {
    spin_status_t st = check_cfg(cfg);
    if (st) return st;
    if ((st = check_rows(cfg, rows))) return st;
    if (!bytes) return fail(SPIN_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = select_workspace_bytes(*cfg, rows);
    return SPIN_OK;
}

static spin_status_t check_layers(int32_t n_layers) {
    if (n_layers < 1 || n_layers > 1024) return fail(SPIN_ERR_INVALID_ARG, "n_layers %d outside [1, 1024]", n_layers);
    return SPIN_OK;
}

static spin_status_t select_impl(const spin_config* cfg, const float* V, const float* D, const float* Vmax,
                                 const int32_t* warm, const int32_t* n_slots, const int32_t* q_pos, int32_t rows,
                                 const int32_t* rho_override, uint64_t step, const uint64_t* step_dev, int32_t layer,
                                 int32_t* blocks, int32_t* n_blocks, int32_t* union_blocks, int32_t* n_union,
                                 void* workspace, size_t workspace_bytes, uint32_t* status, spin_stream_t stream,
                                 int32_t n_layers = 1, const uint32_t* block_age = nullptr) {
    spin_status_t st = check_cfg(cfg);
    if (st) return st;
    if ((st = check_rows(cfg, rows))) return st;
    if ((st = check_layers(n_layers))) return st;
    if ((cfg->explore == SPIN_EXPLORE_BLOCK_AGE) != (block_age != nullptr))
        return fail(SPIN_ERR_INVALID_ARG, cfg->explore == SPIN_EXPLORE_BLOCK_AGE
                                              ? "block-age exploration needs spin_select_blocks_age and an age array"
                                              : "an age array needs explore = SPIN_EXPLORE_BLOCK_AGE");
    const Dims dm = dims_of(*cfg);
    if (dm.MB > kSelectMaxBlocks)
        return fail(SPIN_ERR_CAPACITY, "max_slots %d needs %d blocks; selection supports %d", cfg->max_slots, dm.MB,
                    kSelectMaxBlocks);
    if (!V || !D || !Vmax || !warm || !n_slots || !q_pos || !blocks || !n_blocks)
        return fail(SPIN_ERR_INVALID_ARG, "a required pointer is NULL");
    if (rows > 1 && (!union_blocks || !n_union))
        return fail(SPIN_ERR_INVALID_ARG, "rows > 1 needs union_blocks and n_union");
    if ((union_blocks == nullptr) != (n_union == nullptr))
        return fail(SPIN_ERR_INVALID_ARG, "union_blocks and n_union go together");
    const size_t need = (size_t)n_layers * select_workspace_bytes(*cfg, rows);
    if (!workspace || workspace_bytes < need)
        return fail(SPIN_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu)", need, workspace_bytes);
    if (((uintptr_t)workspace & 255) != 0) return fail(SPIN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    SelectArgs a{V, D, Vmax, warm, n_slots, q_pos, rows, rho_override, step, step_dev, layer, blocks, n_blocks,
                 union_blocks, n_union, reinterpret_cast<float*>(workspace), status, n_layers, block_age};
    return launched(launch_select(*cfg, a, (cudaStream_t)stream), "spin_select_blocks");
}

spin_status_t spin_select_blocks(const spin_config* cfg, const float* V, const float* D, const float* Vmax,
                                 const int32_t* warm, const int32_t* n_slots, const int32_t* q_pos, int32_t rows,
                                 const int32_t* rho_override, uint64_t step, int32_t layer, int32_t* blocks,
                                 int32_t* n_blocks, int32_t* union_blocks, int32_t* n_union, void* workspace,
                                 size_t workspace_bytes, uint32_t* status, spin_stream_t stream) {
    return select_impl(cfg, V, D, Vmax, warm, n_slots, q_pos, rows, rho_override, step, nullptr, layer, blocks,
                       n_blocks, union_blocks, n_union, workspace, workspace_bytes, status, stream);
}

spin_status_t spin_select_blocks_layers(const spin_config* cfg, int32_t n_layers, int32_t layer0, const float* V,
                                        const float* D, const float* Vmax, const int32_t* warm,
                                        const int32_t* n_slots, const int32_t* q_pos, int32_t rows,
                                        const int32_t* rho_override, uint64_t step, const uint64_t* step_dev,
                                        int32_t* blocks, int32_t* n_blocks, int32_t* union_blocks, int32_t* n_union,
                                        void* workspace, size_t workspace_bytes, uint32_t* status,
                                        spin_stream_t stream) {
    return select_impl(cfg, V, D, Vmax, warm, n_slots, q_pos, rows, rho_override, step, step_dev, layer0, blocks,
                       n_blocks, union_blocks, n_union, workspace, workspace_bytes, status, stream, n_layers);
}

spin_status_t spin_select_blocks_age(const spin_config* cfg, const float* V, const float* D, const float* Vmax,
                                     const int32_t* warm, const int32_t* n_slots, const int32_t* q_pos, int32_t rows,
                                     const int32_t* rho_override, uint64_t step, int32_t layer,
                                     const uint32_t* block_age, int32_t* blocks, int32_t* n_blocks,
                                     int32_t* union_blocks, int32_t* n_union, void* workspace,
                                     size_t workspace_bytes, uint32_t* status, spin_stream_t stream) {
    g_err[0] = 0;
    if (!block_age) return fail(SPIN_ERR_INVALID_ARG, "block_age is NULL");
    return select_impl(cfg, V, D, Vmax, warm, n_slots, q_pos, rows, rho_override, step, nullptr, layer, blocks,
                       n_blocks, union_blocks, n_union, workspace, workspace_bytes, status, stream, 1, block_age);
}

spin_status_t spin_select_blocks_dstep(const spin_config* cfg, const float* V, const float* D, const float* Vmax,
                                       const int32_t* warm, const int32_t* n_slots, const int32_t* q_pos,
                                       int32_t rows, const int32_t* rho_override, const uint64_t* step_dev,
                                       int32_t layer, int32_t* blocks, int32_t* n_blocks, int32_t* union_blocks,
                                       int32_t* n_union, void* workspace, size_t workspace_bytes, uint32_t* status,
                                       spin_stream_t stream) {
    if (!step_dev) return fail(SPIN_ERR_INVALID_ARG, "step_dev is NULL");
    return select_impl(cfg, V, D, Vmax, warm, n_slots, q_pos, rows, rho_override, 0, step_dev, layer, blocks,
                       n_blocks, union_blocks, n_union, workspace, workspace_bytes, status, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Allocation-free selection: the block-score scratch lives in this static device array
// instead of a caller workspace, for callers that cannot allocate device memory.  The
// array's device address is looked up once per device (with that device current) on the
// first call and cached; calls that overlap on one device race on the array.
// ---------------------------------------------------------------------------------------
namespace spin {

constexpr size_t kNoAllocScratchEntries = (size_t)1 << 20;  // block-row entries of each of its two arrays
static __device__ __align__(256) float g_select_scratch[2 * kNoAllocScratchEntries];  // 8 MiB

constexpr int kMaxDevices = 128;
static std::mutex g_scratch_mu;
static float* g_scratch_addr[kMaxDevices];

static spin_status_t scratch_of_current_device(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "spin_select_blocks_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(SPIN_ERR_CAPACITY, "device ordinal %d above %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_select_scratch);
        if (e != cudaSuccess || p == nullptr)
            return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                             "spin_select_blocks_noalloc: cudaGetSymbolAddress of the scratch array");
        g_scratch_addr[dev] = reinterpret_cast<float*>(p);
    }
    *out = g_scratch_addr[dev];
    return SPIN_OK;
}

}  // namespace spin

extern "C" {

spin_status_t spin_select_blocks_noalloc(const spin_config* cfg, const float* V, const float* D, const float* Vmax,
                                         const int32_t* warm, const int32_t* n_slots, const int32_t* q_pos,
                                         int32_t rows, const int32_t* rho_override, uint64_t step, int32_t layer,
                                         int32_t* blocks, int32_t* n_blocks, int32_t* union_blocks,
                                         int32_t* n_union, uint32_t* status, spin_stream_t stream) {
    spin_status_t st = check_cfg(cfg);
    if (st) return st;
    if ((st = check_rows(cfg, rows))) return st;
    if (cfg->explore == SPIN_EXPLORE_BLOCK_AGE)
        return fail(SPIN_ERR_INVALID_ARG, "block-age exploration needs spin_select_blocks_age and an age array");
    const Dims dm = dims_of(*cfg);
    if (dm.MB > kSelectMaxBlocks)
        return fail(SPIN_ERR_CAPACITY, "max_slots %d needs %d blocks; selection supports %d", cfg->max_slots, dm.MB,
                    kSelectMaxBlocks);
    const size_t need = (size_t)dm.R * (size_t)rows * (size_t)dm.MB;
    if (need > kNoAllocScratchEntries || select_workspace_bytes(*cfg, rows) > sizeof(g_select_scratch))
        return fail(SPIN_ERR_CAPACITY,
                    "spin_select_blocks_noalloc: n_req * rows * max_blocks = %zu exceeds its built-in scratch of %zu "
                    "entries; use spin_select_blocks with a workspace",
                    need, kNoAllocScratchEntries);
    if (!V || !D || !Vmax || !warm || !n_slots || !q_pos || !blocks || !n_blocks)
        return fail(SPIN_ERR_INVALID_ARG, "a required pointer is NULL");
    if (rows > 1 && (!union_blocks || !n_union))
        return fail(SPIN_ERR_INVALID_ARG, "rows > 1 needs union_blocks and n_union");
    if ((union_blocks == nullptr) != (n_union == nullptr))
        return fail(SPIN_ERR_INVALID_ARG, "union_blocks and n_union go together");
    float* scratch = nullptr;
    if ((st = scratch_of_current_device(&scratch))) return st;
    SelectArgs a{V, D, Vmax, warm, n_slots, q_pos, rows, rho_override, step, nullptr, layer, blocks, n_blocks,
                 union_blocks, n_union, scratch, status, 1};
    return launched(launch_select(*cfg, a, (cudaStream_t)stream), "spin_select_blocks_noalloc");
}

static spin_status_t check_hint(const spin_config* cfg, int32_t rows, const void* hint, size_t hint_bytes) {
    if (!topk_hint_supported(*cfg))
        return fail(SPIN_ERR_UNSUPPORTED, "no hinted top-K for top_k %d with %d blocks (needs top_k <= 2048 and "
                    "at most 8192 blocks)", cfg->top_k, dims_of(*cfg).MB);
    if (!hint) return fail(SPIN_ERR_INVALID_ARG, "hint is NULL");
    if (((uintptr_t)hint & 255) != 0) return fail(SPIN_ERR_INVALID_ARG, "hint must be 256-byte aligned");
    const size_t need = topk_hint_bytes(*cfg, rows);
    if (hint_bytes < need) return fail(SPIN_ERR_INVALID_ARG, "hint of %zu bytes needed (got %zu)", need, hint_bytes);
    return SPIN_OK;
}

static spin_status_t score_impl(const spin_config* cfg, const void* q, const float* w, const void* k_pool,
                                const float* k_scale, int64_t n_pages, const int32_t* block_table, int64_t bt_stride,
                                const int32_t* list, const int32_t* n_list, const int32_t* n_slots, int32_t rows,
                                float* scores, const spin_score_extras* ex, uint32_t* status, spin_stream_t stream) {
    spin_status_t st = check_cfg(cfg);
    if (st) return st;
    if ((st = check_rows(cfg, rows))) return st;
    HintArgs hint{nullptr, nullptr, 0};
    if (ex && ex->topk_hint) {
        if ((st = check_hint(cfg, rows, ex->topk_hint, ex->topk_hint_bytes))) return st;
        hint = topk_hint_args(*cfg, rows, ex->topk_hint);
    }
    const Dims dm = dims_of(*cfg);
    if (!q || !w || !k_pool || !block_table || !list || !n_list || !n_slots || !scores)
        return fail(SPIN_ERR_INVALID_ARG, "a required pointer is NULL");
    if (cfg->k_dtype == SPIN_DTYPE_E4M3 && !k_scale) return fail(SPIN_ERR_INVALID_ARG, "E4M3 keys need k_scale");
    if (n_pages < 0) return fail(SPIN_ERR_INVALID_ARG, "n_pages < 0");
    if (bt_stride < dm.MB) return fail(SPIN_ERR_SHAPE, "bt_stride %lld < max blocks %d", (long long)bt_stride, dm.MB);
    if (((uintptr_t)k_pool & 15) != 0 || (k_scale && ((uintptr_t)k_scale & 15) != 0))
        return fail(SPIN_ERR_INVALID_ARG, "k_pool and k_scale must be 16-byte aligned");
    ScoreArgs a{q, w, k_pool, cfg->k_dtype == SPIN_DTYPE_E4M3 ? k_scale : nullptr, n_pages, block_table, bt_stride,
                list, n_list, n_slots, rows, scores, status, hint};
    int path = cfg->score_path;
    if (path == SPIN_SCORE_AUTO) {
        if (score_tc_supported(*cfg, rows)) path = SPIN_SCORE_TCGEN05;
        else if (score_stream_supported(*cfg, rows)) path = SPIN_SCORE_STREAM;
        else path = SPIN_SCORE_GENERIC;
    }
    cudaStream_t s = (cudaStream_t)stream;
    switch (path) {
        case SPIN_SCORE_GENERIC:
            return launched(launch_score_generic(*cfg, a, s), "spin_indexer_score (generic)");
        case SPIN_SCORE_STREAM:
            if (!score_stream_supported(*cfg, rows))
                return fail(SPIN_ERR_UNSUPPORTED, "no streaming kernel for this shape (needs per-head keys)");
            return launched(launch_score_stream(*cfg, a, s), "spin_indexer_score (stream)");
        case SPIN_SCORE_TCGEN05:
            if (!score_tc_supported(*cfg, rows))
                return fail(SPIN_ERR_UNSUPPORTED, "no tcgen05 kernel for this shape (needs a shared key)");
            return launched(launch_score_tc(*cfg, a, s), "spin_indexer_score (tcgen05)");
    }
    return fail(SPIN_ERR_INVALID_ARG, "score_path");
}

spin_status_t spin_indexer_score(const spin_config* cfg, const void* q, const float* w, const void* k_pool,
                                 const float* k_scale, int64_t n_pages, const int32_t* block_table, int64_t bt_stride,
                                 const int32_t* list, const int32_t* n_list, const int32_t* n_slots, int32_t rows,
                                 float* scores, uint32_t* status, spin_stream_t stream) {
    return score_impl(cfg, q, w, k_pool, k_scale, n_pages, block_table, bt_stride, list, n_list, n_slots, rows,
                      scores, nullptr, status, stream);
}

spin_status_t spin_indexer_score_ex(const spin_config* cfg, const void* q, const float* w, const void* k_pool,
                                    const float* k_scale, int64_t n_pages, const int32_t* block_table,
                                    int64_t bt_stride, const int32_t* list, const int32_t* n_list,
                                    const int32_t* n_slots, int32_t rows, float* scores,
                                    const spin_score_extras* extras, uint32_t* status, spin_stream_t stream) {
    return score_impl(cfg, q, w, k_pool, k_scale, n_pages, block_table, bt_stride, list, n_list, n_slots, rows,
                      scores, extras, status, stream);
}

spin_status_t spin_topk_hint_size(const spin_config* cfg, int32_t rows, size_t* bytes) {
    spin_status_t st = check_cfg(cfg);
    if (st) return st;
    if ((st = check_rows(cfg, rows))) return st;
    if (!bytes) return fail(SPIN_ERR_INVALID_ARG, "bytes is NULL");
    if (!topk_hint_supported(*cfg))
        return fail(SPIN_ERR_UNSUPPORTED, "no hinted top-K for top_k %d with %d blocks (needs top_k <= 2048 and "
                    "at most 8192 blocks)", cfg->top_k, dims_of(*cfg).MB);
    *bytes = topk_hint_bytes(*cfg, rows);
    return SPIN_OK;
}

spin_status_t spin_init_topk_hint(const spin_config* cfg, int32_t rows, void* hint, size_t hint_bytes, int32_t req,
                                  spin_stream_t stream) {
    spin_status_t st = check_cfg(cfg);
    if (st) return st;
    if ((st = check_rows(cfg, rows))) return st;
    if ((st = check_hint(cfg, rows, hint, hint_bytes))) return st;
    if (req >= cfg->n_req) return fail(SPIN_ERR_INVALID_ARG, "req %d >= n_req %d", req, cfg->n_req);
    const size_t rec = (size_t)kHintWords * 4;
    unsigned char* base = reinterpret_cast<unsigned char*>(hint);
    const size_t off = req < 0 ? 0 : (size_t)req * rows * rec;
    const size_t len = (req < 0 ? (size_t)cfg->n_req : 1u) * rows * rec;
    return launched(cudaMemsetAsync(base + off, 0, len, (cudaStream_t)stream), "spin_init_topk_hint");
}

spin_status_t spin_topk_hinted(const spin_config* cfg, const float* scores, const float* w, const int32_t* list,
                               const int32_t* n_list, const int32_t* n_slots, int32_t rows, int32_t* topk_idx,
                               void* hint, size_t hint_bytes, uint32_t* status, spin_stream_t stream) {
    spin_status_t st = check_cfg(cfg);
    if (st) return st;
    if ((st = check_rows(cfg, rows))) return st;
    if (!scores || !w || !list || !n_list || !n_slots || !topk_idx)
        return fail(SPIN_ERR_INVALID_ARG, "a required pointer is NULL");
    if ((st = check_hint(cfg, rows, hint, hint_bytes))) return st;
    return launched(launch_topk_hint(*cfg, scores, w, list, n_list, n_slots, rows, topk_idx,
                                     topk_hint_args(*cfg, rows, hint), status, (cudaStream_t)stream),
                    "spin_topk_hinted");
}

spin_status_t spin_topk(const spin_config* cfg, const float* scores, const int32_t* list, const int32_t* n_list,
                        const int32_t* n_slots, int32_t rows, int32_t* topk_idx, uint32_t* status,
                        spin_stream_t stream) {
    spin_status_t st = check_cfg(cfg);
    if (st) return st;
    if ((st = check_rows(cfg, rows))) return st;
    if (!scores || !list || !n_list || !n_slots || !topk_idx) return fail(SPIN_ERR_INVALID_ARG, "a required pointer is NULL");
    return launched(launch_topk(*cfg, scores, list, n_list, n_slots, rows, topk_idx, status, (cudaStream_t)stream),
                    "spin_topk");
}

static spin_status_t update_impl(const spin_config* cfg, int32_t n_layers, float* V, float* D, float* Vmax,
                                 int32_t* warm, const float* scores, const int32_t* list, const int32_t* n_list,
                                 const int32_t* n_slots, const int32_t* q_pos, uint32_t* status, spin_stream_t stream,
                                 uint32_t* block_age = nullptr, uint64_t age_step = 0) {
    spin_status_t st = check_cfg(cfg);
    if (st) return st;
    if ((st = check_layers(n_layers))) return st;
    if (!V || !D || !Vmax || !warm || !scores || !list || !n_list || !n_slots || !q_pos)
        return fail(SPIN_ERR_INVALID_ARG, "a required pointer is NULL");
    if ((cfg->explore == SPIN_EXPLORE_BLOCK_AGE) != (block_age != nullptr))
        return fail(SPIN_ERR_INVALID_ARG, cfg->explore == SPIN_EXPLORE_BLOCK_AGE
                                              ? "block-age exploration needs spin_update_ema_age and an age array"
                                              : "an age array needs explore = SPIN_EXPLORE_BLOCK_AGE");
    EmaArgs a{V, D, Vmax, warm, scores, 1, list, n_list, n_slots, q_pos, nullptr, status, n_layers, block_age,
              age_step};
    return launched(launch_ema(*cfg, a, (cudaStream_t)stream), "spin_update_ema");
}

static spin_status_t commit_impl(const spin_config* cfg, int32_t n_layers, float* V, float* D, float* Vmax,
                                 int32_t* warm, const float* scores, int32_t rows, const int32_t* union_blocks,
                                 const int32_t* n_union, const int32_t* n_slots, const int32_t* q_pos,
                                 const int32_t* accepted, uint32_t* status, spin_stream_t stream) {
    spin_status_t st = check_cfg(cfg);
    if (st) return st;
    if ((st = check_rows(cfg, rows))) return st;
    if ((st = check_layers(n_layers))) return st;
    if (!V || !D || !Vmax || !warm || !scores || !union_blocks || !n_union || !n_slots || !q_pos || !accepted)
        return fail(SPIN_ERR_INVALID_ARG, "a required pointer is NULL");
    if (cfg->explore == SPIN_EXPLORE_BLOCK_AGE)
        return fail(SPIN_ERR_INVALID_ARG, "block-age exploration has no MTP commit");
    EmaArgs a{V, D, Vmax, warm, scores, rows, union_blocks, n_union, n_slots, q_pos, accepted, status, n_layers};
    return launched(launch_ema(*cfg, a, (cudaStream_t)stream), "spin_commit_mtp");
}

spin_status_t spin_update_ema(const spin_config* cfg, float* V, float* D, float* Vmax, int32_t* warm,
                              const float* scores, const int32_t* list, const int32_t* n_list, const int32_t* n_slots,
                              const int32_t* q_pos, uint32_t* status, spin_stream_t stream) {
    return update_impl(cfg, 1, V, D, Vmax, warm, scores, list, n_list, n_slots, q_pos, status, stream);
}

spin_status_t spin_update_ema_age(const spin_config* cfg, float* V, float* D, float* Vmax, int32_t* warm,
                                  const float* scores, const int32_t* list, const int32_t* n_list,
                                  const int32_t* n_slots, const int32_t* q_pos, uint32_t* block_age, uint64_t step,
                                  uint32_t* status, spin_stream_t stream) {
    g_err[0] = 0;
    if (!block_age) return fail(SPIN_ERR_INVALID_ARG, "block_age is NULL");
    return update_impl(cfg, 1, V, D, Vmax, warm, scores, list, n_list, n_slots, q_pos, status, stream, block_age,
                       step);
}

spin_status_t spin_update_ema_layers(const spin_config* cfg, int32_t n_layers, float* V, float* D, float* Vmax,
                                     int32_t* warm, const float* scores, const int32_t* list, const int32_t* n_list,
                                     const int32_t* n_slots, const int32_t* q_pos, uint32_t* status,
                                     spin_stream_t stream) {
    return update_impl(cfg, n_layers, V, D, Vmax, warm, scores, list, n_list, n_slots, q_pos, status, stream);
}

spin_status_t spin_commit_mtp(const spin_config* cfg, float* V, float* D, float* Vmax, int32_t* warm,
                              const float* scores, int32_t rows, const int32_t* union_blocks, const int32_t* n_union,
                              const int32_t* n_slots, const int32_t* q_pos, const int32_t* accepted, uint32_t* status,
                              spin_stream_t stream) {
    return commit_impl(cfg, 1, V, D, Vmax, warm, scores, rows, union_blocks, n_union, n_slots, q_pos, accepted,
                       status, stream);
}

spin_status_t spin_commit_mtp_layers(const spin_config* cfg, int32_t n_layers, float* V, float* D, float* Vmax,
                                     int32_t* warm, const float* scores, int32_t rows, const int32_t* union_blocks,
                                     const int32_t* n_union, const int32_t* n_slots, const int32_t* q_pos,
                                     const int32_t* accepted, uint32_t* status, spin_stream_t stream) {
    return commit_impl(cfg, n_layers, V, D, Vmax, warm, scores, rows, union_blocks, n_union, n_slots, q_pos,
                       accepted, status, stream);
}

spin_status_t spin_miss_curve(const float* S, int32_t n_req, int64_t s_stride, const int32_t* nb,
                              const int32_t* topk, int32_t top_k, int32_t n_points, float* miss) {
    if (!S || !nb || !topk || !miss) return fail(SPIN_ERR_INVALID_ARG, "S, nb, topk and miss must be non-NULL");
    if (n_req < 1) return fail(SPIN_ERR_INVALID_ARG, "n_req %d < 1", n_req);
    if (top_k < 1) return fail(SPIN_ERR_INVALID_ARG, "top_k %d < 1", top_k);
    if (n_points < 2 || 10000 % (n_points - 1) != 0)
        return fail(SPIN_ERR_INVALID_ARG, "n_points %d: n_points - 1 must divide 10000", n_points);
    for (int32_t r = 0; r < n_req; ++r) {
        if (nb[r] < 1 || (int64_t)nb[r] > s_stride)
            return fail(SPIN_ERR_INVALID_ARG, "request %d: nb %d outside [1, s_stride=%lld]", r, nb[r], (long long)s_stride);
        for (int32_t j = 0; j < nb[r]; ++j)
            if (std::isnan(S[(int64_t)r * s_stride + j]))
                return fail(SPIN_ERR_INVALID_ARG, "request %d: block score %d is NaN", r, j);
        for (int32_t k = 0; k < top_k; ++k) {
            const int32_t id = topk[(int64_t)r * top_k + k];
            if (id < -1 || (int64_t)id >= (int64_t)nb[r] * kBlock)
                return fail(SPIN_ERR_INVALID_ARG, "request %d: top-K id %d outside [-1, %lld)", r, id,
                            (long long)nb[r] * kBlock);
        }
    }
    spin::mean_miss_curve_host(S, n_req, s_stride, nb, topk, top_k, n_points, miss);
    return SPIN_OK;
}

spin_status_t spin_allocate_budgets(const float* miss, int32_t n_layers, int32_t n_points, int32_t target_g,
                                    int32_t g_min, int32_t* g_out, int32_t* rho_bp_out) {
    if (!miss || !g_out) return fail(SPIN_ERR_INVALID_ARG, "miss and g_out must be non-NULL");
    if (n_layers < 1) return fail(SPIN_ERR_INVALID_ARG, "n_layers %d < 1", n_layers);
    if (n_points < 2 || 10000 % (n_points - 1) != 0)
        return fail(SPIN_ERR_INVALID_ARG, "n_points %d: n_points - 1 must divide 10000", n_points);
    if (g_min < 0 || g_min > target_g || target_g > n_points - 1)
        return fail(SPIN_ERR_INVALID_ARG, "need 0 <= g_min (%d) <= target_g (%d) <= n_points - 1 (%d)", g_min,
                    target_g, n_points - 1);
    for (int64_t i = 0; i < (int64_t)n_layers * n_points; ++i)
        if (std::isnan(miss[i])) return fail(SPIN_ERR_INVALID_ARG, "miss[%lld] is NaN", (long long)i);
    spin::allocate_budgets_host(miss, n_layers, n_points, target_g, g_min, g_out);
    if (rho_bp_out)
        for (int32_t l = 0; l < n_layers; ++l)
            rho_bp_out[l] = 10000 - (int32_t)((int64_t)g_out[l] * 10000 / (n_points - 1));
    return SPIN_OK;
}

spin_status_t spin_selftest_wait(int32_t mode, uint64_t limit_ns, uint32_t* status, uint64_t* elapsed_ns,
                                spin_stream_t stream) {
    g_err[0] = 0;
    if (mode < 0 || mode > 2) return fail(SPIN_ERR_INVALID_ARG, "mode %d outside [0, 2]", mode);
    if (!status || !elapsed_ns) return fail(SPIN_ERR_INVALID_ARG, "status and elapsed_ns must be non-NULL");
    if (limit_ns == 0 || limit_ns > 10ull * 1000ull * 1000ull * 1000ull)
        return fail(SPIN_ERR_INVALID_ARG, "limit_ns outside (0, 10 s]");
    return launched(launch_wait_selftest(mode, limit_ns, status, reinterpret_cast<unsigned long long*>(elapsed_ns),
                                         (cudaStream_t)stream),
                    "spin_selftest_wait");
}

const char* spin_version(void) { return "spin-gb300 0.1.0 sm_103a"; }

const char* spin_last_error_string(void) { return g_err; }

}  // extern "C"

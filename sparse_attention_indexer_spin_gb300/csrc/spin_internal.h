// spin_internal.h -- host-side launchers of the SPIN kernels (called by spin_api.cu only).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/spin.h"
#include "spin_common.cuh"

namespace spin {

struct SelectArgs {
    const float* V;
    const float* D;
    const float* Vmax;
    const int32_t* warm;
    const int32_t* n_slots;
    const int32_t* q_pos;
    int rows;
    const int32_t* rho_override;
    uint64_t step;
    const uint64_t* step_dev;  // non-NULL: the kernels read the step here instead
    int layer;
    int32_t* blocks;
    int32_t* n_blocks;
    int32_t* union_blocks;
    int32_t* n_union;
    float* block_scores;  // workspace: S [R][rows][MB] fp32, then exploration draws [R][rows][MB] u32
    uint32_t* status;
    int n_layers;         // layers stacked along the outermost dimension of every array (0 or 1: one)
    const uint32_t* block_age = nullptr;  // block-age exploration: ages [R][MB] replace the draws
};

struct ScoreArgs {
    const void* q;
    const float* w;
    const void* k_pool;
    const float* k_scale;
    int64_t n_pages;
    const int32_t* block_table;
    int64_t bt_stride;
    const int32_t* list;
    const int32_t* n_list;
    const int32_t* n_slots;
    int rows;
    float* scores;
    uint32_t* status;
    HintArgs hint;  // rec == NULL: no candidate collection for the hinted top-K
};

struct EmaArgs {
    float* V;
    float* D;
    float* Vmax;
    int32_t* warm;
    const float* scores;
    int rows;
    const int32_t* list;
    const int32_t* n_list;
    const int32_t* n_slots;
    const int32_t* q_pos;
    const int32_t* accepted;  // NULL: a = 0
    uint32_t* status;
    int n_layers;             // layers stacked along the outermost dimension (0 or 1: one)
    uint32_t* block_age = nullptr;  // block-age exploration: listed blocks get age_step + 1
    uint64_t age_step = 0;
};

size_t select_workspace_bytes(const spin_config& cfg, int rows);

cudaError_t launch_init_state(const spin_config& cfg, float* V, float* D, float* Vmax,
                              int32_t* warm, int req, cudaStream_t s);
cudaError_t launch_select(const spin_config& cfg, const SelectArgs& a, cudaStream_t s);
cudaError_t launch_score_generic(const spin_config& cfg, const ScoreArgs& a, cudaStream_t s);
// Returns cudaErrorNotSupported when the shape has no streaming kernel instance.
cudaError_t launch_score_stream(const spin_config& cfg, const ScoreArgs& a, cudaStream_t s);
bool score_stream_supported(const spin_config& cfg, int rows);
cudaError_t launch_score_tc(const spin_config& cfg, const ScoreArgs& a, cudaStream_t s);
bool score_tc_supported(const spin_config& cfg, int rows);
bool topk_sample_fits(const spin_config& cfg);
cudaError_t launch_topk_sample(const spin_config& cfg, const float* scores, const int32_t* list,
                               const int32_t* n_list, const int32_t* n_slots, int rows, int32_t* topk_idx,
                               uint32_t* status, cudaStream_t s);
cudaError_t launch_topk(const spin_config& cfg, const float* scores, const int32_t* list,
                        const int32_t* n_list, const int32_t* n_slots, int rows,
                        int32_t* topk_idx, uint32_t* status, cudaStream_t s);
cudaError_t launch_ema(const spin_config& cfg, const EmaArgs& a, cudaStream_t s);

// Temporal top-K (spin_topk_hint.cu).
bool topk_hint_supported(const spin_config& cfg);
int topk_hint_cap(const spin_config& cfg);
size_t topk_hint_bytes(const spin_config& cfg, int rows);
HintArgs topk_hint_args(const spin_config& cfg, int rows, void* hint);
cudaError_t launch_topk_hint(const spin_config& cfg, const float* scores, const float* w, const int32_t* list,
                             const int32_t* n_list, const int32_t* n_slots, int rows, int32_t* topk_idx,
                             const HintArgs& h, uint32_t* status, cudaStream_t s);

int device_sm_count();

// Self-test of the bounded mbarrier wait (spin_selftest.cu).
cudaError_t launch_wait_selftest(int mode, uint64_t limit_ns, uint32_t* status, unsigned long long* elapsed_ns,
                                 cudaStream_t s);

// Per-layer block budgets (host functions; spin_budget.cu).  Arguments are validated by the
// C-ABI wrappers.
int64_t budget_blocks_host(int64_t nb, int64_t top_k, int32_t rho_bp);
void mean_miss_curve_host(const float* S, int32_t n_req, int64_t s_stride, const int32_t* nb,
                          const int32_t* topk, int32_t top_k, int32_t n_points, float* miss);
void allocate_budgets_host(const float* miss, int32_t n_layers, int32_t n_points, int32_t target_g,
                           int32_t g_min, int32_t* g_out);

}  // namespace spin

// spin_score_generic.cu -- indexer score for any shape (a slow cross-check kernel).
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention", §2 and Algorithm 1's scoring step:
// z_t[i] = sum_h w_h ReLU(q_{t,h} . k_{i,h}) over the slots of the selected blocks; the
// per-slot FP8 scale multiplies the dot product before the ReLU.
//
// One CTA per (request, list entry); one thread per (row, slot) of the block computes all
// heads sequentially in fp32.  Used for shapes the fast kernels do not cover and as an
// independent GPU cross-check of them.
#include <cuda_fp8.h>

#include "spin_common.cuh"
#include "spin_internal.h"

namespace spin {

__device__ __forceinline__ float load_q(const void* q, int dtype, int64_t idx) {
    if (dtype == SPIN_DTYPE_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(q)[idx]);
    return reinterpret_cast<const float*>(q)[idx];
}

__device__ __forceinline__ float load_k(const void* k, int dtype, int64_t idx) {
    if (dtype == SPIN_DTYPE_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(k)[idx]);
    if (dtype == SPIN_DTYPE_E4M3) {
        __nv_fp8_e4m3 v;
        v.__x = reinterpret_cast<const __nv_fp8_storage_t*>(k)[idx];
        return float(v);
    }
    return reinterpret_cast<const float*>(k)[idx];
}

__global__ void __launch_bounds__(256) score_generic_kernel(spin_config cfg, ScoreArgs a) {
    pdl_begin();
    const Dims dm = dims_of(cfg);
    const int req = blockIdx.y;
    const int k = blockIdx.x;
    const int64_t n = a.n_slots[req];
    const int64_t cnt = a.n_list[req];
    if (n < 0 || n > dm.max_slots || cnt < 0 || cnt > dm.MB) {
        if (k == 0 && threadIdx.x == 0) set_status(a.status, n < 0 || n > dm.max_slots ? SPIN_STATUS_BAD_N : SPIN_STATUS_BAD_LIST);
        return;
    }
    if (k >= cnt) return;
    const int64_t blk = a.list[(int64_t)req * dm.MB + k];
    const int64_t nb = (n + kBlock - 1) / kBlock;
    int64_t page = -1;
    if (blk >= 0 && blk < nb) page = a.block_table[(int64_t)req * a.bt_stride + blk];
    const bool bad_list = !(blk >= 0 && blk < nb);
    const bool bad_page = !bad_list && !(page >= 0 && page < a.n_pages);
    if (threadIdx.x == 0 && (bad_list || bad_page))
        set_status(a.status, bad_list ? SPIN_STATUS_BAD_LIST : SPIN_STATUS_BAD_PAGE);
    const int H = cfg.n_heads, d = cfg.head_dim, rows = a.rows;
    const int64_t slot_elems = (int64_t)cfg.kv_heads * d;
    for (int idx = threadIdx.x; idx < rows * kBlock; idx += blockDim.x) {
        const int r = idx / kBlock, s = idx - r * kBlock;
        const int64_t i = blk * kBlock + s;
        float z = 0.0f;
        if (!bad_list && !bad_page && i < n) {
            const int64_t slot = page * kBlock + s;
            const float scale = a.k_scale ? a.k_scale[slot] : 1.0f;
            const int64_t kbase = slot * slot_elems;
            const int64_t qbase = ((int64_t)req * rows + r) * H * d;
            const float* wr = a.w + ((int64_t)req * rows + r) * H;
            for (int h = 0; h < H; ++h) {
                const int64_t kh = cfg.kv_heads == 1 ? 0 : h;
                float dot = 0.0f;
                for (int c = 0; c < d; ++c)
                    dot = fmaf(load_q(a.q, cfg.q_dtype, qbase + (int64_t)h * d + c),
                               load_k(a.k_pool, cfg.k_dtype, kbase + kh * d + c), dot);
                const float x = scale * dot;
                z = fmaf(wr[h], x > 0.0f ? x : 0.0f, z);
            }
            if (z == 0.0f) z = 0.0f;  // no -0 in the output
        }
        a.scores[(((int64_t)req * rows + r) * dm.MB + k) * kBlock + s] = z;
        // hinted top-K: a live slot (valid block, i < N) at or above its row's threshold
        if (a.hint.rec && !bad_list && i < n) {
            const int64_t rr = (int64_t)req * rows + r;
            const uint32_t thr = hint_threshold(a.hint.rec[rr * kHintWords + kHwGuess], row_wsum(a.w + rr * H, H));
            a.hint.rec[rr * kHintWords + kHwFlags] = 1u;  // (every writer stores the same value)
            const uint32_t key = order_key(z);
            if (thr != 0u && key >= thr) hint_push(a.hint, rr, key, (uint32_t)(k * kBlock + s));
        }
    }
}

cudaError_t launch_score_generic(const spin_config& cfg, const ScoreArgs& a, cudaStream_t s) {
    const Dims dm = dims_of(cfg);
    dim3 grid(dm.MB, dm.R);
    return launch_pdl(score_generic_kernel, grid, dim3(256), 0, s, nullptr, 0, cfg, a);
}

}  // namespace spin

// spin_select.cu -- block prediction and budgeted block selection.
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention": Eq. 1 (predicted slot score
// max(V[i], D[q-i])), Eq. 2 (max-pooling over the block's slots), Algorithm 1's prediction, budget and block top-m steps
// (budget m_t, TopK over block scores), §3.2 practical details (warm-up step is dense;
// sink and newest blocks always kept), §3.2.1 (a share gamma of m_t explores blocks
// drawn at random from those not selected), §3.2.2 (masks of several verifier rows are
// unioned).
//
// Two kernels:
//   block_score_kernel  many CTAs: S[req][row][j] for every block (HBM-bound scan of D
//                       plus the per-block max of V kept in Vmax)
//   select_kernel       one CTA per request: for each row, budget, forced blocks, radix
//                       select of the top blocks, Philox exploration, ordered compaction;
//                       then the union of the rows.
#include <float.h>

#include "spin_common.cuh"
#include "spin_internal.h"

namespace spin {

// ---------------------------------------------------------------------------------------
// S[j] for one (request, row).  Under Eq. 1's max, max_i max(V[i], D[q-i]) over a full
// block equals max(Vmax[j], max_i D[q-i]), so V is read only through its per-block max.
// The additive reading needs V[i] + D[q-i] slot by slot.
// ---------------------------------------------------------------------------------------
constexpr int kBsBlocksPerWarp = 8;

__global__ void __launch_bounds__(256) block_score_kernel(spin_config cfg, const float* __restrict__ V,
                                                          const float* __restrict__ D,
                                                          const float* __restrict__ Vmax,
                                                          const int32_t* __restrict__ warm,
                                                          const int32_t* __restrict__ n_slots,
                                                          const int32_t* __restrict__ q_pos, int rows,
                                                          float* __restrict__ S) {
    const Dims dm = dims_of(cfg);
    const int rr = blockIdx.y;
    const int req = rr / rows, r = rr - req * rows;
    const int64_t n = n_slots[req], q = q_pos[req];
    if (request_check(n, q, rows, dm) != 0u || warm[req] == 0) return;
    const int64_t qr = q + r;
    const int64_t nb = (n + kBlock - 1) / kBlock;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const float* Dq = D + (int64_t)req * dm.DL;
    const float* Vq = V + (int64_t)req * dm.max_slots;
    const float* Vm = Vmax + (int64_t)req * dm.MB;
    float* Sq = S + (int64_t)rr * dm.MB;
    const bool sum = cfg.combine == SPIN_COMBINE_SUM;
    // each warp owns kBsBlocksPerWarp consecutive blocks and issues all their loads first
    for (int64_t j0 = ((int64_t)blockIdx.x * nw + wid) * kBsBlocksPerWarp; j0 < nb;
         j0 += (int64_t)gridDim.x * nw * kBsBlocksPerWarp) {
        float lo[kBsBlocksPerWarp], hi[kBsBlocksPerWarp];
#pragma unroll
        for (int b = 0; b < kBsBlocksPerWarp; ++b) {
            const int64_t i0 = (j0 + b) * kBlock + lane, i1 = i0 + 32;
            lo[b] = i0 < n ? (sum ? __fadd_rn(Vq[i0], Dq[qr - i0]) : Dq[qr - i0]) : -FLT_MAX;
            hi[b] = i1 < n ? (sum ? __fadd_rn(Vq[i1], Dq[qr - i1]) : Dq[qr - i1]) : -FLT_MAX;
        }
        const float vm = (!sum && lane < kBsBlocksPerWarp && j0 + lane < nb) ? Vm[j0 + lane] : -FLT_MAX;
#pragma unroll
        for (int b = 0; b < kBsBlocksPerWarp; ++b) {
            // every block of the loop has at least one slot < N, so the max is a real value
            float m = fmaxf(lo[b], hi[b]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float vmb = __shfl_sync(0xffffffffu, vm, b);
            if (lane == 0 && j0 + b < nb) Sq[j0 + b] = sum ? m : fmaxf(vmb, m);
        }
    }
}

// ---------------------------------------------------------------------------------------
// CTA-wide selection helpers (1024 threads).
// ---------------------------------------------------------------------------------------
constexpr int kSelThreads = 1024;

struct SelShared {
    int hist[256];
    int scan[33];
    int count;
    uint32_t prefix;
    int kk;
};

// Set flag[j] = mark for the k entries with flag[j] == 0 that have the largest keys
// (equal keys: ascending j).  Radix select over 4 digits of 8 bits, then an ordered
// pass for the entries equal to the threshold.
__device__ void top_select(const uint32_t* keys, uint8_t* flag, int n, int k, uint8_t mark, SelShared& sh) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (k <= 0) return;
    // eligible count
    int c = 0;
    for (int j = tid; j < n; j += kSelThreads) c += flag[j] == 0;
    int total;
    block_excl_scan(c, sh.scan, &total);
    if (k >= total) {
        for (int j = tid; j < n; j += kSelThreads)
            if (flag[j] == 0) flag[j] = mark;
        __syncthreads();
        return;
    }
    uint32_t prefix = 0, mask = 0;
    int kk = k;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int b = tid; b < 256; b += kSelThreads) sh.hist[b] = 0;
        __syncthreads();
        // warp-aggregated shared atomics: block scores share their high bits, so many
        // lanes hit the same bin
        const int n_pad = (n + 31) & ~31;
        for (int j = tid; j < n_pad; j += kSelThreads) {
            int bin = -1;
            if (j < n) {
                const uint32_t key = keys[j];
                if (flag[j] == 0 && (key & mask) == prefix) bin = (int)((key >> shift) & 255u);
            }
            const unsigned same = __match_any_sync(0xffffffffu, bin);
            if (bin >= 0 && lane == __ffs(same) - 1) atomicAdd(&sh.hist[bin], __popc(same));
        }
        __syncthreads();
        if (wid == 0) {
            // lane l owns bins 255-8l .. 248-8l (descending)
            int cnt[8], s = 0;
#pragma unroll
            for (int b = 0; b < 8; ++b) { cnt[b] = sh.hist[255 - 8 * lane - b]; s += cnt[b]; }
            const int inc = warp_incl_scan(s);
            const int excl = inc - s;
            const unsigned ball = __ballot_sync(0xffffffffu, inc >= kk);
            const int src = __ffs(ball) - 1;  // first lane whose cumulative count reaches kk
            if (lane == src) {
                int above = excl, digit = 0;
                for (int b = 0; b < 8; ++b) {
                    if (above + cnt[b] >= kk) { digit = 255 - 8 * lane - b; break; }
                    above += cnt[b];
                }
                sh.prefix = prefix | ((uint32_t)digit << shift);
                sh.kk = kk - above;
            }
        }
        __syncthreads();
        prefix = sh.prefix;
        kk = sh.kk;
        mask |= 0xFFu << shift;
        __syncthreads();
    }
    // keys > prefix are taken; of the keys == prefix, the first kk in j order.
    const int chunk = (n + kSelThreads - 1) / kSelThreads;
    const int j0 = min(n, tid * chunk), j1 = min(n, j0 + chunk);
    int eq = 0;
    for (int j = j0; j < j1; ++j) eq += (flag[j] == 0 && keys[j] == prefix);
    int rank = block_excl_scan(eq, sh.scan, &total);
    for (int j = j0; j < j1; ++j) {
        if (flag[j] != 0) continue;
        const uint32_t key = keys[j];
        if (key > prefix) {
            flag[j] = mark;
        } else if (key == prefix) {
            if (rank < kk) flag[j] = mark;
            ++rank;
        }
    }
    __syncthreads();
}

// Ascending list of the j with flag[j] != 0; returns the count.
__device__ int compact_flags(const uint8_t* flag, int n, int32_t* out, SelShared& sh) {
    const int tid = threadIdx.x;
    const int chunk = (n + kSelThreads - 1) / kSelThreads;
    const int j0 = min(n, tid * chunk), j1 = min(n, j0 + chunk);
    int c = 0;
    for (int j = j0; j < j1; ++j) c += flag[j] != 0;
    int total;
    int pos = block_excl_scan(c, sh.scan, &total);
    for (int j = j0; j < j1; ++j)
        if (flag[j] != 0) out[pos++] = j;
    return total;
}

__device__ __forceinline__ int64_t budget_blocks(int64_t nb, int64_t top_k, int32_t rho_bp) {
    const int64_t floor_k = (top_k + kBlock - 1) / kBlock;
    const int64_t keep = ((int64_t)(10000 - rho_bp) * nb + 9999) / 10000;
    const int64_t m = floor_k > keep ? floor_k : keep;
    return m < nb ? m : nb;
}

__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(
    spin_config cfg, const int32_t* __restrict__ warm, const int32_t* __restrict__ n_slots,
    const int32_t* __restrict__ q_pos, int rows, const int32_t* __restrict__ rho_override, uint64_t step,
    int layer, const float* __restrict__ S, int32_t* __restrict__ blocks, int32_t* __restrict__ n_blocks,
    int32_t* __restrict__ union_blocks, int32_t* __restrict__ n_union, uint32_t* status) {
    extern __shared__ __align__(16) unsigned char sel_smem[];
    __shared__ SelShared sh;
    const Dims dm = dims_of(cfg);
    const int MB = dm.MB;
    uint32_t* keys = reinterpret_cast<uint32_t*>(sel_smem);
    uint8_t* flag = sel_smem + (size_t)MB * 4;
    uint8_t* uflag = flag + MB;
    const int req = blockIdx.x, tid = threadIdx.x;
    const int64_t n = n_slots[req], q = q_pos[req];
    uint32_t bad = request_check(n, q, rows, dm);
    int32_t rho = cfg.rho_bp;
    if (rho_override) {
        rho = *rho_override;
        if (rho < 0 || rho > 10000) bad |= SPIN_STATUS_BAD_RHO;
    }
    if (bad) {
        if (tid == 0) {
            set_status(status, bad);
            for (int r = 0; r < rows; ++r) n_blocks[(int64_t)req * rows + r] = 0;
            if (union_blocks && n_union) n_union[req] = 0;
        }
        return;
    }
    const int nb = (int)((n + kBlock - 1) / kBlock);
    const bool is_warm = warm[req] != 0;
    for (int j = tid; j < nb; j += kSelThreads) uflag[j] = 0;
    __syncthreads();
    for (int r = 0; r < rows; ++r) {
        const int64_t rr = (int64_t)req * rows + r;
        if (!is_warm || nb <= 2) {
            // dense warm-up step (and contexts whose every block is forced)
            for (int j = tid; j < nb; j += kSelThreads) flag[j] = 1;
            __syncthreads();
        } else {
            const int64_t m = budget_blocks(nb, cfg.top_k, rho);
            const int64_t f = 2;
            int64_t e = 0, t = 0;
            if (m > f) {
                e = ((int64_t)cfg.gamma_bp * m) / 10000;
                if (e > m - f) e = m - f;
                t = m - f - e;
            }
            const float* Sr = S + rr * MB;
            for (int j = tid; j < nb; j += kSelThreads) {
                const bool forced = (j == 0) || (j == nb - 1);
                flag[j] = forced ? 1 : 0;
                keys[j] = order_key(Sr[j]);
            }
            __syncthreads();
            top_select(keys, flag, nb, (int)t, 1, sh);
            if (e > 0) {
                // smallest Philox key first == largest complement
                for (int j = tid; j < nb; j += kSelThreads)
                    if (flag[j] == 0) keys[j] = ~explore_key(cfg.seed, layer, step, r, req, j);
                __syncthreads();
                top_select(keys, flag, nb, (int)e, 1, sh);
            }
        }
        const int cnt = compact_flags(flag, nb, blocks + rr * MB, sh);
        if (tid == 0) n_blocks[rr] = cnt;
        for (int j = tid; j < nb; j += kSelThreads) uflag[j] |= flag[j];
        __syncthreads();
    }
    if (union_blocks && n_union) {
        const int cnt = compact_flags(uflag, nb, union_blocks + (int64_t)req * MB, sh);
        if (tid == 0) n_union[req] = cnt;
    }
}

size_t select_workspace_bytes(const spin_config& cfg, int rows) {
    const Dims dm = dims_of(cfg);
    size_t b = sizeof(float) * (size_t)dm.R * (size_t)rows * (size_t)dm.MB;
    return (b + 255) & ~(size_t)255;
}

cudaError_t launch_select(const spin_config& cfg, const SelectArgs& a, cudaStream_t s) {
    const Dims dm = dims_of(cfg);
    const int per_cta = (256 / 32) * kBsBlocksPerWarp;
    int gx = (dm.MB + per_cta - 1) / per_cta;
    if (gx > 512) gx = 512;
    dim3 g1(gx, dm.R * a.rows);
    block_score_kernel<<<g1, 256, 0, s>>>(cfg, a.V, a.D, a.Vmax, a.warm, a.n_slots, a.q_pos, a.rows,
                                          a.block_scores);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = ((size_t)dm.MB * 6 + 15) & ~(size_t)15;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    select_kernel<<<dm.R, kSelThreads, smem, s>>>(cfg, a.warm, a.n_slots, a.q_pos, a.rows, a.rho_override,
                                                  a.step, a.layer, a.block_scores, a.blocks, a.n_blocks,
                                                  a.union_blocks, a.n_union, a.status);
    return cudaGetLastError();
}

}  // namespace spin

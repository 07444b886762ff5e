// spin_select.cu -- block prediction and budgeted block selection.
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention": Eq. 1 (predicted slot score
// max(V[i], D[q-i])), Eq. 2 (max-pooling over the block's slots), Algorithm 1's prediction, budget and block top-m steps
// (budget m_t, TopK over block scores), §3.2 practical details (warm-up step is dense;
// sink and newest blocks always kept), §3.2.1 (a share gamma of m_t explores blocks
// drawn at random from those not selected), §3.2.2 (masks of several verifier rows are
// unioned).
//
// Kernels:
//   block_score_kernel  many CTAs: S[req][row][j] for every block (HBM-bound scan of D
//                       plus the per-block max of V kept in Vmax) and the Philox
//                       exploration draw of every block, computed while the loads fly
//   select_reg_kernel   up to 8192 blocks: one CTA per (request, row), keys in registers,
//                       budget, forced blocks, radix select of the top blocks and of the
//                       smallest draws among the rest, ordered compaction; the rows of a
//                       request form a cluster whose first CTA writes their union
//   select_kernel       longer lists: one CTA per request, keys in shared memory, the same
//                       steps row by row, then the union of the rows.
#include <float.h>

#include "spin_common.cuh"
#include "spin_internal.h"

#include <cooperative_groups.h>
namespace cg = cooperative_groups;

namespace spin {

// ---------------------------------------------------------------------------------------
// S[j] for one (request, row).  Under Eq. 1's max, max_i max(V[i], D[q-i]) over a full
// block equals max(Vmax[j], max_i D[q-i]), so V is read only through its per-block max.
// The additive reading needs V[i] + D[q-i] slot by slot.
// ---------------------------------------------------------------------------------------

// Block budget m_t (Algorithm 1's budget step) with rho in basis points.
__device__ __forceinline__ int64_t budget_blocks(int64_t nb, int64_t top_k, int32_t rho_bp) {
    const int64_t floor_k = (top_k + kBlock - 1) / kBlock;
    const int64_t keep = ((int64_t)(10000 - rho_bp) * nb + 9999) / 10000;
    const int64_t m = floor_k > keep ? floor_k : keep;
    return m < nb ? m : nb;
}


// BPW blocks per warp, all their loads issued before the first use: more loads in flight
// per warp pay when many request rows keep every SM busy; few rows want more CTAs instead.
template <int BPW>
__global__ void __launch_bounds__(256) block_score_kernel(spin_config cfg, const float* __restrict__ V,
                                                          const float* __restrict__ D,
                                                          const float* __restrict__ Vmax,
                                                          const int32_t* __restrict__ warm,
                                                          const int32_t* __restrict__ n_slots,
                                                          const int32_t* __restrict__ q_pos, int rows,
                                                          const int32_t* __restrict__ rho_override,
                                                          uint64_t seed, uint64_t step,
                                                          const uint64_t* __restrict__ step_dev, int layer,
                                                          const uint32_t* __restrict__ block_age,
                                                          float* __restrict__ S, uint32_t* __restrict__ X) {
    pdl_begin();
    if (step_dev) step = *step_dev;
    const Dims dm = dims_of(cfg);
    {   // layer blockIdx.z of a stack of layers (0 for a one-layer call)
        const int64_t l = blockIdx.z;
        V += l * dm.R * dm.max_slots;
        D += l * dm.R * dm.DL;
        Vmax += l * dm.R * dm.MB;
        warm += l * dm.R;
        if (rho_override) rho_override += l;
        S += l * dm.R * rows * dm.MB;
        X += l * dm.R * rows * dm.MB;
        layer += (int)l;
    }
    const int rr = blockIdx.y;
    const int req = rr / rows, r = rr - req * rows;
    const int64_t n = n_slots[req], q = q_pos[req];
    if (request_check(n, q, rows, dm) != 0u || warm[req] == 0) return;
    const int64_t qr = q + r;
    const int64_t nb = (n + kBlock - 1) / kBlock;
    // a budget of every block (sparsity 0) selects them all: nothing to predict
    const int32_t rho = rho_override ? *rho_override : cfg.rho_bp;
    if (rho >= 0 && rho <= 10000 && budget_blocks(nb, cfg.top_k, rho) >= nb) return;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const float* Dq = D + (int64_t)req * dm.DL;
    const float* Vq = V + (int64_t)req * dm.max_slots;
    const float* Vm = Vmax + (int64_t)req * dm.MB;
    float* Sq = S + (int64_t)rr * dm.MB;
    uint32_t* Xq = X + (int64_t)rr * dm.MB;
    const bool sum = cfg.combine == SPIN_COMBINE_SUM;
    // the exploration draws of blocks j0 .. j0 + BPW - 1 (used only for blocks that end up
    // unselected): lane l < BPW / 8 computes one Philox output, the draws of the 8 blocks of
    // group j0 / 8 + l
    auto draws = [&](int64_t j0) {
        if (lane < BPW / 8) {
            const int64_t g = j0 / 8 + lane;
            if (g * 8 < nb) {
                uint32_t k8[8];
                if (block_age) {  // block-age exploration (§4.6): the ages are the keys
#pragma unroll
                    for (int h = 0; h < 8; ++h)
                        k8[h] = g * 8 + h < nb ? block_age[(int64_t)req * dm.MB + g * 8 + h] : 0u;
                } else {
                    explore_keys8(seed, layer, step, r, req, g, k8);
                }
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    if (g * 8 + h < nb) Xq[g * 8 + h] = k8[h];
            }
        }
    };
    if (cfg.pooling == SPIN_POOL_A2) {
        // the A2 ablation (§4.6): block-level EMAs, Vb[j] in V and Db at the block offset
        // floor(q / 64) - j in D, combined as Eq. 1 combines V and D
        const int64_t qb = qr / kBlock;
        for (int64_t j0 = ((int64_t)blockIdx.x * nw + wid) * BPW; j0 < nb;
             j0 += (int64_t)gridDim.x * nw * BPW) {
            draws(j0);
            const int64_t j = j0 + lane;
            if (lane < BPW && j < nb) {
                const float v = Vq[j], d = Dq[qb - j];
                Sq[j] = sum ? __fadd_rn(v, d) : fmaxf(v, d);
            }
        }
        return;
    }
    if (cfg.pooling != SPIN_POOL_MAX) {
        // the pooling ablations (§4.6): every slot's prediction, then the block's mean, or
        // the mean of its four largest, summed in the fixed order the interface states
        for (int64_t j0 = ((int64_t)blockIdx.x * nw + wid) * BPW; j0 < nb;
             j0 += (int64_t)gridDim.x * nw * BPW) {
            draws(j0);
            for (int b = 0; b < BPW && j0 + b < nb; ++b) {  // (warp-uniform)
                const int64_t i0 = (j0 + b) * kBlock + lane, i1 = i0 + 32;
                const bool vl = i0 < n, vh = i1 < n;
                auto pred = [&](int64_t i) {
                    const float v = Vq[i], d = Dq[qr - i];
                    return sum ? __fadd_rn(v, d) : fmaxf(v, d);
                };
                const float pl = vl ? pred(i0) : 0.0f, ph = vh ? pred(i1) : 0.0f;
                float score;
                if (cfg.pooling == SPIN_POOL_MEAN) {
                    float t = __fadd_rn(vl ? pl : 0.0f, vh ? ph : 0.0f);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, o));
                    const int cnt = __popc(__ballot_sync(0xffffffffu, vl)) + __popc(__ballot_sync(0xffffffffu, vh));
                    score = __fdiv_rn(t, (float)cnt);
                } else {
                    // the four largest values, one slot at a time (absent slots are -inf)
                    float a = vl ? pl : -INFINITY, c = vh ? ph : -INFINITY;
                    float top[4];
                    int k = 0;
                    for (; k < 4; ++k) {
                        float m = fmaxf(a, c);
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                        if (m == -INFINITY) break;
                        top[k] = m;
                        const unsigned ba = __ballot_sync(0xffffffffu, a == m);
                        if (ba) {
                            if (lane == __ffs(ba) - 1) a = -INFINITY;
                        } else {
                            const unsigned bc = __ballot_sync(0xffffffffu, c == m);
                            if (lane == __ffs(bc) - 1) c = -INFINITY;
                        }
                    }
                    float s4 = top[0];
                    if (k == 2) s4 = __fadd_rn(top[0], top[1]);
                    if (k == 3) s4 = __fadd_rn(__fadd_rn(top[0], top[1]), top[2]);
                    if (k == 4) s4 = __fadd_rn(__fadd_rn(top[0], top[1]), __fadd_rn(top[2], top[3]));
                    score = __fdiv_rn(s4, (float)k);
                }
                if (lane == 0) Sq[j0 + b] = score;
            }
        }
        return;
    }
    // each warp owns BPW consecutive blocks and issues all their loads first
    for (int64_t j0 = ((int64_t)blockIdx.x * nw + wid) * BPW; j0 < nb;
         j0 += (int64_t)gridDim.x * nw * BPW) {
        float lo[BPW], hi[BPW];
#pragma unroll
        for (int b = 0; b < BPW; ++b) {
            const int64_t i0 = (j0 + b) * kBlock + lane, i1 = i0 + 32;
            lo[b] = i0 < n ? (sum ? __fadd_rn(Vq[i0], Dq[qr - i0]) : Dq[qr - i0]) : -FLT_MAX;
            hi[b] = i1 < n ? (sum ? __fadd_rn(Vq[i1], Dq[qr - i1]) : Dq[qr - i1]) : -FLT_MAX;
        }
        const float vm = (!sum && lane < BPW && j0 + lane < nb) ? Vm[j0 + lane] : -FLT_MAX;
        draws(j0);  // while the loads are in flight
#pragma unroll
        for (int b = 0; b < BPW; ++b) {
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


__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(
    spin_config cfg, const int32_t* __restrict__ warm, const int32_t* __restrict__ n_slots,
    const int32_t* __restrict__ q_pos, int rows, const int32_t* __restrict__ rho_override, uint64_t step,
    int layer, const float* __restrict__ S, int32_t* __restrict__ blocks, int32_t* __restrict__ n_blocks,
    int32_t* __restrict__ union_blocks, int32_t* __restrict__ n_union, uint32_t* status,
    const uint64_t* __restrict__ step_dev, const uint32_t* __restrict__ block_age) {
    pdl_begin();
    if (step_dev) step = *step_dev;
    extern __shared__ __align__(16) unsigned char sel_smem[];
    __shared__ SelShared sh;
    const Dims dm = dims_of(cfg);
    const int MB = dm.MB;
    {   // layer blockIdx.y of a stack of layers (0 for a one-layer call)
        const int64_t l = blockIdx.y;
        warm += l * dm.R;
        if (rho_override) rho_override += l;
        S += l * dm.R * rows * MB;
        blocks += l * dm.R * rows * MB;
        n_blocks += l * dm.R * rows;
        if (union_blocks) union_blocks += l * dm.R * MB;
        if (n_union) n_union += l * dm.R;
        layer += (int)l;
    }
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
        if (!is_warm || nb <= 2 || budget_blocks(nb, cfg.top_k, rho) >= nb) {
            // dense: warm-up step, every block forced, or a budget of every block
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
                    if (flag[j] == 0)
                        keys[j] = ~(block_age ? block_age[(int64_t)req * MB + j]
                                              : explore_key(cfg.seed, layer, step, r, req, j));
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

// ---------------------------------------------------------------------------------------
// Register-resident selection (MB <= 512 * 16, rows <= 8): one 512-thread CTA per
// (request, row), rows of a request in one thread-block cluster.  Thread t keeps the keys
// of blocks j = t + 512 i (i < KPT) in registers, so the ascending-j order of equal keys is
// the (i, t) order.  A radix select needs one CTA barrier per 8-bit digit: every warp
// finds the digit itself from the shared histogram, and the three histogram buffers rotate
// so that the buffer a pass fills was cleared two passes earlier.  The union of the rows
// is taken by the cluster's first CTA from the others' selection bitmaps in distributed
// shared memory.
// ---------------------------------------------------------------------------------------
constexpr int kSrThreads = 512;
constexpr int kSrWarps = kSrThreads / 32;
constexpr int kSrMaxKpt = 16;
constexpr int kSrMaxBlocks = kSrThreads * kSrMaxKpt;

struct SrShared {
    __align__(16) int hist[3][256];
    int cnt[kSrMaxKpt * kSrWarps];       // per (i, warp) counts, (i, warp) order
    int base[kSrMaxKpt * kSrWarps + 1];  // their exclusive scan (+ total)
    uint32_t bitmap[kSrMaxBlocks / 32];  // selected blocks of this row, bit j % 32 of word j / 32
};

// Adds the warp's bins (-1: none) to a shared histogram: the lanes that share the first
// active lane's bin with one atomic, the others one atomic each (keys of one warp mostly
// share a bin when they are concentrated, and mostly differ when they are spread).
__device__ __forceinline__ void sr_hist_add(int* h, int bin) {
    const int lane = threadIdx.x & 31;
    const unsigned act = __ballot_sync(0xffffffffu, bin >= 0);
    if (act == 0u) return;
    const int lead = __ffs(act) - 1;
    const int b0 = __shfl_sync(0xffffffffu, bin, lead);
    const unsigned m0 = __ballot_sync(0xffffffffu, bin == b0);
    if (lane == lead) atomicAdd(&h[b0], __popc(m0));
    else if (bin >= 0 && bin != b0) atomicAdd(&h[bin], 1);
}

// Exclusive scan of sh.cnt[0 .. n) in place into sh.base (warp 0), total in sh.base[n].
// Callers bracket it with barriers.
__device__ __forceinline__ void sr_scan_counts(SrShared& sh, int n) {
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    int carry = 0;
    for (int c0 = 0; c0 < n; c0 += 32) {
        const int v = c0 + lane < n ? sh.cnt[c0 + lane] : 0;
        const int inc = warp_incl_scan(v);
        if (c0 + lane < n) sh.base[c0 + lane] = carry + inc - v;
        carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) sh.base[n] = carry;
}

// Marks in `sel` the k eligible entries with the largest keys, equal keys in ascending j.
// Requires 0 < k < (number of eligible entries).  `pass` counts histogram passes across
// calls (buffer rotation); on entry buffers pass % 3 and (pass + 1) % 3 are zero, and
// every pass leaves that so for the next one, also when the digits stop early.
template <int KPT>
__device__ void sr_top(const uint32_t (&key)[KPT], uint32_t elig, uint32_t& sel, int k, int& pass, SrShared& sh) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint32_t prefix = 0, mask = 0;
    int kk = k, n_eq = 0;
    for (int d = 0; d < 4; ++d, ++pass) {
        const int shift = 24 - 8 * d;
        int* h = sh.hist[pass % 3];
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
            const bool in = ((elig >> i) & 1u) && (key[i] & mask) == prefix;
            sr_hist_add(h, in ? (int)((key[i] >> shift) & 255u) : -1);
        }
        __syncthreads();
        // every warp: lane l holds bins 255-8l .. 248-8l (descending key order), read as two
        // 16-byte vectors (a warp reads the 1 KB histogram without bank conflicts)
        const int4 v_hi = reinterpret_cast<const int4*>(h)[63 - 2 * lane];
        const int4 v_lo = reinterpret_cast<const int4*>(h)[62 - 2 * lane];
        const int cnt[8] = {v_hi.w, v_hi.z, v_hi.y, v_hi.x, v_lo.w, v_lo.z, v_lo.y, v_lo.x};
        int sum = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) sum += cnt[b];
        const int inc = warp_incl_scan(sum);
        const unsigned ball = __ballot_sync(0xffffffffu, inc >= kk);
        const int src = __ffs(ball) - 1;
        int above = inc - sum, digit = 0, nbin = 0;
#pragma unroll
        for (int b = 0, found = 0; b < 8; ++b) {
            if (!found) {
                if (above + cnt[b] >= kk) { digit = 255 - 8 * lane - b; nbin = cnt[b]; found = 1; }
                else above += cnt[b];
            }
        }
        digit = __shfl_sync(0xffffffffu, digit, src);
        above = __shfl_sync(0xffffffffu, above, src);
        nbin = __shfl_sync(0xffffffffu, nbin, src);
        // the buffer filled two passes from now was last read before this pass's barrier
        if (tid < 256) sh.hist[(pass + 2) % 3][tid] = 0;
        prefix |= (uint32_t)digit << shift;
        mask |= 0xFFu << shift;
        kk -= above;
        n_eq = nbin;
        if (kk == nbin && d < 3) {
            // every key of the threshold bin is taken: the selection is the eligible keys
            // whose digits so far are >= the prefix, and no tie is left to rank
            ++pass;
#pragma unroll
            for (int i = 0; i < KPT; ++i)
                if (((elig >> i) & 1u) && (key[i] & mask) >= prefix) sel |= 1u << i;
            return;
        }
    }
    // keys above the threshold, then the first kk of the keys equal to it
    uint32_t eq = 0;
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
        if (!((elig >> i) & 1u)) continue;
        if (key[i] > prefix) sel |= 1u << i;
        else if (key[i] == prefix) eq |= 1u << i;
    }
    if (kk == n_eq) {
        sel |= eq;
        return;
    }
    // tie ranks in (i, t) order
    unsigned ball[KPT];
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
        ball[i] = __ballot_sync(0xffffffffu, (eq >> i) & 1u);
        if (lane == 0) sh.cnt[i * kSrWarps + wid] = __popc(ball[i]);
    }
    __syncthreads();
    sr_scan_counts(sh, KPT * kSrWarps);
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < KPT; ++i)
        if (((eq >> i) & 1u) && sh.base[i * kSrWarps + wid] + __popc(ball[i] & lt) < kk) sel |= 1u << i;
    __syncthreads();  // sh.cnt / sh.base are reused
}

// Writes the ascending list of selected j (and the bitmap); returns the count.
template <int KPT>
__device__ int sr_compact(uint32_t sel, int32_t* out, SrShared& sh) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    unsigned ball[KPT];
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
        ball[i] = __ballot_sync(0xffffffffu, (sel >> i) & 1u);
        if (lane == 0) {
            sh.cnt[i * kSrWarps + wid] = __popc(ball[i]);
            sh.bitmap[i * kSrWarps + wid] = ball[i];
        }
    }
    __syncthreads();
    sr_scan_counts(sh, KPT * kSrWarps);
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < KPT; ++i)
        if ((sel >> i) & 1u) out[sh.base[i * kSrWarps + wid] + __popc(ball[i] & lt)] = i * kSrThreads + tid;
    return sh.base[KPT * kSrWarps];
}

template <int KPT>
__global__ void __launch_bounds__(kSrThreads, 1) select_reg_kernel(
    spin_config cfg, const int32_t* __restrict__ warm, const int32_t* __restrict__ n_slots,
    const int32_t* __restrict__ q_pos, int rows, const int32_t* __restrict__ rho_override, uint64_t step,
    int layer, const float* __restrict__ S, const uint32_t* __restrict__ X, int32_t* __restrict__ blocks,
    int32_t* __restrict__ n_blocks, int32_t* __restrict__ union_blocks, int32_t* __restrict__ n_union,
    uint32_t* status) {
    pdl_begin();
    __shared__ SrShared sh;
    const Dims dm = dims_of(cfg);
    const int MB = dm.MB;
    {   // layer blockIdx.y of a stack of layers (0 for a one-layer call)
        const int64_t l = blockIdx.y;
        warm += l * dm.R;
        if (rho_override) rho_override += l;
        S += l * dm.R * rows * MB;
        X += l * dm.R * rows * MB;
        blocks += l * dm.R * rows * MB;
        n_blocks += l * dm.R * rows;
        if (union_blocks) union_blocks += l * dm.R * MB;
        if (n_union) n_union += l * dm.R;
        layer += (int)l;
    }
    const int tid = threadIdx.x;
    const int req = blockIdx.x / rows, r = blockIdx.x % rows;  // a cluster = the rows of a request
    const int64_t rr = (int64_t)req * rows + r;
    // the row's block scores and exploration draws are loaded up front, together with the
    // request's sizes (entries at j >= N/64 are not used)
    float sv[KPT];
    uint32_t xv[KPT];
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
        const int j = i * kSrThreads + tid;
        sv[i] = j < MB ? __ldg(S + rr * MB + j) : 0.0f;
        xv[i] = j < MB ? __ldg(X + rr * MB + j) : 0u;
    }
    const int64_t n = n_slots[req], q = q_pos[req];
    uint32_t bad = request_check(n, q, rows, dm);
    int32_t rho = cfg.rho_bp;
    if (rho_override) {
        rho = *rho_override;
        if (rho < 0 || rho > 10000) bad |= SPIN_STATUS_BAD_RHO;
    }
    // (bad is uniform over the cluster: it depends on the request only)
    if (bad) {
        if (tid == 0) {
            if (r == 0) set_status(status, bad);
            n_blocks[rr] = 0;
            if (r == 0 && union_blocks && n_union) n_union[req] = 0;
        }
        return;
    }
    const int nb = (int)((n + kBlock - 1) / kBlock);
    for (int b = tid; b < 3 * 256; b += kSrThreads) (&sh.hist[0][0])[b] = 0;
    uint32_t valid = 0, sel = 0;
#pragma unroll
    for (int i = 0; i < KPT; ++i)
        if (i * kSrThreads + tid < nb) valid |= 1u << i;
    if (warm[req] == 0 || nb <= 2 || budget_blocks(nb, cfg.top_k, rho) >= nb) {
        // dense: the warm-up step, contexts whose every block is forced, and budgets of
        // every block (forced, top and exploration blocks then cover all of them)
        sel = valid;
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
        uint32_t key[KPT];
        uint32_t elig = 0;
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
            const int j = i * kSrThreads + tid;
            key[i] = 0;
            if (j < nb) {
                if (j == 0 || j == nb - 1) sel |= 1u << i;
                else { key[i] = order_key(sv[i]); elig |= 1u << i; }
            }
        }
        __syncthreads();  // histogram buffers cleared
        int pass = 0;
        const int64_t n_rest = (int64_t)nb - f;
        if (t >= n_rest) sel |= elig;
        else if (t > 0) sr_top<KPT>(key, elig, sel, (int)t, pass, sh);
        if (e > 0) {
            const int64_t n_left = n_rest - t;
            uint32_t elig2 = 0;
#pragma unroll
            for (int i = 0; i < KPT; ++i) {
                if (((elig >> i) & 1u) && !((sel >> i) & 1u)) {
                    elig2 |= 1u << i;
                    // smallest Philox key first == largest complement
                    key[i] = ~xv[i];
                }
            }
            if (e >= n_left) sel |= elig2;
            else sr_top<KPT>(key, elig2, sel, (int)e, pass, sh);
        }
    }
    const int cnt = sr_compact<KPT>(sel, blocks + rr * MB, sh);
    if (tid == 0) n_blocks[rr] = cnt;
    if (rows > 1 && union_blocks && n_union) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();  // every row's bitmap is complete
        if (cluster.block_rank() == 0) {
            const int nwords = (nb + 31) / 32;
            uint32_t u = 0;
            if (tid < nwords)
                for (int p = 0; p < rows; ++p) u |= cluster.map_shared_rank(sh.bitmap, p)[tid];
            // the bitmap words beyond nb's are zero: rows select only j < nb
            int total;
            const int pos0 = block_excl_scan(tid < nwords ? __popc(u) : 0, sh.base, &total);
            int pos = pos0;
            while (u) {
                const int b = __ffs(u) - 1;
                u &= u - 1u;
                union_blocks[(int64_t)req * MB + pos++] = tid * 32 + b;
            }
            if (tid == 0) n_union[req] = total;
        }
        cluster.sync();  // the first CTA has finished reading the others' shared memory
    } else if (union_blocks && n_union) {
        // one row: the union is the row's list
        int32_t* out = union_blocks + (int64_t)req * MB;
        const int32_t* in = blocks + rr * MB;
        __syncthreads();
        for (int c = tid; c < cnt; c += kSrThreads) out[c] = in[c];
        if (tid == 0) n_union[req] = cnt;
    }
}

// ---------------------------------------------------------------------------------------
// A0 (the §4.6 block-reduction ablation, SPIN_POOL_SLOTS): the K slots with the largest
// predicted score (ties: lower slot) are found by the library's top-K over the predictions,
// then expanded to the blocks holding them, with the forced sink and newest blocks; no
// exploration.  Cold requests and budgets of every block select every block, as under A1.
// ---------------------------------------------------------------------------------------

// Predicted slot scores Z [R][rows][MB * 64] in slot order (0 past the context), the
// identity block list [R][MB] and its length nb per request (0 for a request that fails its
// checks, so the top-K skips it).
__global__ void __launch_bounds__(256) slot_pred_kernel(spin_config cfg, const float* __restrict__ V,
                                                        const float* __restrict__ D,
                                                        const int32_t* __restrict__ n_slots,
                                                        const int32_t* __restrict__ q_pos, int rows,
                                                        float* __restrict__ Z, int32_t* __restrict__ list,
                                                        int32_t* __restrict__ n_list) {
    pdl_begin();
    const Dims dm = dims_of(cfg);
    const int rr = blockIdx.y;
    const int req = rr / rows, r = rr - req * rows;
    const int64_t n = n_slots[req], q = q_pos[req];
    const bool ok = request_check(n, q, rows, dm) == 0u;
    const int64_t nb = ok ? (n + kBlock - 1) / kBlock : 0;
    const int64_t qr = q + r;
    const float* Vq = V + (int64_t)req * dm.max_slots;
    const float* Dq = D + (int64_t)req * dm.DL;
    float* Zq = Z + (int64_t)rr * dm.MB * kBlock;
    const bool sum = cfg.combine == SPIN_COMBINE_SUM;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nb * kBlock; i += stride) {
        float z = 0.0f;
        if (i < n) {
            const float v = Vq[i], d = Dq[qr - i];
            z = sum ? __fadd_rn(v, d) : fmaxf(v, d);
        }
        Zq[i] = z;
    }
    if (r == 0) {
        for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < nb; j += stride)
            list[(int64_t)req * dm.MB + j] = (int32_t)j;
        if (blockIdx.x == 0 && threadIdx.x == 0) n_list[req] = (int32_t)nb;
    }
}

// One CTA per request: each row's block set (a bitmap of MB bits in shared memory) from its
// K slot indices and the forced blocks, written in ascending order; the rows' union.
constexpr int kExpThreads = 1024;

__device__ void expand_write(const uint32_t* bits, int nwords, int32_t* out, int32_t* count, int* scan) {
    // ordered compaction of the set bits: a CTA scan of per-thread popcounts
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int per = (nwords + kExpThreads - 1) / kExpThreads;
    const int w0 = tid * per, w1 = min(w0 + per, nwords);
    int c = 0;
    for (int w = w0; w < w1; ++w) c += __popc(bits[w]);
    const int inc = warp_incl_scan(c);
    if (lane == 31) scan[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        const int v = lane < kExpThreads / 32 ? scan[lane] : 0;
        const int vi = warp_incl_scan(v);
        if (lane < kExpThreads / 32) scan[lane] = vi - v;
        if (lane == 31) scan[32] = vi;
    }
    __syncthreads();
    int pos = scan[wid] + inc - c;
    for (int w = w0; w < w1; ++w) {
        uint32_t u = bits[w];
        while (u) {
            const int b = __ffs(u) - 1;
            u &= u - 1u;
            out[pos++] = w * 32 + b;
        }
    }
    if (tid == 0) *count = scan[32];
    __syncthreads();
}

__global__ void __launch_bounds__(kExpThreads) slot_expand_kernel(
    spin_config cfg, const int32_t* __restrict__ warm, const int32_t* __restrict__ n_slots,
    const int32_t* __restrict__ q_pos, int rows, const int32_t* __restrict__ rho_override,
    const int32_t* __restrict__ topk_idx, int32_t* __restrict__ blocks, int32_t* __restrict__ n_blocks,
    int32_t* __restrict__ union_blocks, int32_t* __restrict__ n_union, uint32_t* status) {
    pdl_begin();
    extern __shared__ uint32_t xbits[];  // [2][MB / 32]: a row's blocks, the union
    __shared__ int scan[33];
    const Dims dm = dims_of(cfg);
    const int MB = dm.MB, nw = (MB + 31) / 32;
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
    const int64_t nb = (n + kBlock - 1) / kBlock;
    const bool dense = warm[req] == 0 || nb <= 2 || budget_blocks(nb, cfg.top_k, rho) >= nb;
    uint32_t* rowb = xbits;
    uint32_t* unib = xbits + nw;
    for (int w = tid; w < nw; w += kExpThreads) unib[w] = 0u;
    for (int r = 0; r < rows; ++r) {
        const int64_t rr = (int64_t)req * rows + r;
        __syncthreads();
        for (int w = tid; w < nw; w += kExpThreads) {
            uint32_t v = 0u;
            if (dense) {  // every block j < nb
                const int64_t lo = (int64_t)w * 32;
                if (lo + 32 <= nb) v = 0xffffffffu;
                else if (lo < nb) v = (1u << (nb - lo)) - 1u;
            }
            rowb[w] = v;
        }
        __syncthreads();
        if (!dense) {
            const int32_t* ti = topk_idx + rr * cfg.top_k;
            for (int k = tid; k < cfg.top_k; k += kExpThreads) {
                const int32_t i = ti[k];
                if (i >= 0 && i < n) {
                    const int j = i / kBlock;
                    atomicOr(&rowb[j >> 5], 1u << (j & 31));
                }
            }
            if (tid == 0) {
                atomicOr(&rowb[0], 1u);
                const int last = (int)nb - 1;
                atomicOr(&rowb[last >> 5], 1u << (last & 31));
            }
            __syncthreads();
        }
        for (int w = tid; w < nw; w += kExpThreads) unib[w] |= rowb[w];
        expand_write(rowb, nw, blocks + rr * MB, n_blocks + rr, scan);
    }
    if (union_blocks && n_union) {
        __syncthreads();
        expand_write(unib, nw, union_blocks + (int64_t)req * MB, n_union + req, scan);
    }
}

// Workspace of A0: Z [R][rows][MB * 64] fp32, the identity list [R][MB] and its lengths [R],
// the top-K slots [R][rows][K], each 256-byte aligned.
static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

static size_t slots_workspace_bytes(const spin_config& cfg, int rows) {
    const Dims dm = dims_of(cfg);
    const size_t rrows = (size_t)dm.R * (size_t)rows;
    return align256(sizeof(float) * rrows * (size_t)dm.MB * kBlock) + align256(sizeof(int32_t) * (size_t)dm.R * dm.MB) +
           align256(sizeof(int32_t) * (size_t)dm.R) + align256(sizeof(int32_t) * rrows * (size_t)cfg.top_k);
}

// Every layer of a stack in turn: predictions, the library's top-K over them, expansion.
static cudaError_t launch_select_slots(const spin_config& cfg, const SelectArgs& a, cudaStream_t s) {
    const Dims dm = dims_of(cfg);
    const int L = a.n_layers > 1 ? a.n_layers : 1;
    const size_t per_layer = slots_workspace_bytes(cfg, a.rows);
    const int64_t rrows = (int64_t)dm.R * a.rows;
    const size_t xsmem = sizeof(uint32_t) * 2 * (size_t)((dm.MB + 31) / 32);
    if (xsmem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(slot_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)xsmem);
        if (e != cudaSuccess) return e;
    }
    for (int l = 0; l < L; ++l) {
        unsigned char* ws = reinterpret_cast<unsigned char*>(a.block_scores) + (size_t)l * per_layer;
        float* Z = reinterpret_cast<float*>(ws);
        ws += align256(sizeof(float) * (size_t)rrows * dm.MB * kBlock);
        int32_t* list = reinterpret_cast<int32_t*>(ws);
        ws += align256(sizeof(int32_t) * (size_t)dm.R * dm.MB);
        int32_t* n_list = reinterpret_cast<int32_t*>(ws);
        ws += align256(sizeof(int32_t) * (size_t)dm.R);
        int32_t* topk_idx = reinterpret_cast<int32_t*>(ws);
        const float* V = a.V + (int64_t)l * dm.R * dm.max_slots;
        const float* D = a.D + (int64_t)l * dm.R * dm.DL;
        int gx = (int)((dm.MB * (int64_t)kBlock + 255) / 256);
        if (gx > 64) gx = 64;
        cudaError_t e = launch_pdl(slot_pred_kernel, dim3((unsigned)gx, (unsigned)rrows), dim3(256), 0, s, nullptr, 0,
                                   cfg, V, D, a.n_slots, a.q_pos, a.rows, Z, list, n_list);
        if (e != cudaSuccess) return e;
        e = launch_topk(cfg, Z, list, n_list, a.n_slots, a.rows, topk_idx, a.status, s);
        if (e != cudaSuccess) return e;
        e = launch_pdl(slot_expand_kernel, dim3((unsigned)dm.R), dim3(kExpThreads), xsmem, s, nullptr, 0, cfg,
                       a.warm + (int64_t)l * dm.R, a.n_slots, a.q_pos, a.rows,
                       a.rho_override ? a.rho_override + l : nullptr, (const int32_t*)topk_idx,
                       a.blocks + (int64_t)l * rrows * dm.MB, a.n_blocks + (int64_t)l * rrows,
                       a.union_blocks ? a.union_blocks + (int64_t)l * dm.R * dm.MB : nullptr,
                       a.n_union ? a.n_union + (int64_t)l * dm.R : nullptr, a.status);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Workspace: block scores S [R][rows][MB] (fp32), then exploration draws X [R][rows][MB]
// (u32), each 256-byte aligned.
static size_t select_array_bytes(const spin_config& cfg, int rows) {
    const Dims dm = dims_of(cfg);
    const size_t b = sizeof(float) * (size_t)dm.R * (size_t)rows * (size_t)dm.MB;
    return (b + 255) & ~(size_t)255;
}

size_t select_workspace_bytes(const spin_config& cfg, int rows) {
    if (cfg.pooling == SPIN_POOL_SLOTS) return slots_workspace_bytes(cfg, rows);
    return 2 * select_array_bytes(cfg, rows);
}

// Layer stacks: every array of layer l starts l layer-sizes after layer 0's; the workspace
// holds the n_layers block-score arrays, then the n_layers exploration-draw arrays.
cudaError_t launch_select(const spin_config& cfg, const SelectArgs& a, cudaStream_t s) {
    if (cfg.pooling == SPIN_POOL_SLOTS) return launch_select_slots(cfg, a, s);
    const Dims dm = dims_of(cfg);
    const int L = a.n_layers > 1 ? a.n_layers : 1;
    const bool many_rows = (int64_t)dm.R * a.rows * L >= 8;
    const int per_cta = (256 / 32) * (many_rows ? 16 : 8);
    int gx = (dm.MB + per_cta - 1) / per_cta;
    if (gx > 512) gx = 512;
    dim3 g1(gx, dm.R * a.rows, L);
    float* S = a.block_scores;
    uint32_t* X = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(a.block_scores) +
                                              (size_t)L * select_array_bytes(cfg, a.rows));
    cudaError_t e = launch_pdl(many_rows ? block_score_kernel<16> : block_score_kernel<8>, g1, dim3(256), 0, s,
                               nullptr, 0, cfg, a.V, a.D, a.Vmax, a.warm, a.n_slots, a.q_pos, a.rows,
                               a.rho_override, cfg.seed, a.step, a.step_dev, a.layer, a.block_age, S, X);
    if (e != cudaSuccess) return e;
    if (dm.MB <= kSrMaxBlocks && a.rows >= 1 && a.rows <= 8) {
        const int kpt = dm.MB <= kSrThreads ? 1 : dm.MB <= 2 * kSrThreads ? 2 : dm.MB <= 4 * kSrThreads ? 4
                        : dm.MB <= 8 * kSrThreads ? 8 : 16;
        void (*kern)(spin_config, const int32_t*, const int32_t*, const int32_t*, int, const int32_t*, uint64_t,
                     int, const float*, const uint32_t*, int32_t*, int32_t*, int32_t*, int32_t*, uint32_t*) =
            kpt == 1 ? select_reg_kernel<1> : kpt == 2 ? select_reg_kernel<2> : kpt == 4 ? select_reg_kernel<4>
            : kpt == 8 ? select_reg_kernel<8> : select_reg_kernel<16>;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)a.rows;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        return launch_pdl(kern, dim3((unsigned)(dm.R * a.rows), (unsigned)L), dim3(kSrThreads), 0, s, at, 1, cfg, a.warm,
                          a.n_slots, a.q_pos, a.rows, a.rho_override, a.step, a.layer, (const float*)S,
                          (const uint32_t*)X, a.blocks, a.n_blocks, a.union_blocks, a.n_union, a.status);
    }
    const size_t smem = ((size_t)dm.MB * 6 + 15) & ~(size_t)15;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(select_kernel, dim3(dm.R, L), dim3(kSelThreads), smem, s, nullptr, 0, cfg, a.warm, a.n_slots,
                      a.q_pos, a.rows, a.rho_override, a.step, a.layer, (const float*)a.block_scores, a.blocks,
                      a.n_blocks, a.union_blocks, a.n_union, a.status, a.step_dev, a.block_age);
}

}  // namespace spin

// spin_ema.cu -- EMA update and the deferred MTP replay.
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention":
//   Algorithm 1's EMA update: for every scored slot i,
//       V[i]   <- alpha V[i]   + (1 - alpha) z[i]
//       D[q-i] <- alpha D[q-i] + (1 - alpha) z[i]
//   §3.2.2: with a drafts accepted, the observations of verifier rows 0..a are replayed in
//   order (row r at position q + r); rows above a are discarded.
//
// Both are one kernel: a CTA owns 1024 consecutive slots of one request.  V[i] is a chain
// over the rows r = 0..a at slot i; D[o] is a chain over r at offset o, the slot being
// i = q + r - o.  The CTA owning slot i0 owns offset q - i0 (and the CTA of slot 0 also the
// offsets q+1..q+a), so every location is written by one thread that applies its updates
// in row order: the result is bit-identical to a sequential replay.  The arithmetic is
// t = fl((1 - alpha) z), v = fma(alpha, v, t), with (1 - alpha) rounded to fp32 once.
// Afterwards Vmax (the per-block max of V that block prediction reads) is refreshed for
// the CTA's listed blocks.
#include <float.h>

#include "spin_common.cuh"
#include "spin_internal.h"

namespace spin {

constexpr int kEmaSpan = 1024;
constexpr int kEmaThreads = 256;
constexpr int kEmaMapBlocks = kEmaSpan / kBlock + 2;

// Layer blockIdx.z of a stack of layers: its arrays start l layer-sizes after layer 0's.
__device__ __forceinline__ void ema_layer_offsets(const Dims& dm, EmaArgs& a) {
    const int64_t l = blockIdx.z;
    if (l == 0) return;
    a.V += l * dm.R * dm.max_slots;
    a.D += l * dm.R * dm.DL;
    a.Vmax += l * dm.R * dm.MB;
    a.warm += l * dm.R;
    a.scores += l * dm.R * a.rows * dm.MB * kBlock;
    a.list += l * dm.R * dm.MB;
    a.n_list += l * dm.R;
}

__global__ void __launch_bounds__(kEmaThreads) ema_replay_kernel(spin_config cfg, EmaArgs a) {
    pdl_begin();
    extern __shared__ float zs[];  // [(a+1)][span]
    __shared__ int pos[kEmaMapBlocks];
    const Dims dm = dims_of(cfg);
    ema_layer_offsets(dm, a);
    const int req = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    const int rows = a.rows;
    const int64_t n = a.n_slots[req], q = a.q_pos[req], cnt = a.n_list[req];
    const int A = a.accepted ? a.accepted[req] : 0;
    uint32_t bad = request_check(n, q, rows, dm);
    if (cnt < 0 || cnt > dm.MB) bad |= SPIN_STATUS_BAD_LIST;
    if (A < 0 || A >= rows) bad |= SPIN_STATUS_BAD_ACCEPTED;
    if (bad) {
        if (c == 0 && tid == 0) set_status(a.status, bad);
        return;
    }
    if (c == 0 && tid == 0) a.warm[req] = 1;
    const int64_t lo = (int64_t)c * kEmaSpan;
    if (lo >= n && c > 0) return;
    const int64_t hi = (lo + kEmaSpan < n) ? lo + kEmaSpan : n;  // may be <= lo when n == 0
    const int64_t nb = (n + kBlock - 1) / kBlock;
    const int64_t blk_lo = lo / kBlock;
    const int64_t span = (hi > lo ? hi - lo : 0) + A;  // staged slots [lo, lo + span)
    const int32_t* lst = a.list + (int64_t)req * dm.MB;

    // union position of each block touching [lo, lo + span), or -1: warp 0 finds the first
    // list entry >= blk_lo with a 32-way search (a few dependent loads), then maps the
    // next entries
    if (tid < 32) {
        const int lane = tid;
        int64_t l = 0, h = cnt;  // the answer lies in [l, h]
        while (h - l > 32) {
            const int64_t step = (h - l + 31) / 32;
            const int64_t p = l + (int64_t)lane * step;
            const bool ge = p >= h || lst[p] >= blk_lo;
            const unsigned b = __ballot_sync(0xffffffffu, ge);
            if (b == 0u) {
                l = l + 31 * step + 1;
            } else {
                const int f = __ffs(b) - 1;
                if (f == 0) { h = l; }
                else {
                    const int64_t hf = l + (int64_t)f * step;
                    h = hf < h ? hf : h;
                    l = l + (int64_t)(f - 1) * step + 1;
                }
            }
        }
        const int64_t p = l + lane;
        const bool ge = p >= h || lst[p] >= blk_lo;
        const unsigned b = __ballot_sync(0xffffffffu, ge);
        const int64_t first = b ? l + (__ffs(b) - 1) : h;
        if (lane < kEmaMapBlocks) pos[lane] = -1;
        __syncwarp();
        bool bad_list = false;
        const int64_t k = first + lane;
        if (lane < kEmaMapBlocks && k < cnt) {
            const int64_t blk = lst[k];
            if (blk < 0 || blk >= nb) bad_list = true;
            else if (blk - blk_lo < kEmaMapBlocks) pos[blk - blk_lo] = (int)k;
        }
        if (__any_sync(0xffffffffu, bad_list) && lane == 0) set_status(a.status, SPIN_STATUS_BAD_LIST);
    }
    __syncthreads();
    auto scored = [&](int64_t i) -> int {  // union position of slot i's block, or -1
        if (i < 0 || i >= n || i < lo) return -1;
        const int64_t b = i / kBlock - blk_lo;
        return (b < kEmaMapBlocks) ? pos[b] : -1;
    };

    // stage the observations z_r[i], r <= A, i in [lo, lo + span)
    for (int64_t idx = tid; idx < (int64_t)(A + 1) * span; idx += kEmaThreads) {
        const int r = (int)(idx / span);
        const int64_t i = lo + (idx - (int64_t)r * span);
        const int p = scored(i);
        zs[idx] = p >= 0 ? a.scores[(((int64_t)req * rows + r) * dm.MB + p) * kBlock + (i & 63)] : 0.0f;
    }
    __syncthreads();

    const float alpha = cfg.alpha;
    const float oma = 1.0f - cfg.alpha;
    float* Vq = a.V + (int64_t)req * dm.max_slots;
    float* Dq = a.D + (int64_t)req * dm.DL;

    // V chains
    for (int64_t i = lo + tid; i < hi; i += kEmaThreads) {
        if (scored(i) < 0) continue;
        float v = Vq[i];
        for (int r = 0; r <= A; ++r) v = __fmaf_rn(alpha, v, __fmul_rn(oma, zs[(int64_t)r * span + (i - lo)]));
        Vq[i] = v;
    }
    // D chains: offsets o = q - i0 for i0 in [lo_d, hi)
    const int64_t lo_d = (c == 0) ? -(int64_t)A : lo;
    for (int64_t i0 = lo_d + tid; i0 < hi; i0 += kEmaThreads) {
        const int64_t o = q - i0;
        float d = 0.0f;
        bool any = false;
        for (int r = 0; r <= A; ++r) {
            const int64_t i = i0 + r;
            if (scored(i) < 0) continue;
            if (!any) { d = Dq[o]; any = true; }
            d = __fmaf_rn(alpha, d, __fmul_rn(oma, zs[(int64_t)r * span + (i - lo)]));
        }
        if (any) Dq[o] = d;
    }
    __syncthreads();

    // Vmax of the listed blocks that start inside [lo, hi): one warp per block
    const int lane = tid & 31, wid = tid >> 5;
    for (int b = wid; b < kEmaSpan / kBlock; b += kEmaThreads / 32) {
        const int64_t blk = blk_lo + b;
        if (blk * kBlock >= hi || pos[b] < 0) continue;
        const int64_t i0 = blk * kBlock + lane, i1 = i0 + 32;
        float m = -FLT_MAX;
        if (i0 < dm.max_slots) m = Vq[i0];
        if (i1 < dm.max_slots) m = fmaxf(m, Vq[i1]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) a.Vmax[(int64_t)req * dm.MB + blk] = m;
    }
}

// ---------------------------------------------------------------------------------------
// One-row update (a = 0): each listed slot i is updated once and its offset q - i is
// distinct, so the work splits by list entry with no ordering between threads.  A warp
// takes two list entries (128 slots) per step, issues all their loads together, and
// refreshes the two blocks' Vmax with a warp max; the warps of a request's CTAs stride
// over its list, each reading the next step's list entries before this step's slots.
// ---------------------------------------------------------------------------------------
constexpr int kEmaListWarps = 8;  // warps per CTA

__global__ void __launch_bounds__(256) ema_list_kernel(spin_config cfg, EmaArgs a) {
    pdl_begin();
    const Dims dm = dims_of(cfg);
    ema_layer_offsets(dm, a);
    const int req = blockIdx.y, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t n = a.n_slots[req], q = a.q_pos[req], cnt = a.n_list[req];
    uint32_t bad = request_check(n, q, 1, dm);
    if (cnt < 0 || cnt > dm.MB) bad |= SPIN_STATUS_BAD_LIST;
    if (bad) {
        if (blockIdx.x == 0 && tid == 0) set_status(a.status, bad);
        return;
    }
    if (blockIdx.x == 0 && tid == 0) a.warm[req] = 1;
    const int64_t nb = (n + kBlock - 1) / kBlock;
    const float alpha = cfg.alpha;
    const float oma = 1.0f - cfg.alpha;
    float* Vq = a.V + (int64_t)req * dm.max_slots;
    float* Dq = a.D + (int64_t)req * dm.DL;
    const int32_t* lst = a.list + (int64_t)req * dm.MB;
    const float* zq = a.scores + (int64_t)req * dm.MB * kBlock;
    if (cfg.pooling == SPIN_POOL_A2) {
        // the A2 ablation (§4.6): one observation per scored block, its max over the slots
        // i < N, into the block-level EMAs (Vb[j] in V, Db at floor(q / 64) - j in D)
        const int64_t qb = q / kBlock;
        for (int64_t k = (int64_t)blockIdx.x * kEmaListWarps + wid; k < cnt;
             k += (int64_t)gridDim.x * kEmaListWarps) {
            const int64_t blk = lst[k];
            if (!(blk >= 0 && blk < nb)) {  // (warp-uniform)
                if (lane == 0) set_status(a.status, SPIN_STATUS_BAD_LIST);
                continue;
            }
            float m = -INFINITY;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                if (blk * kBlock + lane + 32 * hh < n) m = fmaxf(m, zq[k * kBlock + lane + 32 * hh]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) {
                const float t = __fmul_rn(oma, m);
                Vq[blk] = __fmaf_rn(alpha, Vq[blk], t);
                Dq[qb - blk] = __fmaf_rn(alpha, Dq[qb - blk], t);
                if (a.block_age) a.block_age[(int64_t)req * dm.MB + blk] = (uint32_t)(a.age_step + 1);
            }
        }
        return;
    }
    const int64_t stride = 2 * (int64_t)gridDim.x * kEmaListWarps;
    int64_t k0 = 2 * ((int64_t)blockIdx.x * kEmaListWarps + wid);
    int64_t nxt[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) nxt[e] = k0 + e < cnt ? lst[k0 + e] : -1;
    for (; k0 < cnt; k0 += stride) {
        int64_t blk[2];
        bool ok[2];
        float z[2][2], v[2][2], d[2][2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int64_t k = k0 + e;
            blk[e] = nxt[e];
            ok[e] = blk[e] >= 0 && blk[e] < nb;
            if (k < cnt && !ok[e] && lane == 0) set_status(a.status, SPIN_STATUS_BAD_LIST);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int64_t i = blk[e] * kBlock + lane + 32 * hh;
                const bool live = ok[e] && i < n;
                z[e][hh] = live ? zq[k * kBlock + lane + 32 * hh] : 0.0f;
                v[e][hh] = (ok[e] && i < dm.max_slots) ? Vq[i] : 0.0f;
                d[e][hh] = live ? Dq[q - i] : 0.0f;
            }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) nxt[e] = k0 + stride + e < cnt ? lst[k0 + stride + e] : -1;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            if (!ok[e]) continue;  // warp-uniform
            float m = -FLT_MAX;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int64_t i = blk[e] * kBlock + lane + 32 * hh;
                if (i < n) {
                    const float t = __fmul_rn(oma, z[e][hh]);
                    v[e][hh] = __fmaf_rn(alpha, v[e][hh], t);
                    Vq[i] = v[e][hh];
                    Dq[q - i] = __fmaf_rn(alpha, d[e][hh], t);
                }
                if (i < dm.max_slots) m = fmaxf(m, v[e][hh]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) {
                a.Vmax[(int64_t)req * dm.MB + blk[e]] = m;
                // block-age exploration (§4.6): the block was observed at this step
                if (a.block_age) a.block_age[(int64_t)req * dm.MB + blk[e]] = (uint32_t)(a.age_step + 1);
            }
        }
    }
}

cudaError_t launch_ema(const spin_config& cfg, const EmaArgs& a, cudaStream_t s) {
    const Dims dm = dims_of(cfg);
    const int L = a.n_layers > 1 ? a.n_layers : 1;
    if (a.accepted == nullptr && a.rows == 1) {
        // about eight CTAs per SM over all requests, at most one step per warp for the longest list
        const int full = (dm.MB + 2 * kEmaListWarps - 1) / (2 * kEmaListWarps);
        const int want = (device_sm_count() * 8 + dm.R * L - 1) / (dm.R * L);
        dim3 grid(want < full ? (want > 0 ? want : 1) : full, dm.R, L);
        return launch_pdl(ema_list_kernel, grid, dim3(256), 0, s, nullptr, 0, cfg, a);
    }
    const int gx = (dm.max_slots + kEmaSpan - 1) / kEmaSpan;
    dim3 grid(gx > 0 ? gx : 1, dm.R, L);
    const size_t smem = sizeof(float) * (size_t)a.rows * (kEmaSpan + a.rows);
    return launch_pdl(ema_replay_kernel, grid, dim3(kEmaThreads), smem, s, nullptr, 0, cfg, a);
}

// ---------------------------------------------------------------------------------------
// Reset after prefill / at a turn start (§3.2 practical details).
// ---------------------------------------------------------------------------------------
__global__ void init_state_kernel(spin_config cfg, float* V, float* D, float* Vmax, int32_t* warm, int req0,
                                  int nreq) {
    pdl_begin();
    const Dims dm = dims_of(cfg);
    const int64_t nv = (int64_t)nreq * dm.max_slots, nd = (int64_t)nreq * dm.DL, nm = (int64_t)nreq * dm.MB;
    float* V0 = V + (int64_t)req0 * dm.max_slots;
    float* D0 = D + (int64_t)req0 * dm.DL;
    float* M0 = Vmax + (int64_t)req0 * dm.MB;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv + nd + nm + nreq; i += stride) {
        if (i < nv) V0[i] = 0.0f;
        else if (i < nv + nd) D0[i - nv] = 0.0f;
        else if (i < nv + nd + nm) M0[i - nv - nd] = 0.0f;
        else warm[req0 + (i - nv - nd - nm)] = 0;
    }
}

cudaError_t launch_init_state(const spin_config& cfg, float* V, float* D, float* Vmax, int32_t* warm, int req,
                              cudaStream_t s) {
    const int req0 = req < 0 ? 0 : req;
    const int nreq = req < 0 ? cfg.n_req : 1;
    const int grid = device_sm_count() * 4;
    return launch_pdl(init_state_kernel, dim3(grid), dim3(256), 0, s, nullptr, 0, cfg, V, D, Vmax, warm, req0,
                      nreq);
}

}  // namespace spin

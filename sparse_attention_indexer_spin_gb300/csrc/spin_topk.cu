// spin_topk.cu -- post-indexer top-K over the freshly scored slots.
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention", Algorithm 1 line 7:
// T_t = TopK(z_t, K) over the slots the indexer scored (the selected blocks), which then
// feeds core attention.  Equal scores at the K-th value go to the lower slot id.
//
// The candidates are the listed blocks' slots i < N, visited in list order, which is
// ascending slot order because block lists are ascending.  A three-pass radix select
// (11 + 11 + 10 bits of the order-preserving 32-bit key) finds the K-th key T and how many
// keys equal to T to keep; one ordered pass then writes the kept slot ids in ascending
// order and pads with -1.  The cluster kernel below is the one used; the single-CTA
// kernel serves candidate sets too large to stage in the cluster's shared memory.
#include <cooperative_groups.h>

#include "spin_common.cuh"
#include "spin_internal.h"

namespace spin {

constexpr int kTopkThreads = 1024;
constexpr int kTopkBins = 2048;

struct TopkShared {
    int hist[kTopkBins];
    int scan[33];
    uint32_t prefix;
    int kk;
    int nvalid;
};

__global__ void __launch_bounds__(kTopkThreads, 1)
topk_kernel(spin_config cfg, const float* __restrict__ scores, const int32_t* __restrict__ list,
            const int32_t* __restrict__ n_list, const int32_t* __restrict__ n_slots, int rows,
            int32_t* __restrict__ topk_idx, uint32_t* status) {
    __shared__ TopkShared sh;
    const Dims dm = dims_of(cfg);
    const int rr = blockIdx.x, req = rr / rows;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int K = cfg.top_k;
    int32_t* out = topk_idx + (int64_t)rr * K;
    const int64_t n = n_slots[req];
    const int64_t cnt = n_list[req];
    if (n < 0 || n > dm.max_slots || cnt < 0 || cnt > dm.MB) {
        if (tid == 0) set_status(status, (n < 0 || n > dm.max_slots) ? SPIN_STATUS_BAD_N : SPIN_STATUS_BAD_LIST);
        for (int k = tid; k < K; k += kTopkThreads) out[k] = -1;
        return;
    }
    const int64_t nb = (n + kBlock - 1) / kBlock;
    const int32_t* lst = list + (int64_t)req * dm.MB;
    const float* sc = scores + (int64_t)rr * dm.MB * kBlock;
    const int64_t C = cnt * kBlock;

    // candidate c is live iff its block is a valid block of this context and i < N
    auto live_slot = [&](int64_t c, int64_t& slot) -> bool {
        const int64_t blk = lst[c >> 6];
        slot = blk * kBlock + (c & 63);
        return blk >= 0 && blk < nb && slot < n;
    };

    int v = 0;
    bool bad_list = false;
    for (int64_t k = tid; k < cnt; k += kTopkThreads) {
        const int64_t blk = lst[k];
        if (blk >= 0 && blk < nb) {
            const int64_t rem = n - blk * kBlock;
            v += (int)(rem < kBlock ? rem : kBlock);
        } else {
            bad_list = true;
        }
    }
    if (bad_list && rr % rows == 0) set_status(status, SPIN_STATUS_BAD_LIST);
    int nvalid;
    block_excl_scan(v, sh.scan, &nvalid);

    uint32_t T = 0;
    int kk = 0;
    const bool take_all = nvalid <= K;
    if (!take_all) {
        uint32_t prefix = 0, mask = 0;
        kk = K;
        const int shifts[3] = {21, 10, 0};
        const int widths[3] = {11, 11, 10};
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = shifts[pass];
            const uint32_t dmask = (1u << widths[pass]) - 1u;
            for (int b = tid; b < kTopkBins; b += kTopkThreads) sh.hist[b] = 0;
            __syncthreads();
            const int64_t C_pad = (C + 31) & ~(int64_t)31;
            for (int64_t c = tid; c < C_pad; c += kTopkThreads) {
                int bin = -1;
                int64_t slot;
                if (c < C && live_slot(c, slot)) {
                    const uint32_t key = order_key(sc[c]);
                    if ((key & mask) == prefix) bin = (int)((key >> shift) & dmask);
                }
                const unsigned same = __match_any_sync(0xffffffffu, bin);
                if (bin >= 0 && lane == __ffs(same) - 1) atomicAdd(&sh.hist[bin], __popc(same));
            }
            __syncthreads();
            if (wid == 0) {
                // lane l owns the 64 bins (dmask - 64 l) down to (dmask - 64 l - 63)
                const int nbins = (int)dmask + 1;
                const int per = nbins / 32;
                int s = 0;
                for (int b = 0; b < per; ++b) s += sh.hist[(int)dmask - per * lane - b];
                const int inc = warp_incl_scan(s);
                const unsigned ball = __ballot_sync(0xffffffffu, inc >= kk);
                const int src = __ffs(ball) - 1;
                if (lane == src) {
                    int above = inc - s, digit = 0;
                    for (int b = 0; b < per; ++b) {
                        const int d = (int)dmask - per * lane - b;
                        const int h = sh.hist[d];
                        if (above + h >= kk) { digit = d; break; }
                        above += h;
                    }
                    sh.prefix = prefix | ((uint32_t)digit << shift);
                    sh.kk = kk - above;
                }
            }
            __syncthreads();
            prefix = sh.prefix;
            kk = sh.kk;
            mask |= dmask << shift;
            __syncthreads();
        }
        T = prefix;
    }

    // ordered pass: keep key > T, and the first kk keys == T; write ascending slot ids
    constexpr int kItems = 4;
    int written = 0, eq_seen = 0;
    for (int64_t base = 0; base < C; base += (int64_t)kTopkThreads * kItems) {
        int32_t ids[kItems];
        uint8_t gt[kItems], eq[kItems];
        int n_eq = 0;
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int64_t c = base + (int64_t)tid * kItems + it;
            gt[it] = eq[it] = 0;
            ids[it] = -1;
            int64_t slot;
            if (c < C && live_slot(c, slot)) {
                ids[it] = (int32_t)slot;
                if (take_all) {
                    gt[it] = 1;
                } else {
                    const uint32_t key = order_key(sc[c]);
                    gt[it] = key > T;
                    eq[it] = key == T;
                }
            }
            n_eq += eq[it];
        }
        int eq_total;
        int eq_rank = eq_seen + block_excl_scan(n_eq, sh.scan, &eq_total);
        int n_keep = 0;
        uint8_t keep[kItems];
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            keep[it] = gt[it];
            if (eq[it]) {
                keep[it] = eq_rank < kk;
                ++eq_rank;
            }
            n_keep += keep[it];
        }
        int keep_total;
        int pos = written + block_excl_scan(n_keep, sh.scan, &keep_total);
#pragma unroll
        for (int it = 0; it < kItems; ++it)
            if (keep[it] && pos < K) out[pos++] = ids[it];
        written += keep_total;
        eq_seen += eq_total;
    }
    for (int k = written + tid; k < K; k += kTopkThreads) out[k] = -1;
}

// ---------------------------------------------------------------------------------------
// Cluster version: the candidates of one (request, row) are split over the 8 CTAs of a
// thread-block cluster in candidate order.  Each CTA keeps its slice's keys in shared
// memory (one global read), builds per-pass histograms with warp-aggregated shared
// atomics, and reads its peers' histograms over distributed shared memory, so all CTAs
// take the same digit decisions.  The ordered write uses the peers' kept counts as the
// output offset of each slice.
// ---------------------------------------------------------------------------------------
constexpr int kTkCluster = 8;

struct TkClusterShared {
    int hist[2][kTopkBins];   // double-buffered local histogram (peers read it)
    int merged[kTopkBins];
    int scan[33];
    int counts[4];            // valid, gt, eq (published to peers)
    uint32_t prefix;
    int kk;
};

__global__ void __cluster_dims__(kTkCluster, 1, 1) __launch_bounds__(kTopkThreads, 1)
topk_cluster_kernel(spin_config cfg, const float* __restrict__ scores, const int32_t* __restrict__ list,
                    const int32_t* __restrict__ n_list, const int32_t* __restrict__ n_slots, int rows,
                    int32_t* __restrict__ topk_idx, uint32_t* status) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ __align__(16) uint32_t keys[];
    __shared__ TkClusterShared sh;
    const Dims dm = dims_of(cfg);
    const int rank = (int)cluster.block_rank();
    const int rr = blockIdx.y, req = rr / rows;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int K = cfg.top_k;
    int32_t* out = topk_idx + (int64_t)rr * K;
    int64_t n = n_slots[req];
    int64_t cnt = n_list[req];
    const bool bad = n < 0 || n > dm.max_slots || cnt < 0 || cnt > dm.MB;
    if (bad) {
        if (rank == 0 && tid == 0) set_status(status, (n < 0 || n > dm.max_slots) ? SPIN_STATUS_BAD_N : SPIN_STATUS_BAD_LIST);
        n = 0;
        cnt = 0;
    }
    const int64_t nb = (n + kBlock - 1) / kBlock;
    const int32_t* lst = list + (int64_t)req * dm.MB;
    const float* sc = scores + (int64_t)rr * dm.MB * kBlock;
    const int64_t C = cnt * kBlock;
    const int64_t c0 = C * rank / kTkCluster, c1 = C * (rank + 1) / kTkCluster;
    const int nloc = (int)(c1 - c0);
    const int nloc_pad = (nloc + 31) & ~31;

    // 1. keys of this slice (0 = not a live candidate; live keys are never 0)
    int v = 0;
    bool bad_list = false;
    for (int i = tid; i < nloc; i += kTopkThreads) {
        const int64_t c = c0 + i;
        const int64_t blk = lst[c >> 6];
        const int64_t slot = blk * kBlock + (c & 63);
        uint32_t key = 0;
        if (blk >= 0 && blk < nb) {
            if (slot < n) key = order_key(sc[c]);
        } else {
            bad_list = true;
        }
        keys[i] = key;
        v += key != 0u;
    }
    if (bad_list && rr % rows == 0) set_status(status, SPIN_STATUS_BAD_LIST);
    int nvalid_loc;
    block_excl_scan(v, sh.scan, &nvalid_loc);
    if (tid == 0) sh.counts[0] = nvalid_loc;
    cluster.sync();
    int nvalid = 0;
    for (int p = 0; p < kTkCluster; ++p) nvalid += cluster.map_shared_rank(&sh.counts[0], p)[0];

    uint32_t T = 0;
    int kk = 0;
    if (nvalid > K) {
        uint32_t prefix = 0, mask = 0;
        kk = K;
        const int shifts[3] = {21, 10, 0};
        const int widths[3] = {11, 11, 10};
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = shifts[pass];
            const uint32_t dmask = (1u << widths[pass]) - 1u;
            int* hist = sh.hist[pass & 1];
            for (int b = tid; b < kTopkBins; b += kTopkThreads) hist[b] = 0;
            __syncthreads();
            for (int i = tid; i < nloc_pad; i += kTopkThreads) {
                int bin = -1;
                if (i < nloc) {
                    const uint32_t key = keys[i];
                    if (key != 0u && (key & mask) == prefix) bin = (int)((key >> shift) & dmask);
                }
                const unsigned same = __match_any_sync(0xffffffffu, bin);
                if (bin >= 0 && lane == __ffs(same) - 1) atomicAdd(&hist[bin], __popc(same));
            }
            cluster.sync();  // local histograms complete and visible to the peers
            const int nbins = (int)dmask + 1;
            for (int b = tid; b < nbins; b += kTopkThreads) {
                int s = 0;
                for (int p = 0; p < kTkCluster; ++p) s += cluster.map_shared_rank(hist, p)[b];
                sh.merged[b] = s;
            }
            __syncthreads();
            if (wid == 0) {
                const int per = nbins / 32;
                int s = 0;
                for (int b = 0; b < per; ++b) s += sh.merged[(int)dmask - per * lane - b];
                const int inc = warp_incl_scan(s);
                const unsigned ball = __ballot_sync(0xffffffffu, inc >= kk);
                const int src = __ffs(ball) - 1;
                if (lane == src) {
                    int above = inc - s, digit = 0;
                    for (int b = 0; b < per; ++b) {
                        const int d = (int)dmask - per * lane - b;
                        const int h = sh.merged[d];
                        if (above + h >= kk) { digit = d; break; }
                        above += h;
                    }
                    sh.prefix = prefix | ((uint32_t)digit << shift);
                    sh.kk = kk - above;
                }
            }
            __syncthreads();
            prefix = sh.prefix;
            kk = sh.kk;
            mask |= dmask << shift;
        }
        T = prefix;
    } else {
        T = 0;   // every live key (> 0) is kept
        kk = 0;
    }

    // 2. per-slice counts -> offsets
    int g = 0, e = 0;
    for (int i = tid; i < nloc; i += kTopkThreads) {
        const uint32_t key = keys[i];
        g += key > T;
        e += (key == T && key != 0u);
    }
    int gt_loc, eq_loc;
    block_excl_scan(g, sh.scan, &gt_loc);
    block_excl_scan(e, sh.scan, &eq_loc);
    if (tid == 0) { sh.counts[1] = gt_loc; sh.counts[2] = eq_loc; }
    cluster.sync();
    // slice p keeps its gt keys and, of its eq keys, those ranked below kk cluster-wide
    int eq_before = 0, out_base = 0, kept_total = 0, eb = 0;
    for (int p = 0; p < kTkCluster; ++p) {
        const int* pc = cluster.map_shared_rank(sh.counts, p);
        const int pk = pc[1] + max(0, min(pc[2], kk - eb));
        if (p < rank) { out_base += pk; eq_before += pc[2]; }
        kept_total += pk;
        eb += pc[2];
    }

    // 3. ordered write of the kept slot ids of this slice
    constexpr int kItems = 4;
    int written = out_base, eq_seen = eq_before;
    for (int base = 0; base < nloc; base += kTopkThreads * kItems) {
        uint8_t gt[kItems], eq[kItems];
        int n_eq = 0;
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int i = base + tid * kItems + it;
            gt[it] = eq[it] = 0;
            if (i < nloc) {
                const uint32_t key = keys[i];
                gt[it] = key > T;
                eq[it] = key == T && key != 0u;
            }
            n_eq += eq[it];
        }
        int eq_total;
        int eq_rank = eq_seen + block_excl_scan(n_eq, sh.scan, &eq_total);
        int n_keep = 0;
        uint8_t keep[kItems];
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            keep[it] = gt[it];
            if (eq[it]) { keep[it] = eq_rank < kk; ++eq_rank; }
            n_keep += keep[it];
        }
        int keep_total;
        int pos = written + block_excl_scan(n_keep, sh.scan, &keep_total);
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            if (keep[it] && pos < K) {
                const int64_t c = c0 + base + tid * kItems + it;
                out[pos++] = (int32_t)((int64_t)lst[c >> 6] * kBlock + (c & 63));
            }
        }
        written += keep_total;
        eq_seen += eq_total;
    }
    if (rank == kTkCluster - 1)
        for (int k = kept_total + tid; k < K; k += kTopkThreads) out[k] = -1;
    cluster.sync();  // no CTA leaves while a peer may still read its shared memory
}

static size_t topk_cluster_smem(const spin_config& cfg) {
    const Dims dm = dims_of(cfg);
    const int64_t per = ((int64_t)dm.MB * kBlock + kTkCluster - 1) / kTkCluster;
    return (size_t)per * 4;
}

cudaError_t launch_topk(const spin_config& cfg, const float* scores, const int32_t* list,
                        const int32_t* n_list, const int32_t* n_slots, int rows, int32_t* topk_idx,
                        uint32_t* status, cudaStream_t s) {
    const size_t smem = topk_cluster_smem(cfg);
    if (smem + sizeof(TkClusterShared) <= 200 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        topk_cluster_kernel<<<dim3(kTkCluster, cfg.n_req * rows), kTopkThreads, smem, s>>>(
            cfg, scores, list, n_list, n_slots, rows, topk_idx, status);
        return cudaGetLastError();
    }
    topk_kernel<<<cfg.n_req * rows, kTopkThreads, 0, s>>>(cfg, scores, list, n_list, n_slots, rows, topk_idx,
                                                          status);
    return cudaGetLastError();
}

}  // namespace spin

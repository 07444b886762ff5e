// spin_topk_rows.cuh -- exact top-K of one (request, row) by one 1024-thread CTA, reading
// the scores from global memory (included by the top-K translation units).
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention", Algorithm 1's top-K step over the
// scored slots; equal scores at the K-th value go to the lower slot id.  A three-pass radix
// select (11 + 11 + 10 bits of the order-preserving key) finds the K-th key T and how many
// keys equal to T to keep; one ordered pass writes the kept slot ids in ascending order and
// pads with -1.
#pragma once

#include "spin_common.cuh"

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

// Candidates are the list's slots i < N in list order (ascending slot order); `lst` holds the
// row's cnt list entries, `sc` its scores, `out` its K outputs.  blockDim.x == kTopkThreads.
__device__ __forceinline__ void topk_exact_row(const float* __restrict__ sc, const int32_t* __restrict__ lst,
                                               int64_t cnt, int64_t n, int K, bool report_list,
                                               int32_t* __restrict__ out, uint32_t* status, TopkShared& sh) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t nb = (n + kBlock - 1) / kBlock;
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
    if (bad_list && report_list) set_status(status, SPIN_STATUS_BAD_LIST);
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

}  // namespace spin

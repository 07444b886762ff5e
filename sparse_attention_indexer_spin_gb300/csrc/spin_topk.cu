// spin_topk.cu -- post-indexer top-K over the freshly scored slots.
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention", Algorithm 1's top-K step:
// T_t = TopK(z_t, K) over the slots the indexer scored (the selected blocks), which then
// feeds core attention.  Equal scores at the K-th value go to the lower slot id.
//
// The candidates are the listed blocks' slots i < N, visited in list order, which is
// ascending slot order because block lists are ascending.  A three-pass radix select
// (11 + 11 + 10 bits of the order-preserving 32-bit key) finds the K-th key T and how many
// keys equal to T to keep; one ordered pass then writes the kept slot ids in ascending
// order and pads with -1.  Launches with at least 32 request rows use the sampled-bracket
// kernel of spin_topk_sample.cu (one CTA per row) when its shared memory fits; fewer rows
// use the 8-CTA cluster kernel below, and the row and single-CTA kernels serve lists too
// long for either.
#include <cooperative_groups.h>

#include "spin_common.cuh"
#include "spin_internal.h"
#include "spin_topk_rows.cuh"

namespace spin {

__global__ void __launch_bounds__(kTopkThreads, 1)
topk_kernel(spin_config cfg, const float* __restrict__ scores, const int32_t* __restrict__ list,
            const int32_t* __restrict__ n_list, const int32_t* __restrict__ n_slots, int rows,
            int32_t* __restrict__ topk_idx, uint32_t* status) {
    pdl_begin();
    __shared__ TopkShared sh;
    const Dims dm = dims_of(cfg);
    const int rr = blockIdx.x, req = rr / rows;
    const int tid = threadIdx.x;
    const int K = cfg.top_k;
    int32_t* out = topk_idx + (int64_t)rr * K;
    const int64_t n = n_slots[req];
    const int64_t cnt = n_list[req];
    if (n < 0 || n > dm.max_slots || cnt < 0 || cnt > dm.MB) {
        if (tid == 0) set_status(status, (n < 0 || n > dm.max_slots) ? SPIN_STATUS_BAD_N : SPIN_STATUS_BAD_LIST);
        for (int k = tid; k < K; k += kTopkThreads) out[k] = -1;
        return;
    }
    topk_exact_row(scores + (int64_t)rr * dm.MB * kBlock, list + (int64_t)req * dm.MB, cnt, n, K, rr % rows == 0,
                   out, status, sh);
}

// ---------------------------------------------------------------------------------------
// Cluster version: the candidates of one (request, row) are split over the 8 CTAs of a
// thread-block cluster in candidate order.  Each CTA keeps its slice's keys in shared
// memory (one global read) and builds per-pass histograms with warp-aggregated shared
// atomics.  The cluster-wide histogram is reduced in distributed shared memory: CTA r
// sums bins [r S, (r+1) S) of every peer (S = bins / 8, 16-byte loads), and every CTA
// then gathers the eight shares, so all CTAs take the same digit decisions from one
// scan.  The live-candidate count is the first pass's histogram total.  The ordered
// write uses the peers' kept counts as the output offset of each slice.
// ---------------------------------------------------------------------------------------
constexpr int kTkCluster = 8;

// candidates of the largest slice, rounded up to whole 16-byte words
__host__ __device__ inline int64_t kTkSliceKeys(const spin_config& cfg) {
    const Dims dm = dims_of(cfg);
    const int64_t per = ((int64_t)dm.MB * kBlock + kTkCluster - 1) / kTkCluster;
    return (per + 3) & ~(int64_t)3;
}

// Adds the warp's bins (-1: none) to a shared histogram: the lanes that share the first
// active lane's bin with one atomic, the others one atomic each.
__device__ __forceinline__ void tk_hist_add(int* h, int bin) {
    const int lane = threadIdx.x & 31;
    const unsigned act = __ballot_sync(0xffffffffu, bin >= 0);
    if (act == 0u) return;
    const int lead = __ffs(act) - 1;
    const int b0 = __shfl_sync(0xffffffffu, bin, lead);
    const unsigned m0 = __ballot_sync(0xffffffffu, bin == b0);
    if (lane == lead) atomicAdd(&h[b0], __popc(m0));
    else if (bin >= 0 && bin != b0) atomicAdd(&h[bin], 1);
}

// Exclusive scan of unsigned words over the CTA (blockDim.x == kTopkThreads); `smem`
// holds 33 words.  Sums wrap modulo 2^32, which two packed 16-bit counts never reach.
__device__ __forceinline__ uint32_t tk_block_excl_scan_u(uint32_t v, uint32_t* smem, uint32_t* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) smem[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        const uint32_t s = smem[lane];
        uint32_t si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) si += t;
        }
        smem[lane] = si - s;
        if (lane == 31) smem[32] = si;
    }
    __syncthreads();
    const uint32_t res = smem[wid] + inc - v;
    *total = smem[32];
    __syncthreads();
    return res;
}

struct TkClusterShared {
    __align__(16) int hist[2][kTopkBins];             // double-buffered local histogram
    __align__(16) int share[kTopkBins / kTkCluster];  // this CTA's bins of the cluster sum
    uint32_t scan[33];
    int counts[4];                                    // gt, eq of the slice (peers read them)
    uint32_t prefix;
    int kk, nbin;
};

__global__ void __cluster_dims__(kTkCluster, 1, 1) __launch_bounds__(kTopkThreads, 1)
topk_cluster_kernel(spin_config cfg, const float* __restrict__ scores, const int32_t* __restrict__ list,
                    const int32_t* __restrict__ n_list, const int32_t* __restrict__ n_slots, int rows,
                    int32_t* __restrict__ topk_idx, uint32_t* status) {
    pdl_begin();
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

    // 1. keys of this slice (0 = not a live candidate; live keys are never 0).  The slice
    // [c0, c1) is a multiple of 8 candidates long and starts 32-byte aligned; the list
    // entry of each group of 4 candidates is read with its scores (16 consecutive groups
    // share one entry) and kept in shared memory for the write.
    int* slist = reinterpret_cast<int*>(keys + kTkSliceKeys(cfg));
    const int64_t e0 = c0 >> 6;
    {
        bool bad_list = false;
        const float4* sc4 = reinterpret_cast<const float4*>(sc + c0);
        uint4* keys4 = reinterpret_cast<uint4*>(keys);
#pragma unroll 4
        for (int i4 = tid; i4 < nloc / 4; i4 += kTopkThreads) {
            const int64_t c = c0 + 4 * (int64_t)i4;
            const int blk = __ldg(lst + (c >> 6));
            const float4 z = __ldg(sc4 + i4);
            if (i4 == 0 || (c & 63) == 0) slist[(c >> 6) - e0] = blk;
            const int64_t slot = (int64_t)blk * kBlock + (c & 63);
            uint4 kv = make_uint4(0u, 0u, 0u, 0u);
            if (blk >= 0 && blk < nb) {
                kv.x = slot + 0 < n ? order_key(z.x) : 0u;
                kv.y = slot + 1 < n ? order_key(z.y) : 0u;
                kv.z = slot + 2 < n ? order_key(z.z) : 0u;
                kv.w = slot + 3 < n ? order_key(z.w) : 0u;
            } else {
                bad_list = true;
            }
            keys4[i4] = kv;
        }
        if (bad_list && rr % rows == 0) set_status(status, SPIN_STATUS_BAD_LIST);
    }

    // 2. radix select of the K-th largest key over 11 + 11 + 10 bits
    uint32_t prefix = 0, mask = 0;
    int kk = K;
    bool keep_all = false, exact_bin = false;
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const uint32_t dmask = pass == 2 ? 1023u : 2047u;
        const int nbins = (int)dmask + 1;
        const int S = nbins / kTkCluster;  // bins of one share: 256 or 128
        int* hist = sh.hist[pass & 1];
        for (int b = tid; b < nbins; b += kTopkThreads) hist[b] = 0;
        __syncthreads();
        for (int i = tid; i < nloc_pad; i += kTopkThreads) {
            int bin = -1;
            if (i < nloc) {
                const uint32_t key = keys[i];
                if (key != 0u && (key & mask) == prefix) bin = (int)((key >> shift) & dmask);
            }
            tk_hist_add(hist, bin);
        }
        cluster.sync();  // local histograms complete and visible to the peers
        if (tid < S / 4) {
            int4 a = make_int4(0, 0, 0, 0);
#pragma unroll
            for (int p = 0; p < kTkCluster; ++p) {
                const int4 h = reinterpret_cast<const int4*>(cluster.map_shared_rank(hist, p) + rank * S)[tid];
                a.x += h.x; a.y += h.y; a.z += h.z; a.w += h.w;
            }
            reinterpret_cast<int4*>(sh.share)[tid] = a;
        }
        cluster.sync();  // shares complete
        // thread t holds bins 4u .. 4u + 3 with u = nbins / 4 - 1 - t: bins in descending order
        const int u = nbins / 4 - 1 - tid;
        int4 h = make_int4(0, 0, 0, 0);
        if (u >= 0) {
            const int owner = (4 * u) / S;
            h = reinterpret_cast<const int4*>(cluster.map_shared_rank(sh.share, owner) + (4 * u - owner * S))[0];
        }
        const int c4 = h.x + h.y + h.z + h.w;
        const int inc = warp_incl_scan(c4);
        if (lane == 31) sh.scan[wid] = (uint32_t)inc;
        __syncthreads();
        const int wtot = (int)sh.scan[lane];
        const int winc = warp_incl_scan(wtot);
        const int total = __shfl_sync(0xffffffffu, winc, 31);
        if (pass == 0 && total <= K) {  // every live candidate is kept (same decision cluster-wide)
            keep_all = true;
            __syncthreads();
            break;
        }
        const int excl = __shfl_sync(0xffffffffu, winc - wtot, wid) + inc - c4;
        if (excl < kk && excl + c4 >= kk) {
            int above = excl, d = 4 * u + 3, nbin = h.w;
            if (above + h.w < kk) { above += h.w; d -= 1; nbin = h.z;
                if (above + h.z < kk) { above += h.z; d -= 1; nbin = h.y;
                    if (above + h.y < kk) { above += h.y; d -= 1; nbin = h.x; } } }
            sh.prefix = prefix | ((uint32_t)d << shift);
            sh.kk = kk - above;
            sh.nbin = nbin;
        }
        __syncthreads();
        prefix = sh.prefix;
        kk = sh.kk;
        mask |= dmask << shift;
        if (kk == sh.nbin && pass < 2) {  // the whole threshold bin is kept: keys >= prefix
            exact_bin = true;
            break;
        }
    }
    // keep_all: every live key (> 0); exact_bin: every key >= prefix (> 0 then), that is
    // > prefix - 1 with no tie kept; otherwise keys > prefix and the first kk equal to it
    const uint32_t T = keep_all ? 0u : exact_bin ? prefix - 1u : prefix;
    if (keep_all || exact_bin) kk = 0;

    // 3. each thread owns a contiguous run of the slice: one packed scan of its gt and eq
    // counts gives the slice totals (published to the peers) and the in-slice offsets
    const int ipt = (nloc + kTopkThreads - 1) / kTopkThreads;
    const int i0 = min(nloc, tid * ipt), i1 = min(nloc, i0 + ipt);
    uint32_t g = 0, e = 0;
    for (int i = i0; i < i1; ++i) {
        const uint32_t key = keys[i];
        g += key > T;
        e += key == T && key != 0u;
    }
    uint32_t tot;
    const uint32_t ex = tk_block_excl_scan_u((g << 16) | e, sh.scan, &tot);
    if (tid == 0) { sh.counts[0] = (int)(tot >> 16); sh.counts[1] = (int)(tot & 0xFFFFu); }
    cluster.sync();
    // slice p keeps its gt keys and, of its eq keys, those ranked below kk cluster-wide
    int eq_before = 0, out_base = 0, kept_total = 0, eb = 0;
    for (int p = 0; p < kTkCluster; ++p) {
        const int* pc = cluster.map_shared_rank(sh.counts, p);
        const int pk = pc[0] + max(0, min(pc[1], kk - eb));
        if (p < rank) { out_base += pk; eq_before += pc[1]; }
        kept_total += pk;
        eb += pc[1];
    }
    const int eq_keep = max(0, kk - eq_before);  // eq keys this slice keeps (its first ones)
    int gb = (int)(ex >> 16), ebf = (int)(ex & 0xFFFFu);
    for (int i = i0; i < i1; ++i) {
        const uint32_t key = keys[i];
        const bool gt = key > T, eq = key == T && key != 0u;
        if (gt || (eq && ebf < eq_keep)) {
            const int pos = out_base + gb + min(ebf, eq_keep);
            if (pos < K) {
                const int64_t c = c0 + i;
                out[pos] = (int32_t)((int64_t)slist[(c >> 6) - e0] * kBlock + (c & 63));
            }
        }
        gb += gt;
        ebf += eq;
    }
    if (rank == kTkCluster - 1)
        for (int k = kept_total + tid; k < K; k += kTopkThreads) out[k] = -1;
    cluster.sync();  // no CTA leaves while a peer may still read its shared memory
}

// ---------------------------------------------------------------------------------------
// Row kernel: one 1024-thread CTA per (request, row), for launches with enough rows to fill
// the GPU.  Pass A reads every candidate once (float4) and builds a 4096-bin histogram of
// the top 12 bits of its key; the bin holding the K-th key is found.  Pass B collects the
// low 20 bits and the candidate index of the keys in that bin (usually a few thousand)
// into shared memory, where two 10-bit radix passes finish the exact threshold.  Pass C
// writes the kept slot ids in candidate (= ascending slot) order.  If the boundary bin
// overflows the collection buffer, the threshold is refined over global memory instead.
// ---------------------------------------------------------------------------------------
constexpr int kTrThreads = 1024;
constexpr int kTrBins = 4096;
constexpr int kTrCollect = 8192;

struct TrShared {
    int hist[kTrBins];
    uint32_t ckey[kTrCollect];  // low 20 bits of the boundary-bin keys
    int ncol;
    int scan[33];
    uint32_t prefix;
    int kk;
};

// block-wide digit search: the digit d with (#keys with digit > d) < kk <= (#keys >= d);
// returns d and the count above it.  nb bins, each warp owning a contiguous descending range.
__device__ __forceinline__ void tr_find_digit(const int* hist, int nbins, int kk, TrShared& sh, int& digit_out,
                                              int& above_out) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = kTrThreads / 32;
    const int per_warp = nbins / nw, per_lane = per_warp / 32;
    // bins of warp w: top = nbins-1 - w*per_warp, descending; lane l owns per_lane of them
    const int top = nbins - 1 - wid * per_warp - lane * per_lane;
    int cnt = 0;
    for (int b = 0; b < per_lane; ++b) cnt += hist[top - b];
    const int inc = warp_incl_scan(cnt);
    __shared__ int wsum[32];
    if (lane == 31) wsum[wid] = inc;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < wid; ++w) before += wsum[w];
    const int excl = before + inc - cnt;
    if (excl < kk && excl + cnt >= kk) {
        int above = excl, digit = top;
        for (int b = 0; b < per_lane; ++b) {
            const int h = hist[top - b];
            if (above + h >= kk) { digit = top - b; break; }
            above += h;
        }
        sh.prefix = (uint32_t)digit;
        sh.kk = above;
    }
    __syncthreads();
    digit_out = (int)sh.prefix;
    above_out = sh.kk;
    __syncthreads();
}

__global__ void __launch_bounds__(kTrThreads, 1)
topk_row_kernel(spin_config cfg, const float* __restrict__ scores, const int32_t* __restrict__ list,
                const int32_t* __restrict__ n_list, const int32_t* __restrict__ n_slots, int rows,
                int32_t* __restrict__ topk_idx, uint32_t* status) {
    pdl_begin();
    extern __shared__ __align__(16) unsigned char tr_smem[];
    TrShared& sh = *reinterpret_cast<TrShared*>(tr_smem);
    int* slist = reinterpret_cast<int*>(tr_smem + sizeof(TrShared));  // the row's list entries
    const Dims dm = dims_of(cfg);
    const int rr = blockIdx.x, req = rr / rows;
    const int tid = threadIdx.x, lane = tid & 31;
    const int K = cfg.top_k;
    int32_t* out = topk_idx + (int64_t)rr * K;
    const int64_t n = n_slots[req];
    const int64_t cnt = n_list[req];
    if (n < 0 || n > dm.max_slots || cnt < 0 || cnt > dm.MB) {
        if (tid == 0) set_status(status, (n < 0 || n > dm.max_slots) ? SPIN_STATUS_BAD_N : SPIN_STATUS_BAD_LIST);
        for (int k = tid; k < K; k += kTrThreads) out[k] = -1;
        return;
    }
    const int64_t nb = (n + kBlock - 1) / kBlock;
    const int32_t* lst = list + (int64_t)req * dm.MB;
    const float4* sc4 = reinterpret_cast<const float4*>(scores + (int64_t)rr * dm.MB * kBlock);
    const int C4 = (int)cnt * (kBlock / 4);
    bool bad_list = false;
    for (int i = tid; i < cnt; i += kTrThreads) {
        const int b = lst[i];
        if (b < 0 || b >= nb) bad_list = true;
        slist[i] = b;
    }
    for (int b = tid; b < kTrBins; b += kTrThreads) sh.hist[b] = 0;
    if (tid == 0) sh.ncol = 0;
    if (bad_list && rr % rows == 0) set_status(status, SPIN_STATUS_BAD_LIST);
    __syncthreads();
    // 4 keys of float4 i4 (0 = not a live candidate)
    auto keys4 = [&](int i4, const float4& z, uint32_t* k4) {
        const int c = 4 * i4;
        const int blk = slist[c >> 6];
        const int64_t slot = (int64_t)blk * kBlock + (c & 63);
        const bool okb = blk >= 0 && blk < nb;
        k4[0] = okb && slot + 0 < n ? order_key(z.x) : 0u;
        k4[1] = okb && slot + 1 < n ? order_key(z.y) : 0u;
        k4[2] = okb && slot + 2 < n ? order_key(z.z) : 0u;
        k4[3] = okb && slot + 3 < n ? order_key(z.w) : 0u;
    };

    // pass A: histogram of the top 12 bits
    int v = 0;
    const int C4pad = (C4 + 31) & ~31;
#pragma unroll 8
    for (int i4 = tid; i4 < C4pad; i4 += kTrThreads) {
        uint32_t k4[4] = {0u, 0u, 0u, 0u};
        if (i4 < C4) keys4(i4, sc4[i4], k4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int bin = k4[e] ? (int)(k4[e] >> 20) : -1;
            const unsigned same = __match_any_sync(0xffffffffu, bin);
            if (bin >= 0 && lane == __ffs(same) - 1) atomicAdd(&sh.hist[bin], __popc(same));
            v += k4[e] != 0u;
        }
    }
    int nvalid;
    block_excl_scan(v, sh.scan, &nvalid);

    uint32_t T = 0;   // full threshold key
    int kk = 0;       // keys == T to keep (lowest candidate index first)
    if (nvalid > K) {
        int d1, above1;
        tr_find_digit(sh.hist, kTrBins, K, sh, d1, above1);
        const int need = K - above1;  // still needed from bin d1
        // pass B: collect the low 20 bits of bin d1's keys
#pragma unroll 8
        for (int i4 = tid; i4 < C4; i4 += kTrThreads) {
            uint32_t k4[4];
            keys4(i4, sc4[i4], k4);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (k4[e] && (int)(k4[e] >> 20) == d1) {
                    const int slot = atomicAdd(&sh.ncol, 1);
                    if (slot < kTrCollect) sh.ckey[slot] = k4[e] & 0xFFFFFu;
                }
        }
        __syncthreads();
        const int ncol = sh.ncol;
        uint32_t prefix = (uint32_t)d1 << 20, mask = 0xFFF00000u;
        int kk2 = need;
        const int shifts[2] = {10, 0};
        for (int pass = 0; pass < 2; ++pass) {
            const int shift = shifts[pass];
            for (int b = tid; b < 1024; b += kTrThreads) sh.hist[b] = 0;
            __syncthreads();
            if (ncol <= kTrCollect) {
                const uint32_t high = (uint32_t)d1 << 20;  // the bin's common top 12 bits
                for (int i = tid; i < ncol; i += kTrThreads) {
                    const uint32_t key = high | sh.ckey[i];
                    if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 1023u], 1);
                }
            } else {  // the boundary bin overflowed the buffer: refine over global memory
#pragma unroll 4
                for (int i4 = tid; i4 < C4; i4 += kTrThreads) {
                    uint32_t k4[4];
                    keys4(i4, sc4[i4], k4);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (k4[e] && (k4[e] & mask) == prefix) atomicAdd(&sh.hist[(k4[e] >> shift) & 1023u], 1);
                }
            }
            __syncthreads();
            int d, above;
            tr_find_digit(sh.hist, 1024, kk2, sh, d, above);
            prefix |= (uint32_t)d << shift;
            mask |= 1023u << shift;
            kk2 -= above;
        }
        T = prefix;
        kk = kk2;
    }

    // pass C: ordered write (keys > T, then the first kk keys == T in candidate order).
    // A thread takes kV consecutive float4 (16 candidates) per round; the next round's
    // loads are issued before this round's scans.
    constexpr int kV = 4, kItems = 4 * kV;
    int written = 0, eq_seen = 0;
    const bool take_all = nvalid <= K;
    float4 zn[kV];
#pragma unroll
    for (int j = 0; j < kV; ++j) {
        const int i4 = tid * kV + j;
        zn[j] = i4 < C4 ? sc4[i4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int base4 = 0; base4 < C4; base4 += kTrThreads * kV) {
        float4 zc[kV];
#pragma unroll
        for (int j = 0; j < kV; ++j) zc[j] = zn[j];
        const int nbase = base4 + kTrThreads * kV;
#pragma unroll
        for (int j = 0; j < kV; ++j) {
            const int i4 = nbase + tid * kV + j;
            if (i4 < C4) zn[j] = sc4[i4];
        }
        uint32_t kx[kItems];
#pragma unroll
        for (int j = 0; j < kV; ++j) {
            const int i4 = base4 + tid * kV + j;
            uint32_t k4[4] = {0u, 0u, 0u, 0u};
            if (i4 < C4) keys4(i4, zc[j], k4);
#pragma unroll
            for (int e = 0; e < 4; ++e) kx[4 * j + e] = k4[e];
        }
        int n_eq = 0;
#pragma unroll
        for (int e = 0; e < kItems; ++e) n_eq += !take_all && kx[e] != 0u && kx[e] == T;
        int eq_total;
        int eq_rank = eq_seen + block_excl_scan(n_eq, sh.scan, &eq_total);
        uint32_t keep = 0;  // bit e: candidate e of this thread is kept
#pragma unroll
        for (int e = 0; e < kItems; ++e) {
            bool kp = take_all ? (kx[e] != 0u) : (kx[e] > T);
            if (!take_all && kx[e] != 0u && kx[e] == T) { kp = eq_rank < kk; ++eq_rank; }
            keep |= (uint32_t)kp << e;
        }
        int keep_total;
        int pos = written + block_excl_scan(__popc(keep), sh.scan, &keep_total);
#pragma unroll
        for (int e = 0; e < kItems; ++e)
            if (((keep >> e) & 1u) && pos < K) {
                const int c = 4 * (base4 + tid * kV) + e;
                out[pos++] = (int32_t)((int64_t)slist[c >> 6] * kBlock + (c & 63));
            }
        written += keep_total;
        eq_seen += eq_total;
    }
    for (int k = written + tid; k < K; k += kTrThreads) out[k] = -1;
}

// keys of the largest slice, then its list entries (a slice spans at most MB / 8 + 2)
static size_t topk_cluster_smem(const spin_config& cfg) {
    return (size_t)kTkSliceKeys(cfg) * 4 + (size_t)(dims_of(cfg).MB / kTkCluster + 2) * 4;
}

cudaError_t launch_topk(const spin_config& cfg, const float* scores, const int32_t* list,
                        const int32_t* n_list, const int32_t* n_slots, int rows, int32_t* topk_idx,
                        uint32_t* status, cudaStream_t s) {
    // enough rows to fill the GPU with one CTA each: the sampled-bracket kernel
    if ((int64_t)cfg.n_req * rows >= 32 && topk_sample_fits(cfg))
        return launch_topk_sample(cfg, scores, list, n_list, n_slots, rows, topk_idx, status, s);
    const Dims dm = dims_of(cfg);
    const size_t row_smem = sizeof(TrShared) + (size_t)dm.MB * 4;
    if ((int64_t)cfg.n_req * rows >= 32 && row_smem <= 200 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)row_smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(topk_row_kernel, dim3(cfg.n_req * rows), dim3(kTrThreads), row_smem, s, nullptr, 0, cfg,
                          scores, list, n_list, n_slots, rows, topk_idx, status);
    }
    const size_t smem = topk_cluster_smem(cfg);
    // (a slice's gt and eq counts share one 32-bit scan word: fewer than 2^16 keys each)
    if (smem + sizeof(TkClusterShared) <= 200 * 1024 && kTkSliceKeys(cfg) < 65536) {
        cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(topk_cluster_kernel, dim3(kTkCluster, cfg.n_req * rows), dim3(kTopkThreads), smem, s,
                          nullptr, 0, cfg, scores, list, n_list, n_slots, rows, topk_idx, status);
    }
    return launch_pdl(topk_kernel, dim3(cfg.n_req * rows), dim3(kTopkThreads), 0, s, nullptr, 0, cfg, scores, list,
                      n_list, n_slots, rows, topk_idx, status);
}

}  // namespace spin

// spin_topk_hint.cu -- temporal top-K: last step's threshold as the guess of this step's.
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention", Algorithm 1's top-K step (the K
// largest fresh scores, equal scores to the lower slot id), computed the way the paper's
// related work ("Guess-Verify-Refine", §5) accelerates the post-indexer top-K: consecutive
// decode steps of one request score the same context with a slowly drifting query, so the
// K-th score moves little from one step to the next.
//
//   guess   the score kernel of this step (spin_indexer_score_ex with the hint) already
//           compared every fresh score with the row's threshold -- the previous step's score
//           at rank K + extra, divided by that step's sum_h |w_h| and multiplied by this
//           step's (the head weights of a step scale all its scores together) -- and appended
//           those at or above it to the row's candidate array (a few per cent of the slots);
//   verify  if at least K and at most cap candidates were found, the top-K lies among them:
//           the K-th key T is >= the guess because K keys are, so every key > T and every
//           key == T was collected;
//   refine  an exact radix select over the candidates (64-bit entries: key, then the
//           complement of the list position, all distinct) gives the K largest entries;
//           they are marked in a bitmap of list positions and written in ascending slot
//           order.  The score at rank K + extra, normalised, becomes the next step's guess.
// A row without a guess, or whose guess found too few or too many candidates, takes the
// cold path: one pass over its scores builds a histogram of the top 12 key bits, the bin
// holding rank K + extra bounds the candidates (refined by the next 12, then the last 8
// bits while that bin alone overflows the candidate array), a last pass collects them, and
// the same refine step follows.  The margin `extra` starts at the geometric middle of [K, cap] minus K,
// doubles after a miss and halves after an overflow.  Only a boundary bin too large for the candidate array (massive ties) falls
// back to exact radix passes over the scores.  Every path returns exactly the top-K of
// spin_topk; the hint only decides how fast.
//
// One 1024-thread CTA per (request, row).  Shared memory: the candidates (cap 8-byte
// entries), the position bitmap (2 words per list entry) and the row's list.
#include "spin_common.cuh"
#include "spin_internal.h"
#include "spin_topk_rows.cuh"

namespace spin {

constexpr int kThThreads = 1024;
constexpr int kThMaxK = 2048;        // cap = 4K rounded up to a power of two, <= 8192
constexpr int kThMaxBlocks = 8192;   // bitmap of the list positions: <= 64 KB
constexpr int kThBinsA = 4096;       // cold pass: top 12 bits of the key
constexpr int kThBins = 2048;        // candidate radix: 11-bit digits of the 64-bit entry

struct ThShared {
    int hist[kThBinsA];
    int scan[33];
    int ncand;
    int digit, above, nbin;
    TopkShared exact;  // the exact fallback's own scratch
};

static_assert(kThThreads == kTopkThreads, "the exact fallback runs with the same CTA");

int topk_hint_cap(const spin_config& cfg) {
    int c = 4096;
    while (c < 4 * cfg.top_k) c <<= 1;
    return c;
}

// Initial rank margin: the guess aims at the geometric middle of [K, cap], where the
// candidate count has as much room to shrink as to grow.
__device__ __forceinline__ uint32_t th_default_extra(int K, int cap) {
    const int mid = (int)sqrtf((float)K * (float)cap);
    return mid > K ? (uint32_t)(mid - K) : 1u;
}

bool topk_hint_supported(const spin_config& cfg) {
    return cfg.top_k <= kThMaxK && dims_of(cfg).MB <= kThMaxBlocks;
}

static size_t hint_rec_bytes(const spin_config& cfg, int rows) {
    return ((size_t)cfg.n_req * rows * kHintWords * 4 + 255) & ~(size_t)255;
}

size_t topk_hint_bytes(const spin_config& cfg, int rows) {
    return hint_rec_bytes(cfg, rows) + (size_t)cfg.n_req * rows * topk_hint_cap(cfg) * 8;
}

HintArgs topk_hint_args(const spin_config& cfg, int rows, void* hint) {
    HintArgs h;
    h.rec = reinterpret_cast<uint32_t*>(hint);
    h.cand = reinterpret_cast<unsigned long long*>(reinterpret_cast<unsigned char*>(hint) +
                                                   hint_rec_bytes(cfg, rows));
    h.cap = topk_hint_cap(cfg);
    return h;
}

// Sum of one value over the CTA (all threads get it).
__device__ __forceinline__ int th_block_sum(int v, ThShared& sh) {
    int tot;
    block_excl_scan(v, sh.scan, &tot);
    return tot;
}

// Digit search over `nbins` bins, scanned from the top: the bin d with
// (# in bins > d) < kk <= (# in bins >= d).  Thread t owns nbins / 1024 consecutive bins in
// descending order.  Leaves d, the count above it and the bin's own count in sh.
__device__ __forceinline__ void th_find_digit(const int* hist, int nbins, int kk, ThShared& sh) {
    const int per = nbins / kThThreads;
    const int top = nbins - 1 - (int)threadIdx.x * per;
    int c = 0;
    for (int b = 0; b < per; ++b) c += hist[top - b];
    int tot;
    const int excl = block_excl_scan(c, sh.scan, &tot);
    if (excl < kk && excl + c >= kk) {
        int above = excl;
        for (int b = 0; b < per; ++b) {
            const int h = hist[top - b];
            if (above + h >= kk) {
                sh.digit = top - b;
                sh.above = above;
                sh.nbin = h;
                break;
            }
            above += h;
        }
    }
    __syncthreads();
}

// Adds this thread's bin (-1: none) to a shared histogram, one atomic per distinct bin of the warp.
__device__ __forceinline__ void th_hist_add(int* hist, int bin) {
    const unsigned same = __match_any_sync(0xffffffffu, bin);
    if (bin >= 0 && (int)(threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&hist[bin], __popc(same));
}

// Threshold U with exactly k of the n (distinct) entries >= U, 1 <= k <= n: radix select over
// 11-bit digits from the top, stopping as soon as the bin holding rank k is needed whole.
__device__ unsigned long long th_kth_entry(const unsigned long long* v, int n, int k, ThShared& sh) {
    unsigned long long prefix = 0ull, mask = 0ull;
    int kk = k;
    for (int pass = 0; pass < 6; ++pass) {
        const int shift = pass < 5 ? 53 - 11 * pass : 0;
        const unsigned long long dmask = pass < 5 ? 2047ull : 511ull;
        for (int b = threadIdx.x; b < kThBins; b += kThThreads) sh.hist[b] = 0;
        __syncthreads();
        for (int i0 = 0; i0 < n; i0 += kThThreads) {
            const int i = i0 + (int)threadIdx.x;
            int bin = -1;
            if (i < n) {
                const unsigned long long x = v[i];
                if ((x & mask) == prefix) bin = (int)((x >> shift) & dmask);
            }
            th_hist_add(sh.hist, bin);
        }
        __syncthreads();
        th_find_digit(sh.hist, kThBins, kk, sh);
        prefix |= (unsigned long long)sh.digit << shift;
        mask |= dmask << shift;
        kk -= sh.above;
        const bool whole = sh.nbin == kk;
        __syncthreads();
        if (whole) break;  // every entry with this prefix is kept: U = the prefix, low bits 0
    }
    return prefix;
}

__global__ void __launch_bounds__(kThThreads, 1)
topk_hint_kernel(spin_config cfg, const float* __restrict__ scores, const float* __restrict__ w,
                 const int32_t* __restrict__ list, const int32_t* __restrict__ n_list,
                 const int32_t* __restrict__ n_slots, int rows, int32_t* __restrict__ topk_idx, HintArgs h,
                 uint32_t* status) {
    pdl_begin();
    extern __shared__ __align__(16) unsigned char th_smem[];
    ThShared& sh = *reinterpret_cast<ThShared*>(th_smem);
    const Dims dm = dims_of(cfg);
    unsigned long long* cand =
        reinterpret_cast<unsigned long long*>(th_smem + ((sizeof(ThShared) + 15) & ~(size_t)15));
    uint32_t* bits = reinterpret_cast<uint32_t*>(cand + h.cap);  // [2 MB]
    int* slist = reinterpret_cast<int*>(bits + 2 * dm.MB);        // [MB]
    const int rr = blockIdx.x, req = rr / rows;
    const int tid = threadIdx.x;
    const int K = cfg.top_k;
    int32_t* out = topk_idx + (int64_t)rr * K;
    uint32_t* rec = h.rec + (int64_t)rr * kHintWords;
    const int64_t n = n_slots[req], cnt = n_list[req];
    const uint32_t guess = rec[kHwGuess], count = rec[kHwCount];
    const uint32_t kmin = K / 8 > 0 ? (uint32_t)(K / 8) : 1u;
    const uint32_t kmax = (uint32_t)(h.cap / 2 - K);
    uint32_t extra = rec[kHwExtra];
    if (extra == 0u) extra = th_default_extra(K, h.cap);
    extra = extra < kmin ? kmin : extra > kmax ? kmax : extra;
    __syncthreads();  // every thread has read the record before thread 0 rewrites it
    if (n < 0 || n > dm.max_slots || cnt < 0 || cnt > dm.MB) {
        if (tid == 0) {
            set_status(status, (n < 0 || n > dm.max_slots) ? SPIN_STATUS_BAD_N : SPIN_STATUS_BAD_LIST);
            rec[kHwGuess] = 0u;
            rec[kHwCount] = 0u;
        }
        for (int k = tid; k < K; k += kThThreads) out[k] = -1;
        return;
    }
    const int64_t nb = (n + kBlock - 1) / kBlock;
    const int64_t C = cnt * kBlock;
    const int W = (int)((C + 31) / 32);  // bitmap words

    bool bad_list = false;
    for (int64_t k = tid; k < cnt; k += kThThreads) {
        const int b = list[(int64_t)req * dm.MB + k];
        if (b < 0 || b >= nb) bad_list = true;
        slist[k] = b;
    }
    if (bad_list && rr % rows == 0) set_status(status, SPIN_STATUS_BAD_LIST);
    for (int wd = tid; wd < W; wd += kThThreads) bits[wd] = 0u;
    if (tid == 0) sh.ncand = 0;
    __syncthreads();

    const bool hit = guess != 0u && count >= (uint32_t)K && count <= (uint32_t)h.cap;
    bool take_all = false, exact = false;
    int nc = 0;
    if (hit) {
        nc = (int)count;
        const unsigned long long* src = h.cand + (int64_t)rr * h.cap;
        for (int i = tid; i < nc; i += kThThreads) cand[i] = src[i];
        __syncthreads();
    } else {
        // cold path.  Keys of four candidates (0: not a live candidate).
        const float4* sc4 = reinterpret_cast<const float4*>(scores + (int64_t)rr * dm.MB * kBlock);
        const int C4 = (int)(C / 4);
        auto keys4 = [&](int i4, uint32_t* k4) {
            const int c = 4 * i4;
            const int blk = slist[c >> 6];
            const int64_t slot = (int64_t)blk * kBlock + (c & 63);
            const bool okb = blk >= 0 && blk < nb;
            const float4 z = sc4[i4];
            k4[0] = okb && slot + 0 < n ? order_key(z.x) : 0u;
            k4[1] = okb && slot + 1 < n ? order_key(z.y) : 0u;
            k4[2] = okb && slot + 2 < n ? order_key(z.z) : 0u;
            k4[3] = okb && slot + 3 < n ? order_key(z.w) : 0u;
        };
        for (int b = tid; b < kThBinsA; b += kThThreads) sh.hist[b] = 0;
        __syncthreads();
        int v = 0;
        const int C4pad = (C4 + 31) & ~31;
        for (int i4 = tid; i4 < C4pad; i4 += kThThreads) {
            uint32_t k4[4] = {0u, 0u, 0u, 0u};
            if (i4 < C4) keys4(i4, k4);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                th_hist_add(sh.hist, k4[e] ? (int)(k4[e] >> 20) : -1);
                v += k4[e] != 0u;
            }
        }
        const int nvalid = th_block_sum(v, sh);  // (its barriers also complete the histogram)
        if (nvalid <= K) {
            take_all = true;
        } else {
            const int kp = (int)min((int64_t)nvalid, (int64_t)K + extra);
            // the bin holding rank kp, by the top 12 bits of the key; while it holds more
            // candidates than fit, refine it by the next 12, then the last 8 bits
            uint32_t tkey = 0u, tmask = 0u;  // collect the live keys >= tkey
            int above = 0, total = 0;
            for (int lvl = 0; lvl < 3; ++lvl) {
                const int shift = lvl == 0 ? 20 : lvl == 1 ? 8 : 0;
                const uint32_t dmask = lvl < 2 ? 4095u : 255u;
                if (lvl > 0) {
                    for (int b = tid; b < kThBinsA; b += kThThreads) sh.hist[b] = 0;
                    __syncthreads();
                    for (int i4 = tid; i4 < C4pad; i4 += kThThreads) {
                        uint32_t k4[4] = {0u, 0u, 0u, 0u};
                        if (i4 < C4) keys4(i4, k4);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            th_hist_add(sh.hist, k4[e] != 0u && (k4[e] & tmask) == tkey
                                                     ? (int)((k4[e] >> shift) & dmask) : -1);
                    }
                    __syncthreads();
                }
                th_find_digit(sh.hist, kThBinsA, kp - above, sh);
                total = above + sh.above + sh.nbin;
                above += sh.above;
                tkey |= (uint32_t)sh.digit << shift;
                tmask |= dmask << shift;
                __syncthreads();
                if (total <= h.cap) break;
            }
            if (total <= h.cap) {
                // collect every live candidate with key >= tkey (all of rank <= kp)
                for (int i4 = tid; i4 < C4pad; i4 += kThThreads) {
                    uint32_t k4[4] = {0u, 0u, 0u, 0u};
                    if (i4 < C4) keys4(i4, k4);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const bool take = k4[e] != 0u && k4[e] >= tkey;
                        const unsigned m = __ballot_sync(0xffffffffu, take);
                        if (m) {
                            const int lane = tid & 31, lead = __ffs(m) - 1;
                            int base = 0;
                            if (lane == lead) base = atomicAdd(&sh.ncand, __popc(m));
                            base = __shfl_sync(0xffffffffu, base, lead);
                            if (take) cand[base + __popc(m & ((1u << lane) - 1u))] =
                                hint_entry(k4[e], (uint32_t)(4 * i4 + e));
                        }
                    }
                }
                __syncthreads();
                nc = sh.ncand;
            } else {
                exact = true;  // a huge boundary bin (massive ties): exact passes over the scores
            }
        }
    }

    uint32_t next_guess = 0u;
    if (exact) {
        topk_exact_row(scores + (int64_t)rr * dm.MB * kBlock, list + (int64_t)req * dm.MB, cnt, n, K, false, out,
                       status, sh.exact);
    } else {
        if (take_all) {
            // every live candidate, as a bitmap of list positions
            for (int wd = tid; wd < W; wd += kThThreads) {
                const int e = wd >> 1;
                const int blk = slist[e];
                uint32_t m = 0u;
                if (blk >= 0 && blk < nb) {
                    const int64_t first = (int64_t)blk * kBlock + (wd & 1) * 32;
                    const int64_t live = n - first;
                    m = live >= 32 ? 0xffffffffu : live <= 0 ? 0u : ((1u << live) - 1u);
                }
                bits[wd] = m;
            }
            __syncthreads();
        } else {
            const unsigned long long U = th_kth_entry(cand, nc, K, sh);
            const int kp = (int)min((int64_t)nc, (int64_t)K + extra);
            // the next guess: the score at rank K + extra over this step's sum of |w_h|
            const float t = key_float((uint32_t)(th_kth_entry(cand, nc, kp, sh) >> 32));
            const float ws = row_wsum(w + (int64_t)rr * cfg.n_heads, cfg.n_heads);
            if (ws > 0.0f) {
                const float g = __fdiv_rn(t, ws);
                if (isfinite(g)) next_guess = order_key(g) == 0u ? 1u : order_key(g);
            }
            for (int i = tid; i < nc; i += kThThreads) {
                const unsigned long long x = cand[i];
                const uint32_t p = ~(uint32_t)(x & 0xffffffffull);
                if (x >= U && (int64_t)p < C) atomicOr(&bits[p >> 5], 1u << (p & 31));
            }
            __syncthreads();
        }
        // ordered write: thread t owns a contiguous run of bitmap words
        const int per = (W + kThThreads - 1) / kThThreads;
        const int w0 = min(W, tid * per), w1 = min(W, w0 + per);
        int mine = 0;
        for (int wd = w0; wd < w1; ++wd) mine += __popc(bits[wd]);
        int total;
        int pos = block_excl_scan(mine, sh.scan, &total);
        for (int wd = w0; wd < w1 && pos < K; ++wd) {
            uint32_t m = bits[wd];
            while (m && pos < K) {
                const int b = __ffs(m) - 1;
                m &= m - 1u;
                const int p = wd * 32 + b;
                out[pos++] = (int32_t)((int64_t)slist[p >> 6] * kBlock + (p & 63));
            }
        }
        for (int k = total + tid; k < K; k += kThThreads) out[k] = -1;
    }

    if (tid == 0) {
        rec[kHwCount] = 0u;
        rec[kHwGuess] = next_guess;
        uint32_t nx = extra;
        if (hit) {
            rec[kHwHit] += 1u;
        } else if (guess == 0u) {
            rec[kHwCold] += 1u;
        } else if (count < (uint32_t)K) {
            rec[kHwMiss] += 1u;
            nx = extra * 2u;
        } else {
            rec[kHwOver] += 1u;
            nx = extra / 2u;
        }
        rec[kHwExtra] = nx < kmin ? kmin : nx > kmax ? kmax : nx;
        if (exact) rec[kHwGlobal] += 1u;
        rec[kHwLast] = count;
    }
}

cudaError_t launch_topk_hint(const spin_config& cfg, const float* scores, const float* w, const int32_t* list,
                             const int32_t* n_list, const int32_t* n_slots, int rows, int32_t* topk_idx,
                             const HintArgs& h, uint32_t* status, cudaStream_t s) {
    const Dims dm = dims_of(cfg);
    const size_t smem = ((sizeof(ThShared) + 15) & ~(size_t)15) + (size_t)h.cap * 8 + (size_t)dm.MB * 12;
    cudaError_t e = cudaFuncSetAttribute(topk_hint_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_hint_kernel, dim3((unsigned)(cfg.n_req * rows)), dim3(kThThreads), smem, s, nullptr, 0,
                      cfg, scores, w, list, n_list, n_slots, rows, topk_idx, h, status);
}

}  // namespace spin

// spin_topk_hint.cu -- temporal top-K: last step's threshold as the guess of this step's.
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention", Algorithm 1's top-K step (the K
// largest fresh scores, equal scores to the lower slot id), computed the way the paper's
// related work ("Guess-Verify-Refine", §5) accelerates the post-indexer top-K: consecutive
// decode steps of one request score the same context with a slowly drifting query, so the
// K-th score moves little from one step to the next.
//
//   guess   every live fresh score is compared with the row's threshold -- the previous
//           step's score at rank K + extra, divided by that step's sum_h |w_h| and multiplied
//           by this step's (the head weights of a step scale all its scores together) -- and
//           those at or above it (a few per cent of the slots) become the candidates.  The
//           streaming and generic score kernels (spin_indexer_score_ex with the hint) do this
//           as they write the scores and mark the record; otherwise (the tensor-core kernel,
//           whose epilogue is its bottleneck) this kernel does it in one pass over the scores;
//   verify  if at least K and at most cap candidates were found, the top-K lies among them:
//           the K-th key T is >= the guess because K keys are, so every key > T and every
//           key == T was collected;
//   refine  an exact radix select over the candidates (64-bit entries: key, then the
//           complement of the list position, all distinct) gives the K largest entries;
//           they are marked in a bitmap of list positions and written in ascending slot
//           order.  The score at rank K + extra, normalised, becomes the next step's guess.
// The candidates' keys all lie between their minimum and maximum, so the radix digits start
// below the bits those two share; the first digit pass also places rank K + extra, whose
// bin's lower edge, normalised, becomes the next step's guess.
// A row without a guess, or whose guess found too few or too many candidates, takes the
// cold path: one pass over its scores counts the live keys and finds their minimum and
// maximum; 12-bit histograms below the shared bits place rank K + extra (refined 12 bits
// at a time while its bin alone overflows the candidate array); a last pass collects every
// live key at or above that bin, and the same refine step follows.  The margin `extra`
// starts at the geometric middle of [K, cap] minus K, doubles after a miss and halves
// after an overflow.  Only a boundary bin too large for the candidate array (massive ties)
// falls back to exact radix passes over the scores.  Every path returns exactly the top-K
// of spin_topk; the hint only decides how fast.
//
// One 1024-thread CTA per (request, row).  Shared memory: the candidates (cap 8-byte
// entries), the position bitmap (2 words per list entry) and the row's list.
#include "spin_common.cuh"
#include "spin_internal.h"
#include "spin_topk_rows.cuh"

namespace spin {

constexpr int kThThreads = 1024;
constexpr int kThMaxK = 2048;        // cap <= 16384 candidates (128 KB of shared memory)
constexpr int kThMaxBlocks = 8192;   // bitmap of the list positions: <= 64 KB
constexpr int kThBinsA = 4096;       // cold pass: top 12 bits of the key
constexpr int kThBins = 2048;        // candidate radix: 11-bit digits of the 64-bit entry
constexpr size_t kThSmemBudget = 220 * 1024;

struct ThShared {
    __align__(16) int hist[kThBinsA];
    int scan[33];
    int ncand;
    int digit, above, nbin, gdigit;
    uint32_t kmin, kmax;  // smallest and largest key of the candidates (or live keys)
    float wsum;           // sum_h |w_h| of the row
    TopkShared exact;     // the exact fallback's own scratch
};

static_assert(kThThreads == kTopkThreads, "the exact fallback runs with the same CTA");

static size_t th_smem_bytes(const spin_config& cfg, int cap) {
    return ((sizeof(ThShared) + 15) & ~(size_t)15) + (size_t)cap * 8 + (size_t)dims_of(cfg).MB * 12;
}

// Candidate capacity per row: 8 K rounded up to a power of two (at least 4096), or 4 K when
// that does not fit in shared memory next to the bitmap and the list.
int topk_hint_cap(const spin_config& cfg) {
    int c = 4096;
    while (c < 8 * cfg.top_k) c <<= 1;
    if (th_smem_bytes(cfg, c) > kThSmemBudget && c > 4096 && c / 2 >= 4 * cfg.top_k) c /= 2;
    return c;
}

// Initial rank margin: the guess aims at the geometric middle of [K, cap], where the
// candidate count has as much room to shrink as to grow.
__device__ __forceinline__ uint32_t th_default_extra(int K, int cap) {
    const int mid = (int)sqrtf((float)K * (float)cap);
    return mid > K ? (uint32_t)(mid - K) : 1u;
}

bool topk_hint_supported(const spin_config& cfg) {
    return cfg.top_k <= kThMaxK && dims_of(cfg).MB <= kThMaxBlocks &&
           th_smem_bytes(cfg, topk_hint_cap(cfg)) <= kThSmemBudget;
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

// Digit search over `nbins` bins (a multiple of 128), scanned from the top, by warp 0 alone:
// the bin d with (# in bins > d) < kk <= (# in bins >= d), for kk and (when kk2 > 0) kk2.
// Lane l first sums its nbins / 32 consecutive bins (16-byte reads); the lane whose range
// holds the rank is then scanned by the whole warp, nbins / 1024 bins a lane.  Leaves d, the
// count above it and the bin's own count in sh (and kk2's digit in sh.gdigit); the caller's
// barrier publishes them.  1 <= kk, kk2 <= the total.
__device__ __forceinline__ void th_find_one(const int* hist, int nbins, int inc, int c, int kk, int* digit,
                                            int* above_out, int* nbin) {
    const int lane = threadIdx.x & 31;
    const int per = nbins / 32;
    const int src = __ffs(__ballot_sync(0xffffffffu, inc >= kk)) - 1;
    const int above0 = __shfl_sync(0xffffffffu, inc - c, src);
    const int q = per / 32;
    const int top = nbins - 1 - src * per - lane * q;
    int c2 = 0;
    for (int b = 0; b < q; ++b) c2 += hist[top - b];
    const int inc2 = above0 + warp_incl_scan(c2);
    const int src2 = __ffs(__ballot_sync(0xffffffffu, inc2 >= kk)) - 1;
    if (lane == src2) {
        int above = inc2 - c2;
        for (int b = 0; b < q; ++b) {
            const int h = hist[top - b];
            if (above + h >= kk) {
                *digit = top - b;
                *above_out = above;
                *nbin = h;
                break;
            }
            above += h;
        }
    }
}

__device__ __forceinline__ void th_find_digit_warp(const int* hist, int nbins, int kk, int kk2, ThShared& sh) {
    const int lane = threadIdx.x & 31;
    const int per = nbins / 32;
    const int4* h4 = reinterpret_cast<const int4*>(hist + (nbins - (lane + 1) * per));
    int c = 0;
#pragma unroll 4
    for (int j = 0; j < per / 4; ++j) {
        const int4 v = h4[j];
        c += v.x + v.y + v.z + v.w;
    }
    const int inc = warp_incl_scan(c);
    th_find_one(hist, nbins, inc, c, kk, &sh.digit, &sh.above, &sh.nbin);
    if (kk2 > 0) {
        int a2, n2;
        th_find_one(hist, nbins, inc, c, kk2, &sh.gdigit, &a2, &n2);
    }
}

// The same over the whole CTA (every thread gets the result; ends with a barrier).
__device__ __forceinline__ void th_find_digit(const int* hist, int nbins, int kk, ThShared& sh, int kk2 = 0) {
    if (threadIdx.x < 32) th_find_digit_warp(hist, nbins, kk, kk2, sh);
    __syncthreads();
}

// Adds this thread's bin (-1: none) to a shared histogram: one atomic for the warp when all
// its lanes share a bin (ties, a narrow score range), else one per lane (the keys of a
// candidate array, below the bits they share, spread over many bins).
__device__ __forceinline__ void th_hist_add(int* hist, int bin) {
    const int b0 = __shfl_sync(0xffffffffu, bin, 0);
    if (__all_sync(0xffffffffu, bin == b0)) {
        if ((threadIdx.x & 31) == 0 && b0 >= 0) atomicAdd(&hist[b0], 32);
    } else if (bin >= 0) {
        atomicAdd(&hist[bin], 1);
    }
}

// Warp-reduced minimum and maximum of a key (0xffffffff / 0 for lanes without one) into sh.
__device__ __forceinline__ void th_minmax(uint32_t lo, uint32_t hi, ThShared& sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if ((threadIdx.x & 31) == 0) {
        atomicMin(&sh.kmin, lo);
        atomicMax(&sh.kmax, hi);
    }
}

// Threshold U with exactly k of the n (distinct) entries >= U, 1 <= k <= n, whose keys all
// lie in [sh.kmin, sh.kmax]: radix select over 11-bit digits starting below the key bits the
// extremes share, stopping as soon as the bin holding rank k is needed whole.  The first
// pass also places rank kp >= k: *guess is the key of its bin's lower edge (at least kp
// entries have a key >= it).
__device__ unsigned long long th_select(const unsigned long long* v, int n, int k, int kp, uint32_t* guess,
                                        ThShared& sh) {
    const uint32_t kmin = sh.kmin, kmax = sh.kmax;
    const int p = kmin == kmax ? 32 : __clz(kmin ^ kmax);  // key bits every entry shares
    unsigned long long mask = p == 0 ? 0ull : (~0ull << (64 - p));
    unsigned long long prefix = ((unsigned long long)kmin << 32) & mask;
    int top = 64 - p, kk = k;
    bool first = true;
    while (top > 0) {
        const int wdt = top < 11 ? top : 11;
        const int shift = top - wdt;
        const unsigned long long dmask = (1ull << wdt) - 1ull;
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
        th_find_digit(sh.hist, kThBins, kk, sh, first ? kp : 0);
        if (first) {
            *guess = (uint32_t)((prefix | ((unsigned long long)sh.gdigit << shift)) >> 32);
            first = false;
        }
        prefix |= (unsigned long long)sh.digit << shift;
        mask |= dmask << shift;
        kk -= sh.above;
        top = shift;
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
    // (thread 0 rewrites the record at the end, after many barriers: every thread has read it)
    float wpart = 0.0f;  // warp 0: its lanes' share of sum_h |w_h|, loaded while the list comes in
    if (tid < 32)
        for (int hh = tid; hh < cfg.n_heads; hh += 32) wpart += fabsf(w[(int64_t)rr * cfg.n_heads + hh]);
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

    // the whole list array (MB entries) is staged, so its loads need not wait for the count;
    // four entries per thread are loaded before any is stored
    bool bad_list = false;
    for (int k0 = tid; k0 < dm.MB; k0 += 4 * kThThreads) {
        int b4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = k0 + u * kThThreads;
            b4[u] = k < dm.MB ? list[(int64_t)req * dm.MB + k] : 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = k0 + u * kThThreads;
            if (k < dm.MB) {
                if (k < cnt && (b4[u] < 0 || b4[u] >= nb)) bad_list = true;
                slist[k] = b4[u];
            }
        }
    }
    if (bad_list && rr % rows == 0) set_status(status, SPIN_STATUS_BAD_LIST);
    for (int wd = tid; wd < W; wd += kThThreads) bits[wd] = 0u;
    if (tid == 0) {
        sh.ncand = 0;
        sh.kmin = 0xffffffffu;
        sh.kmax = 0u;
    }
    if (tid < 32) {  // sum_h |w_h| of the row
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wpart += __shfl_xor_sync(0xffffffffu, wpart, o);
        if (tid == 0) sh.wsum = wpart;
    }
    __syncthreads();

    // Keys of four candidates (0: not a live candidate).
    const float4* sc4 = reinterpret_cast<const float4*>(scores + (int64_t)rr * dm.MB * kBlock);
    const int C4 = (int)(C / 4);
    const int C4pad = (C4 + 31) & ~31;
    auto keys4 = [&](int i4, const float4& z, uint32_t* k4) {
        const int c = 4 * i4;
        const int blk = i4 < C4 ? slist[c >> 6] : -1;  // (padding lanes read nothing)
        const int64_t slot = (int64_t)blk * kBlock + (c & 63);
        const bool okb = blk >= 0 && blk < nb;
        k4[0] = okb && slot + 0 < n ? order_key(z.x) : 0u;
        k4[1] = okb && slot + 1 < n ? order_key(z.y) : 0u;
        k4[2] = okb && slot + 2 < n ? order_key(z.z) : 0u;
        k4[3] = okb && slot + 3 < n ? order_key(z.w) : 0u;
    };
    // body(i4, k4) for every i4 < C4pad (whole warps: C4pad is a multiple of 32; k4 is zero
    // past C4), four 16-byte loads in flight per thread
    auto scan_keys = [&](auto&& body) {
        const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i0 = tid; i0 < C4pad; i0 += 4 * kThThreads) {
            float4 z[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * kThThreads;
                z[u] = i < C4 ? sc4[i] : zero;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * kThThreads;
                if (i < C4pad) {  // (warp-uniform)
                    uint32_t k4[4];
                    keys4(i, z[u], k4);
                    body(i, k4);
                }
            }
        }
    };
    // Appends the warp's keys >= tkey (as candidate entries at position 4 i4 + e) to the shared
    // candidate array.  Each warp fills 32-entry chunks it claims with one atomic (sh.ncand
    // counts the entries claimed); `seen` counts the keys taken, `lo`/`hi` track their extremes.
    // Warp-uniform chunk state: base (-1: none yet) and fill.
    auto collect4 = [&](int i4, const uint32_t* k4, uint32_t tkey, int& cbase, int& cfill, int& seen_w,
                        uint32_t& lo, uint32_t& hi) {
        const int lane = tid & 31;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool take = k4[e] != 0u && k4[e] >= tkey;
            const unsigned m = __ballot_sync(0xffffffffu, take);
            if (m == 0u) continue;
            const int nm = __popc(m), rank = __popc(m & ((1u << lane) - 1u));
            seen_w += nm;
            const int room = cbase < 0 ? 0 : 32 - cfill;
            int nbase = cbase;
            if (nm > room) {  // a new chunk for the rest of the batch
                int b = 0;
                if (lane == 0) b = atomicAdd(&sh.ncand, 32);
                nbase = __shfl_sync(0xffffffffu, b, 0);
            }
            if (take) {
                const int at = rank < room ? cbase + cfill + rank : nbase + (rank - room);
                if (at < h.cap) {
                    cand[at] = hint_entry(k4[e], (uint32_t)(4 * i4 + e));
                    lo = min(lo, k4[e]);
                    hi = max(hi, k4[e]);
                }
            }
            if (nm > room) {
                cbase = nbase;
                cfill = nm - room;
            } else {
                cfill += nm;
            }
        }
    };
    // zero the unfilled tail of the warp's last chunk (entries of key 0 rank below every
    // candidate, so they are never selected)
    auto close_chunk = [&](int cbase, int cfill) {
        const int lane = tid & 31;
        if (cbase >= 0 && lane >= cfill && cbase + lane < h.cap) cand[cbase + lane] = 0ull;
    };

    const bool collected = (rec[kHwFlags] & 1u) != 0u;
    uint32_t seen = count;  // candidates at or above this step's threshold
    int nc_claimed = (int)count;  // entries of the candidate array in use
    bool hit = false;
    if (guess != 0u && collected) {
        // the score kernel collected them
        if (count >= (uint32_t)K && count <= (uint32_t)h.cap) {
            hit = true;
            const unsigned long long* src = h.cand + (int64_t)rr * h.cap;
            uint32_t lo = 0xffffffffu, hi = 0u;
            for (int i0 = tid; i0 < (int)count; i0 += 4 * kThThreads) {  // four loads in flight
                unsigned long long x4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * kThThreads;
                    x4[u] = i < (int)count ? src[i] : 0ull;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * kThThreads;
                    if (i < (int)count) {
                        cand[i] = x4[u];
                        lo = min(lo, (uint32_t)(x4[u] >> 32));
                        hi = max(hi, (uint32_t)(x4[u] >> 32));
                    }
                }
            }
            th_minmax(lo, hi, sh);
            __syncthreads();
        }
    } else if (guess != 0u) {
        // collect them here: one pass over the scores against this step's threshold
        const uint32_t thr = hint_threshold(guess, sh.wsum);
        uint32_t lo = 0xffffffffu, hi = 0u;
        int cbase = -1, cfill = 0, seen_w = 0;
        scan_keys([&](int i4, const uint32_t* k4) { collect4(i4, k4, thr, cbase, cfill, seen_w, lo, hi); });
        close_chunk(cbase, cfill);
        th_minmax(lo, hi, sh);
        seen = (uint32_t)th_block_sum((tid & 31) == 0 ? seen_w : 0, sh);
        // (the claimed chunks, zero tails included, must fit: at most one partial chunk a warp)
        hit = seen >= (uint32_t)K && sh.ncand <= h.cap;
        nc_claimed = sh.ncand;
        __syncthreads();
        if (!hit && tid == 0) {
            sh.ncand = 0;
            sh.kmin = 0xffffffffu;
            sh.kmax = 0u;
        }
        __syncthreads();
    }
    bool take_all = false, exact = false;
    int nc = hit ? nc_claimed : 0;
    int seen_cold = 0;  // live candidates collected by the cold path
    if (!hit) {
        // cold path
        // pass A: live count, smallest and largest live key
        int v = 0;
        uint32_t lo = 0xffffffffu, hi = 0u;
        scan_keys([&](int, const uint32_t* k4) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (k4[e]) {
                    ++v;
                    lo = min(lo, k4[e]);
                    hi = max(hi, k4[e]);
                }
        });
        th_minmax(lo, hi, sh);
        const int nvalid = th_block_sum(v, sh);  // (its barriers also complete the extremes)
        if (nvalid <= K) {
            take_all = true;
        } else {
            // the bin holding rank kp, 12 bits at a time below the bits every live key shares,
            // until the keys at or above it fit the candidate array
            const int kp = (int)min((int64_t)nvalid, (int64_t)K + extra);
            const uint32_t kmn = sh.kmin, kmx = sh.kmax;
            const int pbits = kmn == kmx ? 32 : __clz(kmn ^ kmx);
            uint32_t tmask = pbits == 0 ? 0u : (0xffffffffu << (32 - pbits));
            uint32_t tkey = kmn & tmask;  // collect the live keys >= tkey
            int top = 32 - pbits, above = 0, total = nvalid;
            const int fit = h.cap - 32 * (kThThreads / 32);  // room left for the warps' chunk tails
            while (top > 0 && total > fit) {
                const int wdt = top < 12 ? top : 12;
                const int shift = top - wdt;
                const uint32_t dmask = (1u << wdt) - 1u;
                for (int b = tid; b < kThBinsA; b += kThThreads) sh.hist[b] = 0;
                __syncthreads();
                scan_keys([&](int, const uint32_t* k4) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        th_hist_add(sh.hist, k4[e] != 0u && (k4[e] & tmask) == tkey ? (int)((k4[e] >> shift) & dmask) : -1);
                });
                __syncthreads();
                th_find_digit(sh.hist, kThBinsA, kp - above, sh);
                total = above + sh.above + sh.nbin;
                above += sh.above;
                tkey |= (uint32_t)sh.digit << shift;
                tmask |= dmask << shift;
                top = shift;
                __syncthreads();
            }
            if (total <= fit) {
                // collect every live candidate with key >= tkey (all of rank <= kp)
                if (tid == 0) {
                    sh.kmin = 0xffffffffu;
                    sh.kmax = 0u;
                }
                __syncthreads();
                uint32_t clo = 0xffffffffu, chi = 0u;
                int cbase = -1, cfill = 0, seen_w = 0;
                scan_keys([&](int i4, const uint32_t* k4) { collect4(i4, k4, tkey, cbase, cfill, seen_w, clo, chi); });
                close_chunk(cbase, cfill);
                th_minmax(clo, chi, sh);
                __syncthreads();
                nc = sh.ncand;
                seen_cold = total;
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
            // (nc may include zero entries of chunk tails; the live candidates number `live`)
            const int live = hit ? (int)seen : seen_cold;
            const int kp = (int)min((int64_t)live, (int64_t)K + extra);
            uint32_t gkey = 0u;
            const unsigned long long U = th_select(cand, nc, K, kp, &gkey, sh);
            // the next guess: the score at rank K + extra over this step's sum of |w_h|
            const float ws = sh.wsum;
            if (ws > 0.0f) {
                const float g = __fdiv_rn(key_float(gkey), ws);
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
        rec[kHwFlags] = 0u;
        rec[kHwGuess] = next_guess;
        uint32_t nx = extra;
        if (hit) {
            rec[kHwHit] += 1u;
        } else if (guess == 0u) {
            rec[kHwCold] += 1u;
        } else if (seen < (uint32_t)K) {
            rec[kHwMiss] += 1u;
            nx = extra * 2u;
        } else {
            rec[kHwOver] += 1u;
            nx = extra / 2u;
        }
        rec[kHwExtra] = nx < kmin ? kmin : nx > kmax ? kmax : nx;
        if (exact) rec[kHwGlobal] += 1u;
        rec[kHwLast] = seen;
    }
}

cudaError_t launch_topk_hint(const spin_config& cfg, const float* scores, const float* w, const int32_t* list,
                             const int32_t* n_list, const int32_t* n_slots, int rows, int32_t* topk_idx,
                             const HintArgs& h, uint32_t* status, cudaStream_t s) {
    const size_t smem = th_smem_bytes(cfg, h.cap);
    cudaError_t e = cudaFuncSetAttribute(topk_hint_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_hint_kernel, dim3((unsigned)(cfg.n_req * rows)), dim3(kThThreads), smem, s, nullptr, 0,
                      cfg, scores, w, list, n_list, n_slots, rows, topk_idx, h, status);
}

}  // namespace spin

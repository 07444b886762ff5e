// spin_topk_sample.cu -- post-indexer top-K by a sampled bracket (one CTA per request row).
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention", Algorithm 1's top-K step:
// T_t = TopK(z_t, K) over the slots the indexer scored; equal scores at the K-th value go
// to the lower slot id.  The candidates are the listed blocks' slots i < N in list order,
// which is ascending slot order.
//
// Exact selection with one streaming pass over the scores:
//   1. a fixed sample of 1024 candidates (one per thread) brackets the K-th largest key:
//      two order statistics of the sample, K*1024/C -/+ four standard deviations, found by
//      8-bit radix passes over the sample in registers;
//      (the collected keys share the leading bytes of the bracket's lower end and their
//      maximum, so their radix passes start at the first byte where those differ, and stop
//      once the threshold bin is kept whole)
//   2. one pass over every candidate (a warp reads 128 consecutive scores per float4 load,
//      several loads in flight per thread) writes the keys above the bracket straight into a
//      bitmap of the candidates (shuffles, no atomics) and collects the keys inside the
//      bracket (typically 1-5 % of the candidates) into per-warp segments of shared memory
//      (ballot offsets, no atomics); the comparisons are made on the scores, and the number
//      of live candidates comes from the list;
//   3. if the K-th key is inside the bracket, radix passes over the collected keys give
//      the exact threshold T and the number of keys equal to T to keep; otherwise (a
//      sample that missed, or a bracket holding too many keys, e.g. when all scores tie)
//      the threshold is found by radix passes over all candidates instead;
//   4. equal keys at T are cut in candidate order when not all of them are kept, and the
//      bitmap is read out in candidate order: ascending slot ids, padded with -1.
// Only the sample and the bracket decide the speed; the result is the same either way.
#include "spin_common.cuh"
#include "spin_internal.h"

namespace spin {

constexpr int kTsThreads = 1024;
constexpr int kTsWarps = kTsThreads / 32;
constexpr int kTsSample = kTsThreads;  // one sampled candidate per thread
constexpr int kTsMid = 16384;          // capacity of the collected in-bracket keys
constexpr int kTsMidKpt = kTsMid / kTsThreads;
constexpr int kTsRun = 64;                     // entries a warp claims at least at a time
constexpr int kTsLoads = 4;                    // float4 loads in flight per thread

struct TsShared {
    __align__(16) int hist[6][256];  // radix histograms: 3 rotating buffers x 2 targets
    int red[kTsWarps][5];  // block sums, one slot per use (no barrier needed between uses)
    uint32_t redu[kTsWarps];  // block maximum
    int npool;                // entries of the collection claimed by the warps' runs
    int scan[33];
    int bad_list;
};

__host__ __device__ inline size_t ts_smem_bytes(const spin_config& cfg) {
    const int64_t MB = ((int64_t)cfg.max_slots + kBlock - 1) / kBlock;
    // TsShared | list[MB] | bitmap[2 MB] | eqmap[2 MB] | midkey[kTsMid] | midpos[kTsMid]
    return ((sizeof(TsShared) + 15) & ~(size_t)15) + (size_t)MB * 4 + (size_t)MB * 8 * 2 + (size_t)kTsMid * 8;
}

// The float whose order key is `key` (inverse of order_key for keys of finite floats).
__device__ __forceinline__ float key_to_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Adds the warp's bins (-1: none) to a shared histogram: the lanes that share the first
// active lane's bin with one atomic, the others one atomic each (keys of one warp mostly
// share a bin when they are concentrated, and mostly differ when they are spread).
__device__ __forceinline__ void ts_hist_add(int* h, int bin) {
    const int lane = threadIdx.x & 31;
    const unsigned act = __ballot_sync(0xffffffffu, bin >= 0);
    if (act == 0u) return;
    const int lead = __ffs(act) - 1;
    const int b0 = __shfl_sync(0xffffffffu, bin, lead);
    const unsigned m0 = __ballot_sync(0xffffffffu, bin == b0);
    if (lane == lead) atomicAdd(&h[b0], __popc(m0));
    else if (bin >= 0 && bin != b0) atomicAdd(&h[bin], 1);
}

// Every warp: the digit whose bin holds the kk-th largest key of a 256-bin histogram, the
// number of keys in higher bins and the bin's own count.  Lane l reads bins 255-8l ..
// 248-8l as two 16-byte vectors.
__device__ __forceinline__ void ts_digit(const int* h, int kk, int& digit, int& above, int& nbin) {
    const int lane = threadIdx.x & 31;
    const int4 v_hi = reinterpret_cast<const int4*>(h)[63 - 2 * lane];
    const int4 v_lo = reinterpret_cast<const int4*>(h)[62 - 2 * lane];
    const int cnt[8] = {v_hi.w, v_hi.z, v_hi.y, v_hi.x, v_lo.w, v_lo.z, v_lo.y, v_lo.x};
    int sum = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) sum += cnt[b];
    const int inc = warp_incl_scan(sum);
    const unsigned ball = __ballot_sync(0xffffffffu, inc >= kk);
    const int src = ball ? __ffs(ball) - 1 : 31;
    int ab = inc - sum, dg = 0, nb = 0;
#pragma unroll
    for (int b = 0, found = 0; b < 8; ++b) {
        if (!found) {
            if (ab + cnt[b] >= kk) { dg = 255 - 8 * lane - b; nb = cnt[b]; found = 1; }
            else ab += cnt[b];
        }
    }
    digit = __shfl_sync(0xffffffffu, dg, src);
    above = __shfl_sync(0xffffffffu, ab, src);
    nbin = __shfl_sync(0xffffffffu, nb, src);
}

// Clears the histogram buffers that pass `pass + 2` will fill (they were last read before
// this pass's barrier).
__device__ __forceinline__ void ts_clear_ahead(TsShared& sh, int pass) {
    const int tid = threadIdx.x;
    if (tid < 512) sh.hist[((pass + 2) % 3) * 2 + (tid >> 8)][tid & 255] = 0;
}

// For each target t < NT: the k[t]-th largest (1 <= k[t] <= number of eligible keys) of the
// keys held in registers (KPT per thread, bit i of `elig` marks key[i] eligible).  Returns
// its value T[t] and the number of eligible keys above it.  All threads call it; on entry
// the buffers of passes `pass` and `pass + 1` are zero, and so are they on return.
// The first `d0` bytes of every eligible key are known to equal those of `common`; those
// digit passes are skipped.  With one target and all four digits asked for, the passes stop
// once the threshold bin is taken whole: T is then one below the bin's lowest key, with
// every eligible key above it counted and none equal to it.
// Only the key slots i < nslot (CTA-uniform) are looked at, and only the digits d0 .. d1-1;
// with d1 < 4 the results are the order statistics' leading 8*d1 bits (the rest zero) and
// `above` counts the eligible keys in higher 8*d1-bit bins.
template <int KPT, int NT>
__device__ void ts_kth_regs(const uint32_t (&key)[KPT], uint32_t elig, const int (&k)[NT], uint32_t (&T)[NT],
                            int (&above)[NT], TsShared& sh, int& pass, int d0 = 0, uint32_t common = 0u,
                            int nslot = KPT, int d1 = 4) {
    uint32_t mask = d0 > 0 ? ~(0xFFFFFFFFu >> (8 * d0)) : 0u;
    uint32_t prefix[NT];
    int kk[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) { prefix[t] = common & mask; kk[t] = k[t]; }
    for (int d = d0; d < d1; ++d, ++pass) {
        const int shift = 24 - 8 * d;
        const bool shared_prefix = NT == 2 && prefix[0] == prefix[NT - 1];
        int* h0 = sh.hist[(pass % 3) * 2];
        int* h1 = sh.hist[(pass % 3) * 2 + 1];
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
            if (i >= nslot) break;  // CTA-uniform
            const bool e = (elig >> i) & 1u;
            const int dg = (int)((key[i] >> shift) & 255u);
            ts_hist_add(h0, e && (key[i] & mask) == prefix[0] ? dg : -1);
            if (NT == 2 && !shared_prefix) ts_hist_add(h1, e && (key[i] & mask) == prefix[NT - 1] ? dg : -1);
        }
        __syncthreads();
        int nbin0 = 0;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            int dg, ab, nb;
            ts_digit(t == 0 || shared_prefix ? h0 : h1, kk[t], dg, ab, nb);
            prefix[t] |= (uint32_t)dg << shift;
            kk[t] -= ab;
            if (t == 0) nbin0 = nb;
        }
        ts_clear_ahead(sh, pass);
        mask |= 0xFFu << shift;
        if (NT == 1 && d1 == 4 && d < 3 && kk[0] == nbin0 && prefix[0] != 0u) {
            ++pass;
            T[0] = prefix[0] - 1u;
            above[0] = k[0];
            return;
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) { T[t] = prefix[t]; above[t] = k[t] - kk[t]; }
}

// The candidates as a stream of float4 (4 consecutive candidates of one block).
struct TsCands {
    const float4* sc4;
    const int* slist;  // shared copy of the row's list
    int64_t n, nb;
    int C4;
    __device__ __forceinline__ void keys(int f4, const float4& z, uint32_t (&k)[4], bool& bad) const {
        const int c = 4 * f4;
        const int blk = slist[c >> 6];
        const bool okb = blk >= 0 && blk < nb;
        bad = !okb;
        const int64_t slot = (int64_t)blk * kBlock + (c & 63);
        k[0] = okb && slot + 0 < n ? order_key(z.x) : 0u;
        k[1] = okb && slot + 1 < n ? order_key(z.y) : 0u;
        k[2] = okb && slot + 2 < n ? order_key(z.z) : 0u;
        k[3] = okb && slot + 3 < n ? order_key(z.w) : 0u;
    }
};

// The k-th largest live key over all candidates, by radix passes that re-read the scores
// (the path taken when the sampled bracket does not hold the threshold).
__device__ void ts_kth_stream(const TsCands& cs, int k, uint32_t& T, int& above, TsShared& sh, int& pass) {
    const int tid = threadIdx.x;
    uint32_t prefix = 0, mask = 0;
    int kk = k;
    const int C4pad = (cs.C4 + 31) & ~31;
    for (int d = 0; d < 4; ++d, ++pass) {
        const int shift = 24 - 8 * d;
        int* h = sh.hist[(pass % 3) * 2];
        for (int f4 = tid; f4 < C4pad; f4 += kTsThreads) {
            uint32_t kx[4] = {0u, 0u, 0u, 0u};
            bool bad = false;
            if (f4 < cs.C4) cs.keys(f4, cs.sc4[f4], kx, bad);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                ts_hist_add(h, kx[e] != 0u && (kx[e] & mask) == prefix ? (int)((kx[e] >> shift) & 255u) : -1);
        }
        __syncthreads();
        int dg, ab, nb;
        ts_digit(h, kk, dg, ab, nb);
        ts_clear_ahead(sh, pass);
        prefix |= (uint32_t)dg << shift;
        kk -= ab;
        mask |= 0xFFu << shift;
    }
    T = prefix;
    above = k - kk;
}

// Sum of v over the CTA (all threads call it).
__device__ __forceinline__ int ts_block_sum(int v, TsShared& sh, int slot) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sh.red[wid][slot] = v;
    __syncthreads();
    int s = sh.red[lane][slot];  // kTsWarps == 32: lane w takes warp w's partial
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// One warp's appends to the collection: keys collected, its current run [fill, end) (all
// warp-uniform) and the largest key this thread collected.
struct TsCollect {
    int wcnt, wfill, wend;
    uint32_t kmax;
};

// Step 2, the pass over every candidate.  Each warp takes 32 consecutive float4 (128
// candidates) per step, with kTsLoads steps' loads in flight per thread, and appends its
// in-bracket keys to a run of the collection that it claimed (at least kTsRun entries, one
// shared atomic per claim) at offsets from ballots.  A run given up for a new one has its
// unused entries set to key 0, which no live candidate has, so the collection is the
// claimed prefix with holes of key 0.  HI: the bracket has an upper end, and the keys
// above it are written to the bitmap here; without one nothing is above the bracket.
// Returns this thread's count of keys above the bracket.
template <bool HI>
__device__ __forceinline__ int ts_main_pass(const TsCands& cs, float z_lo, float z_hi, int Cw, uint32_t* bitmap,
                                            uint32_t* midkey, int* midpos, TsShared& sh, TsCollect& col) {
    const int tid = threadIdx.x, lane = tid & 31;
    const unsigned lt = (1u << lane) - 1u;
    const int C4 = cs.C4;
    int gt = 0;
    for (int base = 0; base < C4; base += kTsThreads * kTsLoads) {
        float4 zv[kTsLoads];
#pragma unroll
        for (int u = 0; u < kTsLoads; ++u) {
            const int f4 = base + u * kTsThreads + tid;
            zv[u] = f4 < C4 ? __ldg(cs.sc4 + f4) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < kTsLoads; ++u) {
            const int f4 = base + u * kTsThreads + tid;
            const int ch = f4 >> 5;  // the warp's chunk of 32 float4 (warp-uniform)
            if (32 * ch >= C4) continue;
            // live candidates of this float4: slot < N in a valid block
            int lim = 0;
            if (f4 < C4) {
                const int c = 4 * f4;
                const int blk = cs.slist[c >> 6];
                if (blk >= 0 && blk < cs.nb) {
                    const int64_t room = cs.n - (int64_t)blk * kBlock - (c & 63);
                    lim = room >= 4 ? 4 : (int)max(room, (int64_t)0);
                }
            }
            const float zz[4] = {zv[u].x, zv[u].y, zv[u].z, zv[u].w};
            uint32_t in = 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                in |= (uint32_t)(e < lim && zz[e] >= z_lo && (!HI || zz[e] <= z_hi)) << e;
            if (HI) {
                uint32_t nib = 0u;
#pragma unroll
                for (int e = 0; e < 4; ++e) nib |= (uint32_t)(e < lim && zz[e] > z_hi) << e;
                gt += __popc(nib);
                uint32_t wbits = nib << (4 * (lane & 7));
                wbits |= __shfl_xor_sync(0xffffffffu, wbits, 1);
                wbits |= __shfl_xor_sync(0xffffffffu, wbits, 2);
                wbits |= __shfl_xor_sync(0xffffffffu, wbits, 4);
                if ((lane & 7) == 0 && ch * 4 + (lane >> 3) < Cw) bitmap[ch * 4 + (lane >> 3)] = wbits;
            }
            if (__any_sync(0xffffffffu, in != 0u)) {
                unsigned bal[4];
                int t = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    bal[e] = __ballot_sync(0xffffffffu, (in >> e) & 1u);
                    t += __popc(bal[e]);
                }
                if (col.wfill + t > col.wend) {
                    for (int q = col.wfill + lane; q < min(col.wend, kTsMid); q += 32) midkey[q] = 0u;
                    const int claim = max(kTsRun, (t + 31) & ~31);
                    int b0 = 0;
                    if (lane == 0) b0 = atomicAdd(&sh.npool, claim);
                    col.wfill = __shfl_sync(0xffffffffu, b0, 0);
                    col.wend = col.wfill + claim;
                }
                int off = col.wfill;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if ((in >> e) & 1u) {
                        const int p = off + __popc(bal[e] & lt);
                        const uint32_t kx = order_key(zz[e]);
                        col.kmax = max(col.kmax, kx);
                        if (p < kTsMid) { midkey[p] = kx; midpos[p] = 4 * f4 + e; }
                    }
                    off += __popc(bal[e]);
                }
                col.wfill = off;
                col.wcnt += t;
            }
        }
    }
    for (int q = col.wfill + lane; q < min(col.wend, kTsMid); q += 32) midkey[q] = 0u;
    return gt;
}

// Maximum of v over the CTA (all threads call it).
__device__ __forceinline__ uint32_t ts_block_max(uint32_t v, TsShared& sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) sh.redu[wid] = v;
    __syncthreads();
    uint32_t m = sh.redu[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    return m;
}

__global__ void __launch_bounds__(kTsThreads, 1)
topk_sample_kernel(spin_config cfg, const float* __restrict__ scores, const int32_t* __restrict__ list,
                   const int32_t* __restrict__ n_list, const int32_t* __restrict__ n_slots, int rows,
                   int32_t* __restrict__ topk_idx, uint32_t* status) {
    pdl_begin();
    extern __shared__ __align__(16) unsigned char ts_smem[];
    TsShared& sh = *reinterpret_cast<TsShared*>(ts_smem);
    const Dims dm = dims_of(cfg);
    const int MB = dm.MB;
    int* slist = reinterpret_cast<int*>(ts_smem + ((sizeof(TsShared) + 15) & ~(size_t)15));
    uint32_t* bitmap = reinterpret_cast<uint32_t*>(slist + MB);
    uint32_t* eqmap = bitmap + 2 * (size_t)MB;
    uint32_t* midkey = eqmap + 2 * (size_t)MB;
    int* midpos = reinterpret_cast<int*>(midkey + kTsMid);

    const int rr = blockIdx.x, req = rr / rows;
    const int tid = threadIdx.x, lane = tid & 31;
    const int K = cfg.top_k;
    int32_t* out = topk_idx + (int64_t)rr * K;
    const int64_t n = n_slots[req];
    const int64_t cnt = n_list[req];
    if (n < 0 || n > dm.max_slots || cnt < 0 || cnt > MB) {
        if (tid == 0) set_status(status, (n < 0 || n > dm.max_slots) ? SPIN_STATUS_BAD_N : SPIN_STATUS_BAD_LIST);
        for (int k = tid; k < K; k += kTsThreads) out[k] = -1;
        return;
    }
    const int32_t* lst = list + (int64_t)req * MB;
    const float* sc = scores + (int64_t)rr * MB * kBlock;
    const int C = (int)cnt * kBlock;
    const int Cw = C / 32;
    TsCands cs{reinterpret_cast<const float4*>(sc), slist, n, (n + kBlock - 1) / kBlock, C / 4};

    // sampled candidate of this thread (read straight from global memory while the list is
    // being staged)
    uint32_t skey = 0u;
    const bool use_sample = C > kTsMid;
    if (use_sample) {
        const int c = (int)(((int64_t)tid * C + C / 2) / kTsSample);
        const int blk = __ldg(lst + (c >> 6));
        const int64_t slot = (int64_t)blk * kBlock + (c & 63);
        if (blk >= 0 && blk < cs.nb && slot < n) skey = order_key(__ldg(sc + c));
    }
    for (int i = tid; i < cnt; i += kTsThreads) slist[i] = lst[i];
    if (tid < 512) (&sh.hist[0][0])[tid] = 0;
    if (tid < 1024) (&sh.hist[0][0])[512 + tid] = 0;
    if (tid == 0) { sh.bad_list = 0; sh.npool = 0; }
    int pass = 0;

    // 1. the bracket [key_lo, key_hi] of the K-th largest key
    uint32_t key_hi = 0xFFFFFFFFu, key_lo = 1u;
    const int s_live = ts_block_sum(skey != 0u, sh, 0);  // (its barrier also publishes the above)
    if (use_sample && s_live > 0) {
        // expected sample rank of the K-th key, and four binomial standard deviations around it
        // (fp32: this GPU's fp64 rate is a small fraction of its fp32 rate)
        const float r = (float)K * (float)kTsSample / (float)C;
        const float sd = sqrtf(fmaxf(r * (1.0f - r / (float)kTsSample), 0.0f));
        const int r_hi = (int)floorf(r - 4.0f * sd - 2.0f), r_lo = (int)ceilf(r + 4.0f * sd + 2.0f);
        const int k2[2] = {max(1, min(r_hi, s_live)), max(1, min(r_lo, s_live))};
        uint32_t T2[2];
        int ab2[2];
        const uint32_t sk[1] = {skey};
        // the leading 16 bits of the two order statistics are enough for a bracket: it is
        // widened to the outer edges of their 16-bit bins
        ts_kth_regs<1, 2>(sk, skey != 0u ? 1u : 0u, k2, T2, ab2, sh, pass, 0, 0u, 1, 2);
        if (r_hi >= 1 && r_hi <= s_live) key_hi = T2[0] | 0xFFFFu;
        if (r_lo >= 1 && r_lo <= s_live) key_lo = max(T2[1], 1u);
        if (key_lo > key_hi) key_lo = key_hi;
    }

    // 2. one pass: keys above the bracket -> bitmap, keys inside it -> collected.  The
    // comparisons are made on the scores themselves (the key order is the float order, -0
    // equal to +0); keys are formed only for the collected ones.
    // (keys at or beyond those of +inf and -inf mean no bound on that side)
    const float z_hi = key_hi >= 0xFF800000u ? __int_as_float(0x7f800000) : key_to_float(key_hi);
    const float z_lo = key_lo <= 0x007FFFFFu ? __int_as_float(0xff800000) : key_to_float(key_lo);
    TsCollect col{0, 0, 0, 0u};
    int gt;
    if (key_hi >= 0xFF800000u) {  // no upper end: nothing is above the bracket
        for (int w = tid; w < Cw; w += kTsThreads) bitmap[w] = 0u;
        gt = ts_main_pass<false>(cs, z_lo, z_hi, Cw, bitmap, midkey, midpos, sh, col);
    } else {
        gt = ts_main_pass<true>(cs, z_lo, z_hi, Cw, bitmap, midkey, midpos, sh, col);
    }
    const int wcnt = col.wcnt;
    const uint32_t kmax = col.kmax;
    // live candidates, from the list alone (a listed block outside the context is an error)
    int live = 0;
    bool bad_list = false;
    for (int i = tid; i < cnt; i += kTsThreads) {
        const int blk = slist[i];
        if (blk >= 0 && blk < cs.nb) live += (int)min((int64_t)kBlock, cs.n - (int64_t)blk * kBlock);
        else bad_list = true;
    }
    if (bad_list) sh.bad_list = 1;
    gt = ts_block_sum(gt, sh, 1);  // (its barrier also publishes the collection)
    const int nvalid = ts_block_sum(live, sh, 2);
    const int nmid = ts_block_sum(lane == 0 ? wcnt : 0, sh, 4);
    const int npool = sh.npool;
    if (tid == 0 && sh.bad_list && rr % rows == 0) set_status(status, SPIN_STATUS_BAD_LIST);

    // 3. the exact threshold: keys > T are kept and the first `take_eq` keys == T
    bool eq_cut = false;
    if (nvalid <= K) {
        // every live candidate is kept: the bitmap is the live mask, from the list alone
        for (int w = tid; w < Cw; w += kTsThreads) {
            const int blk = slist[w >> 1];
            uint32_t bits = 0u;
            if (blk >= 0 && blk < cs.nb) {
                const int64_t s0 = (int64_t)blk * kBlock + 32 * (w & 1);
                const int64_t m = n - s0;
                bits = m >= 32 ? 0xFFFFFFFFu : m <= 0 ? 0u : ((1u << m) - 1u);
            }
            bitmap[w] = bits;
        }
    } else if (gt < K && gt + nmid >= K && npool <= kTsMid) {
        uint32_t mk[kTsMidKpt];
        uint32_t elig = 0;
#pragma unroll
        for (int i = 0; i < kTsMidKpt; ++i) {
            const int p = i * kTsThreads + tid;
            mk[i] = p < npool ? midkey[p] : 0u;
            elig |= (uint32_t)(mk[i] != 0u) << i;
        }
        const int k1[1] = {K - gt};
        uint32_t T1[1];
        int ab1[1];
        // every collected key lies in [key_lo, max]: their common leading bytes are known
        const uint32_t kmx = ts_block_max(kmax, sh);
        const uint32_t diff = key_lo ^ kmx;
        const int d0 = diff == 0u ? 3 : min(3, __clz(diff) / 8);
        ts_kth_regs<kTsMidKpt, 1>(mk, elig, k1, T1, ab1, sh, pass, d0, kmx, (npool + kTsThreads - 1) / kTsThreads);
        const uint32_t T = T1[0];
        const int take_eq = K - gt - ab1[0];
        int neq = 0;
#pragma unroll
        for (int i = 0; i < kTsMidKpt; ++i) neq += ((elig >> i) & 1u) && mk[i] == T;
        neq = ts_block_sum(neq, sh, 3);
        eq_cut = neq > take_eq;
        if (eq_cut)
            for (int w = tid; w < Cw; w += kTsThreads) eqmap[w] = 0u;
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kTsMidKpt; ++i) {
            if (!((elig >> i) & 1u)) continue;
            const int c = midpos[i * kTsThreads + tid];
            if (mk[i] > T || (mk[i] == T && !eq_cut)) atomicOr(&bitmap[c >> 5], 1u << (c & 31));
            else if (mk[i] == T) atomicOr(&eqmap[c >> 5], 1u << (c & 31));
        }
        if (eq_cut) {
            __syncthreads();
            // keep the first take_eq equal keys in candidate order
            const int per = (Cw + kTsThreads - 1) / kTsThreads;
            const int w0 = min(Cw, tid * per), w1 = min(Cw, w0 + per);
            int c0 = 0;
            for (int w = w0; w < w1; ++w) c0 += __popc(eqmap[w]);
            int tot;
            int rank = block_excl_scan(c0, sh.scan, &tot);
            for (int w = w0; w < w1 && rank < take_eq; ++w) {
                uint32_t bits = eqmap[w], keep = 0u;
                while (bits && rank < take_eq) {
                    const uint32_t low = bits & (0u - bits);
                    keep |= low;
                    bits ^= low;
                    ++rank;
                }
                if (keep) bitmap[w] |= keep;  // (one thread owns word w here)
            }
        }
    } else {
        // the sampled bracket missed the threshold or overflowed: radix over all candidates
        uint32_t T;
        int ab;
        ts_kth_stream(cs, K, T, ab, sh, pass);
        const int take_eq = K - ab;
        // rebuild the bitmap (keys > T) and the equal keys' map
        int neq = 0;
        for (int w = tid; w < Cw; w += kTsThreads) {
            uint32_t bg = 0u, be = 0u;
            const float4* s4 = cs.sc4 + 8 * w;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t kx[4];
                bool bad;
                cs.keys(8 * w + q, s4[q], kx, bad);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    bg |= (uint32_t)(kx[e] > T) << (4 * q + e);
                    be |= (uint32_t)(kx[e] != 0u && kx[e] == T) << (4 * q + e);
                }
            }
            neq += __popc(be);
            bitmap[w] = bg;
            eqmap[w] = be;
        }
        neq = ts_block_sum(neq, sh, 3);
        eq_cut = neq > take_eq;
        if (!eq_cut) {
            for (int w = tid; w < Cw; w += kTsThreads) bitmap[w] |= eqmap[w];
        } else {
            const int per = (Cw + kTsThreads - 1) / kTsThreads;
            const int w0 = min(Cw, tid * per), w1 = min(Cw, w0 + per);
            int c0 = 0;
            for (int w = w0; w < w1; ++w) c0 += __popc(eqmap[w]);
            int tot;
            int rank = block_excl_scan(c0, sh.scan, &tot);
            for (int w = w0; w < w1 && rank < take_eq; ++w) {
                uint32_t bits = eqmap[w], keep = 0u;
                while (bits && rank < take_eq) {
                    const uint32_t low = bits & (0u - bits);
                    keep |= low;
                    bits ^= low;
                    ++rank;
                }
                if (keep) bitmap[w] |= keep;
            }
        }
    }
    __syncthreads();

    // 4. read the bitmap out in candidate order
    {
        const int per = (Cw + kTsThreads - 1) / kTsThreads;
        const int w0 = min(Cw, tid * per), w1 = min(Cw, w0 + per);
        int c0 = 0;
        for (int w = w0; w < w1; ++w) c0 += __popc(bitmap[w]);
        int total;
        int pos = block_excl_scan(c0, sh.scan, &total);
        for (int w = w0; w < w1; ++w) {
            uint32_t bits = bitmap[w];
            while (bits) {
                const int b = __ffs(bits) - 1;
                bits &= bits - 1u;
                if (pos < K) {
                    const int c = 32 * w + b;
                    out[pos] = (int32_t)((int64_t)slist[c >> 6] * kBlock + (c & 63));
                }
                ++pos;
            }
        }
        for (int k = min(total, K) + tid; k < K; k += kTsThreads) out[k] = -1;
    }
}

bool topk_sample_fits(const spin_config& cfg) { return ts_smem_bytes(cfg) <= 220 * 1024; }

cudaError_t launch_topk_sample(const spin_config& cfg, const float* scores, const int32_t* list,
                               const int32_t* n_list, const int32_t* n_slots, int rows, int32_t* topk_idx,
                               uint32_t* status, cudaStream_t s) {
    const size_t smem = ts_smem_bytes(cfg);
    cudaError_t e = cudaFuncSetAttribute(topk_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_sample_kernel, dim3(cfg.n_req * rows), dim3(kTsThreads), smem, s, nullptr, 0, cfg,
                      scores, list, n_list, n_slots, rows, topk_idx, status);
}

}  // namespace spin

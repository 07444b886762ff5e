// spin_common.cuh -- device helpers shared by the SPIN kernels (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/spin.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "this library is written for sm_103a (GB300) only"
#endif

namespace spin {

constexpr int kBlock = 64;             // slots per logical KV block (one page)
constexpr int kMaxRows = 8;
constexpr int kSelectMaxBlocks = 16384;  // selection kernel keeps one key per block in smem

struct Dims {
    int32_t R, max_slots, max_rows, MB;
    int64_t DL;  // D length per request
};

__host__ __device__ inline Dims dims_of(const spin_config& c) {
    Dims d;
    d.R = c.n_req;
    d.max_slots = c.max_slots;
    d.max_rows = c.max_rows;
    d.MB = (c.max_slots + kBlock - 1) / kBlock;
    d.DL = (int64_t)c.max_slots + c.max_rows;
    return d;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

// Request-level checks shared by selection and the EMA update (reading R9 of the design):
// 0 <= N <= max_slots, N - 1 <= q, q + rows - 1 < max_slots + max_rows.
__device__ __forceinline__ uint32_t request_check(int64_t n, int64_t q, int rows, const Dims& d) {
    uint32_t bad = 0;
    if (n < 0 || n > d.max_slots) bad |= SPIN_STATUS_BAD_N;
    if (q < 0 || (n > 0 && q < n - 1) || q + rows - 1 >= d.DL) bad |= SPIN_STATUS_BAD_QPOS;
    return bad;
}

// Order-preserving map float -> uint32 (larger float -> larger key); -0 maps like +0.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7fffffffu) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------------------
// Temporal top-K hint (spin_topk_hint.cu).  Per (request, row) a record of kHintWords words:
// the guess (order key at or below the coming step's K-th score; 0 = none), the number of
// candidates the score kernel found at or above it, the rank margin of the next guess and
// counters of how the hinted top-K resolved its steps.  The candidates follow the records:
// cap entries per (request, row), each the slot's key in the high word and the complement
// of its list position (list entry * 64 + slot of the block) in the low word, so that the
// K largest entries are the top-K with equal keys taken in ascending position order.
// ---------------------------------------------------------------------------------------
constexpr int kHintWords = 16;
enum HintWord {
    kHwGuess = 0,    // order key of the normalised guess g (0: none, the next top-K takes the
                     // cold path); the score kernel's threshold is g * sum_h |w_h| of its step
    kHwCount = 1,    // candidates found by the score kernel (may exceed cap)
    kHwExtra = 2,    // ranks beyond K at which the next guess is taken (0: K / 2)
    kHwHit = 3,      // steps resolved from the candidates
    kHwMiss = 4,     // steps whose guess found fewer than K candidates
    kHwOver = 5,     // steps whose guess found more candidates than fit
    kHwCold = 6,     // steps without a guess
    kHwGlobal = 7,   // cold steps whose boundary bin did not fit: exact passes over the scores
    kHwLast = 8,     // the last step's candidate count
    kHwFlags = 9     // bit 0: this step's score kernel collected the candidates (else the
                     // top-K kernel collects them from the scores)
};

struct HintArgs {
    uint32_t* rec;              // [R * rows][kHintWords], NULL: no hint
    unsigned long long* cand;   // [R * rows][cap]
    int cap;
};

// Inverse of order_key (the float of a key; key 0x80000000 is +0).
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// sum_h |w_h| of one row's n head weights by one thread: four interleaved partial sums
// (h mod 4), so the loads of a row are in flight together; a fixed order for a given n.
__device__ __forceinline__ float row_wsum(const float* w, int n) {
    float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
    int h = 0;
#pragma unroll 4
    for (; h + 4 <= n; h += 4) {
        s0 = __fadd_rn(s0, fabsf(w[h]));
        s1 = __fadd_rn(s1, fabsf(w[h + 1]));
        s2 = __fadd_rn(s2, fabsf(w[h + 2]));
        s3 = __fadd_rn(s3, fabsf(w[h + 3]));
    }
    for (; h < n; ++h) s0 = __fadd_rn(s0, fabsf(w[h]));
    return __fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3));
}

// Threshold key of a row for this step: the normalised guess times the step's sum of |w_h|
// (the head weights move the scale of every score of a step together), 0 without a guess.
__device__ __forceinline__ uint32_t hint_threshold(uint32_t guess_word, float wsum) {
    if (guess_word == 0u) return 0u;
    const uint32_t k = order_key(__fmul_rn(key_float(guess_word), wsum));
    return k == 0u ? 1u : k;
}

__device__ __forceinline__ unsigned long long hint_entry(uint32_t key, uint32_t pos) {
    return ((unsigned long long)key << 32) | (unsigned long long)(~pos);
}

// Append one candidate with its own atomic (a few per cent of the slots reach the guess).
__device__ __forceinline__ void hint_push(const HintArgs& h, int64_t rr, uint32_t key, uint32_t pos) {
    const uint32_t at = atomicAdd(h.rec + rr * kHintWords + kHwCount, 1u);
    if (at < (uint32_t)h.cap) h.cand[rr * h.cap + at] = hint_entry(key, pos);
}

// ---------------------------------------------------------------------------------------
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2,
// 3", SC'11): ten rounds; each multiplies counter words 0 and 2 by the round multipliers,
// xors the high halves into words 1 and 3 together with the round key, and the key is
// advanced by the Weyl constants between rounds.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void philox4x64_10(uint64_t c[4], uint64_t k0, uint64_t k1) {
    const uint64_t kMul0 = 0xD2E7470EE14C6C93ull, kMul1 = 0xCA5A826395121157ull;
    const uint64_t kWeyl0 = 0x9E3779B97F4A7C15ull, kWeyl1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) { k0 += kWeyl0; k1 += kWeyl1; }
        const uint64_t lo0 = kMul0 * c[0], hi0 = __umul64hi(kMul0, c[0]);
        const uint64_t lo1 = kMul1 * c[2], hi1 = __umul64hi(kMul1, c[2]);
        const uint64_t n0 = hi1 ^ c[1] ^ k0;
        const uint64_t n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
    }
}

// Exploration draws: one Philox4x64-10 output (key {seed, layer}, counter {step, row, req, m})
// serves blocks 8m .. 8m+7; block 8m+h takes 32-bit half h, word h/2, high half first.
__device__ __forceinline__ void explore_keys8(uint64_t seed, int layer, uint64_t step, int row, int req,
                                              int64_t m, uint32_t (&out)[8]) {
    uint64_t c[4] = {step, (uint64_t)(uint32_t)row, (uint64_t)(uint32_t)req, (uint64_t)m};
    philox4x64_10(c, seed, (uint64_t)(uint32_t)layer);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        out[2 * w] = (uint32_t)(c[w] >> 32);
        out[2 * w + 1] = (uint32_t)(c[w] & 0xFFFFFFFFu);
    }
}

__device__ __forceinline__ uint32_t explore_key(uint64_t seed, int layer, uint64_t step, int row,
                                                int req, int64_t j) {
    uint32_t k8[8];
    explore_keys8(seed, layer, step, row, req, j >> 3, k8);
    return k8[j & 7];
}

// ---------------------------------------------------------------------------------------
// Warp / block reductions and scans.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Exclusive scan over the whole CTA (blockDim.x a multiple of 32, <= 1024).  `smem` holds
// 33 ints.  Returns the exclusive prefix; *total receives the block sum.
__device__ __forceinline__ int block_excl_scan(int v, int* smem, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int inc = warp_incl_scan(v);
    if (lane == 31) smem[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        int s = lane < nw ? smem[lane] : 0;
        int si = warp_incl_scan(s);
        if (lane < nw) smem[lane] = si - s;
        if (lane == 31) smem[32] = si;
    }
    __syncthreads();
    int res = smem[wid] + inc - v;
    *total = smem[32];
    __syncthreads();
    return res;
}

// ---------------------------------------------------------------------------------------
// Programmatic dependent launch (PTX ISA: griddepcontrol).  Every kernel of the library is
// launched with programmatic stream serialization allowed and begins with pdl_begin():
// the next kernel on the stream may be scheduled at once (its CTAs take free SM slots
// while this grid runs), and this grid waits, before any other instruction, until the
// previous grid on the stream has completed and its writes are visible.  So no memory
// access of a kernel overlaps its predecessor; only launch latency is hidden.  A kernel
// launched without the attribute passes both instructions at once.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Host side: launch `k` with programmatic stream serialization allowed, plus any extra
// launch attributes (a cluster shape).
template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              const cudaLaunchAttribute* extra, int n_extra, A&&... args) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute at[4];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    for (int i = 0; i < n_extra && i < 3; ++i) at[1 + i] = extra[i];
    lc.attrs = at;
    lc.numAttrs = 1 + (n_extra < 3 ? n_extra : 3);
    return [&](P... coerced) {
        void* pa[] = {const_cast<void*>(static_cast<const void*>(&coerced))...};
        return cudaLaunchKernelExC(&lc, reinterpret_cast<const void*>(k), pa);
    }(static_cast<A&&>(args)...);
}

// ---------------------------------------------------------------------------------------
// mbarrier and bulk-copy primitives (PTX ISA: mbarrier, cp.async.bulk).  Every wait is
// bounded: after kWaitLimitNs of global time it reports failure instead of spinning on.
// ---------------------------------------------------------------------------------------
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on phase `parity`.  Returns false if the limit passed or *abort was set.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u) {
            if (abort_flag && *abort_flag) return false;
            if (global_ns() - t0 > limit_ns) return false;
        }
    }
}

// Contiguous global -> shared copy by the bulk-copy (TMA) engine, completing on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns the OR of `pred` over the participating threads, so a
// group of warps takes the same branch afterwards.
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

}  // namespace spin

// spin_score_stream.cu -- indexer score with a key per head, on CUDA cores.
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention", §2 and Algorithm 1's scoring step:
// z_t[i] = sum_h w_h ReLU(q_{t,h} . k_{i,h}), run only over the slots of the selected
// blocks, read through the paged block table.
//
// With a key per head the work per slot is n_h independent d-long dot products: a batched
// GEMV at about 1 FLOP per key byte, so the kernel is bound by HBM, not by arithmetic,
// and the tensor cores are not used.  Design:
//   * persistent CTAs, each owning a contiguous range of (request, list entry, slot group)
//     chunks; one producer warp streams S-slot chunks of a page (contiguous in the pool)
//     into an NST-deep shared-memory ring with the bulk-copy engine (cp.async.bulk +
//     mbarrier transaction counts), so memory parallelism does not depend on registers;
//   * W consumer warps, each owning a fixed group of n_h/W heads for every slot, keep
//     their heads' query values and weights in registers; a lane covers 16-byte chunks of
//     its heads' keys, the d-long dot is reduced over the d*elt/16 lanes that share a
//     head with xor shuffles, and ReLU(s_i dot) w_h is summed over the warp's heads;
//   * the W per-warp partial sums of a slot are added in a fixed order (deterministic).
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "spin_common.cuh"
#include "spin_internal.h"

namespace spin {

constexpr int kMaxReqStream = 2048;

struct KF32 { static constexpr int kElt = 4; static constexpr int kDtype = SPIN_DTYPE_F32; };
struct KBF16 { static constexpr int kElt = 2; static constexpr int kDtype = SPIN_DTYPE_BF16; };
struct KE4M3 { static constexpr int kElt = 1; static constexpr int kDtype = SPIN_DTYPE_E4M3; };

// Expand a 16-byte chunk of keys into floats and dot it with q (EPC values).
template <class K>
__device__ __forceinline__ float chunk_dot(const uint4& kv, const float* q);

template <>
__device__ __forceinline__ float chunk_dot<KF32>(const uint4& kv, const float* q) {
    float acc = __uint_as_float(kv.x) * q[0];
    acc = fmaf(__uint_as_float(kv.y), q[1], acc);
    acc = fmaf(__uint_as_float(kv.z), q[2], acc);
    acc = fmaf(__uint_as_float(kv.w), q[3], acc);
    return acc;
}

template <>
__device__ __forceinline__ float chunk_dot<KBF16>(const uint4& kv, const float* q) {
    const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        acc = fmaf(__uint_as_float(w[j] << 16), q[2 * j], acc);
        acc = fmaf(__uint_as_float(w[j] & 0xffff0000u), q[2 * j + 1], acc);
    }
    return acc;
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two_codes, __NV_E4M3);
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

template <>
__device__ __forceinline__ float chunk_dot<KE4M3>(const uint4& kv, const float* q) {
    const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 a = e4m3x2_to_float2(w[j] & 0xffffu);
        const float2 b = e4m3x2_to_float2(w[j] >> 16);
        acc = fmaf(a.x, q[4 * j + 0], acc);
        acc = fmaf(a.y, q[4 * j + 1], acc);
        acc = fmaf(b.x, q[4 * j + 2], acc);
        acc = fmaf(b.y, q[4 * j + 3], acc);
    }
    return acc;
}

template <class K, int NH, int D, int W, int MAXR>
struct StreamCfg {
    static constexpr int kElt = K::kElt;
    static constexpr int kSlotBytes = NH * D * kElt;
    static constexpr int kRegionBytes = kSlotBytes / W;         // one warp's heads of a slot
    static constexpr int kU = kRegionBytes / 512;               // 16-byte chunks per lane per slot
    static constexpr int kEPC = 16 / kElt;                      // elements per chunk
    static constexpr int kLPH = D * kElt / 16;                  // lanes sharing a head
    static constexpr int kHPW = NH / W;                         // heads per warp
    static constexpr int kS = (32768 / kSlotBytes) < 1 ? 1 : (32768 / kSlotBytes);  // slots per stage
    static constexpr int kGroups = kBlock / kS;                 // stages per page
    static constexpr int kNST = 3;                              // ring depth
    static constexpr int kStageBytes = kS * kSlotBytes;
    static constexpr int kScaleBytes = (K::kDtype == SPIN_DTYPE_E4M3) ? kS * 4 : 0;
    static constexpr int kThreads = (W + 1) * 32;
    static_assert(kSlotBytes % (W * 512) == 0, "a warp must cover whole 512-byte rows");
    static_assert(32 % kLPH == 0 && kLPH >= 1, "lanes per head must divide the warp");
    static_assert(NH % W == 0, "heads split evenly over warps");
    static_assert(kBlock % kS == 0, "stages tile a page");
    static_assert(kScaleBytes % 16 == 0, "bulk copies move multiples of 16 bytes");
};

struct StreamSmemHeader {
    uint64_t full[4];
    uint64_t empty[4];
    int abort_flag;
    int total_chunks;
};

template <class K, int NH, int D, int W, int MAXR>
__global__ void __launch_bounds__(StreamCfg<K, NH, D, W, MAXR>::kThreads)
score_stream_kernel(spin_config cfg, ScoreArgs a) {
    pdl_begin();
    using C = StreamCfg<K, NH, D, W, MAXR>;
    extern __shared__ __align__(128) unsigned char smem[];
    const Dims dm = dims_of(cfg);
    StreamSmemHeader* hdr = reinterpret_cast<StreamSmemHeader*>(smem);
    int* prefix = reinterpret_cast<int*>(smem + 128);                                  // [R + 1]
    const size_t prefix_bytes = (((size_t)(dm.R + 1) * 4) + 127) & ~(size_t)127;
    unsigned char* stage_base = smem + 128 + prefix_bytes;                             // NST stages
    float* stage_scale = reinterpret_cast<float*>(stage_base + (size_t)C::kNST * C::kStageBytes);
    float* zpart = stage_scale + C::kNST * (C::kScaleBytes / 4);                       // [NST][S][W][MAXR]

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int rows = a.rows;

    // per-request chunk counts -> prefix sums (warp 0)
    if (wid == 0) {
        int carry = 0;
        for (int base = 0; base < dm.R; base += 32) {
            const int r = base + lane;
            int c = 0;
            if (r < dm.R) {
                const int64_t n = a.n_slots[r], cnt = a.n_list[r];
                const bool ok = n >= 0 && n <= dm.max_slots && cnt >= 0 && cnt <= dm.MB;
                if (!ok && blockIdx.x == 0)
                    set_status(a.status, (n < 0 || n > dm.max_slots) ? SPIN_STATUS_BAD_N : SPIN_STATUS_BAD_LIST);
                c = ok ? (int)cnt * C::kGroups : 0;
            }
            const int inc = warp_incl_scan(c);
            if (r < dm.R) prefix[r] = carry + inc - c;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) {
            prefix[dm.R] = carry;
            hdr->total_chunks = carry;
            hdr->abort_flag = 0;
            for (int s = 0; s < C::kNST; ++s) {
                mbar_init(&hdr->full[s], 1);
                mbar_init(&hdr->empty[s], W);
            }
            fence_barrier_init();
        }
    }
    __syncthreads();
    const int total = hdr->total_chunks;
    const int c0 = (int)(((int64_t)total * blockIdx.x) / gridDim.x);
    const int c1 = (int)(((int64_t)total * (blockIdx.x + 1)) / gridDim.x);

    // chunk -> (req, list entry, group, page or -1)
    auto decode = [&](int ch, int& req, int& k, int& g, int64_t& page) {
        int lo = 0, hi = dm.R - 1;
        while (lo < hi) {  // last r with prefix[r] <= ch
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= ch) lo = mid; else hi = mid - 1;
        }
        req = lo;
        const int local = ch - prefix[req];
        k = local / C::kGroups;
        g = local - k * C::kGroups;
        const int64_t n = a.n_slots[req];
        const int64_t nb = (n + kBlock - 1) / kBlock;
        const int64_t blk = a.list[(int64_t)req * dm.MB + k];
        page = -1;
        if (blk >= 0 && blk < nb) {
            const int64_t p = a.block_table[(int64_t)req * a.bt_stride + blk];
            if (p >= 0 && p < a.n_pages) page = p;
        }
    };

    if (wid == W) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            int last_phase[C::kNST];
            for (int st = 0; st < C::kNST; ++st) last_phase[st] = -1;
            for (int ch = c0, it = 0; ch < c1; ++ch, ++it) {
                const int st = it % C::kNST;
                const uint32_t ph = (uint32_t)(it / C::kNST) & 1u;
                if (!mbar_wait(&hdr->empty[st], ph ^ 1u, &hdr->abort_flag)) {
                    hdr->abort_flag = 1;
                    set_status(a.status, SPIN_STATUS_TIMEOUT);
                    break;
                }
                int req, k, g;
                int64_t page;
                decode(ch, req, k, g, page);
                if (page >= 0) {
                    const unsigned char* src = reinterpret_cast<const unsigned char*>(a.k_pool) +
                                               ((size_t)page * kBlock + (size_t)g * C::kS) * C::kSlotBytes;
                    mbar_arrive_expect_tx(&hdr->full[st], C::kStageBytes + C::kScaleBytes);
                    bulk_g2s(stage_base + (size_t)st * C::kStageBytes, src, C::kStageBytes, &hdr->full[st]);
                    if (C::kScaleBytes)
                        bulk_g2s(stage_scale + st * (C::kScaleBytes / 4), a.k_scale + page * kBlock + g * C::kS,
                                 C::kScaleBytes, &hdr->full[st]);
                } else {
                    mbar_arrive(&hdr->full[st]);
                }
                last_phase[st] = (int)ph;
            }
            // never leave with copies in flight: wait (bounded) for the last fill of each stage
            for (int st = 0; st < C::kNST; ++st)
                if (last_phase[st] >= 0 && !mbar_wait(&hdr->full[st], (uint32_t)last_phase[st], nullptr))
                    set_status(a.status, SPIN_STATUS_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------------ consumers
        // registers: this lane's query values and head weights, refreshed per request
        float qreg[MAXR][C::kU][C::kEPC];
        float wreg[MAXR][C::kU];
        int cur_req = -1;
        int h_req = -1;        // hinted top-K: request of the cached threshold of this thread's row
        uint32_t h_thr = 0u;
        for (int ch = c0, it = 0; ch < c1; ++ch, ++it) {
            const int st = it % C::kNST;
            const uint32_t ph = (uint32_t)(it / C::kNST) & 1u;
            int req, k, g;
            int64_t page;
            decode(ch, req, k, g, page);
            if (req != cur_req) {
                cur_req = req;
#pragma unroll
                for (int r = 0; r < MAXR; ++r)
#pragma unroll
                    for (int u = 0; u < C::kU; ++u) {
                        const int cidx = u * 32 + lane;
                        const int head = wid * C::kHPW + cidx / C::kLPH;
                        const int dim0 = (cidx % C::kLPH) * C::kEPC;
                        const bool live = r < rows;
                        const int64_t qoff = (((int64_t)req * rows + (live ? r : 0)) * NH + head) * D + dim0;
#pragma unroll
                        for (int e = 0; e < C::kEPC; ++e) {
                            float v;
                            if (cfg.q_dtype == SPIN_DTYPE_BF16)
                                v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.q)[qoff + e]);
                            else
                                v = reinterpret_cast<const float*>(a.q)[qoff + e];
                            qreg[r][u][e] = live ? v : 0.0f;
                        }
                        wreg[r][u] = live ? a.w[((int64_t)req * rows + r) * NH + head] : 0.0f;
                    }
            }
            const bool ok = mbar_wait(&hdr->full[st], ph, &hdr->abort_flag);
            if (!ok) {
                hdr->abort_flag = 1;
                set_status(a.status, SPIN_STATUS_TIMEOUT);
            }
            if (page < 0 && wid == 0 && lane == 0) {
                const int64_t nb = (a.n_slots[req] + kBlock - 1) / kBlock;
                const int64_t blk = a.list[(int64_t)req * dm.MB + k];
                set_status(a.status, (blk >= 0 && blk < nb) ? SPIN_STATUS_BAD_PAGE : SPIN_STATUS_BAD_LIST);
            }
            float* zp = zpart + (size_t)st * C::kS * W * MAXR;
            if (ok && page >= 0) {
                const unsigned char* sbuf = stage_base + (size_t)st * C::kStageBytes;
                for (int s = 0; s < C::kS; ++s) {
                    const float scale = C::kScaleBytes ? stage_scale[st * (C::kScaleBytes / 4) + s] : 1.0f;
                    const uint4* src = reinterpret_cast<const uint4*>(sbuf + (size_t)s * C::kSlotBytes +
                                                                      (size_t)wid * C::kRegionBytes);
                    float acc[MAXR];
#pragma unroll
                    for (int r = 0; r < MAXR; ++r) acc[r] = 0.0f;
#pragma unroll
                    for (int u = 0; u < C::kU; ++u) {
                        const uint4 kv = src[u * 32 + lane];
#pragma unroll
                        for (int r = 0; r < MAXR; ++r) {
                            float dot = chunk_dot<K>(kv, qreg[r][u]);
#pragma unroll
                            for (int o = 1; o < C::kLPH; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                            const float x = scale * dot;
                            acc[r] = fmaf(wreg[r][u], x > 0.0f ? x : 0.0f, acc[r]);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < MAXR; ++r) {
#pragma unroll
                        for (int o = C::kLPH; o < 32; o <<= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
                    }
                    if (lane == 0) {
#pragma unroll
                        for (int r = 0; r < MAXR; ++r) zp[(s * W + wid) * MAXR + r] = acc[r];
                    }
                }
            }
            // every consumer warp leaves the loop at the same iteration if any wait failed
            const bool fail = named_barrier_or(1, W * 32, !ok);
            __syncwarp();
            if (lane == 0) mbar_arrive(&hdr->empty[st]);
            // fixed-order sum of the W partials, masked to i < N
            const int64_t n = a.n_slots[req];
            for (int t = tid; t < C::kS * rows; t += W * 32) {
                const int s = t / rows, r = t - s * rows;
                float z = 0.0f;
                if (!fail && page >= 0) {
                    for (int ww = 0; ww < W; ++ww) z += zp[(s * W + ww) * MAXR + r];
                }
                const int64_t blk = a.list[(int64_t)req * dm.MB + k];
                const int64_t i = blk * kBlock + (int64_t)g * C::kS + s;
                if (i >= n || z == 0.0f) z = 0.0f;
                a.scores[(((int64_t)req * rows + r) * dm.MB + k) * kBlock + g * C::kS + s] = z;
                // hinted top-K: a live slot (valid block, i < N) at or above its row's threshold
                if (a.hint.rec && blk >= 0 && blk * kBlock < n && i < n) {
                    const int64_t rr = (int64_t)req * rows + r;
                    if (req != h_req) {  // this thread's row r of a new request
                        h_req = req;
                        h_thr = hint_threshold(a.hint.rec[rr * kHintWords + kHwGuess], row_wsum(a.w + rr * NH, NH));
                        a.hint.rec[rr * kHintWords + kHwFlags] = 1u;  // (every writer stores the same value)
                    }
                    const uint32_t key = order_key(z);
                    if (h_thr != 0u && key >= h_thr) hint_push(a.hint, rr, key, (uint32_t)(k * kBlock + g * C::kS + s));
                }
            }
            if (fail) break;
        }
    }
}

template <class K, int NH, int D, int W, int MAXR>
static cudaError_t launch_stream_inst(const spin_config& cfg, const ScoreArgs& a, cudaStream_t s) {
    using C = StreamCfg<K, NH, D, W, MAXR>;
    const Dims dm = dims_of(cfg);
    const size_t prefix_bytes = (((size_t)(dm.R + 1) * 4) + 127) & ~(size_t)127;
    const size_t smem = 128 + prefix_bytes + (size_t)C::kNST * C::kStageBytes + (size_t)C::kNST * C::kScaleBytes +
                        sizeof(float) * (size_t)C::kNST * C::kS * W * MAXR;
    auto kern = score_stream_kernel<K, NH, D, W, MAXR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t max_chunks = (int64_t)dm.R * dm.MB * C::kGroups;
    int64_t grid = (int64_t)device_sm_count() * per_sm;
    if (grid > max_chunks) grid = max_chunks;
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(C::kThreads), smem, s, nullptr, 0, cfg, a);
}

bool score_stream_supported(const spin_config& cfg, int rows) {
    if (cfg.kv_heads != cfg.n_heads || cfg.n_req > kMaxReqStream) return false;
    const int H = cfg.n_heads, d = cfg.head_dim;
    if (cfg.k_dtype == SPIN_DTYPE_F32 && cfg.q_dtype == SPIN_DTYPE_F32 && H == 8 && d == 64) return rows <= 1;
    if (cfg.q_dtype == SPIN_DTYPE_BF16 && H == 64 && d == 128 &&
        (cfg.k_dtype == SPIN_DTYPE_BF16 || cfg.k_dtype == SPIN_DTYPE_E4M3))
        return rows <= 1;
    return false;
}

cudaError_t launch_score_stream(const spin_config& cfg, const ScoreArgs& a, cudaStream_t s) {
    if (!score_stream_supported(cfg, a.rows)) return cudaErrorNotSupported;
    if (cfg.k_dtype == SPIN_DTYPE_F32) return launch_stream_inst<KF32, 8, 64, 4, 1>(cfg, a, s);
    if (cfg.k_dtype == SPIN_DTYPE_BF16) return launch_stream_inst<KBF16, 64, 128, 8, 1>(cfg, a, s);
    return launch_stream_inst<KE4M3, 64, 128, 8, 1>(cfg, a, s);
}

}  // namespace spin

// spin_score_tc.cu -- indexer score with one key shared by all heads, on tcgen05 tensor
// cores (sm_103a).
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention", §2 and Algorithm 1 line 6:
// z_t[i] = sum_h w_h ReLU(q_{t,h} . k_i) over the slots of the selected blocks only.
// With one key per slot shared by the n_h heads (and, for speculative decoding, by the
// rows' queries), the per-tile work is a dense contraction
//     D[slot][row*n_h + h] = sum_c K[slot][c] * Q[row*n_h + h][c]
// of a 128-slot tile (two selected pages) with the 64*rows query vectors, so it runs on
// the tensor cores: M = 128 slots, N = 64*rows, K = d = 128, fp32 accumulation in TMEM.
//
// Warp roles of a persistent CTA (tiles = pairs of selected blocks of one request):
//   warp 0      producer: bf16 keys -> two 2D TMA loads per page straight into the
//               128-byte-swizzled K-major operand layout; FP8 keys -> one bulk copy per
//               page into a raw staging ring
//   warp 1      TMEM owner and MMA issuer (one thread): 8 tcgen05.mma of K = 16 per
//               tile, commits to the operand-release and accumulator-full barriers;
//               stages q (and converts it to f16 for FP8 keys) when the request changes
//   warps 2-5   epilogue: tcgen05.ld of the tile's accumulators (one slot per thread),
//               z = s_i * sum_h w_h max(acc_h, 0) per row, masked to i < N, stored
//   warps 6-9   (FP8 keys only) converters: e4m3 -> f16 (exact) from the raw ring into
//               the swizzled operand layout
// Accumulators are double-buffered in TMEM so the epilogue of tile t overlaps the MMAs
// of tile t+1; every barrier wait is bounded and a timeout unwinds all roles.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "spin_common.cuh"
#include "spin_internal.h"

namespace spin {

constexpr int kTcD = 128;      // head dim (K of the contraction)
constexpr int kTcNH = 64;      // heads
constexpr int kTcM = 128;      // slots per tile (two pages)
constexpr int kTcMaxRows = 4;  // N = 64 * rows <= 256
constexpr int kTcMaxReq = 2048;
constexpr int kTcRegionBytes = kTcM * 128;          // one 64-element K half of a 128-slot tile
constexpr int kTcABytes = 2 * kTcRegionBytes;       // 32 KB operand tile (16-bit elements)
constexpr int kTcRawBytes = 2 * kBlock * kTcD;      // 16 KB: two FP8 pages
constexpr int kTcStagesBf16 = 3;
constexpr int kTcRawStages = 4;
constexpr int kTcAStagesFp8 = 2;

// ------------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 128-byte-swizzle K-major shared-memory matrix descriptor (tcgen05 matrix descriptor):
// start address >> 4, leading byte offset 16 (unused with this swizzle), stride byte
// offset 1024 (8 rows of 128 bytes), version 1, swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B both f16 (fmt 0) or both
// bf16 (fmt 1), both K-major, N >> 3 and M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t ab_fmt, uint32_t n, uint32_t m) {
    return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Byte offset of element c (0..127) of operand row m inside a [rows][128 x 16-bit] K-major
// tile stored as two 128-byte-swizzled regions of region_bytes each.
__device__ __forceinline__ uint32_t sw128_offset(int m, int c, int region_bytes) {
    const int kh = c >> 6, ch = (c & 63) >> 3;
    return (uint32_t)(kh * region_bytes + (m >> 3) * 1024 + (m & 7) * 128 + ((ch ^ (m & 7)) << 4) + (c & 7) * 2);
}

struct TcHdr {
    uint64_t full[kTcRawStages];     // producer -> consumer of a loaded stage
    uint64_t empty[kTcRawStages];    // stage released back to the producer
    uint64_t afull[kTcAStagesFp8];   // FP8: converted operand ready
    uint64_t aempty[kTcAStagesFp8];  // FP8: converted operand consumed by the MMAs
    uint64_t tfull[2];               // accumulator ready
    uint64_t tempty[2];              // accumulator drained by the epilogue
    uint64_t qdone;                  // every issued MMA finished (before q is restaged)
    uint32_t tmem_base;
    int abort_flag;
    int total_tiles;
};

struct TcLayout {
    uint32_t prefix, stage_a, raw, qbuf, wbuf, total;
};

__host__ __device__ inline TcLayout tc_layout(int R, int rows, bool fp8) {
    TcLayout L;
    uint32_t off = 1024;  // header
    L.prefix = off;
    off += ((uint32_t)(R + 1) * 4 + 1023) & ~1023u;
    L.stage_a = off;
    off += (fp8 ? kTcAStagesFp8 : kTcStagesBf16) * kTcABytes;
    L.raw = off;
    if (fp8) off += kTcRawStages * kTcRawBytes;
    L.qbuf = off;
    off += (uint32_t)(64 * rows) * 256;  // two 128-byte regions of N rows
    L.wbuf = off;
    off += 4u * 64 * rows * 4;           // a copy of w per epilogue warp
    L.total = off + 1024;                // slack for 1024-byte alignment of the base
    return L;
}

template <bool FP8>
__global__ void __launch_bounds__(FP8 ? 320 : 192, 1)
score_tc_kernel(spin_config cfg, ScoreArgs a, const __grid_constant__ CUtensorMap kmap) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Dims dm = dims_of(cfg);
    const int rows = a.rows;
    const int N = kTcNH * rows;
    const TcLayout L = tc_layout(dm.R, rows, FP8);
    TcHdr* hdr = reinterpret_cast<TcHdr*>(smem);
    int* prefix = reinterpret_cast<int*>(smem + L.prefix);
    unsigned char* sA = smem + L.stage_a;
    unsigned char* sRaw = smem + L.raw;
    unsigned char* sQ = smem + L.qbuf;
    float* sW = reinterpret_cast<float*>(smem + L.wbuf);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    constexpr int NSA = FP8 ? kTcAStagesFp8 : kTcStagesBf16;  // operand stages
    constexpr int NSL = FP8 ? kTcRawStages : kTcStagesBf16;   // load stages
    const uint32_t tmem_cols = N <= 64 ? 128u : (N <= 128 ? 256u : 512u);

    // ------------------------------------------------------------------ set-up
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
                c = ok ? (int)((cnt + 1) / 2) : 0;
            }
            const int inc = warp_incl_scan(c);
            if (r < dm.R) prefix[r] = carry + inc - c;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) {
            prefix[dm.R] = carry;
            hdr->total_tiles = carry;
            hdr->abort_flag = 0;
            for (int s = 0; s < NSL; ++s) {
                mbar_init(&hdr->full[s], 1);
                mbar_init(&hdr->empty[s], FP8 ? 128 : 1);
            }
            for (int s = 0; s < kTcAStagesFp8; ++s) {
                mbar_init(&hdr->afull[s], 128);
                mbar_init(&hdr->aempty[s], 1);
            }
            for (int s = 0; s < 2; ++s) {
                mbar_init(&hdr->tfull[s], 1);
                mbar_init(&hdr->tempty[s], 128);
            }
            mbar_init(&hdr->qdone, 1);
            fence_barrier_init();
        }
    } else if (wid == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&hdr->tmem_base)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = hdr->tmem_base;
    const int total = hdr->total_tiles;
    const int t0 = (int)(((int64_t)total * blockIdx.x) / gridDim.x);
    const int t1 = (int)(((int64_t)total * (blockIdx.x + 1)) / gridDim.x);

    // tile -> request, first list entry, and the two pages (or -1)
    auto decode = [&](int t, int& req, int& k0, int64_t* page, int64_t* blk) {
        int lo = 0, hi = dm.R - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
        }
        req = lo;
        k0 = 2 * (t - prefix[req]);
        const int64_t n = a.n_slots[req], cnt = a.n_list[req];
        const int64_t nb = (n + kBlock - 1) / kBlock;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            page[h] = -1;
            blk[h] = -1;
            const int64_t k = k0 + h;
            if (k < cnt) {
                const int64_t b = a.list[(int64_t)req * dm.MB + k];
                blk[h] = b;
                if (b >= 0 && b < nb) {
                    const int64_t p = a.block_table[(int64_t)req * a.bt_stride + b];
                    if (p >= 0 && p < a.n_pages) page[h] = p;
                }
            }
        }
    };
    auto fail_wait = [&]() {
        hdr->abort_flag = 1;
        set_status(a.status, SPIN_STATUS_TIMEOUT);
    };

    if (wid == 0) {
        // -------------------------------------------------------------- producer
        if (lane == 0) {
            int last_phase[NSL];
            for (int s = 0; s < NSL; ++s) last_phase[s] = -1;
            for (int t = t0, it = 0; t < t1; ++t, ++it) {
                const int s = it % NSL;
                const uint32_t ph = (uint32_t)(it / NSL) & 1u;
                if (!mbar_wait(&hdr->empty[s], ph ^ 1u, &hdr->abort_flag)) { fail_wait(); break; }
                int req, k0;
                int64_t page[2], blk[2];
                decode(t, req, k0, page, blk);
                uint32_t bytes = 0;
                for (int h = 0; h < 2; ++h)
                    if (page[h] >= 0) bytes += FP8 ? (uint32_t)(kBlock * kTcD) : (uint32_t)(2 * 8192);
                if (bytes == 0) {
                    mbar_arrive(&hdr->full[s]);
                } else {
                    mbar_arrive_expect_tx(&hdr->full[s], bytes);
                    for (int h = 0; h < 2; ++h) {
                        if (page[h] < 0) continue;
                        if (FP8) {
                            const unsigned char* src =
                                reinterpret_cast<const unsigned char*>(a.k_pool) + (size_t)page[h] * kBlock * kTcD;
                            bulk_g2s(sRaw + (size_t)s * kTcRawBytes + h * kBlock * kTcD, src, kBlock * kTcD,
                                     &hdr->full[s]);
                        } else {
                            unsigned char* dst = sA + (size_t)s * kTcABytes + h * 8192;
                            const int y = (int)(page[h] * kBlock);
                            tma_load_2d(dst, &kmap, 0, y, &hdr->full[s]);
                            tma_load_2d(dst + kTcRegionBytes, &kmap, 64, y, &hdr->full[s]);
                        }
                    }
                }
                last_phase[s] = (int)ph;
            }
            for (int s = 0; s < NSL; ++s)
                if (last_phase[s] >= 0 && !mbar_wait(&hdr->full[s], (uint32_t)last_phase[s], nullptr))
                    set_status(a.status, SPIN_STATUS_TIMEOUT);
        }
    } else if (wid == 1) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc = idesc_f16(FP8 ? 0u : 1u, (uint32_t)N, (uint32_t)kTcM);
        int cur_req = -1;
        uint32_t qphase = 0;
        bool issued_any = false;
        for (int t = t0, it = 0; t < t1; ++t, ++it) {
            int req, k0;
            int64_t page[2], blk[2];
            decode(t, req, k0, page, blk);
            if (req != cur_req) {
                if (issued_any) {  // the MMAs of the previous request still read sQ
                    if (lane == 0) tc_commit(&hdr->qdone);
                    __syncwarp();
                    if (!mbar_wait(&hdr->qdone, qphase, &hdr->abort_flag)) { fail_wait(); break; }
                    qphase ^= 1u;
                }
                // stage q[req] (rows x 64 heads x 128 dims) as the K-major B operand
                const int nchunks = N * (kTcD / 8);
                for (int ci = lane; ci < nchunks; ci += 32) {
                    const int nrow = ci / (kTcD / 8), c0 = (ci % (kTcD / 8)) * 8;
                    const int r = nrow / kTcNH, h = nrow % kTcNH;
                    const int64_t qoff = (((int64_t)req * rows + r) * kTcNH + h) * kTcD + c0;
                    uint32_t wv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float f0, f1;
                        if (cfg.q_dtype == SPIN_DTYPE_BF16) {
                            const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(a.q) + qoff;
                            f0 = __bfloat162float(qb[2 * e]);
                            f1 = __bfloat162float(qb[2 * e + 1]);
                        } else {
                            const float* qf = reinterpret_cast<const float*>(a.q) + qoff;
                            f0 = qf[2 * e];
                            f1 = qf[2 * e + 1];
                        }
                        if (FP8) {
                            __half2 hv = __floats2half2_rn(f0, f1);
                            wv[e] = *reinterpret_cast<uint32_t*>(&hv);
                        } else {
                            __nv_bfloat162 bv = __floats2bfloat162_rn(f0, f1);
                            wv[e] = *reinterpret_cast<uint32_t*>(&bv);
                        }
                    }
                    *reinterpret_cast<uint4*>(sQ + sw128_offset(nrow, c0, N * 128)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                fence_async_smem();
                __syncwarp();
                cur_req = req;
            }
            const int sa = it % NSA;
            const uint32_t pha = (uint32_t)(it / NSA) & 1u;
            bool ok = FP8 ? mbar_wait(&hdr->afull[sa], pha, &hdr->abort_flag)
                          : mbar_wait(&hdr->full[sa], pha, &hdr->abort_flag);
            const int acc = it & 1;
            const uint32_t phc = (uint32_t)(it >> 1) & 1u;
            if (ok) ok = mbar_wait(&hdr->tempty[acc], phc ^ 1u, &hdr->abort_flag);
            if (!ok) { fail_wait(); break; }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t a_base = smem_u32(sA + (size_t)sa * kTcABytes);
                const uint32_t b_base = smem_u32(sQ);
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * N);
#pragma unroll
                for (int kh = 0; kh < 2; ++kh)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t adesc = smem_desc_sw128(a_base + kh * kTcRegionBytes + kk * 32);
                        const uint64_t bdesc = smem_desc_sw128(b_base + kh * (N * 128) + kk * 32);
                        tc_mma(d_tmem, adesc, bdesc, idesc, (kh | kk) ? 1u : 0u);
                    }
                tc_commit(FP8 ? &hdr->aempty[sa] : &hdr->empty[sa]);
                tc_commit(&hdr->tfull[acc]);
            }
            issued_any = true;
            __syncwarp();
        }
        // every issued MMA has finished before TMEM is released
        if (issued_any) {
            if (lane == 0) tc_commit(&hdr->qdone);
            __syncwarp();
            if (!mbar_wait(&hdr->qdone, qphase, nullptr)) set_status(a.status, SPIN_STATUS_TIMEOUT);
        }
    } else if (wid < 6) {
        // ------------------------------------------------------------- epilogue
        const int quarter = wid & 3;
        const int m = quarter * 32 + lane;      // slot row of the tile = TMEM lane
        const int h = m >> 6, s = m & 63;
        float* wloc = sW + (size_t)(wid - 2) * N;
        int cur_req = -1;
        for (int t = t0, it = 0; t < t1; ++t, ++it) {
            int req, k0;
            int64_t page[2], blk[2];
            decode(t, req, k0, page, blk);
            if (req != cur_req) {
                __syncwarp();
                for (int i = lane; i < N; i += 32) wloc[i] = a.w[(int64_t)req * rows * kTcNH + i];
                __syncwarp();
                cur_req = req;
            }
            const int acc = it & 1;
            const uint32_t phc = (uint32_t)(it >> 1) & 1u;
            if (!mbar_wait(&hdr->tfull[acc], phc, &hdr->abort_flag)) { fail_wait(); break; }
            tc_fence_after();
            const int64_t k = k0 + h;
            const int64_t n = a.n_slots[req];
            const bool listed = k < a.n_list[req];                      // a real list entry
            const bool live = page[h] >= 0 && blk[h] * kBlock + s < n;  // a slot of the context
            const float scale = (FP8 && page[h] >= 0) ? a.k_scale[page[h] * kBlock + s] : 1.0f;
            if (page[h] < 0 && blk[h] >= 0 && s == 0) {
                const int64_t nb = (n + kBlock - 1) / kBlock;
                set_status(a.status, (blk[h] < nb) ? SPIN_STATUS_BAD_PAGE : SPIN_STATUS_BAD_LIST);
            }
            for (int r = 0; r < rows; ++r) {
                float z = 0.0f;
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    float v[32];
                    const uint32_t taddr =
                        tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * N + r * kTcNH + cb * 32);
                    tc_ld32(taddr, v);
                    const float* wr = wloc + r * kTcNH + cb * 32;
#pragma unroll
                    for (int j = 0; j < 32; ++j) z = fmaf(wr[j], fmaxf(scale * v[j], 0.0f), z);
                }
                if (!live || z == 0.0f) z = 0.0f;
                if (listed) a.scores[(((int64_t)req * rows + r) * dm.MB + k) * kBlock + s] = z;
            }
            tc_fence_before();
            mbar_arrive(&hdr->tempty[acc]);
        }
    } else {
        // ------------------------------------------------------- FP8 converters
        if (FP8) {
            const int ct = tid - 192;  // 0..127
            for (int t = t0, it = 0; t < t1; ++t, ++it) {
                const int rs = it % kTcRawStages;
                const uint32_t phr = (uint32_t)(it / kTcRawStages) & 1u;
                const int sa = it % kTcAStagesFp8;
                const uint32_t pha = (uint32_t)(it / kTcAStagesFp8) & 1u;
                if (!mbar_wait(&hdr->full[rs], phr, &hdr->abort_flag)) { fail_wait(); break; }
                if (!mbar_wait(&hdr->aempty[sa], pha ^ 1u, &hdr->abort_flag)) { fail_wait(); break; }
                int req, k0;
                int64_t page[2], blk[2];
                decode(t, req, k0, page, blk);
                const unsigned char* raw = sRaw + (size_t)rs * kTcRawBytes;
                unsigned char* dstA = sA + (size_t)sa * kTcABytes;
                for (int idx = ct; idx < kTcM * (kTcD / 8); idx += 128) {
                    const int mm = idx >> 4, cc = idx & 15;
                    if (page[mm >> 6] < 0) continue;
                    const uint2 codes = *reinterpret_cast<const uint2*>(raw + mm * kTcD + cc * 8);
                    uint32_t hv[4];
                    const uint32_t cw[2] = {codes.x, codes.y};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(cw[e] & 0xffffu), __NV_E4M3);
                        __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(cw[e] >> 16), __NV_E4M3);
                        hv[2 * e] = (uint32_t)lo.x | ((uint32_t)lo.y << 16);
                        hv[2 * e + 1] = (uint32_t)hi.x | ((uint32_t)hi.y << 16);
                    }
                    *reinterpret_cast<uint4*>(dstA + sw128_offset(mm, cc * 8, kTcRegionBytes)) =
                        make_uint4(hv[0], hv[1], hv[2], hv[3]);
                }
                fence_async_smem();
                mbar_arrive(&hdr->afull[sa]);
                mbar_arrive(&hdr->empty[rs]);
            }
        }
    }

    // ------------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (wid == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(tmem_cols)
                     : "memory");
    }
}

// ------------------------------------------------------------------------------ host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool score_tc_supported(const spin_config& cfg, int rows) {
    return cfg.kv_heads == 1 && cfg.n_heads == kTcNH && cfg.head_dim == kTcD && rows >= 1 && rows <= kTcMaxRows &&
           cfg.n_req <= kTcMaxReq && cfg.q_dtype == SPIN_DTYPE_BF16 &&
           (cfg.k_dtype == SPIN_DTYPE_BF16 || cfg.k_dtype == SPIN_DTYPE_E4M3);
}

cudaError_t launch_score_tc(const spin_config& cfg, const ScoreArgs& a, cudaStream_t s) {
    if (!score_tc_supported(cfg, a.rows)) return cudaErrorNotSupported;
    const Dims dm = dims_of(cfg);
    const bool fp8 = cfg.k_dtype == SPIN_DTYPE_E4M3;
    const TcLayout L = tc_layout(dm.R, a.rows, fp8);
    CUtensorMap map;
    memset(&map, 0, sizeof map);
    if (!fp8) {
        EncodeTiledFn enc = encode_fn();
        if (!enc) return cudaErrorNotSupported;
        const cuuint64_t gdim[2] = {(cuuint64_t)kTcD, (cuuint64_t)a.n_pages * kBlock};
        const cuuint64_t gstride[1] = {(cuuint64_t)kTcD * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)kBlock};
        const cuuint32_t estride[2] = {1, 1};
        if (a.n_pages < 1) return cudaErrorInvalidValue;
        CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.k_pool), gdim, gstride, box,
                         estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    const int64_t max_tiles = (int64_t)dm.R * ((dm.MB + 1) / 2);
    int64_t grid = device_sm_count();
    if (grid > max_tiles) grid = max_tiles;
    if (grid < 1) grid = 1;
    cudaError_t e;
    if (fp8) {
        e = cudaFuncSetAttribute(score_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
        if (e != cudaSuccess) return e;
        score_tc_kernel<true><<<(unsigned)grid, 320, L.total, s>>>(cfg, a, map);
    } else {
        e = cudaFuncSetAttribute(score_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
        if (e != cudaSuccess) return e;
        score_tc_kernel<false><<<(unsigned)grid, 192, L.total, s>>>(cfg, a, map);
    }
    return cudaGetLastError();
}

}  // namespace spin

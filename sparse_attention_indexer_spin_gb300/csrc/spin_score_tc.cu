// spin_score_tc.cu -- indexer score with one key shared by all heads, on tcgen05 tensor
// cores (sm_103a).
//
// "SPIN: Shadow Predictive Indexer for Sparse Attention", §2 and Algorithm 1's scoring step:
// z_t[i] = sum_h w_h ReLU(q_{t,h} . k_i) over the slots of the selected blocks only.
// With one key per slot shared by the n_h heads (and, for speculative decoding, by the
// rows' queries), the per-tile work is a dense contraction
//     D[slot][row*n_h + h] = sum_c K[slot][c] * Q[row*n_h + h][c]
// of a 128-slot tile (two selected pages) with the 64*rows query vectors, so it runs on
// the tensor cores: M = 128 slots, N = 64*rows, K = d = 128, fp32 accumulation in TMEM.
//
// bf16 keys: kind::f16 (bf16 x bf16, exact products).  The keys and q reach shared memory
//   by 2D TMA in the 128-byte-swizzled K-major layout the MMA reads.
// FP8 (e4m3) keys: kind::f8f6f4 straight from the TMA-loaded pages, no conversion.  q is
//   carried as two e4m3 terms: for every (row, head) a power-of-two scale g puts
//   max|q|/g in (224, 448]; hi = e4m3(q/g), lo = e4m3(q/g - hi).  The two terms are two
//   B regions (N = 64 per query row); a tile's four K-steps over the hi terms and four over
//   the lo terms accumulate into the same accumulator, k.(hi + lo), where
//   |q/g - hi - lo| <= 2^-8 |q/g| per element (plus the e4m3 subnormal floor), and the
//   epilogue multiplies by g.  The per-slot dequantisation scale is applied before the ReLU.
// A tcgen05.mma costs a near-constant issue time whatever its N, so the kernel keeps
// the instruction count per tile low and interleaves two tiles (two accumulator chains)
// when TMEM holds four accumulators.
//
// Warp roles of a persistent CTA (tiles = pairs of selected blocks of one request; a CTA
// owns a contiguous range of whole tile pairs):
//   warps 0, 2  producers of the even and odd tiles: one (FP8) or two (bf16) 2D TMA loads
//               per page into a shared-memory ring
//   warps 1, 3  MMA issuers (one elected thread each): 8 tcgen05.mma per tile (FP8: 4 K-steps
//               x hi and lo terms; bf16: 8 K-steps).  Warp 1 takes the even tiles and warp 3
//               the odd ones, two independent accumulator chains.  Warp 1 owns the TMEM
//               allocation.  When the request changes, the issuers wait for their MMAs of
//               the previous one and restage q: FP8, both convert half of the vectors (a
//               quad of lanes per vector, the loads of four vectors in flight per lane);
//               bf16, warp 1 copies the rows by TMA.
//   warps 4-11  epilogue, two warps per TMEM lane quarter taking alternate tiles:
//               tcgen05.ld of a tile's accumulators (one slot per thread),
//               z = sum_h w_h g_h max(s_i acc_h, 0) per row, masked to i < N, stored
// Accumulators are 2-4 deep in TMEM (N <= 128: 4); the epilogue fetches the per-slot FP8
// scales of its next tile while it works on the current one.
// Every warp resolves its tiles' pages 32 at a time (one tile per lane), so the dependent
// list and block-table loads are paid once per 32 tiles; the requests' sizes are read once
// into shared memory with the tile prefix.  Every barrier wait is bounded
// and a timeout unwinds all roles.
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
constexpr int kTcEpiWarps = 8;                      // two per TMEM lane quarter
constexpr int kTcEpiWarp0 = 4;  // warps 0, 2: producers; 1, 3: MMA issuers; 4-11: epilogue
constexpr int kTcThreads = (kTcEpiWarp0 + kTcEpiWarps) * 32;
constexpr int kTcMaxAcc = 4;                        // accumulator buffers in TMEM
// operand ring depth (tiles in flight per CTA): as many as the shared memory budget holds, at
// most kTcStagesMax, an even number (the producers and issuers alternate tiles)
constexpr int kTcStagesMax = 8;
constexpr uint32_t kTcSmemBudget = 220 * 1024;
// FP8 slot scales travel in their own ring: a tile's scales stay until its epilogue has read
// them, i.e. up to (key stages + accumulators) tiles after they were loaded
constexpr int kTcScSlots = 12;
constexpr int kTcScBytes = 128 * 4;  // one tile: 128 slots

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

// Instruction descriptor (kind::f16 and kind::f8f6f4): fp32 accumulator, A and B of the same
// format (kind::f16: 0 = f16, 1 = bf16; kind::f8f6f4: 0 = e4m3), both K-major, N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t idesc_mma(uint32_t ab_fmt, uint32_t n, uint32_t m) {
    return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane, waited for in the same statement.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this thread's TMEM lane, waited for in the same statement.
__device__ __forceinline__ void tc_ld64(uint32_t taddr, float* v) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, "
        "%36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, "
        "%57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}


// max|x| over the 8 bf16 values of one 16-byte word group
__device__ __forceinline__ float amax_u4(float amax, const uint4 u) {
    const uint32_t wds[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        amax = fmaxf(amax, fabsf(__uint_as_float(wds[e] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(wds[e] & 0xffff0000u)));
    }
    return amax;
}

// Scale g of a q row from its max|q|: the power of two with max|q|/g in (224, 448].
__device__ __forceinline__ float q_scale_of(float amax) {
    if (!(amax > 0.0f)) return 1.0f;
    const float t = fmaxf(amax * (1.0f / 448.0f), 1e-30f);
    const uint32_t bits = __float_as_uint(t);
    float g = (bits & 0x7fffffu) ? __uint_as_float((bits & 0x7f800000u) + 0x00800000u) : t;
    if (amax > 448.0f * g) g *= 2.0f;
    return g;
}

// Query vectors handled by a quad of lanes: lane (lane & 3) holds the 32 values
// [32 (lane & 3), 32 (lane & 3) + 32) of the quad's vector as four 16-byte words, and the
// quad agrees on the vector's scale.
__device__ __forceinline__ void quad_load(const __nv_bfloat16* qrow, int lane, uint4 (&u)[4]) {
    const uint4* p = reinterpret_cast<const uint4*>(qrow) + 4 * (lane & 3);
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = p[i];
}

__device__ __forceinline__ float quad_scale(const uint4 (&u)[4]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = amax_u4(amax, u[i]);
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    return q_scale_of(amax);
}

// FP8 query terms of chunk ch (16 values held in u0, u1) of query vector n: hi = e4m3(q/g)
// into the region at sHi, lo = e4m3(q/g - hi) into the region at sLo, row n of each, in the
// 128-byte-swizzled K-major layout the MMA reads.
__device__ __forceinline__ void q8_convert_chunk(const uint4 u0, const uint4 u1, float inv_g, int n, int ch,
                                                 unsigned char* sHi, unsigned char* sLo) {
    const uint32_t wds[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        uint32_t hv = 0, lv = 0;
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
            const uint32_t wd = wds[2 * e + pr];
            const float2 x = make_float2(__uint_as_float(wd << 16) * inv_g, __uint_as_float(wd & 0xffff0000u) * inv_g);
            const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
            const __half2 hf = *reinterpret_cast<const __half2*>(
                &static_cast<const __half2_raw&>(__nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3)));
            const float2 hx = __half22float2(hf);
            const float2 rx = make_float2(x.x - hx.x, x.y - hx.y);
            const __nv_fp8x2_storage_t l2 = __nv_cvt_float2_to_fp8x2(rx, __NV_SATFINITE, __NV_E4M3);
            hv |= (uint32_t)h2 << (16 * pr);
            lv |= (uint32_t)l2 << (16 * pr);
        }
        hw[e] = hv;
        lw[e] = lv;
    }
    const uint32_t o = (uint32_t)((n >> 3) * 1024 + (n & 7) * 128 + ((ch ^ (n & 7)) << 4));
    *reinterpret_cast<uint4*>(sHi + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(sLo + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

struct TileInfo {
    int req, k0, blk0, blk1, page0, page1, n;
};

struct TcHdr {
    uint64_t full[kTcStagesMax];   // tile landed in shared memory
    uint64_t empty[kTcStagesMax];  // tile consumed by the MMAs
    uint64_t tfull[kTcMaxAcc];  // accumulator ready
    uint64_t tempty[kTcMaxAcc]; // accumulator drained by the epilogue
    uint64_t qfull;             // q staged by TMA (bf16 keys)
    uint64_t qdone;             // both issuers' MMAs of the previous request finished (2 arrivals)
    uint64_t qready;            // q of the next request staged (issuer 0 -> issuer 1)
    uint64_t fin[2];            // an issuer's MMAs all finished (teardown)
    uint64_t sfull[kTcScSlots];   // FP8: a tile's slot scales landed
    uint64_t sempty[kTcScSlots];  // FP8: a tile's slot scales read by its epilogue (4 warps)
    uint32_t tmem_base;
    int abort_flag;
    int total_tiles;
};

static_assert(sizeof(TcHdr) <= 1024, "the header fits its 1 KB");

struct TcLayout {
    uint32_t prefix, stage_a, qbuf, wbuf, sbuf, tile_bytes, total;
    int stages;
};

// accumulator buffers that fit in TMEM's 512 columns
__host__ __device__ constexpr int tc_nacc(int n) { return n <= 128 ? 4 : 2; }

__host__ __device__ inline TcLayout tc_layout(int R, int rows, bool fp8) {
    TcLayout L;
    L.tile_bytes = fp8 ? kTcM * kTcD : kTcM * kTcD * 2;  // 16 KB or 32 KB
    uint32_t off = 1024;                                 // header
    L.prefix = off;  // tile prefix [R + 1], then (N, list length) per request [R]
    off += ((uint32_t)(R + 1) * 4 + (uint32_t)R * 8 + 8 + 1023) & ~1023u;
    const uint32_t qbytes = (uint32_t)(64 * rows) * 256;             // two regions of N rows x 128 B
    const uint32_t wbytes = (uint32_t)kTcEpiWarps * 64 * rows * 4;    // w (times g) per epilogue warp
    const uint32_t sbytes = fp8 ? (uint32_t)(kTcScSlots * kTcScBytes) : 0u;  // slot scale ring
    const uint32_t fixed = off + qbytes + wbytes + sbytes + 1024;     // (+ slack for 1024-byte alignment)
    int st = fixed < kTcSmemBudget ? (int)((kTcSmemBudget - fixed) / L.tile_bytes) : 0;
    st = st > kTcStagesMax ? kTcStagesMax : st;
    L.stages = st & ~1;
    L.stage_a = off;
    off += (uint32_t)L.stages * L.tile_bytes;
    L.qbuf = off;
    off += qbytes;
    L.wbuf = off;
    off += wbytes;
    L.sbuf = off;
    off += sbytes;
    L.total = off + 1024;                                // slack for 1024-byte alignment
    return L;
}

template <bool FP8>
__global__ void __launch_bounds__(kTcThreads, 1)
score_tc_kernel(spin_config cfg, ScoreArgs a, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap qmap) {
    pdl_begin();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Dims dm = dims_of(cfg);
    const int rows = a.rows;
    const int NQ = kTcNH * rows;          // query vectors (rows x heads)
    const int N = NQ;                     // MMA N = accumulator columns per tile
    const TcLayout L = tc_layout(dm.R, rows, FP8);
    TcHdr* hdr = reinterpret_cast<TcHdr*>(smem);
    int* prefix = reinterpret_cast<int*>(smem + L.prefix);
    int2* reqinfo = reinterpret_cast<int2*>(smem + L.prefix + (((uint32_t)dm.R + 1) * 4 + 7) / 8 * 8);
    unsigned char* sA = smem + L.stage_a;
    unsigned char* sQ = smem + L.qbuf;
    float* sW = reinterpret_cast<float*>(smem + L.wbuf);
    float* sScale = reinterpret_cast<float*>(smem + L.sbuf);  // FP8: [kTcScSlots][128]
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int NACC = tc_nacc(N);
    const uint32_t tmem_cols = (uint32_t)(NACC * N) <= 256u ? 256u : 512u;
    // bytes of one B region: bf16, one K half of q; FP8, the hi (or lo) terms of q
    const uint32_t qregion = (uint32_t)NQ * 128;
    const int kTcStages = L.stages;

    // ------------------------------------------------------------------ set-up
    if (wid == 0) {
        int carry = 0;
        for (int base = 0; base < dm.R; base += 128) {
            // four chunks of 32 requests, their loads in flight together
            int nn[4], cc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = base + 32 * u + lane;
                nn[u] = r < dm.R ? a.n_slots[r] : 0;
                cc[u] = r < dm.R ? a.n_list[r] : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = base + 32 * u + lane;
                int c = 0;
                if (r < dm.R) {
                    const int64_t n = nn[u], cnt = cc[u];
                    const bool ok = n >= 0 && n <= dm.max_slots && cnt >= 0 && cnt <= dm.MB;
                    if (!ok && blockIdx.x == 0)
                        set_status(a.status, (n < 0 || n > dm.max_slots) ? SPIN_STATUS_BAD_N : SPIN_STATUS_BAD_LIST);
                    c = ok ? 2 * (int)((cnt + 3) / 4) : 0;  // tiles, padded to even: see the issuers
                    reqinfo[r] = make_int2(nn[u], cc[u]);
                }
                const int inc = warp_incl_scan(c);
                if (r < dm.R) prefix[r] = carry + inc - c;
                carry += __shfl_sync(0xffffffffu, inc, 31);
            }
        }
        if (lane == 0) {
            prefix[dm.R] = carry;
            hdr->total_tiles = carry;
            hdr->abort_flag = 0;
            for (int s = 0; s < kTcStages; ++s) {
                mbar_init(&hdr->full[s], 1);
                mbar_init(&hdr->empty[s], 1);
            }
            // two accumulators (N > 128): all eight epilogue warps drain every tile, each
            // parity half of its rows; otherwise four warps drain a tile
            const bool split_rows = tc_nacc(kTcNH * rows) < 4;
            for (int s = 0; s < kTcMaxAcc; ++s) {
                mbar_init(&hdr->tfull[s], 1);
                mbar_init(&hdr->tempty[s], split_rows ? 256 : 128);
            }
            mbar_init(&hdr->qfull, 1);
            mbar_init(&hdr->qdone, 2);
            mbar_init(&hdr->qready, 1);
            mbar_init(&hdr->fin[0], 1);
            mbar_init(&hdr->fin[1], 1);
            for (int c = 0; c < kTcScSlots; ++c) {
                mbar_init(&hdr->sfull[c], 1);
                mbar_init(&hdr->sempty[c], split_rows ? 8 : 4);
            }
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
    // ranges in whole tile pairs: every request contributes an even number of tiles to a
    // range, so the even- and odd-tile pipelines see the same sequence of requests
    const int t0 = 2 * (int)(((int64_t)(total / 2) * blockIdx.x) / gridDim.x);
    const int t1 = 2 * (int)(((int64_t)(total / 2) * (blockIdx.x + 1)) / gridDim.x);

    // FP8: the ten warps that are not producers stage the first request's query terms
    // together (a quarter of a vector per thread) while the producers start loading keys;
    // the issuers wait for them on named barrier 1, the epilogue warps only arrive
    const bool prestaged = FP8 && t0 < t1;
    if (prestaged && wid != 0 && wid != 2) {
        int lo = 0, hi = dm.R - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= t0) lo = mid; else hi = mid - 1;
        }
        const int req0 = lo;
        const int part = (wid == 1 ? 0 : wid == 3 ? 1 : wid - 2) * 32 + lane;  // 0 .. 319
        for (int n0 = 0; n0 < NQ; n0 += 80) {  // 80 quads of lanes, one query vector each
            const int n = n0 + (part >> 2);
            uint4 u[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                          make_uint4(0, 0, 0, 0)};
            if (n < NQ)
                quad_load(reinterpret_cast<const __nv_bfloat16*>(a.q) + ((int64_t)req0 * rows * kTcNH + n) * kTcD,
                          lane, u);
            const float inv_g = 1.0f / quad_scale(u);
            if (n < NQ) {
                q8_convert_chunk(u[0], u[1], inv_g, n, 2 * (lane & 3), sQ, sQ + qregion);
                q8_convert_chunk(u[2], u[3], inv_g, n, 2 * (lane & 3) + 1, sQ, sQ + qregion);
            }
        }
        fence_async_smem();
        if (wid == 1 || wid == 3) named_barrier(1, 320);
        else asm volatile("bar.arrive 1, 320;" ::: "memory");
    }

    // tile -> request, first list entry, its two blocks and their pages (-1: none / invalid)
    auto decode = [&](int t, TileInfo& ti) {
        int lo = 0, hi = dm.R - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
        }
        ti.req = lo;
        ti.k0 = 2 * (t - prefix[lo]);
        const int2 rq = reqinfo[lo];  // (a request that owns tiles passed the checks above)
        const int64_t n = rq.x, cnt = rq.y;
        const int64_t nb = (n + kBlock - 1) / kBlock;
        int bl[2], pg[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            bl[h] = -1;
            pg[h] = -1;
            const int64_t k = ti.k0 + h;
            if (k < cnt) {
                const int64_t b = a.list[(int64_t)lo * dm.MB + k];
                bl[h] = (int)b;
                if (b >= 0 && b < nb) {
                    const int64_t p = a.block_table[(int64_t)lo * a.bt_stride + b];
                    if (p >= 0 && p < a.n_pages) pg[h] = (int)p;
                } else {
                    bl[h] = -2;  // a listed block outside the context
                }
            }
        }
        ti.blk0 = bl[0]; ti.blk1 = bl[1]; ti.page0 = pg[0]; ti.page1 = pg[1];
        ti.n = (int)n;
    };
    // warp-cooperative: lane j resolves tile base + j; tile() broadcasts one tile's info.  FP8:
    // the next batch (base + 32, where every role's next request lands) is resolved ahead in
    // two steps whose loads are consumed only later: its list entries when a batch starts, its
    // block-table entries half-way through it.
    TileInfo mine, pf;
    int batch_base = -1, pf_base = -1, pf_step = 0;  // pf_step: 1 = list entries read, 2 = pages read
    int pf_b0 = -1, pf_b1 = -1, pf_p0 = -1, pf_p1 = -1;
    auto pf_list = [&](int base) {
        pf_base = base;
        pf_step = 1;
        const int t = base + lane;
        pf.req = -1;
        pf_b0 = pf_b1 = -1;
        if (t < t1) {
            int lo = 0, hi = dm.R - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
            }
            pf.req = lo;
            pf.k0 = 2 * (t - prefix[lo]);
            const int2 rq = reqinfo[lo];
            pf.n = rq.x;
            if (pf.k0 < rq.y) pf_b0 = a.list[(int64_t)lo * dm.MB + pf.k0];
            if (pf.k0 + 1 < rq.y) pf_b1 = a.list[(int64_t)lo * dm.MB + pf.k0 + 1];
        }
    };
    auto pf_pages = [&]() {
        pf_step = 2;
        pf_p0 = pf_p1 = -1;
        if (pf.req >= 0) {
            const int64_t nb = ((int64_t)pf.n + kBlock - 1) / kBlock;
            if (pf_b0 >= 0 && pf_b0 < nb) pf_p0 = a.block_table[(int64_t)pf.req * a.bt_stride + pf_b0];
            if (pf_b1 >= 0 && pf_b1 < nb) pf_p1 = a.block_table[(int64_t)pf.req * a.bt_stride + pf_b1];
        }
    };
    auto pf_finish = [&](TileInfo& ti) {  // the same values decode() gives
        ti.req = pf.req;
        ti.k0 = pf.k0;
        ti.n = pf.n;
        const int64_t nb = ((int64_t)pf.n + kBlock - 1) / kBlock;
        const int2 rq = pf.req >= 0 ? reqinfo[pf.req] : make_int2(0, 0);
        int bl[2] = {-1, -1}, pg[2] = {-1, -1};
        const int braw[2] = {pf_b0, pf_b1}, praw[2] = {pf_p0, pf_p1};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (pf.req >= 0 && pf.k0 + h < rq.y) {
                const int b = braw[h];
                bl[h] = b;
                if (b >= 0 && b < nb) {
                    const int p = praw[h];
                    if (p >= 0 && p < a.n_pages) pg[h] = p;
                } else {
                    bl[h] = -2;
                }
            }
        }
        ti.blk0 = bl[0]; ti.blk1 = bl[1]; ti.page0 = pg[0]; ti.page1 = pg[1];
    };
    auto refresh = [&](int t) {  // make the batch hold tile t (t non-decreasing per warp)
        if (!FP8) {  // bf16 tiles take twice as long: their dependent loads hide (measured)
            if (batch_base < 0 || t >= batch_base + 32) {
                batch_base = t;
                if (t + lane < t1) decode(t + lane, mine);
            }
            return;
        }
        if (batch_base < 0 || t >= batch_base + 32) {
            if (t == pf_base && pf_step > 0) {
                if (pf_step == 1) pf_pages();
                if (t + lane < t1) pf_finish(mine);
            } else if (t + lane < t1) {
                decode(t + lane, mine);
            }
            batch_base = t;
            pf_list(t + 32);
        } else if (pf_step == 1 && t - batch_base >= 16) {
            pf_pages();
        }
    };
    auto bc = [&](int v, int t) { return __shfl_sync(0xffffffffu, v, t - batch_base); };
    auto tile = [&](int t) -> TileInfo {
        refresh(t);
        const int j = t - batch_base;
        TileInfo r;
        r.req = __shfl_sync(0xffffffffu, mine.req, j);
        r.k0 = __shfl_sync(0xffffffffu, mine.k0, j);
        r.blk0 = __shfl_sync(0xffffffffu, mine.blk0, j);
        r.blk1 = __shfl_sync(0xffffffffu, mine.blk1, j);
        r.page0 = __shfl_sync(0xffffffffu, mine.page0, j);
        r.page1 = __shfl_sync(0xffffffffu, mine.page1, j);
        r.n = __shfl_sync(0xffffffffu, mine.n, j);
        return r;
    };
    auto fail_wait = [&]() {
        hdr->abort_flag = 1;
        set_status(a.status, SPIN_STATUS_TIMEOUT);
    };

    if (wid == 0 || wid == 2) {
        // -------------------------------------------------------------- producers
        // warp 0 loads the even tiles, warp 2 the odd ones (stages alternate with them)
        const int par = wid >> 1;
        uint32_t issued = 0, phases = 0;        // per stage: ever filled, parity of its last fill
        uint32_t sc_issued = 0, sc_phases = 0;  // the same for the FP8 scale ring
        for (int t = t0 + par, it = par; t < t1; t += 2, it += 2) {
            refresh(t);
            const int page0 = bc(mine.page0, t), page1 = bc(mine.page1, t);
            const int s = it % kTcStages;
            const uint32_t ph = (uint32_t)(it / kTcStages) & 1u;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&hdr->empty[s], ph ^ 1u, &hdr->abort_flag);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                if (lane == 0) fail_wait();
                break;
            }
            if (lane == 0) {
                const uint32_t page_bytes = FP8 ? (uint32_t)(kBlock * kTcD) : (uint32_t)(kBlock * kTcD * 2);
                const uint32_t bytes = (page0 >= 0 ? page_bytes : 0u) + (page1 >= 0 ? page_bytes : 0u);
                if (bytes == 0) {
                    mbar_arrive(&hdr->full[s]);
                } else {
                    mbar_arrive_expect_tx(&hdr->full[s], bytes);
                    unsigned char* stage = sA + (size_t)s * L.tile_bytes;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int page = h ? page1 : page0;
                        if (page < 0) continue;
                        const int y = page * kBlock;
                        // FP8: one 64-row x 128-byte box; bf16: the two 64-element K halves
                        tma_load_2d(stage + h * 8192, &kmap, 0, y, &hdr->full[s]);
                        if (!FP8) tma_load_2d(stage + kTcM * 128 + h * 8192, &kmap, 64, y, &hdr->full[s]);
                    }
                }
            }
            issued |= 1u << s;
            phases = (phases & ~(1u << s)) | (ph << s);
            if (FP8) {
                // the tile's slot scales (256 B per page) into scale-ring entry it % kTcScSlots,
                // once the epilogue of tile it - kTcScSlots has read that entry
                const int c = it % kTcScSlots;
                const uint32_t pc = (uint32_t)(it / kTcScSlots) & 1u;
                int ok2 = 1;
                if (lane == 0) ok2 = mbar_wait(&hdr->sempty[c], pc ^ 1u, &hdr->abort_flag);
                if (!__shfl_sync(0xffffffffu, ok2, 0)) {
                    if (lane == 0) fail_wait();
                    break;
                }
                if (lane == 0) {
                    const uint32_t sb = (page0 >= 0 ? 256u : 0u) + (page1 >= 0 ? 256u : 0u);
                    if (sb == 0) {
                        mbar_arrive(&hdr->sfull[c]);
                    } else {
                        mbar_arrive_expect_tx(&hdr->sfull[c], sb);
                        if (page0 >= 0)
                            bulk_g2s(sScale + c * 128, a.k_scale + (int64_t)page0 * kBlock, 256u, &hdr->sfull[c]);
                        if (page1 >= 0)
                            bulk_g2s(sScale + c * 128 + 64, a.k_scale + (int64_t)page1 * kBlock, 256u, &hdr->sfull[c]);
                    }
                }
                sc_issued |= 1u << c;
                sc_phases = (sc_phases & ~(1u << c)) | (pc << c);
            }
            __syncwarp();
        }
        // never leave with copies in flight: wait (bounded) for the last fill of every entry
        if (lane == 0) {
            for (int s = 0; s < kTcStages; ++s)
                if (((issued >> s) & 1u) && !mbar_wait(&hdr->full[s], (phases >> s) & 1u, nullptr))
                    set_status(a.status, SPIN_STATUS_TIMEOUT);
            for (int c = 0; c < kTcScSlots; ++c)
                if (((sc_issued >> c) & 1u) && !mbar_wait(&hdr->sfull[c], (sc_phases >> c) & 1u, nullptr))
                    set_status(a.status, SPIN_STATUS_TIMEOUT);
        }
    } else if (wid == 1 || wid == 3) {
        // ------------------------------------------------------------ MMA issuers
        // warp 1 issues the even tiles' MMAs, warp 3 the odd ones' (each issuing thread
        // sustains only so many tcgen05.mma, so two double the rate).  Both read sQ: on a
        // request change both commit to qdone, warp 1 waits for both, restages q and
        // signals qready, warp 3 waits for qready.
        // two issuers: with four accumulators each owns two, with two each owns one (the
        // epilogue then drains every tile with all eight warps)
        const int nis = 2;
        const int par = wid >> 1;
        const uint32_t idesc = idesc_mma(FP8 ? 0u : 1u, (uint32_t)N, (uint32_t)kTcM);
        int cur_req = -1;
        uint32_t nchange = 0, qload_phase = 0;
        bool issued_any = false;
        int sa = par, ac = par;  // ring positions of tile `it` (stride nis; S and NACC are even)
        uint32_t pha = 0, phc = 0;
        for (int t = t0 + par, it = par; par < nis && t < t1; t += nis, it += nis) {
            refresh(t);
            const int req = bc(mine.req, t);
            if (req != cur_req) {
                if (nchange > 0) {  // the previous request's MMAs must finish before sQ changes
                    if (lane == 0) tc_commit(&hdr->qdone);
                    __syncwarp();
                }
                if (FP8) {
                    // both issuers restage the query terms (the first request's were staged by ten
                    // warps before the loops): each converts half of the vectors, a quad of lanes
                    // per vector, four vectors' loads per lane in flight
                    if (nchange > 0) {
                        if (!__all_sync(0xffffffffu, mbar_wait(&hdr->qdone, (nchange - 1) & 1u, &hdr->abort_flag))) {
                            fail_wait();
                            break;
                        }
                        for (int p0 = 0; p0 < NQ / 16; p0 += 4) {
                            uint4 u[4][4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int n = par * (NQ / 2) + 8 * (p0 + i) + (lane >> 2);
                                quad_load(reinterpret_cast<const __nv_bfloat16*>(a.q) +
                                              ((int64_t)req * rows * kTcNH + n) * kTcD, lane, u[i]);
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int n = par * (NQ / 2) + 8 * (p0 + i) + (lane >> 2);
                                const float inv_g = 1.0f / quad_scale(u[i]);
                                q8_convert_chunk(u[i][0], u[i][1], inv_g, n, 2 * (lane & 3), sQ, sQ + qregion);
                                q8_convert_chunk(u[i][2], u[i][3], inv_g, n, 2 * (lane & 3) + 1, sQ, sQ + qregion);
                            }
                        }
                        fence_async_smem();
                        named_barrier(2, 64);  // both halves written
                    }
                } else if (par == 0) {
                    if (nchange > 0 && !mbar_wait(&hdr->qdone, (nchange - 1) & 1u, &hdr->abort_flag)) { fail_wait(); break; }
                    // q rows of this request by TMA, straight into the swizzled B layout
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&hdr->qfull, (uint32_t)NQ * kTcD * 2);
                        const int y = req * rows * kTcNH;
                        tma_load_2d(sQ, &qmap, 0, y, &hdr->qfull);
                        tma_load_2d(sQ + qregion, &qmap, 64, y, &hdr->qfull);
                    }
                    __syncwarp();
                    if (!mbar_wait(&hdr->qfull, qload_phase, &hdr->abort_flag)) { fail_wait(); break; }
                    qload_phase ^= 1u;
                    if (lane == 0) mbar_arrive(&hdr->qready);
                } else {
                    if (!mbar_wait(&hdr->qready, nchange & 1u, &hdr->abort_flag)) { fail_wait(); break; }
                }
                ++nchange;
                cur_req = req;
            }
            bool ok = mbar_wait(&hdr->full[sa], pha, &hdr->abort_flag) &&
                      mbar_wait(&hdr->tempty[ac], phc ^ 1u, &hdr->abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { fail_wait(); break; }
            tc_fence_after();
            if (lane == 0) {
                // k-step 0 descriptors; a k-step of 32 bytes adds 2 to the encoded start
                // address, a K half of a bf16 tile adds 16 KB >> 4
                const uint64_t a0 = smem_desc_sw128(smem_u32(sA + (size_t)sa * L.tile_bytes));
                const uint64_t b0 = smem_desc_sw128(smem_u32(sQ));
                const uint32_t d0 = tmem_base + (uint32_t)(ac * N);
                if (FP8) {
                    // k.(q_hi + q_lo): the hi terms' four k-steps, then the lo terms' into the same
                    // accumulator
                    const uint64_t bl = b0 + (qregion >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) tc_mma_f8(d0, a0 + 2 * kk, b0 + 2 * kk, idesc, kk ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) tc_mma_f8(d0, a0 + 2 * kk, bl + 2 * kk, idesc, 1u);
                } else {
                    const uint64_t bh = qregion >> 4;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t ao = (uint64_t)((ks >> 2) * (kTcM * 128 >> 4) + 2 * (ks & 3));
                        const uint64_t bo = (uint64_t)(ks >> 2) * bh + 2 * (ks & 3);
                        tc_mma_f16(d0, a0 + ao, b0 + bo, idesc, ks ? 1u : 0u);
                    }
                }
                tc_commit(&hdr->empty[sa]);
                tc_commit(&hdr->tfull[ac]);
            }
            issued_any = true;
            __syncwarp();
            sa += nis;
            if (sa >= kTcStages) { sa -= kTcStages; pha ^= 1u; }
            ac += nis;
            if (ac >= NACC) { ac -= NACC; phc ^= 1u; }
        }
        // every issued MMA has finished before TMEM is released
        if (issued_any) {
            if (lane == 0) tc_commit(&hdr->fin[par]);
            __syncwarp();
            if (!mbar_wait(&hdr->fin[par], 0u, nullptr)) set_status(a.status, SPIN_STATUS_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------- epilogue
        const int quarter = wid & 3;
        // four accumulators: this warp takes the tiles it with it % 2 == parity, all rows;
        // two: every tile, the rows r with r % 2 == parity (the accumulator frees sooner)
        const int parity = (wid - kTcEpiWarp0) / 4;
        const bool split_rows = NACC < 4;
        const int tstep = split_rows ? 1 : 2;
        const int m = quarter * 32 + lane;      // slot row of the tile = TMEM lane
        const int h = m >> 6, s = m & 63;
        float* wloc = sW + (size_t)(wid - kTcEpiWarp0) * NQ;
        int cur_req = -1;
        for (int t = t0 + (split_rows ? 0 : parity), it = split_rows ? 0 : parity; t < t1; t += tstep, it += tstep) {
            // FP8: this slot's scale, from the scale-ring entry the producer filled for tile it
            // (the warps that drain the tile free the entry once they have read it)
            // the tile's pages and (on a request change) the head weights first: they need no
            // barrier, so their loads overlap the wait for the tile's data
            const TileInfo ti = tile(t);
            const int req = ti.req;
            if (req != cur_req) {
                __syncwarp();
                if (FP8) {
                    // w_n g_n, a quad of lanes per query vector, four vectors' loads in flight
                    for (int p0 = 0; p0 < NQ / 8; p0 += 4) {
                        uint4 u[4][4];
                        float wv[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int n = 8 * (p0 + i) + (lane >> 2);
                            quad_load(reinterpret_cast<const __nv_bfloat16*>(a.q) +
                                          ((int64_t)req * rows * kTcNH + n) * kTcD, lane, u[i]);
                            wv[i] = a.w[(int64_t)req * rows * kTcNH + n];
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float g = quad_scale(u[i]);
                            if ((lane & 3) == 0) wloc[8 * (p0 + i) + (lane >> 2)] = wv[i] * g;
                        }
                    }
                } else {
                    for (int n = lane; n < NQ; n += 32) wloc[n] = a.w[(int64_t)req * rows * kTcNH + n];
                }
                __syncwarp();
                cur_req = req;
            }
            float scale = 1.0f;
            if (FP8) {
                const int c = it % kTcScSlots;
                if (!mbar_wait(&hdr->sfull[c], (uint32_t)(it / kTcScSlots) & 1u, &hdr->abort_flag)) {
                    fail_wait();
                    break;
                }
                scale = sScale[c * 128 + m];
                __syncwarp();
                if (lane == 0) mbar_arrive(&hdr->sempty[c]);
            }
            const int page = h ? ti.page1 : ti.page0;
            const int blk = h ? ti.blk1 : ti.blk0;
            const int64_t k = ti.k0 + h;
            const bool listed = blk != -1;                                    // a real list entry
            const bool live = page >= 0 && (int64_t)blk * kBlock + s < ti.n;  // a slot of the context
            if (listed && page < 0 && s == 0)
                set_status(a.status, blk == -2 ? SPIN_STATUS_BAD_LIST : SPIN_STATUS_BAD_PAGE);
            const int acc = it % NACC;
            const uint32_t phc = (uint32_t)(it / NACC) & 1u;
            if (!mbar_wait(&hdr->tfull[acc], phc, &hdr->abort_flag)) { fail_wait(); break; }
            tc_fence_after();
            const uint32_t trow = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * N);
            // sum_h w_h max(x_h, 0) of one row from its 64 heads' dot products (FP8:
            // k.(q_hi + q_lo) before the per-slot scale s, applied as |s| with sign(s) in x)
            auto head_sum = [&](float* v, int r) -> float {
                if (FP8 && scale < 0.0f) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) v[i] = -v[i];
                }
                float2 z2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
                const float4* wr = reinterpret_cast<const float4*>(wloc + r * kTcNH);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float4 wv = wr[j];
                    const float2 x0 = make_float2(fmaxf(v[4 * j + 0], 0.0f), fmaxf(v[4 * j + 1], 0.0f));
                    const float2 x1 = make_float2(fmaxf(v[4 * j + 2], 0.0f), fmaxf(v[4 * j + 3], 0.0f));
                    const int c = (j & 1) * 2;
                    z2[c] = __ffma2_rn(make_float2(wv.x, wv.y), x0, z2[c]);
                    z2[c + 1] = __ffma2_rn(make_float2(wv.z, wv.w), x1, z2[c + 1]);
                }
                float z = ((z2[0].x + z2[0].y) + (z2[1].x + z2[1].y)) + ((z2[2].x + z2[2].y) + (z2[3].x + z2[3].y));
                if (FP8) z *= fabsf(scale);
                return (!live || z == 0.0f) ? 0.0f : z;
            };
            auto emit = [&](float z, int r) {
                if (listed) a.scores[(((int64_t)req * rows + r) * dm.MB + k) * kBlock + s] = z;
            };
            // this warp's rows (paired TMEM loads measured slower)
            const int rstep = split_rows ? 2 : 1;
            int r = split_rows ? parity : 0;
            for (; r < rows; r += rstep) {
                float v[64];
                tc_ld64(trow + (uint32_t)(r * kTcNH), v);
                emit(head_sum(v, r), r);
            }
            tc_fence_before();
            mbar_arrive(&hdr->tempty[acc]);
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

// 2D tiled map over rows of 128 elements, 128-byte swizzle, box = {inner, box_rows}.
static bool encode_rows(CUtensorMap* map, CUtensorMapDataType dt, int elt, const void* base, int64_t n_rows,
                        uint32_t inner, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || n_rows < 1) return false;
    const cuuint64_t gdim[2] = {(cuuint64_t)kTcD, (cuuint64_t)n_rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)kTcD * elt};
    const cuuint32_t box[2] = {inner, box_rows};
    const cuuint32_t estride[2] = {1, 1};
    return enc(map, dt, 2, const_cast<void*>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool score_tc_supported(const spin_config& cfg, int rows) {
    return cfg.kv_heads == 1 && cfg.n_heads == kTcNH && cfg.head_dim == kTcD && rows >= 1 && rows <= kTcMaxRows &&
           cfg.n_req <= kTcMaxReq && cfg.q_dtype == SPIN_DTYPE_BF16 &&
           (cfg.k_dtype == SPIN_DTYPE_BF16 || cfg.k_dtype == SPIN_DTYPE_E4M3) &&
           tc_layout(cfg.n_req, rows, cfg.k_dtype == SPIN_DTYPE_E4M3).stages >= 2;
}

cudaError_t launch_score_tc(const spin_config& cfg, const ScoreArgs& a, cudaStream_t s) {
    if (!score_tc_supported(cfg, a.rows)) return cudaErrorNotSupported;
    if (((uintptr_t)a.q & 15) != 0 || a.n_pages < 1) return cudaErrorInvalidValue;
    const Dims dm = dims_of(cfg);
    const bool fp8 = cfg.k_dtype == SPIN_DTYPE_E4M3;
    const TcLayout L = tc_layout(dm.R, a.rows, fp8);
    CUtensorMap kmap, qmap;
    memset(&kmap, 0, sizeof kmap);
    memset(&qmap, 0, sizeof qmap);
    const int64_t pool_rows = a.n_pages * kBlock;
    if (fp8) {
        if (!encode_rows(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.k_pool, pool_rows, 128, kBlock))
            return cudaErrorInvalidValue;
    } else {
        if (!encode_rows(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k_pool, pool_rows, 64, kBlock) ||
            !encode_rows(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, (int64_t)dm.R * a.rows * kTcNH, 64,
                         (uint32_t)(kTcNH * a.rows)))
            return cudaErrorInvalidValue;
    }
    const int64_t max_tiles = (int64_t)dm.R * ((dm.MB + 1) / 2);
    int64_t grid = device_sm_count();
    if (grid > max_tiles) grid = max_tiles;
    if (grid < 1) grid = 1;
    cudaError_t e;
    if (fp8) {
        e = cudaFuncSetAttribute(score_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
        if (e != cudaSuccess) return e;
        return launch_pdl(score_tc_kernel<true>, dim3((unsigned)grid), dim3(kTcThreads), L.total, s, nullptr, 0,
                          cfg, a, kmap, qmap);
    } else {
        e = cudaFuncSetAttribute(score_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
        if (e != cudaSuccess) return e;
        return launch_pdl(score_tc_kernel<false>, dim3((unsigned)grid), dim3(kTcThreads), L.total, s, nullptr, 0,
                          cfg, a, kmap, qmap);
    }
}

}  // namespace spin

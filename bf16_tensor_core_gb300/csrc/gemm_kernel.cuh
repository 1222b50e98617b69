// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   C <- alpha * op(A) * op(B) + beta * C + bias,  f16/bf16 operands, f32 accumulation in TMEM.
//
// Design (prior art: "Optimizing GEMMs using tcgen05 - Part 2"):
//  * TMA loads with 128-byte swizzle into a STAGES-deep shared-memory ring guarded by
//    mbarrier expect_tx / complete_tx (section 5.1), BK = 64 so one operand row is one
//    128-byte swizzle span (section 7.3, "BK=64");
//  * warp specialisation: warp 0 lane 0 produces (waits "slot free", arms, issues copies),
//    warp 1 lane 0 issues tcgen05.mma and commits each slot back (section 5.2);
//  * BN = 256 with the accumulator in 256 TMEM columns (section 6.1); the 2-SM variant runs
//    one tcgen05.mma.cta_group::2 with M = 256 per cluster, each CTA loading its own 128 A
//    rows and half of B, both CTAs' copies completing on the leader's barrier (section 6.2);
//  * unlike the page's final kernel the grid is persistent: each cluster walks output tiles
//    in grouped raster order and owns TWO TMEM accumulators (2 x BN columns), so the
//    epilogue of tile i overlaps the mainloop of tile i+1 (the first item of section 8);
//    descriptors are derived per slot without rebuilding (third item of section 8);
//  * epilogue warps 2..5 drain TMEM with tcgen05.ld.32x32b (warp w reads lanes 32*(w%4)..),
//    apply alpha / beta / bias in f32, round to the output type, and write C either through
//    128-byte-swizzled shared memory and TMA tensor stores (section 7.2's idea, full 128-byte
//    lines) or, when C's layout does not allow TMA, with masked vector stores.
//
// Every wait is bounded (global-timer limit); on expiry the kernel records the failure in a
// device status word, lets in-flight copies and MMAs land, frees TMEM and returns.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx_sm103.cuh"

namespace gb300 {

enum : int { OUT_F16 = 0, OUT_BF16 = 1, OUT_F32 = 2 };  // same codes as gemm_dtype_t
enum : int { ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_EPILOGUE = 3 };
enum : unsigned { STATUS_TIMEOUT = 1u };

struct KernelParams {
    int M, N, K;
    int tiles_m, tiles_n, num_tiles, k_tiles;
    int raster_group;
    int a_mn, b_mn;            // 0: operand K-major in memory, 1: MN-major
    int a_3d, b_3d;            // 1: the operand's tensor map is 3-D and one box covers the whole stage
    uint32_t idesc;            // tcgen05 instruction descriptor (kind::f16)
    void* C;
    long long ldc;             // elements
    const void* bias;          // N elements of the output type, or nullptr
    float alpha, beta;
    int use_tma_store;         // write C with TMA tensor stores (with beta != 0, C_in boxes arrive by TMA loads)
    int c_vec_ok;              // C rows may be accessed with 16-byte vectors
    unsigned long long* status;
    unsigned long long timeout_ns;
    long long debug_skip_stage;  // test only: cluster 0's producer never issues this stage
    // Stream-K (sk_enabled != 0): tiles [0, dp_tiles) are walked data-parallel; the k-iterations of
    // tiles [dp_tiles, num_tiles) are divided evenly over the clusters (sk_base or sk_base + 1 each,
    // the first sk_extra clusters taking one more).  Each cluster's range is contiguous, so only its
    // first segment can start inside a tile (k0 > 0): that segment's f32 partial goes to the
    // cluster's slot of sk_partials and its flags are raised to `epoch`.  The segment that starts a
    // tile (the head, always a cluster's last) waits for the clusters after it that cover the rest
    // of the tile -- one when ranges are at least k_tiles long, several when a tile is split K-wise
    // over more clusters than there are tiles -- and adds their partials in cluster order.
    int sk_enabled;
    int dp_tiles;
    long long sk_base;
    int sk_extra;
    float* sk_partials;        // [cluster][cta rank][BN / 4][128 rows][4] f32
    unsigned* sk_flags;        // [cluster][cta rank][epilogue warp]
    unsigned epoch;            // launch counter of the handle, never 0
    // Q4_0 B (kernels built with kQ4): N rows of K/32 blocks of 18 bytes at pitch ldbq bytes.
    const uint8_t* bq;
    long long ldbq;
    int kblocks;               // K / 32
};

enum : int { UNIT_FULL = 0, UNIT_HEAD = 1, UNIT_TAIL = 2 };

struct Unit {
    int tile;
    int k0, k1;   // k-tile range [k0, k1) of this tile computed here
    int kind;     // UNIT_FULL, UNIT_HEAD (adds the partials of the following clusters), UNIT_TAIL (writes a partial)
};

// First stream-K iteration of cluster c.
__device__ __forceinline__ long long sk_range_start(const KernelParams& p, int c) {
    return static_cast<long long>(c) * p.sk_base + min(c, p.sk_extra);
}

// The deterministic sequence of work units of one cluster, identical in every role.
struct UnitIter {
    int next_dp, dp_limit, stride;
    long long it, it_end;

    __device__ __forceinline__ void init(const KernelParams& p, int cluster, int num_clusters) {
        next_dp = cluster;
        stride = num_clusters;
        dp_limit = p.sk_enabled ? p.dp_tiles : p.num_tiles;
        if (p.sk_enabled) {
            it = sk_range_start(p, cluster);
            it_end = it + p.sk_base + (cluster < p.sk_extra ? 1 : 0);
        } else {
            it = it_end = 0;
        }
    }

    __device__ __forceinline__ bool next(const KernelParams& p, Unit& u) {
        if (next_dp < dp_limit) {
            u.tile = next_dp;
            u.k0 = 0;
            u.k1 = p.k_tiles;
            u.kind = UNIT_FULL;
            next_dp += stride;
            return true;
        }
        if (it < it_end) {
            const long long rel = it / p.k_tiles;
            const int k0 = static_cast<int>(it - rel * p.k_tiles);
            const long long seg_end = min((rel + 1) * p.k_tiles, it_end);
            u.tile = p.dp_tiles + static_cast<int>(rel);
            u.k0 = k0;
            u.k1 = k0 + static_cast<int>(seg_end - it);
            u.kind = (k0 == 0 && u.k1 == p.k_tiles) ? UNIT_FULL : (k0 == 0 ? UNIT_HEAD : UNIT_TAIL);
            it = seg_end;
            return true;
        }
        return false;
    }
};

template <int kCtaGroup, int kBN, int kStages, int kBKc = 64, bool kQ4 = false>
struct TileConfig {
    static constexpr int kBM = 128;                    // rows per CTA (TMEM lanes)
    static constexpr int kBK = kBKc;                   // K per stage: 64 or 128
    static constexpr int kKChunks = kBK / 64;          // 64-wide K chunks (one 128-byte swizzle span each)
    static constexpr int kBNC = kBN / kCtaGroup;       // B columns each CTA loads
    static constexpr int kABytes = kBM * kBK * 2;      // 16 or 32 KB
    static constexpr int kBBytes = kBNC * kBK * 2;
    static constexpr int kAChunkBytes = kBM * 128;     // one 64-wide K chunk of a K-major A tile
    static constexpr int kBChunkBytes = kBNC * 128;    // one 64-wide K chunk of a K-major B tile
    static constexpr int kSlabBytes = kBK * 128;       // one 64-wide MN slab of an MN-major tile
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kRingBytes = kStages * kStageBytes;
    // Eight epilogue warps: warps w and w+4 read the same 32 TMEM lanes and split the columns.
    // With Q4_0 B, four of them are dequantisation warps instead and four drain all columns.
    static constexpr int kEpiWarps = kQ4 ? 4 : 8;
    static constexpr int kDqWarps = kQ4 ? 4 : 0;
    static constexpr int kEpiCols = kBN / (kEpiWarps / 4);   // accumulator columns one warp drains
    static constexpr int kEpiBufBytes = 32 * 128;      // 32 rows x 128 bytes, one staging buffer per warp
    static constexpr int kEpiBytes = kEpiWarps * kEpiBufBytes;
    static constexpr int kSmemBytes = kRingBytes + kEpiBytes + 1024;  // + alignment slack
    static constexpr int kThreads = 64 + 32 * (kEpiWarps + kDqWarps);
    static constexpr int kMmaN = kBN < 256 ? kBN : 256; // N of one tcgen05.mma (at most 256)
    static constexpr int kNHalves = kBN / kMmaN;       // MMAs per K step that cover the tile's N
    static constexpr int kHalfCols = kMmaN / kCtaGroup; // B columns of one MMA that a CTA holds
    static constexpr int kAccCols = kBN;               // f32 accumulator columns per buffer
    static constexpr int kAccBufs = (2 * kBN <= 512) ? 2 : 1;   // TMEM has 512 columns
    static constexpr int kTmemCols = (kAccBufs * kBN <= 32) ? 32 : (kAccBufs * kBN <= 64) ? 64
                                     : (kAccBufs * kBN <= 128) ? 128 : (kAccBufs * kBN <= 256) ? 256 : 512;
    static_assert(kBN % 64 == 0 && kBN <= 512, "BN must be a multiple of 64, at most 512");
    static_assert(kBN <= 256 || kBN % 256 == 0, "BN above 256 must be a multiple of 256");
    static_assert(kBK == 64 || kBK == 128, "BK must be 64 or 128");
    static_assert(kHalfCols % 64 == 0, "each CTA loads whole 64-column B slabs");
    static_assert(kSmemBytes <= 232448 - 512, "shared memory budget");
    static_assert(!kQ4 || (kBNC == 128 && kBK == 128 && kNHalves == 1),
                  "Q4_0 B: one dequantisation lane per B row (128 per CTA), four blocks per stage");
};

__device__ __forceinline__ void tile_coords(const KernelParams& p, int t, int& mb, int& nb) {
    const int per_group = p.raster_group * p.tiles_n;
    const int g = t / per_group;
    const int first = g * p.raster_group;
    const int gm = min(p.tiles_m - first, p.raster_group);
    const int local = t - g * per_group;
    mb = first + local % gm;
    nb = local / gm;
}

template <int kClusterCtas>
__device__ __forceinline__ void report_error(const KernelParams& p, int role, int tile, int stage,
                                             volatile int* abort_flag) {
    *abort_flag = 1;
    if constexpr (kClusterCtas > 1) {
        const uint32_t me = cluster_ctarank();
        for (uint32_t r = 0; r < static_cast<uint32_t>(kClusterCtas); ++r)
            if (r != me) st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), r), 1u);
    }
    const unsigned long long code = static_cast<unsigned long long>(STATUS_TIMEOUT) |
                                    (static_cast<unsigned long long>(role & 0xff) << 8) |
                                    (static_cast<unsigned long long>(stage & 0xffff) << 16) |
                                    (static_cast<unsigned long long>(static_cast<uint32_t>(tile)) << 32);
    atomicCAS(p.status, 0ull, code);
}

// ---------------------------------------------------------------- epilogue helpers
template <int kOut>
__device__ __forceinline__ float load_out(const void* base, long long idx) {
    if constexpr (kOut == OUT_F32) return static_cast<const float*>(base)[idx];
    else if constexpr (kOut == OUT_F16) return __half2float(static_cast<const __half*>(base)[idx]);
    else return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
}

template <int kOut>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (kOut == OUT_F16) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// The two 16-bit values of a packed word (low half first), widened to f32.
template <int kOut>
__device__ __forceinline__ void unpack2(uint32_t w, float& lo, float& hi) {
    if constexpr (kOut == OUT_F16) {
        lo = __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
        hi = __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
    } else {
        lo = __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(w & 0xffffu)));
        hi = __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(w >> 16)));
    }
}

// v[0..31] = alpha * acc + beta * cin + bias for columns col0 .. col0+31, C_in already in registers.
template <int kOut>
__device__ __forceinline__ void epilogue_math_cin(const KernelParams& p, const uint32_t (&acc)[32], float (&v)[32],
                                                  const float (&cin)[32], int col0) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(acc[i]);
    if (p.alpha != 1.0f) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= p.alpha;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = fmaf(p.beta, cin[i], v[i]);
    if (p.bias != nullptr) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col0 + i < p.N) v[i] += load_out<kOut>(p.bias, col0 + i);
    }
}

// v[0..31] = alpha * acc + beta * C_in + bias for columns col0 .. col0+31 of `row`.
template <int kOut>
__device__ __forceinline__ void epilogue_math(const KernelParams& p, const uint32_t (&acc)[32], float (&v)[32],
                                              int row, int col0) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(acc[i]);
    if (p.alpha != 1.0f) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= p.alpha;
    }
    if (p.beta != 0.0f && row < p.M) {
        const long long base = static_cast<long long>(row) * p.ldc + col0;
        if (p.c_vec_ok && col0 + 32 <= p.N) {
            if constexpr (kOut == OUT_F32) {
                const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.C) + base);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 c = src[j];
                    v[4 * j + 0] = fmaf(p.beta, c.x, v[4 * j + 0]);
                    v[4 * j + 1] = fmaf(p.beta, c.y, v[4 * j + 1]);
                    v[4 * j + 2] = fmaf(p.beta, c.z, v[4 * j + 2]);
                    v[4 * j + 3] = fmaf(p.beta, c.w, v[4 * j + 3]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = fmaf(p.beta, load_out<kOut>(p.C, base + i), v[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (col0 + i < p.N) v[i] = fmaf(p.beta, load_out<kOut>(p.C, base + i), v[i]);
        }
    }
    if (p.bias != nullptr) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col0 + i < p.N) v[i] += load_out<kOut>(p.bias, col0 + i);
    }
}

// Masked direct stores of 32 values of one row.
template <int kOut>
__device__ __forceinline__ void store_row_direct(const KernelParams& p, const float (&v)[32], int row, int col0) {
    if (row >= p.M) return;
    const long long base = static_cast<long long>(row) * p.ldc + col0;
    if (p.c_vec_ok && col0 + 32 <= p.N) {
        if constexpr (kOut == OUT_F32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.C) + base);
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.C) + base);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                dst[j] = make_uint4(pack2<kOut>(v[8 * j + 0], v[8 * j + 1]), pack2<kOut>(v[8 * j + 2], v[8 * j + 3]),
                                    pack2<kOut>(v[8 * j + 4], v[8 * j + 5]), pack2<kOut>(v[8 * j + 6], v[8 * j + 7]));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if (col0 + i < p.N) {
                if constexpr (kOut == OUT_F32) static_cast<float*>(p.C)[base + i] = v[i];
                else if constexpr (kOut == OUT_F16) static_cast<__half*>(p.C)[base + i] = __float2half_rn(v[i]);
                else static_cast<__nv_bfloat16*>(p.C)[base + i] = __float2bfloat16_rn(v[i]);
            }
        }
    }
}

// Ask L2 for the C_in lines of `row`, columns [col0, col0 + kCols) clipped to N, while the
// accumulator is still being computed: the epilogue then reads them from L2 instead of HBM.
template <int kOut, int kCols>
__device__ __forceinline__ void prefetch_c_rows(const KernelParams& p, int row, int col0) {
    if (row >= p.M || col0 >= p.N) return;
    constexpr int kElt = (kOut == OUT_F32) ? 4 : 2;
    const char* base = static_cast<const char*>(p.C) + (static_cast<long long>(row) * p.ldc + col0) * kElt;
    const int bytes = (min(kCols, p.N - col0)) * kElt;
    const int first = static_cast<int>(reinterpret_cast<uintptr_t>(base) & 127u);
    for (int off = -first; off < bytes; off += 128)
        asm volatile("prefetch.global.L2 [%0];" :: "l"(reinterpret_cast<uint64_t>(base + max(off, 0))));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// Stream-K partials.  Inside one CTA's slot the data of epilogue warp ew (its 32 rows x kCols
// columns) is one contiguous block [kCols / 4 column quads][32 lanes][4 f32]: a warp store of one
// quad is 512 contiguous bytes, and 64 columns (8 KB) are one contiguous piece.
constexpr uint32_t kFixPieceBytes = 64 * 32 * 4;   // 64 columns x 32 rows of f32
constexpr int kFixBufs = 3;                        // pieces in flight per warp

// Head fix-up: add the partials of `count` consecutive clusters (slots `stride` floats apart,
// `first` already at this warp's block) into this warp's accumulator columns in TMEM, in cluster
// order.  The head is always its cluster's last unit, so the operand ring is idle: each warp stages
// pieces through its own kFixBufs x 8 KB of it with bulk copies, kFixBufs in flight.
template <int kCols>
__device__ __forceinline__ bool head_fixup(uint32_t tbase, int lane, const float* first, int count, size_t stride,
                                           uint32_t region, uint32_t bar0, uint64_t timeout_ns,
                                           const volatile int* abort_flag) {
    static_assert(kCols % 64 == 0, "whole 64-column pieces");
    constexpr int kPieces = kCols / 64;
    const int n = count * kPieces;
    auto issue = [&](int i) {
        const int src = i / kPieces;
        const int pc = i - src * kPieces;
        const uint32_t b = static_cast<uint32_t>(i % kFixBufs);
        mbar_arrive_expect_tx(bar0 + 8u * b, kFixPieceBytes);
        bulk_load_g2s(region + b * kFixPieceBytes, first + static_cast<size_t>(src) * stride + pc * (64 * 32),
                      kFixPieceBytes, bar0 + 8u * b);
    };
    if (lane == 0) {
        fence_proxy_async_global();   // the flags were acquired by this thread in the generic proxy
        for (int i = 0; i < n && i < kFixBufs; ++i) issue(i);
    }
    __syncwarp();
#pragma unroll 1
    for (int i = 0; i < n; ++i) {
        const uint32_t b = static_cast<uint32_t>(i % kFixBufs);
        bool ok = mbar_wait_bounded(bar0 + 8u * b, static_cast<uint32_t>((i / kFixBufs) & 1), timeout_ns, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) return false;
        const uint32_t buf = region + b * kFixPieceBytes;
        const uint32_t tpiece = tbase + static_cast<uint32_t>((i % kPieces) * 64);
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
            uint32_t acc[32];
            tmem_ld_32x32b_x32(tpiece + cc * 32, acc);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 v = ld_shared_f4(buf + static_cast<uint32_t>(((cc * 8 + j) * 32 + lane) * 16));
                acc[4 * j + 0] = __float_as_uint(__uint_as_float(acc[4 * j + 0]) + v.x);
                acc[4 * j + 1] = __float_as_uint(__uint_as_float(acc[4 * j + 1]) + v.y);
                acc[4 * j + 2] = __float_as_uint(__uint_as_float(acc[4 * j + 2]) + v.z);
                acc[4 * j + 3] = __float_as_uint(__uint_as_float(acc[4 * j + 3]) + v.w);
            }
            tmem_st_32x32b_x32(tpiece + cc * 32, acc);
        }
        tmem_wait_st();
        __syncwarp();
        if (lane == 0 && i + kFixBufs < n) {
            fence_proxy_async_smem();   // this warp's reads of the buffer precede the next copy into it
            issue(i + kFixBufs);
        }
    }
    return true;
}

// One warp drains its 32 TMEM lanes (32 rows) x kCols columns of one accumulator buffer, starting at
// tile column pcol0 (tbase already points there).
//   out_part != nullptr: a stream-K tail segment; the raw f32 sums go to this warp's block of the
//   partial slot (layout above), C is untouched.
//   With beta != 0 on the TMA path, each box of C_in is first TMA-loaded into the warp's staging
//   buffer (completing on cin_bar; *cin_uses counts this warp's loads for the barrier parity), read
//   back row per lane, and the result overwrites it in place before the TMA store.
template <int kOut, int kCols>
__device__ __forceinline__ bool epilogue_tile(const KernelParams& p, const CUtensorMap* tmC, uint32_t tbase,
                                              int row0, int col_base, int lane, uint32_t stage_buf,
                                              float* out_part, uint32_t cin_bar, uint32_t* cin_uses,
                                              const volatile int* abort_flag) {
    const int row = row0 + lane;
    if (out_part != nullptr) {
        float4* dst = reinterpret_cast<float4*>(out_part);
#pragma unroll 1
        for (int c = 0; c < kCols / 32; ++c) {
            uint32_t acc[32];
            tmem_ld_32x32b_x32(tbase + c * 32, acc);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j)
                __stcg(&dst[(c * 8 + j) * 32 + lane],
                       make_float4(__uint_as_float(acc[4 * j]), __uint_as_float(acc[4 * j + 1]),
                                   __uint_as_float(acc[4 * j + 2]), __uint_as_float(acc[4 * j + 3])));
        }
        return true;
    }
    if (p.use_tma_store) {
        // A chunk is one 128-byte line per row: 64 columns of a 16-bit type, 32 of f32.
        constexpr int kChunk = (kOut == OUT_F32) ? 32 : 64;
        const bool warp_rows_in = row0 < p.M;
        const uint32_t row_addr = stage_buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll 1
        for (int c = 0; c < kCols / kChunk; ++c) {
            const int col0 = col_base + c * kChunk;
            const bool box_in = warp_rows_in && col0 < p.N;   // warp-uniform
            const bool with_cin = box_in && p.beta != 0.0f;
            if (with_cin && lane == 0) {
                bulk_wait_group_read<0>();                    // the previous store has read the buffer
                mbar_arrive_expect_tx(cin_bar, 32u * 128u);
                tma_load_2d(stage_buf, tmC, col0, row0, cin_bar);
            }
            uint32_t words[32];
            uint32_t acc0[32], acc1[32];
            tmem_ld_32x32b_x32(tbase + c * (kChunk == 32 ? 32 : 64), acc0);
            if constexpr (kChunk == 64) tmem_ld_32x32b_x32(tbase + c * 64 + 32, acc1);
            tmem_wait_ld();
            float v[32];
            if (with_cin) {
                const bool ok = mbar_wait_bounded(cin_bar, *cin_uses & 1u, p.timeout_ns, abort_flag);
                ++*cin_uses;
                if (!__all_sync(0xffffffffu, ok)) return false;
                // Row `lane` of the box: 16-byte piece j sits at piece j ^ (lane & 7) (128-byte swizzle).
                uint32_t cw[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 q = ld_shared_f4(row_addr + ((static_cast<uint32_t>(j) ^ (static_cast<uint32_t>(lane) & 7u)) * 16u));
                    cw[4 * j + 0] = __float_as_uint(q.x);
                    cw[4 * j + 1] = __float_as_uint(q.y);
                    cw[4 * j + 2] = __float_as_uint(q.z);
                    cw[4 * j + 3] = __float_as_uint(q.w);
                }
                float cin[32];
                if constexpr (kOut == OUT_F32) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) cin[i] = __uint_as_float(cw[i]);
                    epilogue_math_cin<kOut>(p, acc0, v, cin, col0);
#pragma unroll
                    for (int i = 0; i < 32; ++i) words[i] = __float_as_uint(v[i]);
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) unpack2<kOut>(cw[16 * h + i], cin[2 * i], cin[2 * i + 1]);
                        epilogue_math_cin<kOut>(p, h == 0 ? acc0 : acc1, v, cin, col0 + 32 * h);
#pragma unroll
                        for (int i = 0; i < 16; ++i) words[16 * h + i] = pack2<kOut>(v[2 * i], v[2 * i + 1]);
                    }
                }
            } else {
                epilogue_math<kOut>(p, acc0, v, row, col0);
                if constexpr (kOut == OUT_F32) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) words[i] = __float_as_uint(v[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) words[i] = pack2<kOut>(v[2 * i], v[2 * i + 1]);
                    epilogue_math<kOut>(p, acc1, v, row, col0 + 32);
#pragma unroll
                    for (int i = 0; i < 16; ++i) words[16 + i] = pack2<kOut>(v[2 * i], v[2 * i + 1]);
                }
            }
            if (!box_in) continue;                            // whole box outside C
            if (!with_cin && lane == 0) bulk_wait_group_read<0>();   // the previous store has read the buffer
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t piece = static_cast<uint32_t>(j) ^ (static_cast<uint32_t>(lane) & 7u);  // 128B swizzle
                st_shared_v4(row_addr + piece * 16u, words[4 * j], words[4 * j + 1], words[4 * j + 2], words[4 * j + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(tmC, col0, row0, stage_buf);
                bulk_commit_group();
            }
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < kCols / 32; ++c) {
            const int col0 = col_base + c * 32;
            uint32_t acc[32];
            tmem_ld_32x32b_x32(tbase + c * 32, acc);
            tmem_wait_ld();
            if (col0 >= p.N) continue;
            float v[32];
            epilogue_math<kOut>(p, acc, v, row, col0);
            store_row_direct<kOut>(p, v, row, col0);
        }
    }
    return true;
}

__device__ __forceinline__ void st_release_gpu(unsigned* addr, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* addr) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
    return v;
}

// Bounded wait for a stream-K flag written by another cluster of this grid (all clusters are
// co-resident: the grid never exceeds the device's active-cluster capacity).
__device__ __forceinline__ bool wait_flag_bounded(const unsigned* flag, unsigned want, uint64_t timeout_ns,
                                                  const volatile int* abort_flag) {
    if (ld_acquire_gpu(flag) == want) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        __nanosleep(64);
        if (ld_acquire_gpu(flag) == want) return true;
        if ((i & 31u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > timeout_ns) return false;
        }
    }
}

// ---------------------------------------------------------------- Q4_0 B operand
// Block format ("02 . 8m/8m(2) -- Tiled wmma f16 prefill GEMM", section 3.2): an f16 scale d and
// 16 bytes q; weight i is the low nibble of q[i], weight 16+i its high nibble, value d * (q - 8)
// rounded to f16.  Four blocks (128 K) of one B row per stage.
struct Q4Row {
    uint32_t d[4];      // f16 scale bits of each block (0: out of range, all weights 0)
    uint32_t q[4][4];   // the 16 nibble bytes of each block as four little-endian words
};

__device__ __forceinline__ void q4_load_row(const KernelParams& p, int n, int kt, Q4Row& r) {
    const int b0 = kt * 4;
    const uint8_t* row = p.bq + static_cast<long long>(n) * p.ldbq;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        if (n < p.N && b0 + b < p.kblocks) {
            // Blocks are 18 bytes, so only 2-byte alignment is guaranteed: nine 16-bit loads.
            const uint16_t* h = reinterpret_cast<const uint16_t*>(row + static_cast<long long>(b0 + b) * 18);
            uint32_t v[9];
#pragma unroll
            for (int i = 0; i < 9; ++i) v[i] = __ldg(h + i);
            r.d[b] = v[0];
#pragma unroll
            for (int w = 0; w < 4; ++w) r.q[b][w] = v[1 + 2 * w] | (v[2 + 2 * w] << 16);
        } else {
            r.d[b] = 0u;
#pragma unroll
            for (int w = 0; w < 4; ++w) r.q[b][w] = 0x88888888u;    // nibble 8: weight 0
        }
    }
}

// Two weights from the low (hi_half = 0) or high nibbles of bytes 2j and 2j+1 of word w, as f16x2
// d * (q - 8): 0x6400 | q is the f16 1024 + q, minus 1032 is q - 8 exactly, and the product with
// d is one correctly rounded f16 multiplication.
__device__ __forceinline__ uint32_t q4_pair(uint32_t w, int j, bool high, __half2 d2) {
    const uint32_t bytes = __byte_perm(w, 0u, j == 0 ? 0x4140u : 0x4342u);   // byte 2j -> [7:0], 2j+1 -> [23:16]
    const uint32_t nib = high ? ((bytes >> 4) & 0x000F000Fu) : (bytes & 0x000F000Fu);
    const uint32_t biased = nib | 0x64006400u;
    __half2 h = *reinterpret_cast<const __half2*>(&biased);
    h = __hsub2(h, __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6408u))));   // - 1032
    h = __hmul2(h, d2);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Write row `row` (0..127) of the stage's K-major, 128-byte-swizzled B tile: 128 K = two 64-wide
// chunks of 128 bytes; block b covers 16-byte pieces 4*(b%2)..+3 of chunk b/2.
__device__ __forceinline__ void q4_store_row(uint32_t sb, int row, const Q4Row& r, uint32_t chunk_bytes) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const __half2 d2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(r.d[b])));
        const uint32_t base = sb + static_cast<uint32_t>(b >> 1) * chunk_bytes + static_cast<uint32_t>(row) * 128u;
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
            // pieces 0,1: weights 0..15 = low nibbles of q[0..15]; pieces 2,3: weights 16..31 = high nibbles.
            const bool high = pc >= 2;
            const int w0 = (pc & 1) * 2;          // q words holding bytes 8*(pc&1) .. +7
            const uint32_t x0 = q4_pair(r.q[b][w0], 0, high, d2);
            const uint32_t x1 = q4_pair(r.q[b][w0], 1, high, d2);
            const uint32_t x2 = q4_pair(r.q[b][w0 + 1], 0, high, d2);
            const uint32_t x3 = q4_pair(r.q[b][w0 + 1], 1, high, d2);
            const uint32_t piece = static_cast<uint32_t>(4 * (b & 1) + pc) ^ (static_cast<uint32_t>(row) & 7u);
            st_shared_v4(base + piece * 16u, x0, x1, x2, x3);
        }
    }
}

// ---------------------------------------------------------------- the kernel
// kPairs == 2 (with kCtaGroup == 2): a 4-CTA cluster of two 2-SM pairs stacked along M.  Both pairs
// need the same B columns, so each pair loads half of every B stage and multicasts it to the
// matching CTA of the other pair: the cluster reads B from L2 once for 512 output rows.
// kQ4: B is Q4_0-quantised; dequantisation warps (after the epilogue warps) write each stage's
// B tile into shared memory instead of the producer's TMA copies.
template <int kCtaGroup, int kPairs, int kBN, int kStages, int kBK, int kOut, bool kQ4 = false>
__global__ void __launch_bounds__(TileConfig<kCtaGroup, kBN, kStages, kBK, kQ4>::kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const KernelParams p) {
    using Cfg = TileConfig<kCtaGroup, kBN, kStages, kBK, kQ4>;
    static_assert(!kQ4 || kPairs == 1, "Q4_0 B is built for one 2-SM pair per cluster");
    static_assert(kPairs == 1 || kCtaGroup == 2, "pairs of CTAs need cta_group::2");
    static_assert(kPairs == 1 || Cfg::kNHalves == 1, "B multicast is built for one MMA per K step");
    static_assert(Cfg::kRingBytes >= Cfg::kEpiWarps * kFixBufs * static_cast<int>(kFixPieceBytes),
                  "the head fix-up stages its pieces in the operand ring");
    constexpr int kClusterCtas = kCtaGroup * kPairs;
    constexpr int kClusterRows = Cfg::kBM * kClusterCtas;      // output rows of one cluster tile
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages];
    __shared__ __align__(8) uint64_t bar_empty[kStages];
    __shared__ __align__(8) uint64_t bar_tfull[2];
    __shared__ __align__(8) uint64_t bar_tempty[2];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ __align__(8) uint64_t bar_fix[Cfg::kEpiWarps * kFixBufs];   // stream-K head fix-up pieces
    __shared__ __align__(8) uint64_t bar_cin[Cfg::kEpiWarps];              // C_in boxes (beta != 0, TMA path)
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (kClusterCtas > 1) ? cluster_ctarank() : 0u;
    const uint32_t prank = rank & static_cast<uint32_t>(kCtaGroup - 1);   // rank within the 2-SM pair
    const uint32_t pair = rank / kCtaGroup;                                // which pair of the cluster
    const uint32_t lrank = rank - prank;                                   // MMA-issuing CTA of my pair
    const uint16_t pair_mask = static_cast<uint16_t>(((1u << kCtaGroup) - 1u) << lrank);
    const uint16_t all_mask = static_cast<uint16_t>((1u << kClusterCtas) - 1u);
    const int cluster_id = blockIdx.x / kClusterCtas;
    const int num_clusters = gridDim.x / kClusterCtas;
    const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t epi_smem = ring + Cfg::kRingBytes;
    volatile int* abort_flag = &s_abort;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < kStages; ++s) {
            // The producer's arrive (with the TMA byte count), plus one arrive per dequantisation
            // warp of every CTA of the pair when B is dequantised in shared memory.
            mbar_init(smem_u32(&bar_full[s]), 1 + Cfg::kDqWarps * kCtaGroup);
            mbar_init(smem_u32(&bar_empty[s]), kPairs);   // one commit from each pair that reads the slot
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_tfull[b]), 1);
            mbar_init(smem_u32(&bar_tempty[b]), Cfg::kEpiWarps * kCtaGroup);
        }
        mbar_init(smem_u32(&bar_drain), 1);
        for (int b = 0; b < Cfg::kEpiWarps * kFixBufs; ++b) mbar_init(smem_u32(&bar_fix[b]), 1);
        for (int b = 0; b < Cfg::kEpiWarps; ++b) mbar_init(smem_u32(&bar_cin[b]), 1);
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (p.use_tma_store) prefetch_tensormap(&tmC);
    }
    if (warp == 1) tmem_alloc<kCtaGroup>(smem_u32(&s_tmem_base), Cfg::kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kClusterCtas > 1) cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem_base = s_tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            long long gstage = 0;
            const uint32_t tx_bytes = static_cast<uint32_t>((kQ4 ? Cfg::kABytes : Cfg::kStageBytes) * kCtaGroup);
            bool ok = true;
            UnitIter units;
            units.init(p, cluster_id, num_clusters);
            Unit u;
            while (ok && units.next(p, u)) {
                int mb, nb;
                tile_coords(p, u.tile, mb, nb);
                const int m0 = mb * kClusterRows + static_cast<int>(rank) * Cfg::kBM;
                const int n0 = nb * kBN + static_cast<int>(prank) * Cfg::kBNC;   // (kNHalves == 1)
                for (int kt = u.k0; kt < u.k1; ++kt) {
                    if (!mbar_wait_bounded(smem_u32(&bar_empty[stage]), phase ^ 1u, p.timeout_ns, abort_flag)) {
                        if (!*abort_flag) report_error<kClusterCtas>(p, ROLE_PRODUCER, u.tile, static_cast<int>(stage), abort_flag);
                        ok = false;
                        break;
                    }
                    const bool skip = (gstage == p.debug_skip_stage) && cluster_id == 0;
                    if (!skip) {
                        const uint32_t full_local = smem_u32(&bar_full[stage]);
                        const uint32_t full_bar = (kCtaGroup == 2) ? mapa_shared(full_local, lrank) : full_local;
                        if (prank == 0) mbar_arrive_expect_tx(full_local, tx_bytes);
                        const uint32_t sa = ring + stage * Cfg::kStageBytes;
                        const uint32_t sb = sa + Cfg::kABytes;
                        const int k0 = kt * Cfg::kBK;
                        auto load = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1) {
                            if constexpr (kCtaGroup == 2) tma_load_2d_pair(dst, map, c0, c1, full_bar);
                            else tma_load_2d(dst, map, c0, c1, full_bar);
                        };
                        auto load3 = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2) {
                            if constexpr (kCtaGroup == 2) tma_load_3d_pair(dst, map, c0, c1, c2, full_bar);
                            else tma_load_3d(dst, map, c0, c1, c2, full_bar);
                        };
                        if (!p.a_mn) {
                            if (p.a_3d) {
                                load3(sa, &tmA, 0, m0, kt * Cfg::kKChunks);   // box {64, 128 M, K chunks}
                            } else {
#pragma unroll
                                for (int c = 0; c < Cfg::kKChunks; ++c)  // box {64 K, 128 M} per K chunk
                                    load(sa + static_cast<uint32_t>(c * Cfg::kAChunkBytes), &tmA, k0 + 64 * c, m0);
                            }
                        } else {
                            if (p.a_3d) {
                                load3(sa, &tmA, 0, k0, m0 / 64);          // box {64, BK K, 2 M slabs}
                            } else {
                                load(sa, &tmA, m0, k0);                   // box {64 M, BK K} slabs
                                load(sa + static_cast<uint32_t>(Cfg::kSlabBytes), &tmA, m0 + 64, k0);
                            }
                        }
                        if constexpr (kQ4) {
                            // B arrives from the dequantisation warps.
                        } else if constexpr (kPairs == 1) {
                            // For each MMA N half h the CTA holds columns
                            // [nb*BN + h*kMmaN + prank*kHalfCols, +kHalfCols).
#pragma unroll
                            for (int h = 0; h < Cfg::kNHalves; ++h) {
                                const int nh = nb * kBN + h * Cfg::kMmaN + static_cast<int>(prank) * Cfg::kHalfCols;
                                if (!p.b_mn) {
                                    if (p.b_3d) {                         // box {64, kHalfCols N, K chunks}
                                        load3(sb, &tmB, 0, nh, kt * Cfg::kKChunks);
                                    } else {
#pragma unroll
                                        for (int c = 0; c < Cfg::kKChunks; ++c)  // box {64 K, kHalfCols N} per K chunk
                                            load(sb + static_cast<uint32_t>(c * Cfg::kBChunkBytes + h * Cfg::kHalfCols * 128),
                                                 &tmB, k0 + 64 * c, nh);
                                    }
                                } else {
                                    const uint32_t dh = sb + static_cast<uint32_t>(h * (Cfg::kHalfCols / 64) * Cfg::kSlabBytes);
                                    if (p.b_3d) {                         // box {64, BK K, N slabs}
                                        load3(dh, &tmB, 0, k0, nh / 64);
                                    } else {
#pragma unroll
                                        for (int j = 0; j < Cfg::kHalfCols / 64; ++j)  // box {64 N, BK K} slabs
                                            load(dh + static_cast<uint32_t>(j * Cfg::kSlabBytes), &tmB, nh + 64 * j, k0);
                                    }
                                }
                            }
                        } else {
                            // This pair loads part `pair` of the CTA's B columns and multicasts it to
                            // the CTA with the same rank-in-pair in every pair of the cluster.
                            constexpr int kPart = Cfg::kBNC / kPairs;     // B columns per part
                            const uint16_t mc = static_cast<uint16_t>(((1u << prank) | (1u << (prank + 2))));
                            const int nb0 = n0 + kPart * static_cast<int>(pair);
                            if (!p.b_mn) {
                                // rows [pair * kPart, +kPart) of every K chunk: box {64 K, kPart N}
                                const uint32_t db = sb + pair * static_cast<uint32_t>(kPart * 128);
#pragma unroll
                                for (int c = 0; c < Cfg::kKChunks; ++c)
                                    tma_load_2d_pair_mc(db + static_cast<uint32_t>(c * Cfg::kBChunkBytes), &tmB,
                                                        k0 + 64 * c, nb0, full_bar, mc);
                            } else {
                                // slabs [pair * kPart / 64, +kPart / 64): box {64 N, BK K}
                                const uint32_t db = sb + pair * static_cast<uint32_t>((kPart / 64) * Cfg::kSlabBytes);
#pragma unroll
                                for (int j = 0; j < kPart / 64; ++j)
                                    tma_load_2d_pair_mc(db + static_cast<uint32_t>(j * Cfg::kSlabBytes), &tmB,
                                                        nb0 + 64 * j, k0, full_bar, mc);
                            }
                        }
                    }
                    ++gstage;
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader CTA)
        if (lane == 0 && prank == 0) {
            // K-major operand: 8-row groups 1024 bytes apart (SBO); a K=16 step is +32 bytes inside a
            // 64-wide K chunk, and the next chunk starts one chunk (rows x 128 bytes) further.
            // MN-major operand: 64-element slabs BK x 128 bytes apart (LBO), 8-row K groups 1024
            // bytes apart (SBO); a K=16 step is +2048 bytes.
            const uint32_t a_lbo = p.a_mn ? static_cast<uint32_t>(Cfg::kSlabBytes) : 16u;
            const uint32_t b_lbo = p.b_mn ? static_cast<uint32_t>(Cfg::kSlabBytes) : 16u;
            uint64_t a_koff[Cfg::kBK / 16], b_koff[Cfg::kBK / 16], b_hoff[Cfg::kNHalves];
#pragma unroll
            for (int k = 0; k < Cfg::kBK / 16; ++k) {
                a_koff[k] = (p.a_mn ? 2048u * k : static_cast<uint32_t>((k >> 2) * Cfg::kAChunkBytes + (k & 3) * 32)) >> 4;
                b_koff[k] = (p.b_mn ? 2048u * k : static_cast<uint32_t>((k >> 2) * Cfg::kBChunkBytes + (k & 3) * 32)) >> 4;
            }
            // Start of N half h inside a B stage: its slabs (MN-major) or its rows (K-major).
#pragma unroll
            for (int h = 0; h < Cfg::kNHalves; ++h)
                b_hoff[h] = (p.b_mn ? static_cast<uint32_t>(h * (Cfg::kHalfCols / 64) * Cfg::kSlabBytes)
                                    : static_cast<uint32_t>(h * Cfg::kHalfCols * 128)) >> 4;
            const uint64_t a_desc0 = smem_desc_sw128(ring, a_lbo, 1024u);
            const uint64_t b_desc0 = smem_desc_sw128(ring + Cfg::kABytes, b_lbo, 1024u);
            const uint64_t stage_step = static_cast<uint64_t>(Cfg::kStageBytes >> 4);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            UnitIter units;
            units.init(p, cluster_id, num_clusters);
            Unit u;
            while (ok && units.next(p, u)) {
                if (!mbar_wait_bounded<kCtaGroup == 2>(smem_u32(&bar_tempty[acc]), acc_phase ^ 1u, p.timeout_ns,
                                                       abort_flag)) {
                    if (!*abort_flag) report_error<kClusterCtas>(p, ROLE_MMA, u.tile, 100 + static_cast<int>(acc), abort_flag);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * static_cast<uint32_t>(Cfg::kAccCols);
                for (int kt = u.k0; kt < u.k1; ++kt) {
                    // With dequantised B the peer CTA's warps arrive on this barrier too (release at
                    // cluster scope), so the wait acquires at cluster scope.
                    if (!mbar_wait_bounded<kQ4 && kCtaGroup == 2>(smem_u32(&bar_full[stage]), phase, p.timeout_ns,
                                                                  abort_flag)) {
                        if (!*abort_flag) report_error<kClusterCtas>(p, ROLE_MMA, u.tile, static_cast<int>(stage), abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t ad = a_desc0 + stage * stage_step;
                    const uint64_t bd = b_desc0 + stage * stage_step;
#pragma unroll
                    for (int k = 0; k < Cfg::kBK / 16; ++k)
#pragma unroll
                        for (int h = 0; h < Cfg::kNHalves; ++h)
                            mma_f16<kCtaGroup>(d_tmem + static_cast<uint32_t>(h * Cfg::kMmaN), ad + a_koff[k],
                                               bd + b_hoff[h] + b_koff[k], p.idesc, (kt > u.k0 || k > 0) ? 1u : 0u);
                    mma_commit<kCtaGroup>(smem_u32(&bar_empty[stage]), all_mask);  // slot free in every CTA it feeds
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit<kCtaGroup>(smem_u32(&bar_tfull[acc]), pair_mask);  // accumulator ready
                if (++acc == static_cast<uint32_t>(Cfg::kAccBufs)) { acc = 0; acc_phase ^= 1u; }
            }
            // Drain: every MMA this thread issued has completed once bar_drain flips.  This wait
            // ignores the abort flag (only the time limit ends it): TMEM is freed after it.
            mma_commit<kCtaGroup>(smem_u32(&bar_drain), pair_mask);
            volatile int never = 0;
            mbar_wait_bounded(smem_u32(&bar_drain), 0u, p.timeout_ns, &never);
        }
    } else if (warp < 2 + Cfg::kEpiWarps) {
        // ------------------------------------------------------------ epilogue warps
        const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
        const int ew = warp - 2;
        const int pcol0 = (ew / 4) * Cfg::kEpiCols;   // first tile column this warp drains
        const uint32_t stage_buf = epi_smem + static_cast<uint32_t>(ew) * Cfg::kEpiBufBytes;
        const size_t slot_floats = static_cast<size_t>(kClusterCtas) * 128 * kBN;
        // This warp's block inside a CTA slot of the partials.
        const size_t warp_block = static_cast<size_t>(rank) * 128 * kBN + static_cast<size_t>(ew) * Cfg::kEpiCols * 32;
        uint32_t acc = 0, acc_phase = 0, cin_uses = 0;
        UnitIter units;
        units.init(p, cluster_id, num_clusters);
        Unit u;
        while (units.next(p, u)) {
            int mb, nb;
            tile_coords(p, u.tile, mb, nb);
            const int row0 = mb * kClusterRows + static_cast<int>(rank) * Cfg::kBM + quarter * 32;
            if (p.beta != 0.0f && u.kind != UNIT_TAIL)
                prefetch_c_rows<kOut, Cfg::kEpiCols>(p, row0 + lane, nb * kBN + pcol0);
            bool ok = mbar_wait_bounded(smem_u32(&bar_tfull[acc]), acc_phase, p.timeout_ns, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0 && !*abort_flag)
                    report_error<kClusterCtas>(p, ROLE_EPILOGUE, u.tile, 200 + static_cast<int>(acc), abort_flag);
                break;
            }
            tc_fence_after_sync();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   acc * static_cast<uint32_t>(Cfg::kAccCols) + static_cast<uint32_t>(pcol0);
            float* out_part = nullptr;
            if (u.kind == UNIT_TAIL) {
                out_part = p.sk_partials + static_cast<size_t>(cluster_id) * slot_floats + warp_block;
            } else if (u.kind == UNIT_HEAD) {
                // The rest of this tile, [k1, k_tiles), is the first unit of each following cluster
                // whose range starts before the tile ends.
                const long long tile_end = static_cast<long long>(u.tile - p.dp_tiles + 1) * p.k_tiles;
                int n = 0;
                bool ready = true;
                for (int src = cluster_id + 1; src < num_clusters && sk_range_start(p, src) < tile_end; ++src, ++n) {
                    const unsigned* flag =
                        p.sk_flags + (static_cast<size_t>(src) * kClusterCtas + rank) * Cfg::kEpiWarps + ew;
                    if (lane == 0 && ready) ready = wait_flag_bounded(flag, p.epoch, p.timeout_ns, abort_flag);
                }
                ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
                if (ready) {
                    ready = head_fixup<Cfg::kEpiCols>(
                        tbase, lane, p.sk_partials + static_cast<size_t>(cluster_id + 1) * slot_floats + warp_block, n,
                        slot_floats, ring + static_cast<uint32_t>(ew) * kFixBufs * kFixPieceBytes,
                        smem_u32(&bar_fix[ew * kFixBufs]), p.timeout_ns, abort_flag);
                }
                if (!ready) {
                    if (lane == 0 && !*abort_flag)
                        report_error<kClusterCtas>(p, ROLE_EPILOGUE, u.tile, 300 + quarter, abort_flag);
                    break;
                }
            }
            if (!epilogue_tile<kOut, Cfg::kEpiCols>(p, &tmC, tbase, row0, nb * kBN + pcol0, lane, stage_buf, out_part,
                                                    smem_u32(&bar_cin[ew]), &cin_uses, abort_flag)) {
                if (lane == 0 && !*abort_flag)
                    report_error<kClusterCtas>(p, ROLE_EPILOGUE, u.tile, 400 + quarter, abort_flag);
                break;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                const uint32_t te = smem_u32(&bar_tempty[acc]);
                if constexpr (kCtaGroup == 2) mbar_arrive_cluster(mapa_shared(te, lrank));
                else mbar_arrive_local(te);
                if (u.kind == UNIT_TAIL) {
                    // Every lane's partial stores precede this release (warp barrier, then fence).
                    __threadfence();
                    st_release_gpu(p.sk_flags + (static_cast<size_t>(cluster_id) * kClusterCtas + rank) * Cfg::kEpiWarps + ew,
                                   p.epoch);
                }
            }
            if (++acc == static_cast<uint32_t>(Cfg::kAccBufs)) { acc = 0; acc_phase ^= 1u; }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    } else if constexpr (kQ4) {
        // ------------------------------------------------------------ Q4_0 dequantisation warps
        // Lane `row` of warp dw owns B row dw * 32 + lane of this CTA's 128 (one output column n).
        // Raw blocks of the next stage are loaded while the current one waits for its slot.
        const int row = (warp - 2 - Cfg::kEpiWarps) * 32 + lane;
        UnitIter units;
        units.init(p, cluster_id, num_clusters);
        Unit u;
        bool valid = units.next(p, u);
        int kt = valid ? u.k0 : 0;
        auto row_of = [&](const Unit& uu) {
            int mb, nb;
            tile_coords(p, uu.tile, mb, nb);
            return nb * kBN + static_cast<int>(prank) * Cfg::kBNC + row;
        };
        Q4Row cur, nxt;
        int cur_tile = valid ? u.tile : 0;
        if (valid) q4_load_row(p, row_of(u), kt, cur);
        uint32_t stage = 0, phase = 0;
        while (valid) {
            // Advance to the next (unit, k-tile) and prefetch its raw blocks.
            const int this_tile = cur_tile;
            if (++kt >= u.k1) {
                valid = units.next(p, u);
                kt = valid ? u.k0 : 0;
            }
            if (valid) {
                cur_tile = u.tile;
                q4_load_row(p, row_of(u), kt, nxt);
            }
            bool ok = mbar_wait_bounded(smem_u32(&bar_empty[stage]), phase ^ 1u, p.timeout_ns, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0 && !*abort_flag)
                    report_error<kClusterCtas>(p, ROLE_PRODUCER, this_tile, 500 + static_cast<int>(stage), abort_flag);
                break;
            }
            q4_store_row(ring + stage * Cfg::kStageBytes + Cfg::kABytes, row, cur, Cfg::kBChunkBytes);
            asm volatile("fence.proxy.async;" ::: "memory");   // generic writes -> the MMA's async reads
            __syncwarp();
            if (lane == 0) {
                const uint32_t full_local = smem_u32(&bar_full[stage]);
                if constexpr (kCtaGroup == 2) mbar_arrive_cluster(mapa_shared(full_local, lrank));
                else mbar_arrive_local(full_local);
            }
            cur = nxt;
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
    }

    // ---------------------------------------------------------------- teardown
    if (threadIdx.x == 0 && *abort_flag) {
        // A bounded settle so copies issued before the abort land before shared memory goes away.
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 200000ull) { }
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kClusterCtas > 1) cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<kCtaGroup>(tmem_base, Cfg::kTmemCols);
    }
}

}  // namespace gb300

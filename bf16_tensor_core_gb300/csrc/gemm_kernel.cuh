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
    int c_trans;               // the kernel computes C^T: its element (i, j) is C[j * ldc + i]; the bias is
                               // indexed by i (direct stores only)
    int c_vec_ok;              // C rows may be accessed with 16-byte vectors
    int bias_vec_ok;           // the bias is 16-byte aligned: 32 of its values load as 16-byte vectors
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
    // Split K as a reduce-scatter (sk_rs = S dividing the epilogue warp count, with sk_enabled, no whole
    // tiles and every tile split over exactly S consecutive clusters with equal k ranges): part r of a
    // tile owns the blocks (32 rows x the warp's columns) of epilogue warps ew with ew * S / warps == r.
    // A warp whose block another part owns writes its partial and raises its flag; an owning warp waits
    // for the S - 1 flags of the same warp in the tile's other parts, adds their partials and stores its
    // block of C.  So every part moves (S - 1) / S of a tile instead of one head reading all S - 1.
    int sk_rs;
    // 1 (with sk_rs, 1-SM configs of 64-wide tiles, the transposed product): the S parts of a tile are the
    // S CTAs of one thread-block cluster, and the blocks travel through distributed shared memory
    // instead of global partials and flags.  Each owning warp arms a barrier for S - 1 blocks and tells
    // the same warp of every other part that its slice of the (now idle) operand ring is free; each of
    // those warps then stores its accumulator block straight into that slice (st.async, completing on
    // the owner's barrier); the owner adds the S blocks in part order and stores its block of C.
    int rs_cluster;
    // 1: whole tiles of odd waves walk their k-tiles from the last to the first, so the first operand
    // slabs such a tile reads are the ones the tiles of the wave before read last (still in L2).
    int k_alternate;
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
    int rev;      // 1: the range is walked from k1 - 1 down to k0
    // The k-tile of the unit's i-th stage.
    __device__ __forceinline__ int kt_at(int i) const { return rev ? k1 - 1 - i : k0 + i; }
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
            u.rev = p.k_alternate ? (next_dp / stride) & 1 : 0;   // the wave's parity
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
            u.rev = 0;
            it = seg_end;
            return true;
        }
        return false;
    }
};

template <int kCtaGroup, int kBN, int kStages, int kBKc = 64, bool kQ4 = false, int kElt = 2>
struct TileConfig {
    static constexpr int kBM = 128;                    // rows per CTA (TMEM lanes)
    static constexpr int kBK = kBKc;                   // K per stage
    static constexpr int kEltBytes = kElt;             // 2: f16 / bf16 inputs, 1: 8-bit floats
    static constexpr int kKChunkElems = 128 / kElt;    // K elements of one 128-byte swizzle span
    static constexpr int kKChunks = kBK / kKChunkElems;   // swizzle-span-wide K chunks per stage
    static constexpr int kKPerMma = 32 / kElt;         // K of one tcgen05.mma: 16 (kind::f16), 32 (kind::f8f6f4)
    static constexpr int kMmasPerStage = kBK / kKPerMma;
    static constexpr int kBNC = kBN / kCtaGroup;       // B columns each CTA loads
    static constexpr int kABytes = kBM * kBK * kElt;   // 16 or 32 KB
    static constexpr int kBBytes = kBNC * kBK * kElt;
    static constexpr int kAChunkBytes = kBM * 128;     // one 64-wide K chunk of a K-major A tile
    static constexpr int kBChunkBytes = kBNC * 128;    // one 64-wide K chunk of a K-major B tile
    static constexpr int kSlabBytes = kBK * 128;       // one 64-wide MN slab of an MN-major tile
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kRingBytes = kStages * kStageBytes;
    // Eight epilogue warps: warps w and w+4 read the same 32 TMEM lanes and split the columns.
    // With Q4_0 B, four epilogue warps drain all columns and eight dequantisation warps follow.
    static constexpr int kEpiWarps = kQ4 ? 4 : 8;
    static constexpr int kDqWarps = kQ4 ? 8 : 0;
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
    static_assert(kBK * kElt == 128 || kBK * kElt == 256, "a stage is one or two 128-byte swizzle spans of K");
    static_assert(kElt == 2 || !kQ4, "Q4_0 weights dequantise to f16");
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

// v[i] += bias[col0 + i] for the columns inside C.  col0 is a multiple of 32 and the same for every lane,
// so with a 16-byte aligned bias the 32 values arrive as broadcast 16-byte loads.
template <int kOut>
__device__ __forceinline__ void add_bias(const KernelParams& p, float (&v)[32], int col0) {
    if (p.bias == nullptr) return;
    if (!p.bias_vec_ok || col0 + 32 > p.N) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col0 + i < p.N) v[i] += load_out<kOut>(p.bias, col0 + i);
        return;
    }
    if constexpr (kOut == OUT_F32) {
        const float4* b4 = reinterpret_cast<const float4*>(static_cast<const float*>(p.bias) + col0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 b = __ldg(b4 + j);
            v[4 * j + 0] += b.x;
            v[4 * j + 1] += b.y;
            v[4 * j + 2] += b.z;
            v[4 * j + 3] += b.w;
        }
    } else {
        const uint4* b4 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.bias) + col0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 b = __ldg(b4 + j);
            const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float lo, hi;
                unpack2<kOut>(w[h], lo, hi);
                v[8 * j + 2 * h] += lo;
                v[8 * j + 2 * h + 1] += hi;
            }
        }
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
    add_bias<kOut>(p, v, col0);
}

// v[0..31] = alpha * acc + beta * C_in + bias for columns col0 .. col0+31 of `row` (kTrans: of the
// transposed product, whose element (row, col) is C[col * ldc + row] and whose bias follows `row`).
template <int kOut, bool kTrans = false>
__device__ __forceinline__ void epilogue_math(const KernelParams& p, const uint32_t (&acc)[32], float (&v)[32],
                                              int row, int col0) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(acc[i]);
    if (p.alpha != 1.0f) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= p.alpha;
    }
    if constexpr (kTrans) {
        if (p.beta != 0.0f && row < p.M) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (col0 + i < p.N)
                    v[i] = fmaf(p.beta, load_out<kOut>(p.C, static_cast<long long>(col0 + i) * p.ldc + row), v[i]);
        }
        if (p.bias != nullptr && row < p.M) {
            const float b = load_out<kOut>(p.bias, row);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] += b;
        }
        return;
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
    add_bias<kOut>(p, v, col0);
}

// Masked direct stores of 32 values of one row.
template <int kOut, bool kTrans = false>
__device__ __forceinline__ void store_row_direct(const KernelParams& p, const float (&v)[32], int row, int col0) {
    if (row >= p.M) return;
    if constexpr (kTrans) {   // column `row` of C: for each j the lanes of a warp write consecutive addresses
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if (col0 + i < p.N) {
                const long long idx = static_cast<long long>(col0 + i) * p.ldc + row;
                if constexpr (kOut == OUT_F32) static_cast<float*>(p.C)[idx] = v[i];
                else if constexpr (kOut == OUT_F16) static_cast<__half*>(p.C)[idx] = __float2half_rn(v[i]);
                else static_cast<__nv_bfloat16*>(p.C)[idx] = __float2bfloat16_rn(v[i]);
            }
        }
        return;
    }
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

// The same for the transposed product: the warp's block of C^T is kernel rows row0 .. row0 + 31 and
// kernel columns col0 .. col0 + kCols - 1, i.e. 32 consecutive elements of each of C's rows col0 + j;
// lane l asks for rows col0 + l, col0 + 32 + l, ...
template <int kOut, int kCols>
__device__ __forceinline__ void prefetch_c_block_trans(const KernelParams& p, int row0, int col0, int lane) {
    if (row0 >= p.M) return;
    constexpr int kElt = (kOut == OUT_F32) ? 4 : 2;
#pragma unroll
    for (int t = 0; t < kCols / 32; ++t) {
        const int j = col0 + 32 * t + lane;
        if (j >= p.N) break;
        const char* a = static_cast<const char*>(p.C) + (static_cast<long long>(j) * p.ldc + row0) * kElt;
        asm volatile("prefetch.global.L2 [%0];" :: "l"(reinterpret_cast<uint64_t>(a)));
        const int last = min(32, p.M - row0) * kElt - 1;   // the block's last byte in this row
        if (((reinterpret_cast<uintptr_t>(a) & 127u) + last) >= 128u)
            asm volatile("prefetch.global.L2 [%0];" :: "l"(reinterpret_cast<uint64_t>(a + last)));
    }
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

// A warp's whole 32 x 32 block of the transposed product, 16-bit output: lane l holds v[i] =
// C[col0 + i][row0 + l].  The block goes through the warp's staging buffer (row i of C at i * 64 bytes)
// so that each lane then writes 16-byte pieces of C's rows instead of 32 two-byte stores.  Needs the
// whole block inside C and 16-byte aligned C rows (row0 is a multiple of 32).
template <int kOut>
__device__ __forceinline__ void store_block_trans_staged(const KernelParams& p, const float (&v)[32], int row0,
                                                         int col0, int lane, uint32_t buf) {
    static_assert(kOut != OUT_F32, "16-bit outputs");
    constexpr int kElt = 2;
    constexpr int kPieces = 32 * kElt / 16;          // 16-byte pieces per row of the block
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t a = buf + static_cast<uint32_t>((i * 32 + lane) * kElt);
        const unsigned short h = static_cast<unsigned short>(pack2<kOut>(v[i], 0.0f) & 0xffffu);
        asm volatile("st.shared.u16 [%0], %1;" :: "r"(a), "h"(h) : "memory");
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < kPieces; ++k) {
        const int c = lane + 32 * k;
        const int i = c / kPieces, piece = c % kPieces;
        const float4 w = ld_shared_f4(buf + static_cast<uint32_t>(i * 32 * kElt + piece * 16));
        char* dst = static_cast<char*>(p.C) + (static_cast<long long>(col0 + i) * p.ldc + row0) * kElt + piece * 16;
        *reinterpret_cast<float4*>(dst) = w;
    }
    __syncwarp();   // the buffer is free again
}

// Stream-K partials.  Inside one CTA's slot the data of epilogue warp ew (its 32 rows x kCols
// columns) is one contiguous block [kCols / 4 column quads][32 lanes][4 f32]: a warp store of one
// quad is 512 contiguous bytes, and 64 columns (8 KB) are one contiguous piece.
constexpr uint32_t kFixPieceBytes = 64 * 32 * 4;   // at most 64 columns x 32 rows of f32 per piece
constexpr int kFixBufs = 3;                        // pieces in flight per warp

// Head fix-up: add the partials of `count` consecutive clusters (slots `stride` floats apart,
// `first` already at this warp's block; slot `hole`, if given, is skipped) into this warp's
// accumulator columns in TMEM, in cluster order.  The head is always its cluster's last unit, so the
// operand ring is idle: each warp stages pieces through its own kFixBufs x 8 KB of it with bulk
// copies, kFixBufs in flight.
template <int kCols>
__device__ __forceinline__ bool head_fixup(uint32_t tbase, int lane, const float* first, int count, size_t stride,
                                           uint32_t region, uint32_t bar0, uint64_t timeout_ns,
                                           const volatile int* abort_flag, int hole = 1 << 30) {
    constexpr int kPieceCols = kCols < 64 ? kCols : 64;
    static_assert(kPieceCols % 32 == 0 && kCols % kPieceCols == 0, "whole pieces of 32 or 64 columns");
    constexpr int kPieces = kCols / kPieceCols;
    constexpr uint32_t kPieceBytes = kPieceCols * 32 * 4;
    const int n = count * kPieces;
    auto issue = [&](int i) {
        const int j = i / kPieces;
        const int pc = i - j * kPieces;
        const int src = j + (j >= hole ? 1 : 0);   // sources skip slot `hole` (the caller's own)
        const uint32_t b = static_cast<uint32_t>(i % kFixBufs);
        mbar_arrive_expect_tx(bar0 + 8u * b, kPieceBytes);
        bulk_load_g2s(region + b * kFixPieceBytes, first + static_cast<size_t>(src) * stride + pc * (kPieceCols * 32),
                      kPieceBytes, bar0 + 8u * b);
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
        const uint32_t tpiece = tbase + static_cast<uint32_t>((i % kPieces) * kPieceCols);
#pragma unroll 1
        for (int cc = 0; cc < kPieceCols / 32; ++cc) {
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
//   cin_ring != 0 (the cluster's last unit, whose operand ring is idle): all of the warp's C_in boxes
//   are loaded at once, each into its own 4 KB at cin_ring, and each result is stored from there, so
//   the boxes do not wait for one another's round trips.
//   kLean (a CTA of 14 warps, 128 registers each): the second 32-column half of a 16-bit box is read from
//   TMEM only after the first half is packed, so that the two halves are never live together.
//   parts > 0 (transposed 32-column blocks only, KernelParams::rs_cluster): the accumulator is part `self`
//   of the tile's `parts` partial sums and the others' blocks are in shared memory at parts_smem + 4 KB x
//   part (slot `self` free, each block [8 column quads][32 lanes][4 f32]); the block's value is
//   ((x_0 + x_1) + x_2) + ... in part order.
template <int kOut, int kCols, bool kTrans = false, bool kLean = false>
__device__ __forceinline__ bool epilogue_tile(const KernelParams& p, const CUtensorMap* tmC, uint32_t tbase,
                                              int row0, int col_base, int lane, uint32_t stage_buf,
                                              float* out_part, uint32_t cin_bar, uint32_t* cin_uses,
                                              const volatile int* abort_flag, uint32_t cin_ring = 0,
                                              uint32_t parts_smem = 0, int parts = 0, int self = 0) {
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
    // A chunk is one 128-byte line per row: 64 columns of a 16-bit type, 32 of f32.  A warp whose
    // columns do not fill whole chunks (a 64-wide tile with 16-bit output) uses direct stores.
    constexpr int kChunk = (kOut == OUT_F32) ? 32 : 64;
    constexpr bool kWholeBoxes = kCols % kChunk == 0;
    if (kWholeBoxes && !kTrans && p.use_tma_store) {
        const bool warp_rows_in = row0 < p.M;
        constexpr int kBoxes = kCols / kChunk;
        const bool ring_cin = cin_ring != 0 && p.beta != 0.0f && warp_rows_in;   // warp-uniform
        if (ring_cin) {
            int nbox = 0;
#pragma unroll 1
            for (int c = 0; c < kBoxes; ++c) nbox += (col_base + c * kChunk < p.N) ? 1 : 0;
            if (nbox > 0) {
                __syncwarp();
                if (lane == 0) {
                    fence_proxy_async_smem();   // earlier generic reads of this region (a fix-up) precede the copies
                    mbar_arrive_expect_tx(cin_bar, static_cast<uint32_t>(nbox) * 32u * 128u);
#pragma unroll 1
                    for (int c = 0; c < kBoxes; ++c)
                        if (col_base + c * kChunk < p.N)
                            tma_load_2d(cin_ring + static_cast<uint32_t>(c) * 4096u, tmC, col_base + c * kChunk, row0,
                                        cin_bar);
                }
                const bool ok = mbar_wait_bounded(cin_bar, *cin_uses & 1u, p.timeout_ns, abort_flag);
                ++*cin_uses;
                if (!__all_sync(0xffffffffu, ok)) return false;
            }
        }
#pragma unroll 1
        for (int c = 0; c < kBoxes; ++c) {
            const int col0 = col_base + c * kChunk;
            const bool box_in = warp_rows_in && col0 < p.N;   // warp-uniform
            const bool with_cin = box_in && p.beta != 0.0f;
            const uint32_t buf = ring_cin ? cin_ring + static_cast<uint32_t>(c) * 4096u : stage_buf;
            const uint32_t row_addr = buf + static_cast<uint32_t>(lane) * 128u;
            if (with_cin && !ring_cin && lane == 0) {
                bulk_wait_group_read<0>();                    // the previous store has read the buffer
                mbar_arrive_expect_tx(cin_bar, 32u * 128u);
                tma_load_2d(stage_buf, tmC, col0, row0, cin_bar);
            }
            uint32_t words[32];
            uint32_t acc0[32], acc1[kLean ? 1 : 32];
            tmem_ld_32x32b_x32(tbase + c * (kChunk == 32 ? 32 : 64), acc0);
            if constexpr (kChunk == 64 && !kLean) tmem_ld_32x32b_x32(tbase + c * 64 + 32, acc1);
            tmem_wait_ld();
            // The second half of a 16-bit box (kLean: read into acc0 once the first half is packed).
            auto second_half = [&]() -> const uint32_t (&)[32] {
                if constexpr (kLean) {
                    tmem_ld_32x32b_x32(tbase + c * 64 + 32, acc0);
                    tmem_wait_ld();
                    return acc0;
                } else {
                    return acc1;
                }
            };
            float v[32];
            if (with_cin) {
                if (!ring_cin) {
                    const bool ok = mbar_wait_bounded(cin_bar, *cin_uses & 1u, p.timeout_ns, abort_flag);
                    ++*cin_uses;
                    if (!__all_sync(0xffffffffu, ok)) return false;
                }
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
                        if (h == 0) epilogue_math_cin<kOut>(p, acc0, v, cin, col0);
                        else epilogue_math_cin<kOut>(p, second_half(), v, cin, col0 + 32);
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
                    epilogue_math<kOut>(p, second_half(), v, row, col0 + 32);
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
                tma_store_2d(tmC, col0, row0, buf);
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
            if constexpr (kTrans && kCols == 32) {
                if (parts > 0) {
                    // This warp's own block joins the others at its part's slot; then the sum runs in
                    // part order.
                    const uint32_t own = parts_smem + static_cast<uint32_t>(self) * 4096u;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        st_shared_v4(own + static_cast<uint32_t>((q * 32 + lane) * 16), acc[4 * q], acc[4 * q + 1],
                                     acc[4 * q + 2], acc[4 * q + 3]);
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float4 sum = ld_shared_f4(parts_smem + static_cast<uint32_t>((q * 32 + lane) * 16));
                        for (int i = 1; i < parts; ++i) {
                            const float4 e = ld_shared_f4(parts_smem + static_cast<uint32_t>(i) * 4096u +
                                                          static_cast<uint32_t>((q * 32 + lane) * 16));
                            sum.x += e.x; sum.y += e.y; sum.z += e.z; sum.w += e.w;
                        }
                        acc[4 * q + 0] = __float_as_uint(sum.x);
                        acc[4 * q + 1] = __float_as_uint(sum.y);
                        acc[4 * q + 2] = __float_as_uint(sum.z);
                        acc[4 * q + 3] = __float_as_uint(sum.w);
                    }
                }
            }
            if (col0 >= p.N) continue;
            float v[32];
            epilogue_math<kOut, kTrans>(p, acc, v, row, col0);
            if constexpr (kTrans && kCols == 32 && kOut != OUT_F32) {
                // The warp's whole block inside C (warp-uniform): 16-byte stores through the staging buffer
                // (f32 rows are already written 128 bytes per warp instruction).
                if (p.c_vec_ok && row0 + 32 <= p.M && col0 + 32 <= p.N) {
                    store_block_trans_staged<kOut>(p, v, row0, col0, lane, stage_buf);
                    continue;
                }
            }
            store_row_direct<kOut, kTrans>(p, v, row, col0);
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

// Each stream-K flag has one consumer, which sets it back to 0 once it has the partial: the next
// launch then finds every flag at 0 whatever its epoch, so replaying a launch with the same epoch
// (a CUDA graph) cannot see a stale flag.
__device__ __forceinline__ void clear_flag(unsigned* flag) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(flag), "r"(0u) : "memory");
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
// rounded to f16.  A stage covers 128 K = four blocks of each B row.  Lane l of a dequantisation
// warp works on block l / 8 of rows (l % 8) + 8 * pass, so a warp's loads cover the 72 contiguous
// stage bytes of eight rows and each 8-lane phase of its stores one K chunk of eight rows.
constexpr int kQ4RegStages = 2;        // stages of raw blocks held in registers (loaded this many stages early)

// The lane's blocks of one stage (one per pass) exactly as loaded (rows 4-byte aligned, so a block starts 0
// or 2 bytes past a 4-byte boundary, which is the parity of its index):
//   even block: w[0..3] = bytes 0..15, w[4] = bytes 16..17;
//   odd block:  w[0] = bytes 0..1 (the scale), w[1..4] = bytes 2..17 (the nibbles).
// A block outside the matrix is all zero: scale 0, so every weight is 0.
constexpr int kQ4Passes = 2;           // B rows per dequantisation lane per stage (8 warps x 8 rows per pass)

struct Q4Raw {
    uint32_t w[kQ4Passes][5];
};

__device__ __forceinline__ void q4_load_raw(const KernelParams& p, const int (&rows)[kQ4Passes], int blk, Q4Raw& r) {
    const bool odd = (blk & 1) != 0;
#pragma unroll
    for (int ps = 0; ps < kQ4Passes; ++ps) {
        if (rows[ps] < p.N && blk < p.kblocks) {
            const uint8_t* b = p.bq + static_cast<long long>(rows[ps]) * p.ldbq + static_cast<long long>(blk) * 18;
            if (!odd) {
                const uint32_t* w = reinterpret_cast<const uint32_t*>(b);
                r.w[ps][0] = __ldg(w);
                r.w[ps][1] = __ldg(w + 1);
                r.w[ps][2] = __ldg(w + 2);
                r.w[ps][3] = __ldg(w + 3);
                r.w[ps][4] = __ldg(reinterpret_cast<const uint16_t*>(b + 16));
            } else {
                const uint32_t* w = reinterpret_cast<const uint32_t*>(b + 2);
                r.w[ps][0] = __ldg(reinterpret_cast<const uint16_t*>(b));
                r.w[ps][1] = __ldg(w);
                r.w[ps][2] = __ldg(w + 1);
                r.w[ps][3] = __ldg(w + 2);
                r.w[ps][4] = __ldg(w + 3);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 5; ++i) r.w[ps][i] = 0u;
        }
    }
}

// d * (nibble - 8) for the nibbles of two packed bytes (in bits 0..3 and 16..19 of x, other bits
// ignored), as f16x2: 0x6400 | q is the f16 1024 + q, minus 1032 is q - 8 exactly, and the product
// with d is one correctly rounded f16 multiplication.
__device__ __forceinline__ uint32_t q4_two(uint32_t x, __half2 d2) {
    const uint32_t biased = (x & 0x000F000Fu) | 0x64006400u;
    __half2 h = *reinterpret_cast<const __half2*>(&biased);
    h = __hsub2(h, __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6408u))));   // - 1032
    h = __hmul2(h, d2);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// The lane's blocks converted to f16, ready to store: per pass 16 words = four 16-byte pieces
// (piece 0 holds weights 0..7, the low nibbles of bytes 0..7; piece 1 weights 8..15; pieces 2
// and 3 the high nibbles of the same bytes, weights 16..31).
struct Q4Half {
    uint32_t v[kQ4Passes][16];
};

__device__ __forceinline__ void q4_convert(const Q4Raw& r, bool odd, Q4Half& h) {
#pragma unroll
    for (int ps = 0; ps < kQ4Passes; ++ps) {
        uint32_t dbits, q[4];
        if (!odd) {
            dbits = r.w[ps][0] & 0xffffu;
            q[0] = __byte_perm(r.w[ps][0], r.w[ps][1], 0x5432u);
            q[1] = __byte_perm(r.w[ps][1], r.w[ps][2], 0x5432u);
            q[2] = __byte_perm(r.w[ps][2], r.w[ps][3], 0x5432u);
            q[3] = __byte_perm(r.w[ps][3], r.w[ps][4], 0x5432u);
        } else {
            dbits = r.w[ps][0];
            q[0] = r.w[ps][1];
            q[1] = r.w[ps][2];
            q[2] = r.w[ps][3];
            q[3] = r.w[ps][4];
        }
        const __half2 d2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(dbits)));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t sh = q[i] >> 4;   // byte k's high nibble now in its low nibble
            h.v[ps][2 * i] = q4_two(__byte_perm(q[i], 0u, 0x4140u), d2);
            h.v[ps][2 * i + 1] = q4_two(__byte_perm(q[i], 0u, 0x4342u), d2);
            h.v[ps][8 + 2 * i] = q4_two(__byte_perm(sh, 0u, 0x4140u), d2);
            h.v[ps][8 + 2 * i + 1] = q4_two(__byte_perm(sh, 0u, 0x4342u), d2);
        }
    }
}

// Write the converted blocks into the stage's K-major, 128-byte-swizzled B tile: row `row0 + 8 *
// pass` (0..127), block b (0..3) = 32 K = 16-byte pieces 4*(b%2)..+3 of the 64-wide chunk b/2.
__device__ __forceinline__ void q4_store(uint32_t sb, int row0, int b, const Q4Half& h, uint32_t chunk_bytes) {
#pragma unroll
    for (int ps = 0; ps < kQ4Passes; ++ps) {
        const int row = row0 + 8 * ps;
        const uint32_t base = sb + static_cast<uint32_t>(b >> 1) * chunk_bytes + static_cast<uint32_t>(row) * 128u;
        const uint32_t sw = static_cast<uint32_t>(row) & 7u;
        const uint32_t pb = 4u * static_cast<uint32_t>(b & 1);
#pragma unroll
        for (int pc = 0; pc < 4; ++pc)
            st_shared_v4(base + (((pb + static_cast<uint32_t>(pc)) ^ sw) * 16u), h.v[ps][4 * pc], h.v[ps][4 * pc + 1],
                         h.v[ps][4 * pc + 2], h.v[ps][4 * pc + 3]);
    }
}

// A walk over one cluster's (unit, k-tile) stages in the order every role uses.
struct StageWalk {
    UnitIter units;
    Unit u;
    int i;        // stage index inside the unit
    int kt;       // its k-tile
    bool valid;
    __device__ __forceinline__ void init(const KernelParams& p, int cluster, int num_clusters) {
        units.init(p, cluster, num_clusters);
        valid = units.next(p, u);
        i = 0;
        kt = valid ? u.kt_at(0) : 0;
    }
    __device__ __forceinline__ void advance(const KernelParams& p) {
        if (++i >= u.k1 - u.k0) {
            valid = units.next(p, u);
            i = 0;
        }
        kt = valid ? u.kt_at(i) : 0;
    }
};

// ---------------------------------------------------------------- the kernel
// kCtaGroup == 2: a cluster is one 2-SM pair; rank 0 issues the MMAs for both CTAs.
// kQ4: B is Q4_0-quantised; dequantisation warps (after the epilogue warps) write each stage's
// B tile into shared memory instead of the producer's TMA copies.
// kElt == 1: 8-bit float operands (E4M3 / E5M2), both K-major, multiplied by kind::f8f6f4 MMAs.
template <int kCtaGroup, int kBN, int kStages, int kBK, int kOut, bool kQ4 = false, int kElt = 2>
__global__ void __launch_bounds__(TileConfig<kCtaGroup, kBN, kStages, kBK, kQ4, kElt>::kThreads, kQ4 ? 1 : 0)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const KernelParams p) {
    using Cfg = TileConfig<kCtaGroup, kBN, kStages, kBK, kQ4, kElt>;
    static_assert(Cfg::kRingBytes >= Cfg::kEpiWarps * kFixBufs * static_cast<int>(kFixPieceBytes),
                  "the head fix-up stages its pieces in the operand ring");
    constexpr int kClusterCtas = kCtaGroup;
    constexpr int kClusterRows = Cfg::kBM * kClusterCtas;      // output rows of one cluster tile
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages];
    __shared__ __align__(8) uint64_t bar_empty[kStages];
    __shared__ __align__(8) uint64_t bar_tfull[2];
    __shared__ __align__(8) uint64_t bar_tempty[2];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ __align__(8) uint64_t bar_fix[Cfg::kEpiWarps * kFixBufs];   // stream-K head fix-up pieces
    __shared__ __align__(8) uint64_t bar_cin[Cfg::kEpiWarps];              // C_in boxes (beta != 0, TMA path)
    __shared__ __align__(8) uint64_t bar_rsx[Cfg::kEpiWarps];              // rs_cluster: blocks in / owner ready
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (kClusterCtas > 1) ? cluster_ctarank() : 0u;
    const uint32_t prank = rank;                                           // rank within the 2-SM pair
    const uint32_t lrank = 0;                                              // MMA-issuing CTA of the pair
    const int cluster_id = blockIdx.x / kClusterCtas;
    const int num_clusters = gridDim.x / kClusterCtas;
    const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t epi_smem = ring + Cfg::kRingBytes;
    volatile int* abort_flag = &s_abort;

    // The TMA copies of one operand stage -- k-tile kt of output tile (mb, nb) -- into sa / sb, completing on
    // full_bar; with `prefetch` the same boxes are only brought into L2.
    auto stage_copies = [&](int mb, int nb, int kt, uint32_t sa, uint32_t sb, uint32_t full_bar, bool prefetch) {
        const int m0 = mb * kClusterRows + static_cast<int>(rank) * Cfg::kBM;
        const int k0 = kt * Cfg::kBK;
        auto load = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1) {
            if (prefetch) tma_prefetch_2d(map, c0, c1);
            else if constexpr (kCtaGroup == 2) tma_load_2d_pair(dst, map, c0, c1, full_bar);
            else tma_load_2d(dst, map, c0, c1, full_bar);
        };
        auto load3 = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2) {
            if (prefetch) tma_prefetch_3d(map, c0, c1, c2);
            else if constexpr (kCtaGroup == 2) tma_load_3d_pair(dst, map, c0, c1, c2, full_bar);
            else tma_load_3d(dst, map, c0, c1, c2, full_bar);
        };
        if (!p.a_mn) {
            if (p.a_3d) {
                load3(sa, &tmA, 0, m0, kt * Cfg::kKChunks);   // box {64, 128 M, K chunks}
            } else {
#pragma unroll
                for (int c = 0; c < Cfg::kKChunks; ++c)  // box {one swizzle span of K, 128 M} per chunk
                    load(sa + static_cast<uint32_t>(c * Cfg::kAChunkBytes), &tmA, k0 + Cfg::kKChunkElems * c, m0);
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
        } else {
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
                        for (int c = 0; c < Cfg::kKChunks; ++c)  // box {one span of K, kHalfCols N} per chunk
                            load(sb + static_cast<uint32_t>(c * Cfg::kBChunkBytes + h * Cfg::kHalfCols * 128),
                                 &tmB, k0 + Cfg::kKChunkElems * c, nh);
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
        }
    };
    if (threadIdx.x == (kQ4 ? 0 : 64)) {
        // The first ring of operand stages of this cluster's first unit into L2 before anything else: the
        // kernel before this one on the stream may still be running (the waits below come later), and the
        // loads of these stages then hit L2.  Lane 0 of the first epilogue warp issues them, so that thread 0
        // initialises the barriers at once and the set-up barrier releases sooner (with Q4_0 B thread 0 does,
        // whose kernel has no registers to spare for it in the epilogue warps).
        UnitIter first_units;
        first_units.init(p, cluster_id, num_clusters);
        Unit fu;
        if (first_units.next(p, fu)) {
            int mb, nb;
            tile_coords(p, fu.tile, mb, nb);
            const int n = min(kStages, fu.k1 - fu.k0);
            for (int i = 0; i < n; ++i) stage_copies(mb, nb, fu.kt_at(i), 0u, 0u, 0u, true);
        }
    }
    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < kStages; ++s) {
            // The producer's arrive (with the TMA byte count), plus one arrive from the dequantisation
            // warps of every CTA of the pair when B is dequantised in shared memory.
            mbar_init(smem_u32(&bar_full[s]), 1 + (kQ4 ? kCtaGroup : 0));
            mbar_init(smem_u32(&bar_empty[s]), 1);        // one commit from the pair's MMA issuer
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_tfull[b]), 1);
            mbar_init(smem_u32(&bar_tempty[b]), Cfg::kEpiWarps * kCtaGroup);
        }
        mbar_init(smem_u32(&bar_drain), 1);
        for (int b = 0; b < Cfg::kEpiWarps * kFixBufs; ++b) mbar_init(smem_u32(&bar_fix[b]), 1);
        for (int b = 0; b < Cfg::kEpiWarps; ++b) mbar_init(smem_u32(&bar_cin[b]), 1);
        for (int b = 0; b < Cfg::kEpiWarps; ++b) mbar_init(smem_u32(&bar_rsx[b]), 1);
        fence_barrier_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (p.use_tma_store) prefetch_tensormap(&tmC);
    }
    if (warp == 1) {
        __syncwarp();    // tcgen05.alloc is .aligned: the whole warp, converged (lane 0 prefetched alone above)
        tmem_alloc<kCtaGroup>(smem_u32(&s_tmem_base), Cfg::kTmemCols);
    }
    tc_fence_before_sync();
    cta_sync_all();
    if constexpr (kClusterCtas > 1) cluster_sync();
    else if (p.rs_cluster) cluster_sync();      // the other parts arrive on this CTA's barriers
    tc_fence_after_sync();
    const uint32_t tmem_base = s_tmem_base;
    // The set-up above touched no global memory; everything below may read what the previous kernel
    // on the stream wrote, or overwrite what it reads.
    griddep_launch_dependents();
    griddep_wait();

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
                for (int i = 0; i < u.k1 - u.k0; ++i) {
                    const int kt = u.kt_at(i);
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
                        stage_copies(mb, nb, kt, sa, sb, full_bar, false);
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
            // (An MMA covers 32 bytes of K in either input width, so 4 MMAs span one 128-byte chunk.)
            uint64_t a_koff[Cfg::kMmasPerStage], b_koff[Cfg::kMmasPerStage], b_hoff[Cfg::kNHalves];
#pragma unroll
            for (int k = 0; k < Cfg::kMmasPerStage; ++k) {
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
                for (int i = 0; i < u.k1 - u.k0; ++i) {
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
                    for (int k = 0; k < Cfg::kMmasPerStage; ++k)
#pragma unroll
                        for (int h = 0; h < Cfg::kNHalves; ++h) {
                            const uint32_t dt = d_tmem + static_cast<uint32_t>(h * Cfg::kMmaN);
                            const uint32_t accum = (i > 0 || k > 0) ? 1u : 0u;
                            if constexpr (kElt == 1) mma_f8<kCtaGroup>(dt, ad + a_koff[k], bd + b_hoff[h] + b_koff[k], p.idesc, accum);
                            else mma_f16<kCtaGroup>(dt, ad + a_koff[k], bd + b_hoff[h] + b_koff[k], p.idesc, accum);
                        }
                    mma_commit_pair<kCtaGroup>(smem_u32(&bar_empty[stage]), 1u);  // slot free in both CTAs
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair<kCtaGroup>(smem_u32(&bar_tfull[acc]), 1u);  // accumulator ready
                if (++acc == static_cast<uint32_t>(Cfg::kAccBufs)) { acc = 0; acc_phase ^= 1u; }
            }
            // Drain: every MMA this thread issued has completed once bar_drain flips.  This wait
            // ignores the abort flag (only the time limit ends it): TMEM is freed after it.
            mma_commit_pair<kCtaGroup>(smem_u32(&bar_drain), 1u);
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
        // The slice of the operand ring this warp may use once the ring is idle (its cluster's last unit).
        constexpr uint32_t kRingSlice = (static_cast<uint32_t>(Cfg::kRingBytes) / Cfg::kEpiWarps) & ~4095u;
        constexpr int kCinBoxes = Cfg::kEpiCols / ((kOut == OUT_F32) ? 32 : 64);
        constexpr bool kRingCin = kRingSlice >= static_cast<uint32_t>(kCinBoxes) * 4096u;
        const uint32_t ring_slice = ring + static_cast<uint32_t>(ew) * kRingSlice;
        UnitIter units;
        units.init(p, cluster_id, num_clusters);
        Unit u, u_next;
        bool have = units.next(p, u);
        while (have) {
            const bool more = units.next(p, u_next);
            int mb, nb;
            tile_coords(p, u.tile, mb, nb);
            const int row0 = mb * kClusterRows + static_cast<int>(rank) * Cfg::kBM + quarter * 32;
            if (p.beta != 0.0f && u.kind != UNIT_TAIL) {        // C_in into L2 while the MMAs run
                if (!p.c_trans) prefetch_c_rows<kOut, Cfg::kEpiCols>(p, row0 + lane, nb * kBN + pcol0);
                else prefetch_c_block_trans<kOut, Cfg::kEpiCols>(p, row0, nb * kBN + pcol0, lane);
            }
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
            uint32_t parts_smem = 0;   // rs_cluster owner: the other parts' blocks, 4 KB per part
            int parts = 0, self_part = 0;
            bool sent = false;         // rs_cluster: this warp's block went to its owner; no C block here
            if (kCtaGroup == 1 && !kQ4 && Cfg::kEpiCols == 32 && p.rs_cluster && p.sk_rs > 1 && u.kind != UNIT_FULL) {
                // The S parts of the tile are the S CTAs of this thread-block cluster.  The owner of
                // warp ew's block is part ew * S / warps; its owner warps take S x 4 KB each of its ring.
                const int S = p.sk_rs;
                const uint32_t r = cluster_ctarank();
                const int per_owner = Cfg::kEpiWarps / S;
                const uint32_t owner = static_cast<uint32_t>(ew / per_owner);
                const uint32_t region = ring + static_cast<uint32_t>(ew - static_cast<int>(owner) * per_owner) *
                                                   static_cast<uint32_t>(S) * 4096u;
                const uint32_t bar = smem_u32(&bar_rsx[ew]);
                bool ready;
                if (owner == r) {
                    if (lane == 0) {
                        // Arm for the S - 1 blocks, then tell the same warp of every other part that
                        // this slice of the idle ring may be written.
                        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(S - 1) * 4096u);
                        for (int j = 0; j < S; ++j)
                            if (j != static_cast<int>(r)) mbar_arrive_cluster(mapa_shared(bar, static_cast<uint32_t>(j)));
                    }
                    ready = mbar_wait_bounded<true>(bar, 0u, p.timeout_ns, abort_flag);
                    parts_smem = region;
                    parts = S;
                    self_part = static_cast<int>(r);
                } else {
                    // Wait for the owner's word, then store the block into its slot of the owner's slice.
                    ready = mbar_wait_bounded<true>(bar, 0u, p.timeout_ns, abort_flag);
                    if (__all_sync(0xffffffffu, ready)) {
                        uint32_t a[32];
                        tmem_ld_32x32b_x32(tbase, a);
                        tmem_wait_ld();
                        const uint32_t slot = region + r * 4096u + static_cast<uint32_t>(lane) * 16u;
                        const uint32_t rbar = mapa_shared(bar, owner);
#pragma unroll
                        for (int q = 0; q < 8; ++q)    // [quad][lane][4 f32], as the owner reads it
                            st_async_v4(mapa_shared(slot + static_cast<uint32_t>(q) * 512u, owner), a[4 * q], a[4 * q + 1],
                                        a[4 * q + 2], a[4 * q + 3], rbar);
                        sent = true;
                    }
                }
                if (!__all_sync(0xffffffffu, ready)) {
                    if (lane == 0 && !*abort_flag)
                        report_error<kClusterCtas>(p, ROLE_EPILOGUE, u.tile, 300 + quarter, abort_flag);
                    break;
                }
            } else if (p.sk_rs > 1 && u.kind != UNIT_FULL) {
                // Reduce-scatter split (one unit per cluster, parts of a tile in consecutive clusters).
                const int S = p.sk_rs;
                const int r = cluster_id % S;
                if (ew * S / Cfg::kEpiWarps != r) {
                    out_part = p.sk_partials + static_cast<size_t>(cluster_id) * slot_floats + warp_block;
                } else {
                    const int c0 = cluster_id - r;
                    bool ready = true;
                    for (int src = c0; src < c0 + S; ++src) {
                        if (src == cluster_id) continue;
                        const unsigned* flag =
                            p.sk_flags + (static_cast<size_t>(src) * kClusterCtas + rank) * Cfg::kEpiWarps + ew;
                        if (lane == 0 && ready) ready = wait_flag_bounded(flag, p.epoch, p.timeout_ns, abort_flag);
                    }
                    ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
                    if (ready) {
                        ready = head_fixup<Cfg::kEpiCols>(
                            tbase, lane, p.sk_partials + static_cast<size_t>(c0) * slot_floats + warp_block, S - 1,
                            slot_floats, ring + static_cast<uint32_t>(ew) * kFixBufs * kFixPieceBytes,
                            smem_u32(&bar_fix[ew * kFixBufs]), p.timeout_ns, abort_flag, r);
                    }
                    if (ready && lane == 0) {
                        for (int src = c0; src < c0 + S; ++src)
                            if (src != cluster_id)
                                clear_flag(p.sk_flags + (static_cast<size_t>(src) * kClusterCtas + rank) * Cfg::kEpiWarps + ew);
                    }
                    if (!ready) {
                        if (lane == 0 && !*abort_flag)
                            report_error<kClusterCtas>(p, ROLE_EPILOGUE, u.tile, 300 + quarter, abort_flag);
                        break;
                    }
                }
            } else if (u.kind == UNIT_TAIL) {
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
                if (ready && lane == 0) {
                    for (int src = cluster_id + 1; src < cluster_id + 1 + n; ++src)
                        clear_flag(p.sk_flags + (static_cast<size_t>(src) * kClusterCtas + rank) * Cfg::kEpiWarps + ew);
                }
                if (!ready) {
                    if (lane == 0 && !*abort_flag)
                        report_error<kClusterCtas>(p, ROLE_EPILOGUE, u.tile, 300 + quarter, abort_flag);
                    break;
                }
            }
            bool drained;
            if (sent)
                drained = true;
            else if (!kQ4 && p.c_trans)     // (the transposed product never takes Q4_0 weights)
                drained = epilogue_tile<kOut, Cfg::kEpiCols, !kQ4>(p, &tmC, tbase, row0, nb * kBN + pcol0, lane, stage_buf,
                                                                   out_part, smem_u32(&bar_cin[ew]), &cin_uses, abort_flag,
                                                                   0u, parts_smem, parts, self_part);
            else
                drained = epilogue_tile<kOut, Cfg::kEpiCols, false, kQ4>(p, &tmC, tbase, row0, nb * kBN + pcol0, lane, stage_buf,
                                                             out_part, smem_u32(&bar_cin[ew]), &cin_uses, abort_flag,
                                                             (kRingCin && !more) ? ring_slice : 0u);
            if (!drained) {
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
                if (out_part != nullptr) {
                    // Every lane's partial stores precede this release: the warp barrier above orders
                    // them before it, and a release is cumulative.
                    st_release_gpu(p.sk_flags + (static_cast<size_t>(cluster_id) * kClusterCtas + rank) * Cfg::kEpiWarps + ew,
                                   p.epoch);
                }
            }
            if (++acc == static_cast<uint32_t>(Cfg::kAccBufs)) { acc = 0; acc_phase ^= 1u; }
            u = u_next;
            have = more;
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    } else if constexpr (kQ4) {
        // ------------------------------------------------------------ Q4_0 dequantisation warps
        // Warp dw covers B rows dw * 16 .. +15 of this CTA's 128 (output columns); lane l takes block
        // l % 4 of rows dw * 16 + l / 4 + 8 * pass.  Two walks over the same stages: `conv` is the
        // next stage to store, `load` runs kQ4RegStages further ahead filling raw register buffers.
        // (An L2 prefetch walk further ahead was measured to slow the loop down.)  Each stage is converted
        // into registers while the MMA still works on earlier stages; once its slot is free only the
        // shared-memory stores, a fence, a barrier among the four warps and one arrive remain.
        static_assert(Cfg::kDqWarps * 8 * kQ4Passes == Cfg::kBNC, "every B row of the CTA has one lane group");
        const int dw = warp - 2 - Cfg::kEpiWarps;
        // Lanes 8j..8j+7 take block j of eight consecutive rows: each 8-lane phase of a 16-byte
        // shared store then covers eight rows of one K chunk, whose swizzled pieces are all distinct.
        const int row0 = dw * 8 * kQ4Passes + (lane & 7);
        const int bl = lane >> 3;
        // The rows of a unit change only with its tile: keep the last tile's answer.
        int memo_tile = -1, memo_n0 = 0;
        auto rows_of = [&](const Unit& uu, int (&rows)[kQ4Passes]) {
            if (uu.tile != memo_tile) {
                int mb, nb;
                tile_coords(p, uu.tile, mb, nb);
                memo_tile = uu.tile;
                memo_n0 = nb * kBN + static_cast<int>(prank) * Cfg::kBNC + row0;
            }
#pragma unroll
            for (int ps = 0; ps < kQ4Passes; ++ps) rows[ps] = memo_n0 + 8 * ps;
        };
        StageWalk conv, load;
        conv.init(p, cluster_id, num_clusters);
        load.init(p, cluster_id, num_clusters);
        auto load_one = [&](Q4Raw& r) {
            if (!load.valid) return;
            int rows[kQ4Passes];
            rows_of(load.u, rows);
            q4_load_raw(p, rows, load.kt * 4 + bl, r);
            load.advance(p);
        };
        Q4Raw r0, r1;
        Q4Half h;
        load_one(r0);
        load_one(r1);
        const bool odd = (bl & 1) != 0;
        if (conv.valid) q4_convert(r0, odd, h);
        load_one(r0);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        // Store the converted stage, then convert the one held in `next` and refill `next`.
        auto store_one = [&](Q4Raw& next) {
            if (!ok || !conv.valid) return;
            const bool got = mbar_wait_bounded(smem_u32(&bar_empty[stage]), phase ^ 1u, p.timeout_ns, abort_flag);
            // Every wait above is bounded, so all four warps reach this barrier; it ANDs their
            // outcomes so that they leave together on a failure (none is left at a barrier).
            uint32_t all_got;
            asm volatile("{\n\t.reg .pred pin, pout;\n\t"
                         "setp.ne.u32 pin, %1, 0;\n\t"
                         "barrier.red.and.pred pout, 1, %2, pin;\n\t"
                         "selp.u32 %0, 1, 0, pout;\n\t}"
                         : "=r"(all_got) : "r"(got ? 1u : 0u), "n"(Cfg::kDqWarps * 32) : "memory");
            if (!all_got) {
                if (lane == 0 && !got && !*abort_flag)
                    report_error<kClusterCtas>(p, ROLE_PRODUCER, conv.u.tile, 500 + static_cast<int>(stage), abort_flag);
                ok = false;
                return;
            }
            q4_store(ring + stage * Cfg::kStageBytes + Cfg::kABytes, row0, bl, h, Cfg::kBChunkBytes);
            // This CTA's generic shared-memory writes -> the MMA's async-proxy reads.
            fence_proxy_async_smem();
            // The four dequantisation warps of this CTA meet (no exit path lies between the barrier
            // above and this one); one thread arrives for all of them.
            asm volatile("barrier.sync 1, %0;" :: "n"(Cfg::kDqWarps * 32) : "memory");
            if (dw == 0 && lane == 0) {
                const uint32_t full_local = smem_u32(&bar_full[stage]);
                if constexpr (kCtaGroup == 2) {
                    if (prank == 0) mbar_arrive_local(full_local);
                    else mbar_arrive_cluster(mapa_shared(full_local, lrank));
                } else {
                    mbar_arrive_local(full_local);
                }
            }
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
            conv.advance(p);
            if (conv.valid) q4_convert(next, odd, h);
            load_one(next);
        };
        static_assert(kQ4RegStages == 2, "two rotating raw register buffers");
        while (ok && conv.valid) {
            store_one(r1);
            store_one(r0);
        }
    }

    // ---------------------------------------------------------------- teardown
    if (threadIdx.x == 0 && *abort_flag) {
        // A bounded settle so copies issued before the abort land before shared memory goes away.
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 200000ull) { }
    }
    tc_fence_before_sync();
    cta_sync_all();
    if constexpr (kClusterCtas > 1) cluster_sync();
    else if (p.rs_cluster) cluster_sync();      // no part leaves while another may still write into it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<kCtaGroup>(tmem_base, Cfg::kTmemCols);
    }
}

}  // namespace gb300

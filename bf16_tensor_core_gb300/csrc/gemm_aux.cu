// Auxiliary kernels around the tcgen05 GEMM:
//  * repack of a 16-bit operand whose byte pitch is not a multiple of 16 into a workspace with a
//    16-byte pitch (TMA tensor maps require 16-byte-multiple strides);
//  * the K == 0 epilogue, C = beta * C + bias (the product of an empty sum is zero).
#include <algorithm>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"
#include "gemm_launch.h"
#include "q4_block.cuh"

namespace gb300 {

// Copy rows x cols blocks of 16-bit elements from pitch `lds` to a pitch `ldd` that is a multiple
// of 8 elements (16 bytes) on a 16-byte-aligned destination; destination columns [cols, ldd) are
// zero-filled.  Both jobs of a launch share one flat space of work items (a row segment of
// 32 x kRepackChunks destination chunks of 16 bytes).  The source row starts o bytes past a 16-byte
// boundary (o even); lane l reads the aligned 16-byte source chunk under its destination chunk with one
// vector load, takes the following aligned chunk from lane l + 1 by a shuffle (lane 31 loads it), and
// shifts the 32 bytes right by o.  All of a lane's loads are issued before any is used.  An aligned
// chunk is read only when it holds at least one byte of the row, so every load stays inside the
// 16-byte granules of the source rows.
constexpr int kRepackChunks = 4;   // destination chunks per lane per work item

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Bytes [o, o + 16) of the 32 bytes lo:hi (little-endian words), o even and below 16.
__device__ __forceinline__ uint4 shift_right_bytes(const uint4& lo, const uint4& hi, uint32_t o) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const uint32_t sh = (o & 3u) * 8u;   // 0 or 16
    uint32_t r[4];
    switch (o >> 2) {                     // uniform across the warp (one row per work item)
#define GB300_REPACK_CASE(WS)                                                               \
        case WS:                                                                            \
            _Pragma("unroll") for (int i = 0; i < 4; ++i) r[i] = __funnelshift_r(w[i + WS], w[i + WS + 1], sh); \
            break;
        GB300_REPACK_CASE(0)
        GB300_REPACK_CASE(1)
        GB300_REPACK_CASE(2)
        default:
        GB300_REPACK_CASE(3)
#undef GB300_REPACK_CASE
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

__global__ void __launch_bounds__(256) repack_u16_kernel(RepackJobs jobs, long long items0, long long items) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
    constexpr int kSeg = 32 * kRepackChunks;                   // destination chunks per work item
    for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5); w < items;
         w += warps) {
        const bool second = w >= items0;
        const RepackJob j = second ? jobs.job[1] : jobs.job[0];   // (no dynamic index into the parameter)
        const long long wi = second ? w - items0 : w;
        const long long chunks = j.ldd / 8;
        const long long segs = (chunks + kSeg - 1) / kSeg;
        const long long r = wi / segs;
        const long long seg0 = (wi - r * segs) * kSeg;
        const char* row = reinterpret_cast<const char*>(j.src + r * j.lds);
        const uint32_t o = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(row) & 15u);
        const char* base = row - o;                            // 16-byte aligned
        const long long row_bytes = 2 * j.cols;                // valid source bytes of the row
        const long long valid = o + row_bytes;                 // ... measured from `base`
        uint4 cur[kRepackChunks], nxt[kRepackChunks];
#pragma unroll
        for (int u = 0; u < kRepackChunks; ++u) {
            const long long c = seg0 + u * 32 + lane;          // destination chunk
            cur[u] = make_uint4(0u, 0u, 0u, 0u);
            nxt[u] = make_uint4(0u, 0u, 0u, 0u);
            // (also for c == chunks: lane l - 1 takes that chunk's bytes when the row is misaligned)
            if (16 * c < valid) cur[u] = ld_nc_v4(base + 16 * c);
            if (lane == 31 && c < chunks && 16 * (c + 1) < valid && o != 0) nxt[u] = ld_nc_v4(base + 16 * (c + 1));
        }
#pragma unroll
        for (int u = 0; u < kRepackChunks; ++u) {
            const long long c = seg0 + u * 32 + lane;
            uint4 hi;
            hi.x = __shfl_down_sync(0xffffffffu, cur[u].x, 1);
            hi.y = __shfl_down_sync(0xffffffffu, cur[u].y, 1);
            hi.z = __shfl_down_sync(0xffffffffu, cur[u].z, 1);
            hi.w = __shfl_down_sync(0xffffffffu, cur[u].w, 1);
            if (lane == 31) hi = nxt[u];
            if (c >= chunks) continue;
            uint4 v = o != 0 ? shift_right_bytes(cur[u], hi, o) : cur[u];
            const long long e0 = 8 * c;                        // first element of the chunk
            if (e0 + 8 > j.cols) {                             // zero the elements at and past `cols`
                const long long keep = j.cols > e0 ? j.cols - e0 : 0;   // 0..7 elements
                uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const long long k0 = 2 * i;
                    if (k0 >= keep) wds[i] = 0u;
                    else if (k0 + 1 >= keep) wds[i] &= 0xffffu;
                }
                v = make_uint4(wds[0], wds[1], wds[2], wds[3]);
            }
            *reinterpret_cast<uint4*>(j.dst + r * j.ldd + e0) = v;
        }
    }
}

cudaError_t launch_repack_u16(const RepackJobs& jobs, int num_sms, cudaStream_t stream, bool pdl) {
    if (jobs.n <= 0) return cudaSuccess;
    long long counts[2] = {0, 0};
    for (int i = 0; i < jobs.n; ++i) {
        const RepackJob& j = jobs.job[i];
        if (j.ldd % 8 != 0 || j.ldd < j.cols || (reinterpret_cast<uintptr_t>(j.dst) & 15u) != 0 ||
            (reinterpret_cast<uintptr_t>(j.src) & 1u) != 0)
            return cudaErrorInvalidValue;
        counts[i] = j.rows * ((j.ldd / 8 + 32 * kRepackChunks - 1) / (32 * kRepackChunks));
    }
    const long long items = counts[0] + counts[1];
    if (items <= 0) return cudaSuccess;
    // 64 registers per thread: four 256-thread blocks fit on an SM, and the grid is one such wave.
    long long blocks = (items + 7) / 8;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 152) * 4;
    if (blocks > cap) blocks = cap;
    return launch_ex(repack_u16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pdl, jobs,
                     counts[0], items);
}

// Q4_0 weights -> f16 ("02 . 8m/8m(2) -- Tiled wmma f16 prefill GEMM", section 3.2: an f16 scale d
// and 16 bytes per 32 weights; weight i is the low nibble of byte i, weight 16+i its high nibble;
// value d * (q - 8) formed in f32, exact, then rounded to f16).  One thread per block.
__global__ void __launch_bounds__(256) dequant_q4_0_kernel(const uint8_t* __restrict__ bq, long long ldbq,
                                                           long long N, long long nblocks, __half* __restrict__ out,
                                                           long long ldo) {
    griddep_launch_dependents();
    griddep_wait();
    const long long total = N * nblocks;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < total; g += stride) {
        const long long n = g / nblocks, b = g - n * nblocks;
        const uint16_t* h = reinterpret_cast<const uint16_t*>(bq + n * ldbq + b * 18);
        const float d = __half2float(__ushort_as_half(__ldg(h)));
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t two = __ldg(h + 1 + i);                  // bytes 2i (low) and 2i+1 (high)
            const uint32_t b0 = two & 0xffu, b1 = two >> 8;
            // weights 2i, 2i+1 from the low nibbles; 16+2i, 16+2i+1 from the high nibbles
            const __half2 lo = __floats2half2_rn(d * static_cast<float>(static_cast<int>(b0 & 15u) - 8),
                                                 d * static_cast<float>(static_cast<int>(b1 & 15u) - 8));
            const __half2 hi = __floats2half2_rn(d * static_cast<float>(static_cast<int>(b0 >> 4) - 8),
                                                 d * static_cast<float>(static_cast<int>(b1 >> 4) - 8));
            packed[i] = *reinterpret_cast<const uint32_t*>(&lo);
            packed[8 + i] = *reinterpret_cast<const uint32_t*>(&hi);
        }
        __half* dst = out + n * ldo + b * 32;
        if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int j = 0; j < 4; ++j) d4[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
        } else if ((reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
            uint32_t* d32 = reinterpret_cast<uint32_t*>(dst);
#pragma unroll
            for (int j = 0; j < 16; ++j) d32[j] = packed[j];
        } else {
            uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                d16[2 * j] = static_cast<uint16_t>(packed[j] & 0xffffu);
                d16[2 * j + 1] = static_cast<uint16_t>(packed[j] >> 16);
            }
        }
    }
}

// The same pass for 16-byte aligned rows and output (the common case): warp w takes 32 consecutive
// blocks of one row at a time (576 bytes in, 2 KB out).  The input arrives with 16-byte loads into
// shared memory, lane l dequantises block l there (f16 1024 + q, minus 1032, times d: one rounding,
// the same value as above), and the 2 KB leave as 16-byte stores that cover it contiguously.
constexpr int kDqWarpsPerCta = 8;
constexpr int kDqStagePitch = 80;     // bytes per block in the staging buffer (64 + 16: no bank conflicts)

__global__ void __launch_bounds__(kDqWarpsPerCta * 32) dequant_q4_0_rows_kernel(const uint8_t* __restrict__ bq,
                                                                                 long long ldbq, long long N,
                                                                                 int nblocks, __half* __restrict__ out,
                                                                                 long long ldo) {
    __shared__ __align__(16) uint8_t raw[kDqWarpsPerCta][576];
    __shared__ __align__(16) uint8_t stage[kDqWarpsPerCta][32 * kDqStagePitch];
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gpr = (nblocks + 31) / 32;                    // groups of 32 blocks per row
    const long long groups = N * gpr;
    const uint32_t raw_s = static_cast<uint32_t>(__cvta_generic_to_shared(raw[warp]));
    for (long long g = static_cast<long long>(blockIdx.x) * kDqWarpsPerCta + warp; g < groups;
         g += static_cast<long long>(gridDim.x) * kDqWarpsPerCta) {
        const long long n = g / gpr;
        const int b0 = static_cast<int>(g - n * gpr) * 32;
        const int nb = min(32, nblocks - b0);
        const uint8_t* src = bq + n * ldbq + 18LL * b0;
        const int bytes = 18 * nb;
        const int full = bytes & ~15;
        for (int off = 16 * lane; off < full; off += 512)
            *reinterpret_cast<uint4*>(&raw[warp][off]) = __ldg(reinterpret_cast<const uint4*>(src + off));
        for (int off = full + 2 * lane; off < bytes; off += 64)
            *reinterpret_cast<uint16_t*>(&raw[warp][off]) = __ldg(reinterpret_cast<const uint16_t*>(src + off));
        __syncwarp();
        if (lane < nb) {
            uint32_t v[16];
            q4_block_weights(q4_block_shared(raw_s, lane), v);
            uint4* st = reinterpret_cast<uint4*>(&stage[warp][lane * kDqStagePitch]);
#pragma unroll
            for (int j = 0; j < 4; ++j) st[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        __syncwarp();
        uint4* dst = reinterpret_cast<uint4*>(out + n * ldo + 32LL * b0);
        for (int i = lane; i < 4 * nb; i += 32)
            dst[i] = *reinterpret_cast<const uint4*>(&stage[warp][(i >> 2) * kDqStagePitch + (i & 3) * 16]);
        __syncwarp();
    }
}

cudaError_t launch_dequant_q4_0(const void* bq, long long ldbq, long long N, long long K, void* out, long long ldo,
                                int num_sms, cudaStream_t stream, bool pdl) {
    const long long nblocks = K / 32;
    const long long total = N * nblocks;
    if (total <= 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(bq) & 15u) == 0 && ldbq % 16 == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0 &&
        ldo % 8 == 0 && nblocks < (1LL << 30)) {
        const long long groups = N * ((nblocks + 31) / 32);
        long long ctas = (groups + kDqWarpsPerCta - 1) / kDqWarpsPerCta;
        const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 152) * 8;
        if (ctas > cap) ctas = cap;
        return launch_ex(dequant_q4_0_rows_kernel, dim3(static_cast<unsigned>(ctas)), dim3(kDqWarpsPerCta * 32), 0,
                         stream, pdl, static_cast<const uint8_t*>(bq), ldbq, N, static_cast<int>(nblocks),
                         static_cast<__half*>(out), ldo);
    }
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 152) * 8;
    if (blocks > cap) blocks = cap;
    return launch_ex(dequant_q4_0_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pdl,
                     static_cast<const uint8_t*>(bq), ldbq, N, nblocks, static_cast<__half*>(out), ldo);
}

template <int kOut>
__global__ void scale_bias_kernel(void* C, long long ldc, const void* bias, float beta, long long M, long long N) {
    griddep_launch_dependents();
    griddep_wait();
    const long long total = M * N;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const long long r = i / N, c = i - r * N;
        const long long idx = r * ldc + c;
        float v = 0.0f;
        if (beta != 0.0f) v = beta * load_out<kOut>(C, idx);
        if (bias) v += load_out<kOut>(bias, c);
        if constexpr (kOut == OUT_F32) static_cast<float*>(C)[idx] = v;
        else if constexpr (kOut == OUT_F16) static_cast<__half*>(C)[idx] = __float2half_rn(v);
        else static_cast<__nv_bfloat16*>(C)[idx] = __float2bfloat16_rn(v);
    }
}

cudaError_t launch_scale_bias(int out, void* C, long long ldc, const void* bias, float beta, long long M,
                              long long N, int num_sms, cudaStream_t stream, bool pdl) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    long long blocks = (M * N + 255) / 256;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 152) * 8;
    if (blocks > cap) blocks = cap;
    const dim3 g(static_cast<unsigned>(blocks));
    switch (out) {
        case OUT_F16: return launch_ex(scale_bias_kernel<OUT_F16>, g, dim3(256), 0, stream, pdl, C, ldc, bias, beta, M, N);
        case OUT_BF16: return launch_ex(scale_bias_kernel<OUT_BF16>, g, dim3(256), 0, stream, pdl, C, ldc, bias, beta, M, N);
        case OUT_F32: return launch_ex(scale_bias_kernel<OUT_F32>, g, dim3(256), 0, stream, pdl, C, ldc, bias, beta, M, N);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300

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
// of 8 elements (16 bytes) on a 16-byte-aligned destination.  A warp moves 32 consecutive 16-byte
// destination chunks of one row; each chunk is read with the widest loads the source address allows
// (one 16-byte load, four 4-byte loads, or eight 2-byte loads) and written with one 16-byte store.
// Destination columns [cols, ldd) are zero-filled.  blockIdx.y selects the job (A or B).
__global__ void __launch_bounds__(256) repack_u16_kernel(RepackJobs jobs) {
    const RepackJob j = blockIdx.y == 0 ? jobs.job[0] : jobs.job[1];   // (no dynamic index into the parameter)
    const long long chunks = j.ldd / 8;
    const long long segs = (chunks + 31) / 32;
    const long long items = j.rows * segs;
    const int lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
    for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5); w < items;
         w += warps) {
        const long long r = w / segs;
        const long long chunk = (w - r * segs) * 32 + lane;
        if (chunk >= chunks) continue;
        const long long c0 = chunk * 8;
        const uint16_t* src = j.src + r * j.lds + c0;
        uint4 out;
        if (c0 + 8 <= j.cols) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(src);
            if ((a & 15u) == 0) {
                out = __ldg(reinterpret_cast<const uint4*>(src));
            } else if ((a & 3u) == 0) {
                const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src);
                out = make_uint4(__ldg(s32), __ldg(s32 + 1), __ldg(s32 + 2), __ldg(s32 + 3));
            } else {
                uint32_t wds[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    wds[i] = static_cast<uint32_t>(__ldg(src + 2 * i)) | (static_cast<uint32_t>(__ldg(src + 2 * i + 1)) << 16);
                out = make_uint4(wds[0], wds[1], wds[2], wds[3]);
            }
        } else {
            uint32_t wds[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (c0 + i < j.cols) wds[i / 2] |= static_cast<uint32_t>(__ldg(src + i)) << (16 * (i & 1));
            out = make_uint4(wds[0], wds[1], wds[2], wds[3]);
        }
        *reinterpret_cast<uint4*>(j.dst + r * j.ldd + c0) = out;
    }
}

cudaError_t launch_repack_u16(const RepackJobs& jobs, int num_sms, cudaStream_t stream) {
    if (jobs.n <= 0) return cudaSuccess;
    long long items = 0;
    for (int i = 0; i < jobs.n; ++i) {
        const RepackJob& j = jobs.job[i];
        if (j.ldd % 8 != 0 || j.ldd < j.cols || (reinterpret_cast<uintptr_t>(j.dst) & 15u) != 0 ||
            (reinterpret_cast<uintptr_t>(j.src) & 1u) != 0)
            return cudaErrorInvalidValue;
        items = std::max(items, j.rows * ((j.ldd / 8 + 31) / 32));
    }
    if (items <= 0) return cudaSuccess;
    long long blocks = (items + 7) / 8;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 152) * 8;
    if (blocks > cap) blocks = cap;
    repack_u16_kernel<<<dim3(static_cast<unsigned>(blocks), static_cast<unsigned>(jobs.n)), 256, 0, stream>>>(jobs);
    return cudaGetLastError();
}

// Q4_0 weights -> f16 ("02 . 8m/8m(2) -- Tiled wmma f16 prefill GEMM", section 3.2: an f16 scale d
// and 16 bytes per 32 weights; weight i is the low nibble of byte i, weight 16+i its high nibble;
// value d * (q - 8) formed in f32, exact, then rounded to f16).  One thread per block.
__global__ void __launch_bounds__(256) dequant_q4_0_kernel(const uint8_t* __restrict__ bq, long long ldbq,
                                                           long long N, long long nblocks, __half* __restrict__ out,
                                                           long long ldo) {
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
                                int num_sms, cudaStream_t stream) {
    const long long nblocks = K / 32;
    const long long total = N * nblocks;
    if (total <= 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(bq) & 15u) == 0 && ldbq % 16 == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0 &&
        ldo % 8 == 0 && nblocks < (1LL << 30)) {
        const long long groups = N * ((nblocks + 31) / 32);
        long long ctas = (groups + kDqWarpsPerCta - 1) / kDqWarpsPerCta;
        const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 152) * 8;
        if (ctas > cap) ctas = cap;
        dequant_q4_0_rows_kernel<<<static_cast<unsigned>(ctas), kDqWarpsPerCta * 32, 0, stream>>>(
            static_cast<const uint8_t*>(bq), ldbq, N, static_cast<int>(nblocks), static_cast<__half*>(out), ldo);
        return cudaGetLastError();
    }
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 152) * 8;
    if (blocks > cap) blocks = cap;
    dequant_q4_0_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint8_t*>(bq), ldbq, N, nblocks, static_cast<__half*>(out), ldo);
    return cudaGetLastError();
}

template <int kOut>
__global__ void scale_bias_kernel(void* C, long long ldc, const void* bias, float beta, long long M, long long N) {
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
                              long long N, int num_sms, cudaStream_t stream) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    long long blocks = (M * N + 255) / 256;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 152) * 8;
    if (blocks > cap) blocks = cap;
    const unsigned g = static_cast<unsigned>(blocks);
    switch (out) {
        case OUT_F16: scale_bias_kernel<OUT_F16><<<g, 256, 0, stream>>>(C, ldc, bias, beta, M, N); break;
        case OUT_BF16: scale_bias_kernel<OUT_BF16><<<g, 256, 0, stream>>>(C, ldc, bias, beta, M, N); break;
        case OUT_F32: scale_bias_kernel<OUT_F32><<<g, 256, 0, stream>>>(C, ldc, bias, beta, M, N); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gb300

// Auxiliary kernels around the tcgen05 GEMM:
//  * repack of a 16-bit operand whose byte pitch is not a multiple of 16 into a workspace with a
//    16-byte pitch (TMA tensor maps require 16-byte-multiple strides);
//  * the K == 0 epilogue, C = beta * C + bias (the product of an empty sum is zero).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"
#include "gemm_launch.h"

namespace gb300 {

// Copy a rows x cols block of 16-bit elements from pitch `lds` to pitch `ldd` (elements).
// When both pitches are even and cols is even, pairs move as 32-bit words.
__global__ void repack_u16_kernel(const uint16_t* __restrict__ src, long long lds, uint16_t* __restrict__ dst,
                                  long long ldd, long long rows, long long cols, int pairs) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    if (pairs) {
        const long long wc = cols / 2;
        const long long total = rows * wc;
        for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
            const long long r = i / wc, c = i - r * wc;
            const uint32_t w = *reinterpret_cast<const uint32_t*>(src + r * lds + 2 * c);
            *reinterpret_cast<uint32_t*>(dst + r * ldd + 2 * c) = w;
        }
    } else {
        const long long total = rows * cols;
        for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
            const long long r = i / cols, c = i - r * cols;
            dst[r * ldd + c] = src[r * lds + c];
        }
    }
}

cudaError_t launch_repack_u16(const void* src, long long lds, void* dst, long long ldd, long long rows,
                              long long cols, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const int pairs = ((lds % 2) == 0 && (ldd % 2) == 0 && (cols % 2) == 0 &&
                       (reinterpret_cast<uintptr_t>(src) % 4) == 0 && (reinterpret_cast<uintptr_t>(dst) % 4) == 0)
                          ? 1 : 0;
    const long long work = pairs ? rows * (cols / 2) : rows * cols;
    long long blocks = (work + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    repack_u16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(src), lds, static_cast<uint16_t*>(dst), ldd, rows, cols, pairs);
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

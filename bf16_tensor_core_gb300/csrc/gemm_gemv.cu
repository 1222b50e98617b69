// Products with very few rows of C (M <= 8) against weights stored N x K (K contiguous): the
// decode shape of "Matrix Multiplication: The Operation Behind Modern AI" (section "The shape a
// language model actually runs": one 4096 x 4096 weight, M input vectors, intensity ~1 FLOP/B),
// which is bound by streaming the weights from HBM, not by the tensor cores.
//
//   C[m][n] = alpha * sum_k A[m][k] * W[n][k] + beta * C[m][n] + bias[n]
//
// A CTA owns kGemvRows consecutive weight rows and its kGemvWarps warps split K.  Per step every lane
// loads 16 bytes (8 weights) of each row -- 512 contiguous bytes per row per warp instruction, two
// steps in flight -- and the matching 8 values of every A row through L1 (A is small and shared by
// all CTAs), accumulating in f32.  Lane partials are summed with shuffles, warp partials through
// shared memory in warp order, and the epilogue is applied in f32.  Many small CTAs per SM keep
// enough bytes in flight to stream the weights at HBM speed.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"
#include "gemm_launch.h"
#include "q4_block.cuh"

namespace gb300 {

namespace {

constexpr int kGemvRows = 4;       // weight rows per CTA (every warp carries all of them)
constexpr int kGemvWarps = 8;      // warps per CTA (they split K)

template <bool kBf16>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t;
        if constexpr (kBf16) t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
        else t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// The f32 epilogue of element (m, n): alpha * s + beta * C_in + bias, rounded to the output type.
template <int kOut>
__device__ __forceinline__ void store_gemv_out(const GemvParams& p, int m, int n, float s) {
    const long long idx = static_cast<long long>(m) * p.ldc + n;
    float v = p.alpha * s;
    if (p.beta != 0.0f) v = fmaf(p.beta, load_out<kOut>(p.C, idx), v);
    if (p.bias != nullptr) v += load_out<kOut>(p.bias, n);
    if constexpr (kOut == OUT_F32) static_cast<float*>(p.C)[idx] = v;
    else if constexpr (kOut == OUT_F16) static_cast<__half*>(p.C)[idx] = __float2half_rn(v);
    else static_cast<__nv_bfloat16*>(p.C)[idx] = __float2bfloat16_rn(v);
}

// kM rows of C; kOut: output type; kBf16: bf16 operands (else f16).
template <int kM, int kOut, bool kBf16>
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_kernel(GemvParams p) {
    __shared__ float part[kGemvWarps][kGemvRows][kM];
    griddep_launch_dependents();
    const int n0 = blockIdx.x * kGemvRows;
    // This CTA's weight rows into L2 while the kernel before it may still run (see tma_prefetch_2d).
    if (threadIdx.x < kGemvRows && n0 + static_cast<int>(threadIdx.x) < p.N)
        bulk_prefetch_l2(static_cast<const uint8_t*>(p.W) + static_cast<long long>(n0 + threadIdx.x) * p.ldw_bytes,
                         static_cast<uint32_t>(p.K) * 2u);
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunks = p.K / 8;                                     // 8 values per chunk (K % 8 == 0)
    const int per_warp = (chunks + kGemvWarps - 1) / kGemvWarps;
    const int c_begin = warp * per_warp;
    const int c_end = min(chunks, c_begin + per_warp);
    const uint8_t* W = static_cast<const uint8_t*>(p.W);
    const uint8_t* A = static_cast<const uint8_t*>(p.A);
    float acc[kGemvRows][kM];
#pragma unroll
    for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
        for (int m = 0; m < kM; ++m) acc[r][m] = 0.0f;
    // Row r's chunk c at byte offset (n0 + r) * ldw_bytes + 16 c; rows past N contribute zeros.
    auto load = [&](int c, uint4 (&w)[kGemvRows]) {
#pragma unroll
        for (int r = 0; r < kGemvRows; ++r) {
            if (n0 + r < p.N && c < c_end)
                w[r] = ldg_stream(W + static_cast<long long>(n0 + r) * p.ldw_bytes + static_cast<long long>(c) * 16);
            else
                w[r] = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    auto fma_chunk = [&](int c, const uint4 (&w)[kGemvRows]) {
        float wf[kGemvRows][8];
#pragma unroll
        for (int r = 0; r < kGemvRows; ++r) unpack8<kBf16>(w[r], wf[r]);
#pragma unroll
        for (int m = 0; m < kM; ++m) {
            float af[8];
            unpack8<kBf16>(__ldg(reinterpret_cast<const uint4*>(A + static_cast<long long>(m) * p.lda_bytes +
                                                                static_cast<long long>(c) * 16)), af);
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[r][m] = fmaf(af[j], wf[r][j], acc[r][m]);
        }
    };
    // Two chunks in flight per lane and row.
    for (int c = c_begin + lane; c < c_end; c += 64) {
        uint4 w0[kGemvRows], w1[kGemvRows];
        load(c, w0);
        load(c + 32, w1);
        fma_chunk(c, w0);
        if (c + 32 < c_end) fma_chunk(c + 32, w1);
    }
#pragma unroll
    for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
        for (int m = 0; m < kM; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);
            if (lane == 0) part[warp][r][m] = acc[r][m];
        }
    __syncthreads();
    if (threadIdx.x < kGemvRows * kM) {
        const int r = threadIdx.x / kM, m = threadIdx.x - (threadIdx.x / kM) * kM;
        const int n = n0 + r;
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kGemvWarps; ++w) s += part[w][r][m];
        if (n < p.N) store_gemv_out<kOut>(p, m, n, s);
    }
}

template <int kM, int kOut>
cudaError_t launch_m(const GemvParams& p, bool bf16, int blocks, cudaStream_t s, bool pdl) {
    auto kern = bf16 ? &gemv_kernel<kM, kOut, true> : &gemv_kernel<kM, kOut, false>;
    return launch_ex(kern, dim3(blocks), dim3(kGemvWarps * 32), 0, s, pdl, p);
}

template <int kOut>
cudaError_t launch_out(const GemvParams& p, bool bf16, int blocks, cudaStream_t s, bool pdl) {
    switch (p.M) {
        case 1: return launch_m<1, kOut>(p, bf16, blocks, s, pdl);
        case 2: return launch_m<2, kOut>(p, bf16, blocks, s, pdl);
        case 3: return launch_m<3, kOut>(p, bf16, blocks, s, pdl);
        case 4: return launch_m<4, kOut>(p, bf16, blocks, s, pdl);
        case 5: return launch_m<5, kOut>(p, bf16, blocks, s, pdl);
        case 6: return launch_m<6, kOut>(p, bf16, blocks, s, pdl);
        case 7: return launch_m<7, kOut>(p, bf16, blocks, s, pdl);
        case 8: return launch_m<8, kOut>(p, bf16, blocks, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------- Q4_0 weights
// The same product with W given as Q4_0 blocks ("02 . 8m/8m(2) -- Tiled wmma f16 prefill GEMM",
// section 3.2: per 32 weights an f16 scale d and 16 bytes q, weight i the low nibble of q[i] and
// weight 16+i its high nibble, value d * (q - 8) rounded to f16).  At decode the weights are read
// once at 4.5 bits each, so the kernel streams the blocks and multiplies as it dequantises: a CTA
// owns kQ4Rows weight rows; thread t takes blocks t, t + kQ4Threads, ... of all of them (a warp's
// loads of one row cover 576 contiguous bytes), dequantises each block exactly as the tensor-core
// path does (f16 1024 + q, minus 1032, times d, one rounding) and accumulates a * w in f32.
constexpr int kQ4Rows = 4;           // weight rows per CTA
constexpr int kQ4Threads = 128;      // threads per CTA (they split the blocks of a row)

// acc + a.lo * w.lo + a.hi * w.hi, each product exact (two f16 values) and each sum rounded in f32.
__device__ __forceinline__ float fma2_f16_f32(uint32_t a2, uint32_t w2, float acc) {
    asm("{\n\t.reg .b16 al, ah, wl, wh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, wl, %0;\n\t"
        "fma.rn.f32.f16 %0, ah, wh, %0;\n\t}"
        : "+f"(acc) : "r"(a2), "r"(w2));
    return acc;
}

template <int kM, int kOut>
__global__ void __launch_bounds__(kQ4Threads) gemv_q4_0_kernel(GemvParams p) {
    constexpr int kWarps = kQ4Threads / 32;
    __shared__ float part[kWarps][kQ4Rows][kM];
    griddep_launch_dependents();
    const int n0 = blockIdx.x * kQ4Rows;
    const int nblk = p.K / 32;
    // This CTA's block rows into L2 while the kernel before it may still run (see tma_prefetch_2d); a row
    // starts at any 2-byte boundary, so the range is widened to the 16-byte granules that hold it.
    if (threadIdx.x < kQ4Rows && n0 + static_cast<int>(threadIdx.x) < p.N) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(static_cast<const uint8_t*>(p.W) +
                                                        static_cast<long long>(n0 + threadIdx.x) * p.ldw_bytes);
        const uintptr_t lo = a & ~static_cast<uintptr_t>(15), hi = (a + 18ull * nblk + 15) & ~static_cast<uintptr_t>(15);
        bulk_prefetch_l2(reinterpret_cast<const void*>(lo), static_cast<uint32_t>(hi - lo));
    }
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint8_t* Bq = static_cast<const uint8_t*>(p.W);
    const uint8_t* A = static_cast<const uint8_t*>(p.A);
    float acc[kQ4Rows][kM];
#pragma unroll
    for (int r = 0; r < kQ4Rows; ++r)
#pragma unroll
        for (int m = 0; m < kM; ++m) acc[r][m] = 0.0f;
    for (int b = threadIdx.x; b < nblk; b += kQ4Threads) {
        // All rows' loads first, then the arithmetic; rows past N are zero blocks (scale 0).
        Q4Block raw[kQ4Rows];
#pragma unroll
        for (int r = 0; r < kQ4Rows; ++r) {
            if (n0 + r < p.N) raw[r] = q4_block_global(Bq + static_cast<long long>(n0 + r) * p.ldw_bytes + 18LL * b);
            else raw[r] = Q4Block{0u, {0u, 0u, 0u, 0u}};
        }
        uint32_t w[kQ4Rows][16];
#pragma unroll
        for (int r = 0; r < kQ4Rows; ++r) q4_block_weights(raw[r], w[r]);
#pragma unroll
        for (int m = 0; m < kM; ++m) {
            const uint4* ap = reinterpret_cast<const uint4*>(A + static_cast<long long>(m) * p.lda_bytes + 64LL * b);
#pragma unroll
            for (int pc = 0; pc < 4; ++pc) {
                const uint4 a = __ldg(ap + pc);
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int r = 0; r < kQ4Rows; ++r) acc[r][m] = fma2_f16_f32(aw[j], w[r][4 * pc + j], acc[r][m]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kQ4Rows; ++r)
#pragma unroll
        for (int m = 0; m < kM; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);
            if (lane == 0) part[warp][r][m] = acc[r][m];
        }
    __syncthreads();
    if (threadIdx.x < kQ4Rows * kM) {
        const int r = threadIdx.x / kM, m = threadIdx.x - (threadIdx.x / kM) * kM;
        const int n = n0 + r;
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += part[w][r][m];
        if (n < p.N) store_gemv_out<kOut>(p, m, n, s);
    }
}

template <int kM, int kOut>
cudaError_t launch_q4_m(const GemvParams& p, int blocks, cudaStream_t s, bool pdl) {
    return launch_ex(gemv_q4_0_kernel<kM, kOut>, dim3(blocks), dim3(kQ4Threads), 0, s, pdl, p);
}

template <int kOut>
cudaError_t launch_q4_out(const GemvParams& p, int blocks, cudaStream_t s, bool pdl) {
    switch (p.M) {
        case 1: return launch_q4_m<1, kOut>(p, blocks, s, pdl);
        case 2: return launch_q4_m<2, kOut>(p, blocks, s, pdl);
        case 3: return launch_q4_m<3, kOut>(p, blocks, s, pdl);
        case 4: return launch_q4_m<4, kOut>(p, blocks, s, pdl);
        case 5: return launch_q4_m<5, kOut>(p, blocks, s, pdl);
        case 6: return launch_q4_m<6, kOut>(p, blocks, s, pdl);
        case 7: return launch_q4_m<7, kOut>(p, blocks, s, pdl);
        case 8: return launch_q4_m<8, kOut>(p, blocks, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gemv_q4_0(int out, const GemvParams& p, int num_sms, cudaStream_t stream, bool pdl) {
    (void)num_sms;
    if (p.M < 1 || p.M > kGemvMaxM || p.N <= 0 || p.K <= 0 || p.K % 32 != 0 || p.ldw_bytes % 2 != 0 ||
        p.ldw_bytes < p.K / 32 * 18 || (reinterpret_cast<uintptr_t>(p.W) & 1u) != 0 || p.lda_bytes % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(p.A) & 15u) != 0)
        return cudaErrorInvalidValue;
    const long long blocks = (p.N + kQ4Rows - 1) / kQ4Rows;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    switch (out) {
        case OUT_F16: return launch_q4_out<OUT_F16>(p, static_cast<int>(blocks), stream, pdl);
        case OUT_BF16: return launch_q4_out<OUT_BF16>(p, static_cast<int>(blocks), stream, pdl);
        case OUT_F32: return launch_q4_out<OUT_F32>(p, static_cast<int>(blocks), stream, pdl);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv(int out, bool bf16, const GemvParams& p, int num_sms, cudaStream_t stream, bool pdl) {
    (void)num_sms;
    if (p.M < 1 || p.M > kGemvMaxM || p.N <= 0 || p.K <= 0 || p.K % 8 != 0) return cudaErrorInvalidValue;
    const long long blocks = (p.N + kGemvRows - 1) / kGemvRows;   // one row group per CTA
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    switch (out) {
        case OUT_F16: return launch_out<OUT_F16>(p, bf16, static_cast<int>(blocks), stream, pdl);
        case OUT_BF16: return launch_out<OUT_BF16>(p, bf16, static_cast<int>(blocks), stream, pdl);
        case OUT_F32: return launch_out<OUT_F32>(p, bf16, static_cast<int>(blocks), stream, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300

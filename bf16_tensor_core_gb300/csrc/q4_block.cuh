// Q4_0 block decoding shared by the CUDA-core small-M kernel and the separate dequantisation pass
// ("02 . 8m/8m(2) -- Tiled wmma f16 prefill GEMM", section 3.2: an f16 scale d, then 16 bytes q;
// weight i is the low nibble of q[i], weight 16+i its high nibble, value d * (q - 8) rounded to f16).
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "gemm_kernel.cuh"

namespace gb300 {

// One block as the scale bits and the 16 nibble bytes in four words, from words holding its 18
// bytes: w0..w3 from the block start and a 16-bit tail w4 (block on a 4-byte boundary), or the
// 16-bit scale w0 and w1..w4 (block 2 bytes past one).
struct Q4Block {
    uint32_t d;
    uint32_t q[4];
};

__device__ __forceinline__ Q4Block q4_block_from_words(bool aligned4, uint32_t w0, uint32_t w1, uint32_t w2,
                                                       uint32_t w3, uint32_t w4) {
    Q4Block r;
    if (aligned4) {
        r.d = w0 & 0xffffu;
        r.q[0] = __byte_perm(w0, w1, 0x5432u);
        r.q[1] = __byte_perm(w1, w2, 0x5432u);
        r.q[2] = __byte_perm(w2, w3, 0x5432u);
        r.q[3] = __byte_perm(w3, w4, 0x5432u);
    } else {
        r.d = w0;
        r.q[0] = w1;
        r.q[1] = w2;
        r.q[2] = w3;
        r.q[3] = w4;
    }
    return r;
}

// A block in global memory at any 2-byte alignment (read-only path; L1 keeps the lines that a
// warp's consecutive blocks share).
__device__ __forceinline__ Q4Block q4_block_global(const uint8_t* b) {
    if ((reinterpret_cast<uintptr_t>(b) & 2u) == 0) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(b);
        return q4_block_from_words(true, __ldg(w), __ldg(w + 1), __ldg(w + 2), __ldg(w + 3),
                                   __ldg(reinterpret_cast<const unsigned short*>(b + 16)));
    }
    const uint32_t* w = reinterpret_cast<const uint32_t*>(b + 2);
    return q4_block_from_words(false, __ldg(reinterpret_cast<const unsigned short*>(b)), __ldg(w), __ldg(w + 1),
                               __ldg(w + 2), __ldg(w + 3));
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_shared_u16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
    return v;
}

// Block b of blocks packed from shared address s (16-byte aligned): it starts 18 b bytes in.
__device__ __forceinline__ Q4Block q4_block_shared(uint32_t s, int b) {
    const uint32_t a = s + 18u * static_cast<uint32_t>(b);
    if ((b & 1) == 0)
        return q4_block_from_words(true, ld_shared_u32(a), ld_shared_u32(a + 4), ld_shared_u32(a + 8),
                                   ld_shared_u32(a + 12), ld_shared_u16(a + 16));
    return q4_block_from_words(false, ld_shared_u16(a), ld_shared_u32(a + 2), ld_shared_u32(a + 6),
                               ld_shared_u32(a + 10), ld_shared_u32(a + 14));
}

// The block's 32 weights as f16 pairs: word j holds weights 2j (low half) and 2j + 1.
__device__ __forceinline__ void q4_block_weights(const Q4Block& b, uint32_t (&v)[16]) {
    const __half2 d2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(b.d)));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t hi = b.q[i] >> 4;
        v[2 * i] = q4_two(__byte_perm(b.q[i], 0u, 0x4140u), d2);
        v[2 * i + 1] = q4_two(__byte_perm(b.q[i], 0u, 0x4342u), d2);
        v[8 + 2 * i] = q4_two(__byte_perm(hi, 0u, 0x4140u), d2);
        v[8 + 2 * i + 1] = q4_two(__byte_perm(hi, 0u, 0x4342u), d2);
    }
}

}  // namespace gb300

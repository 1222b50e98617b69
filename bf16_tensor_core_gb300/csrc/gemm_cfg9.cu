// Kernel configuration 9: cta_group::1, output tile 128 x 64, 8-bit inputs, BK 256, 4-stage ring
// (transposed skinny products).
#include "gemm_kernel.cuh"
#include "gemm_launch.h"

namespace gb300 {

const void* cfg9_kernel(int out) {
    switch (out) {
        case OUT_F16: return reinterpret_cast<const void*>(&gemm_tc_kernel<1, 64, 4, 256, OUT_F16, false, 1>);
        case OUT_BF16: return reinterpret_cast<const void*>(&gemm_tc_kernel<1, 64, 4, 256, OUT_BF16, false, 1>);
        case OUT_F32: return reinterpret_cast<const void*>(&gemm_tc_kernel<1, 64, 4, 256, OUT_F32, false, 1>);
        default: return nullptr;
    }
}

cudaError_t cfg9_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p) {
    switch (out) {
        case OUT_F16: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<1, 64, 4, 256, OUT_F16, false, 1>, a, b, c, p);
        case OUT_BF16: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<1, 64, 4, 256, OUT_BF16, false, 1>, a, b, c, p);
        case OUT_F32: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<1, 64, 4, 256, OUT_F32, false, 1>, a, b, c, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300

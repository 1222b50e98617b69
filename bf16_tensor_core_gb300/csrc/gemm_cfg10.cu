// Kernel configuration 10: cta_group::1, output tile 128 x 128, 8-bit inputs, BK 128, 6-stage ring.
#include "gemm_kernel.cuh"
#include "gemm_launch.h"

namespace gb300 {

const void* cfg10_kernel(int out) {
    switch (out) {
        case OUT_F16: return reinterpret_cast<const void*>(&gemm_tc_kernel<1, 128, 6, 128, OUT_F16, false, 1>);
        case OUT_BF16: return reinterpret_cast<const void*>(&gemm_tc_kernel<1, 128, 6, 128, OUT_BF16, false, 1>);
        case OUT_F32: return reinterpret_cast<const void*>(&gemm_tc_kernel<1, 128, 6, 128, OUT_F32, false, 1>);
        default: return nullptr;
    }
}

cudaError_t cfg10_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                         const CUtensorMap& c, const KernelParams& p) {
    switch (out) {
        case OUT_F16: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<1, 128, 6, 128, OUT_F16, false, 1>, a, b, c, p);
        case OUT_BF16: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<1, 128, 6, 128, OUT_BF16, false, 1>, a, b, c, p);
        case OUT_F32: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<1, 128, 6, 128, OUT_F32, false, 1>, a, b, c, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300

// Kernel configuration 3: cta_group::2 (2-SM pair), output tile 256 x 128, BK 64, 8-stage ring.
#include "gemm_kernel.cuh"
#include "gemm_launch.h"

namespace gb300 {

const void* cfg3_kernel(int out) {
    switch (out) {
        case OUT_F16: return reinterpret_cast<const void*>(&gemm_tc_kernel<2, 128, 8, 64, OUT_F16>);
        case OUT_BF16: return reinterpret_cast<const void*>(&gemm_tc_kernel<2, 128, 8, 64, OUT_BF16>);
        case OUT_F32: return reinterpret_cast<const void*>(&gemm_tc_kernel<2, 128, 8, 64, OUT_F32>);
        default: return nullptr;
    }
}

cudaError_t cfg3_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p) {
    switch (out) {
        case OUT_F16: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<2, 128, 8, 64, OUT_F16>, a, b, c, p);
        case OUT_BF16: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<2, 128, 8, 64, OUT_BF16>, a, b, c, p);
        case OUT_F32: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<2, 128, 8, 64, OUT_F32>, a, b, c, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300

// Kernel configuration 6: cta_group::2 (2-SM pair), output tile 256 x 256, BK 128, 3-stage ring,
// B dequantised from Q4_0 blocks in shared memory.
#include "gemm_kernel.cuh"
#include "gemm_launch.h"

namespace gb300 {

const void* cfg6_kernel(int out) {
    switch (out) {
        case OUT_F16: return reinterpret_cast<const void*>(&gemm_tc_kernel<2, 256, 3, 128, OUT_F16, true>);
        case OUT_BF16: return reinterpret_cast<const void*>(&gemm_tc_kernel<2, 256, 3, 128, OUT_BF16, true>);
        case OUT_F32: return reinterpret_cast<const void*>(&gemm_tc_kernel<2, 256, 3, 128, OUT_F32, true>);
        default: return nullptr;
    }
}

cudaError_t cfg6_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p) {
    switch (out) {
        case OUT_F16: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<2, 256, 3, 128, OUT_F16, true>, a, b, c, p);
        case OUT_BF16: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<2, 256, 3, 128, OUT_BF16, true>, a, b, c, p);
        case OUT_F32: return cudaLaunchKernelEx(&lc, &gemm_tc_kernel<2, 256, 3, 128, OUT_F32, true>, a, b, c, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300

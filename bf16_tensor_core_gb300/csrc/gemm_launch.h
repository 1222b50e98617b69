// Host-side view of the kernel configurations (no device code).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gb300 {

struct KernelParams;

// Launch `kernel` with cudaLaunchKernelEx; with `pdl` the launch allows programmatic stream
// serialization, so it may be scheduled while the previous kernel on the stream finishes (every
// kernel here waits with griddepcontrol.wait before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                      Args&&... args) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&lc, kernel, static_cast<KArgs>(args)...);
}

struct ConfigDesc {
    int id;
    int cta_group;
    int block_n;
    int block_k;      // K per pipeline stage (64 or 128)
    int stages;
    int smem_bytes;
    int threads;
    int b_q4;         // 1: B is Q4_0-quantised and dequantised in shared memory by the kernel
    int in_bytes;     // operand element size: 2 (f16 / bf16) or 1 (8-bit floats)
};

constexpr int kNumConfigs = 11;
constexpr int kNumOut = 3;  // OUT_F16, OUT_BF16, OUT_F32

// Static description of config `id` (nullptr if out of range).
const ConfigDesc* config_desc(int id);

// Kernel entry for config `id` and output type `out` (for attributes and occupancy queries).
const void* config_kernel(int id, int out);

// Launch config `id` on `grid_ctas` CTAs on `stream`, in thread-block clusters of `cluster_ctas` CTAs
// (the config's cta_group, or the split parts of a tile for KernelParams::rs_cluster).
cudaError_t config_launch(int id, int out, int grid_ctas, int cluster_ctas, cudaStream_t stream, bool pdl,
                          const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c, const KernelParams& p);

// Per-config translation units.
const void* cfg0_kernel(int out);
cudaError_t cfg0_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p);
const void* cfg1_kernel(int out);
cudaError_t cfg1_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p);
const void* cfg2_kernel(int out);
cudaError_t cfg2_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p);
const void* cfg3_kernel(int out);
cudaError_t cfg3_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p);
const void* cfg4_kernel(int out);
cudaError_t cfg4_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p);
const void* cfg5_kernel(int out);
cudaError_t cfg5_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p);
const void* cfg6_kernel(int out);
cudaError_t cfg6_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p);
const void* cfg7_kernel(int out);
cudaError_t cfg7_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p);
const void* cfg8_kernel(int out);
cudaError_t cfg8_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p);
const void* cfg9_kernel(int out);
cudaError_t cfg9_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KernelParams& p);
const void* cfg10_kernel(int out);
cudaError_t cfg10_launch(int out, const cudaLaunchConfig_t& lc, const CUtensorMap& a, const CUtensorMap& b,
                         const CUtensorMap& c, const KernelParams& p);

// Few rows of C against weights stored N x K (gemm_gemv.cu): CUDA-core kernel for M <= kGemvMaxM.
constexpr int kGemvMaxM = 8;
struct GemvParams {
    const void* A;           // M x K row-major, 16-bit, 16-byte aligned, row pitch lda_bytes (multiple of 16)
    long long lda_bytes;
    const void* W;           // N x K, K contiguous, 16-byte aligned, row pitch ldw_bytes (multiple of 16)
    long long ldw_bytes;
    void* C;                 // M x N row-major, ldc elements
    long long ldc;
    const void* bias;
    float alpha, beta;
    int M, N, K;             // K a multiple of 8
};
cudaError_t launch_gemv(int out, bool bf16, const GemvParams& p, int num_sms, cudaStream_t stream, bool pdl);
// The same with W given as Q4_0 blocks: W = the block rows (2-byte aligned), ldw_bytes = their even
// pitch (>= K/32*18), K a multiple of 32, A f16 with a 16-byte aligned base and pitch.
cudaError_t launch_gemv_q4_0(int out, const GemvParams& p, int num_sms, cudaStream_t stream, bool pdl);

// Auxiliary kernels (gemm_aux.cu).
struct RepackJob {
    const uint16_t* src;   // rows x cols elements at pitch lds (2-byte aligned)
    long long lds;
    uint16_t* dst;         // rows x ldd elements, 16-byte aligned, ldd a multiple of 8 and >= cols
    long long ldd;
    long long rows, cols;
};
struct RepackJobs {
    RepackJob job[2];
    int n;                 // jobs in use (0..2), all moved by one launch
};
cudaError_t launch_repack_u16(const RepackJobs& jobs, int num_sms, cudaStream_t stream, bool pdl);
cudaError_t launch_dequant_q4_0(const void* bq, long long ldbq, long long N, long long K, void* out, long long ldo,
                                int num_sms, cudaStream_t stream, bool pdl);
cudaError_t launch_scale_bias(int out, void* C, long long ldc, const void* bias, float beta, long long M,
                              long long N, int num_sms, cudaStream_t stream, bool pdl);

}  // namespace gb300

// Host side of the C ABI declared in include/gemm.h: handle, validation, planning, tensor-map
// cache, operand repack, stream-K buffers, dispatch and error reporting.  The only device code
// here is the file-scope scratch of gemm_run_noalloc.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/gemm.h"
#include "gemm_kernel.cuh"
#include "gemm_launch.h"

using namespace gb300;

namespace {

// ---------------------------------------------------------------- configuration table
template <int CG, int BN, int ST, int BK, bool Q4 = false, int ELT = 2>
constexpr ConfigDesc make_desc(int id) {
    return ConfigDesc{id, CG, BN, BK, ST, TileConfig<CG, BN, ST, BK, Q4, ELT>::kSmemBytes,
                      TileConfig<CG, BN, ST, BK, Q4, ELT>::kThreads, Q4 ? 1 : 0, ELT};
}

const ConfigDesc kConfigs[kNumConfigs] = {
    make_desc<1, 256, 4, 64>(0),   // 1 SM, 128 x 256 tile
    make_desc<2, 256, 6, 64>(1),   // 2-SM pair, 256 x 256 tile
    make_desc<1, 128, 6, 64>(2),   // 1 SM, 128 x 128 tile
    make_desc<2, 128, 8, 64>(3),   // 2-SM pair, 256 x 128 tile
    make_desc<2, 256, 3, 128>(4),  // 2-SM pair, 256 x 256 tile, 128-wide K stages
    make_desc<2, 512, 4, 64>(5),   // 2-SM pair, 256 x 512 tile (two N=256 MMAs per K step)
    make_desc<2, 256, 3, 128, true>(6),  // as 4, B dequantised from Q4_0 blocks in shared memory
    make_desc<1, 64, 4, 128>(7),   // 1 SM, 128 x 64 tile: the short side of a transposed skinny product
    make_desc<2, 256, 3, 256, false, 1>(8),  // 8-bit inputs: 2-SM pair, 256 x 256 tile, BK 256
    make_desc<1, 64, 4, 256, false, 1>(9),   // 8-bit inputs: 1 SM, 128 x 64 tile (transposed skinny)
    make_desc<1, 128, 6, 128, false, 1>(10), // 8-bit inputs: 1 SM, 128 x 128 tile
};

// Mainloop efficiency per config (measured k-iteration time of one long-K tile against the
// config's tensor-core time at 1.9 GHz, cold L2, GB300): small tiles need more operand bytes per
// flop and are bound by the TMA load rate per SM.  Config 5 is derated for its single accumulator
// (its epilogue does not overlap the next tile); config 6 runs at the rate of its dequantisation
// warps (2048 x 11008 x 4096 in 260 us), not of its MMAs.
const double kConfigEfficiency[kNumConfigs] = {0.73, 0.78, 0.40, 0.39, 0.85, 0.75, 0.31, 0.40, 0.85, 0.40, 0.40};

int cluster_ctas(const ConfigDesc& d) { return d.cta_group; }
int block_m(const ConfigDesc& d) { return 128 * cluster_ctas(d); }

enum FaultSite { FAULT_NONE = 0, FAULT_OPTIN = 1, FAULT_TMAP = 2, FAULT_LAUNCH = 4, FAULT_ALLOC = 8 };

int read_fault_env() {
    // Host-side fault injection for tests: GEMM_TEST_FAIL=optin,tmap,launch,alloc
    const char* e = std::getenv("GEMM_TEST_FAIL");
    if (!e) return FAULT_NONE;
    int f = FAULT_NONE;
    std::string s(e);
    if (s.find("optin") != std::string::npos) f |= FAULT_OPTIN;
    if (s.find("tmap") != std::string::npos) f |= FAULT_TMAP;
    if (s.find("launch") != std::string::npos) f |= FAULT_LAUNCH;
    if (s.find("alloc") != std::string::npos) f |= FAULT_ALLOC;
    return f;
}

int elt_bytes(int dt) { return dt == GEMM_F32 ? 4 : (dt == GEMM_E4M3 || dt == GEMM_E5M2) ? 1 : 2; }
bool is_f8(int dt) { return dt == GEMM_E4M3 || dt == GEMM_E5M2; }
int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// What a device offers each config: SM count, co-resident clusters, the tensor-map encoder.
struct DevInfo {
    int num_sms = 0;
    int slots[kNumConfigs] = {};                 // clusters of each config that fit at once
    int rs_slots[kNumConfigs][3] = {};           // 1-SM 64-wide configs: clusters of 2, 4, 8 CTAs that fit
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
};

// Opt every kernel into its shared memory (never inside a capture window), count the clusters
// of each config that fit, resolve the encoder.  `dev` must be current.
gemm_status_t query_device(int dev, bool force_optin_failure, DevInfo* info) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&info->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;
    for (int c = 0; c < kNumConfigs; ++c) {
        const ConfigDesc* d = config_desc(c);
        for (int outk = 0; outk < kNumOut; ++outk) {
            cudaError_t ea = force_optin_failure ? cudaErrorInvalidValue
                             : cudaFuncSetAttribute(config_kernel(c, outk), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    d->smem_bytes);
            if (ea != cudaSuccess) {
                cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
        }
        const int csize = cluster_ctas(*d);
        int n = info->num_sms;
        if (csize > 1) {
            cudaLaunchConfig_t lc = {};
            lc.gridDim = dim3((unsigned)(info->num_sms - info->num_sms % csize), 1, 1);
            lc.blockDim = dim3((unsigned)d->threads, 1, 1);
            lc.dynamicSmemBytes = (size_t)d->smem_bytes;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)csize;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            lc.attrs = attr;
            lc.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, config_kernel(c, OUT_F16), &lc) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
        }
        info->slots[c] = n;
        // The split parts of a tile as one cluster (KernelParams::rs_cluster): 1-SM configs of 64-wide tiles.
        if (d->cta_group == 1 && d->block_n == 64 && !d->b_q4) {
            for (int i = 0; i < 3; ++i) {
                cudaLaunchConfig_t lc = {};
                lc.gridDim = dim3((unsigned)((info->num_sms >> (i + 1)) << (i + 1)), 1, 1);
                lc.blockDim = dim3((unsigned)d->threads, 1, 1);
                lc.dynamicSmemBytes = (size_t)d->smem_bytes;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = 2u << i;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                lc.attrs = attr;
                lc.numAttrs = 1;
                int m = 0;
                if (cudaOccupancyMaxActiveClusters(&m, config_kernel(c, OUT_F16), &lc) != cudaSuccess) {
                    cudaGetLastError();
                    m = 0;
                }
                info->rs_slots[c][i] = m;
            }
        }
    }
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    info->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return GEMM_OK;
}

// A 2-D or 3-D tiled tensor map: dims[0] contiguous, strides in bytes for dims 1..rank-1.
struct TmapDesc {
    const void* ptr;
    CUtensorMapDataType dt;
    int rank;
    uint64_t dims[3];
    uint64_t strides[2];
    uint32_t box[3];
    bool operator==(const TmapDesc& o) const {
        if (ptr != o.ptr || dt != o.dt || rank != o.rank) return false;
        for (int i = 0; i < rank; ++i)
            if (dims[i] != o.dims[i] || box[i] != o.box[i]) return false;
        for (int i = 0; i + 1 < rank; ++i)
            if (strides[i] != o.strides[i]) return false;
        return true;
    }
};

TmapDesc tmap2d(const void* ptr, CUtensorMapDataType dt, uint64_t d0, uint64_t d1, uint64_t stride, uint32_t b0,
                uint32_t b1) {
    return TmapDesc{ptr, dt, 2, {d0, d1, 1}, {stride, 0}, {b0, b1, 1}};
}

TmapDesc tmap3d(const void* ptr, CUtensorMapDataType dt, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
    return TmapDesc{ptr, dt, 3, {d0, d1, d2}, {s1, s2}, {b0, b1, b2}};
}

struct TmapEntry {
    TmapDesc key;
    CUtensorMap map;
};

}  // namespace

struct gemm_ctx {
    int device = 0;
    DevInfo dev;
    gemm_options_t opt{};
    unsigned long long* d_status = nullptr;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    std::string err;
    std::vector<TmapEntry> cache;
    size_t cache_next = 0;
    int faults = FAULT_NONE;
    bool force_2d = false;          // GEMM_TMA_RANK=2 (tuning): never use 3-D operand maps
    bool k_forward = false;         // GEMM_K_ORDER=forward (tuning): every tile walks K upwards
    int64_t launches = 0;
    unsigned* sk_flags = nullptr;   // zeroed at creation; raised to the launch epoch, reset by their consumer
    float* sk_part = nullptr;       // stream-K partials (grown on demand)
    size_t sk_part_bytes = 0;
    void* q4_ws = nullptr;          // f16 weights of the separate Q4_0 dequantisation pass (grown on demand)
    size_t q4_ws_bytes = 0;
    unsigned epoch = 0;
    gemm_plan_t last_plan{};        // plan of the last successful gemm_run
    bool has_plan = false;
};

namespace {

gemm_status_t fail(gemm_handle_t h, gemm_status_t s, const std::string& msg) {
    if (h) h->err = msg;
    return s;
}

gemm_status_t cuda_fail(gemm_handle_t h, const char* what, cudaError_t e) {
    return fail(h, GEMM_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Time model of one config on one shape, in microseconds, used to choose the config and the
// schedule.  A k-iteration of a cluster costs the CTA's FLOPs at the tensor rate scaled by the
// config's efficiency; the exposed epilogue moves one CTA row block of C; a stream-K fix-up costs
// one partial write plus one partial read per contributing cluster at a per-SM copy rate.
struct Schedule {
    int clusters = 0;
    int stream_k = 0;
    int dp_tiles = 0;
    double est_us = 0.0;
};

constexpr double kFlopPerUsPerSm = 8192.0 * 1900.0;   // dense f16 FLOP per SM-clock x clock (MHz)
constexpr double kSmBytesPerUs = 150.0e3;             // one SM's copy rate to or from L2 (B/us)
constexpr double kLaunchUs = 2.0;                     // prologue and pipeline fill of one launch
constexpr double kStreamKUs = 4.5;                    // measured fixed cost of a stream-K schedule (partial
                                                      // stores, flag release and acquire, the extra unit)
constexpr int kMaxSplit = 8;                          // clusters sharing one tile (split-K)
// Stream-K ranges start at staggered k offsets, so concurrent clusters share few operand lines in
// L2.  Once A and B together fill most of L2 those iterations come largely from DRAM and run slower
// than data-parallel ones.  Splitting only the partial last wave then beats splitting a wave and a
// half (GB300, f16: 4096 x 4096 x 16384 324 vs 386 us, 4096 x 4096 x 8192 176 vs 188 us, 8192^3 625
// vs 628 us), while 4096^3, whose operands fit, keeps the longer ranges (88 vs 92 us).  A factor of
// 1.2 on the stream-K iterations, over the fixed stream-K cost, reproduces those choices.
constexpr double kL2FitBytes = 80.0e6;
constexpr double kSkIterSlowdown = 1.2;

Schedule schedule(const ConfigDesc& d, double eff, int64_t M, int64_t N, int64_t K, int P, int stream_k,
                  int out_bytes, float beta) {
    const int64_t bm = block_m(d);
    const int64_t T = ((M + bm - 1) / bm) * ((N + d.block_n - 1) / d.block_n);
    const int64_t kt = (K + d.block_k - 1) / d.block_k;
    const double t_iter = 2.0 * 128.0 * d.block_n * d.block_k / (eff * kFlopPerUsPerSm);
    const double t_epi = 128.0 * d.block_n * out_bytes * (beta != 0.0f ? 2.0 : 1.0) / kSmBytesPerUs;
    const double t_part = 128.0 * d.block_n * 4.0 / kSmBytesPerUs;
    // Data-parallel: whole waves of whole tiles.
    Schedule best;
    best.clusters = (int)std::min<int64_t>(T, P);
    best.est_us = kLaunchUs + (double)((T + P - 1) / P) * kt * t_iter + t_epi;
    if (stream_k == 0 || kt < 2) return best;
    const double operand_bytes = ((double)M * K + (double)K * N) * d.in_bytes;
    const double sk_slow = operand_bytes > kL2FitBytes ? kSkIterSlowdown : 1.0;
    auto consider = [&](int C, int64_t dp_tiles) {
        const int64_t sk_iters = (T - dp_tiles) * kt;
        const int64_t base = sk_iters / C, extra = sk_iters % C;
        if (base < 1) return;
        const int64_t per = base + (extra ? 1 : 0);
        // Partials the busiest head adds: the ranges that start strictly inside one tile.
        int64_t srcs = 0, run = 0, run_tile = -1;
        for (int64_t c = 1; c < C; ++c) {
            const int64_t st = c * base + std::min<int64_t>(c, extra);
            if (st % kt == 0) continue;
            run = (st / kt == run_tile) ? run + 1 : 1;
            run_tile = st / kt;
            srcs = std::max(srcs, run);
        }
        if (srcs > kMaxSplit - 1) return;
        Schedule s;
        s.clusters = C;
        s.stream_k = 1;
        s.dp_tiles = (int)dp_tiles;
        // The fix-up, costed as one head reading every other part's partial.  (A clean split runs as a
        // reduce-scatter, which moves less per SM; the planner keeps the head's cost for it, measured
        // to choose no worse than before on the small-M and long-K shapes.)
        const double fix = (1 + srcs) * t_part;
        s.est_us = kLaunchUs + kStreamKUs + (double)(dp_tiles / C) * kt * t_iter + per * t_iter * sk_slow + fix + t_epi;
        if (stream_k == 1 ? (!best.stream_k || s.est_us < best.est_us) : s.est_us < best.est_us * 0.99) best = s;
    };
    if (T > P) {
        if (T % P != 0) {
            consider(P, (T / P - 1) * P);   // the last wave and a half split K-wise: long ranges, few partials
            consider(P, (T / P) * P);       // only the partial last wave: short ranges, more partials per tile
        }
    } else {
        for (int64_t split = 2; split <= kMaxSplit; ++split)  // fewer tiles than clusters: split K
            consider((int)std::min<int64_t>(P, T * split), 0);
    }
    return best;
}

// Tile rows per raster group.  Each group re-reads every B panel, so fewer groups read less of B; a
// group's A panels should stay in L2 while its waves walk along N.  Up to 16 tile rows: one or two
// groups of at most 8 (square waves).  Beyond: as few groups of at most 16 rows as cover them, while a
// group's A panels take at most 64 MiB.  8192^3 (32 rows of 256): two groups of 16 read 995 MB of DRAM
// per launch against 1046 MB for four groups of 8, and run 1-2 % faster; 6144^2 x 4096: two groups of 12.
int raster_group_for(int tiles_m, int block_m, int64_t K, int in_bytes) {
    if (tiles_m <= 16) return std::min(tiles_m, 8);
    const int groups = (tiles_m + 15) / 16;
    const int g = (tiles_m + groups - 1) / groups;
    if ((double)g * block_m * (double)K * in_bytes > 64.0 * 1024 * 1024) return 8;
    return g;
}

// One product as the kernels see it.  transpose() gives C^T = op(B)^T op(A)^T: M and N swap and
// each operand's stored array is reused with the opposite layout code.  A B stored K x N (N
// contiguous, ROW) is the M-contiguous COL operand A' of the transposed product, a B stored N x K
// (COL) its K-contiguous ROW A'; an A stored M x K (ROW) is the COL operand B' (stored N' x K'),
// an A stored K x M (COL) the ROW B' (stored K' x N').
struct Problem {
    int64_t M, N, K;
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    int la, lb;
};

Problem transpose(const Problem& q) {
    return Problem{q.N, q.M, q.K, q.B, q.ldb, q.A, q.lda, q.lb == GEMM_ROW ? GEMM_COL : GEMM_ROW,
                   q.la == GEMM_ROW ? GEMM_COL : GEMM_ROW};
}

// Whether the CUDA-core kernel can take a product: a few rows of C, 16-bit operands, A row-major and
// B stored N x K, both with 16-byte row pitches, K a multiple of 8.
bool gemv_applies(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int din, int la, int lb, int b_q4) {
    return !b_q4 && (din == GEMM_F16 || din == GEMM_BF16) && M >= 1 && M <= kGemvMaxM && N >= 1 && K >= 8 &&
           la == GEMM_ROW && lb == GEMM_COL && K % 8 == 0 && (lda * 2) % 16 == 0 && (ldb * 2) % 16 == 0 &&
           K < (1LL << 30);
}

// Whether a call takes the CUDA-core kernel: on request (skinny 2) or automatically.
bool use_gemv(int skinny, int config, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int din, int la,
              int lb, int b_q4) {
    if (skinny == 2) return true;
    return skinny == -1 && config == -1 && N > 64 && gemv_applies(M, N, K, lda, ldb, din, la, lb, b_q4);
}

// Whether a call computes the transposed product: only on request (skinny 1), or automatically for
// a few rows of C against many columns when the config is automatic.
bool use_transposed(int skinny, int config, int64_t M, int64_t N, int b_q4) {
    if (b_q4) return false;
    if (skinny == 1) return true;
    return skinny == -1 && config == -1 && M <= 64 && N > 64;
}

// How gemm_run_q4_0 computes a product.
enum Q4Route {
    Q4_FUSED = 0,       // the tensor-core kernel with dequantisation warps (config 6)
    Q4_GEMV = 1,        // the CUDA-core kernel that dequantises as it multiplies (M <= 8)
    Q4_TWO_PASS = 2,    // the separate dequantisation pass into the handle's workspace, then the f16 GEMM
};

constexpr double kDequantBytesPerUs = 3.7e6;          // measured rate of the separate pass (read + write)

bool q4_gemv_applies(int64_t M, int64_t lda, int la) {
    return M >= 1 && M <= kGemvMaxM && la == GEMM_ROW && (lda * 2) % 16 == 0;
}

// Estimated time of the separate pass over N x K weights (18 bytes read and 64 written per block).
double q4_dequant_us(int64_t N, int64_t K) {
    return kLaunchUs + static_cast<double>(N) * (K / 32) * (18 + 64) / kDequantBytesPerUs;
}

Schedule plan_schedule(const gemm_plan_t& pl, int64_t M, int64_t N, int64_t K, const int* slots, int cluster_cap,
                       int stream_k, int dout, float beta) {
    int s = slots[pl.config];
    if (cluster_cap > 0) s = std::min(s, cluster_cap);
    return schedule(kConfigs[pl.config], kConfigEfficiency[pl.config], M, N, K, s, stream_k, elt_bytes(dout), beta);
}

gemm_status_t plan_impl(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int din, int dout,
                        int la, int lb, float beta, const int* slots, int config, int stream_k, int cluster_cap,
                        gemm_plan_t* out, std::string* err, int b_q4, int c_trans);

// The route of a Q4_0 product and its plan (the fused kernel's, or the f16 GEMM's after the
// separate pass).  config >= 0 without Q4_0 weights asks for the separate pass and that config;
// skinny 2 asks for the CUDA-core kernel.  Automatically: the CUDA-core kernel for M <= 8, else
// the faster of the fused kernel and the separate pass by the time model (the fused kernel
// dequantises B once per row of output tiles, the pass once in all).
gemm_status_t plan_q4(int64_t M, int64_t N, int64_t K, int64_t lda, int la, int64_t ldbq, int64_t ldc, int dout,
                      float beta, const int* slots, int config, int stream_k, int skinny, int cluster_cap,
                      gemm_plan_t* out, std::string* err, Q4Route* route) {
    *route = Q4_FUSED;
    const bool two_pass_cfg = config >= 0 && config < kNumConfigs && !kConfigs[config].b_q4;
    gemm_status_t st = plan_impl(M, N, K, lda, ldbq, ldc, GEMM_F16, dout, la, GEMM_COL, beta, slots,
                                 two_pass_cfg ? -1 : config, stream_k, cluster_cap, out, err, 1, 0);
    if (st != GEMM_OK || M == 0 || N == 0 || K == 0) return st;
    if (skinny < -1 || skinny > 2) { *err = "skinny must be -1, 0, 1 or 2"; return GEMM_ERR_INVALID_ARG; }
    if (skinny == 2 || (skinny == -1 && config == -1 && q4_gemv_applies(M, lda, la))) {
        if (!q4_gemv_applies(M, lda, la)) {
            *err = "the CUDA-core Q4_0 kernel takes M <= 8 row-major f16 activations with a 16-byte pitch";
            return GEMM_ERR_UNSUPPORTED;
        }
        std::memset(out, 0, sizeof(*out));
        out->config = -1;
        out->kernels = 1;
        out->gemv = 1;
        *route = Q4_GEMV;
        return GEMM_OK;
    }
    bool two_pass = two_pass_cfg;
    gemm_plan_t f16plan;
    if (two_pass || (config == -1 && M > 64)) {
        st = plan_impl(M, N, K, lda, K, ldc, GEMM_F16, dout, la, GEMM_COL, beta, slots, two_pass_cfg ? config : -1,
                       stream_k, cluster_cap, &f16plan, err, 0, 0);
        if (st != GEMM_OK) return st;
        if (!two_pass) {
            const double fused = plan_schedule(*out, M, N, K, slots, cluster_cap, stream_k, dout, beta).est_us;
            const double sep = q4_dequant_us(N, K) +
                               plan_schedule(f16plan, M, N, K, slots, cluster_cap, stream_k, dout, beta).est_us;
            two_pass = sep < fused;
        }
    }
    if (two_pass) {
        *out = f16plan;
        out->q4_dequant = 1;
        out->kernels += 1;
        out->workspace_bytes += round_up(N * K * 2, 256);
        *route = Q4_TWO_PASS;
    }
    return GEMM_OK;
}

// Pure host planning: validation, config choice, grid, stream-K split and workspace.
//   slots[c]     clusters of config c that fit on the device at once
//   cluster_cap  optional cap on launched clusters (0 = none)
//   b_q4         1: B is Q4_0 weights (N rows of K/32 18-byte blocks, ldb = row pitch in bytes)
gemm_status_t plan_impl(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int din, int dout,
                        int la, int lb, float beta, const int* slots, int config, int stream_k, int cluster_cap,
                        gemm_plan_t* out, std::string* err, int b_q4 = 0, int c_trans = 0) {
    std::memset(out, 0, sizeof(*out));
    out->config = -1;
    if (M < 0 || N < 0 || K < 0) { *err = "M, N and K must be >= 0"; return GEMM_ERR_INVALID_ARG; }
    const int64_t kMaxDim = (int64_t)1 << 31;
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) { *err = "M, N and K must be < 2^31"; return GEMM_ERR_INVALID_ARG; }
    if (din != GEMM_F16 && din != GEMM_BF16 && !is_f8(din)) {
        *err = "dtype_in must be GEMM_F16, GEMM_BF16, GEMM_E4M3 or GEMM_E5M2"; return GEMM_ERR_INVALID_ARG;
    }
    if (dout != GEMM_F16 && dout != GEMM_BF16 && dout != GEMM_F32) { *err = "dtype_out must be F16, BF16 or F32"; return GEMM_ERR_INVALID_ARG; }
    if ((la != GEMM_ROW && la != GEMM_COL) || (lb != GEMM_ROW && lb != GEMM_COL)) { *err = "layout must be GEMM_ROW or GEMM_COL"; return GEMM_ERR_INVALID_ARG; }
    const int in_bytes = elt_bytes(din);
    if (is_f8(din) && (la != GEMM_ROW || lb != GEMM_COL)) {
        *err = "8-bit inputs need K-major operands (layoutA GEMM_ROW, layoutB GEMM_COL)"; return GEMM_ERR_UNSUPPORTED;
    }
    const int64_t a_inner = la == GEMM_ROW ? K : M;
    const int64_t b_inner = lb == GEMM_ROW ? N : K;
    if (lda < std::max<int64_t>(1, a_inner)) { *err = "lda too small"; return GEMM_ERR_INVALID_ARG; }
    if (b_q4) {
        if (din != GEMM_F16) { *err = "Q4_0 weights take f16 activations"; return GEMM_ERR_INVALID_ARG; }
        if (K % 32 != 0) { *err = "K must be a multiple of 32 (whole Q4_0 blocks)"; return GEMM_ERR_INVALID_ARG; }
        if (ldb < std::max<int64_t>(1, K / 32 * 18) || ldb % 2 != 0) {
            *err = "ldbq must be even and at least K/32*18 bytes"; return GEMM_ERR_INVALID_ARG;
        }
    } else if (ldb < std::max<int64_t>(1, b_inner)) { *err = "ldb too small"; return GEMM_ERR_INVALID_ARG; }
    // (In the transposed product the kernel's rows are C's columns: C's pitch covers M here.)
    if (ldc < std::max<int64_t>(1, c_trans ? M : N)) { *err = "ldc too small"; return GEMM_ERR_INVALID_ARG; }
    if (config < -1 || config >= kNumConfigs) { *err = "no such config"; return GEMM_ERR_UNSUPPORTED; }
    if (config >= 0 && kConfigs[config].b_q4 != b_q4) {
        *err = b_q4 ? "this config does not take Q4_0 weights" : "this config only takes Q4_0 weights";
        return GEMM_ERR_UNSUPPORTED;
    }
    if (config >= 0 && kConfigs[config].in_bytes != in_bytes) {
        *err = "this config is built for another input width"; return GEMM_ERR_UNSUPPORTED;
    }
    if (stream_k < -1 || stream_k > 1) { *err = "stream_k must be -1, 0 or 1"; return GEMM_ERR_INVALID_ARG; }
    if (M == 0 || N == 0) { out->kernels = 0; return GEMM_OK; }
    if (K == 0) { out->kernels = 1; return GEMM_OK; }

    auto slots_of = [&](int c) {
        int s = slots[c];
        if (cluster_cap > 0) s = std::min(s, cluster_cap);
        return s;
    };
    const int out_bytes = elt_bytes(dout);
    int best = config;
    if (best < 0) {
        double best_us = 1e300;
        for (int c = 0; c < kNumConfigs; ++c) {
            const int s = slots_of(c);
            if (s <= 0 || kConfigs[c].b_q4 != b_q4 || kConfigs[c].in_bytes != in_bytes) continue;
            const Schedule sc = schedule(kConfigs[c], kConfigEfficiency[c], M, N, K, s, stream_k, out_bytes, beta);
            if (sc.est_us < best_us * (1.0 - 1e-9)) { best_us = sc.est_us; best = c; }
        }
        if (best < 0) { *err = "no config fits on this device"; return GEMM_ERR_UNSUPPORTED; }
    }
    const ConfigDesc& d = kConfigs[best];
    const int P = slots_of(best);
    if (P <= 0) { *err = "clusters of this config do not fit"; return GEMM_ERR_UNSUPPORTED; }
    const Schedule sc = schedule(d, kConfigEfficiency[best], M, N, K, P, stream_k, out_bytes, beta);
    out->config = best;
    out->cta_group = d.cta_group;
    out->block_m = block_m(d);
    out->block_n = d.block_n;
    out->block_k = d.block_k;
    out->stages = d.stages;
    out->tiles_m = (int)((M + out->block_m - 1) / out->block_m);
    out->tiles_n = (int)((N + out->block_n - 1) / out->block_n);
    out->clusters = sc.clusters;
    out->raster_group = raster_group_for(out->tiles_m, out->block_m, K, in_bytes);
    // TMA stores move 128-byte rows: each epilogue warp must drain whole ones (a 64-wide tile with
    // 16-bit output does not: its eight warps take 32 columns each).
    const int warp_cols = d.block_n / (d.b_q4 ? 1 : 2);
    out->tma_store = (!c_trans && (ldc * out_bytes) % 16 == 0 && warp_cols * out_bytes >= 128) ? 1 : 0;
    out->transposed = c_trans;
    // Q4_0 rows are read with 4-byte loads: a pitch that is not a multiple of 4 bytes is repacked
    // (as 16-bit units) to a 16-byte pitch.
    out->repack_b = b_q4 ? (ldb % 4 != 0) : (ldb * in_bytes) % 16 != 0;
    out->repack_a = (lda * in_bytes) % 16 != 0;
    // The repack moves 16-bit units: an 8-bit operand needs an even pitch and an even row.
    if (is_f8(din) && ((out->repack_a && (lda % 2 || a_inner % 2)) || (out->repack_b && (ldb % 2 || b_inner % 2)))) {
        *err = "8-bit operands with an odd pitch or odd K whose pitch is not a multiple of 16 bytes";
        return GEMM_ERR_UNSUPPORTED;
    }
    const int64_t unit = 16 / in_bytes;      // elements per 16 bytes
    int64_t ws = 0;
    if (out->repack_a) ws += round_up((la == GEMM_ROW ? M : K) * round_up(a_inner, unit) * in_bytes, 256);
    if (out->repack_b && b_q4) ws += round_up(N * round_up(K / 32 * 9, 8) * 2, 256);
    else if (out->repack_b) ws += round_up((lb == GEMM_ROW ? K : N) * round_up(b_inner, unit) * in_bytes, 256);
    if (sc.stream_k) {
        out->stream_k = 1;
        out->dp_tiles = sc.dp_tiles;
        out->sk_partial_bytes = round_up((int64_t)sc.clusters * cluster_ctas(d) * 128 * d.block_n * 4, 256);
    }
    out->workspace_bytes = ws + out->sk_partial_bytes;
    out->kernels = 1 + ((out->repack_a || out->repack_b) ? 1 : 0);
    return GEMM_OK;
}

uint32_t make_idesc(int din, int a_mn, int b_mn, int mma_m, int mma_n) {
    // tcgen05 instruction descriptor, kind::f16: D f32 (bits 4-5 = 1); A/B format 0 f16, 1 bf16
    // (bits 7-9, 10-12); A/B major 0 K, 1 MN (bits 15, 16); N >> 3 (bits 17-22); M >> 4 (24-28).
    // kind::f16: 0 f16, 1 bf16; kind::f8f6f4: 0 E4M3, 1 E5M2 (same fields)
    const uint32_t fmt = (din == GEMM_BF16 || din == GEMM_E5M2) ? 1u : 0u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(mma_n >> 3) << 17) | ((uint32_t)(mma_m >> 4) << 24);
}

// Tensor-map encoder used by the launch: cached per handle, or direct.
using TmapFn = std::function<gemm_status_t(const TmapDesc&, CUtensorMap*)>;

gemm_status_t encode_tmap(PFN_cuTensorMapEncodeTiled_v12000 encode, const TmapDesc& d, CUtensorMap* out) {
    const cuuint64_t dims[3] = {d.dims[0], d.dims[1], d.dims[2]};
    const cuuint64_t strides[2] = {d.strides[0], d.strides[1]};
    const cuuint32_t box[3] = {d.box[0], d.box[1], d.box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(out, d.dt, (cuuint32_t)d.rank, const_cast<void*>(d.ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Everything the GEMM launch needs once operands are TMA-addressable.
struct LaunchArgs {
    const gemm_plan_t* plan;
    int64_t M, N, K;
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    void* C;
    int64_t ldc;
    int din, dout, la, lb;
    float alpha, beta;
    const void* bias;
    unsigned long long* status;
    unsigned long long timeout_ns;
    long long debug_skip_stage;
    int raster_group;           // 0 = the plan's
    float* sk_partials;
    unsigned* sk_flags;
    unsigned epoch;
    cudaStream_t stream;
    bool force_2d;              // tuning: one 2-D box per slab even where a 3-D box would do
    int c_trans = 0;            // the product is C^T (see Problem / transpose)
    bool pdl = true;            // launch with programmatic stream serialization
    bool k_alternate = true;    // whole tiles of odd waves walk K downwards (L2 reuse between waves)
    const DevInfo* dev = nullptr;  // the device's cluster capacities (split parts as clusters); null: not used
    int* split_cluster_out = nullptr;  // receives KernelParams::rs_cluster of the launch
};

// Whether a stream-K schedule splits every tile over the same number S of consecutive clusters with
// equal k ranges, S dividing the config's epilogue warp count (8, or 4 with Q4_0 B): the kernel then
// reduces the partials as a reduce-scatter (each part finishes 1/S of the tile's epilogue blocks)
// instead of through one head per tile.
bool rs_split(int64_t dp_tiles, int64_t clusters, int64_t tiles, int64_t k_tiles, int epi_warps) {
    if (dp_tiles != 0 || tiles <= 0 || clusters % tiles != 0) return false;
    const int64_t S = clusters / tiles;
    return S >= 2 && epi_warps % S == 0 && k_tiles % S == 0;
}

// Encode the tensor maps, fill the kernel parameters and launch the planned config.
gemm_status_t launch_planned(const LaunchArgs& a, const TmapFn& tmap, const char** what, cudaError_t* cuda_err) {
    const gemm_plan_t& plan = *a.plan;
    const ConfigDesc* d = config_desc(plan.config);
    const CUtensorMapDataType tin = is_f8(a.din) ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                    : a.din == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint64_t ib = (uint64_t)elt_bytes(a.din);
    const uint32_t ce = (uint32_t)(128 / ib);     // K elements of one 128-byte swizzle span
    // B columns one TMA box covers: a CTA's share of one MMA's N.
    const int mma_n = std::min(d->block_n, 256);
    const uint32_t b_box_n = (uint32_t)(mma_n / d->cta_group);
    const uint32_t bk = (uint32_t)d->block_k;
    const uint32_t kchunks = bk / ce;
    const uint64_t M = (uint64_t)a.M, N = (uint64_t)a.N, K = (uint64_t)a.K;
    CUtensorMap ta, tb, tc;
    std::memset(&tc, 0, sizeof(tc));
    // Where the extents divide evenly, a 3-D view (64-element slabs as the outer dimension) lets one
    // TMA instruction fill a whole operand stage; otherwise one 2-D box per 64-element slab.
    int a_3d = 0, b_3d = 0;
    const bool allow_3d = !a.force_2d;
    *what = "tensor map of A";
    gemm_status_t st = GEMM_ERR_CUDA;
    if (a.la == GEMM_ROW) {  // K-major
        if (allow_3d && K % ce == 0) {
            st = tmap(tmap3d(a.A, tin, ce, M, K / ce, (uint64_t)a.lda * ib, 128, ce, 128, kchunks), &ta);
            a_3d = st == GEMM_OK;
        }
        if (!a_3d) st = tmap(tmap2d(a.A, tin, K, M, (uint64_t)a.lda * ib, ce, 128), &ta);
    } else {                 // M-major
        if (allow_3d && M % 64 == 0) {
            st = tmap(tmap3d(a.A, tin, 64, K, M / 64, (uint64_t)a.lda * 2, 128, 64, bk, 2), &ta);
            a_3d = st == GEMM_OK;
        }
        if (!a_3d) st = tmap(tmap2d(a.A, tin, M, K, (uint64_t)a.lda * 2, 64, bk), &ta);
    }
    if (st != GEMM_OK) return st;
    *what = "tensor map of B";
    st = GEMM_ERR_CUDA;
    if (d->b_q4) {           // B is read by the kernel's dequantisation warps, not by TMA
        std::memset(&tb, 0, sizeof(tb));
        st = GEMM_OK;
    } else if (a.lb == GEMM_ROW) {  // N-major
        if (allow_3d && N % 64 == 0) {
            st = tmap(tmap3d(a.B, tin, 64, K, N / 64, (uint64_t)a.ldb * 2, 128, 64, bk, b_box_n / 64), &tb);
            b_3d = st == GEMM_OK;
        }
        if (!b_3d) st = tmap(tmap2d(a.B, tin, N, K, (uint64_t)a.ldb * 2, 64, bk), &tb);
    } else {                 // K-major
        if (allow_3d && d->block_n <= 256 && K % ce == 0) {
            st = tmap(tmap3d(a.B, tin, ce, N, K / ce, (uint64_t)a.ldb * ib, 128, ce, b_box_n, kchunks), &tb);
            b_3d = st == GEMM_OK;
        }
        if (!b_3d) st = tmap(tmap2d(a.B, tin, K, N, (uint64_t)a.ldb * ib, ce, b_box_n), &tb);
    }
    if (st != GEMM_OK) return st;
    const int eb = elt_bytes(a.dout);
    const bool c_aligned = (reinterpret_cast<uintptr_t>(a.C) % 16) == 0 && (a.ldc * eb) % 16 == 0;
    const int use_tma_store = (plan.tma_store && c_aligned && !a.c_trans) ? 1 : 0;
    if (use_tma_store) {
        *what = "tensor map of C";
        const CUtensorMapDataType tcd = a.dout == GEMM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                        : a.dout == GEMM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const uint32_t box0 = a.dout == GEMM_F32 ? 32 : 64;   // one 128-byte line per row
        st = tmap(tmap2d(a.C, tcd, N, M, (uint64_t)a.ldc * eb, box0, 32), &tc);
        if (st != GEMM_OK) return st;
    }
    KernelParams p;
    std::memset(&p, 0, sizeof(p));
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.tiles_m = plan.tiles_m;
    p.tiles_n = plan.tiles_n;
    p.num_tiles = plan.tiles_m * plan.tiles_n;
    p.k_tiles = (int)((a.K + d->block_k - 1) / d->block_k);
    p.raster_group = a.raster_group > 0 ? std::min(a.raster_group, plan.tiles_m) : plan.raster_group;
    p.a_mn = a.la == GEMM_COL ? 1 : 0;
    p.b_mn = (a.lb == GEMM_ROW && !d->b_q4) ? 1 : 0;
    if (d->b_q4) {
        p.bq = static_cast<const uint8_t*>(a.B);
        p.ldbq = a.ldb;
        p.kblocks = (int)(a.K / 32);
    }
    p.a_3d = a_3d;
    p.b_3d = b_3d;
    p.idesc = make_idesc(a.din, p.a_mn, p.b_mn, 128 * d->cta_group, mma_n);
    p.C = a.C;
    p.ldc = a.ldc;
    p.bias = a.bias;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.use_tma_store = use_tma_store;
    p.c_trans = a.c_trans;
    p.c_vec_ok = c_aligned ? 1 : 0;
    p.bias_vec_ok = (a.bias != nullptr && (reinterpret_cast<uintptr_t>(a.bias) % 16) == 0) ? 1 : 0;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.debug_skip_stage = a.debug_skip_stage;
    p.k_alternate = a.k_alternate ? 1 : 0;
    if (plan.stream_k) {
        const long long sk_total = (long long)(p.num_tiles - plan.dp_tiles) * p.k_tiles;
        p.sk_enabled = 1;
        p.dp_tiles = plan.dp_tiles;
        p.sk_base = sk_total / plan.clusters;
        p.sk_extra = (int)(sk_total % plan.clusters);
        p.sk_partials = a.sk_partials;
        p.sk_flags = a.sk_flags;
        p.epoch = a.epoch;
        const int S = plan.clusters / p.num_tiles;   // whole tiles split over S clusters each: reduce-scatter
        if (rs_split(plan.dp_tiles, plan.clusters, p.num_tiles, p.k_tiles, d->b_q4 ? 4 : 8)) p.sk_rs = S;
    }
    // The transposed skinny product's split parts exchange their blocks inside a thread-block cluster
    // when every tile's cluster of S CTAs fits on the device at once.
    int launch_cluster = cluster_ctas(*d);
    if (p.sk_rs > 1 && a.c_trans && a.dev != nullptr && d->cta_group == 1 && d->block_n == 64 && !d->b_q4) {
        const int i = p.sk_rs == 2 ? 0 : p.sk_rs == 4 ? 1 : p.sk_rs == 8 ? 2 : -1;
        if (i >= 0 && a.dev->rs_slots[plan.config][i] >= p.num_tiles) {
            p.rs_cluster = 1;
            launch_cluster = p.sk_rs;
        }
    }
    if (a.split_cluster_out) *a.split_cluster_out = p.rs_cluster;
    *what = "GEMM kernel launch";
    cudaError_t e = config_launch(plan.config, a.dout == GEMM_F32 ? OUT_F32 : (a.dout == GEMM_F16 ? OUT_F16 : OUT_BF16),
                                  plan.clusters * cluster_ctas(*d), launch_cluster, a.stream, a.pdl, ta, tb, tc, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *cuda_err = e;
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

// Repack the operands whose byte pitch TMA cannot use into `ws` (16-byte pitch), both in one
// launch.  Updates the operand pointers and leading dimensions; counts launches.
cudaError_t repack_operands(const gemm_plan_t& plan, int64_t M, int64_t N, int64_t K, int la, int lb, void* ws,
                            const void** A, int64_t* lda, const void** B, int64_t* ldb, int num_sms,
                            cudaStream_t s, bool pdl, int64_t* launches, const char** what, int b_q4 = 0,
                            int in_bytes = 2) {
    char* w = static_cast<char*>(ws);
    RepackJobs jobs{};
    // 8-bit operands (in_bytes 1) move as pairs: their pitch and row length are even (checked by the plan).
    const int64_t pair = in_bytes == 1 ? 2 : 1;
    if (plan.repack_a) {
        const int64_t rows = la == GEMM_ROW ? M : K;
        const int64_t cols = (la == GEMM_ROW ? K : M) / pair;
        const int64_t ld = round_up(cols, 8);
        jobs.job[jobs.n++] = RepackJob{static_cast<const uint16_t*>(*A), *lda / pair, reinterpret_cast<uint16_t*>(w),
                                       ld, rows, cols};
        *A = w;
        *lda = ld * pair;
        w += round_up(rows * ld * 2, 256);
    }
    if (plan.repack_b && b_q4) {   // Q4_0 rows (ldb in bytes, even) moved as 16-bit units
        const int64_t cols = K / 32 * 9;
        const int64_t ld = round_up(cols, 8);
        jobs.job[jobs.n++] = RepackJob{static_cast<const uint16_t*>(*B), *ldb / 2, reinterpret_cast<uint16_t*>(w), ld,
                                       N, cols};
        *B = w;
        *ldb = ld * 2;
    } else if (plan.repack_b) {
        const int64_t rows = lb == GEMM_ROW ? K : N;
        const int64_t cols = (lb == GEMM_ROW ? N : K) / pair;
        const int64_t ld = round_up(cols, 8);
        jobs.job[jobs.n++] = RepackJob{static_cast<const uint16_t*>(*B), *ldb / pair, reinterpret_cast<uint16_t*>(w),
                                       ld, rows, cols};
        *B = w;
        *ldb = ld * pair;
    }
    if (jobs.n == 0) return cudaSuccess;
    *what = "repack of the operands";
    cudaError_t e = launch_repack_u16(jobs, num_sms, s, pdl);
    if (e != cudaSuccess) return e;
    ++*launches;
    return cudaSuccess;
}

gemm_status_t get_tmap_cached(gemm_handle_t h, const TmapDesc& key, CUtensorMap* out) {
    for (const TmapEntry& e : h->cache)
        if (e.key == key) { *out = e.map; return GEMM_OK; }
    if (h->faults & FAULT_TMAP) return fail(h, GEMM_ERR_CUDA, "cuTensorMapEncodeTiled: forced failure (GEMM_TEST_FAIL=tmap)");
    CUtensorMap m;
    if (encode_tmap(h->dev.encode, key, &m) != GEMM_OK) {
        char buf[256];
        std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed: rank %d dims {%llu,%llu,%llu} box {%u,%u,%u}",
                      key.rank, (unsigned long long)key.dims[0], (unsigned long long)key.dims[1],
                      (unsigned long long)key.dims[2], key.box[0], key.box[1], key.box[2]);
        return fail(h, GEMM_ERR_CUDA, buf);
    }
    const size_t kCacheSize = 32;
    if (h->cache.size() < kCacheSize) {
        h->cache.push_back(TmapEntry{key, m});
    } else {
        h->cache[h->cache_next] = TmapEntry{key, m};
        h->cache_next = (h->cache_next + 1) % kCacheSize;
    }
    *out = m;
    return GEMM_OK;
}

gemm_status_t ensure_buffer(gemm_handle_t h, void** buf, size_t* have, size_t bytes, const char* what) {
    if (bytes <= *have) return GEMM_OK;
    if (h->faults & FAULT_ALLOC) return fail(h, GEMM_ERR_OOM, std::string(what) + ": forced failure (GEMM_TEST_FAIL=alloc)");
    if (*buf) { cudaFree(*buf); *buf = nullptr; *have = 0; }
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(h, GEMM_ERR_OOM, std::string(what) + " cudaMalloc: " + cudaGetErrorString(e));
    }
    *buf = p;
    *have = bytes;
    return GEMM_OK;
}

struct DeviceGuard {
    int prev = -1;
    bool changed = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
            if (cudaSetDevice(dev) == cudaSuccess) changed = true;
        }
    }
    ~DeviceGuard() {
        if (changed) cudaSetDevice(prev);
    }
};

}  // namespace

namespace gb300 {

const ConfigDesc* config_desc(int id) { return (id >= 0 && id < kNumConfigs) ? &kConfigs[id] : nullptr; }

const void* config_kernel(int id, int out) {
    switch (id) {
        case 0: return cfg0_kernel(out);
        case 1: return cfg1_kernel(out);
        case 2: return cfg2_kernel(out);
        case 3: return cfg3_kernel(out);
        case 4: return cfg4_kernel(out);
        case 5: return cfg5_kernel(out);
        case 6: return cfg6_kernel(out);
        case 7: return cfg7_kernel(out);
        case 8: return cfg8_kernel(out);
        case 9: return cfg9_kernel(out);
        case 10: return cfg10_kernel(out);
        default: return nullptr;
    }
}

cudaError_t config_launch(int id, int out, int grid_ctas, int cluster, cudaStream_t stream, bool pdl,
                          const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c, const KernelParams& p) {
    const ConfigDesc* d = config_desc(id);
    if (!d) return cudaErrorInvalidValue;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)grid_ctas, 1, 1);
    lc.blockDim = dim3((unsigned)d->threads, 1, 1);
    lc.dynamicSmemBytes = (size_t)d->smem_bytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = pdl ? 2 : 1;
    switch (id) {
        case 0: return cfg0_launch(out, lc, a, b, c, p);
        case 1: return cfg1_launch(out, lc, a, b, c, p);
        case 2: return cfg2_launch(out, lc, a, b, c, p);
        case 3: return cfg3_launch(out, lc, a, b, c, p);
        case 4: return cfg4_launch(out, lc, a, b, c, p);
        case 5: return cfg5_launch(out, lc, a, b, c, p);
        case 6: return cfg6_launch(out, lc, a, b, c, p);
        case 7: return cfg7_launch(out, lc, a, b, c, p);
        case 8: return cfg8_launch(out, lc, a, b, c, p);
        case 9: return cfg9_launch(out, lc, a, b, c, p);
        case 10: return cfg10_launch(out, lc, a, b, c, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gb300

extern "C" {

void gemm_options_default(gemm_options_t* opt) {
    if (!opt) return;
    std::memset(opt, 0, sizeof(*opt));
    opt->struct_size = (int)sizeof(gemm_options_t);
    opt->config = -1;
    opt->timeout_ms = 2000;
    opt->sync_check = 0;
    opt->raster_group = 0;
    opt->max_clusters = 0;
    opt->debug_skip_stage = -1;
    opt->stream_k = -1;
    opt->skinny = -1;
    opt->pdl = 1;
}

const char* gemm_status_string(gemm_status_t s) {
    switch (s) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
        case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
        case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
        case GEMM_ERR_OOM: return "GEMM_ERR_OOM";
        default: return "GEMM_ERR_UNKNOWN";
    }
}

int gemm_num_configs(void) { return kNumConfigs; }

gemm_status_t gemm_config_info(int id, gemm_config_info_t* out) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    const ConfigDesc* d = config_desc(id);
    if (!d) return GEMM_ERR_UNSUPPORTED;
    out->id = d->id;
    out->cta_group = d->cta_group;
    out->block_m = block_m(*d);
    out->block_n = d->block_n;
    out->block_k = d->block_k;
    out->stages = d->stages;
    out->smem_bytes = d->smem_bytes;
    out->threads = d->threads;
    out->b_q4_0 = d->b_q4;
    out->in_bytes = d->in_bytes;
    return GEMM_OK;
}

gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                        gemm_dtype_t dtype_in, gemm_dtype_t dtype_out, gemm_layout_t layoutA, gemm_layout_t layoutB,
                        float beta, int num_sms, int max_clusters, int config, int stream_k, gemm_plan_t* out) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    if (num_sms <= 0) return GEMM_ERR_INVALID_ARG;
    if (max_clusters <= 0) max_clusters = num_sms / 2;
    int slots[kNumConfigs];
    for (int c = 0; c < kNumConfigs; ++c) {
        const ConfigDesc& d = kConfigs[c];
        slots[c] = d.cta_group == 1 ? num_sms : max_clusters;
    }
    std::string err;
    gemm_status_t st = plan_impl(M, N, K, lda, ldb, ldc, dtype_in, dtype_out, layoutA, layoutB, beta, slots, config,
                                 stream_k, 0, out, &err);
    if (st != GEMM_OK || M == 0 || N == 0 || K == 0) return st;
    if (use_gemv(-1, config, M, N, K, lda, ldb, dtype_in, layoutA, layoutB, 0)) {
        std::memset(out, 0, sizeof(*out));
        out->config = -1;
        out->kernels = 1;
        out->gemv = 1;
        return GEMM_OK;
    }
    if (!use_transposed(-1, config, M, N, 0)) return st;
    const Problem q = transpose(Problem{M, N, K, nullptr, lda, nullptr, ldb, layoutA, layoutB});
    return plan_impl(q.M, q.N, K, q.lda, q.ldb, ldc, dtype_in, dtype_out, q.la, q.lb, beta, slots, config, stream_k, 0,
                     out, &err, 0, 1);
}

gemm_status_t gemm_create(gemm_handle_t* out, int device, const gemm_options_t* opt) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    gemm_options_t o;
    gemm_options_default(&o);
    if (opt) {
        if (opt->struct_size != (int)sizeof(gemm_options_t)) return GEMM_ERR_INVALID_ARG;
        o = *opt;
    }
    if (o.config < -1 || o.config >= kNumConfigs || o.timeout_ms <= 0 || o.raster_group < 0 || o.max_clusters < 0 ||
        o.stream_k < -1 || o.stream_k > 1 || o.pdl < 0 || o.pdl > 1)
        return GEMM_ERR_INVALID_ARG;
    int count = 0;
    cudaError_t e = cudaGetDeviceCount(&count);
    if (e != cudaSuccess) { cudaGetLastError(); return GEMM_ERR_CUDA; }
    if (device < 0 || device >= count) return GEMM_ERR_INVALID_ARG;

    gemm_ctx* h = new (std::nothrow) gemm_ctx();
    if (!h) return GEMM_ERR_OOM;
    h->device = device;
    h->opt = o;
    h->faults = read_fault_env();
    if (const char* r = std::getenv("GEMM_TMA_RANK")) h->force_2d = std::atoi(r) == 2;
    if (const char* r = std::getenv("GEMM_K_ORDER")) h->k_forward = std::string(r) == "forward";
    DeviceGuard guard(device);
    gemm_status_t st = query_device(device, (h->faults & FAULT_OPTIN) != 0, &h->dev);
    if (st != GEMM_OK) {
        delete h;
        return st;
    }
    e = cudaMalloc(&h->d_status, 64);
    if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, 64);
    // One flag per (CTA of the grid, epilogue warp) for the stream-K hand-off.
    const size_t flag_bytes = (size_t)h->dev.num_sms * 8 * sizeof(unsigned);
    if (e == cudaSuccess) e = cudaMalloc(&h->sk_flags, flag_bytes);
    if (e == cudaSuccess) e = cudaMemset(h->sk_flags, 0, flag_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        if (h->d_status) cudaFree(h->d_status);
        if (h->sk_flags) cudaFree(h->sk_flags);
        delete h;
        return GEMM_ERR_OOM;
    }
    *out = h;
    return GEMM_OK;
}

gemm_status_t gemm_destroy(gemm_handle_t h) {
    if (!h) return GEMM_OK;
    {
        DeviceGuard guard(h->device);
        cudaDeviceSynchronize();
        if (h->ws) cudaFree(h->ws);
        if (h->d_status) cudaFree(h->d_status);
        if (h->sk_flags) cudaFree(h->sk_flags);
        if (h->sk_part) cudaFree(h->sk_part);
        if (h->q4_ws) cudaFree(h->q4_ws);
    }
    delete h;
    return GEMM_OK;
}

const char* gemm_last_error(gemm_handle_t h) { return h ? h->err.c_str() : "null handle"; }

int64_t gemm_launch_count(gemm_handle_t h) { return h ? h->launches : 0; }

gemm_status_t gemm_last_plan(gemm_handle_t h, gemm_plan_t* out) {
    if (!h || !out || !h->has_plan) return GEMM_ERR_INVALID_ARG;
    *out = h->last_plan;
    return GEMM_OK;
}

gemm_status_t gemm_get_device_status(gemm_handle_t h, void* stream) {
    if (!h) return GEMM_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(h, "cudaStreamSynchronize", e);
    unsigned long long word = 0;
    e = cudaMemcpy(&word, h->d_status, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(h, "reading the status word", e);
    if (word == 0) return GEMM_OK;
    e = cudaMemset(h->d_status, 0, sizeof(word));
    if (e != cudaSuccess) return cuda_fail(h, "clearing the status word", e);
    // An aborted launch may leave stream-K flags raised; reset them so that no later launch (a graph
    // replay repeats its epoch) can take one for a fresh partial.
    e = cudaMemset(h->sk_flags, 0, (size_t)h->dev.num_sms * 8 * sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(h, "clearing the stream-K flags", e);
    const unsigned code = (unsigned)(word & 0xff);
    const unsigned role = (unsigned)((word >> 8) & 0xff);
    const unsigned stage = (unsigned)((word >> 16) & 0xffff);
    const unsigned tile = (unsigned)(word >> 32);
    static const char* roles[] = {"?", "producer", "mma", "epilogue"};
    char buf[256];
    std::snprintf(buf, sizeof(buf), "device wait expired: code %u role %s tile %u stage %u", code,
                  roles[role < 4 ? role : 0], tile, stage);
    h->err = buf;
    return GEMM_ERR_TIMEOUT;
}

}  // extern "C"

namespace {

// The handle's raster_group option, when set, replaces the planner's choice in the plan itself, so
// that gemm_last_plan reports the group the kernel runs with.
void apply_raster_option(const gemm_ctx* h, gemm_plan_t* plan) {
    if (h->opt.raster_group > 0 && plan->tiles_m > 0) plan->raster_group = std::min(h->opt.raster_group, plan->tiles_m);
}

// The body of gemm_run and gemm_run_q4_0 (b_q4 = 1: B is Q4_0 weights at row pitch ldb bytes).
gemm_status_t run_impl(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                       int64_t ldb, void* C, int64_t ldc, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                       gemm_layout_t layoutA, gemm_layout_t layoutB, float alpha, float beta, const void* bias,
                       void* stream, int b_q4) {
    if (!h) return GEMM_ERR_INVALID_ARG;
    h->err.clear();
    gemm_plan_t plan;
    std::string err;
    gemm_status_t st = plan_impl(M, N, K, lda, ldb, ldc, dtype_in, dtype_out, layoutA, layoutB, beta, h->dev.slots,
                                 h->opt.config, h->opt.stream_k, h->opt.max_clusters, &plan, &err, b_q4);
    if (st != GEMM_OK) return fail(h, st, err);
    apply_raster_option(h, &plan);
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C) return fail(h, GEMM_ERR_INVALID_ARG, "C is NULL");
    if (K > 0 && (!A || !B)) return fail(h, GEMM_ERR_INVALID_ARG, "A or B is NULL");
    if (K > 0 && (reinterpret_cast<uintptr_t>(A) % 16) != 0)
        return fail(h, GEMM_ERR_ALIGNMENT, "A must be 16-byte aligned");
    if (K > 0 && (reinterpret_cast<uintptr_t>(B) % (b_q4 ? 2 : 16)) != 0)
        return fail(h, GEMM_ERR_ALIGNMENT, b_q4 ? "Q4_0 weights must be 2-byte aligned" : "B must be 16-byte aligned");
    if (b_q4 && K > 0 && !plan.repack_b && (reinterpret_cast<uintptr_t>(B) % 4) != 0) {
        // The rows start 2 bytes past a 4-byte boundary: repack them like an odd pitch.
        plan.repack_b = 1;
        plan.workspace_bytes += round_up(N * round_up(K / 32 * 9, 8) * 2, 256);
        plan.kernels = 2;
    }
    if (K > 0 && use_gemv(h->opt.skinny, h->opt.config, M, N, K, lda, ldb, dtype_in, layoutA, layoutB, b_q4)) {
        if (!gemv_applies(M, N, K, lda, ldb, dtype_in, layoutA, layoutB, b_q4) ||
            (reinterpret_cast<uintptr_t>(B) % 16) != 0)
            return fail(h, GEMM_ERR_UNSUPPORTED, "the CUDA-core small-M kernel does not take this product");
        DeviceGuard guard(h->device);
        if (h->faults & FAULT_LAUNCH) return fail(h, GEMM_ERR_CUDA, "kernel launch: forced failure (GEMM_TEST_FAIL=launch)");
        GemvParams gp{A, lda * 2, B, ldb * 2, C, ldc, bias, alpha, beta, (int)M, (int)N, (int)K};
        const int out_kind = dtype_out == GEMM_F32 ? OUT_F32 : (dtype_out == GEMM_F16 ? OUT_F16 : OUT_BF16);
        cudaError_t e = launch_gemv(out_kind, dtype_in == GEMM_BF16, gp, h->dev.num_sms, static_cast<cudaStream_t>(stream),
                                    h->opt.pdl != 0);
        if (e != cudaSuccess) return cuda_fail(h, "small-M kernel launch", e);
        h->launches += 1;
        gemm_plan_t gplan{};
        gplan.config = -1;
        gplan.kernels = 1;
        gplan.gemv = 1;
        h->last_plan = gplan;
        h->has_plan = true;
        if (h->opt.sync_check) return gemm_get_device_status(h, stream);
        return GEMM_OK;
    }
    // The product the kernels compute: C itself, or C^T for a few rows of C against many columns.
    Problem q{M, N, K, A, lda, B, ldb, layoutA, layoutB};
    const bool trans = K > 0 && use_transposed(h->opt.skinny, h->opt.config, M, N, b_q4);
    if (trans) {
        q = transpose(q);
        st = plan_impl(q.M, q.N, K, q.lda, q.ldb, ldc, dtype_in, dtype_out, q.la, q.lb, beta, h->dev.slots,
                       h->opt.config, h->opt.stream_k, h->opt.max_clusters, &plan, &err, 0, 1);
        if (st != GEMM_OK) return fail(h, st, err);
    }
    DeviceGuard guard(h->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int out_kind = dtype_out == GEMM_F32 ? OUT_F32 : (dtype_out == GEMM_F16 ? OUT_F16 : OUT_BF16);
    if (h->faults & FAULT_LAUNCH) return fail(h, GEMM_ERR_CUDA, "kernel launch: forced failure (GEMM_TEST_FAIL=launch)");

    if (K == 0) {
        cudaError_t e = launch_scale_bias(out_kind, C, ldc, bias, beta, M, N, h->dev.num_sms, s, h->opt.pdl != 0);
        if (e != cudaSuccess) return cuda_fail(h, "scale/bias kernel launch", e);
        h->launches += 1;
    } else {
        const void* a_ptr = q.A;
        const void* b_ptr = q.B;
        int64_t lda_eff = q.lda, ldb_eff = q.ldb;
        const char* what = "";
        if (plan.repack_a || plan.repack_b) {
            st = ensure_buffer(h, &h->ws, &h->ws_bytes, (size_t)(plan.workspace_bytes - plan.sk_partial_bytes),
                               "workspace allocation");
            if (st != GEMM_OK) return st;
            cudaError_t e = repack_operands(plan, q.M, q.N, K, q.la, q.lb, h->ws, &a_ptr, &lda_eff, &b_ptr, &ldb_eff,
                                            h->dev.num_sms, s, h->opt.pdl != 0, &h->launches, &what, b_q4,
                                            elt_bytes(dtype_in));
            if (e != cudaSuccess) return cuda_fail(h, what, e);
        }
        if (plan.stream_k) {
            void* part = h->sk_part;
            st = ensure_buffer(h, &part, &h->sk_part_bytes, (size_t)plan.sk_partial_bytes, "stream-K partials");
            h->sk_part = static_cast<float*>(part);
            if (st != GEMM_OK) return st;
            if (++h->epoch == 0) ++h->epoch;
        }
        LaunchArgs la{&plan, q.M, q.N, K, a_ptr, lda_eff, b_ptr, ldb_eff, C, ldc, dtype_in, dtype_out, q.la, q.lb,
                      alpha, beta, bias, h->d_status, (unsigned long long)h->opt.timeout_ms * 1000000ull,
                      h->opt.debug_skip_stage, h->opt.raster_group, h->sk_part, h->sk_flags, h->epoch, s,
                      h->force_2d, trans ? 1 : 0, h->opt.pdl != 0, !h->k_forward, &h->dev, &plan.split_cluster};
        TmapFn tmap = [h](const TmapDesc& desc, CUtensorMap* m) { return get_tmap_cached(h, desc, m); };
        cudaError_t ce = cudaSuccess;
        st = launch_planned(la, tmap, &what, &ce);
        if (st != GEMM_OK) return ce != cudaSuccess ? cuda_fail(h, what, ce) : st;
        h->launches += 1;
    }
    h->last_plan = plan;
    h->has_plan = true;
    if (h->opt.sync_check) return gemm_get_device_status(h, stream);
    return GEMM_OK;
}

}  // namespace

extern "C" {

gemm_status_t gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                       int64_t ldb, void* C, int64_t ldc, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                       gemm_layout_t layoutA, gemm_layout_t layoutB, float alpha, float beta, const void* bias,
                       void* stream) {
    return run_impl(h, M, N, K, A, lda, B, ldb, C, ldc, dtype_in, dtype_out, layoutA, layoutB, alpha, beta, bias,
                    stream, 0);
}

gemm_status_t gemm_run_q4_0(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                            gemm_layout_t layoutA, const void* Bq, int64_t ldbq, void* C, int64_t ldc,
                            gemm_dtype_t dtype_out, float alpha, float beta, const void* bias, void* stream) {
    if (!h) return GEMM_ERR_INVALID_ARG;
    h->err.clear();
    gemm_plan_t plan;
    std::string err;
    Q4Route route;
    gemm_status_t st = plan_q4(M, N, K, lda, layoutA, ldbq, ldc, dtype_out, beta, h->dev.slots, h->opt.config,
                               h->opt.stream_k, h->opt.skinny, h->opt.max_clusters, &plan, &err, &route);
    if (st != GEMM_OK) return fail(h, st, err);
    apply_raster_option(h, &plan);
    if (route == Q4_FUSED || M == 0 || N == 0 || K == 0)
        return run_impl(h, M, N, K, A, lda, Bq, ldbq, C, ldc, GEMM_F16, dtype_out, layoutA, GEMM_COL, alpha, beta,
                        bias, stream, 1);
    if (!C) return fail(h, GEMM_ERR_INVALID_ARG, "C is NULL");
    if (!A || !Bq) return fail(h, GEMM_ERR_INVALID_ARG, "A or B is NULL");
    if ((reinterpret_cast<uintptr_t>(A) % 16) != 0) return fail(h, GEMM_ERR_ALIGNMENT, "A must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(Bq) % 2) != 0)
        return fail(h, GEMM_ERR_ALIGNMENT, "Q4_0 weights must be 2-byte aligned");
    DeviceGuard guard(h->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (h->faults & FAULT_LAUNCH) return fail(h, GEMM_ERR_CUDA, "kernel launch: forced failure (GEMM_TEST_FAIL=launch)");
    if (route == Q4_GEMV) {
        GemvParams gp{A, lda * 2, Bq, ldbq, C, ldc, bias, alpha, beta, (int)M, (int)N, (int)K};
        const int out_kind = dtype_out == GEMM_F32 ? OUT_F32 : (dtype_out == GEMM_F16 ? OUT_F16 : OUT_BF16);
        cudaError_t e = launch_gemv_q4_0(out_kind, gp, h->dev.num_sms, s, h->opt.pdl != 0);
        if (e != cudaSuccess) return cuda_fail(h, "Q4_0 small-M kernel launch", e);
        h->launches += 1;
        h->last_plan = plan;
        h->has_plan = true;
        if (h->opt.sync_check) return gemm_get_device_status(h, stream);
        return GEMM_OK;
    }
    // The separate pass writes the N x K f16 weights (pitch K) that the f16 GEMM then reads.
    st = ensure_buffer(h, &h->q4_ws, &h->q4_ws_bytes, (size_t)round_up(N * K * 2, 256), "dequantised weights");
    if (st != GEMM_OK) return st;
    cudaError_t e = launch_dequant_q4_0(Bq, ldbq, N, K, h->q4_ws, K, h->dev.num_sms, s, h->opt.pdl != 0);
    if (e != cudaSuccess) return cuda_fail(h, "Q4_0 dequantisation launch", e);
    h->launches += 1;
    st = run_impl(h, M, N, K, A, lda, h->q4_ws, K, C, ldc, GEMM_F16, dtype_out, layoutA, GEMM_COL, alpha, beta, bias,
                  stream, 0);
    if (st != GEMM_OK) return st;
    h->last_plan.q4_dequant = 1;
    h->last_plan.kernels += 1;
    h->last_plan.workspace_bytes += round_up(N * K * 2, 256);
    return GEMM_OK;
}

gemm_status_t gemm_plan_q4_0(int64_t M, int64_t N, int64_t K, int64_t lda, gemm_layout_t layoutA, int64_t ldbq,
                             int64_t ldc, gemm_dtype_t dtype_out, float beta, int num_sms, int max_clusters,
                             int config, int stream_k, gemm_plan_t* out) {
    if (!out || num_sms <= 0) return GEMM_ERR_INVALID_ARG;
    if (max_clusters <= 0) max_clusters = num_sms / 2;
    int slots[kNumConfigs];
    for (int c = 0; c < kNumConfigs; ++c) {
        const ConfigDesc& d = kConfigs[c];
        slots[c] = d.cta_group == 1 ? num_sms : max_clusters;
    }
    std::string err;
    Q4Route route;
    return plan_q4(M, N, K, lda, layoutA, ldbq, ldc, dtype_out, beta, slots, config, stream_k, -1, 0, out, &err,
                   &route);
}

gemm_status_t gemm_dequant_q4_0(const void* Bq, int64_t ldbq, int64_t N, int64_t K, void* out, int64_t ldo,
                                void* stream) {
    if (N < 0 || K < 0 || K % 32 != 0) return GEMM_ERR_INVALID_ARG;
    if (ldbq < K / 32 * 18 || ldbq % 2 != 0 || ldo < K) return GEMM_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return GEMM_OK;
    if (!Bq || !out) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(Bq) % 2) != 0 || (reinterpret_cast<uintptr_t>(out) % 2) != 0)
        return GEMM_ERR_ALIGNMENT;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    cudaError_t e = launch_dequant_q4_0(Bq, ldbq, N, K, out, ldo, sms, static_cast<cudaStream_t>(stream), true);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

}  // extern "C"

// ============================================================================================
// gemm_run_noalloc: the same product for callers that must not allocate device memory.
//
// Its only scratch need is the operand repack (a 16-bit operand whose byte pitch is not a
// multiple of 16 is copied to a 16-byte pitch before the TMA can read it).  Here that scratch is
// a file-scope device array of fixed size, loaded with this library's module, instead of the
// handle-owned workspace that gemm_run grows with cudaMalloc.  Host code cannot use the array's
// name as a device address: per device, the first call looks the address up with
// cudaGetSymbolAddress (with that device current) and every launch receives that pointer.
// This entry point never uses the stream-K schedule, which needs partial buffers.
// ============================================================================================
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_BYTES];
static __device__ unsigned long long g_noalloc_status;  // bounded-wait word of these calls

constexpr int kNoallocMaxDevices = 64;

struct NoallocDevice {
    std::once_flag once;
    gemm_status_t setup_status = GEMM_ERR_CUDA;
    DevInfo info;
    void* scratch = nullptr;                 // device address of g_noalloc_scratch
    unsigned long long* status = nullptr;    // device address of g_noalloc_status
};

NoallocDevice g_noalloc_dev[kNoallocMaxDevices];

// One-time set-up on the current device `dev`: shared-memory opt-in, occupancy, the tensor-map
// encoder and the device addresses of the file-scope scratch and status word.
void noalloc_setup(int dev, NoallocDevice& nd) {
    nd.setup_status = query_device(dev, false, &nd.info);
    if (nd.setup_status != GEMM_OK) return;
    if (cudaGetSymbolAddress(&nd.scratch, g_noalloc_scratch) != cudaSuccess || !nd.scratch ||
        cudaGetSymbolAddress(reinterpret_cast<void**>(&nd.status), g_noalloc_status) != cudaSuccess ||
        !nd.status) {
        cudaGetLastError();
        nd.scratch = nullptr;
        nd.status = nullptr;
        nd.setup_status = GEMM_ERR_CUDA;
        return;
    }
    if (cudaMemset(nd.status, 0, sizeof(unsigned long long)) != cudaSuccess) {
        cudaGetLastError();
        nd.setup_status = GEMM_ERR_CUDA;
        return;
    }
    nd.setup_status = GEMM_OK;
}

}  // namespace

extern "C" gemm_status_t gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                                          int64_t ldb, void* C, int64_t ldc, gemm_dtype_t dtype_in,
                                          gemm_dtype_t dtype_out, gemm_layout_t layoutA, gemm_layout_t layoutB,
                                          float alpha, float beta, const void* bias, void* stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kNoallocMaxDevices) return GEMM_ERR_UNSUPPORTED;
    NoallocDevice& nd = g_noalloc_dev[dev];
    std::call_once(nd.once, noalloc_setup, dev, std::ref(nd));
    if (nd.setup_status != GEMM_OK) return nd.setup_status;

    // Validation and planning (shared with gemm_plan); the message sink reserves its buffer once
    // per thread, so reporting an invalid argument does not grow it.
    static thread_local std::string sink(64, '\0');
    gemm_plan_t plan;
    gemm_status_t st = plan_impl(M, N, K, lda, ldb, ldc, dtype_in, dtype_out, layoutA, layoutB, beta, nd.info.slots, -1,
                                 0, 0, &plan, &sink);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C) return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B)) return GEMM_ERR_INVALID_ARG;
    if (K > 0 && ((reinterpret_cast<uintptr_t>(A) % 16) != 0 || (reinterpret_cast<uintptr_t>(B) % 16) != 0))
        return GEMM_ERR_ALIGNMENT;
    if (plan.workspace_bytes > (int64_t)GEMM_NOALLOC_SCRATCH_BYTES) return GEMM_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int out_kind = dtype_out == GEMM_F32 ? OUT_F32 : (dtype_out == GEMM_F16 ? OUT_F16 : OUT_BF16);
    if (K == 0) {
        return launch_scale_bias(out_kind, C, ldc, bias, beta, M, N, nd.info.num_sms, s, true) == cudaSuccess
                   ? GEMM_OK : GEMM_ERR_CUDA;
    }
    // Repack into the file-scope scratch.  Every byte the GEMM then reads is written by this call
    // first, so nothing in the scratch has to start at zero.
    const void* a_ptr = A;
    const void* b_ptr = B;
    int64_t lda_eff = lda, ldb_eff = ldb, launches = 0;
    const char* what = "";
    if (repack_operands(plan, M, N, K, layoutA, layoutB, nd.scratch, &a_ptr, &lda_eff, &b_ptr, &ldb_eff,
                        nd.info.num_sms, s, true, &launches, &what, 0, elt_bytes(dtype_in)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    LaunchArgs la{&plan, M, N, K, a_ptr, lda_eff, b_ptr, ldb_eff, C, ldc, dtype_in, dtype_out, layoutA, layoutB,
                  alpha, beta, bias, nd.status, 2000ull * 1000000ull, -1, 0, nullptr, nullptr, 0, s, false};
    const PFN_cuTensorMapEncodeTiled_v12000 enc = nd.info.encode;
    TmapFn tmap = [enc](const TmapDesc& desc, CUtensorMap* m) { return encode_tmap(enc, desc, m); };
    cudaError_t ce = cudaSuccess;
    return launch_planned(la, tmap, &what, &ce);
}

extern "C" gemm_status_t gemm_noalloc_get_device_status(void* stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kNoallocMaxDevices) return GEMM_ERR_UNSUPPORTED;
    NoallocDevice& nd = g_noalloc_dev[dev];
    std::call_once(nd.once, noalloc_setup, dev, std::ref(nd));
    if (nd.setup_status != GEMM_OK) return nd.setup_status;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    unsigned long long word = 0;
    if (cudaMemcpy(&word, nd.status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (word == 0) return GEMM_OK;
    if (cudaMemset(nd.status, 0, sizeof(word)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_ERR_TIMEOUT;
}

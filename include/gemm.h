/*
 * gemm.h - C ABI of the GB300 (sm_103a) dense GEMM library  libgemm_gb300.so
 *
 *   C <- alpha * op(A) * op(B) + beta * C + bias
 *
 * The operation is the dense matrix product C_ij = sum_k A_ik * B_kj
 * (2*M*N*K flops) defined in "Matrix Multiplication: The Operation Behind
 * Modern AI" (opening definition; section "One formula for every matmul"),
 * with f16/bf16 operands and f32 accumulation as in "Optimizing GEMMs using
 * tcgen05 - Part 2" (fp16 in, fp32 accumulate, section 5 onward) and the NT
 * prefill GEMM of "02 - Tiled wmma f16 prefill GEMM" (section 3.2, B stored
 * as od x id, i.e. N x K).  alpha, beta and the per-column bias form the
 * fused epilogue (tcgen05 worklog, section 7: epilogue after the TMEM drain).
 *
 * Conventions
 *   A is M x K, B is K x N, C is M x N; all matrices are dense, element
 *   strides 1, leading dimensions in ELEMENTS.
 *   layoutA  GEMM_ROW: A stored M x K row-major (K contiguous, lda >= K)
 *            GEMM_COL: A stored K x M row-major (M contiguous, lda >= M)
 *   layoutB  GEMM_ROW: B stored K x N row-major (N contiguous, ldb >= N)
 *            GEMM_COL: B stored N x K row-major (K contiguous, ldb >= K)
 *   C        always row-major M x N (ldc >= N), dtype_out.
 *   bias     NULL or N elements of dtype_out, added to every row, NOT scaled
 *            by alpha:  C_ij = alpha * S_ij + beta * C_ij + bias_j.
 *   beta == 0: C is not read (NaN in C does not propagate).
 *   K == 0:   C = beta * C + bias.   M == 0 or N == 0: no-op.
 *   dtype_in in {GEMM_F16, GEMM_BF16} (A and B share it), or the 8-bit floats
 *   GEMM_E4M3 / GEMM_E5M2 (OCP FP8 formats; the matrix-multiplication page's
 *   closing caveat names FP8 tensor cores).  8-bit inputs are multiplied by
 *   kind::f8f6f4 MMAs with f32 accumulation and need K-major operands:
 *   layoutA GEMM_ROW and layoutB GEMM_COL (else GEMM_ERR_UNSUPPORTED); an odd
 *   byte pitch or odd K with an unaligned pitch is GEMM_ERR_UNSUPPORTED too.
 *   dtype_out in {GEMM_F32, GEMM_F16, GEMM_BF16}; the output is rounded to
 *   nearest-even from the f32 epilogue value.
 *
 * Memory and ownership
 *   A, B, C and bias are caller-owned DEVICE pointers on the handle's device;
 *   the library never frees them.  A and B must be 16-byte aligned.  A leading
 *   dimension whose byte pitch is not a multiple of 16 (e.g. lda = 2050 f16) is
 *   legal: the operand is repacked into a handle-owned workspace with a 16-byte
 *   pitch before the product (counted in the call's time).  The handle owns
 *   that workspace (grown on demand, reused), the tensor-map cache and a
 *   device status word.
 *
 * Asynchrony and streams
 *   gemm_run only enqueues work on `stream` (a cudaStream_t passed as void*;
 *   NULL = the legacy default stream) and returns.  Shared-memory opt-in for
 *   every kernel instantiation happens in gemm_create, never inside a call
 *   (cf. the prefill GEMM page, section 3.3: setting the attribute inside a
 *   graph-capture window fails silently).  A call that grows the workspace
 *   allocates device memory, so warm such shapes up before capturing a graph.
 *   Once warm, calls may be captured into a CUDA graph and the graph replayed
 *   any number of times: the stream-K hand-off flags are reset by the kernel
 *   that consumes them, so a replayed launch never sees a stale flag.  Calls
 *   of one handle share its workspace, so they must not run concurrently on
 *   several streams.  A handle must not be used by two host threads at once.
 *
 * Errors
 *   Every entry point returns a gemm_status_t; nothing calls exit or abort.
 *   Detail of the last failure is kept per handle (gemm_last_error).  Device
 *   waits inside the kernels are bounded: on expiry a kernel records
 *   {code, role, tile, stage} in the status word and returns cleanly;
 *   gemm_get_device_status reports it as GEMM_ERR_TIMEOUT.
 *
 * Environment (read once, by gemm_create; none is needed in normal use)
 *   GEMM_TEST_FAIL=optin|tmap|launch|alloc  (tests) force that host error path
 *                                           of the handle; the names combine.
 *   GEMM_TMA_RANK=2     (tuning) one 2-D TMA box per 64-element slab even where
 *                       a 3-D box would fill a whole operand stage.
 *   GEMM_K_ORDER=forward (tuning) every tile walks K upwards; by default whole
 *                       tiles of odd waves walk it downwards for L2 reuse.
 */
#ifndef GB300_GEMM_H
#define GB300_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_ctx* gemm_handle_t; /* opaque, owned by the library */

typedef enum { GEMM_F16 = 0, GEMM_BF16 = 1, GEMM_F32 = 2, GEMM_E4M3 = 3, GEMM_E5M2 = 4 } gemm_dtype_t;
typedef enum { GEMM_ROW = 0, GEMM_COL = 1 } gemm_layout_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,  /* negative size, ld too small, NULL with nonzero size, bad dtype/layout */
    GEMM_ERR_UNSUPPORTED = 2,  /* device is not sm_103 (compute capability 10.3), or no such config   */
    GEMM_ERR_ALIGNMENT = 3,    /* A or B base pointer not 16-byte aligned                              */
    GEMM_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed; see gemm_last_error              */
    GEMM_ERR_TIMEOUT = 5,      /* a bounded device wait expired (read by gemm_get_device_status)        */
    GEMM_ERR_OOM = 6           /* workspace or handle allocation failed                                 */
} gemm_status_t;

/* Options for gemm_create.  Fill with gemm_options_default, then change fields. */
typedef struct {
    int struct_size;      /* sizeof(gemm_options_t), set by gemm_options_default              */
    int config;           /* -1: choose per call; else a kernel config id (gemm_config_info)  */
    int timeout_ms;       /* limit of every bounded device wait (default 2000)                */
    int sync_check;       /* 1: gemm_run synchronises the stream and reads the status word    */
    int raster_group;     /* output-tile rows per raster group; 0 = automatic (gemm_plan)     */
    int max_clusters;     /* cap on persistent clusters (0 = as many as fit on the device)    */
    int debug_skip_stage; /* TEST ONLY: the producer of cluster 0 never issues this k-stage,
                             so the MMA issuer's bounded wait expires (-1 = off)              */
    int stream_k;         /* tail-wave balancing: -1 automatic, 0 off, 1 whenever possible   */
    int skinny;           /* products with few rows of C: -1 automatic (config -1 only): the
                             CUDA-core kernel for M <= 8 with B stored N x K (16-bit, K a
                             multiple of 8, 16-byte row pitch), else C^T = op(B)^T op(A)^T
                             for M <= 64 < N; 0 never; 1 always C^T; 2 always the CUDA-core
                             kernel (GEMM_ERR_UNSUPPORTED where it does not apply)            */
    int pdl;              /* 1 (default): launch with programmatic stream serialization, so a
                             kernel's set-up (barriers, tensor memory, descriptor prefetch)
                             overlaps the end of the kernel before it on the stream; each
                             kernel still waits for its predecessors to complete before it
                             touches global memory.  0: plain stream order               */
} gemm_options_t;

/* Description of a kernel configuration. */
typedef struct {
    int id;
    int cta_group;     /* 1: one CTA per output tile; 2: a 2-SM cluster issues cta_group::2 MMAs */
    int block_m;       /* output-tile rows (128 * cta_group)                                      */
    int block_n;       /* output-tile columns (= MMA N)                                           */
    int block_k;       /* K elements per pipeline stage (64 = one 128-byte swizzle span)          */
    int stages;        /* depth of the shared-memory ring                                         */
    int smem_bytes;    /* dynamic shared memory per CTA                                           */
    int threads;       /* threads per CTA                                                         */
    int b_q4_0;        /* 1: B is Q4_0 weights dequantised in shared memory (gemm_run_q4_0 only)  */
    int in_bytes;      /* operand element size: 2 (f16 / bf16) or 1 (E4M3 / E5M2)                */
} gemm_config_info_t;

/* What gemm_run would do for a problem (pure host computation, no device needed). */
typedef struct {
    int config;            /* chosen config id                                              */
    int cta_group, block_m, block_n, block_k, stages;
    int tiles_m, tiles_n;  /* output tiles                                                  */
    int clusters;          /* persistent clusters launched (grid = clusters * cta_group)    */
    int raster_group;      /* tile rows per raster group: up to 16 tile rows, groups of up
                              to 8; beyond, as few groups of at most 16 as cover them
                              while a group's A panels take at most 64 MiB, else 8.  In
                              gemm_last_plan, the handle's raster_group option when set */
    int tma_store;         /* 1: epilogue moves C boxes by TMA (C_in loads when beta != 0,
                              then tensor stores); 0: per-row st.global / ld.global        */
    int repack_a, repack_b;/* 1: operand copied to a 16-byte pitch workspace first          */
    int64_t workspace_bytes; /* repack workspace + stream-K partials                        */
    int kernels;           /* kernel launches the call makes                                */
    int stream_k;          /* 1: the last wave(s) are split evenly by k-iterations          */
    int dp_tiles;          /* tiles walked whole before the stream-K region                 */
    int64_t sk_partial_bytes; /* part of workspace_bytes holding stream-K f32 partials      */
    int transposed;        /* 1: the kernel computes C^T = op(B)^T op(A)^T; tiles_m, tiles_n,
                              block_m, block_n and repack_a/_b then describe that product
                              (its rows are C's columns) and C is written by direct stores    */
    int gemv;              /* 1: the CUDA-core kernel for a few rows of C (no tensor cores, no
                              tiles; config is -1)                                             */
    int q4_dequant;        /* 1 (gemm_run_q4_0): the Q4_0 weights are first dequantised by the
                              separate pass into the handle's workspace; the other fields
                              describe the f16 GEMM that follows (kernels counts both)         */
    int split_cluster;     /* 1 (gemm_last_plan only; gemm_plan, which queries no device, reports
                              0): the split-K parts of each tile ran as one thread-block cluster
                              and exchanged their partial sums through distributed shared memory */
} gemm_plan_t;

/* Fill *opt with defaults (config -1, timeout 2000 ms, no sync check, automatic raster). */
void gemm_options_default(gemm_options_t* opt);

/* Create a handle on CUDA device `device` (opt NULL = defaults).  Checks that the device is
 * sm_103, opts every kernel into its dynamic shared memory, resolves cuTensorMapEncodeTiled and
 * allocates the device status word.  *out is NULL on failure. */
gemm_status_t gemm_create(gemm_handle_t* out, int device, const gemm_options_t* opt);

/* Enqueue C <- alpha*op(A)*op(B) + beta*C + bias on `stream`.  See the conventions above. */
gemm_status_t gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                       const void* A, int64_t lda, const void* B, int64_t ldb,
                       void* C, int64_t ldc,
                       gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                       gemm_layout_t layoutA, gemm_layout_t layoutB,
                       float alpha, float beta, const void* bias, void* stream);

/* gemm_run_q4_0 - the same product with Q4_0-quantised weights as B ("02 . 8m/8m(2) -- Tiled
 * wmma f16 prefill GEMM (LANDED)": section 3.2 gives the block format and the separate dequant
 * pass, section 2.3 names the dequant-in-GEMM fused kernel as its successor).  One of three routes:
 *   - fused: the tensor-core kernel whose dequantisation warps write each B stage into shared
 *     memory (config 6);
 *   - small M: a CUDA-core kernel that dequantises each block in registers as it multiplies
 *     (M <= 8, A row-major with a 16-byte pitch; automatic, or the handle's skinny option 2);
 *   - separate pass: gemm_dequant_q4_0 into a workspace the handle owns (N*K*2 bytes, grown on
 *     demand) followed by the f16 GEMM on it (chosen when the time model says it is faster, or
 *     when the handle's config option names a config without Q4_0 weights, which then runs the
 *     f16 GEMM).
 * Every route computes the same value per element: the dequantised weight rounded to f16, times
 * the f16 activation, summed in f32.
 *   C (M x N) <- alpha * op(A) * W^T + beta * C + bias, W the N x K dequantised weights.
 *   A: f16 activations, layoutA as in gemm_run, 16-byte aligned.
 *   Bq: N rows (one per output column) of K/32 blocks of 18 bytes at a row pitch of ldbq bytes
 *       (ldbq even, >= K/32*18); 2-byte aligned.  Block: little-endian f16 scale d, then 16 bytes
 *       q[0..15]; weight i of the block is the low nibble of q[i], weight 16+i the high nibble;
 *       its value is d * (nibble - 8) rounded to f16, exactly as gemm_dequant_q4_0 writes it, and
 *       the product then runs on the f16 tensor cores with f32 accumulation.
 *   K must be a multiple of 32 (whole blocks).  C, ldc, dtype_out, alpha, beta, bias, stream and
 *   the returned codes are those of gemm_run (GEMM_ERR_UNSUPPORTED for skinny 2 where the
 *   small-M kernel does not apply). */
gemm_status_t gemm_run_q4_0(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                            const void* A, int64_t lda, gemm_layout_t layoutA,
                            const void* Bq, int64_t ldbq,
                            void* C, int64_t ldc, gemm_dtype_t dtype_out,
                            float alpha, float beta, const void* bias, void* stream);

/* gemm_dequant_q4_0 - the separate dequantisation pass of the same page (section 3.2): writes the
 * N x K f16 weights (row n at out + n * ldo elements, ldo >= K) from Q4_0 blocks laid out as for
 * gemm_run_q4_0, on the current device and `stream`.  K a multiple of 32; Bq and out 2-byte
 * aligned.  Needs no handle; returns GEMM_ERR_INVALID_ARG / GEMM_ERR_ALIGNMENT / GEMM_ERR_CUDA. */
gemm_status_t gemm_dequant_q4_0(const void* Bq, int64_t ldbq, int64_t N, int64_t K,
                                void* out, int64_t ldo, void* stream);

/* Free the handle and everything it owns (waits for its device work first).  NULL is a no-op. */
gemm_status_t gemm_destroy(gemm_handle_t h);

/* Static, human-readable name of a status code. */
const char* gemm_status_string(gemm_status_t s);

/* Detail of the handle's last failure ("" if none).  Valid until the next call on h. */
const char* gemm_last_error(gemm_handle_t h);

/* Synchronise `stream`, read and clear the device status word.  Returns GEMM_ERR_TIMEOUT (with
 * role, tile and stage in gemm_last_error) if a bounded wait expired since the last read. */
gemm_status_t gemm_get_device_status(gemm_handle_t h, void* stream);

/* Plan a call without running it: validation, config choice, grid, repack and workspace.
 * beta: as for gemm_run (beta != 0 rules out the TMA-store epilogue, which never reads C);
 * the plan assumes C is 16-byte aligned.  num_sms: the device's SM count (e.g. 152);
 * max_clusters: co-resident 2-SM clusters (0 = num_sms / 2).  config: -1 automatic, else a
 * config id.  stream_k: as in gemm_options_t.  Uses no device. */
gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                        gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                        gemm_layout_t layoutA, gemm_layout_t layoutB, float beta,
                        int num_sms, int max_clusters, int config, int stream_k, gemm_plan_t* out);

/* The same for gemm_run_q4_0 (automatic skinny option): the plan's gemv, q4_dequant or neither
 * field says which of the three routes the call takes. */
gemm_status_t gemm_plan_q4_0(int64_t M, int64_t N, int64_t K, int64_t lda, gemm_layout_t layoutA,
                             int64_t ldbq, int64_t ldc, gemm_dtype_t dtype_out, float beta,
                             int num_sms, int max_clusters, int config, int stream_k, gemm_plan_t* out);

/* Number of kernel configurations and their descriptions (ids 0 .. gemm_num_configs()-1). */
int gemm_num_configs(void);
gemm_status_t gemm_config_info(int id, gemm_config_info_t* out);

/* Kernels launched through this handle since it was created. */
int64_t gemm_launch_count(gemm_handle_t h);

/* The plan of the handle's last successful gemm_run (config, tiles, clusters launched, stream-K
 * split, repacks).  GEMM_ERR_INVALID_ARG before the first call or for NULL arguments. */
gemm_status_t gemm_last_plan(gemm_handle_t h, gemm_plan_t* out);

/* Size of the fixed device scratch that gemm_run_noalloc uses for operand repacks. */
#define GEMM_NOALLOC_SCRATCH_BYTES (32u << 20)

/* gemm_run_noalloc - the same product as gemm_run, for callers that cannot allocate.
 *
 * The pages have no counterpart to this entry point; it exists for the library's users.  Some
 * callers must not allocate device memory: an application whose device memory is owned by
 * another allocator (a framework's caching pool, or a budget carved out up front) cannot let a
 * library call cudaMalloc behind that allocator's back, and a latency-critical loop cannot afford
 * cudaMalloc / cudaFree, which may synchronise the whole device.  This call takes no handle and
 * calls no cudaMalloc, cudaFree or other allocating routine.  Arguments, layouts, semantics and
 * the returned codes are those of gemm_run (on the current device, on `stream`), except:
 *   - Scratch: an operand whose byte pitch is not a multiple of 16 is repacked into a file-scope
 *     device array of GEMM_NOALLOC_SCRATCH_BYTES (32 MiB) that every GPU loading this library's
 *     module holds until the process exits.  A call whose repack needs more than that returns
 *     GEMM_ERR_UNSUPPORTED without launching anything.  Operands with 16-byte pitches use no
 *     scratch at all.
 *   - Set-up: the first call on each device opts the kernels into their shared memory, queries
 *     the device and looks up the scratch's device address (cudaGetSymbolAddress) with that
 *     device current.  Make that first call before any stream capture begins.
 *   - Sharing: every call on a device uses the same scratch, which keeps the previous call's
 *     contents; this call writes every byte it later reads, so nothing has to start at zero.
 *     Calls whose work overlaps on the GPU (for example on two streams) race on the scratch:
 *     order them on one stream or with events.
 *   - Errors: there is no handle, hence no gemm_last_error text.  The return code covers
 *     validation and launch only: a bounded device wait that expires later records into a
 *     library-internal word per device, which gemm_noalloc_get_device_status reads and clears.
 */
gemm_status_t gemm_run_noalloc(int64_t M, int64_t N, int64_t K,
                               const void* A, int64_t lda, const void* B, int64_t ldb,
                               void* C, int64_t ldc,
                               gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                               gemm_layout_t layoutA, gemm_layout_t layoutB,
                               float alpha, float beta, const void* bias, void* stream);

/* gemm_noalloc_get_device_status - synchronise `stream`, then read and clear the status word that
 * gemm_run_noalloc's kernels write on the current device when a bounded wait expires.  Returns
 * GEMM_OK, GEMM_ERR_TIMEOUT (a wait expired since the last read: the output of that call is
 * incomplete) or GEMM_ERR_CUDA.  Like gemm_run_noalloc it allocates nothing; its first call on a
 * device performs the same one-time set-up. */
gemm_status_t gemm_noalloc_get_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_H */

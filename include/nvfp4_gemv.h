/*
 * nvfp4_gemv.h: C ABI of the GB300 (sm_103a) NVFP4 block-scaled batched GEMV.
 *
 * The operation (kernelbot "nvfp4-gemv" submission 103289, `cute_kernel`:
 * each output accumulates a*sfa*b*sfb over K in FP32 and is stored with
 * `.to(Float16)`; submission 69953's docstring names the shapes):
 *
 *   c[m,l] = fp16( sum_{k<K} E2M1(a[m,k,l]) * E4M3(sfa[m,k/16,l])
 *                          * E2M1(b[k,l])   * E4M3(sfb[k/16,l]) )
 *
 * Element formats: E2M1 is FP4 (sign, 2 exponent bits, 1 mantissa bit; no
 * Inf/NaN); E4M3 is finite-only FP8 (0x7F/0xFF are NaN).  Two E2M1 codes are
 * packed per byte along K, the lower k in the low nibble (the pages' torch
 * tensors are `float4_e2m1fn_x2`, so "k is halved").  One E4M3 scale covers
 * 16 consecutive K elements (`sf_vec_size = 16`).
 *
 * Memory layouts (all row-major, batch L outermost; submission 103289's
 * `cute_jit_kernel` gives A the strides (k, 1, m*k) and c the strides
 * (1, 1, m)):
 *   a   : uint8 [L][M][K/2]          packed E2M1, row stride K/2 bytes
 *   b   : uint8 [L][K/2]             packed E2M1 (dense: no N padding)
 *   c   : fp16  [L][M]               output, written, never read
 *   sfa, sfb in one of two layouts, chosen by `sf_layout`:
 *     NVFP4_SF_PLAIN          sfa uint8 [L][M][K/16], sfb uint8 [L][K/16]
 *     NVFP4_SF_PERMUTED_128x4 the pre-permuted tensor [32, 4, rest_m, 4,
 *        rest_k, L] of submission 103289 (`permuted_to_blocked`), stored
 *        L-outermost in 128x4 atoms of 512 bytes: byte (m, kb) of batch l is
 *        at ((l*rest_m + m/128)*rest_k + kb/4)*512 + (m%32)*16
 *        + ((m/32)%4)*4 + kb%4, rest_m = ceil(rows/128), rest_k = ceil(K/64)
 *        (both sized with ceil_div as in submission 69953's
 *        `to_blocked_batch`; padding rows and, when K % 64 != 0, the padding
 *        blocks of the last atom column hold 0x00).
 *        For sfb, rows = 1 (row 0 of each atom is used).
 *        nvfp4_repack_scales() produces this layout from the plain one.
 *
 * Ownership and execution: every pointer is device memory owned by the
 * caller (or memory the device can address, such as mapped pinned host
 * memory).  No call allocates, frees, synchronizes or keeps per-call state
 * (the two wait diagnostics at the end, nvfp4_tensor_wait_timeouts and
 * nvfp4_selftest_bounded_wait, synchronize); all work is enqueued on
 * `stream` (NULL = the legacy default stream), so the compute calls may be
 * captured into CUDA graphs.  Kernels are launched with
 * programmatic stream serialization: they wait for the preceding work on the
 * stream before reading any input, so stream order is preserved.
 *
 * Errors: arguments are validated on the host before anything is launched,
 * and a failing call launches nothing unless it returns NVFP4_ERR_CUDA.
 */
#ifndef NVFP4_GEMV_H
#define NVFP4_GEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t is a pointer to this opaque driver type. */
struct CUstream_st;

typedef enum {
  NVFP4_SF_PLAIN = 0,
  NVFP4_SF_PERMUTED_128x4 = 1
} nvfp4_sf_layout_t;

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_VALUE = 1,     /* NULL pointer with non-empty data, negative size, bad enum */
  NVFP4_ERR_UNSUPPORTED_SHAPE = 2, /* K % 16 != 0, a size beyond the limits below, or a
                                      shape the selected kernel cannot run */
  NVFP4_ERR_MISALIGNED = 3,        /* pointer alignment rule broken (see each call) */
  NVFP4_ERR_CUDA = 4               /* a CUDA runtime call failed; see nvfp4_last_cuda_error() */
} nvfp4_status_t;

/*
 * Batched GEMV, c[m,l] as defined above.
 *
 *   a, b, sfa, sfb : inputs in the layouts above (sf_layout selects the scale layout)
 *   c              : output, fp16 [L][M]
 *   M, K, L        : rows, reduction length (elements), batch count
 *   sf_layout      : NVFP4_SF_PLAIN or NVFP4_SF_PERMUTED_128x4
 *   stream         : CUDA stream (cudaStream_t)
 *
 * Shapes: M, L >= 0 and K >= 0 with K % 16 == 0 (whole 16-element scale
 * blocks; the pages' kernels take K % 64 == 0, their K tile and scale atom
 * `mma_tiler_mnk = (128, 1, 64)`, and K % 64 != 0 runs on the blockwise
 * kernel).  M == 0 or L == 0 is a no-op
 * (pointers may be NULL).  K == 0 writes +0 to every c (a, b, sfa, sfb may be
 * NULL).  Limits: K <= 2^30, M*L < 2^40.
 * Alignment: a and b 16-byte aligned, sfa and sfb 32-byte aligned (the
 * pages' `assumed_align` of 16 and 32), c 2-byte aligned.  (A 16-byte
 * aligned a is never run on the direct kernel, whose 256-bit loads need 32.)
 * Accuracy: on the CUDA-core kernels each 16-element block's dot product is
 * exact and blocks are scaled and summed in FP32; the tensor-core kernel
 * (which nvfp4_gemv runs for large streams in either scale layout, see
 * nvfp4_gemv_plan) sums in FP32 in the MMA's own order.
 * c is rounded to nearest even (overflow gives +-Inf; a NaN scale gives NaN)
 * and stays within 1e-3 * sum|terms| + 1 fp16 ulp of the exact result.
 * Results are bitwise reproducible run to run.  The FP32 summation order
 * follows the launch schedule, which the library picks per shape and scale
 * layout; under one CUDA-core schedule (nvfp4_gemv_explicit) the two layouts
 * give identical bits.
 * Execution detail: before waiting for the preceding work on the stream, the
 * kernel may ask the L2 to prefetch lines of a (a hint that returns no data;
 * every input is read only after that work has completed).
 */
nvfp4_status_t nvfp4_gemv(const void* a, const void* b, const void* sfa, const void* sfb,
                          void* c, int64_t M, int64_t K, int64_t L, int sf_layout,
                          struct CUstream_st* stream);

/*
 * Output activation of nvfp4_gemv_ex and nvfp4_gemm_small_n, applied in fp32
 * to y = alpha * sum + bias before the fp16 rounding: c = fp16(act(y)).  The
 * pages list none; these are the usual MLP activations, with NaN in -> NaN out:
 *   NVFP4_ACT_NONE      act(y) = y
 *   NVFP4_ACT_RELU      act(y) = y > 0 ? y : +0
 *   NVFP4_ACT_SILU      act(y) = y / (1 + exp(-y))
 *   NVFP4_ACT_GELU_TANH act(y) = y/2 * (1 + tanh(sqrt(2/pi) * (y + 0.044715 y^3)))
 *   NVFP4_ACT_GELU_ERF  act(y) = y/2 * (1 + erf(y / sqrt(2)))
 * Accuracy: act is evaluated with CUDA's fp32 expf, tanhf and erff; |act'| <=
 * 1.13 for all five, so c stays within 1.13 * (1e-3 * |alpha| * sum|terms|) + 1
 * fp16 ulp of act applied to the exact value (plus the fp32 evaluation error,
 * a few fp32 ulps).
 */
typedef enum {
  NVFP4_ACT_NONE = 0,
  NVFP4_ACT_RELU = 1,
  NVFP4_ACT_SILU = 2,
  NVFP4_ACT_GELU_TANH = 3,
  NVFP4_ACT_GELU_ERF = 4
} nvfp4_activation_t;

/*
 * Options of nvfp4_gemv_ex.  Zero-initialised fields other than alpha give
 * the plain call; {1.0f, NULL, 0, 0, NVFP4_ACT_NONE} is exactly nvfp4_gemv.
 *
 *   alpha            : fp32 output scale: c = fp16(alpha * sum + bias).  A
 *                      global per-tensor scale of this kind is mentioned in a
 *                      removed docstring line of submission 69575; the pages
 *                      never apply one (alpha = 1).
 *   bias             : NULL, or fp16 [L][M] (row stride M) added after the
 *                      scaling; 2-byte aligned.  With a bias the scaling and the
 *                      addition are one fp32 fused multiply-add before the fp16
 *                      rounding.
 *   b_batch_stride   : bytes from batch l to batch l+1 of b; 0 = K/2 (dense).
 *                      Otherwise >= K/2 and a multiple of 16: b may be row 0 of
 *                      an N-padded [L][N][K/2] buffer such as the one
 *                      submission 103289's host code builds (stride N*K/2).
 *   sfb_batch_stride : bytes from batch l to batch l+1 of sfb; 0 = dense
 *                      (K/16 plain, ceil(K/64)*512 permuted).  Otherwise at least
 *                      that, and a multiple of 4 (plain) or 16 (permuted).
 *   activation       : nvfp4_activation_t, applied last (see above).
 * Violations: a stride below the dense size or an unknown activation ->
 * NVFP4_ERR_INVALID_VALUE; a stride or bias pointer off its alignment ->
 * NVFP4_ERR_MISALIGNED.
 */
typedef struct {
  float alpha;
  const void* bias;
  int64_t b_batch_stride;
  int64_t sfb_batch_stride;
  int32_t activation;
} nvfp4_gemv_options_t;

/*
 * nvfp4_gemv with options (NULL options = nvfp4_gemv).  Same arguments,
 * rules, schedule and accuracy contract; the tolerance scales with |alpha|.
 */
nvfp4_status_t nvfp4_gemv_ex(const void* a, const void* b, const void* sfa, const void* sfb,
                             void* c, int64_t M, int64_t K, int64_t L, int sf_layout,
                             const nvfp4_gemv_options_t* options, struct CUstream_st* stream);

/* The GEMV kernels (CUDA-core kernels 0 and 1 share their arithmetic). */
typedef enum {
  /* Warps load up to 8 rows' 32-byte K chunks straight into registers with
   * 256-bit loads, then compute.  Needs a 32-byte aligned a. */
  NVFP4_KERNEL_DIRECT = 0,
  /* Each lane copies its rows' chunks and scale words into a 3-slot
   * per-warp shared-memory ring with cp.async, so every warp keeps two tasks
   * in flight while it computes one.  The default for every K > 0; needs
   * k_split no larger than the K steps, ceil(K/64 / lanes_per_row). */
  NVFP4_KERNEL_PIPELINED = 1,
  /* The tensor cores' block-scaled MMA (tcgen05 kind::mxf4nvf4, 16-element
   * E4M3 blocks, M = 128 tiles, b padded to N = 16 with zero rows), fed by
   * TMA.  The 128x4 atom of the pre-permuted layout is the MMA's scale
   * layout; plain scales (K % 256 == 0, a sfb batch stride that is a
   * multiple of 16 bytes) arrive as 16 bytes per row and 256-element stage,
   * and the MMA warp writes them out as atoms in shared memory before the
   * MMAs (the same atoms, so the same bits as pre-permuted scales).
   * k_split = CTAs per cluster (1, 2, 4 or 8, at most ceil(K/256))
   * splitting each tile's K range, summed in cluster rank order through
   * distributed shared memory; ctas a multiple of k_split (the clusters are
   * persistent over the L*ceil(M/128) tiles); lanes_per_row = pipeline
   * stages per CTA (2 or 4: 4, 3 or 2 CTAs of 2 stages share an SM, 2 of 4).
   * The MMA sums in fp32 in an order of its own: c meets the same accuracy
   * contract, not the CUDA-core kernels' bits.  The MMA reads scale codes as
   * unsigned magnitudes; the kernel folds every negative sfa or sfb code into
   * the sign bits of the 16 elements it scales before the MMA, so signed,
   * subnormal and NaN codes give the E4M3 result.  nvfp4_gemv runs it with
   * M >= 1024 where it was measured faster than the pipelined kernel: at
   * least 512 MB of A with K <= 8192 (either layout; plain scales with
   * K % 256 == 0 and, through nvfp4_gemv_ex, a sfb batch stride that is a
   * multiple of 16), or, for pre-permuted scales, 128-row tiles
   * (L * ceil(M/128)) filling 80-100% of one wave of 2 CTAs per SM with
   * K >= 6144, or more tiles than that wave holds and at least 128 MB of A
   * (any K); nvfp4_gemm_small_n uses it for N >= 2. */
  NVFP4_KERNEL_TENSOR = 2,
  /* Tensor-core block dots with the scales applied on the CUDA cores: A is
   * streamed by TMA in one box per tile of up to 128 rows (rows handed out to
   * one CTA per SM in units of 8), 512-element K stages (256 when K % 256 !=
   * 0), a ring of lanes_per_row slots (2..32; 0 = the most that fit); the
   * block-scaled MMA runs with unit A scales and constant selector B scales
   * so that it writes each 16-element block's dot to its own accumulator
   * column, and the epilogue adds dot * sfa * sfb in fp32 from the signed
   * E4M3 codes, block by block in K order (bits independent of grid, ring
   * depth and scale layout).  k_split must be 1.  Plain scales need
   * K % 256 == 0.  Selected explicitly only: measured on GB300 it matches the
   * pipelined kernel on the largest streams and is slower on smaller ones. */
  NVFP4_KERNEL_BLOCKDOT = 3,
  /* CUDA cores, any K % 16 == 0: each warp takes a group of 4 rows, each lane
   * whole 16-element blocks (8 bytes of a row of A, one aligned load whatever
   * K % 64 is), b's block decoded once for the 4 rows, then a shuffle sum over
   * the lanes.  Block arithmetic as in kernels 0 and 1; the fp32 sums run in
   * an order fixed by K alone.  lanes_per_row must be 32 and k_split 1.
   * nvfp4_gemv runs it for K % 64 != 0; the other kernels need K % 64 == 0
   * (NVFP4_ERR_UNSUPPORTED_SHAPE otherwise). */
  NVFP4_KERNEL_BLOCKWISE = 4
} nvfp4_kernel_t;

/*
 * nvfp4_gemv with the kernel and launch schedule given instead of chosen
 * (for tuning and for testing every schedule; same arguments, rules and
 * results contract as nvfp4_gemv).  kernel: nvfp4_kernel_t;
 * lanes_per_row in {4, 8, 16, 32}: lanes sharing a row; k_split in
 * {1, 2, 4, 8}: warps splitting a row's K range; ctas in [1, 2^31): grid size.
 * The summation order, and so the last bits of c, depend on (kernel,
 * lanes_per_row, k_split); any valid schedule meets the accuracy contract.
 * Invalid schedule values give NVFP4_ERR_INVALID_VALUE.
 */
nvfp4_status_t nvfp4_gemv_explicit(const void* a, const void* b, const void* sfa,
                                   const void* sfb, void* c, int64_t M, int64_t K, int64_t L,
                                   int sf_layout, int kernel, int lanes_per_row, int k_split,
                                   int64_t ctas, struct CUstream_st* stream);

/*
 * Small-N NVFP4 GEMM (a decode batch of N <= 16 vectors per batch): for each
 * batch l, vector n < N and row m,
 *   c[l][n][m] = fp16(alpha * sum_k E2M1(a[m,k,l]) * E4M3(sfa[m,k/16,l])
 *                                   * E2M1(b[n,k,l]) * E4M3(sfb[n,k/16,l]) + bias[l][n][m]),
 * N GEMVs that share one pass over A.  (Submission 103289's
 * `cute_jit_kernel` gives b a stride of 128 padded columns, made for
 * torch._scaled_mm; here b has the N rows given.)
 * Layouts: a [L][M][K/2] as for nvfp4_gemv; b [L][N][K/2], row n of batch l
 * at b + l*b_batch_stride + n*K/2 (b_batch_stride 0 = N*K/2); scales
 * pre-permuted only: sfa as for nvfp4_gemv, sfb the permuted form of
 * [L][N][K/16] (one 128-row atom block per batch, rows 0..N-1:
 * nvfp4_repack_scales with rows = N), batch stride sfb_batch_stride
 * (0 = (K/64)*512); c fp16 [L][N][M]; bias fp16 [L][N][M] or NULL.
 * N = 1 is nvfp4_gemv_ex with permuted scales (kernel and schedule chosen as
 * nvfp4_gemv chooses them); N >= 2 runs the tensor-core kernel
 * (NVFP4_KERNEL_TENSOR), whose cost does not grow with N.  Shapes: M, L >= 0, 0 <= N <= 16 (N > 16: UNSUPPORTED_SHAPE),
 * K % 64 == 0 (K = 0 gives c = fp16(bias) or zeros).  Alignment: a and b
 * 16 bytes, sfa and sfb 32 bytes; c and bias 2 bytes; batch strides as for
 * nvfp4_gemv_ex.
 */
nvfp4_status_t nvfp4_gemm_small_n(const void* a, const void* b, const void* sfa, const void* sfb,
                                  void* c, int64_t M, int64_t N, int64_t K, int64_t L,
                                  const nvfp4_gemv_options_t* options, struct CUstream_st* stream);

/*
 * nvfp4_gemm_small_n (N >= 1, always the tensor-core kernel, default options)
 * with its schedule given: stages (2 or 4) pipeline stages per CTA, k_split
 * (1, 2, 4 or 8, at most ceil(K/256); 1 when K = 0) CTAs per cluster
 * splitting each 128-row tile's K range, ctas in [1, 2^31) a multiple of
 * k_split.  Invalid values give NVFP4_ERR_INVALID_VALUE.
 */
nvfp4_status_t nvfp4_gemm_small_n_explicit(const void* a, const void* b, const void* sfa,
                                           const void* sfb, void* c, int64_t M, int64_t N,
                                           int64_t K, int64_t L, int stages, int k_split,
                                           int64_t ctas, struct CUstream_st* stream);

/*
 * The tensor-core schedule nvfp4_gemm_small_n uses for N >= 2 (computed for
 * any N in 1..16): stages per CTA, CTAs per cluster, grid size, and
 * optionally (resident_ctas non-NULL) the CTAs of that kernel resident at once
 * on the current device.  Queries the device (occupancy; cached per device).
 */
nvfp4_status_t nvfp4_gemm_small_n_plan(int64_t M, int64_t N, int64_t K, int64_t L,
                                       int* stages, int* k_split, int64_t* ctas,
                                       int* resident_ctas);

/*
 * Scale repack: plain [L][rows][K/16] E4M3 -> the 128x4-atom pre-permuted
 * layout above (submission 69953, `to_blocked_batch`; submission 69575,
 * `blocked_transform_kernel`).  A byte permutation, bit-exact; padding rows
 * rows..128*rest_m-1 of the last atom row, and blocks K/16..4*rest_k-1 of the
 * last atom column when K % 64 != 0, are written as 0x00.  dst must hold
 * nvfp4_permuted_scale_bytes(rows, K, L) bytes and must not overlap src.
 * Use rows = M for sfa and rows = 1 for sfb.
 * Shapes: rows, L >= 0, K % 16 == 0 (empty is a no-op).
 * Alignment: src 4-byte aligned; dst 16-byte aligned.  With K % 256 == 0 and a
 * 16-byte aligned src a shared-memory-free kernel runs; the result is the same.
 */
nvfp4_status_t nvfp4_repack_scales(const void* src, void* dst, int64_t rows, int64_t K,
                                   int64_t L, struct CUstream_st* stream);

/* Bytes of a permuted scale tensor: L * ceil(rows/128) * ceil(K/64) * 512.
 * Returns 0 for invalid arguments (negative sizes or K % 16 != 0). */
size_t nvfp4_permuted_scale_bytes(int64_t rows, int64_t K, int64_t L);

/* Static, human-readable name of a status code. */
const char* nvfp4_status_string(int status);

/* The cudaError_t of the most recent NVFP4_ERR_CUDA on the calling thread
 * (0 if none). */
int nvfp4_last_cuda_error(void);

/* Waits of the tensor-core kernel that gave up: every wait of that kernel on
 * a pipeline barrier is bounded (2 s), and a wait that runs out is counted
 * here and makes its thread skip the rest of its work (the launch's c is
 * then not valid).  Synchronises the device; reset != 0 clears the count
 * after reading it.  Returns the count, or -1 on a CUDA error. */
int nvfp4_tensor_wait_timeouts(int reset);

/* Device self-test of that bounded wait (the one the tensor-core and block-dot
 * kernels use on their pipeline barriers), made so that a wait runs out
 * without hanging anything: one warp initialises two shared-memory barriers
 * for one arrival each, arrives on the first, then waits on phase 0 of each.
 * Expected: *completed = 1 (the first wait returned at once), *gave_up = 1 (the
 * second gave up: nothing arrives on it), *timeouts = 1 (the give-up was
 * counted) and *waited_ns about 2e9 (the wait limit, measured with the global
 * timer).  The self-test has its own counter (nvfp4_tensor_wait_timeouts is
 * not changed) and leaves the context usable.  Synchronises `stream`; takes
 * about 2 s.  NULL outputs give NVFP4_ERR_INVALID_VALUE, a CUDA failure
 * NVFP4_ERR_CUDA. */
nvfp4_status_t nvfp4_selftest_bounded_wait(int* completed, int* gave_up, int* timeouts,
                                           int64_t* waited_ns, struct CUstream_st* stream);

/*
 * Launch plan of nvfp4_gemv, computed on the host only (no GPU needed), for
 * inspection and tests.  kernel = -1 gives the plan nvfp4_gemv uses, an
 * nvfp4_kernel_t value that kernel's plan (NVFP4_ERR_UNSUPPORTED_SHAPE if it
 * cannot run the shape).  num_sms is the device's multiprocessor count and
 * ctas_per_sm the number of the CUDA-core kernel's CTAs resident per SM (pass
 * 0 to use the compiled-in default of 2).  nvfp4_gemv picks: the blockwise
 * kernel for K % 64 != 0; the direct kernel for K = 0 and for plain scales up
 * to 512 KB of A; the tensor-core kernel with M >= 1024 and either at least
 * 512 MB of A with K <= 8192 (plain scales: K % 256 == 0), or, for
 * pre-permuted scales, 80-100% of 2 * num_sms tiles of 128 rows with
 * K >= 6144 or more than 2 * num_sms such tiles with at least 128 MB of A;
 * the pipelined kernel otherwise.
 * For the tensor-core kernel the plan assumes 4 resident 2-stage CTAs (or 2
 * 4-stage ones) per SM (nvfp4_gemm_small_n_plan gives the schedule rule); for the block-dot kernel, one CTA per SM and up to
 * 227 KB of shared memory.
 */
typedef struct {
  int kernel;         /* nvfp4_kernel_t */
  int lanes_per_row;  /* lanes of a warp that share one row (32-byte K chunk
                         each); tensor-core kernel: pipeline stages per CTA;
                         block-dot kernel: ring slots; blockwise: 32 */
  int k_split;        /* warps of a CTA that split one row's K range;
                         tensor-core kernel: CTAs per cluster; block-dot: 1 */
  int rows_per_pass;  /* rows a warp reduces at once; tensor-core and
                         block-dot kernels: 128 (a tile); blockwise: rows a
                         CTA takes at once (8 warps x 4) */
  int threads_per_cta;
  int64_t ctas;       /* grid size */
  int64_t steps;      /* K chunks per lane per row, ceil(K/64 / lanes_per_row);
                         tensor-core kernel: 256-element K stages, ceil(K/256);
                         block-dot kernel: ceil(K/512) (ceil(K/256) when
                         K % 256 != 0); blockwise: ceil(K/16 / 32) */
} nvfp4_gemv_plan_t;

nvfp4_status_t nvfp4_gemv_plan(int64_t M, int64_t K, int64_t L, int sf_layout, int kernel,
                               int num_sms, int ctas_per_sm, nvfp4_gemv_plan_t* out);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GEMV_H */

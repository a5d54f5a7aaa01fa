// Host/device interface between the C ABI layer and the kernels.
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

namespace nvfp4 {

constexpr int kGemvThreads = 256;   // 8 warps per CTA
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kGemvMinCtasPerSm = 2;  // __launch_bounds__ occupancy floor
constexpr int kRowsPerPass = 8;     // rows one warp reduces at once (direct kernel)

// Pipelined (cp.async) kernel: row items per lane per task, ring slots per
// warp, and the per-warp slot size (A chunks [item][lane][32 B], then scale
// words [item][lane][4 B]).
constexpr int kAsyncItems = 4;
constexpr int kAsyncStages = 3;
constexpr int kAsyncStageBytes = kAsyncItems * (32 * 32 + 32 * 4);
constexpr int kAsyncSmemBytes = kGemvWarps * kAsyncStages * kAsyncStageBytes;

enum KernelKind {
  kKernelDirect = 0,
  kKernelAsync = 1,
  kKernelTensor = 2,
  kKernelBlockDot = 3,
  kKernelBlockwise = 4
};

// Everything a GEMV kernel needs, by value (kernel parameter space).
struct GemvParams {
  const uint8_t* a;
  const uint8_t* b;
  const uint8_t* sfa;
  const uint8_t* sfb;
  uint16_t* c;        // fp16 bits
  int64_t M;
  int64_t rows_per_l; // rows visited per batch: M (plain) or 128*rest_m (permuted)
  int64_t rows_total; // rows_per_l * L
  int64_t units_q;    // partition of T = units_q*ctas + units_r units of rows (a unit is
  int32_t units_r;    //   one row, or one aligned row group) evenly over the CTAs
  int32_t prefetch_tasks;  // pipelined kernel: tasks per warp prefetched into L2 (1 or 2)
  int64_t b_stride;   // bytes from batch l to l+1 of b
  int64_t sfb_stride; // bytes from batch l to l+1 of sfb
  float alpha;        // output scale (1 = none)
  const uint16_t* bias;  // fp16 [L][M] added after scaling, or null
  int32_t half_k;     // K/2: bytes of one packed row
  int32_t blocks;     // K/16: scale bytes of one plain row
  int32_t kchunks;    // K/64: 32-byte chunks per row (one per 128x4 atom column)
  int32_t steps;      // ceil(kchunks / lanes_per_row)
  int32_t rest_m;     // ceil(M/128)
  int32_t rest_k;     // ceil(K/64): atom columns of a pre-permuted row
  int32_t activation; // nvfp4_activation_t applied to the output
};

struct GemvPlan {
  int kernel;         // KernelKind
  int lanes_per_row;  // 4, 8, 16 or 32
  int k_split;        // 1, 2, 4 or 8 warps per row range
  int groups;         // pipelined kernel: row groups per pass (1, 2 or 4); direct: 1
  int64_t ctas;
  int64_t steps;
};

// Host-only schedule choice (no CUDA calls) for one kernel, or for the
// kernel the library picks (kernel = -1).  Returns false if the kernel cannot
// run the shape (caller validates the shape first).
bool plan_gemv(int64_t M, int64_t K, int64_t L, bool permuted, int kernel, int num_sms,
               int ctas_per_sm, GemvPlan* out);
// Row groups per pass of the pipelined kernel for a launch shape: enough for
// the longest row-lane range, rounded up to 1, 2 or 4; 2 (several passes)
// when the range needs more than 4.
int async_groups(int64_t M, int64_t L, bool permuted, int lanes_per_row, int k_split,
                 int64_t ctas);
// Rows one warp reduces at once under a plan.
int rows_per_pass(const GemvPlan& plan);

// Occupancy of the GEMV kernel family on the current device (CTAs per SM).
cudaError_t gemv_ctas_per_sm(int* out);

// Scale repack: occupancy (CTAs per SM) and launch over at most max_ctas CTAs.
cudaError_t repack_ctas_per_sm(int* out);
// Any K % 16 == 0: the last atom column of a K % 64 != 0 repack is padded
// with 0x00.
cudaError_t launch_repack(const uint8_t* src, uint8_t* dst, int64_t rows, int64_t K, int64_t L,
                          int64_t max_ctas, cudaStream_t stream);

constexpr int kTcThreadsPerCta = 224;  // tensor-core kernel: 7 warps

// Tensor-core kernel (gemv_tc.cu): N (1..16) rows of b (row n at
// b + l*p.b_stride + n*b_row_stride), c [L][N][M]; stages (2 or 4) per CTA;
// ctas CTAs in clusters of ks, each cluster splitting a 128-row tile's K
// range ks ways.  Pre-permuted scales, or with plain (N = 1, K % 256 == 0,
// p.sfb_stride % 16 == 0) the plain layouts.
cudaError_t launch_gemv_tc(const GemvParams& p, int64_t N, int64_t L, int64_t b_row_stride,
                           int stages, int ks, int64_t ctas, cudaStream_t stream,
                           bool plain = false);
// Clusters of ks tensor-core CTAs that can be resident at once.
cudaError_t tc_max_active_clusters(int stages, int64_t N, int ks, int* out);
// Bounded waits of the tensor-core kernel that gave up (read, then optionally
// cleared; synchronous).
cudaError_t tc_wait_timeouts(int reset, int* out);

// Block-dot kernel (gemv_blockdot.cu): tensor-core 16-element block dots
// (selector scales), E4M3 scales applied on the CUDA cores.  One CTA of
// kBlockDotThreads threads per SM, a ring of `stages` (2..kBlockDotMaxStages)
// K-stage slots of slot_rows rows and blockdot_column_blocks(K) 128-byte
// column blocks; rows handed out in units of blockdot_unit_rows() (8) rows.
// Needs K > 0; plain scales also K % 256 == 0.
constexpr int kBlockDotThreads = 192;
constexpr int kBlockDotMaxStages = 32;
int blockdot_unit_rows(bool permuted);
// 128-byte column blocks per K stage: 2 when K % 256 == 0, else 1.
int blockdot_column_blocks(int64_t K);
// Rows of a ring slot for a launch over `ctas` CTAs (the longest tile).
int blockdot_slot_rows(int64_t M, int64_t L, bool permuted, int64_t ctas);
size_t blockdot_smem_bytes(bool permuted, int column_blocks, int slot_rows, int stages);
// Most ring slots that fit smem_per_cta bytes of dynamic shared memory.
int blockdot_max_stages(bool permuted, int column_blocks, int slot_rows, size_t smem_per_cta);
cudaError_t launch_blockdot(const GemvParams& p, bool permuted, int64_t L, int stages,
                            int64_t ctas, cudaStream_t stream);
cudaError_t blockdot_wait_timeouts(int reset, int* out);

// Blockwise kernel (gemv_blockwise.cu): one 16-element block per lane and
// step, any K % 16 == 0; groups of kBlockwiseRows rows over the grid's warps
// (kGemvThreads threads per CTA).
constexpr int kBlockwiseRows = 4;
cudaError_t launch_gemv_blockwise(const GemvParams& p, bool permuted, int64_t ctas,
                                  cudaStream_t stream);

// Per-layout GEMV launchers (gemv_plain.cu, gemv_permuted.cu).
cudaError_t launch_gemv_plain(const GemvParams& p, const GemvPlan& plan, cudaStream_t stream);
cudaError_t launch_gemv_permuted(const GemvParams& p, const GemvPlan& plan, cudaStream_t stream);
cudaError_t launch_async_plain(const GemvParams& p, const GemvPlan& plan, cudaStream_t stream);
cudaError_t launch_async_permuted(const GemvParams& p, const GemvPlan& plan, cudaStream_t stream);

}  // namespace nvfp4

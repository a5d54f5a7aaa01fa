// C ABI: argument validation, launch planning and dispatch.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>

#include "internal.h"
#include "nvfp4_gemv.h"
#include "selftest.h"

namespace nvfp4 {

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kMaxDevices = 128;
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_gemv_occ[kMaxDevices];
std::atomic<int> g_repack_occ[kMaxDevices];

// Resident clusters of the tensor-core kernel per device, stage count (2, 4),
// column count (1, 2, 4, 8, 16) and cluster size (1, 2, 4, 8); 0 = not queried.
std::atomic<int> g_tc_clusters[kMaxDevices][2][5][4];

constexpr int64_t kMaxK = int64_t(1) << 30;
constexpr int64_t kMaxRows = int64_t(1) << 40;  // M * L
constexpr int64_t kMaxM = (int64_t(1) << 31) - 1;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

nvfp4_status_t cuda_failure(cudaError_t err) {
  g_last_cuda_error = (int)err;
  (void)cudaGetLastError();  // clear a non-sticky launch error
  return NVFP4_ERR_CUDA;
}

// Multiprocessor count and kernel occupancies of the current device, cached
// per device (a benign race: concurrent first calls store the same values).
cudaError_t device_info(int* sms, int* gemv_occ, int* repack_occ) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int s = g_sms[dev].load(std::memory_order_relaxed);
  int g = g_gemv_occ[dev].load(std::memory_order_relaxed);
  int r = g_repack_occ[dev].load(std::memory_order_relaxed);
  if (s <= 0 || g <= 0 || r <= 0) {
    err = cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = gemv_ctas_per_sm(&g);
    if (err != cudaSuccess) return err;
    err = repack_ctas_per_sm(&r);
    if (err != cudaSuccess) return err;
    if (g < 1) g = 1;
    if (r < 1) r = 1;
    g_sms[dev].store(s, std::memory_order_relaxed);
    g_gemv_occ[dev].store(g, std::memory_order_relaxed);
    g_repack_occ[dev].store(r, std::memory_order_relaxed);
  }
  if (sms) *sms = s;
  if (gemv_occ) *gemv_occ = g;
  if (repack_occ) *repack_occ = r;
  return cudaSuccess;
}

nvfp4_status_t validate_gemv_shape(int64_t M, int64_t K, int64_t L, int sf_layout) {
  if (M < 0 || K < 0 || L < 0) return NVFP4_ERR_INVALID_VALUE;
  if (sf_layout != NVFP4_SF_PLAIN && sf_layout != NVFP4_SF_PERMUTED_128x4)
    return NVFP4_ERR_INVALID_VALUE;
  if (K % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (K > kMaxK || M > kMaxM) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (M != 0 && L > kMaxRows / M) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return NVFP4_OK;
}

// a and b 16-byte aligned (submission 103289's `assumed_align=16`), the
// scales 32-byte aligned (its `assumed_align=32`), c 2-byte aligned.  The
// direct kernel's 256-bit loads of a also need a 32-byte aligned a.
nvfp4_status_t validate_gemv_pointers(const void* a, const void* b, const void* sfa,
                                      const void* sfb, const void* c, int64_t K) {
  if (c == nullptr) return NVFP4_ERR_INVALID_VALUE;
  if (K > 0 && (a == nullptr || b == nullptr || sfa == nullptr || sfb == nullptr))
    return NVFP4_ERR_INVALID_VALUE;
  if (!aligned(c, 2)) return NVFP4_ERR_MISALIGNED;
  if (K > 0 && (!aligned(a, 16) || !aligned(b, 16) || !aligned(sfa, 32) || !aligned(sfb, 32)))
    return NVFP4_ERR_MISALIGNED;
  return NVFP4_OK;
}

// The options of a plain nvfp4_gemv call: no output scale or bias, dense b
// and sfb (strides 0 = dense).
const nvfp4_gemv_options_t kDefaultOptions = {1.0f, nullptr, 0, 0, NVFP4_ACT_NONE};

bool activation_ok(int32_t act) { return act >= NVFP4_ACT_NONE && act <= NVFP4_ACT_GELU_ERF; }

// Option checks shared by the entry points that take options.
nvfp4_status_t validate_options(const nvfp4_gemv_options_t& o, int64_t K, int sf_layout) {
  if (o.b_batch_stride < 0 || o.sfb_batch_stride < 0) return NVFP4_ERR_INVALID_VALUE;
  if (!activation_ok(o.activation)) return NVFP4_ERR_INVALID_VALUE;
  if (o.b_batch_stride != 0 && o.b_batch_stride < K / 2) return NVFP4_ERR_INVALID_VALUE;
  if (o.b_batch_stride % 16 != 0) return NVFP4_ERR_MISALIGNED;
  const bool permuted = sf_layout == NVFP4_SF_PERMUTED_128x4;
  const int64_t sfb_dense = permuted ? (K + 63) / 64 * 512 : K / 16;
  if (o.sfb_batch_stride != 0 && o.sfb_batch_stride < sfb_dense) return NVFP4_ERR_INVALID_VALUE;
  if (o.sfb_batch_stride % (permuted ? 16 : 4) != 0) return NVFP4_ERR_MISALIGNED;
  if (o.bias != nullptr && !aligned(o.bias, 2)) return NVFP4_ERR_MISALIGNED;
  return NVFP4_OK;
}

GemvParams make_params(const void* a, const void* b, const void* sfa, const void* sfb, void* c,
                       int64_t M, int64_t K, int64_t L, bool permuted, const GemvPlan& plan,
                       const nvfp4_gemv_options_t& opt) {
  GemvParams p;
  p.a = static_cast<const uint8_t*>(a);
  p.b = static_cast<const uint8_t*>(b);
  p.sfa = static_cast<const uint8_t*>(sfa);
  p.sfb = static_cast<const uint8_t*>(sfb);
  p.c = static_cast<uint16_t*>(c);
  p.M = M;
  p.rest_m = (int32_t)((M + 127) / 128);
  p.rest_k = (int32_t)((K + 63) / 64);
  p.rows_per_l = permuted ? (int64_t)p.rest_m * 128 : M;
  p.rows_total = p.rows_per_l * L;
  p.half_k = (int32_t)(K / 2);
  p.blocks = (int32_t)(K / 16);
  p.kchunks = (int32_t)(K / 64);
  p.steps = (int32_t)plan.steps;
  // rows per partition unit: the pipelined kernel hands permuted-scale rows
  // out in aligned groups of its item rows, everything else row by row
  const int64_t unit =
      (plan.kernel == kKernelAsync && permuted) ? kAsyncItems * (32 / plan.lanes_per_row) : 1;
  const int64_t units = p.rows_total / unit;
  p.units_q = units / plan.ctas;
  p.units_r = (int32_t)(units % plan.ctas);
  // L2 prefetch ahead of the dependency wait: one task per warp when the call
  // gives each warp fewer than 4 tasks (4 KB of A each) on average, else two
  // (measured on GB300: more prefetch delays the first copies of small calls)
  const int64_t four_tasks = plan.ctas * kGemvWarps * 4 * (int64_t)kAsyncItems * 32 * 32;
  const int64_t half_k = K / 2;
  p.prefetch_tasks = (half_k > 0 && M * L >= (four_tasks + half_k - 1) / half_k) ? 2 : 1;
  p.b_stride = opt.b_batch_stride != 0 ? opt.b_batch_stride : K / 2;
  p.sfb_stride = opt.sfb_batch_stride != 0 ? opt.sfb_batch_stride
                                           : (permuted ? (int64_t)p.rest_k * 512 : K / 16);
  p.alpha = opt.alpha;
  p.bias = static_cast<const uint16_t*>(opt.bias);
  p.activation = opt.activation;
  return p;
}

nvfp4_status_t run_gemv(const void* a, const void* b, const void* sfa, const void* sfb, void* c,
                        int64_t M, int64_t K, int64_t L, int sf_layout, const GemvPlan& plan,
                        const nvfp4_gemv_options_t& opt, cudaStream_t stream) {
  const bool permuted = sf_layout == NVFP4_SF_PERMUTED_128x4;
  const GemvParams p = make_params(a, b, sfa, sfb, c, M, K, L, permuted, plan, opt);
  cudaError_t err;
  if (plan.kernel == kKernelBlockwise)
    err = launch_gemv_blockwise(p, permuted, plan.ctas, stream);
  else if (plan.kernel == kKernelBlockDot)
    err = launch_blockdot(p, permuted, L, plan.lanes_per_row, plan.ctas, stream);
  else if (plan.kernel == kKernelTensor)
    err = launch_gemv_tc(p, 1, L, K / 2, plan.lanes_per_row, plan.k_split, plan.ctas, stream,
                         !permuted);
  else if (plan.kernel == kKernelAsync)
    err = permuted ? launch_async_permuted(p, plan, stream) : launch_async_plain(p, plan, stream);
  else
    err = permuted ? launch_gemv_permuted(p, plan, stream) : launch_gemv_plain(p, plan, stream);
  if (err != cudaSuccess) return cuda_failure(err);
  return NVFP4_OK;
}

int log2_small(int64_t v) {  // v in {1, 2, 4, 8, 16}
  int r = 0;
  while ((int64_t(1) << r) < v) ++r;
  return r;
}

// Clusters of ks tensor-core CTAs (stages, N columns) resident at once on the
// current device, cached.
cudaError_t tc_resident_clusters(int stages, int64_t N, int ks, int* out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const int nc = N <= 1 ? 1 : N <= 2 ? 2 : N <= 4 ? 4 : N <= 8 ? 8 : 16;
  std::atomic<int>& slot = g_tc_clusters[dev][stages == 4 ? 1 : 0][log2_small(nc)][log2_small(ks)];
  int v = slot.load(std::memory_order_relaxed);
  if (v <= 0) {
    err = tc_max_active_clusters(stages, N, ks, &v);
    if (err != cudaSuccess) return err;
    if (v < 1) v = 1;
    slot.store(v, std::memory_order_relaxed);
  }
  *out = v;
  return cudaSuccess;
}

// Tensor-core schedule (measured on GB300 over the decode-batch shapes, cold
// L2).  slots2 / slots4 = CTAs of 2 / 4 stages resident at once.
//  * When the L*ceil(M/128) tiles fit in one wave of 4-stage CTAs: 4 stages
//    (two ring slots per MMA chain, so a chain's next copies are in flight
//    while it issues MMAs) and the largest cluster size k_split whose tiles
//    times k_split still fit (at most 4 when more than 8 columns are summed
//    across the cluster, at most 8, each CTA keeping 2 K stages); one CTA per
//    tile and rank.  (M7168_N8_K2048_L4: 11.2 us against 11.8 with the rule
//    below; M7168_N16_K16384_L1: 20.6 against 25.5.)  Tiles filling 80-99% of
//    the wave with 24-32 K stages get no split either: one CTA per tile, which
//    skips the cluster barriers, beat clusters of 2 on every resident CTA
//    by 2.1-3.9% on 9 of 10 such GEMVs and GEMMs in alternating runs and
//    tied on the 10th (e.g. M4096_K7168_L8 23.28 against 23.98 us).
//  * When they fit in one wave of 2-stage CTAs (but not of 4-stage ones): 4
//    stages on every resident 4-stage CTA (persistent), with clusters of 2
//    only when that leaves each rank strictly fewer K stages over the waves
//    of tiles (waves = tiles over resident clusters, rounded up, times the
//    rank's K stages), else no split.  Alternating runs on 9 such small-N
//    GEMMs: the best of (2 or 4 stages) x (cluster 1 or 2) or within 1.3% of
//    it on every one, and 0.9-19% faster than the earlier 2-stage rule (e.g.
//    M4096_N2_K16384_L12 74.2 against 92.1 us, M10240_N4_K16384_L6 91.3
//    against 96.5).
//  * Larger problems: 4 stages on every resident 4-stage CTA (persistent
//    clusters), in clusters of 2 once K has 32 or more stages, else 1.
//    Measured on 9 GEMV shapes of 0.6-1.2 GB (both scale layouts) and 7
//    small-N GEMMs: the best schedule of (2 or 4 stages) x (cluster 1, 2, 4)
//    everywhere but M8192_K12288_L8 (2.5% from it), e.g. M16384_K8192_L16
//    176.6 us against 182.5 with the rule above, M32768_K8192_L4 90.9 against
//    100.4, M16384_N16_K8192_L8 93.5 against 129.1.
void tc_rule(int64_t M, int64_t N, int64_t K, int64_t L, int64_t slots2, int64_t slots4,
             int* stages, int* k_split, int64_t* ctas) {
  const int64_t tiles = L * ((M + 127) / 128);
  const int64_t kst = (K + 255) / 256;
  const int ks_max = N > 8 ? 4 : 8;
  int ks = 1;
  if (tiles <= slots4) {
    while (ks < ks_max && 4 * ks <= kst && tiles * 2 * ks <= slots4) ks *= 2;
    *stages = 4;
    *k_split = ks;
    *ctas = tiles * ks;
    return;
  }
  if (tiles > slots2) {
    ks = kst >= 32 ? 2 : 1;
    const int64_t resident = slots4 / ks > 0 ? slots4 / ks : 1;
    *stages = 4;
    *k_split = ks;
    *ctas = (tiles < resident ? tiles : resident) * ks;
    return;
  }
  const int64_t pairs = slots4 / 2;  // resident clusters of 2 four-stage CTAs
  if (pairs > 0 && kst >= 2) {
    const int64_t w1 = (tiles + slots4 - 1) / slots4 * kst;
    const int64_t w2 = (tiles + pairs - 1) / pairs * ((kst + 1) / 2);
    if (w2 < w1) ks = 2;
  }
  const int64_t resident = slots4 / ks > 0 ? slots4 / ks : 1;
  *stages = 4;
  *k_split = ks;
  *ctas = (tiles < resident ? tiles : resident) * ks;
}

// Shapes the block-dot kernel can run: K > 0; plain scales need K % 256 == 0
// (their rows of K/16 bytes are TMA boxes, whose row stride must be a multiple
// of 16 bytes) and a sfb batch stride that keeps 16-byte alignment; batches
// and rows are 32-bit TMA coordinates.
bool blockdot_shape_ok(int64_t M, int64_t K, int64_t L, bool permuted) {
  if (K <= 0 || M < 1 || L < 1 || M > 0x7fffffff || L > 0x7fffffff) return false;
  return permuted || K % 256 == 0;
}

// Dynamic shared memory a block-dot CTA may use (one CTA per SM: the 227 KB
// opt-in limit less the kernel's static barriers).
constexpr size_t kBlockDotSmemBudget = 232448 - 1024;

// Block-dot schedule: one CTA per SM (no more than the row units), and the
// deepest ring of K-stage slots that fits.
void blockdot_rule(int64_t M, int64_t K, int64_t L, bool permuted, int num_sms, int* stages,
                   int64_t* ctas) {
  const int64_t ur = blockdot_unit_rows(permuted);
  const int64_t units = L * ((M + ur - 1) / ur);
  int64_t n = num_sms;
  if (units < n) n = units;
  if (n < 1) n = 1;
  *ctas = n;
  *stages = blockdot_max_stages(permuted, blockdot_column_blocks(K),
                                blockdot_slot_rows(M, L, permuted, n), kBlockDotSmemBudget);
}

// The rule above with the CTAs of the 2- and 4-stage kernels resident on this
// device.
cudaError_t plan_tc(int64_t M, int64_t N, int64_t K, int64_t L, int* stages, int* k_split,
                    int64_t* ctas) {
  int slots = 0;
  int slots4 = 0;
  cudaError_t err = tc_resident_clusters(2, N, 1, &slots);
  if (err == cudaSuccess) err = tc_resident_clusters(4, N, 1, &slots4);
  if (err != cudaSuccess) return err;
  tc_rule(M, N, K, L, slots, slots4, stages, k_split, ctas);
  return cudaSuccess;
}

// Checks of the small-N GEMM arguments shared by both entry points.
nvfp4_status_t validate_gemm(const void* a, const void* b, const void* sfa, const void* sfb,
                             const void* c, int64_t M, int64_t N, int64_t K, int64_t L,
                             const nvfp4_gemv_options_t& o) {
  if (M < 0 || N < 0 || K < 0 || L < 0) return NVFP4_ERR_INVALID_VALUE;
  if (K % 64 != 0 || N > 16) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (K > kMaxK || M > kMaxM) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (M != 0 && L > kMaxRows / M) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (L * ((M + 127) / 128) > 0x7fffffff) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (o.b_batch_stride < 0 || o.sfb_batch_stride < 0) return NVFP4_ERR_INVALID_VALUE;
  if (!activation_ok(o.activation)) return NVFP4_ERR_INVALID_VALUE;
  if (o.b_batch_stride != 0 && o.b_batch_stride < N * (K / 2)) return NVFP4_ERR_INVALID_VALUE;
  if (o.sfb_batch_stride != 0 && o.sfb_batch_stride < (K / 64) * 512) return NVFP4_ERR_INVALID_VALUE;
  if (o.b_batch_stride % 16 != 0 || o.sfb_batch_stride % 16 != 0) return NVFP4_ERR_MISALIGNED;
  if (M == 0 || N == 0 || L == 0) return NVFP4_OK;
  if (c == nullptr) return NVFP4_ERR_INVALID_VALUE;
  if (K > 0 && (a == nullptr || b == nullptr || sfa == nullptr || sfb == nullptr))
    return NVFP4_ERR_INVALID_VALUE;
  if (!aligned(c, 2) || (o.bias != nullptr && !aligned(o.bias, 2))) return NVFP4_ERR_MISALIGNED;
  if (K > 0 && (!aligned(a, 16) || !aligned(b, 16) || !aligned(sfa, 32) || !aligned(sfb, 32)))
    return NVFP4_ERR_MISALIGNED;
  return NVFP4_OK;
}

nvfp4_status_t run_gemm_tc(const void* a, const void* b, const void* sfa, const void* sfb,
                           void* c, int64_t M, int64_t N, int64_t K, int64_t L, int stages,
                           int ks, int64_t ctas, const nvfp4_gemv_options_t& opt,
                           cudaStream_t stream) {
  GemvPlan plan;
  plan.kernel = kKernelTensor;
  plan.lanes_per_row = stages;
  plan.k_split = ks;
  plan.groups = 1;
  plan.ctas = ctas;
  plan.steps = 1;
  GemvParams p = make_params(a, b, sfa, sfb, c, M, K, L, true, plan, opt);
  if (opt.b_batch_stride == 0) p.b_stride = N * (K / 2);
  const cudaError_t err = launch_gemv_tc(p, N, L, K / 2, stages, ks, ctas, stream);
  if (err != cudaSuccess) return cuda_failure(err);
  return NVFP4_OK;
}

}  // namespace

int rows_per_pass(const GemvPlan& plan) {
  if (plan.kernel == kKernelTensor || plan.kernel == kKernelBlockDot) return 128;  // a tile of A rows
  if (plan.kernel == kKernelBlockwise) return kBlockwiseRows * kGemvWarps;
  return plan.kernel == kKernelAsync ? kAsyncItems * (32 / plan.lanes_per_row) * plan.groups
                                     : kRowsPerPass;
}

namespace {

// Rows of the longest row-lane range: CTA ranges differ by at most one unit
// (a row, or an aligned group of rows for permuted scales) and a CTA's range
// is cut evenly among its 8/k_split row lanes.
int64_t max_rows_per_row_lane(int64_t M, int64_t L, bool permuted, int lanes_per_row,
                              int k_split, int64_t ctas) {
  const int64_t nr = kAsyncItems * (32 / lanes_per_row);
  const int64_t unit = permuted ? nr : 1;
  const int64_t rows_per_l = permuted ? (M + 127) / 128 * 128 : M;
  const int64_t t = rows_per_l * L / unit;
  const int64_t per_cta = (t + ctas - 1) / ctas;
  const int64_t lanes = kGemvWarps / k_split;
  return (per_cta + lanes - 1) / lanes * unit;
}

// Relative cost of a pipelined schedule.  Dominant term: the average number
// of tasks per warp (one task = one row group at one K step), which charges
// the lanes left idle when K/64 is not a multiple of the row width.  Then:
// passes of more than 4 K steps per warp, charged for sweeping their rows'
// columns over a long window (DRAM locality); the busiest row lane's decoded
// b chunks and row groups (pass-end work).  The weights were fitted to
// measured sweeps of all 16 schedules on GB300 over the benchmark shapes and
// several other decode-sized shapes (M 512..28672, K 1024..16384, L 1..16,
// both scale layouts); ties go to the wider row, then the smaller split.
double async_cost(int64_t M, int64_t L, bool permuted, int64_t kchunks, int lpr, int ks,
                  int64_t ctas) {
  const int64_t nr = kAsyncItems * (32 / lpr);
  const int64_t steps = (kchunks + lpr - 1) / lpr;
  const int64_t steps_w = (steps + ks - 1) / ks;
  const int64_t rows_per_l = permuted ? (M + 127) / 128 * 128 : M;
  const double avg_rows = (double)(rows_per_l * L) / (double)(ctas * (kGemvWarps / ks));
  const double avg_tasks = avg_rows / (double)nr * (double)steps_w;
  const int64_t rows = max_rows_per_row_lane(M, L, permuted, lpr, ks, ctas);
  const int64_t ngroups = (rows + nr - 1) / nr;
  const int64_t g = ngroups <= 1 ? 1 : ngroups <= 2 ? 2 : ngroups <= 4 ? 4 : 2;
  const int64_t passes = (ngroups + g - 1) / g;
  const int64_t b_chunks = steps_w > 1 ? passes * steps_w : 1;
  const double long_pass = (double)(ngroups * steps_w * (steps_w > 4 ? steps_w - 4 : 0));
  return 1000.0 * avg_tasks + 4.8 * (double)b_chunks + 5.6 * (double)ngroups + 32.8 * long_pass;
}

}  // namespace

int async_groups(int64_t M, int64_t L, bool permuted, int lanes_per_row, int k_split,
                 int64_t ctas) {
  const int64_t nr = kAsyncItems * (32 / lanes_per_row);
  const int64_t rows = max_rows_per_row_lane(M, L, permuted, lanes_per_row, k_split, ctas);
  const int64_t g = (rows + nr - 1) / nr;
  // a range of more than 4 groups takes several passes anyway; there the
  // 2-group kernel (fewer live accumulators) is as fast or faster
  return g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 2;
}

// The schedule (see gemv_kernel.cuh and gemv_async.cuh for what each knob
// means):
//  * kernel: the pipelined (cp.async) kernel for every K > 0; the direct
//    kernel writes the zeros of K == 0;
//  * tiny problems with plain scales (up to 512 KB of A): the direct kernel,
//    rows narrow enough for at most 4 K steps, those steps split over warps,
//    one CTA per 8 KB of A (measured, see above);
//  * ctas: one wave of resident CTAs (SMs x occupancy), fewer for tiny
//    problems (at least 2 rows per CTA: short, long-K problems still spread
//    their K splits over many SMs), and at most 64 for the pipelined kernel
//    on plain scales up to 2 MB of A;
//  * pipelined kernel: (lanes_per_row, k_split) minimising the cost model
//    above over 32/16/8/4 lanes (16/8/4 for permuted scales) and splits
//    1..8 no larger than the chunk steps (ties go to the wider row, then the
//    smaller split), with the row groups per pass that cover the longest
//    row-lane range (at most 4, beyond that several passes);
//  * direct kernel: the width among 32/16/8/4 lanes that leaves the fewest
//    idle lane slots over K/64 chunks, and the smallest split that still
//    gives each row lane of 8/k_split warps a full pass of rows, capped by
//    the number of chunk steps.
bool plan_gemv(int64_t M, int64_t K, int64_t L, bool permuted, int kernel, int num_sms,
               int ctas_per_sm, GemvPlan* out) {
  if (M < 0 || K < 0 || L < 0 || num_sms < 1 || ctas_per_sm < 1 || out == nullptr) return false;
  if (kernel < -1 || kernel > kKernelBlockwise) return false;
  const int64_t kchunks = K / 64;
  // K % 64 != 0 (K a multiple of 16): the blockwise kernel alone runs it
  if (kernel == -1 && K % 64 != 0) kernel = kKernelBlockwise;
  if (kernel == kKernelBlockwise) {
    const int64_t groups = L * ((M + kBlockwiseRows - 1) / kBlockwiseRows);
    const int64_t warps = (int64_t)num_sms * ctas_per_sm * kGemvWarps;
    out->kernel = kKernelBlockwise;
    out->lanes_per_row = 32;
    out->k_split = 1;
    out->groups = 1;
    out->ctas = std::max<int64_t>(1, (std::min(groups, warps) + kGemvWarps - 1) / kGemvWarps);
    out->steps = (K / 16 + 31) / 32;
    return true;
  }
  if (K % 64 != 0) return false;
  // bytes of A, saturated (M*L < 2^40 and K/2 <= 2^29 can pass 2^63)
  const int64_t a_bytes =
      K / 2 > 0 && M * L > INT64_MAX / (K / 2) ? INT64_MAX : M * L * (K / 2);
  // Tiny problems with plain scales (measured on GB300 over 16 KB .. 2 MB of
  // A): the launch and the first DRAM access dominate, and fewer, fuller CTAs
  // finish first.  Up to 512 KB the direct kernel does best with rows narrow
  // enough for at most 4 K steps, those steps split over warps and one CTA
  // per 8 KB of A (e.g. M128_K256_L1: 1.50 against 1.73 us); up to 2 MB the
  // pipelined kernel does best on at most 64 CTAs.  (Pre-permuted scales keep
  // the general schedule: the same rule was slower for some of them.)
  const bool small_plain = !permuted && kchunks > 0 && a_bytes <= (int64_t(2) << 20);
  const bool tiny = kernel == -1 && small_plain && a_bytes <= (int64_t(512) << 10);
  // The tensor-core kernel where it was measured faster than the pipelined
  // kernel (GB300, cold L2):
  //  * large streams, either scale layout (plain: K % 256 == 0): from 512 MB
  //    of A with K <= 8192, by 2.6-9.4% plain and 1-11% pre-permuted on 7
  //    shapes of 0.6-1.2 GB (M16384_K8192_L16 plain 176.6 against 182.0 us,
  //    M65536_K1024_L16 88.9 against 98.2); with plain scales slower at
  //    K >= 12288 and below 500 MB;
  //  * one wave, pre-permuted scales: tiles (L*ceil(M/128)) filling 80-100% of
  //    the resident 4-stage CTAs, one CTA per tile, with K >= 6144: faster on
  //    13 of 14 such shapes by 0.4-21% (M4096_K7168_L8 24.6 against 25.1 us),
  //    1% slower at K = 4096; with 74% filled (224 tiles) 7% slower.  (Plain
  //    scales there: 25.2 against 23.3 us.)
  //  * more than one wave of tiles with pre-permuted scales, from 128 MB of
  //    A, any K: faster on 15 of 16 such shapes of 128 MB-1 GB with K from
  //    1024 to 16384, by 0.8-8.8% (M32768_K2048_L8 46.5 against 51.0 us,
  //    M8192_K6144_L8 37.7 against 40.3, M16384_K16384_L8 179.9 against
  //    185.3), 0.4% slower on M8192_K4096_L8.  Below 128 MB it depends on the
  //    shape (4 of 10 faster, 6 up to 8% slower); with plain scales, whose
  //    atom layout costs the MMA warp a step per stage, 5 of 6 such shapes
  //    were slower.
  // Elsewhere (a K split, a partial wave, short K) the pipelined kernel is
  // faster.  The block-dot kernel is explicit only (level at best).
  const int64_t tc_tiles = L * ((M + 127) / 128);
  const int64_t slots4 = (int64_t)num_sms * 2;  // 4-stage tensor-core CTAs resident
  const bool tensor_large =
      K <= 8192 && a_bytes >= (int64_t(512) << 20) && (permuted || K % 256 == 0);
  const bool tensor_wave =
      permuted && K >= 6144 && tc_tiles <= slots4 && 5 * tc_tiles >= 4 * slots4;
  const bool tensor_waves =
      permuted && tc_tiles > slots4 && a_bytes >= (int64_t(128) << 20);
  const bool tensor_pays =
      M >= 1024 && tc_tiles <= 0x7fffffff && (tensor_large || tensor_wave || tensor_waves);
  if (kernel == -1)
    kernel = tiny || kchunks == 0 ? kKernelDirect : tensor_pays ? kKernelTensor : kKernelAsync;
  if (kernel == kKernelBlockDot) {
    if (!blockdot_shape_ok(M, K, L, permuted)) return false;
    int stages = 2;
    int64_t ctas = 1;
    blockdot_rule(M, K, L, permuted, num_sms, &stages, &ctas);
    out->kernel = kKernelBlockDot;
    out->lanes_per_row = stages;
    out->k_split = 1;
    out->groups = 1;
    out->ctas = ctas;
    const int64_t stage_chunks = 4 * blockdot_column_blocks(K);  // 64-element chunks per stage
    out->steps = (kchunks + stage_chunks - 1) / stage_chunks;
    return true;
  }
  if (kernel == kKernelTensor) {
    // plain scales: 16-byte scale rows per 256-element stage (K % 256 == 0)
    if (kchunks == 0 || (!permuted && K % 256 != 0)) return false;
    // host-only estimate: 4 CTAs of the 2-stage kernel or 2 of the 4-stage
    // kernel resident per SM (the launch recomputes the schedule from this
    // device's limits)
    int stages = 2, ks = 1;
    int64_t ctas = 1;
    tc_rule(M, 1, K, L, (int64_t)num_sms * 4, (int64_t)num_sms * 2, &stages, &ks, &ctas);
    out->kernel = kKernelTensor;
    out->lanes_per_row = stages;
    out->k_split = ks;
    out->groups = 1;
    out->ctas = ctas;
    out->steps = (K + 255) / 256;
    return true;
  }
  if (kernel == kKernelAsync && kchunks == 0) return false;
  const int64_t rows = M * L;
  int64_t ctas = (int64_t)num_sms * ctas_per_sm;
  const int64_t by_rows = (rows + 1) / 2;
  if (by_rows < ctas) ctas = by_rows;
  if (tiny && a_bytes / 8192 < ctas) ctas = a_bytes / 8192;
  if (kernel == kKernelAsync && small_plain && ctas > 64) ctas = 64;
  if (ctas < 1) ctas = 1;
  int lpr = 32, ks = 1;
  if (tiny) {
    lpr = 32;
    for (int cand : {4, 8, 16, 32}) {
      if ((kchunks + cand - 1) / cand <= 4) {
        lpr = cand;
        break;
      }
    }
    const int64_t steps = (kchunks + lpr - 1) / lpr;
    while (2 * ks <= 4 && 2 * ks <= steps) ks *= 2;
    out->kernel = kKernelDirect;
    out->lanes_per_row = lpr;
    out->k_split = ks;
    out->groups = 1;
    out->ctas = ctas;
    out->steps = steps;
    return true;
  }
  // permuted scales with plenty of rows: 4 lanes per row, whose 32-row
  // groups read whole 128-byte lines of the scale atoms, and the even K split
  // that leaves about 2 K steps per warp (measured: 4-16% faster than the
  // model's choice on the large permuted shapes, slower when rows are scarce)
  const int64_t steps4 = (kchunks + 3) / 4;
  int ks4 = 1;
  while (ks4 < kGemvWarps && (steps4 + ks4 - 1) / ks4 > 2) ks4 *= 2;
  const bool narrow = kernel == kKernelAsync && permuted && steps4 % ks4 == 0 &&
                      steps4 / ks4 <= 4 &&
                      (M + 127) / 128 * 128 * L >= 24 * ctas * (kGemvWarps / ks4);
  if (narrow) {
    lpr = 4;
    ks = ks4;
  } else if (kernel == kKernelAsync) {
    double best = -1.0;
    for (int cand : {32, 16, 8, 4}) {
      // a lane's permuted scale run is 16 bytes: with 32 lanes per row it is
      // half of a 32-byte sector whose other half another task reads
      if (permuted && cand == 32) continue;
      const int64_t steps = (kchunks + cand - 1) / cand;
      for (int k = 1; k <= kGemvWarps && k <= steps; k *= 2) {
        const double c = async_cost(M, L, permuted, kchunks, cand, k, ctas);
        if (best < 0.0 || c < best - 1e-9) {
          best = c;
          lpr = cand;
          ks = k;
        }
      }
    }
  } else {
    int64_t best_slots = -1;
    for (int cand : {32, 16, 8, 4}) {
      const int64_t slots = (kchunks + cand - 1) / cand * cand;
      if (best_slots < 0 || slots < best_slots) {
        best_slots = slots;
        lpr = cand;
      }
    }
    const int64_t steps = (kchunks + lpr - 1) / lpr;
    while (ks < kGemvWarps && 2 * ks <= steps && rows * ks < ctas * kGemvWarps * kRowsPerPass)
      ks *= 2;
  }
  out->kernel = kernel;
  out->lanes_per_row = lpr;
  out->k_split = ks;
  out->groups = kernel == kKernelAsync ? async_groups(M, L, permuted, lpr, ks, ctas) : 1;
  out->ctas = ctas;
  out->steps = (kchunks + lpr - 1) / lpr;
  return true;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

nvfp4_status_t nvfp4_gemv(const void* a, const void* b, const void* sfa, const void* sfb,
                          void* c, int64_t M, int64_t K, int64_t L, int sf_layout,
                          struct CUstream_st* stream) {
  return nvfp4_gemv_ex(a, b, sfa, sfb, c, M, K, L, sf_layout, nullptr, stream);
}

nvfp4_status_t nvfp4_gemv_ex(const void* a, const void* b, const void* sfa, const void* sfb,
                             void* c, int64_t M, int64_t K, int64_t L, int sf_layout,
                             const nvfp4_gemv_options_t* options, struct CUstream_st* stream) {
  nvfp4_status_t st = validate_gemv_shape(M, K, L, sf_layout);
  if (st != NVFP4_OK) return st;
  const nvfp4_gemv_options_t& opt = options ? *options : kDefaultOptions;
  st = validate_options(opt, K, sf_layout);
  if (st != NVFP4_OK) return st;
  if (M == 0 || L == 0) return NVFP4_OK;
  st = validate_gemv_pointers(a, b, sfa, sfb, c, K);
  if (st != NVFP4_OK) return st;
  int sms = 0, occ = 0;
  cudaError_t err = device_info(&sms, &occ, nullptr);
  if (err != cudaSuccess) return cuda_failure(err);
  GemvPlan plan;
  const bool permuted = sf_layout == NVFP4_SF_PERMUTED_128x4;
  if (!plan_gemv(M, K, L, permuted, -1, sms, occ, &plan)) return NVFP4_ERR_INVALID_VALUE;
  // the direct kernel loads a with 256-bit loads: a 16-byte aligned a takes
  // the pipelined kernel (K = 0 reads nothing); the tensor-core kernel reads
  // plain sfb rows through a tensor map: a batch stride that is not a
  // multiple of 16 bytes takes the pipelined kernel
  if (((plan.kernel == kKernelDirect && K > 0 && !aligned(a, 32)) ||
       (plan.kernel == kKernelTensor && !permuted && opt.sfb_batch_stride % 16 != 0)) &&
      !plan_gemv(M, K, L, permuted, kKernelAsync, sms, occ, &plan))
    return NVFP4_ERR_INVALID_VALUE;
  return run_gemv(a, b, sfa, sfb, c, M, K, L, sf_layout, plan, opt, (cudaStream_t)stream);
}

nvfp4_status_t nvfp4_gemv_explicit(const void* a, const void* b, const void* sfa,
                                   const void* sfb, void* c, int64_t M, int64_t K, int64_t L,
                                   int sf_layout, int kernel, int lanes_per_row, int k_split,
                                   int64_t ctas, struct CUstream_st* stream) {
  nvfp4_status_t st = validate_gemv_shape(M, K, L, sf_layout);
  if (st != NVFP4_OK) return st;
  if (kernel != kKernelDirect && kernel != kKernelAsync && kernel != kKernelTensor &&
      kernel != kKernelBlockDot && kernel != kKernelBlockwise)
    return NVFP4_ERR_INVALID_VALUE;
  const bool permuted = sf_layout == NVFP4_SF_PERMUTED_128x4;
  if (kernel == kKernelBlockwise) {
    // 32 lanes per row group, k_split 1
    if (lanes_per_row != 32 || k_split != 1 || ctas < 1 || ctas > 0x7fffffff)
      return NVFP4_ERR_INVALID_VALUE;
    if (M == 0 || L == 0) return NVFP4_OK;
    st = validate_gemv_pointers(a, b, sfa, sfb, c, K);
    if (st != NVFP4_OK) return st;
    GemvPlan plan;
    plan.kernel = kKernelBlockwise;
    plan.lanes_per_row = 32;
    plan.k_split = 1;
    plan.groups = 1;
    plan.ctas = ctas;
    plan.steps = (K / 16 + 31) / 32;
    return run_gemv(a, b, sfa, sfb, c, M, K, L, sf_layout, plan, kDefaultOptions,
                    (cudaStream_t)stream);
  }
  // the other kernels move 64-element chunks
  if (K % 64 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (kernel == kKernelBlockDot) {
    // lanes_per_row = ring slots (0: the most that fit), k_split 1
    if (k_split != 1 || ctas < 1 || ctas > 0x7fffffff || lanes_per_row < 0 ||
        lanes_per_row == 1 || lanes_per_row > kBlockDotMaxStages)
      return NVFP4_ERR_INVALID_VALUE;
    if (!blockdot_shape_ok(M < 1 ? 1 : M, K, L < 1 ? 1 : L, permuted)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || L == 0) return NVFP4_OK;
    st = validate_gemv_pointers(a, b, sfa, sfb, c, K);
    if (st != NVFP4_OK) return st;
    const int slot_rows = blockdot_slot_rows(M, L, permuted, ctas);
    const int most = blockdot_max_stages(permuted, blockdot_column_blocks(K), slot_rows,
                                         kBlockDotSmemBudget);
    if (lanes_per_row > most) return NVFP4_ERR_INVALID_VALUE;
    GemvPlan plan;
    plan.kernel = kKernelBlockDot;
    plan.lanes_per_row = lanes_per_row == 0 ? most : lanes_per_row;
    plan.k_split = 1;
    plan.groups = 1;
    plan.ctas = ctas;
    plan.steps = (K + 255) / 256;
    return run_gemv(a, b, sfa, sfb, c, M, K, L, sf_layout, plan, kDefaultOptions,
                    (cudaStream_t)stream);
  }
  // lanes per row; for the tensor-core kernel, pipeline stages per CTA
  if (kernel == kKernelTensor ? (lanes_per_row != 2 && lanes_per_row != 4)
                              : (lanes_per_row != 4 && lanes_per_row != 8 &&
                                 lanes_per_row != 16 && lanes_per_row != 32))
    return NVFP4_ERR_INVALID_VALUE;
  if (k_split != 1 && k_split != 2 && k_split != 4 && k_split != 8) return NVFP4_ERR_INVALID_VALUE;
  if (ctas < 1 || ctas > 0x7fffffff) return NVFP4_ERR_INVALID_VALUE;
  const int64_t steps = (K / 64 + lanes_per_row - 1) / lanes_per_row;
  // the pipelined kernel needs a K range and a step for every K-split warp
  if (kernel == kKernelAsync && (K == 0 || k_split > steps)) return NVFP4_ERR_INVALID_VALUE;
  // the tensor-core kernel: clusters of k_split CTAs that each take at least
  // one 256-element K stage of every 128-row tile; plain scales with
  // K % 256 == 0 only
  if (kernel == kKernelTensor) {
    if (K == 0) return NVFP4_ERR_INVALID_VALUE;
    if (!permuted && K % 256 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (k_split > (K + 255) / 256 || ctas % k_split != 0) return NVFP4_ERR_INVALID_VALUE;
    if (L * ((M + 127) / 128) > 0x7fffffff) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  }
  if (M == 0 || L == 0) return NVFP4_OK;
  st = validate_gemv_pointers(a, b, sfa, sfb, c, K);
  if (st != NVFP4_OK) return st;
  if (kernel == kKernelDirect && K > 0 && !aligned(a, 32)) return NVFP4_ERR_MISALIGNED;
  GemvPlan plan;
  plan.kernel = kernel;
  plan.lanes_per_row = lanes_per_row;
  plan.k_split = k_split;
  plan.ctas = ctas;
  plan.steps = steps;
  plan.groups = kernel == kKernelAsync
                    ? async_groups(M, L, sf_layout == NVFP4_SF_PERMUTED_128x4, lanes_per_row,
                                   k_split, ctas)
                    : 1;
  return run_gemv(a, b, sfa, sfb, c, M, K, L, sf_layout, plan, kDefaultOptions,
                  (cudaStream_t)stream);
}

nvfp4_status_t nvfp4_repack_scales(const void* src, void* dst, int64_t rows, int64_t K,
                                   int64_t L, struct CUstream_st* stream) {
  if (rows < 0 || K < 0 || L < 0) return NVFP4_ERR_INVALID_VALUE;
  if (K % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (K > kMaxK || rows > kMaxM) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (rows != 0 && L > kMaxRows / rows) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0 || K == 0 || L == 0) return NVFP4_OK;
  if (src == nullptr || dst == nullptr) return NVFP4_ERR_INVALID_VALUE;
  if (!aligned(src, 4) || !aligned(dst, 16)) return NVFP4_ERR_MISALIGNED;
  int sms = 0, occ = 0;
  cudaError_t err = device_info(&sms, nullptr, &occ);
  if (err != cudaSuccess) return cuda_failure(err);
  err = launch_repack(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), rows, K, L,
                      (int64_t)sms * occ, (cudaStream_t)stream);
  if (err != cudaSuccess) return cuda_failure(err);
  return NVFP4_OK;
}

size_t nvfp4_permuted_scale_bytes(int64_t rows, int64_t K, int64_t L) {
  if (rows < 0 || K < 0 || L < 0 || K % 16 != 0) return 0;
  return (size_t)(L * ((rows + 127) / 128) * ((K + 63) / 64) * 512);
}

const char* nvfp4_status_string(int status) {
  switch (status) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_ERR_INVALID_VALUE: return "NVFP4_ERR_INVALID_VALUE";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "NVFP4_ERR_UNSUPPORTED_SHAPE";
    case NVFP4_ERR_MISALIGNED: return "NVFP4_ERR_MISALIGNED";
    case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
    default: return "NVFP4_ERR_UNKNOWN";
  }
}

nvfp4_status_t nvfp4_gemm_small_n(const void* a, const void* b, const void* sfa, const void* sfb,
                                  void* c, int64_t M, int64_t N, int64_t K, int64_t L,
                                  const nvfp4_gemv_options_t* options, struct CUstream_st* stream) {
  const nvfp4_gemv_options_t& opt = options ? *options : kDefaultOptions;
  nvfp4_status_t st = validate_gemm(a, b, sfa, sfb, c, M, N, K, L, opt);
  if (st != NVFP4_OK || M == 0 || N == 0 || L == 0) return st;
  if (N == 1)
    return nvfp4_gemv_ex(a, b, sfa, sfb, c, M, K, L, NVFP4_SF_PERMUTED_128x4, &opt, stream);
  int stages = 2, ks = 1;
  int64_t ctas = 1;
  const cudaError_t err = plan_tc(M, N, K, L, &stages, &ks, &ctas);
  if (err != cudaSuccess) return cuda_failure(err);
  return run_gemm_tc(a, b, sfa, sfb, c, M, N, K, L, stages, ks, ctas, opt, (cudaStream_t)stream);
}

nvfp4_status_t nvfp4_gemm_small_n_explicit(const void* a, const void* b, const void* sfa,
                                           const void* sfb, void* c, int64_t M, int64_t N,
                                           int64_t K, int64_t L, int stages, int k_split,
                                           int64_t ctas, struct CUstream_st* stream) {
  nvfp4_status_t st = validate_gemm(a, b, sfa, sfb, c, M, N, K, L, kDefaultOptions);
  if (st != NVFP4_OK) return st;
  if (stages != 2 && stages != 4) return NVFP4_ERR_INVALID_VALUE;
  if (k_split != 1 && k_split != 2 && k_split != 4 && k_split != 8) return NVFP4_ERR_INVALID_VALUE;
  if (k_split > 1 && k_split > (K + 255) / 256) return NVFP4_ERR_INVALID_VALUE;
  if (ctas < 1 || ctas > 0x7fffffff || ctas % k_split != 0) return NVFP4_ERR_INVALID_VALUE;
  if (M == 0 || N == 0 || L == 0) return NVFP4_OK;
  return run_gemm_tc(a, b, sfa, sfb, c, M, N, K, L, stages, k_split, ctas, kDefaultOptions,
                     (cudaStream_t)stream);
}

nvfp4_status_t nvfp4_gemm_small_n_plan(int64_t M, int64_t N, int64_t K, int64_t L,
                                       int* stages, int* k_split, int64_t* ctas,
                                       int* resident_ctas) {
  if (stages == nullptr || k_split == nullptr || ctas == nullptr) return NVFP4_ERR_INVALID_VALUE;
  nvfp4_status_t st = validate_gemm(nullptr, nullptr, nullptr, nullptr, nullptr, 0, N, K, L,
                                    kDefaultOptions);
  if (st != NVFP4_OK) return st;
  if (M < 0 || M > kMaxM || (M != 0 && L > kMaxRows / M)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (L * ((M + 127) / 128) > 0x7fffffff) return NVFP4_ERR_UNSUPPORTED_SHAPE;  // 128-row tiles
  cudaError_t err = plan_tc(M, N < 1 ? 1 : N, K, L, stages, k_split, ctas);
  if (err == cudaSuccess && resident_ctas != nullptr)
    err = tc_resident_clusters(*stages, N < 1 ? 1 : N, 1, resident_ctas);
  if (err != cudaSuccess) return cuda_failure(err);
  return NVFP4_OK;
}

int nvfp4_last_cuda_error(void) { return g_last_cuda_error; }

int nvfp4_tensor_wait_timeouts(int reset) {
  int v = 0, w = 0;
  cudaError_t err = tc_wait_timeouts(reset, &v);
  if (err == cudaSuccess) err = blockdot_wait_timeouts(reset, &w);
  if (err != cudaSuccess) {
    g_last_cuda_error = (int)err;
    (void)cudaGetLastError();
    return -1;
  }
  return v + w;
}

nvfp4_status_t nvfp4_selftest_bounded_wait(int* completed, int* gave_up, int* timeouts,
                                           int64_t* waited_ns, struct CUstream_st* stream) {
  if (completed == nullptr || gave_up == nullptr || timeouts == nullptr || waited_ns == nullptr)
    return NVFP4_ERR_INVALID_VALUE;
  WaitSelftest r = {};
  const cudaError_t err = run_wait_selftest((cudaStream_t)stream, &r);
  if (err != cudaSuccess) return cuda_failure(err);
  *completed = r.completed;
  *gave_up = r.gave_up;
  *timeouts = r.timeouts;
  *waited_ns = r.waited_ns;
  return NVFP4_OK;
}

nvfp4_status_t nvfp4_gemv_plan(int64_t M, int64_t K, int64_t L, int sf_layout, int kernel,
                               int num_sms, int ctas_per_sm, nvfp4_gemv_plan_t* out) {
  if (out == nullptr || num_sms < 1 || ctas_per_sm < 0) return NVFP4_ERR_INVALID_VALUE;
  nvfp4_status_t st = validate_gemv_shape(M, K, L, sf_layout);
  if (st != NVFP4_OK) return st;
  GemvPlan plan;
  if (kernel < -1 || kernel > kKernelBlockwise) return NVFP4_ERR_INVALID_VALUE;
  if (!plan_gemv(M, K, L, sf_layout == NVFP4_SF_PERMUTED_128x4, kernel, num_sms,
                 ctas_per_sm > 0 ? ctas_per_sm : kGemvMinCtasPerSm, &plan))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  out->kernel = plan.kernel;
  out->lanes_per_row = plan.lanes_per_row;
  out->k_split = plan.k_split;
  out->rows_per_pass = rows_per_pass(plan);
  out->threads_per_cta = plan.kernel == kKernelTensor     ? kTcThreadsPerCta
                         : plan.kernel == kKernelBlockDot ? kBlockDotThreads
                                                          : kGemvThreads;
  out->ctas = plan.ctas;
  out->steps = plan.steps;
  return NVFP4_OK;
}

}  // extern "C"

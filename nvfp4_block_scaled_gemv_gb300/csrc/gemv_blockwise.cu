// NVFP4 block-scaled batched GEMV for any K % 16 == 0 (CUDA cores, sm_103a).
//
// The other kernels move 64-element (32-byte) K chunks, one 128x4 scale-atom
// column at a time, and need K % 64 == 0.  Here a lane takes whole 16-element
// scale blocks: with K % 16 == 0 a row of A is K/2 bytes, a multiple of 8, so
// every block is one aligned 8-byte load wherever K ends.  The arithmetic per
// block is the other kernels' (exact half2 block dot, exact scaling by sfa,
// one fp32 fma with sfb; gemv_kernel.cuh).
//
// Work split: the rows of every batch are cut into groups of kBlockwiseRows
// rows (plain scales: consecutive rows, the last group of a batch may be
// shorter; pre-permuted scales: rows m, m + 32, m + 64, m + 96 of a 128-row
// atom block, whose scales for 4 consecutive blocks are one 16-byte run of
// the atom, rows past M skipped); warp w of the grid takes groups w,
// w + warps, ...  In a group, lane j takes blocks j, j + 32, j + 64, ...,
// kBwUnroll of them per step: it first issues every load of the step (the
// blocks of b, their sfb bytes, and each row's A blocks and sfa bytes) and
// only then decodes and accumulates, so each warp keeps kBwUnroll x
// kBlockwiseRows x 256 bytes of A in flight.  Each lane accumulates its rows'
// blocks in K order; a shuffle butterfly then sums the 32 lanes of each row.
// The summation order depends only on K, so results are reproducible and the
// same for both scale layouts and any grid.
//
// Pre-permuted scales for K % 64 != 0: the last 128x4 atom column holds the
// K/16 % 4 remaining blocks and 0x00 padding (nvfp4_repack_scales writes it
// so); byte (m, kb) of batch l is at ((l*rest_m + m/128)*rest_k + kb/4)*512
// + (m%32)*16 + ((m/32)%4)*4 + kb%4 with rest_k = ceil(K/64).
#include "gemv_kernel.cuh"

namespace nvfp4 {

namespace {

constexpr int kBwUnroll = 4;  // blocks per lane and step

__device__ __forceinline__ uint2 ld_stream_64(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_cached_64(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_byte(const uint8_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_cached_128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <bool PERM>
__global__ void __launch_bounds__(kGemvThreads, 2)
    nvfp4_gemv_blockwise_kernel(const GemvParams p) {
  constexpr int R = kBlockwiseRows, U = kBwUnroll;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * kGemvWarps;
  static_assert(R == 4, "a permuted group is the 4 rows of one 16-byte atom run");
  const int64_t groups_per_l = PERM ? (int64_t)p.rest_m * 32 : (p.M + R - 1) / R;
  const int64_t groups = groups_per_l * (p.rows_total / p.rows_per_l);

  pdl_launch_dependents();
  pdl_wait();

  for (int64_t g = (int64_t)blockIdx.x * kGemvWarps + (threadIdx.x >> 5); g < groups; g += warps) {
    const int64_t l = g / groups_per_l;
    const int64_t gi = g - l * groups_per_l;
    // row r of the group is m0 + r*dm; live[r]: the row is below M
    const int64_t m0 = PERM ? (gi >> 5) * 128 + (gi & 31) : gi * R;
    const int64_t dm = PERM ? 32 : 1;
    bool live[R];
#pragma unroll
    for (int r = 0; r < R; ++r) live[r] = m0 + r * dm < p.M;
    if (!live[0]) continue;  // an all-padding group of the last atom block
    const uint8_t* brow = p.b + l * p.b_stride;
    const uint8_t* sbrow = p.sfb + l * p.sfb_stride;
    // the group's rows (dead rows repeat row 0; they are never loaded)
    const uint8_t* arow[R];
    const uint8_t* srow[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int64_t m = live[r] ? m0 + r * dm : m0;
      arow[r] = p.a + (l * p.M + m) * p.half_k;
      srow[r] = p.sfa + (PERM ? ((l * p.rest_m + (m >> 7)) * p.rest_k) * 512 + (m & 31) * 16
                              : (l * p.M + m) * p.blocks);
    }
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;
    for (int64_t j0 = lane; j0 < p.blocks; j0 += 32 * U) {
      // every load of the step first (blocks past K/16 and rows past the
      // group's nr are not loaded)
      uint2 bw[U], aw[U][R];
      uint32_t sbc[U], sac[U][R];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j = j0 + 32 * u;
        const bool in = j < p.blocks;
        // scale byte of block j: at j (plain) or (j/4)*512 + j%4 (permuted,
        // byte 4r of the group's 16-byte run for row r)
        const int64_t sj = PERM ? (j >> 2) * 512 + (j & 3) : j;
        bw[u] = in ? ld_cached_64(brow + 8 * j) : make_uint2(0u, 0u);
        sbc[u] = in ? ld_byte(sbrow + sj) : 0u;
        if constexpr (PERM) {
          const uint4 run = in ? ld_cached_128(srow[0] + (j >> 2) * 512) : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t words[4] = {run.x, run.y, run.z, run.w};
#pragma unroll
          for (int r = 0; r < R; ++r) sac[u][r] = (words[r] >> (8 * (j & 3))) & 0xffu;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const bool ld = in && live[r];
          aw[u][r] = ld ? ld_stream_64(arow[r] + 8 * j) : make_uint2(0u, 0u);
          if constexpr (!PERM) sac[u][r] = ld ? ld_byte(srow[r] + sj) : 0u;
        }
      }
      // then the arithmetic, block by block in K order
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (j0 + 32 * u < p.blocks) {
          uint32_t bh[8];
          {
            uint32_t lo[4], hi[4];
            e2m1x8_to_f16x2x4(bw[u].x, lo);
            e2m1x8_to_f16x2x4(bw[u].y, hi);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              bh[t] = lo[t];
              bh[4 + t] = hi[t];
            }
          }
          const float sb = f16_lo_to_f32(e4m3x2_to_f16x2(sbc[u]));
#pragma unroll
          for (int r = 0; r < R; ++r)
            if (live[r])
              acc[r] = block_accumulate<false>(block_dot(aw[u][r].x, aw[u][r].y, bh),
                                               e4m3x2_to_f16x2(sac[u][r]), sb, acc[r]);
        }
      }
    }
    // lanes 8r..8r+7 end with row r's sum
    const float v = lane_reduce<R, 16>(acc, lane);
    const int r = lane >> 3;
    if ((lane & 7) == 0 && m0 + r * dm < p.M) {
      const int64_t idx = l * p.M + m0 + r * dm;
      p.c[idx] = finish_output(p, v, idx);
    }
  }
}

}  // namespace

cudaError_t launch_gemv_blockwise(const GemvParams& p, bool permuted, int64_t ctas,
                                  cudaStream_t stream) {
  void (*kern)(GemvParams) =
      permuted ? nvfp4_gemv_blockwise_kernel<true> : nvfp4_gemv_blockwise_kernel<false>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace nvfp4

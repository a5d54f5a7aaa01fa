// NVFP4 block-scaled batched GEMV for any K % 16 == 0 (CUDA cores, sm_103a).
//
// The other kernels move 64-element (32-byte) K chunks, one 128x4 scale-atom
// column at a time, and need K % 64 == 0.  Here a lane takes whole 16-element
// scale blocks: with K % 16 == 0 a row of A is K/2 bytes, a multiple of 8, so
// every block is one aligned 8-byte load wherever K ends.  The arithmetic per
// block is the other kernels' (exact half2 block dot, exact scaling by sfa,
// one fp32 fma with sfb; gemv_kernel.cuh).
//
// Work split: the rows of every batch are cut into groups of 4 (the last group
// of a batch may be shorter); warp w of the grid takes groups w, w + warps,
// ...  In a group, lane j takes blocks j, j + 32, ..., decodes b's block once
// for the 4 rows, and accumulates each row's blocks in K order; a shuffle
// butterfly then sums the 32 lanes of each row.  The summation order depends
// only on K, so results are reproducible and the same for both scale layouts.
//
// Pre-permuted scales for K % 64 != 0: the last 128x4 atom column holds the
// K/16 % 4 remaining blocks and 0x00 padding (nvfp4_repack_scales writes it
// so); byte (m, kb) of batch l is at ((l*rest_m + m/128)*rest_k + kb/4)*512
// + (m%32)*16 + ((m/32)%4)*4 + kb%4 with rest_k = ceil(K/64).
#include "gemv_kernel.cuh"

namespace nvfp4 {

namespace {

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

// Byte offset of scale (m, kb) of batch l.
template <bool PERM>
__device__ __forceinline__ int64_t bw_scale_offset(const GemvParams& p, int64_t l, int64_t m,
                                                   int64_t kb) {
  if (!PERM) return (l * p.M + m) * p.blocks + kb;
  return ((l * p.rest_m + (m >> 7)) * p.rest_k + (kb >> 2)) * 512 + (m & 31) * 16 +
         ((m >> 5) & 3) * 4 + (kb & 3);
}

template <bool PERM>
__global__ void __launch_bounds__(kGemvThreads)
    nvfp4_gemv_blockwise_kernel(const GemvParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * kGemvWarps;
  const int64_t groups_per_l = (p.M + kBlockwiseRows - 1) / kBlockwiseRows;
  const int64_t groups = groups_per_l * (p.rows_total / p.rows_per_l);

  pdl_launch_dependents();
  pdl_wait();

  for (int64_t g = (int64_t)blockIdx.x * kGemvWarps + (threadIdx.x >> 5); g < groups; g += warps) {
    const int64_t l = g / groups_per_l;
    const int64_t m0 = (g - l * groups_per_l) * kBlockwiseRows;
    const int nr = p.M - m0 < kBlockwiseRows ? (int)(p.M - m0) : kBlockwiseRows;
    const uint8_t* brow = p.b + l * p.b_stride;
    const uint8_t* sbrow = p.sfb + l * p.sfb_stride;
    float acc[kBlockwiseRows] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t j = lane; j < p.blocks; j += 32) {
      // b's block j, decoded once for the group's rows
      const uint2 bw = ld_cached_64(brow + 8 * j);
      uint32_t bh[8];
      {
        uint32_t lo[4], hi[4];
        e2m1x8_to_f16x2x4(bw.x, lo);
        e2m1x8_to_f16x2x4(bw.y, hi);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          bh[t] = lo[t];
          bh[4 + t] = hi[t];
        }
      }
      const uint32_t sbc = ld_byte(sbrow + (PERM ? (j >> 2) * 512 + (j & 3) : j));
      const float sb = f16_lo_to_f32(e4m3x2_to_f16x2(sbc));
#pragma unroll
      for (int r = 0; r < kBlockwiseRows; ++r) {
        if (r < nr) {
          const int64_t m = m0 + r;
          const uint2 aw = ld_stream_64(p.a + (l * p.M + m) * p.half_k + 8 * j);
          const uint32_t sac = ld_byte(p.sfa + bw_scale_offset<PERM>(p, l, m, j));
          acc[r] = block_accumulate<false>(block_dot(aw.x, aw.y, bh), e4m3x2_to_f16x2(sac), sb,
                                           acc[r]);
        }
      }
    }
    // lanes 8r..8r+7 end with row r's sum
    const float v = lane_reduce<kBlockwiseRows, 16>(acc, lane);
    const int r = lane >> 3;
    if ((lane & 7) == 0 && r < nr) {
      const int64_t idx = l * p.M + m0 + r;
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

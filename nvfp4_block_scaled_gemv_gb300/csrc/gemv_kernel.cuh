// NVFP4 block-scaled batched GEMV kernel (CUDA cores, sm_103a).
//
// Computes c[m,l] = fp16(sum_k E2M1(a)*E4M3(sfa)*E2M1(b)*E4M3(sfb)), the
// per-element product the k-tile loop of `cute_kernel` (kernelbot nvfp4-gemv
// submission 103289) accumulates, regrouped per 16-element scale block:
//   c = sum_blocks (sfa*sfb) * sum_{16} a*b.
//
// Work split (one grid sized to the SMs, no atomics, no scratch memory):
//   * The rows of all batches, L*M of them, are cut into gridDim.x contiguous
//     ranges that differ by at most one row; each CTA takes one range.
//   * A CTA's 8 warps form 8/KS row lanes of KS warps each; a row lane takes a
//     contiguous share of the CTA's rows and walks it in passes of up to 8
//     rows of one batch.  The KS warps of a row lane split each row's K range
//     and add their partial sums through shared memory.
//   * Inside a warp, LPR lanes share a row: lane kc owns the 32-byte A chunks
//     kt = s*LPR + kc (one 128x4 scale-atom column: 64 elements, 4 blocks),
//     so each warp-wide 256-bit load reads LPR*32 contiguous bytes of each of
//     32/LPR rows.
//
// Arithmetic: A and b nibbles are decoded with cvt.rn.f16x2.e2m1x2 and
// multiplied with fma.rn.f16x2; all products are multiples of 1/4 below 36
// in magnitude and each half2 lane sums 8 of them, so every partial sum is
// exact in fp16.  The two halves times sfa go to fp32 exactly (two mixed
// fp16 x fp16 + fp32 fmas), and one fp32 fma adds that times sfb (exact
// product) to the accumulator.  Lane partials are
// combined by a shuffle butterfly; the summation order depends only on
// (K, LPR, KS), so results are reproducible and identical for both scale
// layouts.
#pragma once
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

// The order rows are visited in.  Plain scales: m = 0..M-1.  Permuted
// scales: inside each 128-row atom block, the 8 rows of a pass are those whose
// scale bytes share one 32-byte sector of the atom: m%32 in {2j, 2j+1} and
// all four (m/32)%4.
template <bool PERM>
__device__ __forceinline__ int64_t visited_row(int64_t rp) {
  if (!PERM) return rp;
  const int q = (int)(rp & 127);
  const int j = q >> 3, t = q & 7;
  return (rp & ~(int64_t)127) + 32 * (t >> 1) + 2 * j + (t & 1);
}

// Units [begin, end) of row lane wr (of WR) in this CTA.  CTA b takes units
// [floor(T*b/ctas), floor(T*(b+1)/ctas)) of the T = units_q*ctas + units_r
// units (the extra units spread evenly over the grid), computed as
// units_q*b + floor(units_r*b/ctas) with a 32-bit division whenever
// units_r*b fits; a CTA's units are cut evenly (to one unit) among its row
// lanes.
__device__ __forceinline__ int64_t cta_first_unit(const GemvParams& p, uint64_t b) {
  const uint64_t n = (uint64_t)gridDim.x;
  const uint64_t rb = (uint64_t)p.units_r * b;
  const uint64_t extra = rb <= 0xffffffffull ? (uint64_t)((uint32_t)rb / (uint32_t)n) : rb / n;
  return (int64_t)((uint64_t)p.units_q * b + extra);
}
template <int WR>
__device__ __forceinline__ void row_lane_units(const GemvParams& p, int wr, int64_t& begin,
                                               int64_t& end) {
  const int64_t c0 = cta_first_unit(p, blockIdx.x);
  const uint64_t len = (uint64_t)(cta_first_unit(p, blockIdx.x + 1ull) - c0);
  begin = c0 + (int64_t)(len * (uint64_t)wr / WR);
  end = c0 + (int64_t)(len * (uint64_t)(wr + 1) / WR);
}

// Batch of visit row r (32-bit division whenever the rows fit in 32 bits).
__device__ __forceinline__ int batch_of(const GemvParams& p, int64_t r) {
  if (p.rows_total <= 0xffffffffll) return (int)((uint32_t)r / (uint32_t)p.rows_per_l);
  return (int)(r / p.rows_per_l);
}

// c[idx] from the row's fp32 sum v: fp16(alpha * v + bias[idx]) rounded to
// nearest even, with one fp32 rounding before it (a fused multiply-add when
// there is a bias; alpha = 1 without one gives v itself).
__device__ __forceinline__ uint16_t finish_output(const GemvParams& p, float v, int64_t idx) {
  return finish_value(v, p.alpha, p.bias, p.activation, idx);
}

// Byte offset of the 4 scale bytes (blocks 4kt..4kt+3) of row m, chunk 0.
template <bool PERM>
__device__ __forceinline__ int64_t scale_row_offset(const GemvParams& p, int64_t l, int64_t m) {
  if (!PERM) return (l * p.M + m) * p.blocks;
  return ((l * p.rest_m + (m >> 7)) * p.rest_k) * 512 + (m & 31) * 16 + ((m >> 5) & 3) * 4;
}

template <bool PERM>
__device__ __forceinline__ int64_t scale_chunk_stride() {
  return PERM ? 512 : 4;
}

// Dot product of one 16-element block of one row with the matching block of
// b (bh: 8 half2 holding b's elements 2j, 2j+1), as an f16x2 pair of partial
// sums: every product is a multiple of 1/4 below 36 in magnitude and each
// half2 lane sums 8 of them, so both halves are exact.
__device__ __forceinline__ uint32_t block_dot(uint32_t w0, uint32_t w1, const uint32_t (&bh)[8]) {
  uint32_t d0[4], d1[4];
  e2m1x8_to_f16x2x4(w0, d0);
  e2m1x8_to_f16x2x4(w1, d1);
  uint32_t h = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) h = hfma2(d0[j], bh[j], h);
#pragma unroll
  for (int j = 0; j < 4; ++j) h = hfma2(d1[j], bh[4 + j], h);
  return h;
}

// acc + (block dot) * sfa * sfb: the dot's two halves times sfa exactly
// (f16x2_sum_times; sfa is the HI or low half of the f16x2 sa2), then one fp32
// fma with sfb (exact product, one rounding).
template <bool HI>
__device__ __forceinline__ float block_accumulate(uint32_t h, uint32_t sa2, float sb, float acc) {
  return fmaf(f16x2_sum_times<HI>(h, sa2), sb, acc);
}

// E4M3 scale of block blk (0..3) of a 4-byte scale word, as fp32 (exact).
__device__ __forceinline__ float scale_of(uint32_t word, int blk) {
  const uint32_t h = e4m3x2_to_f16x2(word >> (16 * (blk >> 1)));
  return (blk & 1) ? f16_hi_to_f32(h) : f16_lo_to_f32(h);
}

// Sum each of NV values over the lanes that differ in bits OFF, OFF/2, ..., 1.
// Each level halves the values a lane keeps (the upper half when the lane's
// OFF bit is set), so the result for value index i ends in the lanes whose
// bits OFF..OFF/(NV/2) spell i.
template <int NV, int OFF>
__device__ __forceinline__ float lane_reduce(const float (&v)[NV], int lane) {
  if constexpr (NV == 1) {
    float x = v[0];
#pragma unroll
    for (int o = OFF; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
  } else {
    constexpr int H = NV / 2;
    const bool upper = (lane & OFF) != 0;
    float w[H];
#pragma unroll
    for (int t = 0; t < H; ++t) {
      const float send = upper ? v[t] : v[t + H];
      const float keep = upper ? v[t + H] : v[t];
      w[t] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
    }
    return lane_reduce<H, OFF / 2>(w, lane);
  }
}

template <int LPR, int KS, bool PERM>
__global__ void __launch_bounds__(kGemvThreads, kGemvMinCtasPerSm)
    nvfp4_gemv_kernel(const GemvParams p) {
  constexpr int RI = 32 / LPR;            // rows per warp-wide load
  constexpr int NI = kRowsPerPass / RI;   // loads per lane per chunk step
  constexpr int WR = kGemvWarps / KS;     // row lanes per CTA
  static_assert(LPR >= 4 && LPR <= 32 && (LPR & (LPR - 1)) == 0, "LPR in {4,8,16,32}");
  static_assert(KS >= 1 && KS <= kGemvWarps && (kGemvWarps % KS) == 0, "KS divides the warps per CTA");
  __shared__ float red[KS > 1 ? WR : 1][KS][kRowsPerPass];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wr = warp / KS, ks = warp % KS;
  const int sub = lane / LPR, kc = lane % LPR;

  pdl_launch_dependents();

  int64_t r_begin, r_end;
  row_lane_units<WR>(p, wr, r_begin, r_end);

  pdl_wait();

  int64_t l = r_begin < r_end ? batch_of(p, r_begin) : 0;
  for (int64_t r = r_begin; r < r_end;) {
    if (r >= (l + 1) * p.rows_per_l) ++l;  // passes never cross a batch
    const int64_t batch_end = (l + 1) * p.rows_per_l;
    const int64_t pass_end = min(min(r_end, r + kRowsPerPass), batch_end);
    const int cnt = (int)(pass_end - r);
    const int64_t rp0 = r - l * p.rows_per_l;

    int64_t a_off[NI], s_off[NI];
    bool valid[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int rho = i * RI + sub;
      const int64_t m = visited_row<PERM>(rp0 + rho);
      valid[i] = rho < cnt && m < p.M;
      a_off[i] = (l * p.M + m) * p.half_k;
      s_off[i] = scale_row_offset<PERM>(p, l, m);
    }
    const uint8_t* brow = p.b + l * p.b_stride;
    const uint8_t* sbrow = p.sfb + l * p.sfb_stride;

    float acc[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) acc[i] = 0.f;

    for (int s = ks; s < p.steps; s += KS) {
      const int kt = s * LPR + kc;
      if (kt < p.kchunks) {
        uint32_t av[NI][8];
        uint32_t sw[NI];
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          if (valid[i]) {
            ld_stream_256(p.a + a_off[i] + (int64_t)kt * 32, av[i]);
            sw[i] = ld_scale_32(p.sfa + s_off[i] + kt * scale_chunk_stride<PERM>());
          }
        }
        uint32_t bw[8];
        ld_shared_2x128(brow + (int64_t)kt * 32, bw);
        const uint32_t sbw = ld_scale_32(sbrow + kt * scale_chunk_stride<PERM>());
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          uint32_t bh[8];
          {
            uint32_t lo[4], hi[4];
            e2m1x8_to_f16x2x4(bw[2 * blk], lo);
            e2m1x8_to_f16x2x4(bw[2 * blk + 1], hi);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              bh[j] = lo[j];
              bh[4 + j] = hi[j];
            }
          }
          const float sb = scale_of(sbw, blk);
#pragma unroll
          for (int i = 0; i < NI; ++i) {
            if (valid[i]) {
              const uint32_t h = block_dot(av[i][2 * blk], av[i][2 * blk + 1], bh);
              const uint32_t sa2 = e4m3x2_to_f16x2(sw[i] >> (16 * (blk >> 1)));
              acc[i] = (blk & 1) ? block_accumulate<true>(h, sa2, sb, acc[i])
                                 : block_accumulate<false>(h, sa2, sb, acc[i]);
            }
          }
        }
      }
    }

    float v = lane_reduce<NI, LPR / 2>(acc, lane);
    const int rho_out = ((kc >> 2) & (NI - 1)) * RI + sub;
    const bool holder = (kc & 3) == 0;
    if constexpr (KS > 1) {
      if (holder) red[wr][ks][rho_out] = v;
      named_barrier_sync(1 + wr, 32 * KS);
      if (ks == 0 && holder) {
        float t = red[wr][0][rho_out];
#pragma unroll
        for (int j = 1; j < KS; ++j) t += red[wr][j][rho_out];
        v = t;
      }
      named_barrier_sync(1 + wr, 32 * KS);
    }
    if ((KS == 1 || ks == 0) && holder && rho_out < cnt) {
      const int64_t m = visited_row<PERM>(rp0 + rho_out);
      if (m < p.M) p.c[l * p.M + m] = finish_output(p, v, l * p.M + m);
    }
    r = pass_end;
  }
}

template <bool PERM>
cudaError_t launch_gemv_layout(const GemvParams& p, const GemvPlan& plan, cudaStream_t stream) {
  void (*kern)(GemvParams) = nullptr;
#define NVFP4_CASE(LPR_, KS_) \
  if (plan.lanes_per_row == LPR_ && plan.k_split == KS_) kern = nvfp4_gemv_kernel<LPR_, KS_, PERM>;
#define NVFP4_CASES_KS(LPR_) \
  NVFP4_CASE(LPR_, 1) NVFP4_CASE(LPR_, 2) NVFP4_CASE(LPR_, 4) NVFP4_CASE(LPR_, 8)
  NVFP4_CASES_KS(4)
  NVFP4_CASES_KS(8)
  NVFP4_CASES_KS(16)
  NVFP4_CASES_KS(32)
#undef NVFP4_CASES_KS
#undef NVFP4_CASE
  if (kern == nullptr) return cudaErrorInvalidConfiguration;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.ctas, 1, 1);
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace nvfp4

// NVFP4 block-scaled batched GEMV (sm_103a): 16-element block dots on the
// tensor cores, E4M3 scales applied on the CUDA cores.
//
//   c[m,l] = fp16( sum_blocks E4M3(sfa[m,j,l]) * E4M3(sfb[j,l]) * dot16_j(a[m,l], b[l]) )
//
// The per-element form a*sfa*b*sfb of `cute_kernel` (kernelbot nvfp4-gemv
// submission 103289) regrouped per 16-element scale block: dot16_j is the
// unscaled dot product of block j, and every one is exact in fp32 (products
// are multiples of 1/4 below 36, sums of 16 of them below 2^10).
//
// Block dots on the tensor cores.  The block-scaled MMA (kind::mxf4nvf4,
// M = 128, N = 16, K = 64, a 16-element scale per row and block) does the
// block separation itself: every row of its B operand holds b's bytes (one
// TMA copy replicates them, through a tensor map whose row stride is zero),
// A's scales are all 1.0, and B's scales are a constant selector: for the MMA
// of 64-element chunk c of a 128-byte column block, B row n = 4*c + j has scale
// 1.0 on block j and 0 on the other three blocks, and every other row has
// scale 0.  That MMA therefore writes, in accumulator column 4*c + j, the dot
// of A's block j of chunk c with b's, and zeros in the other columns; a
// column block's 4 MMAs accumulate into 16 columns holding its 16 block dots
// of every row.  (E2M1 has no Inf or NaN, so the zero scales give exact
// zeros; the selector and unit scales are written to TMEM once.)
//
// A K stage is CB column blocks (CB = 2, 512 elements, when K % 256 == 0;
// else 1): every copy, wait and commit costs a thread 50 to 170 cycles
// whatever its size, so a stage carries as many bytes as the ring allows.
//
// Scales on the CUDA cores.  Each epilogue thread owns one row of the tile:
// it reads the row's 16*CB block dots from TMEM, decodes the sfa and sfb
// codes with cvt.rn.f16x2.e4m3x2 (exact, signed, NaN kept), forms
// sfa*sfb exactly in fp32 and adds dot * (sfa*sfb) to an fp32 accumulator,
// block by block in K order.  Signed and NaN scale codes are thus read as
// E4M3 (the MMA's own scale path reads unsigned UE4M3 codes).
//
// Work split: rows are handed out in units of 8 rows, all batches in one
// sequence; CTA i takes a contiguous range of units (ranges differ by at most
// one unit) and walks it in tiles of at most slot_rows rows that never cross
// a batch (nor, for pre-permuted scales, a 128-row atom block), each over the
// whole K.  No partial sums leave a CTA, and the summation order of a row
// depends only on K.  (With pre-permuted scales, CTAs that share an atom
// block each copy the block's atoms; they reach those stages at about the
// same time, so the second copy is mostly served by the L2.)
//
// Roles of a CTA (192 threads):
//   warp 0      one lane issues each K stage's 4 copies into a ring slot: A
//               as one TMA box of slot_rows rows x CB column blocks of 128
//               bytes (128-byte swizzle), plain sfa as one box of slot_rows x
//               16*CB bytes (or the stage's permuted atoms as one bulk copy),
//               b's bytes replicated into 16 swizzled rows per column block,
//               and the stage's sfb bytes; all complete one mbarrier;
//   warp 1      allocates TMEM and writes the unit and selector scales; per
//               stage one lane issues the 4*CB MMAs into one of kBdD
//               accumulator buffers and commits it to the epilogue (each MMA
//               costs the thread about 110 cycles; a second issuing warp,
//               alternating stages, gave results that varied from run to run
//               on the largest workloads, so one thread issues them all);
//   warps 2..5  the epilogue (one TMEM lane quarter, i.e. 32 rows, each).
// A ring slot is free again once the 4 epilogue warps have read its scale
// bytes, which they do after the slot's MMAs have completed.  Before the
// dependency wait, the producer asks the L2 to prefetch the A boxes of its
// first stages.
//
// One lane per warp waits on an mbarrier (then __syncwarp): threads polling a
// barrier slow down every barrier operation of the CTA.  Every wait gives up
// after 2 s of global time, counts a timeout (nvfp4_tensor_wait_timeouts) and
// makes its warp skip the rest of its work; control flow stays uniform so
// TMEM is always freed.
#include <cstdint>
#include <cstring>

#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace nvfp4 {

__device__ int g_bd_timeouts;

namespace {

constexpr int kBdThreads = kBlockDotThreads;  // 6 warps
constexpr int kBdD = 4;                       // accumulator buffers of 16*CB TMEM columns
constexpr uint32_t kBdTmemCols = 256;
// The constant scales: 4 columns of unit scales for A, then 4 x 4 columns of
// B's selector scales of chunks 0..3.
constexpr uint32_t kBdScales = 16 * 2 * kBdD;  // first scale column
static_assert(kBdScales + 20 <= kBdTmemCols, "TMEM columns");
constexpr uint32_t kBdIdesc = tc::mxf4nvf4_idesc(16);
constexpr uint32_t kBdBBytes = 16 * 128;      // B of one column block: b's 128 bytes in 16 rows
constexpr uint32_t kBdAtoms = 5 * 512;        // the unit atom and the 4 selector atoms
// sfb bytes of one stage (at most 32 used, 128 for pre-permuted scales); a
// tiled TMA copy's shared-memory destination is 128-byte aligned
constexpr uint32_t kBdSfbSlot = 128;

struct BdParams {
  CUtensorMap tmap_a;    // CB = 2: uint8 {128, M, K/256, L}, box {128, slot_rows, 2, 1};
                         // CB = 1: uint8 {K/2, M, L}, box {128, slot_rows, 1}; 128-byte swizzle
  CUtensorMap tmap_s;    // plain sfa: uint8 {K/16, M, L}, box {16*CB, slot_rows, 1}
  CUtensorMap tmap_b;    // b replicated: CB = 2 {128, 16 (stride 0), K/256, L}, box {128, 16, 2, 1};
                         // CB = 1 {K/2, 16 (stride 0), L}, box {128, 16, 1}; 128-byte swizzle
  CUtensorMap tmap_sfb;  // pre-permuted sfb: {16 bytes, rest_k atoms (stride 512), L}, box {16, 4*CB, 1}
  const uint8_t* sfa;    // pre-permuted atoms [L][rest_m][rest_k][512]
  const uint8_t* sfb;    // plain sfb: batch l at sfb + l*sfb_stride
  uint16_t* c;           // fp16 [L][M]
  const uint16_t* bias;  // fp16 [L][M], or null
  float alpha;
  int32_t activation;    // nvfp4_activation_t
  int64_t M;
  int64_t sfb_stride;
  int64_t units_per_l;   // 8-row units per batch
  int64_t units_q;       // the L*units_per_l units = units_q*ctas + units_r,
  int32_t units_r;       //   spread evenly over the CTAs
  int32_t rest_m, rest_k, kstages;  // kstages = ceil(rest_k / (4*CB))
  int32_t slot_rows;     // A rows per ring slot (a multiple of 8, <= 128)
  int32_t stages;        // ring slots
  int32_t prefetch_stages;  // stages whose A boxes are prefetched before the dependency wait
  uint32_t off_b, off_sfa, off_sfbv, off_unit;  // shared-memory offsets
  uint32_t sfa_slot_bytes;
};

// First unit of CTA i: units_q*i + floor(units_r*i/ctas).
__device__ __forceinline__ int64_t bd_first_unit(const BdParams& p, uint64_t i) {
  return (int64_t)((uint64_t)p.units_q * i + ((uint64_t)p.units_r * i) / (uint64_t)gridDim.x);
}

// The tiles of one CTA: maximal runs of its units inside one batch (and one
// 128-row atom block for pre-permuted scales), at most slot_rows rows each.
// Every tile is copied as one box of slot_rows rows, placed inside the CTA's
// own rows of the batch where it can be (so the rows it adds are ones this
// CTA copies anyway, mostly from the L2): starting at the tile's first row,
// or ending at the CTA's last row of the batch.
template <bool PERM>
struct BdTiles {
  static constexpr int UR = 8;  // rows per unit
  int64_t u_begin, u, u_end;    // the CTA's units; the next tile's first unit
  int64_t m0;    // first row of the tile (in its batch)
  int64_t box0;  // first row of the tile's box (may precede the batch: zero fill)
  int l;         // batch
  int rows;      // rows of the tile that exist (< M)

  __device__ __forceinline__ bool next(const BdParams& p) {
    if (u >= u_end) return false;
    // (a 32-bit division whenever the units fit: the 64-bit one is a long
    // software sequence on the producer's critical path)
    l = u_end <= 0xffffffffll ? (int)((uint32_t)u / (uint32_t)p.units_per_l)
                              : (int)(u / p.units_per_l);
    const int64_t l0 = (int64_t)l * p.units_per_l;
    const int64_t uu = u - l0;
    m0 = uu * UR;
    int64_t n = u_end - u;
    if (p.units_per_l - uu < n) n = p.units_per_l - uu;
    if (p.slot_rows / UR < n) n = p.slot_rows / UR;
    if (PERM && (128 - (m0 & 127)) / UR < n) n = (128 - (m0 & 127)) / UR;
    u += n;
    rows = (int)(p.M - m0 < n * UR ? p.M - m0 : n * UR);
    // the CTA's rows of batch l: [lo, hi)
    const int64_t lo = (u_begin > l0 ? u_begin - l0 : 0) * UR;
    int64_t hi = (u_end - l0 < p.units_per_l ? u_end - l0 : p.units_per_l) * UR;
    if (hi > p.M) hi = p.M;
    box0 = hi - lo >= p.slot_rows ? (m0 < hi - p.slot_rows ? m0 : hi - p.slot_rows) : lo;
    return true;
  }
};

// fp32 -> fp16 output (the epilogue of every kernel).
__device__ __forceinline__ uint16_t bd_finish(const BdParams& p, float v, int64_t idx) {
  return finish_value(v, p.alpha, p.bias, p.activation, idx);
}

// sfa * sfb of one block, exact in fp32: the low (HI = false) or high halves
// of two f16x2 holding decoded E4M3 scales, multiplied by a mixed
// fp16 x fp16 + fp32 fma (4 significant bits each, so nothing rounds).
template <bool HI>
__device__ __forceinline__ float scale_product(uint32_t a2, uint32_t b2) {
  float t;
  if (HI)
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, 0f00000000;\n\t}"
        : "=f"(t)
        : "r"(a2), "r"(b2));
  else
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, 0f00000000;\n\t}"
        : "=f"(t)
        : "r"(a2), "r"(b2));
  return t;
}

// acc + sum over the 4 blocks of one 64-element chunk of dot * sfa * sfb, in
// block order; sa, sb hold the chunk's 4 scale codes (block j in byte j).
__device__ __forceinline__ float chunk_accumulate(const float* dot, uint32_t sa, uint32_t sb,
                                                  float acc) {
  const uint32_t a01 = e4m3x2_half_to_f16x2<false>(sa), a23 = e4m3x2_half_to_f16x2<true>(sa);
  const uint32_t b01 = e4m3x2_half_to_f16x2<false>(sb), b23 = e4m3x2_half_to_f16x2<true>(sb);
  acc = fmaf(dot[0], scale_product<false>(a01, b01), acc);
  acc = fmaf(dot[1], scale_product<true>(a01, b01), acc);
  acc = fmaf(dot[2], scale_product<false>(a23, b23), acc);
  acc = fmaf(dot[3], scale_product<true>(a23, b23), acc);
  return acc;
}

// The A (and replicated b) copies of stage s: column blocks CB*s.. (CB = 2)
// or the 128 bytes at 128*s (CB = 1).
template <int CB>
__device__ __forceinline__ void tma_stage(uint32_t dst, const CUtensorMap* map, int s, int row,
                                          int l, uint32_t bar) {
  if constexpr (CB == 1)
    tc::tma_load_3d(dst, map, s * 128, row, l, bar);
  else
    tc::tma_load_4d(dst, map, 0, row, CB * s, l, bar);
}

template <bool PERM, int CB>
__global__ void __launch_bounds__(kBdThreads, 1)
    nvfp4_blockdot_kernel(const __grid_constant__ BdParams p) {
  constexpr int NC = 4 * CB;  // 64-element chunks per stage
  extern __shared__ uint8_t bd_smem[];
  __shared__ __align__(8) uint64_t bars[2 * kBlockDotMaxStages + 2 * kBdD + 1];
  __shared__ uint32_t tmem_slot;

  const uint32_t raw = smem_u32(bd_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzled tiles want 1024-byte alignment
  uint8_t* const gen = bd_smem - raw;            // generic pointer = gen + shared address
  const int S = p.stages;
  const uint32_t cb_bytes = (uint32_t)p.slot_rows * 128u;  // one column block of an A slot
  const uint32_t a_slot_bytes = CB * cb_bytes;
  const uint32_t a_s = base, b_s = base + p.off_b, sfa_s = base + p.off_sfa;
  const uint32_t sfbv_s = base + p.off_sfbv, unit_s = base + p.off_unit;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](uint32_t st) { return bar0 + 8u * st; };
  auto empty_bar = [&](uint32_t st) { return bar0 + 8u * (kBlockDotMaxStages + st); };
  auto dfull_bar = [&](uint32_t d) { return bar0 + 8u * (2 * kBlockDotMaxStages + d); };
  auto dempty_bar = [&](uint32_t d) { return bar0 + 8u * (2 * kBlockDotMaxStages + kBdD + d); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kBlockDotMaxStages + 2 * kBdD);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  BdTiles<PERM> tiles0;
  tiles0.u_begin = tiles0.u = bd_first_unit(p, blockIdx.x);
  tiles0.u_end = bd_first_unit(p, blockIdx.x + 1ull);

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int st = 0; st < S; ++st) {
      tc::mbar_init(full_bar(st), 1);
      tc::mbar_init(empty_bar(st), 4);  // the 4 epilogue warps
    }
    for (int d = 0; d < kBdD; ++d) {
      tc::mbar_init(dfull_bar(d), 1);
      tc::mbar_init(dempty_bar(d), 4);
    }
    tc::mbar_init(drain_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the scale atoms (the pre-permuted 128x4 layout: byte (row n, block j) at
  // n*16 + j for n < 32): atom 0 all 1.0 (E4M3 0x38) for A; atom 1 + c the
  // selector of chunk c for B, 1.0 at (4*c + j, j) and 0 elsewhere
  for (uint32_t i = threadIdx.x; i < kBdAtoms / 4; i += kBdThreads) {
    const uint32_t atom = i / 128, byte0 = 4 * (i % 128);
    uint32_t w = 0;
    for (uint32_t k = 0; k < 4; ++k) {
      const uint32_t n = (byte0 + k) / 16, j = (byte0 + k) % 16;
      const bool one = atom == 0 || (j < 4 && n == 4 * (atom - 1) + j);
      w |= (one ? 0x38u : 0u) << (8 * k);
    }
    *reinterpret_cast<uint32_t*>(gen + unit_s + 4 * i) = w;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
  if (warp == 1) tc::alloc(smem_u32(&tmem_slot), kBdTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;


  if (warp == 0) {
    if (lane == 0) {
      // the first stages' A boxes, ahead of the dependency wait (the L2 is
      // coherent: the copies after the wait still read what earlier work on
      // the stream wrote)
      {
        BdTiles<PERM> t = tiles0;
        int n = 0;
        while (n < p.prefetch_stages && t.next(p)) {
          for (int s = 0; s < p.kstages && n < p.prefetch_stages; ++s, ++n) {
            if constexpr (CB == 1)
              tc::tma_prefetch_3d(&p.tmap_a, s * 128, (int)t.box0, t.l);
            else
              tc::tma_prefetch_4d(&p.tmap_a, 0, (int)t.box0, CB * s, t.l);
          }
        }
      }
      pdl_wait();
      BdTiles<PERM> t = tiles0;
      uint32_t slot = 0, ph = 0;
      while (t.next(p)) {
        const uint8_t* sfa_blk =
            PERM ? p.sfa + (((int64_t)t.l * p.rest_m + (t.m0 >> 7)) * p.rest_k) * 512 : nullptr;
        const uint8_t* sfb_l = p.sfb + (int64_t)t.l * p.sfb_stride;
        for (int s = 0; s < p.kstages;
             ++s, slot = slot + 1 == (uint32_t)S ? 0 : slot + 1, ph ^= slot == 0 ? 1u : 0u) {
          if (!tc::mbar_wait<false>(empty_bar(slot), ph ^ 1u, ok, &g_bd_timeouts)) continue;
          const int nks = min(NC, p.rest_k - NC * s);  // chunks of this stage
          const uint32_t fb = full_bar(slot);
          const uint32_t sfa_bytes = PERM ? 512u * (uint32_t)nks : 16u * CB * (uint32_t)p.slot_rows;
          const uint32_t sfb_bytes = PERM ? 64u * CB : 16u * (uint32_t)((nks + 3) / 4);
          tc::mbar_expect_tx(fb, a_slot_bytes + sfa_bytes + CB * kBdBBytes + sfb_bytes);
          const uint32_t s_dst = sfa_s + slot * p.sfa_slot_bytes;
          tma_stage<CB>(a_s + slot * a_slot_bytes, &p.tmap_a, s, (int)t.box0, t.l, fb);
          if (PERM)
            tc::bulk_load(s_dst, sfa_blk + (int64_t)s * NC * 512, 512u * (uint32_t)nks, fb);
          else
            tc::tma_load_3d(s_dst, &p.tmap_s, s * 16 * CB, (int)t.box0, t.l, fb);
          tma_stage<CB>(b_s + slot * CB * kBdBBytes, &p.tmap_b, s, 0, t.l, fb);
          if (PERM)  // the first 16 bytes (row 0's scales) of the stage's sfb atoms
            tc::tma_load_3d(sfbv_s + slot * kBdSfbSlot, &p.tmap_sfb, 0, NC * s, t.l, fb);
          else
            tc::bulk_load(sfbv_s + slot * kBdSfbSlot, sfb_l + (int64_t)s * 16 * CB, sfb_bytes, fb);
        }
      }
      // copies still in flight land before the CTA can exit: the epilogue
      // releases a slot only after reading it, so waiting for every slot to
      // be released once more covers the last fill of each
      bool drain_ok = ok;
      for (int k = 0; k < S; ++k) {
        tc::mbar_wait<false>(empty_bar(slot), ph ^ 1u, drain_ok, &g_bd_timeouts);
        slot = slot + 1 == (uint32_t)S ? 0 : slot + 1;
        ph ^= slot == 0 ? 1u : 0u;
      }
    } else {
      pdl_wait();
    }
  } else if (warp == 1) {
    pdl_wait();
    if (lane == 0) {
      // unit scales for A, and B's selector of each chunk (4 columns each)
      const uint32_t scales = tmem + kBdScales;
      tc::copy_atom(scales, tc::desc_atom(unit_s));
      for (uint32_t c = 0; c < 4; ++c)
        tc::copy_atom(scales + 4 * (c + 1), tc::desc_atom(unit_s + 512 * (c + 1)));
      BdTiles<PERM> t = tiles0;
      uint32_t slot = 0, ph = 0, d = 0, dph = 0;
      while (t.next(p)) {
        for (int s = 0; s < p.kstages; ++s, slot = slot + 1 == (uint32_t)S ? 0 : slot + 1,
                 ph ^= slot == 0 ? 1u : 0u, d = (d + 1) % kBdD, dph ^= d == 0 ? 1u : 0u) {
          if (!tc::mbar_wait2(full_bar(slot), ph, dempty_bar(d), dph ^ 1u, ok, &g_bd_timeouts))
            continue;
          tc::fence_after();
          const int nks = min(NC, p.rest_k - NC * s);
          const uint32_t a_addr = a_s + slot * a_slot_bytes, b_addr = b_s + slot * CB * kBdBBytes;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            if (c < nks) {
              const uint32_t cb = c / 4, cc = c % 4;
              tc::mma(tmem + 16u * (CB * d + cb), tc::desc_sw128(a_addr + cb * cb_bytes + 32u * cc),
                      tc::desc_sw128(b_addr + cb * kBdBBytes + 32u * cc), kBdIdesc, scales,
                      scales + 4u * (cc + 1), cc > 0);
            }
          }
          tc::commit(dfull_bar(d));
        }
      }
      // every MMA and TMEM copy of this warp has finished before TMEM is released
      tc::commit(drain_bar);
      bool drain_ok = true;
      tc::mbar_wait<false>(drain_bar, 0, drain_ok, &g_bd_timeouts);
    }
    __syncwarp();
  } else {
    pdl_wait();
    const uint32_t q = (uint32_t)(warp & 3);  // the TMEM lane quarter this warp may read
    const int row = (int)(32 * q) + lane;     // box row = TMEM lane
    BdTiles<PERM> t = tiles0;
    uint32_t slot = 0, ph = 0, d = 0, dph = 0;
    while (t.next(p)) {
      const int64_t m = t.box0 + row;  // the row of box row `row`
      const bool mine = m >= t.m0 && m < t.m0 + t.rows;
      // pre-permuted: the row's 4-byte word inside each atom of its block
      const uint32_t perm_off = (uint32_t)((m & 31) * 16 + ((m >> 5) & 3) * 4);
      float acc = 0.f;
      for (int s = 0; s < p.kstages; ++s, slot = slot + 1 == (uint32_t)S ? 0 : slot + 1,
               ph ^= slot == 0 ? 1u : 0u, d = (d + 1) % kBdD, dph ^= d == 0 ? 1u : 0u) {
        const int nks = min(NC, p.rest_k - NC * s);
        if (lane == 0) tc::mbar_wait2(full_bar(slot), ph, dfull_bar(d), dph, ok, &g_bd_timeouts);
        __syncwarp();
        // one decision for the warp: the TMEM load below is warp-collective
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        float dot[16 * CB];
        uint32_t sa[NC], sb[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) sa[c] = sb[c] = 0;
        if (ok) {
          tc::fence_after();
          tc::tmem_load_cols<16 * CB>(tmem + 16u * CB * d + ((32u * q) << 16), dot);
          const uint32_t sfa_slot = sfa_s + slot * p.sfa_slot_bytes;
          const uint32_t sfb_slot = sfbv_s + slot * kBdSfbSlot;
          if (!PERM) {
            if (row < p.slot_rows) {
#pragma unroll
              for (int h = 0; h < CB; ++h) {
                const uint4 v =
                    *reinterpret_cast<const uint4*>(gen + sfa_slot + 16u * (CB * row + h));
                sa[4 * h] = v.x, sa[4 * h + 1] = v.y, sa[4 * h + 2] = v.z, sa[4 * h + 3] = v.w;
              }
            }
#pragma unroll
            for (int h = 0; h < CB; ++h) {
              const uint4 w = *reinterpret_cast<const uint4*>(gen + sfb_slot + 16u * h);
              sb[4 * h] = w.x, sb[4 * h + 1] = w.y, sb[4 * h + 2] = w.z, sb[4 * h + 3] = w.w;
            }
          } else {
#pragma unroll
            for (int c = 0; c < NC; ++c) {
              if (c < nks) {
                sa[c] = *reinterpret_cast<const uint32_t*>(gen + sfa_slot + 512u * c + perm_off);
                sb[c] = *reinterpret_cast<const uint32_t*>(gen + sfb_slot + 16u * c);
              }
            }
          }
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) {  // the accumulator buffer and the slot's scale bytes are read
          tc::mbar_arrive(dempty_bar(d));
          tc::mbar_arrive(empty_bar(slot));
        }
        if (ok) {
#pragma unroll
          for (int c = 0; c < NC; ++c)
            if (c < nks) acc = chunk_accumulate(dot + 4 * c, sa[c], sb[c], acc);
        }
      }
      if (ok && mine) {
        const int64_t idx = (int64_t)t.l * p.M + m;
        p.c[idx] = bd_finish(p, acc, idx);
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tmem, kBdTmemCols);
  }
}

// Shared-memory layout of one CTA for a ring of `stages` slots of slot_rows
// rows and CB column blocks: A slots, B tiles, the scale atoms, sfa slots,
// sfb bytes.
struct BdLayout {
  uint32_t off_b, off_sfa, off_sfbv, off_unit, total, sfa_slot_bytes;
};

BdLayout bd_layout(bool permuted, int cb, int slot_rows, int stages) {
  BdLayout o;
  const uint32_t S = (uint32_t)stages, CB = (uint32_t)cb;
  o.sfa_slot_bytes = permuted ? 2048u * CB : 16u * CB * (uint32_t)slot_rows;
  o.off_b = S * CB * 128u * (uint32_t)slot_rows;  // A slots: multiples of 1024 bytes
  o.off_unit = o.off_b + S * CB * kBdBBytes;      // 1024-byte aligned
  o.off_sfa = o.off_unit + kBdAtoms;              // slots: multiples of 128 bytes
  o.off_sfbv = o.off_sfa + S * o.sfa_slot_bytes;
  o.total = o.off_sfbv + S * kBdSfbSlot;
  // the MMA reads 128 rows (16 KB) from the start of each column block of an
  // A slot, past a short one into what follows: the last slot's last column
  // block's window stays inside the allocation
  const uint32_t window = (S * CB - 1) * 128u * (uint32_t)slot_rows + 16384u;
  if (o.total < window) o.total = window;
  return o;
}

template <bool PERM>
using BdKernel = void (*)(BdParams);

}  // namespace

int blockdot_unit_rows(bool) { return 8; }

int blockdot_column_blocks(int64_t K) { return K % 256 == 0 ? 2 : 1; }

int blockdot_slot_rows(int64_t M, int64_t L, bool permuted, int64_t ctas) {
  const int64_t ur = blockdot_unit_rows(permuted);
  const int64_t units = L * ((M + ur - 1) / ur);
  const int64_t per_cta = ctas > 0 ? (units + ctas - 1) / ctas * ur : ur;
  int64_t rows = per_cta < 128 ? per_cta : 128;
  const int64_t batch = (M + ur - 1) / ur * ur;
  if (batch < rows) rows = batch;
  return (int)rows;
}

size_t blockdot_smem_bytes(bool permuted, int cb, int slot_rows, int stages) {
  return (size_t)bd_layout(permuted, cb, slot_rows, stages).total + 1024u;  // + alignment slack
}

int blockdot_max_stages(bool permuted, int cb, int slot_rows, size_t smem_per_cta) {
  int s = kBlockDotMaxStages;
  while (s > 1 && blockdot_smem_bytes(permuted, cb, slot_rows, s) > smem_per_cta) --s;
  return s;
}

cudaError_t launch_blockdot(const GemvParams& gp, bool permuted, int64_t L, int stages,
                            int64_t ctas, cudaStream_t stream) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  const int64_t K = 2 * (int64_t)gp.half_k;
  const int cb = blockdot_column_blocks(K);
  const int slot_rows = blockdot_slot_rows(gp.M, L, permuted, ctas);
  if (stages < 2 || stages > kBlockDotMaxStages) return cudaErrorInvalidValue;
  const BdLayout lay = bd_layout(permuted, cb, slot_rows, stages);
  BdParams p;
  memset(&p, 0, sizeof(p));
  const cuuint64_t half_k = (cuuint64_t)gp.half_k, M = (cuuint64_t)gp.M, LL = (cuuint64_t)L;
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  auto enc = [&](CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                 const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  sw == CU_TENSOR_MAP_SWIZZLE_128B ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                                   : CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const cuuint32_t rows = (cuuint32_t)slot_rows;
  bool good = true;
  if (cb == 2) {
    // A as {128 bytes, rows, column blocks, batches}: a box lands as
    // [column block][row][128 bytes]; b likewise with 16 rows of stride 0
    const cuuint64_t ad[4] = {128, M, half_k / 128, LL};
    const cuuint64_t as[3] = {half_k, 128, half_k * M};
    const cuuint32_t ab[4] = {128, rows, 2, 1};
    good = good && enc(&p.tmap_a, gp.a, 4, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B);
    const cuuint64_t bd[4] = {128, 16, half_k / 128, LL};
    const cuuint64_t bs[3] = {0, 128, (cuuint64_t)gp.b_stride};
    const cuuint32_t bb[4] = {128, 16, 2, 1};
    good = good && enc(&p.tmap_b, gp.b, 4, bd, bs, bb, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const cuuint64_t ad[3] = {half_k, M, LL};
    const cuuint64_t as[2] = {half_k, half_k * M};
    const cuuint32_t ab[3] = {128, rows, 1};
    good = good && enc(&p.tmap_a, gp.a, 3, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B);
    const cuuint64_t bd[3] = {half_k, 16, LL};
    const cuuint64_t bs[2] = {0, (cuuint64_t)gp.b_stride};
    const cuuint32_t bb[3] = {128, 16, 1};
    good = good && enc(&p.tmap_b, gp.b, 3, bd, bs, bb, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!permuted) {
    const cuuint64_t blocks = (cuuint64_t)gp.blocks;
    const cuuint64_t sd[3] = {blocks, M, LL};
    const cuuint64_t ss[2] = {blocks, blocks * M};
    const cuuint32_t sbx[3] = {16u * (cuuint32_t)cb, rows, 1};
    good = good && enc(&p.tmap_s, gp.sfa, 3, sd, ss, sbx, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    // the first 16 bytes of each sfb atom (row 0's scales in bytes 0..3)
    const cuuint64_t fd[3] = {16, (cuuint64_t)gp.rest_k, LL};
    const cuuint64_t fs[2] = {512, (cuuint64_t)gp.sfb_stride};
    const cuuint32_t fb[3] = {16, 4u * (cuuint32_t)cb, 1};
    good = good && enc(&p.tmap_sfb, gp.sfb, 3, fd, fs, fb, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (!good) return cudaErrorInvalidValue;
  const int64_t ur = blockdot_unit_rows(permuted);
  p.sfa = gp.sfa;
  p.sfb = gp.sfb;
  p.c = gp.c;
  p.bias = gp.bias;
  p.alpha = gp.alpha;
  p.activation = gp.activation;
  p.M = gp.M;
  p.sfb_stride = gp.sfb_stride;
  p.units_per_l = (gp.M + ur - 1) / ur;
  const int64_t units = L * p.units_per_l;
  p.units_q = units / ctas;
  p.units_r = (int32_t)(units % ctas);
  p.rest_m = gp.rest_m;
  p.rest_k = gp.rest_k;
  p.kstages = (gp.rest_k + 4 * cb - 1) / (4 * cb);
  p.slot_rows = slot_rows;
  p.stages = stages;
  p.prefetch_stages = stages;
  p.off_b = lay.off_b;
  p.off_sfa = lay.off_sfa;
  p.off_sfbv = lay.off_sfbv;
  p.off_unit = lay.off_unit;
  p.sfa_slot_bytes = lay.sfa_slot_bytes;

  void (*kern)(BdParams) = permuted ? (cb == 2 ? nvfp4_blockdot_kernel<true, 2>
                                               : nvfp4_blockdot_kernel<true, 1>)
                                    : (cb == 2 ? nvfp4_blockdot_kernel<false, 2>
                                               : nvfp4_blockdot_kernel<false, 1>);
  const size_t smem = blockdot_smem_bytes(permuted, cb, slot_rows, stages);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(kBdThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t blockdot_wait_timeouts(int reset, int* out) {
  cudaError_t err = cudaMemcpyFromSymbol(out, g_bd_timeouts, sizeof(int));
  if (err != cudaSuccess || !reset) return err;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_bd_timeouts, &zero, sizeof(int));
}

}  // namespace nvfp4

// NVFP4 block-scaled batched GEMV, per-warp cp.async pipelined kernel (sm_103a).
//
// Same work split and arithmetic as the direct kernel (gemv_kernel.cuh): CTA
// row ranges balanced to one row, row lanes of KS warps, LPR lanes per row,
// 32-byte K chunks per lane, exact half2 block dots, fp32 block scaling, a
// shuffle butterfly over the lanes of a row and a fixed-order shared-memory
// sum over the K-split warps.  What changes is how A reaches the registers:
//
//   * A warp's work is a sequence of tasks, one task = one K step of one pass
//     (kAsyncItems row items per lane).  Each lane copies its own A chunks and
//     scale words of a task into a per-warp ring of kAsyncStages shared-memory
//     slots with cp.async, and waits for them with its own wait_group: a lane
//     only ever reads bytes it copied, so no cross-lane synchronisation is
//     needed and no register holds in-flight data.
//   * The warp keeps kAsyncStages - 1 tasks in flight while it computes one,
//     so every warp streams continuously instead of alternating between a
//     burst of loads and a burst of arithmetic.
//   * The lane's 32 bytes of b (and its sfb word) are loaded into registers
//     one task ahead.
#pragma once
#include "gemv_kernel.cuh"

namespace nvfp4 {

// Row order of the pipelined kernel.  Plain scales: m = 0..M-1.  Permuted
// scales: inside each 128-row atom block, pass c (NR = 4*RI rows) holds the
// rows 32*g + c*RI + sub for g = 0..3 and sub < RI, in slot order g*RI + sub.
// The lane that takes the four rows g = 0..3 of one (c*RI + sub) finds their
// scale words side by side: the 16 bytes at ((m%32)*16) of each atom.
template <bool PERM, int RI>
__device__ __forceinline__ int64_t async_row(int64_t rp) {
  if (!PERM) return rp;
  constexpr int NR = 4 * RI;
  const int q = (int)(rp & 127);
  const int chunk = q / NR, t = q % NR;
  return (rp & ~(int64_t)127) + 32 * (t / RI) + chunk * RI + (t % RI);
}

// The (pass, K step) tasks of one warp: passes of NR = NI*RI rows of one
// batch over the row lane's range and, in each pass, the steps ks, ks + KS,
// ... below p.steps (the planner keeps KS <= steps, so every pass has one).
// What a lane needs per pass (pointers to its item-0 row of A, scales and
// c, and which items are real rows) is computed once when the pass starts;
// item i sits a fixed kernel-wide stride further, and a task adds only its K
// offset.
template <int LPR, bool PERM>
struct TaskCursor {
  static constexpr int NI = kAsyncItems, RI = 32 / LPR, NR = NI * RI;
  static constexpr int ROW_STEP = PERM ? 32 : RI;  // rows between a lane's items
  int64_t r, end;        // first visit-order row of the pass, end of the range
  int64_t l_begin;       // first visit row of the pass's batch
  int64_t l_end;         // first visit row of the next batch
  int64_t lm;            // l * M
  int l, cnt, s;
  bool done;
  uint32_t valid;        // bit i: the lane's item i is a real row
  const uint8_t* a0;     // the lane's item-0 row of A
  const uint8_t* s0;     // plain: its scale row; permuted: its 16-byte atom run (kt = 0)
  int64_t c0;            // index of its item-0 output

  __device__ __forceinline__ void start_pass(const GemvParams& p, int ks, int sub) {
    done = r >= end;
    if (done) return;
    if (r >= l_end) {  // passes never cross a batch, and advance by at most one
      ++l;
      l_begin = l_end;
      l_end += p.rows_per_l;
      lm += p.M;
    }
    const int64_t left = min(end, l_end) - r;
    cnt = left < NR ? (int)left : NR;
    s = ks;
    const int64_t rp = r - l_begin;  // visit row of the pass inside its batch
    valid = 0;
    if (!PERM) {
      c0 = lm + rp + sub;
      s0 = p.sfa + c0 * p.blocks;
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (i * RI + sub < cnt) valid |= 1u << i;
    } else {
      const int64_t m0 = async_row<true, RI>(rp + sub);  // item i is row m0 + 32*i
      c0 = lm + m0;
      s0 = p.sfa + (((int64_t)l * p.rest_m + (m0 >> 7)) * p.rest_k) * 512 + (m0 & 31) * 16;
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (i * RI + sub < cnt && m0 + 32 * i < p.M) valid |= 1u << i;
    }
    a0 = p.a + c0 * p.half_k;
  }
  __device__ __forceinline__ void init(const GemvParams& p, int64_t begin, int64_t e, int ks,
                                       int sub) {
    r = begin;
    end = e;
    l = (int)(begin < e ? begin / p.rows_per_l : 0);
    l_begin = (int64_t)l * p.rows_per_l;
    l_end = l_begin + p.rows_per_l;
    lm = (int64_t)l * p.M;
    start_pass(p, ks, sub);
  }
  __device__ __forceinline__ void advance(const GemvParams& p, int ks, int KS, int sub) {
    s += KS;
    if (s >= p.steps) {
      r += cnt;
      start_pass(p, ks, sub);
    }
  }
};

template <int LPR, int KS, bool PERM>
__global__ void __launch_bounds__(kGemvThreads, kGemvMinCtasPerSm)
    nvfp4_gemv_async_kernel(const GemvParams p) {
  using Cursor = TaskCursor<LPR, PERM>;
  constexpr int NI = Cursor::NI;           // row items per lane per task
  constexpr int RI = Cursor::RI;           // rows per warp-wide item
  constexpr int NR = Cursor::NR;           // rows per pass
  constexpr int WR = kGemvWarps / KS;      // row lanes per CTA
  constexpr int S = kAsyncStages;
  constexpr int SFA_OFF = NI * 1024;       // scale words ([lane][item] words) follow the A chunks
  static_assert(LPR >= NI && LPR <= 32 && (LPR & (LPR - 1)) == 0, "LPR in {4,8,16,32}");
  static_assert(KS >= 1 && KS <= kGemvWarps && (kGemvWarps % KS) == 0, "KS divides 8");
  extern __shared__ __align__(128) uint8_t ring_smem[];
  __shared__ float red[KS > 1 ? WR : 1][KS][NR];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wr = warp / KS, ks = warp % KS;
  const int sub = lane / LPR, kc = lane % LPR;
  const uint32_t ring = smem_u32(ring_smem) + (uint32_t)(warp * S * kAsyncStageBytes);
  const uint8_t* ring_gen = ring_smem + warp * S * kAsyncStageBytes;
  // a lane reads its 32-byte chunk as two 16-byte halves, lanes whose K chunk
  // index has bit 2 set taking the upper half first (spreads a quarter-warp
  // over all 32 banks; keyed on the chunk, so a row's arithmetic does not
  // depend on which lane group holds it)
  const bool swp = ((kc >> 2) & 1) != 0;
  const int h0 = swp ? 16 : 0;
  const uint32_t rot16 = swp ? 16u : 0u;

  pdl_launch_dependents();

  // Plain: ranges balanced to one row.  Permuted: balanced to one aligned
  // NR-row chunk (chunks never straddle a 128-row block or a batch).
  const int64_t unit = PERM ? NR : 1;
  const int64_t T = p.rows_total / unit;
  const int64_t c0 = T * (int64_t)blockIdx.x / gridDim.x;
  const int64_t c1 = T * (int64_t)(blockIdx.x + 1) / gridDim.x;
  const int64_t r_begin = (c0 + (c1 - c0) * wr / WR) * unit;
  const int64_t r_end = (c0 + (c1 - c0) * (wr + 1) / WR) * unit;

  pdl_wait();

  const int64_t a_step = (int64_t)Cursor::ROW_STEP * p.half_k;
  const int64_t s_step = (int64_t)Cursor::ROW_STEP * p.blocks;

  // copy this lane's part of task t (A chunks and scale words of its rows)
  auto issue = [&](const Cursor& t, int slot) {
    const int kt = t.s * LPR + kc;
    if (kt >= p.kchunks) return;
    const uint32_t a_dst = ring + (uint32_t)(slot * kAsyncStageBytes + lane * 32);
    const uint32_t s_dst = ring + (uint32_t)(slot * kAsyncStageBytes + SFA_OFF + lane * 16);
    const uint8_t* a_src = t.a0 + kt * 32;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      if (t.valid & (1u << i)) {
        cp_async_16(a_dst + i * 1024, a_src + i * a_step);
        cp_async_16(a_dst + i * 1024 + 16, a_src + i * a_step + 16);
        if (!PERM) cp_async_4(s_dst + i * 4, t.s0 + kt * 4 + i * s_step);
      }
    }
    // permuted: the four rows m0 + 32*i of this lane are one 16-byte run of
    // the atom (padding rows of the last block included, read as 0x00)
    if (PERM) cp_async_16(s_dst, t.s0 + (int64_t)kt * 512);
  };
  auto load_b = [&](int l, int kt, uint32_t (&w)[8], uint32_t& sw) {
    if (kt < p.kchunks) {
      ld_shared_256(p.b + (int64_t)l * p.half_k + kt * 32, w);
      sw = ld_scale_32(p.sfb + (PERM ? ((int64_t)l * p.rest_k + kt) * 512
                                     : (int64_t)l * p.blocks + kt * 4));
    }
  };

  Cursor ld, cp;
  ld.init(p, r_begin, r_end, ks, sub);
  cp = ld;
#pragma unroll
  for (int j = 0; j < S - 1; ++j) {
    if (!ld.done) {
      issue(ld, j);
      ld.advance(p, ks, KS, sub);
    }
    cp_async_commit();
  }
  // b (and sfb) of the task being computed, and of the next one when it differs
  uint32_t bw[8] = {0, 0, 0, 0, 0, 0, 0, 0}, sbw = 0;
  uint32_t bw_n[8] = {0, 0, 0, 0, 0, 0, 0, 0}, sbw_n = 0;
  if (!cp.done) load_b(cp.l, cp.s * LPR + kc, bw, sbw);

  float acc[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) acc[i] = 0.f;
  int slot = 0;
  bool pending_b = false;

  while (!cp.done) {
    // the slot computed in the previous iteration is free again
    if (!ld.done) {
      issue(ld, (slot + S - 1) % S);
      ld.advance(p, ks, KS, sub);
    }
    cp_async_commit();
    // the next task's b: same K step of the next pass, or the next step;
    // it changes unless there is one step per row and the batch stays
    const bool last_step = cp.s + KS >= p.steps;
    const bool more = !last_step || cp.r + cp.cnt < cp.end;
    const int s_n = last_step ? ks : cp.s + KS;
    const int l_n = (last_step && cp.r + cp.cnt >= cp.l_end) ? cp.l + 1 : cp.l;
    // b loaded during the previous task moves in only now, so its load
    // latency is hidden behind a whole task's compute
    if (pending_b) {
#pragma unroll
      for (int j = 0; j < 8; ++j) bw[j] = bw_n[j];
      sbw = sbw_n;
      pending_b = false;
    }
    const bool new_b = more && (s_n != cp.s || l_n != cp.l);
    if (new_b) {
      load_b(l_n, s_n * LPR + kc, bw_n, sbw_n);
      pending_b = true;
    }
    cp_async_wait<S - 1>();

    const int kt = cp.s * LPR + kc;
    if (kt < p.kchunks) {
      // Lanes with bit 2 set process the chunk's second 16-byte half (blocks
      // 2, 3) first; their b words and scale bytes are rotated to match, so the
      // block order inside registers stays static.
      const uint8_t* a_slot = ring_gen + slot * kAsyncStageBytes + lane * 32;
      const uint4 sw4 =
          *reinterpret_cast<const uint4*>(ring_gen + slot * kAsyncStageBytes + SFA_OFF + lane * 16);
      const uint32_t sws[4] = {sw4.x, sw4.y, sw4.z, sw4.w};
      uint32_t bwr[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bwr[j] = swp ? bw[4 + j] : bw[j];
        bwr[4 + j] = swp ? bw[j] : bw[4 + j];
      }
      const uint32_t sbwr = __funnelshift_l(sbw, sbw, rot16);
      uint32_t saw[NI];
#pragma unroll
      for (int i = 0; i < NI; ++i) saw[i] = __funnelshift_l(sws[i], sws[i], rot16);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint32_t bh0[8], bh1[8];
        {
          uint32_t q[4];
          e2m1x8_to_f16x2x4(bwr[4 * j], q);
#pragma unroll
          for (int t = 0; t < 4; ++t) bh0[t] = q[t];
          e2m1x8_to_f16x2x4(bwr[4 * j + 1], q);
#pragma unroll
          for (int t = 0; t < 4; ++t) bh0[4 + t] = q[t];
          e2m1x8_to_f16x2x4(bwr[4 * j + 2], q);
#pragma unroll
          for (int t = 0; t < 4; ++t) bh1[t] = q[t];
          e2m1x8_to_f16x2x4(bwr[4 * j + 3], q);
#pragma unroll
          for (int t = 0; t < 4; ++t) bh1[4 + t] = q[t];
        }
        const float sb0 = scale_of(sbwr, 2 * j), sb1 = scale_of(sbwr, 2 * j + 1);
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          if (cp.valid & (1u << i)) {
            const uint4 x = *reinterpret_cast<const uint4*>(a_slot + i * 1024 + ((j * 16) ^ h0));
            const uint32_t sa2 = e4m3x2_to_f16x2(saw[i] >> (16 * j));
            acc[i] = block_accumulate<false>(block_dot(x.x, x.y, bh0), sa2, sb0, acc[i]);
            acc[i] = block_accumulate<true>(block_dot(x.z, x.w, bh1), sa2, sb1, acc[i]);
          }
        }
      }
    }

    if (last_step) {
      float v = lane_reduce<NI, LPR / 2>(acc, lane);
      const int rho_out = (kc / (LPR / NI)) * RI + sub;
      const bool holder = (kc % (LPR / NI)) == 0;
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
      // a holder keeps item rho_out / RI of its own lane group (rho_out % RI
      // == sub), so its cursor knows the row
      const int item = rho_out / RI;
      if ((KS == 1 || ks == 0) && holder && (cp.valid & (1u << item)))
        p.c[cp.c0 + item * Cursor::ROW_STEP] = __half_as_ushort(__float2half_rn(v));
#pragma unroll
      for (int i = 0; i < NI; ++i) acc[i] = 0.f;
    }
    cp.advance(p, ks, KS, sub);
    slot = (slot + 1 == S) ? 0 : slot + 1;
  }
  cp_async_wait<0>();
}

template <bool PERM>
cudaError_t launch_async_layout(const GemvParams& p, const GemvPlan& plan, cudaStream_t stream) {
  void (*kern)(GemvParams) = nullptr;
#define NVFP4_CASE(LPR_, KS_) \
  if (plan.lanes_per_row == LPR_ && plan.k_split == KS_) kern = nvfp4_gemv_async_kernel<LPR_, KS_, PERM>;
#define NVFP4_CASES_KS(LPR_) \
  NVFP4_CASE(LPR_, 1) NVFP4_CASE(LPR_, 2) NVFP4_CASE(LPR_, 4) NVFP4_CASE(LPR_, 8)
  NVFP4_CASES_KS(4)
  NVFP4_CASES_KS(8)
  NVFP4_CASES_KS(16)
  NVFP4_CASES_KS(32)
#undef NVFP4_CASES_KS
#undef NVFP4_CASE
  if (kern == nullptr) return cudaErrorInvalidConfiguration;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAsyncSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.ctas, 1, 1);
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.dynamicSmemBytes = kAsyncSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace nvfp4

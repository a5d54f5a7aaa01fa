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

// The (pass, K step) tasks of one warp: passes of up to NR rows of one batch
// over the row lane's range and, in each pass, the steps ks, ks + KS, ...
// below p.steps (the planner keeps KS <= steps, so every pass has one).
template <int NR>
struct TaskCursor {
  int64_t r, l, end;
  int cnt, s;
  bool done;

  __device__ __forceinline__ void start_pass(const GemvParams& p, int ks) {
    done = r >= end;
    if (done) return;
    l = r / p.rows_per_l;
    cnt = (int)(min(min(end, r + NR), (l + 1) * p.rows_per_l) - r);
    s = ks;
  }
  __device__ __forceinline__ void init(const GemvParams& p, int64_t begin, int64_t e, int ks) {
    r = begin;
    end = e;
    start_pass(p, ks);
  }
  __device__ __forceinline__ void advance(const GemvParams& p, int ks, int KS) {
    s += KS;
    if (s >= p.steps) {
      r += cnt;
      start_pass(p, ks);
    }
  }
};

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

template <int LPR, int KS, bool PERM>
__global__ void __launch_bounds__(kGemvThreads, kGemvMinCtasPerSm)
    nvfp4_gemv_async_kernel(const GemvParams p) {
  constexpr int NI = kAsyncItems;          // row items per lane per task
  constexpr int RI = 32 / LPR;             // rows per warp-wide item
  constexpr int NR = NI * RI;              // rows per pass
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

  // copy this lane's part of task t (A chunks and scale words of its rows)
  auto issue = [&](const TaskCursor<NR>& t, int slot) {
    const int kt = t.s * LPR + kc;
    if (kt >= p.kchunks) return;
    const uint32_t a_dst = ring + (uint32_t)(slot * kAsyncStageBytes + lane * 32);
    const uint32_t s_dst = ring + (uint32_t)(slot * kAsyncStageBytes + SFA_OFF + lane * 16);
    const int64_t rp0 = t.r - t.l * p.rows_per_l;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int rho = i * RI + sub;
      if (rho < t.cnt) {
        const int64_t m = async_row<PERM, RI>(rp0 + rho);
        if (m < p.M) {
          const uint8_t* src = p.a + (t.l * p.M + m) * p.half_k + (int64_t)kt * 32;
          cp_async_16(a_dst + i * 1024, src);
          cp_async_16(a_dst + i * 1024 + 16, src + 16);
          if (!PERM) cp_async_4(s_dst + i * 4, p.sfa + (t.l * p.M + m) * p.blocks + kt * 4);
        }
      }
    }
    if (PERM) {
      // rows g = 0..3 of this lane: one 16-byte run of the atom (padding rows
      // of the last block are in the atom too and read as 0x00)
      const int64_t m0 = async_row<PERM, RI>(rp0 + sub);
      cp_async_16(s_dst, p.sfa + ((t.l * p.rest_m + (m0 >> 7)) * p.rest_k + kt) * 512 +
                             (m0 & 31) * 16);
    }
  };
  auto load_b = [&](const TaskCursor<NR>& t, uint32_t (&w)[8], uint32_t& sw) {
    const int kt = t.s * LPR + kc;
    if (kt < p.kchunks) {
      ld_shared_256(p.b + t.l * p.half_k + (int64_t)kt * 32, w);
      sw = ld_scale_32(p.sfb + (PERM ? (t.l * p.rest_k + kt) * 512 : t.l * p.blocks + kt * 4));
    }
  };

  TaskCursor<NR> ld, cp;
  ld.init(p, r_begin, r_end, ks);
  cp = ld;
#pragma unroll
  for (int j = 0; j < S - 1; ++j) {
    if (!ld.done) {
      issue(ld, j);
      ld.advance(p, ks, KS);
    }
    cp_async_commit();
  }
  uint32_t bw_n[8] = {0, 0, 0, 0, 0, 0, 0, 0}, sbw_n = 0;
  if (!cp.done) load_b(cp, bw_n, sbw_n);

  float acc[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) acc[i] = 0.f;
  int slot = 0;

  while (!cp.done) {
    // the slot computed in the previous iteration is free again
    if (!ld.done) {
      issue(ld, (slot + S - 1) % S);
      ld.advance(p, ks, KS);
    }
    cp_async_commit();
    uint32_t bw[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) bw[j] = bw_n[j];
    const uint32_t sbw = sbw_n;
    TaskCursor<NR> nxt = cp;
    nxt.advance(p, ks, KS);
    if (!nxt.done) load_b(nxt, bw_n, sbw_n);
    cp_async_wait<S - 1>();

    const int kt = cp.s * LPR + kc;
    const int64_t rp0 = cp.r - cp.l * p.rows_per_l;
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
      bool valid[NI];
      uint32_t saw[NI];
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int rho = i * RI + sub;
        valid[i] = rho < cp.cnt && async_row<PERM, RI>(rp0 + rho) < p.M;
        saw[i] = __funnelshift_l(sws[i], sws[i], rot16);
      }
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
          if (valid[i]) {
            const uint4 x = *reinterpret_cast<const uint4*>(a_slot + i * 1024 + ((j * 16) ^ h0));
            const uint32_t sa2 = e4m3x2_to_f16x2(saw[i] >> (16 * j));
            acc[i] = block_accumulate<false>(block_dot(x.x, x.y, bh0), sa2, sb0, acc[i]);
            acc[i] = block_accumulate<true>(block_dot(x.z, x.w, bh1), sa2, sb1, acc[i]);
          }
        }
      }
    }

    const bool pass_end = nxt.done || nxt.r != cp.r;
    if (pass_end) {
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
      if ((KS == 1 || ks == 0) && holder && rho_out < cp.cnt) {
        const int64_t m = async_row<PERM, RI>(rp0 + rho_out);
        if (m < p.M) p.c[cp.l * p.M + m] = __half_as_ushort(__float2half_rn(v));
      }
#pragma unroll
      for (int i = 0; i < NI; ++i) acc[i] = 0.f;
    }
    cp = nxt;
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

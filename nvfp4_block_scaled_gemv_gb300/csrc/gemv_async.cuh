// NVFP4 block-scaled batched GEMV, per-warp cp.async pipelined kernel (sm_103a).
//
// Same arithmetic as the direct kernel (gemv_kernel.cuh): LPR lanes per row,
// 32-byte K chunks per lane, exact half2 block dots, fp32 block scaling, a
// shuffle butterfly over the lanes of a row and a fixed-order shared-memory
// sum over the KS warps that split a row's K range.  What differs is how A
// reaches the registers and how a warp orders its work:
//
//   * A row lane's rows are cut into passes of up to G groups of NR rows,
//     never crossing a batch.  A pass runs the warp's K steps outermost and
//     its groups innermost; one task = one group at one K step (kAsyncItems
//     row items per lane).  The lane's chunk of b is decoded once per K step
//     and serves every group, and the partial sums are reduced and stored
//     once per pass.
//   * Each lane copies its own A chunks and scale words of a task into a
//     per-warp ring of kAsyncStages shared-memory slots with cp.async and
//     waits for them with its own wait_group: a lane only ever reads bytes it
//     copied, so there is no cross-lane synchronisation and no spin-wait.
//   * The warp keeps kAsyncStages - 1 tasks in flight while it computes one.
//     The loader runs that far ahead of the compute and hands it, per task,
//     the mask of items it copied.
//   * The next K step's b words are loaded while the current step computes
//     and decoded when that step begins.
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

// The (K step, group) tasks of one warp.  A row lane's range is cut into
// passes of up to G groups of NR = NI*RI rows, a pass never crossing a batch;
// inside a pass the warp's K steps ks, ks + KS, ... (below p.steps; the
// planner keeps KS <= steps, so every pass has one) run outermost and the
// groups innermost, so one decoded chunk of b serves every group of the pass
// and the partial sums are reduced and stored once per pass.  The cursor is
// pure bookkeeping: the loader turns a task into addresses when it issues it.
template <int LPR, int G>
struct TaskCursor {
  static constexpr int NI = kAsyncItems, RI = 32 / LPR, NR = NI * RI;
  int64_t r, end;         // first visit-order row of the pass, end of the range
  int64_t l_begin, l_end; // visit rows of the pass's batch
  int l;                  // the pass's batch
  int cnt;                // rows in the pass, at most G*NR
  int ng;                 // groups in the pass, ceil(cnt / NR)
  int s, g;               // the task: K step and group
  bool done;

  __device__ __forceinline__ void start_pass(const GemvParams& p, int ks) {
    done = r >= end;
    if (done) return;
    if (r >= l_end) {  // passes never cross a batch, and advance by at most one
      ++l;
      l_begin = l_end;
      l_end += p.rows_per_l;
    }
    const int64_t left = min(end, l_end) - r;
    cnt = left < G * NR ? (int)left : G * NR;
    ng = (cnt + NR - 1) / NR;
    s = ks;
    g = 0;
  }
  __device__ __forceinline__ void init(const GemvParams& p, int64_t begin, int64_t e, int ks) {
    r = begin;
    end = e;
    l = begin < e ? batch_of(p, begin) : 0;
    l_begin = (int64_t)l * p.rows_per_l;
    l_end = l_begin + p.rows_per_l;
    start_pass(p, ks);
  }
  __device__ __forceinline__ void advance(const GemvParams& p, int ks, int KS) {
    if (++g < ng) return;
    g = 0;
    s += KS;
    if (s >= p.steps) {
      r += cnt;
      start_pass(p, ks);
    }
  }
};

// Which of a lane's NI items (rows first + i*RI of the pass, first = the
// lane's offset inside the pass) are real rows.  m0 is the row of item 0;
// permuted item i is row m0 + 32*i, and rows past M are atom padding.
template <int LPR, bool PERM>
__device__ __forceinline__ uint32_t item_mask(int first, int cnt, int64_t m0, int64_t M) {
  constexpr int NI = kAsyncItems, RI = 32 / LPR;
  uint32_t v = 0;
#pragma unroll
  for (int i = 0; i < NI; ++i)
    if (first + i * RI < cnt && (!PERM || m0 + 32 * i < M)) v |= 1u << i;
  return v;
}

template <int LPR, int KS, bool PERM, int G>
__global__ void __launch_bounds__(kGemvThreads, kGemvMinCtasPerSm)
    nvfp4_gemv_async_kernel(const GemvParams p) {
  using Cursor = TaskCursor<LPR, G>;
  constexpr int NI = Cursor::NI;           // row items per lane per task
  constexpr int RI = Cursor::RI;           // rows per warp-wide item
  constexpr int NR = Cursor::NR;           // rows per group
  constexpr int WR = kGemvWarps / KS;      // row lanes per CTA
  constexpr int S = kAsyncStages;
  constexpr int SFA_OFF = NI * 1024;       // scale words ([lane][item] words) follow the A chunks
  static_assert(LPR >= NI && LPR <= 32 && (LPR & (LPR - 1)) == 0, "LPR in {4,8,16,32}");
  static_assert(KS >= 1 && KS <= kGemvWarps && (kGemvWarps % KS) == 0, "KS divides the warps per CTA");
  static_assert(G == 1 || G == 2 || G == 4, "G in {1,2,4}");
  extern __shared__ __align__(128) uint8_t ring_smem[];
  __shared__ float red[KS > 1 ? WR : 1][KS][KS > 1 ? G * NR : 1];

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
  constexpr int64_t unit = PERM ? NR : 1;
  int64_t r_begin, r_end;
  row_lane_units<WR>(p, wr, r_begin, r_end);
  r_begin *= unit;
  r_end *= unit;

  const int64_t a_step = (int64_t)(PERM ? 32 : RI) * p.half_k;  // item i -> i+1 of A
  const int64_t s_step = (int64_t)RI * p.blocks;                // same for plain scales
  const int64_t a_group = (int64_t)NR * p.half_k;               // plain: group g -> g+1
  const int64_t s_group = (int64_t)NR * p.blocks;

  const uint64_t a_pol = l2_evict_first_policy();
  // plain: the lane's item-0 row of A and of the scales in group 0 of the
  // loader's current pass (recomputed when the pass changes)
  int64_t base_r = -1;
  const uint8_t* a_pass = p.a;
  const uint8_t* s_pass = p.sfa;

  // Copy this lane's part of task t (A chunks and scale words of its items);
  // returns which items were copied (none when the lane's K chunk is past K).
  auto issue = [&](const Cursor& t, int slot) -> uint32_t {
    const int kt = t.s * LPR + kc;
    if (kt >= p.kchunks) return 0u;
    const uint32_t a_dst = ring + (uint32_t)(slot * kAsyncStageBytes + lane * 32);
    const uint32_t s_dst = ring + (uint32_t)(slot * kAsyncStageBytes + SFA_OFF + lane * 16);
    const uint8_t* a_src;
    const uint8_t* s_src;
    int64_t m0 = 0;
    if (!PERM) {
      if (t.r != base_r) {
        base_r = t.r;
        const int64_t row = (int64_t)t.l * p.M + (t.r - t.l_begin) + sub;
        a_pass = p.a + row * p.half_k;
        s_pass = p.sfa + row * p.blocks;
      }
      a_src = a_pass + t.g * a_group + kt * 32;
      s_src = s_pass + t.g * s_group + kt * 4;
    } else {
      m0 = async_row<true, RI>(t.r - t.l_begin + t.g * NR + sub);
      a_src = p.a + ((int64_t)t.l * p.M + m0) * p.half_k + kt * 32;
      // the four rows m0 + 32*i of this lane are one 16-byte run of the atom
      // (padding rows of the last block included, read as 0x00)
      s_src = p.sfa + (((int64_t)t.l * p.rest_m + (m0 >> 7)) * p.rest_k + kt) * 512 +
              (m0 & 31) * 16;
    }
    const uint32_t valid = item_mask<LPR, PERM>(t.g * NR + sub, t.cnt, m0, p.M);
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      if (valid & (1u << i)) {
        cp_async_16_ef(a_dst + i * 1024, a_src + i * a_step, a_pol);
        cp_async_16_ef(a_dst + i * 1024 + 16, a_src + i * a_step + 16, a_pol);
        if (!PERM) cp_async_4(s_dst + i * 4, s_src + i * s_step);
      }
    }
    if (PERM) cp_async_16(s_dst, s_src);
    return valid;
  };
  // Ask the L2 for the A lines of task t (used before the dependency wait:
  // the L2 is coherent, so the copies issued after the wait still read what
  // earlier work on the stream wrote; the prefetch only starts the DRAM
  // traffic while that work finishes).
  auto prefetch_task = [&](const Cursor& t) {
    const int kt = t.s * LPR + kc;
    if (kt >= p.kchunks) return;
    int64_t m0 = 0, row;
    if (!PERM) {
      row = (int64_t)t.l * p.M + (t.r - t.l_begin) + t.g * NR + sub;
    } else {
      m0 = async_row<true, RI>(t.r - t.l_begin + t.g * NR + sub);
      row = (int64_t)t.l * p.M + m0;
    }
    const uint8_t* a_src = p.a + row * p.half_k + kt * 32;
    const uint32_t valid = item_mask<LPR, PERM>(t.g * NR + sub, t.cnt, m0, p.M);
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (valid & (1u << i)) prefetch_l2(a_src + i * a_step);
  };
  auto load_b = [&](int l, int kt, uint32_t (&w)[8], uint32_t& sw) {
    if (kt < p.kchunks) {
      ld_shared_2x128(p.b + (int64_t)l * p.b_stride + kt * 32, w);
      sw = ld_scale_32(p.sfb + (int64_t)l * p.sfb_stride + (PERM ? (int64_t)kt * 512 : kt * 4));
    }
  };

  Cursor ld, cp;
  ld.init(p, r_begin, r_end, ks);
  cp = ld;
  {
    Cursor pf = ld;
    for (int j = 0; j < S - 1 && j < p.prefetch_tasks && !pf.done; ++j) {
      prefetch_task(pf);
      pf.advance(p, ks, KS);
    }
  }
  pdl_wait();
  // b (and sfb) words of the next K step whose chunk differs from the one
  // decoded (the first one requested ahead of the A stream); decoded: the
  // lane's four blocks in its half-swapped order
  uint32_t bw_n[8] = {0, 0, 0, 0, 0, 0, 0, 0}, sbw_n = 0;
  bool b_pending = false;
  if (!cp.done) {
    load_b(cp.l, cp.s * LPR + kc, bw_n, sbw_n);
    b_pending = true;
  }
  // items copied per task in flight, oldest first (the slot order)
  uint32_t mq[S];
#pragma unroll
  for (int j = 0; j < S; ++j) mq[j] = 0u;
#pragma unroll
  for (int j = 0; j < S - 1; ++j) {
    if (!ld.done) {
      mq[j] = issue(ld, j);
      ld.advance(p, ks, KS);
    }
    cp_async_commit();
  }
  uint32_t bh[4][8];
  float sb[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    sb[q] = 0.f;
#pragma unroll
    for (int t = 0; t < 8; ++t) bh[q][t] = 0;
  }

  float acc[G][NI];
#pragma unroll
  for (int gg = 0; gg < G; ++gg)
#pragma unroll
    for (int i = 0; i < NI; ++i) acc[gg][i] = 0.f;
  int slot = 0;

  while (!cp.done) {
    // the slot computed in the previous iteration is free again; refill it
    // first, so the copies never queue behind a wait for b
    mq[S - 1] = 0u;
    if (!ld.done) {
      mq[S - 1] = issue(ld, (slot + S - 1) % S);
      ld.advance(p, ks, KS);
    }
    cp_async_commit();
    const bool last_step = cp.s + KS >= p.steps;
    if (cp.g == 0) {
      if (b_pending) {
        // the chunk loaded during the previous step is decoded only now, so
        // its load latency hides behind a whole step's compute
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t w0 = swp ? bw_n[(2 * q + 4) & 7] : bw_n[2 * q];
          const uint32_t w1 = swp ? bw_n[(2 * q + 5) & 7] : bw_n[2 * q + 1];
          uint32_t d[4];
          e2m1x8_to_f16x2x4(w0, d);
#pragma unroll
          for (int t = 0; t < 4; ++t) bh[q][t] = d[t];
          e2m1x8_to_f16x2x4(w1, d);
#pragma unroll
          for (int t = 0; t < 4; ++t) bh[q][4 + t] = d[t];
        }
        const uint32_t sbwr = __funnelshift_l(sbw_n, sbw_n, rot16);
#pragma unroll
        for (int q = 0; q < 4; ++q) sb[q] = scale_of(sbwr, q);
        b_pending = false;
      }
      // the next step's chunk: the same pass's next step, else the first step
      // of the next pass (whose batch may be the next one)
      const bool more = !last_step || cp.r + cp.cnt < cp.end;
      const int s_n = last_step ? ks : cp.s + KS;
      const int l_n = (last_step && cp.r + cp.cnt >= cp.l_end) ? cp.l + 1 : cp.l;
      if (more && (s_n != cp.s || l_n != cp.l)) {
        load_b(l_n, s_n * LPR + kc, bw_n, sbw_n);
        b_pending = true;
      }
    }
    cp_async_wait<S - 1>();

    const uint32_t valid = mq[0];
    // whole tasks (every lane, every item) take a branch-free path, so the
    // items' independent dependency chains can interleave
    const bool full = __all_sync(0xffffffffu, valid == (1u << NI) - 1u);
    if (valid != 0u) {
      // Lanes with bit 2 set process the chunk's second 16-byte half (blocks
      // 2, 3) first; their b blocks and scale bytes are rotated to match, so
      // the block order inside registers stays static.
      const uint8_t* a_slot = ring_gen + slot * kAsyncStageBytes + lane * 32;
      const uint4 sw4 =
          *reinterpret_cast<const uint4*>(ring_gen + slot * kAsyncStageBytes + SFA_OFF + lane * 16);
      const uint32_t sws[4] = {sw4.x, sw4.y, sw4.z, sw4.w};
      uint32_t saw[NI];
#pragma unroll
      for (int i = 0; i < NI; ++i) saw[i] = __funnelshift_l(sws[i], sws[i], rot16);
      auto item = [&](float& a, int i, int j) {
        const uint4 x = *reinterpret_cast<const uint4*>(a_slot + i * 1024 + ((j * 16) ^ h0));
        const uint32_t sa2 =
            j ? e4m3x2_half_to_f16x2<true>(saw[i]) : e4m3x2_half_to_f16x2<false>(saw[i]);
        a = block_accumulate<false>(block_dot(x.x, x.y, bh[2 * j]), sa2, sb[2 * j], a);
        a = block_accumulate<true>(block_dot(x.z, x.w, bh[2 * j + 1]), sa2, sb[2 * j + 1], a);
      };
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        if (gg != cp.g) continue;
        if (full) {
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int i = 0; i < NI; ++i) item(acc[gg][i], i, j);
        } else {
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int i = 0; i < NI; ++i)
              if (valid & (1u << i)) item(acc[gg][i], i, j);
        }
      }
    }

    if (last_step && cp.g == cp.ng - 1) {
      // end of the pass: every group's rows are complete in this warp
      const int rho_out = (kc / (LPR / NI)) * RI + sub;
      const bool holder = (kc % (LPR / NI)) == 0;
      float v[G];
#pragma unroll
      for (int gg = 0; gg < G; ++gg)
        if (gg < cp.ng) v[gg] = lane_reduce<NI, LPR / 2>(acc[gg], lane);
      if constexpr (KS > 1) {
        if (holder) {
#pragma unroll
          for (int gg = 0; gg < G; ++gg)
            if (gg < cp.ng) red[wr][ks][gg * NR + rho_out] = v[gg];
        }
        named_barrier_sync(1 + wr, 32 * KS);
        if (ks == 0 && holder) {
#pragma unroll
          for (int gg = 0; gg < G; ++gg) {
            if (gg < cp.ng) {
              float t = red[wr][0][gg * NR + rho_out];
#pragma unroll
              for (int j = 1; j < KS; ++j) t += red[wr][j][gg * NR + rho_out];
              v[gg] = t;
            }
          }
        }
        named_barrier_sync(1 + wr, 32 * KS);
      }
      if ((KS == 1 || ks == 0) && holder) {
        const int64_t rp = cp.r - cp.l_begin;
        const int64_t lm = (int64_t)cp.l * p.M;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          if (gg < cp.ng && gg * NR + rho_out < cp.cnt) {
            const int64_t m = PERM ? async_row<true, RI>(rp + gg * NR + rho_out)
                                   : rp + gg * NR + rho_out;
            if (!PERM || m < p.M) p.c[lm + m] = finish_output(p, v[gg], lm + m);
          }
        }
      }
#pragma unroll
      for (int gg = 0; gg < G; ++gg)
#pragma unroll
        for (int i = 0; i < NI; ++i) acc[gg][i] = 0.f;
    }
    cp.advance(p, ks, KS);
    slot = (slot + 1 == S) ? 0 : slot + 1;
#pragma unroll
    for (int j = 0; j + 1 < S; ++j) mq[j] = mq[j + 1];
  }
  cp_async_wait<0>();
}

template <bool PERM>
cudaError_t launch_async_layout(const GemvParams& p, const GemvPlan& plan, cudaStream_t stream) {
  void (*kern)(GemvParams) = nullptr;
#define NVFP4_CASE(LPR_, KS_, G_)                                             \
  if (plan.lanes_per_row == LPR_ && plan.k_split == KS_ && plan.groups == G_) \
    kern = nvfp4_gemv_async_kernel<LPR_, KS_, PERM, G_>;
#define NVFP4_CASES_G(LPR_, KS_) NVFP4_CASE(LPR_, KS_, 1) NVFP4_CASE(LPR_, KS_, 2) NVFP4_CASE(LPR_, KS_, 4)
#define NVFP4_CASES_KS(LPR_) \
  NVFP4_CASES_G(LPR_, 1) NVFP4_CASES_G(LPR_, 2) NVFP4_CASES_G(LPR_, 4) NVFP4_CASES_G(LPR_, 8)
  NVFP4_CASES_KS(4)
  NVFP4_CASES_KS(8)
  NVFP4_CASES_KS(16)
  NVFP4_CASES_KS(32)
#undef NVFP4_CASES_KS
#undef NVFP4_CASES_G
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

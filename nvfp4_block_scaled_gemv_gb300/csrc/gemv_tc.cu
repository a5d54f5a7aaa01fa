// NVFP4 block-scaled batched GEMV on the tensor cores (tcgen05, sm_103a),
// pre-permuted scales only.
//
// The hardware block-scaled MMA (kind::mxf4nvf4, 16-element blocks with E4M3
// scales, scale_vec::4X) computes, for a 128-row tile of A and an N = 16 row
// operand B, D[m][n] += sum_k E2M1(a[m][k]) * sfa[m][k/16] * E2M1(b[n][k]) *
// sfb[n][k/16] over K = 64 per instruction, accumulating in fp32 in tensor
// memory (TMEM).  The GEMV puts b in row 0 of B (rows 1..15 are zeros) and
// keeps column 0 of D.  The 128x4 scale atom of the pre-permuted layout is
// byte for byte the source the 32x128b.warpx4 TMEM copy expects, so one atom
// (512 B) feeds one MMA's scales with no repacking.
//
// One CTA (192 threads):
//   warp 0      one lane issues the copies of each stage: A as a 128-row x
//               128-byte TMA tile (128-byte swizzle), b's 128-byte chunk as a
//               1-row TMA tile, and the stage's 4 sfa atoms and 4 sfb atoms as
//               two 2 KB bulk copies (consecutive atoms are adjacent in memory);
//   warp 1      allocates TMEM; one lane copies each stage's scale atoms into
//               TMEM (tcgen05.cp) and issues the stage's 4 MMAs, then commits
//               the stage back to the producer and, at the end of a tile, the
//               accumulator to the epilogue;
//   warps 2..5  read the accumulator (one TMEM lane quarter each), and either
//               store c or send the partial sums to the cluster's rank 0.
// Split K: the KS CTAs of a cluster share every tile, each taking a
// contiguous range of 256-element K stages (the rank that takes an extra
// stage rotates from tile to tile); ranks 1..KS-1 store their partial sums
// into rank 0's shared memory (distributed shared memory) and rank 0 adds
// them in rank order, so the result does not depend on timing.
// Clusters are persistent: cluster i takes tiles i, i + clusters, ...
//
// Every wait on an mbarrier gives up after kWaitNs of global time, counts a
// timeout in a device word the host can read, and the thread then skips its
// remaining work; control flow stays uniform so every thread reaches the
// cluster barriers and TMEM is always freed.
#include <cstdint>
#include <cstring>

#include <cuda.h>  // CUtensorMap (the type only; the encoder is looked up at run time)
#include <cudaTypedefs.h>

#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

__device__ int g_tc_timeouts;

namespace {

constexpr int kTcThreads = 192;
constexpr int kTcStages = 6;
constexpr int kTcMaxCluster = 8;
constexpr uint32_t kTcABytes = 128 * 128;   // 128 rows x 256 elements
constexpr uint32_t kTcBBytes = 16 * 128;    // 16 rows x 256 elements (row 0 = b)
constexpr uint32_t kTcSfBytes = 4 * 512;    // 4 scale atoms (K = 256)
constexpr uint32_t kTcStageBytes = kTcABytes + kTcBBytes + 2 * kTcSfBytes;
constexpr uint32_t kTcRedBytes = 2 * kTcMaxCluster * 128 * 4;
constexpr uint32_t kTcSmemBytes = kTcStages * kTcStageBytes + kTcRedBytes + 1024;
constexpr uint32_t kTmemCols = 256;
// TMEM columns: accumulators [2][16] at 0, sfa [stage][4 atoms][4 cols] at 32,
// sfb likewise after them
constexpr uint32_t kTmemSfa = 32;
constexpr uint32_t kTmemSfb = kTmemSfa + kTcStages * 16;
static_assert(kTmemSfb + kTcStages * 16 <= kTmemCols, "TMEM columns");
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s

// Instruction descriptor of the block-scaled MMA: A and B E2M1 (format 1),
// both K-major, N = 16 (N/8 at bit 17), UE4M3 scales (bit 23 clear),
// M = 128 (M/16 at bit 24), scale ids 0, dense K = 64.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

struct TcParams {
  CUtensorMap tmap_a;  // uint8 {K/2, M, L}, box {128, 128, 1}, 128-byte swizzle
  CUtensorMap tmap_b;  // uint8 {K/2, L}, box {128, 1}, 128-byte swizzle
  const uint8_t* sfa;  // permuted [L][rest_m][rest_k][512]
  const uint8_t* sfb;  // permuted, one 128-row block per batch: [L][rest_k][512] (stride below)
  uint16_t* c;
  const uint16_t* bias;
  float alpha;
  int64_t M;
  int64_t sfb_stride;
  int32_t rest_m, rest_k, kstages, tiles;
};

// fp32 -> fp16 output with the optional scale and bias: the same formula as
// the CUDA-core kernels' epilogue.
__device__ __forceinline__ uint16_t finish_output_tc(float alpha, const uint16_t* bias, float v,
                                                     int64_t idx) {
  const float o = bias ? fmaf(v, alpha, __half2float(__ushort_as_half(bias[idx]))) : v * alpha;
  return __half_as_ushort(__float2half_rn(o));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Acquire at cluster scope: the phase was completed by arrivals from other
// CTAs of the cluster whose prior shared-memory stores must be visible.
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;"
      "\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase of the given parity; false (and ok cleared, one
// timeout counted) if it did not complete within kWaitNs, or if ok was
// already clear.
template <bool CLUSTER>
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, bool& ok) {
  if (!ok) return false;
  if (CLUSTER ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (CLUSTER ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
    if ((i & 255u) == 0 && global_ns() - t0 > kWaitNs) {
      atomicAdd(&g_tc_timeouts, 1);
      ok = false;
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// The same shared-memory offset in the CTA of the given cluster rank.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ void st_remote_f32(uint32_t cluster_addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptors (64-bit): start address >> 4 in bits
// 0-13, leading byte offset >> 4 in 16-29, stride byte offset >> 4 in
// 32-45, descriptor version 1 in 46-47, layout in 61-63.
// K-major operand tile in the 128-byte swizzled layout the TMA writes: rows
// of 128 bytes, 8-row groups 1024 bytes apart; the K step inside the swizzle
// span moves the start address by 32 bytes.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// A scale atom as the 32 x 128-bit copy source: 32 rows of 16 bytes, no
// swizzle, 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t desc_atom(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_copy_atom(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t sfa,
                                       uint32_t sfb, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"((uint32_t)accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}
// Arrive on the mbarrier once every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1)
    nvfp4_gemv_tc_kernel(const __grid_constant__ TcParams p) {
  constexpr int S = kTcStages;
  extern __shared__ uint8_t tc_smem[];
  __shared__ __align__(8) uint64_t bars[2 * S + 9];
  __shared__ uint32_t tmem_slot;

  const uint32_t raw = smem_u32(tc_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzled tiles want 1024-byte alignment
  const uint32_t a_s = base;
  const uint32_t b_s = a_s + S * kTcABytes;
  const uint32_t sfa_s = b_s + S * kTcBBytes;
  const uint32_t sfb_s = sfa_s + S * kTcSfBytes;
  const uint32_t red_s = sfb_s + S * kTcSfBytes;
  const float* red = reinterpret_cast<const float*>(tc_smem + (red_s - raw));
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int st) { return bar0 + 8u * st; };
  auto empty_bar = [&](int st) { return bar0 + 8u * (S + st); };
  const uint32_t dfull_bar = bar0 + 8u * (2 * S);       // [2]
  const uint32_t dempty_bar = bar0 + 8u * (2 * S + 2);  // [2]
  const uint32_t rfull_bar = bar0 + 8u * (2 * S + 4);   // [2] (rank 0)
  const uint32_t rfree_bar = bar0 + 8u * (2 * S + 6);   // [2] (ranks > 0)
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ks = cluster_size(), rank = cluster_rank();
  const int cid = (int)(blockIdx.x / ks), nclusters = (int)(gridDim.x / ks);
  const int ntiles = cid < p.tiles ? (p.tiles - cid + nclusters - 1) / nclusters : 0;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int st = 0; st < S; ++st) {
      mbar_init(full_bar(st), 1);
      mbar_init(empty_bar(st), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(dfull_bar + 8u * i, 1);
      mbar_init(dempty_bar + 8u * i, 128);
      mbar_init(rfull_bar + 8u * i, ks > 1 ? (ks - 1) * 128 : 1);
      mbar_init(rfree_bar + 8u * i, 128);
    }
    mbar_init(drain_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // rows 1..15 of every B stage stay zero (the b copy writes row 0 only)
  for (uint32_t i = threadIdx.x; i < S * kTcBBytes / 16; i += kTcThreads) {
    if ((i % (kTcBBytes / 16)) >= 128 / 16)
      *reinterpret_cast<uint4*>(tc_smem + (b_s - raw) + 16 * i) = make_uint4(0, 0, 0, 0);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every CTA's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;

  // The contiguous K-stage range of this rank for the cluster's j-th tile.
  auto stage_range = [&](int j, int& s0, int& cnt) {
    const int per = p.kstages / (int)ks, extra = p.kstages % (int)ks;
    const int rr = (int)((rank + (uint32_t)j) % ks);
    cnt = per + (rr < extra ? 1 : 0);
    s0 = rr * per + (rr < extra ? rr : extra);
  };

  if (warp == 0) {
    int issued = 0;
    if (lane == 0) {
      if (ntiles > 0) {  // the first stages' A lines, ahead of the dependency wait
        int s0, cnt;
        stage_range(0, s0, cnt);
        const int l = cid / p.rest_m, mt = cid % p.rest_m;
        for (int i = 0; i < cnt && i < S; ++i) tma_prefetch_3d(&p.tmap_a, (s0 + i) * 128, mt * 128, l);
      }
      pdl_wait();
      int st = 0;
      uint32_t ph = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int t = cid + j * nclusters;
        const int l = t / p.rest_m, mt = t % p.rest_m;
        int s0, cnt;
        stage_range(j, s0, cnt);
        for (int i = 0; i < cnt; ++i) {
          const int s = s0 + i;
          const int nk = min(4, p.rest_k - 4 * s);
          if (mbar_wait<false>(empty_bar(st), ph ^ 1u, ok)) {
            const uint32_t fb = full_bar(st);
            mbar_expect_tx(fb, kTcABytes + 128u + 2u * (uint32_t)nk * 512u);
            tma_load_3d(a_s + st * kTcABytes, &p.tmap_a, s * 128, mt * 128, l, fb);
            tma_load_2d(b_s + st * kTcBBytes, &p.tmap_b, s * 128, l, fb);
            bulk_load(sfa_s + st * kTcSfBytes,
                      p.sfa + (((int64_t)l * p.rest_m + mt) * p.rest_k + 4 * s) * 512,
                      (uint32_t)nk * 512u, fb);
            bulk_load(sfb_s + st * kTcSfBytes, p.sfb + (int64_t)l * p.sfb_stride + (int64_t)s * 2048,
                      (uint32_t)nk * 512u, fb);
            ++issued;
          }
          if (++st == S) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      // copies still in flight land before the CTA can exit: the last phase
      // issued on each stage (a phase already consumed passes at once)
      bool drain_ok = true;
      for (int k = 0; k < S && k < issued; ++k) {
        const int i_last = issued - 1 - k;
        mbar_wait<false>(full_bar(i_last % S), (uint32_t)((i_last / S) & 1), drain_ok);
      }
    } else {
      pdl_wait();
    }
  } else if (warp == 1) {
    pdl_wait();
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int acc = j & 1;
        const uint32_t d = tmem + (uint32_t)(16 * acc);
        mbar_wait<false>(dempty_bar + 8u * acc, ((uint32_t)(j >> 1) & 1u) ^ 1u, ok);
        tc_fence_after();
        int s0, cnt;
        stage_range(j, s0, cnt);
        for (int i = 0; i < cnt; ++i) {
          const int s = s0 + i;
          const int nk = min(4, p.rest_k - 4 * s);
          if (mbar_wait<false>(full_bar(st), ph, ok)) {
            tc_fence_after();
            for (int kk = 0; kk < nk; ++kk) {
              tc_copy_atom(tmem + kTmemSfa + (uint32_t)(16 * st + 4 * kk),
                           desc_atom(sfa_s + st * kTcSfBytes + 512u * kk));
              tc_copy_atom(tmem + kTmemSfb + (uint32_t)(16 * st + 4 * kk),
                           desc_atom(sfb_s + st * kTcSfBytes + 512u * kk));
            }
            for (int kk = 0; kk < nk; ++kk)
              tc_mma(d, desc_sw128(a_s + st * kTcABytes + 32u * kk),
                     desc_sw128(b_s + st * kTcBBytes + 32u * kk),
                     tmem + kTmemSfa + (uint32_t)(16 * st + 4 * kk),
                     tmem + kTmemSfb + (uint32_t)(16 * st + 4 * kk), i > 0 || kk > 0);
            tc_commit(empty_bar(st));
          }
          if (++st == S) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (ok) tc_commit(dfull_bar + 8u * acc);
      }
      // every MMA and TMEM copy has finished before TMEM is released
      tc_commit(drain_bar);
      bool drain_ok = true;
      mbar_wait<false>(drain_bar, 0, drain_ok);
    }
    __syncwarp();
  } else {
    pdl_wait();
    const uint32_t q = (uint32_t)(warp & 3);  // the TMEM lane quarter this warp may read
    const int r = (int)(32 * q) + lane;       // row inside the tile
    for (int j = 0; j < ntiles; ++j) {
      const int t = cid + j * nclusters;
      const int l = t / p.rest_m, mt = t % p.rest_m;
      const int acc = j & 1;
      mbar_wait<false>(dfull_bar + 8u * acc, (uint32_t)(j >> 1) & 1u, ok);
      ok = __all_sync(0xffffffffu, ok);  // the TMEM load below is warp-collective
      float part = 0.f;
      if (ok) {
        tc_fence_after();
        uint32_t v;
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];"
                     : "=r"(v)
                     : "r"(tmem + (uint32_t)(16 * acc) + ((32u * q) << 16)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        part = __uint_as_float(v);
      }
      tc_fence_before();
      mbar_arrive(dempty_bar + 8u * acc);
      const int64_t m = (int64_t)mt * 128 + r;
      const int buf = j & 1;
      const uint32_t use = (uint32_t)(j >> 1);
      if (ks == 1) {
        if (ok && m < p.M) p.c[(int64_t)l * p.M + m] = finish_output_tc(p.alpha, p.bias, part, (int64_t)l * p.M + m);
      } else if (rank != 0) {
        // wait until rank 0 has read this buffer's previous use, then send
        mbar_wait<true>(rfree_bar + 8u * buf, (use & 1u) ^ 1u, ok);
        const uint32_t slot = red_s + 4u * (uint32_t)((buf * kTcMaxCluster + (int)rank) * 128 + r);
        st_remote_f32(map_rank(slot, 0), part);
        mbar_arrive_remote(map_rank(rfull_bar + 8u * buf, 0));
      } else {
        float sum = part;
        if (mbar_wait<true>(rfull_bar + 8u * buf, use & 1u, ok)) {
          for (uint32_t k = 1; k < ks; ++k) sum += red[(buf * kTcMaxCluster + (int)k) * 128 + r];
        }
        for (uint32_t k = 1; k < ks; ++k) mbar_arrive_remote(map_rank(rfree_bar + 8u * buf, k));
        if (ok && m < p.M) p.c[(int64_t)l * p.M + m] = finish_output_tc(p.alpha, p.bias, sum, (int64_t)l * p.M + m);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no peer still reads or signals this CTA's shared memory
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link
// against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

cudaError_t tc_launch_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[2], int ks,
                             int64_t ctas, cudaStream_t stream) {
  cudaError_t err = cudaFuncSetAttribute(nvfp4_gemv_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
  if (err != cudaSuccess) return err;
  cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = kTcSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemv_tc(const GemvParams& gp, int64_t L, int ks, int64_t ctas,
                           cudaStream_t stream) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  TcParams p;
  memset(&p, 0, sizeof(p));
  const cuuint64_t half_k = (cuuint64_t)gp.half_k;
  {
    const cuuint64_t dims[3] = {half_k, (cuuint64_t)gp.M, (cuuint64_t)L};
    const cuuint64_t strides[2] = {half_k, half_k * (cuuint64_t)gp.M};
    const cuuint32_t box[3] = {128, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&p.tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(gp.a), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {half_k, (cuuint64_t)L};
    const cuuint64_t strides[1] = {(cuuint64_t)gp.b_stride};
    const cuuint32_t box[2] = {128, 1};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&p.tmap_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(gp.b), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  p.sfa = gp.sfa;
  p.sfb = gp.sfb;
  p.c = gp.c;
  p.bias = gp.bias;
  p.alpha = gp.alpha;
  p.M = gp.M;
  p.sfb_stride = gp.sfb_stride;
  p.rest_m = gp.rest_m;
  p.rest_k = gp.rest_k;
  p.kstages = (gp.rest_k + 3) / 4;
  p.tiles = (int32_t)(L * gp.rest_m);
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cudaError_t err = tc_launch_config(cfg, attr, ks, ctas, stream);
  if (err != cudaSuccess) return err;
  return cudaLaunchKernelEx(&cfg, nvfp4_gemv_tc_kernel, p);
}

cudaError_t tc_max_active_clusters(int ks, int* out) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cudaError_t err = tc_launch_config(cfg, attr, ks, ks, nullptr);
  if (err != cudaSuccess) return err;
  cfg.numAttrs = 1;  // the cluster shape alone
  return cudaOccupancyMaxActiveClusters(out, nvfp4_gemv_tc_kernel, &cfg);
}

cudaError_t tc_wait_timeouts(int reset, int* out) {
  cudaError_t err = cudaMemcpyFromSymbol(out, g_tc_timeouts, sizeof(int));
  if (err != cudaSuccess || !reset) return err;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_tc_timeouts, &zero, sizeof(int));
}

}  // namespace nvfp4

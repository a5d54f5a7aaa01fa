// NVFP4 block-scaled batched GEMV and small-N GEMM on the tensor cores
// (tcgen05, sm_103a): pre-permuted scales, and plain scales for the GEMV.
//
// The hardware block-scaled MMA (kind::mxf4nvf4, 16-element blocks with E4M3
// scales, scale_vec::4X) computes, for a 128-row tile of A and an N = 16 row
// operand B, D[m][n] += sum_k E2M1(a[m][k]) * sfa[m][k/16] * E2M1(b[n][k]) *
// sfb[n][k/16] over K = 64 per instruction, accumulating in fp32 in tensor
// memory (TMEM).  Rows 0..N-1 of B hold the N <= 16 vectors (one for the
// GEMV), the other rows are zeros, and the epilogue reads columns 0..N-1 of
// D.  The 128x4 scale atom of the pre-permuted layout is byte for byte the
// source of one 32x128b.warpx4 TMEM copy, so the scales need no repacking:
// one sfa atom and one sfb atom (512 B each) feed one MMA.  (An MMA's scale
// address in TMEM is a 4-column-aligned copy destination.)  Plain scales (the
// GEMV, K % 256 == 0): a stage's 16 scale bytes of each of the tile's 128
// rows arrive as one TMA box, and the MMA warp writes them out as the stage's
// 4 atoms in shared memory before its TMEM copies (the atoms a repack would
// have made, so the result is the same bits); a TMA box cannot make the atom
// itself, whose 4-byte runs are narrower than a box's 16-byte minimum row.
//
// One CTA (224 threads):
//   warp 0      one lane issues the copies of each 256-element K stage: A as
//               a 128-row x 128-byte TMA tile (128-byte swizzle), b as an
//               N-row TMA tile, and the stage's 4 sfa atoms and 4 sfb atoms as
//               two 2 KB bulk copies (consecutive atoms are adjacent);
//   warps 1, 6  two independent MMA chains (warp 1 also allocates TMEM):
//               chain c takes the stages i with i % 2 == c of every tile,
//               through a ring of its own, into its own (double-buffered)
//               accumulator; one lane copies the stage's 8 atoms into TMEM
//               (tcgen05.cp) and issues its MMAs, then commits the stage back
//               to the producer and, at the end of a tile, the accumulator to
//               the epilogue;
//   warps 2..5  read and add the two accumulators (one TMEM lane quarter each),
//               and either store c or hand their partial sums to the cluster's
//               rank 0.
// The copies and MMAs of one chain complete one after another; a CTA has two
// chains of 1 or 2 stages each, and several CTAs share an SM, so independent
// chains overlap.
// Split K: the KS CTAs of a cluster share every tile, each taking a
// contiguous range of 256-element K stages (the rank that takes an extra
// stage rotates from tile to tile); ranks 1..KS-1 leave their partial sums
// in their own shared memory and rank 0 reads them (distributed shared
// memory) and adds them in rank order, so the result does not depend on
// timing or on the grid.
// Clusters are persistent: cluster i takes tiles i, i + clusters, ...
//
// Scale signs: the MMA reads each scale byte as an unsigned magnitude, so
// before a stage's MMAs the MMA warp folds every negative sfa or sfb code into
// the sign bits of the 16 E2M1 elements it scales (fold_scale_signs); a stage
// whose codes all have the sign bit clear (the benchmark's) costs that warp
// one vote over its scale bytes (any_negative_scale).
//
// Every wait on an mbarrier gives up after kWaitNs of global time, counts a
// timeout in a device word the host can read, and the thread then skips its
// remaining work; control flow stays uniform so every thread reaches the
// cluster barriers and TMEM is always freed.
#include <atomic>
#include <cstdint>
#include <cstring>

#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace nvfp4 {

__device__ int g_tc_timeouts;

namespace {

constexpr int kTcThreads = kTcThreadsPerCta;  // 7 warps
constexpr uint32_t kTcABytes = 128 * 128;   // 128 rows x 256 elements
constexpr uint32_t kTcBBytes = 16 * 128;    // 16 rows x 256 elements (rows 0..N-1 = b)
constexpr uint32_t kTcSfBytes = 4 * 512;    // 4 scale atoms (K = 256)

// TMEM columns a CTA allocates: accumulators [2 chains][2][16], then sfa and
// sfb [stage][4 atoms][4 columns] each (a power of two, at least 32).
__host__ __device__ constexpr uint32_t tc_tmem_cols(int stages) { return stages <= 2 ? 128u : 256u; }
// Plain scales also stage each K stage's sfa box ([128 rows][16 bytes]) and
// sfb bytes (16 of a 128-byte slot) before they are laid out as atoms.
constexpr uint32_t kTcPlainStageBytes = kTcSfBytes + 128;
constexpr uint32_t tc_smem_bytes(int stages, int nc, bool plain = false) {
  return (uint32_t)stages * (kTcABytes + kTcBBytes + 2 * kTcSfBytes) +
         2u * (uint32_t)nc * 128u * 4u + 1024u + (plain ? (uint32_t)stages * kTcPlainStageBytes : 0u);
}
static_assert(64 + 32 * 2 <= tc_tmem_cols(2) && 64 + 32 * 4 <= tc_tmem_cols(4), "TMEM columns");
// The SM's 512 TMEM columns are never oversubscribed, so an allocation never
// waits for another CTA: shared memory (228 KB per SM, 1 KB of it reserved
// per CTA) admits at most 4 CTAs of 2 stages (128 columns), at most 2 of 4
// stages (256), and 2-stage CTAs beside a 4-stage one at most 2.
static_assert(5 * (tc_smem_bytes(2, 1) + 1024) > 228 * 1024, "at most 4 CTAs of 2 stages");
static_assert(3 * (tc_smem_bytes(4, 1) + 1024) > 228 * 1024, "at most 2 CTAs of 4 stages");
static_assert((tc_smem_bytes(4, 1) + 1024) + 3 * (tc_smem_bytes(2, 1) + 1024) > 228 * 1024,
              "at most 2 CTAs of 2 stages beside one of 4");

// Instruction descriptor: N = 16 rows of B (see tc::mxf4nvf4_idesc).
constexpr uint32_t kIdesc = tc::mxf4nvf4_idesc(16);

struct TcParams {
  CUtensorMap tmap_a;  // uint8 {K/2, M, L}, box {128, 128, 1}, 128-byte swizzle
  CUtensorMap tmap_b;  // uint8 {K/2, N, L}, box {128, N, 1}, 128-byte swizzle
  CUtensorMap tmap_sfa;  // plain sfa (GEMV): uint8 {K/16, M, L}, box {16, 128, 1}
  CUtensorMap tmap_sfb;  // plain sfb (GEMV): uint8 {K/16, L} (batch stride sfb_stride), box {16, 1}
  const uint8_t* sfa;  // permuted [L][rest_m][rest_k][512]
  const uint8_t* sfb;  // permuted, one 128-row block per batch (rows 0..N-1): [L][rest_k][512]
  uint16_t* c;         // fp16 [L][N][M]
  const uint16_t* bias;  // fp16 [L][N][M], or null
  float alpha;
  int64_t M;
  int64_t sfb_stride;  // bytes from batch l to l+1 of sfb
  int32_t N, rest_m, rest_k, kstages, tiles;
  int32_t activation;  // nvfp4_activation_t
};

// A CTA's first K stages whose A lines are prefetched into the L2 before the
// dependency wait (the copies themselves wait for it).  Measured on GB300 with
// back-to-back calls: 2 beat 0, 4 and 8 (M7168_N8_K2048_L4 9.17 us against
// 10.18, 9.47 and 9.78; M4096_K7168_L8 23.6 against 24.2-24.0); each prefetch
// costs the producer lane about as much as a copy.
constexpr int kTcPrefetchStages = 2;


// The MMA reads each scale byte as an unsigned E4M3 magnitude (the sign bit
// is ignored).  A negative scale is folded into the operand it scales: for
// every scale byte of the stage with the sign bit set, the 16 E2M1 elements it
// scales (8 bytes of one row of the A tile, or of one vector's row of the B
// tile) get their sign bits flipped in shared memory, so the MMA's product
// |scale| * (-x) is the signed one (exact: E2M1 negation only flips a bit).
// A NaN code (0x7F, 0xFF) stays NaN either way.  The warp scans the stage's
// nk sfa and nk sfb atoms, 16 bytes per lane and step; returns whether any
// element was flipped (the caller then fences the writes for the tensor
// cores).  B rows past the tile's 16 are never written (their atom rows are
// padding).
static __device__ __noinline__ bool fold_scale_signs(uint8_t* gen, uint32_t a_tile, uint32_t b_tile,
                                                 uint32_t sfa_atoms, uint32_t sfb_atoms, int nk,
                                                 int lane) {
  bool flipped = false;
  for (int j = lane; j < 2 * 32 * nk; j += 32) {
    const bool is_b = j >= 32 * nk;
    const int jj = is_b ? j - 32 * nk : j;  // 16-byte run: atom kk = jj / 32, atom row i = jj % 32
    const uint4 v = *reinterpret_cast<const uint4*>(gen + (is_b ? sfb_atoms : sfa_atoms) + 16u * jj);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (((w[0] | w[1] | w[2] | w[3]) & 0x80808080u) == 0) continue;
    const int kk = jj / 32, i = jj % 32;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        if (!((w[g] >> (8 * blk + 7)) & 1u)) continue;
        const int r = 32 * g + i;  // tile row (A) or vector (B) of this scale byte
        if (is_b && r >= 16) continue;
        // byte 32*kk + 8*blk of row r in the 128-byte swizzled tile
        const uint32_t unit = (uint32_t)(2 * kk + blk / 2) ^ (uint32_t)(r & 7);
        const uint32_t off = (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u + unit * 16u +
                             8u * (uint32_t)(blk & 1);
        uint64_t* q = reinterpret_cast<uint64_t*>(gen + (is_b ? b_tile : a_tile) + off);
        *q ^= 0x8888888888888888ull;
        flipped = true;
      }
    }
  }
  return flipped;
}

__device__ __forceinline__ uint32_t lds_or4(uint32_t addr) {
  uint32_t x, y, z, w;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(x), "=r"(y), "=r"(z), "=r"(w)
               : "r"(addr));
  return x | y | z | w;
}

// Whether any of the stage's nk sfa and nk sfb atoms holds a code with the
// sign bit set (a warp vote; the benchmark's codes never do).  Every lane
// issues its loads (16 bytes per atom) before testing any, so the common
// all-positive stage costs the MMA warp one round of shared-memory latency;
// fold_scale_signs then runs only for stages that need it.
__device__ __forceinline__ bool any_negative_scale(uint32_t sfa_atoms, uint32_t sfb_atoms, int nk,
                                                   int lane) {
  uint32_t acc = 0;
  if (nk == 4) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      acc |= lds_or4(sfa_atoms + 512u * kk + 16u * lane);
      acc |= lds_or4(sfb_atoms + 512u * kk + 16u * lane);
    }
  } else {
    for (int kk = 0; kk < nk; ++kk) {
      acc |= lds_or4(sfa_atoms + 512u * kk + 16u * lane);
      acc |= lds_or4(sfb_atoms + 512u * kk + 16u * lane);
    }
  }
  return __any_sync(0xffffffffu, (acc & 0x80808080u) != 0u);
}

// Plain scales (GEMV, N = 1): lane i of the MMA warp turns the staged
// [128 rows][16 bytes] sfa box of a stage into its 4 atoms (atom kk holds,
// at byte 16*i + 4*g + b, the scale of block 4*kk + b of row 32*g + i: one
// 16-byte load per g, one 16-byte store per atom) and lanes 0..3 copy the
// stage's sfb word kk into row 0 of sfb atom kk (the other rows stay zero).
// Returns whether any of those codes has the sign bit set (a warp vote).
__device__ __forceinline__ bool plain_scales_to_atoms(uint8_t* gen, uint32_t staged_sfa,
                                                      uint32_t staged_sfb, uint32_t sfa_atoms,
                                                      uint32_t sfb_atoms, int lane) {
  uint32_t w[4][4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint4 v = *reinterpret_cast<const uint4*>(gen + staged_sfa + 16u * (32u * g + lane));
    w[g][0] = v.x;
    w[g][1] = v.y;
    w[g][2] = v.z;
    w[g][3] = v.w;
  }
  const uint32_t sbw = lane < 4 ? *reinterpret_cast<const uint32_t*>(gen + staged_sfb + 4u * lane) : 0u;
  uint32_t any = sbw;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    *reinterpret_cast<uint4*>(gen + sfa_atoms + 512u * kk + 16u * lane) =
        make_uint4(w[0][kk], w[1][kk], w[2][kk], w[3][kk]);
    any |= w[0][kk] | w[1][kk] | w[2][kk] | w[3][kk];
  }
  if (lane < 4) *reinterpret_cast<uint32_t*>(gen + sfb_atoms + 512u * lane) = sbw;
  return __any_sync(0xffffffffu, (any & 0x80808080u) != 0u);
}

// S: pipeline stages per CTA (2 or 4; fewer stages let more CTAs share an SM,
// whose independent copy+MMA chains then overlap).  NC: accumulator columns
// read back (a power of two >= N, the rows of B that hold data).  PLAIN: the
// GEMV with plain scales (N = 1), which the MMA warps lay out as atoms.
template <int S, int NC, bool PLAIN>
__global__ void __launch_bounds__(kTcThreads, 1)
    nvfp4_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t tc_smem[];
  __shared__ __align__(8) uint64_t bars[2 * S + 9];
  __shared__ uint32_t tmem_slot;

  const uint32_t raw = smem_u32(tc_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzled tiles want 1024-byte alignment
  const uint32_t a_s = base;
  const uint32_t b_s = a_s + S * kTcABytes;
  const uint32_t sfa_s = b_s + S * kTcBBytes;
  const uint32_t sfb_s = sfa_s + S * kTcSfBytes;
  const uint32_t red_s = sfb_s + S * kTcSfBytes;  // this CTA's partial sums [2][128][NC]
  const uint32_t stg_s = red_s + 2u * NC * 128u * 4u;  // plain: staged sfa [S][2 KB], sfb [S][128]
  auto staged_sfa = [&](int st) { return stg_s + (uint32_t)st * kTcSfBytes; };
  auto staged_sfb = [&](int st) { return stg_s + (uint32_t)S * kTcSfBytes + 128u * st; };
  uint8_t* const gen = tc_smem - raw;            // generic pointer = gen + shared address
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int st) { return bar0 + 8u * st; };
  auto empty_bar = [&](int st) { return bar0 + 8u * (S + st); };
  const uint32_t dfull_bar = bar0 + 8u * (2 * S);       // [2]
  const uint32_t dempty_bar = bar0 + 8u * (2 * S + 2);  // [2]
  const uint32_t rfull_bar = bar0 + 8u * (2 * S + 4);   // [2] (rank 0)
  const uint32_t rfree_bar = bar0 + 8u * (2 * S + 6);   // [2] (ranks > 0)
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 8);
  // TMEM columns: accumulators [2 chains][2][16], sfa and sfb [stage][4 atoms][4]
  constexpr uint32_t kSfaCol = 64, kSfbCol = 64 + 16 * S, kTmemCols = tc_tmem_cols(S);
  // stage slots per MMA chain: chain c owns slots c*SC .. c*SC + SC - 1
  constexpr int SC = S / 2;
  static_assert(S % 2 == 0, "two chains of equal rings");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ks = tc::cluster_size(), rank = tc::cluster_rank();
  const int cid = (int)(blockIdx.x / ks), nclusters = (int)(gridDim.x / ks);
  // tiles of this cluster: cid, cid + nclusters, ... below p.tiles (< 2^31)
  const int ntiles =
      cid < p.tiles ? (int)(((int64_t)p.tiles - cid + nclusters - 1) / nclusters) : 0;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int st = 0; st < S; ++st) {
      tc::mbar_init(full_bar(st), 1);
      tc::mbar_init(empty_bar(st), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(dfull_bar + 8u * i, 2);  // one commit per MMA chain
      tc::mbar_init(dempty_bar + 8u * i, 128);
      tc::mbar_init(rfull_bar + 8u * i, ks > 1 ? (ks - 1) * 128 : 1);
      tc::mbar_init(rfree_bar + 8u * i, 128);
    }
    tc::mbar_init(drain_bar, 2);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // rows N..15 of every B stage start as zeros and are never written again
  // (the b copy fills rows 0..N-1 only)
  for (uint32_t i = threadIdx.x; i < S * kTcBBytes / 16; i += kTcThreads)
    if ((int)((i % (kTcBBytes / 16)) / 8) >= p.N)
      *reinterpret_cast<uint4*>(gen + b_s + 16 * i) = make_uint4(0, 0, 0, 0);
  // plain scales: rows 1..127 of every sfb atom stay zero
  if constexpr (PLAIN)
    for (uint32_t i = threadIdx.x; i < S * kTcSfBytes / 16; i += kTcThreads)
      *reinterpret_cast<uint4*>(gen + sfb_s + 16 * i) = make_uint4(0, 0, 0, 0);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc::fence_before();
  __syncthreads();
  // every CTA's barriers are initialised before any remote arrive (clusters
  // of one CTA have no remote traffic: the barrier cost them ~0.5 us per CTA)
  if (ks > 1) tc::cluster_sync();
  tc::fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;

  // The contiguous K-stage range of this rank for tile t (the rank that takes
  // an extra stage rotates with t, so the split, and the rounding, depend on
  // the tile and the cluster size only, not on the grid).
  auto stage_range = [&](int t, int& s0, int& cnt) {
    const int per = p.kstages / (int)ks, extra = p.kstages % (int)ks;
    const int rr = (int)((rank + (uint32_t)t) % ks);
    cnt = per + (rr < extra ? 1 : 0);
    s0 = rr * per + (rr < extra ? rr : extra);
  };

  if (warp == 0) {
    if (lane == 0) {
      if (ntiles > 0) {  // the first stages' A lines, ahead of the dependency wait
        int s0, cnt;
        stage_range(cid, s0, cnt);
        const int l = cid / p.rest_m, mt = cid % p.rest_m;
        for (int i = 0; i < cnt && i < kTcPrefetchStages; ++i)
          tc::tma_prefetch_3d(&p.tmap_a, (s0 + i) * 128, mt * 128, l);
      }
      pdl_wait();
      // stage i of a tile goes to MMA chain i % 2, through that chain's ring
      int pos[2] = {0, 0}, issued[2] = {0, 0};
      uint32_t ph[2] = {0u, 0u};
      for (int j = 0; j < ntiles; ++j) {
        const int t = cid + j * nclusters;
        const int l = t / p.rest_m, mt = t % p.rest_m;
        int s0, cnt;
        stage_range(t, s0, cnt);
        for (int i = 0; i < cnt; ++i) {
          const int s = s0 + i;
          const int nk = min(4, p.rest_k - 4 * s);
          const int c = i & 1, st = c * SC + pos[c];
          if (tc::mbar_wait<false>(empty_bar(st), ph[c] ^ 1u, ok, &g_tc_timeouts)) {
            const uint32_t fb = full_bar(st);
            if constexpr (PLAIN) {
              // the stage's 16 scale bytes of every row, and of b (a whole box
              // either way; blocks past K arrive as zeros)
              tc::mbar_expect_tx(fb, kTcABytes + 128u * (uint32_t)p.N + kTcSfBytes + 16u);
            } else {
              tc::mbar_expect_tx(fb, kTcABytes + 128u * (uint32_t)p.N + 2u * (uint32_t)nk * 512u);
            }
            tc::tma_load_3d(a_s + st * kTcABytes, &p.tmap_a, s * 128, mt * 128, l, fb);
            tc::tma_load_3d(b_s + st * kTcBBytes, &p.tmap_b, s * 128, 0, l, fb);
            if constexpr (PLAIN) {
              tc::tma_load_3d(staged_sfa(st), &p.tmap_sfa, s * 16, mt * 128, l, fb);
              tc::tma_load_2d(staged_sfb(st), &p.tmap_sfb, s * 16, l, fb);
            } else {
              tc::bulk_load(sfa_s + st * kTcSfBytes,
                        p.sfa + (((int64_t)l * p.rest_m + mt) * p.rest_k + 4 * s) * 512,
                        (uint32_t)nk * 512u, fb);
              tc::bulk_load(sfb_s + st * kTcSfBytes, p.sfb + (int64_t)l * p.sfb_stride + (int64_t)s * 2048,
                        (uint32_t)nk * 512u, fb);
            }
            ++issued[c];
          }
          if (++pos[c] == SC) {
            pos[c] = 0;
            ph[c] ^= 1u;
          }
        }
      }
      // copies still in flight land before the CTA can exit: the last phase
      // issued on each slot (a phase already consumed passes at once)
      bool drain_ok = true;
      for (int c = 0; c < 2; ++c)
        for (int k = 0; k < SC && k < issued[c]; ++k) {
          const int i_last = issued[c] - 1 - k;
          tc::mbar_wait<false>(full_bar(c * SC + i_last % SC), (uint32_t)((i_last / SC) & 1), drain_ok, &g_tc_timeouts);
        }
    } else {
      pdl_wait();
    }
  } else if (warp == 1 || warp == 6) {
    // MMA chain c takes the stages i with i % 2 == c of every tile into its own
    // accumulator; the two chains' copies and MMAs run independently
    pdl_wait();
    const int c = warp == 1 ? 0 : 1;
    int pos = 0;
    uint32_t ph = 0;
    for (int j = 0; j < ntiles; ++j) {
      const int acc = j & 1;
      const uint32_t d = tmem + (uint32_t)(16 * (2 * c + acc));
      if (lane == 0) tc::mbar_wait<false>(dempty_bar + 8u * acc, ((uint32_t)(j >> 1) & 1u) ^ 1u, ok, &g_tc_timeouts);
      int s0, cnt;
      stage_range(cid + j * nclusters, s0, cnt);
      bool first = true;
      for (int i = c; i < cnt; i += 2) {
        const int s = s0 + i;
        const int nk = min(4, p.rest_k - 4 * s);
        const int st = c * SC + pos;
        if (lane == 0) tc::mbar_wait<false>(full_bar(st), ph, ok, &g_tc_timeouts);
        __syncwarp();  // (orders lane 0's acquire before the other lanes' reads)
        if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0) {
          // plain scales: lay the stage's scales out as atoms first (written
          // through the generic proxy, read by the tensor cores' copies)
          bool neg;
          if constexpr (PLAIN) {
            neg = plain_scales_to_atoms(gen, staged_sfa(st), staged_sfb(st), sfa_s + st * kTcSfBytes,
                                        sfb_s + st * kTcSfBytes, lane);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          } else {
            neg = any_negative_scale(sfa_s + st * kTcSfBytes, sfb_s + st * kTcSfBytes, nk, lane);
          }
          // signed scales: fold negative codes into the operands' sign bits
          if (neg) {
            const bool flipped =
                fold_scale_signs(gen, a_s + st * kTcABytes, b_s + st * kTcBBytes,
                                 sfa_s + st * kTcSfBytes, sfb_s + st * kTcSfBytes, nk, lane);
            if (__any_sync(0xffffffffu, flipped))
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // for the tensor cores
          }
          __syncwarp();
        }
        if (lane == 0 && ok) {
          tc::fence_after();
          for (int kk = 0; kk < nk; ++kk) {
            tc::copy_atom(tmem + kSfaCol + (uint32_t)(16 * st + 4 * kk),
                         tc::desc_atom(sfa_s + st * kTcSfBytes + 512u * kk));
            tc::copy_atom(tmem + kSfbCol + (uint32_t)(16 * st + 4 * kk),
                         tc::desc_atom(sfb_s + st * kTcSfBytes + 512u * kk));
          }
          for (int kk = 0; kk < nk; ++kk)
            tc::mma(d, tc::desc_sw128(a_s + st * kTcABytes + 32u * kk),
                    tc::desc_sw128(b_s + st * kTcBBytes + 32u * kk), kIdesc,
                   tmem + kSfaCol + (uint32_t)(16 * st + 4 * kk),
                   tmem + kSfbCol + (uint32_t)(16 * st + 4 * kk), !first || kk > 0);
          tc::commit(empty_bar(st));
        }
        first = false;
        if (++pos == SC) {
          pos = 0;
          ph ^= 1u;
        }
      }
      // a chain with no stage in this tile commits at once (its accumulator is
      // not read)
      if (lane == 0 && ok) tc::commit(dfull_bar + 8u * acc);
    }
    if (lane == 0) {
      // every MMA and TMEM copy of this chain has finished before TMEM is released
      tc::commit(drain_bar);
      bool drain_ok = true;
      tc::mbar_wait<false>(drain_bar, 0, drain_ok, &g_tc_timeouts);
    }
    __syncwarp();
  } else {
    pdl_wait();
    const uint32_t q = (uint32_t)(warp & 3);  // the TMEM lane quarter this warp may read
    const int r = (int)(32 * q) + lane;       // row inside the tile
    float* const red = reinterpret_cast<float*>(gen + red_s);
    for (int j = 0; j < ntiles; ++j) {
      const int t = cid + j * nclusters;
      const int l = t / p.rest_m, mt = t % p.rest_m;
      const int acc = j & 1;
      tc::mbar_wait<false>(dfull_bar + 8u * acc, (uint32_t)(j >> 1) & 1u, ok, &g_tc_timeouts);
      ok = __all_sync(0xffffffffu, ok);  // the TMEM load below is warp-collective
      float part[NC];
#pragma unroll
      for (int n = 0; n < NC; ++n) part[n] = 0.f;
      int s0, cnt;
      stage_range(t, s0, cnt);
      if (ok && cnt > 0) {  // K = 0: the sums are zero and no MMA ran
        tc::fence_after();
        tc::tmem_load_cols<NC>(tmem + (uint32_t)(16 * acc) + ((32u * q) << 16), part);
        if (cnt > 1) {  // chain 1 took the odd stages
          float odd[NC];
          tc::tmem_load_cols<NC>(tmem + (uint32_t)(16 * (2 + acc)) + ((32u * q) << 16), odd);
#pragma unroll
          for (int n = 0; n < NC; ++n) part[n] += odd[n];
        }
      }
      tc::fence_before();
      tc::mbar_arrive(dempty_bar + 8u * acc);
      const int64_t m = (int64_t)mt * 128 + r;
      const int buf = j & 1;
      const uint32_t use = (uint32_t)(j >> 1);
      if (ks > 1 && rank != 0) {
        // wait until rank 0 has read this buffer's previous use, then publish
        tc::mbar_wait<true>(rfree_bar + 8u * buf, (use & 1u) ^ 1u, ok, &g_tc_timeouts);
        // this row's NC partials side by side: [buf][row][NC]
#pragma unroll
        for (int n = 0; n < NC; ++n) red[(buf * 128 + r) * NC + n] = part[n];
        tc::mbar_arrive_remote(tc::map_rank(rfull_bar + 8u * buf, 0));
        continue;
      }
      if (ks > 1) {
        const bool got = tc::mbar_wait<true>(rfull_bar + 8u * buf, use & 1u, ok, &g_tc_timeouts);
        // each rank's NC partials of this row in vector loads, added in rank order
        if (got) {
          const uint32_t own = red_s + 4u * (uint32_t)((buf * 128 + r) * NC);
          for (uint32_t k = 1; k < ks; ++k) {
            float v[NC];
            tc::ld_remote_vec<NC>(tc::map_rank(own, k), v);
#pragma unroll
            for (int n = 0; n < NC; ++n) part[n] += v[n];
          }
        }
        for (uint32_t k = 1; k < ks; ++k) tc::mbar_arrive_remote(tc::map_rank(rfree_bar + 8u * buf, k));
      }
      if (ok && m < p.M) {
#pragma unroll
        for (int n = 0; n < NC; ++n) {
          if (n < p.N) {
            const int64_t idx = ((int64_t)l * p.N + n) * p.M + m;
            p.c[idx] = finish_value(part[n], p.alpha, p.bias, p.activation, idx);
          }
        }
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  if (ks > 1) tc::cluster_sync();  // no peer still reads or signals this CTA's shared memory
  if (warp == 1) {
    tc::fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

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

namespace {

using TcKernel = void (*)(TcParams);

// The kernel instance for (stages, columns read back, plain scales); null if
// none (plain scales: the GEMV, one column).
TcKernel tc_kernel_for(int stages, int nc, bool plain = false) {
  if (plain) {
    if (nc != 1) return nullptr;
    return stages == 2 ? nvfp4_tc_kernel<2, 1, true> : stages == 4 ? nvfp4_tc_kernel<4, 1, true> : nullptr;
  }
#define NVFP4_TC(S_, NC_) \
  if (stages == S_ && nc == NC_) return nvfp4_tc_kernel<S_, NC_, false>;
  NVFP4_TC(2, 1) NVFP4_TC(2, 2) NVFP4_TC(2, 4) NVFP4_TC(2, 8) NVFP4_TC(2, 16)
  NVFP4_TC(4, 1) NVFP4_TC(4, 2) NVFP4_TC(4, 4) NVFP4_TC(4, 8) NVFP4_TC(4, 16)
#undef NVFP4_TC
  return nullptr;
}

int tc_columns(int64_t n) { return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : n <= 8 ? 8 : 16; }

cudaError_t tc_launch_config(TcKernel kern, int stages, int nc, cudaLaunchConfig_t& cfg,
                             cudaLaunchAttribute (&attr)[2], int ks, int64_t ctas,
                             cudaStream_t stream, bool plain = false) {
  const uint32_t smem = tc_smem_bytes(stages, nc, plain);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  // all of the unified L1/shared storage as shared memory: the kernel reads
  // nothing through L1, and more CTAs per SM overlap their copy+MMA chains
  err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
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

// The static_asserts above, on the current device: shared memory must keep
// the CTAs resident on one SM within its 512 TMEM columns (at most 4 CTAs of
// 2 stages, 2 of 4 stages, 2 of 2 stages beside one of 4), so that no
// tcgen05.alloc ever waits for another CTA.  The smallest footprints (one
// column of B) are the ones that pack most CTAs.  Checked once per device.
cudaError_t tc_tmem_never_oversubscribed(bool* ok) {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cached[kMaxDevices];  // 0 unknown, 1 ok, 2 not
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c != 0) {
      *ok = c == 1;
      return cudaSuccess;
    }
  }
  int smem_sm = 0, reserved = 0;
  if ((err = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
          cudaSuccess ||
      (err = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
          cudaSuccess)
    return err;
  int64_t cta[2];
  for (int i = 0; i < 2; ++i) {
    cudaFuncAttributes fa;
    if ((err = cudaFuncGetAttributes(&fa, tc_kernel_for(2 + 2 * i, 1))) != cudaSuccess) return err;
    cta[i] = (int64_t)tc_smem_bytes(2 + 2 * i, 1) + (int64_t)fa.sharedSizeBytes + reserved;
  }
  *ok = 5 * cta[0] > smem_sm && 3 * cta[1] > smem_sm && cta[1] + 3 * cta[0] > smem_sm;
  if (dev >= 0 && dev < kMaxDevices) cached[dev].store(*ok ? 1 : 2, std::memory_order_relaxed);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemv_tc(const GemvParams& gp, int64_t N, int64_t L, int64_t b_row_stride,
                           int stages, int ks, int64_t ctas, cudaStream_t stream, bool plain) {
  const int nc = tc_columns(N);
  TcKernel kern = tc_kernel_for(stages, nc, plain);
  if (kern == nullptr || N < 1 || N > 16) return cudaErrorInvalidValue;
  // plain scales: 16-byte rows of sfa and sfb per stage through tensor maps
  // (row and batch strides multiples of 16 bytes: K % 256 == 0)
  if (plain && (gp.half_k % 128 != 0 || gp.sfb_stride % 16 != 0)) return cudaErrorInvalidValue;
  bool tmem_ok = false;
  cudaError_t terr = tc_tmem_never_oversubscribed(&tmem_ok);
  if (terr != cudaSuccess) return terr;
  if (!tmem_ok) return cudaErrorNotSupported;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr && gp.half_k > 0) return cudaErrorNotSupported;
  TcParams p;
  memset(&p, 0, sizeof(p));
  const cuuint64_t half_k = (cuuint64_t)gp.half_k;
  if (half_k > 0) {  // K = 0 reads nothing
    const cuuint64_t dims[3] = {half_k, (cuuint64_t)gp.M, (cuuint64_t)L};
    const cuuint64_t strides[2] = {half_k, half_k * (cuuint64_t)gp.M};
    const cuuint32_t box[3] = {128, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&p.tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(gp.a), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (half_k > 0) {
    const cuuint64_t dims[3] = {half_k, (cuuint64_t)N, (cuuint64_t)L};
    const cuuint64_t strides[2] = {(cuuint64_t)b_row_stride, (cuuint64_t)gp.b_stride};
    const cuuint32_t box[3] = {128, (cuuint32_t)N, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&p.tmap_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(gp.b), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (plain && half_k > 0) {
    const cuuint64_t blocks = (cuuint64_t)gp.blocks;
    const cuuint64_t sd[3] = {blocks, (cuuint64_t)gp.M, (cuuint64_t)L};
    const cuuint64_t ss[2] = {blocks, blocks * (cuuint64_t)gp.M};
    const cuuint32_t sbox[3] = {16, 128, 1};
    const cuuint64_t fd[2] = {blocks, (cuuint64_t)L};
    const cuuint64_t fs[1] = {(cuuint64_t)gp.sfb_stride};
    const cuuint32_t fbox[2] = {16, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&p.tmap_sfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(gp.sfa), sd, ss,
               sbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(&p.tmap_sfb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(gp.sfb), fd, fs,
               fbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  p.sfa = gp.sfa;
  p.sfb = gp.sfb;
  p.c = gp.c;
  p.bias = gp.bias;
  p.alpha = gp.alpha;
  p.activation = gp.activation;
  p.M = gp.M;
  p.sfb_stride = gp.sfb_stride;
  p.N = (int32_t)N;
  p.rest_m = gp.rest_m;
  p.rest_k = gp.rest_k;
  p.kstages = (gp.rest_k + 3) / 4;
  p.tiles = (int32_t)(L * gp.rest_m);
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cudaError_t err = tc_launch_config(kern, stages, nc, cfg, attr, ks, ctas, stream, plain);
  if (err != cudaSuccess) return err;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t tc_max_active_clusters(int stages, int64_t N, int ks, int* out) {
  const int nc = tc_columns(N);
  TcKernel kern = tc_kernel_for(stages, nc);
  if (kern == nullptr) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cudaError_t err = tc_launch_config(kern, stages, nc, cfg, attr, ks, ks, nullptr);
  if (err != cudaSuccess) return err;
  // CTAs per SM from the per-CTA limits: shared memory (with the per-CTA
  // reservation), registers, threads, and TMEM (512 columns per SM).  The
  // occupancy queries answer one CTA per SM for this kernel, while measured
  // runs place several per SM (twice the throughput with two).
  cudaFuncAttributes fa;
  err = cudaFuncGetAttributes(&fa, kern);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0, smem_sm = 0, reserved = 0, regs_sm = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess ||
      (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
      (err = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
          cudaSuccess ||
      (err = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
          cudaSuccess ||
      (err = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) !=
          cudaSuccess)
    return err;
  const int smem_cta = (int)tc_smem_bytes(stages, nc) + (int)fa.sharedSizeBytes + reserved;
  const int regs_cta = ((fa.numRegs * 32 + 255) / 256 * 256) * (kTcThreads / 32);
  int per_sm = smem_sm / smem_cta;
  if (regs_cta > 0 && regs_sm / regs_cta < per_sm) per_sm = regs_sm / regs_cta;
  if (2048 / kTcThreads < per_sm) per_sm = 2048 / kTcThreads;
  const int by_tmem = 512 / (int)tc_tmem_cols(stages);
  if (by_tmem < per_sm) per_sm = by_tmem;
  if (per_sm < 1) per_sm = 1;
  *out = sms * per_sm / ks > 0 ? sms * per_sm / ks : 1;
  return cudaSuccess;
}

cudaError_t tc_wait_timeouts(int reset, int* out) {
  cudaError_t err = cudaMemcpyFromSymbol(out, g_tc_timeouts, sizeof(int));
  if (err != cudaSuccess || !reset) return err;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_tc_timeouts, &zero, sizeof(int));
}

}  // namespace nvfp4

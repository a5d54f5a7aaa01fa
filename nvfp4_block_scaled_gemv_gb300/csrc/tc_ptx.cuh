// Inline-PTX helpers shared by the tensor-core kernels (sm_103a): mbarriers
// with bounded waits, TMA and bulk copies, distributed shared memory, and the
// tcgen05 operations (TMEM copy, MMA, commit, load).
#pragma once
#include <cstdint>

#include <cuda.h>  // CUtensorMap (the type only; the encoder is looked up at run time)
#include <cudaTypedefs.h>

#include "ptx.cuh"

namespace nvfp4 {
namespace tc {

// A wait on an mbarrier gives up after this much global time.
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s

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

// Slow path of mbar_wait: poll with a short sleep between tries (so waiting
// threads leave the issue slots and the barrier unit to the threads doing the
// work) until the phase completes or kWaitNs of global time pass.
template <bool CLUSTER>
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, int* timeouts) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (CLUSTER ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
    if (i > 8) __nanosleep(32);
    if ((i & 255u) == 0 && global_ns() - t0 > kWaitNs) {
      atomicAdd(timeouts, 1);
      return false;
    }
  }
}

// Bounded wait for the phase of the given parity; false (and ok cleared, one
// timeout counted in *timeouts) if it did not complete within kWaitNs, or if
// ok was already clear.  One thread per warp should wait (then __syncwarp):
// many threads polling one barrier slow down the barrier unit for everyone.
template <bool CLUSTER>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, bool& ok, int* timeouts) {
  if (!ok) return false;
  if (CLUSTER ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
  ok = mbar_wait_slow<CLUSTER>(bar, parity, timeouts);
  return ok;
}

// Bounded wait for two phases at once: both tries are in flight together, so
// two barriers that are usually complete cost one round trip.
__device__ __forceinline__ bool mbar_wait2(uint32_t bar1, uint32_t parity1, uint32_t bar2,
                                           uint32_t parity2, bool& ok, int* timeouts) {
  if (!ok) return false;
  uint32_t d1, d2;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%2], %3;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q, [%4], %5;\n\t"
      "selp.u32 %0, 1, 0, p;\n\tselp.u32 %1, 1, 0, q;\n\t}"
      : "=r"(d1), "=r"(d2)
      : "r"(bar1), "r"(parity1), "r"(bar2), "r"(parity2)
      : "memory");
  if (d1 && d2) return true;
  ok = (d1 || mbar_wait_slow<false>(bar1, parity1, timeouts)) &&
       (d2 || mbar_wait_slow<false>(bar2, parity2, timeouts));
  return ok;
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
// NC consecutive floats at a distributed-shared-memory address (16-byte
// aligned for NC >= 4), loaded with as few vector loads as fit.
template <int NC>
__device__ __forceinline__ void ld_remote_vec(uint32_t cluster_addr, float (&v)[NC]) {
  if constexpr (NC >= 4) {
#pragma unroll
    for (int i = 0; i < NC / 4; ++i)
      asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(v[4 * i]), "=f"(v[4 * i + 1]), "=f"(v[4 * i + 2]), "=f"(v[4 * i + 3])
                   : "r"(cluster_addr + 16u * i));
  } else if constexpr (NC == 2) {
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                 : "=f"(v[0]), "=f"(v[1])
                 : "r"(cluster_addr));
  } else {
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v[0]) : "r"(cluster_addr));
  }
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

// Tiled TMA load of a 2D box at (x, y) into shared memory, completing on the
// mbarrier (transaction bytes = the whole box, out-of-bounds fill included).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Tiled TMA load of a 3D box at (x, y, z) into shared memory, completing on
// the mbarrier (transaction bytes = the whole box, out-of-bounds fill
// included).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(map),
               "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
// Contiguous bulk copy global -> shared (both 16-byte aligned, bytes a
// multiple of 16), completing on the mbarrier.
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

// Instruction descriptor of the block-scaled MMA kind::mxf4nvf4: A and B E2M1
// (format 1, bits 7 and 10), both K-major, N/8 at bit 17, UE4M3 scales (bit
// 23 clear), M = 128 (M/16 at bit 24), scale ids 0, dense K = 64.  The
// hardware reads each scale byte as an unsigned E4M3 magnitude: the sign bit
// of a code is ignored (0x81..0xFE read as 0x01..0x7E); 0x7F and 0xFF are NaN.
__host__ __device__ constexpr uint32_t mxf4nvf4_idesc(uint32_t n) {
  return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void copy_atom(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}
// D (fp32, TMEM) = A x B (+ D when accumulate), 128 x N x 64, block-scaled by
// the scale vectors at TMEM addresses sfa and sfb.
__device__ __forceinline__ void mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                    uint32_t sfa, uint32_t sfb, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}
// Arrive on the mbarrier once every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void alloc(uint32_t slot_saddr, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

// Columns 0..NC-1 of this warp's 32 TMEM lanes (lane i of the warp gets
// row 32*quarter + i), as fp32.
template <int NC>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float (&out)[NC]) {
  uint32_t v[NC];
  if constexpr (NC == 1) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v[0]) : "r"(taddr));
  } else if constexpr (NC == 2) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];"
                 : "=r"(v[0]), "=r"(v[1])
                 : "r"(taddr));
  } else if constexpr (NC == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "r"(taddr));
  } else if constexpr (NC == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr));
  } else if constexpr (NC == 32) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
  } else {
    static_assert(NC == 16, "NC in {1, 2, 4, 8, 16, 32}");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int n = 0; n < NC; ++n) out[n] = __uint_as_float(v[n]);
}

}  // namespace tc

// cuTensorMapEncodeTiled, looked up once through the runtime (no link
// against the driver library); null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace nvfp4

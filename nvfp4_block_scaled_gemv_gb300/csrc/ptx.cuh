// Inline-PTX helpers for sm_103a: streaming loads, packed FP4/FP8 decode,
// half2 FMA and programmatic-dependent-launch control.
#pragma once
#include <cstdint>

namespace nvfp4 {

// 256-bit load of streamed data (read once): bypass L1, ask L2 for 256-byte
// prefetch granules.  p must be 32-byte aligned.
__device__ __forceinline__ void ld_stream_256(const void* p, uint32_t (&r)[8]) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::256B.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "l"(p));
}

// 32 bytes of data many warps re-read (the vector b) as two 128-bit loads
// with normal L1 caching (b needs only 16-byte alignment).
__device__ __forceinline__ void ld_shared_2x128(const void* p, uint32_t (&r)[8]) {
  asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%8];\n\t"
               "ld.global.nc.v4.b32 {%4,%5,%6,%7}, [%8+16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}

// 32-bit load of scale bytes (their 32-byte sectors are shared by
// neighbouring rows, so L1 allocation is kept).  p must be 4-byte aligned.
__device__ __forceinline__ uint32_t ld_scale_32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Four packed bytes of E2M1 pairs -> four f16x2 (byte j -> out[j]).  The
// word is split into byte registers first, so no shifts are needed.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

// Two E4M3 codes (the low, or with HI the high, 16 bits of v) -> f16x2.
// Exact; NaN stays NaN.
template <bool HI>
__device__ __forceinline__ uint32_t e4m3x2_half_to_f16x2(uint32_t v) {
  uint32_t out;
  if (HI)
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}"
        : "=r"(out)
        : "r"(v));
  else
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t}"
        : "=r"(out)
        : "r"(v));
  return out;
}

// Two E4M3 codes (low 16 bits of v) -> f16x2.  Exact; NaN stays NaN.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t out;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(out)
      : "r"(v));
  return out;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ float f16_lo_to_f32(uint32_t h) {
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}"
      : "=f"(f)
      : "r"(h));
  return f;
}

__device__ __forceinline__ float f16_hi_to_f32(uint32_t h) {
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, hi;\n\t}"
      : "=f"(f)
      : "r"(h));
  return f;
}

// (h.lo + h.hi) * s exactly in fp32, where h holds two fp16 partial sums and
// s is the low (HI = false) or high half of the f16x2 s2.  Both fused
// multiply-adds take fp16 operands and an fp32 addend; with the partial sums
// multiples of 1/4 below 2^10 and s an E4M3 value (4 significant bits), every
// intermediate fits in 24 bits, so nothing rounds.
template <bool HI>
__device__ __forceinline__ float f16x2_sum_times(uint32_t h, uint32_t s2) {
  float t;
  if (HI)
    asm("{\n\t.reg .b16 l, u, a, b;\n\tmov.b32 {l, u}, %1;\n\tmov.b32 {a, b}, %2;\n\t"
        "fma.rn.f32.f16 %0, l, b, 0f00000000;\n\tfma.rn.f32.f16 %0, u, b, %0;\n\t}"
        : "=f"(t)
        : "r"(h), "r"(s2));
  else
    asm("{\n\t.reg .b16 l, u, a, b;\n\tmov.b32 {l, u}, %1;\n\tmov.b32 {a, b}, %2;\n\t"
        "fma.rn.f32.f16 %0, l, a, 0f00000000;\n\tfma.rn.f32.f16 %0, u, a, %0;\n\t}"
        : "=f"(t)
        : "r"(h), "r"(s2));
  return t;
}

// Per-thread asynchronous copies global -> shared (completion tracked per
// thread with commit/wait groups).  16-byte copies bypass L1 (streamed data);
// 4-byte copies go through L1 (scale words whose 32-byte sectors neighbouring
// rows share).  Addresses must be aligned to the copy size.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// L2 policy for data read exactly once: its lines are the first to go, so
// streaming A does not push out lines that are still to be used (b, and A
// lines prefetched for the next call).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// cp_async_16 with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void cp_async_16_ef(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol) : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Hint: bring the line holding p into L2 (no data returned, no ordering).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Programmatic dependent launch: block until the preceding grid on the
// stream has completed and its writes are visible (a no-op when the launch
// carries no programmatic dependency).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next grid on the stream to begin launching.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace nvfp4

// Output epilogue shared by every kernel (sm_103a):
//   c = fp16_rne(act(alpha * v + bias))
// v the fp32 dot product, alpha the fp32 output scale, bias an optional fp16
// [L][M] (or [L][N][M]) addend fused with the scaling into one fp32 FMA, act
// one of the nvfp4_activation_t codes.
#pragma once
#include <cstdint>

#include <cuda_fp16.h>

namespace nvfp4 {

// act(y) in fp32 (the codes of nvfp4_activation_t); NaN stays NaN.  Kept out
// of line: every kernel's epilogue runs once per output, at the end of a CTA's
// work, from a cold instruction cache, and the inlined transcendental code of
// every output column made that tail measurably longer for calls that use no
// activation.
static __device__ __noinline__ float activate(float y, int act) {
  switch (act) {
    case 1:  // ReLU (+0 for y <= 0)
      return y > 0.f ? y : (y != y ? y : 0.f);
    case 2:  // SiLU: y * sigmoid(y)
      return y / (1.f + expf(-y));
    case 3: {  // GELU, tanh form
      const float u = 0.7978845608028654f * fmaf(0.044715f * y, y * y, y);
      return 0.5f * y * (1.f + tanhf(u));
    }
    case 4:  // GELU, erf form
      return 0.5f * y * (1.f + erff(y * 0.7071067811865476f));
    default:
      return y;
  }
}

__device__ __forceinline__ uint16_t finish_value(float v, float alpha, const uint16_t* bias,
                                                 int act, int64_t idx) {
  float o = bias ? fmaf(v, alpha, __half2float(__ushort_as_half(bias[idx]))) : v * alpha;
  if (act != 0) o = activate(o, act);
  return __half_as_ushort(__float2half_rn(o));
}

}  // namespace nvfp4

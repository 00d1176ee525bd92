// fp8.cuh -- FP8 (E4M3) storage of the compacted KV cache.
//
// Method ("Inference-Time Hyper-Scaling with KV Cache Compression",
// paper-notes page, "Related work"): quantizing the KV cache is orthogonal to
// DMS's sparsification and the two combine.  The pages fix no scheme; the one
// here stores every retained K and V row (one token, one KV head) as D E4M3
// codes with a float32 scale:
//   scale = amax / 448 (float32; a row of zeros gets scale 1),
//   code  = E4M3(x / scale), the float32 quotient rounded to nearest, ties to
//           even, saturated to +-448,
// and the row stands for code * scale.
#pragma once

#include "dms_device.cuh"

namespace dms {

constexpr float kE4m3Max = 448.0f;

// Two floats -> two E4M3 codes (round to nearest even, saturating); lo goes to
// the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (low byte first) -> two floats (exact: E4M3 values are f16 values).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t v) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(v)));
  float2 f;
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(f.x), "=f"(f.y)
      : "r"(h));
  return f;
}

// Quantize one token's K and V rows of one head into their FP8 slot rows, by a
// whole warp (all 32 lanes call it).  Lane c < CH holds K chunk c (8 bf16) in
// `in`, lane CH + c holds V chunk c; other lanes are idle.  krow / vrow are the
// slot's K row (D codes + the 16-byte scale chunk) and V row (D codes).
template <int D>
__device__ __forceinline__ void quantize_kv_rows(uint4 in, uint8_t* krow, uint8_t* vrow, int lane) {
  constexpr int CH = D / 8;
  const bool active = lane < 2 * CH;
  float x[8];
  {
    const float2 a = bf16x2_to_float2(in.x), b = bf16x2_to_float2(in.y);
    const float2 c = bf16x2_to_float2(in.z), d = bf16x2_to_float2(in.w);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
  }
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) amax = fmaxf(amax, active ? fabsf(x[e]) : 0.f);
  // max over the CH lanes of this row (groups of CH lanes are aligned)
#pragma unroll
  for (int off = CH / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f;
  uint2 codes;
  codes.x = f32x2_to_e4m3x2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale)) |
            (f32x2_to_e4m3x2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale)) << 16);
  codes.y = f32x2_to_e4m3x2(__fdiv_rn(x[4], scale), __fdiv_rn(x[5], scale)) |
            (f32x2_to_e4m3x2(__fdiv_rn(x[6], scale), __fdiv_rn(x[7], scale)) << 16);
  const float vscale = __shfl_sync(0xffffffffu, scale, CH);
  if (lane < CH) {
    reinterpret_cast<uint2*>(krow)[lane] = codes;
  } else if (active) {
    reinterpret_cast<uint2*>(vrow)[lane - CH] = codes;
  }
  if (lane == 0)
    *reinterpret_cast<uint4*>(krow + D) = make_uint4(__float_as_uint(scale), __float_as_uint(vscale), 0u, 0u);
}

}  // namespace dms

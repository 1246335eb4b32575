// e4m3 quantisation of new 16-bit K/V values, shared by the FP8 write kernel
// and the FP8 partition kernel's fused write: code = e4m3(float32(x) /
// scale), IEEE float32 division, round to nearest even, magnitudes beyond
// 448 saturated to +-448 ("PagedAttention internals", section 06: the block
// is the quantisation group; each block and KV head has its scale).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace pkv {
namespace fp8 {

__device__ __forceinline__ float widen16(uint32_t bits, bool bf16) {
  return bf16 ? __uint_as_float(bits << 16) : __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

// Two floats -> two e4m3 codes, `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_satfinite(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four 16-bit values (w01: elements 0, 1; w23: elements 2, 3) -> four codes,
// element 0 in the low byte.
__device__ __forceinline__ uint32_t quantize4(uint32_t w01, uint32_t w23, float scale, bool bf16) {
  const uint32_t e01 = e4m3x2_satfinite(__fdiv_rn(widen16(w01 & 0xffffu, bf16), scale),
                                        __fdiv_rn(widen16(w01 >> 16, bf16), scale));
  const uint32_t e23 = e4m3x2_satfinite(__fdiv_rn(widen16(w23 & 0xffffu, bf16), scale),
                                        __fdiv_rn(widen16(w23 >> 16, bf16), scale));
  return e01 | (e23 << 16);
}

}  // namespace fp8
}  // namespace pkv

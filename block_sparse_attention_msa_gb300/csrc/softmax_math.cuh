// Softmax arithmetic shared by the attention kernels: the SFU exponential, a three-input max
// and packed fp32 pair operations (one instruction for two values).
#pragma once

#include <stdint.h>

namespace msa {

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed fp32 pair arithmetic (one instruction for two lanes of data) and a three-input max.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1) {
  asm("{\n .reg .b64 ra, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rd, {%0, %1};\n"
      " add.rn.f32x2 rd, rd, ra;\n mov.b64 {%0, %1}, rd;\n}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}
__device__ __forceinline__ void mul2(float& d0, float& d1, float b0, float b1) {
  asm("{\n .reg .b64 rb, rd;\n mov.b64 rb, {%2, %3};\n mov.b64 rd, {%0, %1};\n"
      " mul.rn.f32x2 rd, rd, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "+f"(d0), "+f"(d1)
      : "f"(b0), "f"(b1));
}

}  // namespace msa

// store_fwht.cuh -- the 64-point transform the store builds run per half row.
//
// A row of 128 values is rotated by H128 = [[H64, H64], [H64, -H64]]
// (Sylvester order).  With two threads per row, thread h forms
// x_lo + x_hi (h = 0) or x_lo - x_hi (h = 1) and transforms those 64 values
// with H64: the result is elements 64h .. 64h + 63 of the row times H128,
// unnormalised.  The stride-64 butterflies thus come first, where the
// 128-point transform (fwht128_packed) runs them last, so the two sum in a
// different order and may differ in the last bit.
#pragma once

#include <cuda_runtime.h>

namespace h3kv {

// Unnormalised 64-point fast Walsh-Hadamard transform of x in place
// (Sylvester order): y_j = sum_i x_i (-1)^popcount(i & j).  Stride 1 runs in
// scalar; strides 2 .. 32 run two butterflies at a time in packed fp32
// (a + b with one add, a - b as fma(b, -1, a), both exactly rounded), so
// every value equals the scalar transform's.
__device__ __forceinline__ void fwht64_packed(float (&x)[64]) {
#pragma unroll
  for (int i = 0; i < 64; i += 2) {
    const float a = x[i], b = x[i + 1];
    x[i] = a + b;
    x[i + 1] = a - b;
  }
  const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
  for (int h = 2; h < 64; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
      if ((i & h) == 0) {
        const float2 a = make_float2(x[i], x[i + 1]);
        const float2 b = make_float2(x[i + h], x[i + h + 1]);
        const float2 sum = __fadd2_rn(a, b);
        const float2 dif = __ffma2_rn(b, neg1, a);
        x[i] = sum.x;
        x[i + 1] = sum.y;
        x[i + h] = dif.x;
        x[i + h + 1] = dif.y;
      }
    }
  }
}

}  // namespace h3kv

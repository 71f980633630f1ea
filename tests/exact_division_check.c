// Exhaustive host checks of the kvi8r store build's scale arithmetic
// (store_build.cu: div127, rcp_scale), in IEEE fp32 with a fused fma:
//  (1) q1 = fma(fma(-q0, 127, a), y, q0), q0 = a * y, y = RN(1/127), equals a / 127 (RN) for every
//      non-negative finite fp32 a;
//  (2) y1 = fma(fma(-p, y0, 1), y0, y0) equals 1 / p (RN) for every p = RN(sf * c), sf a positive finite
//      fp16 value, c = 11.313708498984761f, and every y0 within 2 ulp of 1 / p.
// (The same quotient step with 448 fails where the quotient is subnormal, and the same reciprocal step
// for an arbitrary s fails from starts 2 ulp away on some significands: the kvf8s build keeps the
// library's division and reciprocal.)
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float half_to_float(uint16_t h) {
  uint32_t e = (h >> 10) & 31, m = h & 1023;
  if (e == 0) return ldexpf((float)m, -24);
  return ldexpf((float)(m | 1024), (int)e - 25);
}
int main(void) {
  volatile float d127 = 127.0f, one = 1.0f;
  const float y = one / d127;
  uint64_t bad = 0, n = 0;
  for (uint32_t u = 0; u <= 0x7F7FFFFFu; ++u) {
    const float a = f_of(u);
    const float q0 = a * y;
    const float r = fmaf(-q0, 127.0f, a);
    const float q1 = fmaf(r, y, q0);
    const float ref = a / d127;
    if (u_of(q1) != u_of(ref)) { if (bad < 5) printf("div mismatch a=%a q1=%a ref=%a\n", a, q1, ref); ++bad; }
    ++n;
  }
  printf("division by 127: %llu of %llu mismatch\n", (unsigned long long)bad, (unsigned long long)n);
  const float c = 11.313708498984761f;
  uint64_t bad2 = 0, n2 = 0;
  for (uint32_t h = 1; h <= 0x7BFFu; ++h) {
    const float sf = half_to_float((uint16_t)h);
    const float p = sf * c;
    const float ref = one / p;
    for (int k = -2; k <= 2; ++k) {
      const float y0 = f_of(u_of(ref) + (uint32_t)k);
      const float e = fmaf(-p, y0, 1.0f);
      const float y1 = fmaf(e, y0, y0);
      if (u_of(y1) != u_of(ref)) { if (bad2 < 5) printf("rcp mismatch sf=%a p=%a k=%d y1=%a ref=%a\n", sf, p, k, y1, ref); ++bad2; }
      ++n2;
    }
  }
  printf("reciprocal of fp16 scale * sqrt(128): %llu of %llu mismatch\n", (unsigned long long)bad2, (unsigned long long)n2);
  return (bad || bad2) ? 1 : 0;
}

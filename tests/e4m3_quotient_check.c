// Host check of the kvf8s store build's V codes: code = e4m3(v / s), the
// quotient rounded once, exactly, to the nearest e4m3 value (ties to the even
// code, saturating at 448), where s = RN(b / 448) for a bf16 channel absmax b
// and v is any bf16 value with |v| <= b.  The build forms it in fp32 with
// r = RN(1/s), r16 = r 2^16 (e4m3_quotient2 in store_f8.cu, restated here):
// t = RN(v r); if t lies within a few fp32 ulps of an e4m3 rounding boundary
// m, the value sent to the conversion is RN(m + RN(v - m s) r16), which sits
// on the quotient's side of m (or is m on an exact tie); otherwise t itself.
//
// Checked on every (b, v) pair with b a positive finite bf16 value (b / 448
// not zero) and v one of the bf16 values in [0, b]; a sample of the negative
// values checks that the sign carries through.  Reference: binary search of
// the e4m3 grid with exact comparisons (for a grid value or midpoint c, at
// most five significant bits, c s is exact in double, and so is the sign of
// v - c s).  Below an absmax of 2^-100 the fp32 intermediates go subnormal
// and the procedure is not exact; those channels are counted apart.
//
// Usage: e4m3_quotient_check [stride]  (every stride-th absmax; default 1)
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static double grid[127];  // the non-negative e4m3 values, in code order

static void make_grid(void) {
  for (int c = 0; c < 127; ++c) {
    const int e = c >> 3, m = c & 7;
    grid[c] = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  }
}

// code (0..126) of the nearest e4m3 value to the non-negative a / s, ties to
// the even code, saturating; a and s as doubles holding fp32 values
static int round_exact(double a, double s) {
  if (a >= grid[126] * s) return 126;
  int lo = 0, hi = 126;  // grid[lo] * s <= a < grid[hi] * s
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (grid[mid] * s <= a) lo = mid;
    else hi = mid;
  }
  const double d = a - 0.5 * (grid[lo] + grid[hi]) * s;
  if (d > 0) return hi;
  if (d < 0) return lo;
  return (lo & 1) ? hi : lo;
}

// the conversion of one fp32 value (cvt.rn.satfinite.e4m3), as a signed code
static int cvt_e4m3(float x) {
  const int c = round_exact(fabs((double)x), 1.0);
  return x < 0 ? -c : c;
}

static float full_value(float v, float s, float r, float r16) {
  const float t = v * r;
  const float at = fabsf(t);
  const int sub = at < 0x1p-6f;
  const uint32_t ub = u_of(sub ? at + 0x1p-6f : at);
  const float mu = f_of((ub & 0xFFF00000u) | 0x00080000u);
  const float mk = copysignf(sub ? mu - 0x1p-6f : mu, t);
  const int near = ((ub & 0xFFFFFu) - 0x7FFFDu) < 7u;
  const float tn = fmaf(fmaf(-mk, s, v), r16, mk);
  return near ? tn : t;
}

int main(int argc, char **argv) {
  const int stride = argc > 1 ? atoi(argv[1]) : 1;
  const float tiny = 0x1p-100f;  // the smallest absmax the procedure is exact for
  make_grid();
  uint64_t pairs = 0, bad = 0, bad_tiny = 0, sym_bad = 0;
  float max_b_bad = 0.0f;
  for (uint32_t bb = 1; bb <= 0x7F7Fu; bb += (uint32_t)stride) {
    const float b = f_of(bb << 16);
    const float s = b / 448.0f;
    if (s == 0.0f) continue;  // the channel is dropped (its codes are zero)
    const float r = 1.0f / s, r16 = r * 65536.0f;
    for (uint32_t vb = 0; vb <= bb; ++vb) {
      const float v = f_of(vb << 16);
      const int got = cvt_e4m3(full_value(v, s, r, r16));
      ++pairs;
      if (got != round_exact((double)v, (double)s)) {
        if (b < tiny) {
          ++bad_tiny;
          if (b > max_b_bad) max_b_bad = b;
        } else {
          ++bad;
        }
      }
      if ((vb & 63u) == 0 && cvt_e4m3(full_value(-v, s, r, r16)) != -got) ++sym_bad;
    }
  }
  printf("pairs %llu\n", (unsigned long long)pairs);
  printf("absmax >= 2^-100: %llu mismatch\n", (unsigned long long)bad);
  printf("sign symmetry: %llu mismatch\n", (unsigned long long)sym_bad);
  printf("absmax < 2^-100: %llu mismatch (largest such absmax %a)\n", (unsigned long long)bad_tiny,
         (double)max_b_bad);
  return (bad || sym_bad) ? 1 : 0;
}

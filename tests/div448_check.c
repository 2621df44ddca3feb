/* div448_check.c -- checks the identity the fp8 kernels use for a block's
   scale, amax / 448 rounded to nearest, without a division: with
   y = RN(1/448), q0 = RN(a y), r = RN(a - 448 q0) and q = RN(q0 + r y)
   (one correction with the exact remainder, the method for divisors known
   in advance of Brisebarre, Muller and Raina), q == RN(a / 448) for every
   binary32 a in [2^-120, FLT_MAX].  The kernels take IEEE division for
   smaller amax, whose quotients are subnormal.

   Usage: div448_check STEP [nocorr|below]
     Runs over every STEP-th positive binary32 bit pattern a in
     [2^-120, FLT_MAX] and compares q with the IEEE quotient a / 448.0f.
     "nocorr" takes q0 itself (a control: it must fail somewhere);
     "below" runs over the patterns below 2^-120 instead, where the method
     is not used (failures there are expected and only counted).
   Prints "cases N mismatches M" and exits 0.
   Built with OpenMP (-fopenmp) the patterns are split over threads; without
   it the pragma is ignored. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float u2f(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint32_t f2u(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

int main(int argc, char **argv) {
  const long step = argc > 1 ? atol(argv[1]) : 1;
  const int nocorr = argc > 2 && strcmp(argv[2], "nocorr") == 0;
  const int below = argc > 2 && strcmp(argv[2], "below") == 0;
  const uint32_t lo_in = f2u(0x1p-120f), hi_in = f2u(3.4028234e38f);
  const uint32_t lo = below ? 1u : lo_in, hi = below ? lo_in - 1u : hi_in;
  const long n_pat = ((long)(hi - lo) + step) / step;
  const float y = 1.0f / 448.0f;
  long long n = 0, bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : n, bad)
  for (long i = 0; i < n_pat; ++i) {
    const float a = u2f(lo + (uint32_t)(i * step));
    const float q0 = a * y;
    const float q = nocorr ? q0 : fmaf(fmaf(-q0, 448.0f, a), y, q0);
    n++;
    if (f2u(q) != f2u(a / 448.0f)) bad++;
  }
  printf("cases %lld mismatches %lld\n", n, bad);
  return 0;
}

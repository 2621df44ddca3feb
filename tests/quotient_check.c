/* quotient_check.c -- checks the identity the fp8 dispatch kernels use to
   quantise bf16 rows without dividing: for y = RN(1/b), q0 = RN(x y),
   e = RN(b q0 - x) and q = RN(q0 - e y) (one correction with the exact
   remainder, after Markstein), q = RN(x / b).  The kernels compute it on -x and
   -y (so that x = -0 keeps its sign); this program does the same, in binary32
   with fmaf.

   Usage: quotient_check STEP [exact|nocorr|unsigned] [K]
     Runs over b = B * 2^k for k in {-60, -59, -40, -1, 0, 1, 40, 59, 60} and
     every STEP-th binary32 significand B in [1, 2), and over every finite bf16
     x (both signs, zeros, subnormals) with |x / b| < 1024.  Requires
       |x/b| >= 2^-12:  q == RN32(x / b), bit for bit;
       |x/b| <  2^-12:  |q| < 2^-10 (rounds to an E4M3 zero) with x's sign.
     The reference RN32(x / b) is the double quotient rounded to binary32: x
     has 8 significant bits, so x / b is never within 2^-48 relative of a
     binary32 midpoint unless on it, which it cannot be, and the double
     rounding is exact.
     Controls, which must fail, so that the check is seen to detect a wrong
     result: "nocorr" takes q0 itself (no correction); "unsigned" runs the
     steps on x and y, with e = RN(x - b q0) and q = RN(q0 + e y), where x = -0
     comes out +0.
     K, if given, replaces the nine exponents by that one.
   Prints "cases N exact_mismatches A small_failures B" and exits 0.
   Built with OpenMP (-fopenmp) the scale significands are split over threads;
   without it the pragma is ignored.

   With STEP 1 and k = 0 this is every binary32 b in [1, 2); scaling x and b
   by the same power of two changes no rounding while every intermediate stays
   normal, which covers b in [2^-60, 2^60]. */
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
  const long step = argc > 1 ? atol(argv[1]) : 4096;
  const int nocorr = argc > 2 && strcmp(argv[2], "nocorr") == 0;
  const int unsig = argc > 2 && strcmp(argv[2], "unsigned") == 0;
  static const int all_ks[] = {-60, -59, -40, -1, 0, 1, 40, 59, 60};
  int one_k[1];
  const int *ks = all_ks;
  unsigned nk = sizeof all_ks / sizeof all_ks[0];
  if (argc > 3) {
    one_k[0] = atoi(argv[3]);
    ks = one_k;
    nk = 1;
  }
  const long nm = ((1L << 23) + step - 1) / step;
  long long n = 0, bad_exact = 0, bad_small = 0;
  for (unsigned ki = 0; ki < nk; ++ki) {
#pragma omp parallel for schedule(dynamic, 16) reduction(+ : n, bad_exact, bad_small)
    for (long mi = 0; mi < nm; ++mi) {
      const uint32_t m = (uint32_t)(mi * step);
      const float b = ldexpf(u2f(0x3F800000u | m), ks[ki]);
      const float y = 1.0f / b, ny = -y;
      for (uint32_t xb = 0; xb < 0x10000u; ++xb) {
        if ((xb & 0x7F80u) == 0x7F80u) continue; /* inf, nan */
        const float x = u2f(xb << 16), nx = -x;
        const double qd = (double)x / (double)b;
        if (fabs(qd) >= 1024.0) continue;
        float q;
        if (unsig) {
          const float q0 = x * y;
          q = fmaf(fmaf(-b, q0, x), y, q0);
        } else {
          const float q0 = nx * ny;
          q = nocorr ? q0 : fmaf(fmaf(b, q0, nx), ny, q0);
        }
        n++;
        if (fabs(qd) >= 0x1p-12) {
          if (f2u(q) != f2u((float)qd)) bad_exact++;
        } else if (!(fabsf(q) < 0x1p-10f) || (signbit(q) != 0) != (signbit(x) != 0)) {
          bad_small++;
        }
      }
    }
  }
  printf("cases %lld exact_mismatches %lld small_failures %lld\n", n, bad_exact, bad_small);
  return 0;
}

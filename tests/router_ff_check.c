/* router_ff_check.c -- checks the router's softmax arithmetic: the weights
   e^(l_k - l_max) / sum_j e^(l_j - l_max) computed in float-float (binary32
   pairs) with a Cody-Waite reduced Taylor exponential, as the router kernel
   computes them, against the same weights in binary64.

   The steps are those of the kernel, in binary32 with fmaf and
   round-to-nearest (build with -ffp-contract=off so that no product and sum
   are fused behind the code's back):
     d = l_k - l_max as a float-float (TwoSum, exact);
     e^d for d >= -64: N = rint(32 d_h / ln 2) = 32 m + j, r = d - N (L1 +
       L2 + L3) as a float-float (L1 + L2 + L3 = ln 2 / 32), e^r = 1 + r +
       r^2 (1/2 + r/6 + r^2/24 + r^3/120) with the part after r in binary32
       and the two additions in float-float, times the float-float 2^(j/32)
       and 2^m; below -64 (and for -inf) in binary64;
     the sum of the K exponentials by a butterfly of float-float additions;
     w = RN(q + RN(rem y)), y ~ 1 / S_h, q = RN(e_h y), rem = e - q S.

   Usage: router_ff_check STEP ROWS [full|noL2|f32sum|rcpU]
     exp: every STEP-th binary32 d in [-64, 0] (bit patterns of -0 .. -64),
       plus ROWS * 8 differences of random logit pairs (non-zero low parts);
       reports the largest relative error of e_h + e_l against exp() in
       binary64, as a power of two (about 2^-36; the test requires below
       2^-35).
     softmax: ROWS random rows of K = 1..32 logits (N(0, s), s in {0.5, 1, 3,
       10}, some rounded to integers for exact ties), the weights against
       RN32 of the binary64 softmax; counts weights one ulp apart (the test
       allows 0.1% of them) and more than one ulp apart (must be none).
     "rcpU" (U = -2 .. 2) moves y = RN(1/S_h) by U ulps: the kernel takes y
       from the hardware's approximate reciprocal, and the corrected
       quotient must come out the same within these bounds for any such y.
     Controls, which must fail, so that the check is seen to detect a wrong
     result: "noL2" reduces by N L1 alone; "f32sum" adds the exponentials'
     high parts in binary32.
   Prints "exp_cases N exp_err_log2 X ulp1 A ulp2plus B rows R" and exits 0. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  float h, l;
} ff;

static int mode_nol2 = 0, mode_f32sum = 0, rcp_ulps = 0;

static ff two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  const float e = (a - (s - bb)) + (b - bb);
  ff r = {s, e};
  return r;
}
static ff fast_two_sum(float a, float b) {
  const float s = a + b;
  ff r = {s, b - (s - a)};
  return r;
}
static ff ff_add(ff a, ff b) {
  const ff s = two_sum(a.h, b.h);
  return fast_two_sum(s.h, s.l + (a.l + b.l));
}
static ff ff_mul(ff a, ff b) {
  const float p = a.h * b.h;
  float e = fmaf(a.h, b.h, -p);
  e = fmaf(a.h, b.l, fmaf(a.l, b.h, e));
  return fast_two_sum(p, e);
}
/* 2^(j/32) as float-float pairs (hi, lo), the kernel's table. */
static const float exp2_32[64] = {
    0x1p+0f, 0x0p+0f, 0x1.059b0ep+0f, -0x1.9d4f52p-25f, 0x1.0b5586p+0f, 0x1.9f3122p-25f,
    0x1.11301ep+0f, -0x1.fdb496p-25f, 0x1.172b84p+0f, -0x1.c15742p-27f, 0x1.1d4874p+0f, -0x1.d2e8cap-25f,
    0x1.2387a6p+0f, 0x1.ceac48p-25f, 0x1.29e9e0p+0f, -0x1.5c0424p-25f, 0x1.306fe0p+0f, 0x1.4636e2p-25f,
    0x1.371a74p+0f, -0x1.18aac6p-25f, 0x1.3dea64p+0f, 0x1.824684p-25f, 0x1.44e086p+0f, 0x1.8624b4p-30f,
    0x1.4bfdaep+0f, -0x1.593abcp-25f, 0x1.5342b6p+0f, -0x1.2c5610p-25f, 0x1.5ab07ep+0f, -0x1.5bd5ecp-27f,
    0x1.6247ecp+0f, -0x1.f8b550p-25f, 0x1.6a09e6p+0f, 0x1.9fcef4p-26f, 0x1.71f75ep+0f, 0x1.1d8beep-25f,
    0x1.7a1148p+0f, -0x1.829fd0p-25f, 0x1.82589ap+0f, -0x1.accc7cp-26f, 0x1.8ace54p+0f, 0x1.15506ep-27f,
    0x1.93737cp+0f, -0x1.e64744p-25f, 0x1.9c4918p+0f, 0x1.51f848p-27f, 0x1.a5503cp+0f, -0x1.b83b54p-25f,
    0x1.ae89fap+0f, -0x1.a94b14p-26f, 0x1.b7f770p+0f, -0x1.a09438p-25f, 0x1.c199bep+0f, -0x1.3d56b2p-27f,
    0x1.cb720ep+0f, -0x1.8837ccp-27f, 0x1.d5818ep+0f, -0x1.822dbcp-27f, 0x1.dfc974p+0f, -0x1.908c94p-25f,
    0x1.ea4afap+0f, 0x1.52486cp-27f, 0x1.f50766p+0f, -0x1.246eb0p-26f};

static ff ff_exp_neg(float dh, float dl) {
  const float kInv = 0x1.715476p+5f;
  const float kL1 = 0x1.62ep-6f, kL2 = 0x1.0bfbe8p-20f, kL3 = 0x1.cf79acp-45f;
  const float n = rintf(dh * kInv);
  const int ni = (int)n;
  const int j = ni & 31, m = ni >> 5;
  const float th = exp2_32[2 * j], tl = exp2_32[2 * j + 1];
  const float r1 = dh - n * kL1;
  float p2 = n * kL2, p2e = fmaf(n, kL2, -p2), l3 = n * kL3;
  if (mode_nol2) p2 = p2e = l3 = 0.0f;
  const ff s = two_sum(r1, -p2);
  const float low = ((s.l - p2e) + dl) - l3;
  const ff r = fast_two_sum(s.h, low);
  float q = fmaf(r.h, 0x1.111112p-7f, 0x1.555556p-5f);
  q = fmaf(q, r.h, 0x1.555556p-3f);
  q = fmaf(q, r.h, 0.5f);
  const float pr = (r.h * r.h) * q;
  ff one = {1.0f, 0.0f}, prf = {pr, 0.0f}, tt = {th, tl};
  const ff t = ff_add(one, ff_add(r, prf));
  const ff u = ff_mul(t, tt);
  const float two_m = ldexpf(1.0f, m);
  ff out = {u.h * two_m, u.l * two_m};
  return out;
}

/* The kernel's weights for one row of K logits sorted descending (lane k
   holds v[k]).  The butterfly: level l adds lanes k and k ^ 2^l. */
static void ff_softmax(int K, const float *v, float *w) {
  ff e[32], s[32];
  double z[32];
  int slow[32];
  int lg = 1;
  while ((1 << lg) < K) ++lg;
  const int L = 1 << lg;
  for (int k = 0; k < L; ++k) {
    e[k].h = e[k].l = 0.0f;
    slow[k] = 0;
    z[k] = 0.0;
    if (k < K) {
      const ff d = two_sum(v[k], -v[0]);
      if (d.h >= -64.0f) {
        e[k] = ff_exp_neg(d.h, d.l);
      } else {
        slow[k] = 1;
        z[k] = exp((double)v[k] - (double)v[0]);
        e[k].h = (float)z[k];
        e[k].l = (float)(z[k] - (double)e[k].h);
      }
    }
    s[k] = e[k];
    if (mode_f32sum) s[k].l = 0.0f;
  }
  for (int l = 0; l < lg; ++l) {
    ff t[32];
    for (int k = 0; k < L; ++k) t[k] = ff_add(s[k], s[k ^ (1 << l)]);
    memcpy(s, t, sizeof(ff) * (size_t)L);
  }
  for (int k = 0; k < K; ++k) {
    const ff S = s[k];
    if (!slow[k]) {
      float y = 1.0f / S.h;
      for (int u = 0; u < rcp_ulps; ++u) y = nextafterf(y, INFINITY);
      for (int u = 0; u > rcp_ulps; --u) y = nextafterf(y, 0.0f);
      const float q = e[k].h * y;
      const float pr = q * S.h;
      const float pe = fmaf(q, S.h, -pr);
      const float rem = ((e[k].h - pr) - pe) + (e[k].l - q * S.l);
      w[k] = q + rem * y;
    } else {
      w[k] = (float)(z[k] / ((double)S.h + (double)S.l));
    }
  }
}

static void oracle_softmax(int K, const float *v, float *w) {
  double z[32], sum = 0.0;
  for (int k = 0; k < K; ++k) {
    z[k] = exp((double)v[k] - (double)v[0]);
    sum += z[k];
  }
  for (int k = 0; k < K; ++k) w[k] = (float)(z[k] / sum);
}

static uint64_t rng = 0x9E3779B97F4A7C15ull;
static uint64_t next_u64(void) { /* splitmix64 */
  uint64_t z = (rng += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
static double uniform(void) { return (double)(next_u64() >> 11) * 0x1.0p-53; }
static float normal(void) {
  const double u1 = uniform() + 0x1.0p-60, u2 = uniform();
  return (float)(sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2));
}
static int cmp_desc(const void *a, const void *b) {
  const float x = *(const float *)a, y = *(const float *)b;
  return (x < y) - (x > y);
}
static double rel_err(ff e, double ref) {
  return fabs(((double)e.h + (double)e.l) - ref) / ref;
}
static uint32_t f2u(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

int main(int argc, char **argv) {
  if (argc < 3) return 2;
  const uint32_t step = (uint32_t)strtoul(argv[1], NULL, 10);
  const long rows = strtol(argv[2], NULL, 10);
  if (argc > 3) {
    mode_nol2 = strcmp(argv[3], "noL2") == 0;
    mode_f32sum = strcmp(argv[3], "f32sum") == 0;
    if (strncmp(argv[3], "rcp", 3) == 0) rcp_ulps = atoi(argv[3] + 3);
  }
  double worst = 0.0;
  long cases = 0;
  const uint32_t hi = f2u(-64.0f);
  for (uint32_t u = 0x80000000u; u <= hi; u += step) {
    float d;
    memcpy(&d, &u, 4);
    const double err = rel_err(ff_exp_neg(d, 0.0f), exp((double)d));
    if (err > worst) worst = err;
    ++cases;
  }
  for (long i = 0; i < rows * 8; ++i) {
    const float a = normal() * 8.0f, b = normal() * 8.0f;
    const float m = a > b ? a : b, v = a > b ? b : a;
    const ff d = two_sum(v, -m);
    if (!(d.h >= -64.0f)) continue;
    const double err = rel_err(ff_exp_neg(d.h, d.l), exp((double)v - (double)m));
    if (err > worst) worst = err;
    ++cases;
  }
  static const float sig[4] = {0.5f, 1.0f, 3.0f, 10.0f};
  long ulp1 = 0, ulp2 = 0;
  for (long r = 0; r < rows; ++r) {
    const int K = 1 + (int)(next_u64() % 32);
    const float s = sig[next_u64() % 4];
    const int ties = next_u64() % 4 == 0;
    float v[32], w[32], wo[32];
    for (int k = 0; k < K; ++k) v[k] = ties ? rintf(normal() * s) : normal() * s;
    qsort(v, (size_t)K, sizeof(float), cmp_desc);
    ff_softmax(K, v, w);
    oracle_softmax(K, v, wo);
    for (int k = 0; k < K; ++k) {
      const int64_t du = (int64_t)f2u(w[k]) - (int64_t)f2u(wo[k]);
      const int64_t a = du < 0 ? -du : du;
      if (a == 1) ++ulp1;
      else if (a > 1) ++ulp2;
    }
  }
  printf("exp_cases %ld exp_err_log2 %.2f ulp1 %ld ulp2plus %ld rows %ld\n", cases,
         worst > 0 ? log2(worst) : -999.0, ulp1, ulp2, rows);
  return 0;
}

/* router_ff_check.c -- checks the router's softmax arithmetic: the weights
   e^(l_k - l_max) / sum_j e^(l_j - l_max) computed in float-float (binary32
   pairs) with a Cody-Waite reduced Taylor exponential, as the router kernel
   computes them, against the same weights in binary64.

   The steps are those of the kernel, in binary32 with fmaf and
   round-to-nearest (build with -ffp-contract=off so that no product and sum
   are fused behind the code's back):
     d = l_k - l_max as a float-float (TwoSum, exact);
     e^d for d >= -64: n = rint(d_h / ln 2), r = d - n (L1 + L2 + L3) as a
       float-float, e^r = 1 + r (1 + r (1/2 + r (1/6 + r Q(r)))) with Q (the
       terms r^4/4! .. r^9/9! over r^3) in binary32, the product r Q exact,
       and the outer steps in float-float, times 2^n; below -64 (and for
       -inf) in binary64;
     the sum of the K exponentials by a butterfly of float-float additions;
     w = RN(q + RN(rem / S_h)), q = RN(e_h / S_h), rem = e - q S.

   Usage: router_ff_check STEP ROWS [full|noL2|f32sum]
     exp: every STEP-th binary32 d in [-64, 0] (bit patterns of -0 .. -64),
       plus ROWS * 8 differences of random logit pairs (non-zero low parts);
       reports the largest relative error of e_h + e_l against exp() in
       binary64, as a power of two (about 2^-34; the test requires below
       2^-33.5).
     softmax: ROWS random rows of K = 1..32 logits (N(0, s), s in {0.5, 1, 3,
       10}, some rounded to integers for exact ties), the weights against
       RN32 of the binary64 softmax; counts weights one ulp apart (the test
       allows 0.1% of them) and more than one ulp apart (must be none).
     Controls, which must fail, so that the check is seen to detect a wrong
     result: "noL2" reduces by n L1 alone; "f32sum" adds the exponentials'
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

static int mode_nol2 = 0, mode_f32sum = 0;

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
static ff ff_horner(float c, ff r, ff t) {
  ff cc = {c, 0.0f};
  return ff_add(cc, ff_mul(r, t));
}

static ff ff_exp_neg(float dh, float dl) {
  const float kInvLn2 = 0x1.715476p+0f;
  const float kL1 = 0x1.62e4p-1f, kL2 = 0x1.7f7d1cp-20f, kL3 = 0x1.ef357ap-45f;
  const float n = rintf(dh * kInvLn2);
  const float r1 = dh - n * kL1;
  float p2 = n * kL2, p2e = fmaf(n, kL2, -p2), l3 = n * kL3;
  if (mode_nol2) p2 = p2e = l3 = 0.0f;
  const ff s = two_sum(r1, -p2);
  const float low = ((s.l - p2e) + dl) - l3;
  const ff r = fast_two_sum(s.h, low);
  float q = 0x1.71de3ap-19f;
  q = fmaf(q, r.h, 0x1.a01a02p-16f);
  q = fmaf(q, r.h, 0x1.a01a02p-13f);
  q = fmaf(q, r.h, 0x1.6c16c2p-10f);
  q = fmaf(q, r.h, 0x1.111112p-7f);
  q = fmaf(q, r.h, 0x1.555556p-5f);
  const float rqh = r.h * q;
  ff c6 = {0x1.555556p-3f, -0x1.555556p-28f}, rq = {rqh, fmaf(r.l, q, fmaf(r.h, q, -rqh))};
  ff t = ff_add(c6, rq);
  t = ff_horner(0.5f, r, t);
  t = ff_horner(1.0f, r, t);
  t = ff_horner(1.0f, r, t);
  const float two_n = ldexpf(1.0f, (int)n);
  ff out = {t.h * two_n, t.l * two_n};
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
      const float q = e[k].h / S.h;
      const float pr = q * S.h;
      const float pe = fmaf(q, S.h, -pr);
      const float rem = ((e[k].h - pr) - pe) + (e[k].l - q * S.l);
      w[k] = q + rem / S.h;
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

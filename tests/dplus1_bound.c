/* Bound of the SwiGLU kernels' fast denominator against the specification.
 *
 * The specification's denominator is d = fl32(1 + exp_spec(t)), exp_spec a
 * Cody-Waite reduction (n = rint(t log2 e), r = (t - n ln2_hi) - n ln2_lo)
 * and a degree-7 Taylor polynomial in Horner form, every multiply and add
 * rounded on its own.  The kernels' fast path evaluates the same steps with
 * fused multiply-adds.  For every binary32 t in [-17, 88] taken with the
 * given stride this program compares the two and prints how many differ and
 * by how much (in binary32 ulps and relative).  Build without contraction
 * (-ffp-contract=off) so that the specification side stays unfused.
 *
 * usage: dplus1_bound STRIDE
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float bits_to_float(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t float_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

int main(int argc, char** argv) {
  const uint32_t stride = argc > 1 ? (uint32_t)strtoul(argv[1], NULL, 10) : 1u;
  const float log2e = bits_to_float(0x3FB8AA3Bu), ln2_hi = bits_to_float(0x3F317000u),
              ln2_lo = bits_to_float(0x3805FDF4u);
  /* 1/7!, 1/6!, 1/5!, 1/4!, 1/3!, 1/2, 1, 1 (highest power first) */
  const float coef[8] = {bits_to_float(0x39500D01u), bits_to_float(0x3AB60B61u), bits_to_float(0x3C088889u),
                         bits_to_float(0x3D2AAAABu), bits_to_float(0x3E2AAAABu), 0.5f, 1.0f, 1.0f};
  long long n = 0, differ = 0, max_ulp = 0;
  double max_rel = 0.0;
  for (int neg = 0; neg < 2; ++neg) {
    const uint32_t top = neg ? float_to_bits(17.0f) : float_to_bits(88.0f);
    for (uint32_t a = 0; a <= top; a += stride) {
      const float t = bits_to_float(a | (neg ? 0x80000000u : 0u));
      const float nn = rintf(t * log2e);
      const int ni = (int)nn;
      volatile float v;
      /* specification: separately rounded steps */
      float p = nn * ln2_hi;
      v = t - p;
      float r = v;
      p = nn * ln2_lo;
      v = r - p;
      r = v;
      float q = coef[0];
      for (int k = 1; k < 8; ++k) {
        const float m = q * r;
        v = m + coef[k];
        q = v;
      }
      v = 1.0f + ldexpf(q, ni);
      const float d_spec = v;
      /* fast path: fused multiply-adds */
      float rf = fmaf(-nn, ln2_hi, t);
      rf = fmaf(-nn, ln2_lo, rf);
      float qf = coef[0];
      for (int k = 1; k < 8; ++k) qf = fmaf(qf, rf, coef[k]);
      v = 1.0f + ldexpf(qf, ni);
      const float d_fast = v;
      ++n;
      if (float_to_bits(d_spec) != float_to_bits(d_fast)) {
        ++differ;
        long long du = (long long)float_to_bits(d_spec) - (long long)float_to_bits(d_fast);
        if (du < 0) du = -du;
        const double rel = fabs((double)d_fast / (double)d_spec - 1.0);
        if (rel > max_rel) max_rel = rel;
        if (du > max_ulp) max_ulp = du;
      }
    }
  }
  printf("n=%lld differ=%lld max_ulp=%lld max_rel_over_2^-24=%.4f\n", n, differ, max_ulp,
         max_rel / ldexp(1.0, -24));
  return 0;
}

/* The quantiser computes each group scale fl32(a / 448), a = max(amax, 1e-10),
 * as q0 = RN(a * y), y = RN(1/448), r = a - q0 * 448 (exact), q = RN(q0 + r * y)
 * with both corrections as fused multiply-adds (Markstein's corrected
 * reciprocal product).  This program checks that for every fp32 a from 1e-10
 * to the largest finite value the result equals the IEEE quotient a / 448
 * (the host's division, IEEE 754 correctly rounded), and prints the number of
 * mismatches.  Built with -ffp-contract=off: every operation is as written. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

int main(void) {
  const float y = 0x1.24924ap-9f;
  if (y != 1.0f / 448.0f) { printf("constant is not RN(1/448)\n"); return 2; }
  const float lo = 1e-10f;
  uint32_t b0;
  memcpy(&b0, &lo, 4);
  uint64_t bad = 0, n = 0;
  for (uint32_t b = b0; b < 0x7F800000u; ++b) {
    float a;
    memcpy(&a, &b, 4);
    const float want = a / 448.0f;
    const float q0 = a * y;
    const float r = fmaf(-q0, 448.0f, a);
    const float q = fmaf(r, y, q0);
    uint32_t wb, qb;
    memcpy(&wb, &want, 4);
    memcpy(&qb, &q, 4);
    bad += (wb != qb);
    ++n;
  }
  printf("checked %llu mismatches %llu\n", (unsigned long long)n, (unsigned long long)bad);
  return bad != 0;
}

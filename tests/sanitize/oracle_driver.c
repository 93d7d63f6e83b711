/* Runs the CPU oracle's entry points on small cases under AddressSanitizer and
 * UndefinedBehaviorSanitizer (including the fail-closed paths).  Built and run
 * by tests/test_sanitizers.py; returns non-zero on a failed check. */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include "pskv_oracle.h"

#define CHECK(c)                                                          \
  do {                                                                    \
    if (!(c)) {                                                           \
      fprintf(stderr, "check failed: %s:%d %s\n", __FILE__, __LINE__, #c); \
      return 1;                                                           \
    }                                                                     \
  } while (0)

static float frand(unsigned *s) {
  *s = *s * 1664525u + 1013904223u;
  return ((float)(*s >> 8) / 16777216.0f) * 2.0f - 1.0f;
}

int main(void) {
  enum { NP = 6, PS = 16, H = 2, D = 8, B = 2, HQ = 4, STRIDE = 3 };
  static float k[NP * H * PS * D], v[NP * H * PS * D], q[B * HQ * D];
  unsigned seed = 1;
  for (int i = 0; i < NP * H * PS * D; ++i) {
    k[i] = frand(&seed);
    v[i] = frand(&seed);
  }
  for (int i = 0; i < B * HQ * D; ++i) q[i] = frand(&seed);
  int32_t tables[B * STRIDE] = {3, 0, 5, 1, 4, 2};
  int32_t lens[B] = {40, 17};
  orc_pool pool = {k, v, ORC_F32, NP, PS, H, D, D};
  double out[B * HQ * D], out2[B * HQ * D];
  CHECK(orc_decode_direct(&pool, q, tables, STRIDE, lens, NULL, NULL, B, HQ, 0.35, out) == ORC_OK);
  CHECK(orc_decode_online(&pool, q, tables, STRIDE, lens, NULL, NULL, B, HQ, 0.35, 4, 7, 2, out2) ==
        ORC_OK);
  for (int i = 0; i < B * HQ * D; ++i) CHECK(fabs(out[i] - out2[i]) < 1e-12);
  int32_t first[B] = {0, 100}, lo[B] = {9, 110};
  CHECK(orc_decode_direct(&pool, q, tables, STRIDE, lens, first, lo, B, HQ, 0.35, out) == ORC_OK);
  int32_t bad_tables[B * STRIDE] = {3, 0, 99, 1, 4, 2};
  CHECK(orc_decode_direct(&pool, q, bad_tables, STRIDE, lens, NULL, NULL, B, HQ, 0.35, out) ==
        ORC_ERR_BAD_PAGE);
  int32_t zero[B] = {0, 5};
  CHECK(orc_decode_direct(&pool, q, tables, STRIDE, zero, NULL, NULL, B, HQ, 0.35, out) ==
        ORC_ERR_INVALID);

  double oa[D] = {0}, ob[D] = {0}, om[D];
  double m, l;
  CHECK(orc_merge(-INFINITY, 0.0, oa, 0.5, 2.0, ob, D, &m, &l, om) == ORC_OK);
  CHECK(orc_merge(-INFINITY, 1.0, oa, 0.5, 2.0, ob, D, &m, &l, om) == ORC_ERR_STATE);
  CHECK(orc_merge(NAN, 1.0, oa, 0.5, 2.0, ob, D, &m, &l, om) == ORC_ERR_STATE);
  CHECK(orc_finalize(-INFINITY, 0.0, oa, D, om) == ORC_ERR_STATE);

  float kn[1 * H * D] = {0}, vn[1 * H * D] = {0};
  int32_t row_of[1] = {1}, pos_of[1] = {40}, lease[B] = {3, 2};
  CHECK(orc_append_rows(k, v, &pool, kn, vn, row_of, pos_of, 1, tables, STRIDE, lease, B) ==
        ORC_ERR_PAST_PAGES);
  pos_of[0] = 20;
  CHECK(orc_append_rows(k, v, &pool, kn, vn, row_of, pos_of, 1, tables, STRIDE, lease, B) == ORC_OK);

  size_t a, b, c, t;
  CHECK(orc_partial_scratch_bytes(1, 32, 512, 32, &a, &b, &c, &t) == ORC_OK && t == 2105344);
  CHECK(orc_partial_scratch_bytes((int64_t)1 << 40, (int64_t)1 << 20, 512, 1024, &a, &b, &c, &t) ==
        ORC_ERR_OVERFLOW);
  puts("oracle driver ok");
  return 0;
}

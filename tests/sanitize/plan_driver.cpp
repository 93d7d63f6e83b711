// Exercises the CUDA library's host-only planning and argument checks
// (pskv_plan.cpp) under AddressSanitizer and UndefinedBehaviorSanitizer.
// Built and run by tests/test_sanitizers.py; returns non-zero on a failed check.
#include <cstdint>
#include <cstdio>
#include <vector>

#include "pskv_plan.h"

#define CHECK(c)                                               \
  do {                                                         \
    if (!(c)) {                                                \
      std::fprintf(stderr, "check failed: %s:%d %s\n", __FILE__, __LINE__, #c); \
      return 1;                                                \
    }                                                          \
  } while (0)

int main() {
  using namespace pskv;
  alignas(16) static char fake_k[64], fake_v[64];
  pskv_layout_desc d{};
  d.num_pages = 10;
  d.page_size = 256;
  d.num_kv_heads = 4;
  d.head_dim_k = d.head_dim_v = 512;
  d.kv_dtype = PSKV_DTYPE_BF16;
  d.format = PSKV_FORMAT_SPLIT;
  d.k_pool = fake_k;
  d.v_pool = fake_v;
  CHECK(check_layout_desc(&d) == PSKV_OK);
  pskv_layout_desc e = d;
  e.num_pages = (int64_t)1 << 62;
  CHECK(check_layout_desc(&e) != PSKV_OK);
  e = d;
  e.page_size = 17;
  CHECK(check_layout_desc(&e) == PSKV_ERR_INVALID_ARG);
  e = d;
  e.k_pool = fake_k + 4;
  CHECK(check_layout_desc(&e) == PSKV_ERR_INVALID_ARG);
  CHECK(check_layout_desc(nullptr) == PSKV_ERR_INVALID_ARG);
  e = d;
  e.format = PSKV_FORMAT_FOLDED;
  CHECK(check_layout_desc(&e) == PSKV_ERR_UNSUPPORTED);  // folded needs head_dim_k = head_dim_v / 4
  e.head_dim_k = 128;
  CHECK(check_layout_desc(&e) == PSKV_OK);
  e.kv_dtype = PSKV_DTYPE_F32;
  CHECK(check_layout_desc(&e) == PSKV_ERR_UNSUPPORTED);

  WorkspacePlan w;
  CHECK(plan_workspace(1, 32, 512, 32, 16, &w) == PSKV_OK);
  CHECK(w.groups == 2 && w.total % 256 == 0 && w.o_off >= w.l_off + 32 * 32 * 4);
  CHECK(plan_workspace(INT64_MAX / 2, 32, 512, 1024, 16, &w) == PSKV_ERR_OVERFLOW);
  CHECK(plan_workspace((int64_t)1 << 30, (int64_t)1 << 30, 512, 1024, 16, &w) == PSKV_ERR_OVERFLOW);
  CHECK(plan_workspace(0, 32, 512, 32, 16, &w) == PSKV_ERR_INVALID_ARG);

  pskv_layout lay{d, 2, 1024, 1024};
  std::vector<int32_t> lens = {1, 256 * 4, 7};
  CHECK(check_lengths(&lay, 3, 4, lens.data()) == PSKV_OK);
  lens[1] = 256 * 4 + 1;
  CHECK(check_lengths(&lay, 3, 4, lens.data()) == PSKV_ERR_INVALID_ARG);
  lens[1] = 0;
  CHECK(check_lengths(&lay, 3, 4, lens.data()) == PSKV_ERR_INVALID_ARG);

  std::vector<int32_t> one = {40002};
  CHECK(plan_splits(304, 1, 4, one.data()) == 76);                // every slot
  CHECK(plan_splits(304, 1, 4, one.data(), kFillBytes32) == 64);  // 27/32 of 76
  CHECK(plan_splits(152, 1, 4, one.data()) == 38);
  std::vector<int32_t> window = {1024};                           // 64 tiles: 3 per piece
  CHECK(plan_splits(608, 1, 16, window.data(), kFillBytes32) == 21);
  std::vector<int32_t> tiny = {5};
  CHECK(plan_splits(304, 1, 4, tiny.data()) == 1);
  std::vector<int32_t> ragged = {131072, 1, 5000, 17, 90000};
  const int p = plan_splits(304, 5, 4, ragged.data());
  CHECK(p >= 1 && p <= PSKV_AUTO_MAX_SPLITS);
  std::vector<int32_t> big(4096, INT32_MAX);
  CHECK(plan_splits(INT32_MAX, 4096, 4, big.data()) <= PSKV_AUTO_MAX_SPLITS);

  // tensor-memory prefill: a wave or more of blocks runs unsplit
  CHECK(plan_tc_splits(1024, 152, 64) == 1);
  CHECK(plan_tc_splits(128, 76, 166) == 1);
  CHECK(plan_tc_splits(32, 152, 1000) == 5);   // ceil(152 / 32)
  CHECK(plan_tc_splits(32, 152, 8) == 2);      // at most 8 / 4 partitions
  CHECK(plan_tc_splits(5, 152, 100000) == 31); // ceil(152 / 5)
  CHECK(plan_tc_splits(2, 152, 100000) == 32); // capped at 32
  CHECK(plan_tc_splits(0, 152, 10) == 1);
  CHECK(plan_verify_splits(4, 152, 313) == 38);   // one wave: floor(152 / 4)
  CHECK(plan_verify_splits(5, 152, 313) == 30);   // 150 CTAs, not a second wave of 3
  CHECK(plan_verify_splits(4, 152, 20) == 10);    // two tiles per partition at least
  CHECK(plan_verify_splits(4, 152, 1) == 1);
  CHECK(plan_verify_splits(152, 152, 313) == 1);
  CHECK(plan_verify_splits(1, 152, 100000) == 152);
  CHECK(plan_verify_splits(0, 152, 10) == 1);

  std::vector<int32_t> rows = {0, 1}, pos = {3, 600}, lease = {1, 2};
  CHECK(check_append_host(&lay, 2, 4, 2, rows.data(), pos.data(), lease.data()) ==
        PSKV_ERR_PAST_PAGES);
  pos[1] = 511;
  CHECK(check_append_host(&lay, 2, 4, 2, rows.data(), pos.data(), lease.data()) == PSKV_OK);
  rows[1] = 7;
  CHECK(check_append_host(&lay, 2, 4, 2, rows.data(), pos.data(), lease.data()) ==
        PSKV_ERR_INVALID_ARG);

  CHECK(pick_kernel(PSKV_DTYPE_BF16, 512, 8) == kKernelMma);
  CHECK(pick_kernel(PSKV_DTYPE_BF16, 256, 8) == kKernelMma);
  CHECK(pick_kernel(PSKV_DTYPE_F32, 512, 8) == kKernelSimt);
  CHECK(pick_kernel(PSKV_DTYPE_BF16, 256, 2) == kKernelMma);
  CHECK(pick_kernel(PSKV_DTYPE_BF16, 256, 16) == kKernelSimt);
  CHECK(pick_kernel(PSKV_DTYPE_BF16, 512, 16) == -1);
  CHECK(pick_kernel(PSKV_DTYPE_BF16, 128, 8) == -1);
  CHECK(pick_kernel(PSKV_DTYPE_BF16, 512, 8, PSKV_FORMAT_FOLDED) == kKernelMma);
  CHECK(pick_kernel(PSKV_DTYPE_BF16, 256, 16, PSKV_FORMAT_FOLDED) == -1);
  std::puts("plan driver ok");
  return 0;
}

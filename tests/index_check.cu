// Host-side check of the decode kernels' index checks (compiled and run by
// tests/test_index_checks.py, no GPU needed): checked_len, page_in_pool and
// splits_holding_tokens from csrc/kvq_internal.cuh -- the functions every decode kernel
// calls on the lengths and block-table entries it reads from device memory -- are driven
// here with in-range and out-of-range values, which never go near a GPU.
#include <climits>
#include <cstdio>

#include "../quantized_decode_attention_rht_gb300/csrc/kvq_internal.cuh"

using namespace kvq;

static int failures = 0;

static void expect(bool ok, const char* what, long long a, long long b) {
  if (!ok) {
    printf("FAIL %s (%lld, %lld)\n", what, a, b);
    ++failures;
  }
}

int main() {
  const int page = 16;
  for (int max_pages : {0, 1, 7, 4096, 1 << 20}) {
    const long long cap = (long long)max_pages * page;
    for (long long len : {-(1LL << 31), -17LL, -1LL, 0LL, 1LL, cap - 1, cap, cap + 1, cap + 16, (long long)INT_MAX}) {
      if (len < INT_MIN || len > INT_MAX) continue;
      int bits = 0;
      const int got = checked_len((int)len, max_pages, page, &bits);
      const bool in_range = len >= 0 && len <= cap;
      if (in_range) {
        expect(got == len && bits == 0, "in-range length kept", len, cap);
      } else {
        expect(bits == KVQ_DEVERR_SEQ_LEN, "out-of-range length flagged", len, cap);
        expect(got == (len < 0 ? 0 : cap), "out-of-range length clamped", len, got);
      }
      expect(got >= 0 && got <= cap, "checked length inside the block table", got, cap);
    }
  }
  for (int num_pages : {0, 1, 5, 1 << 24}) {
    for (long long phys : {(long long)INT_MIN, -2LL, -1LL, 0LL, 1LL, (long long)num_pages - 1, (long long)num_pages,
                           (long long)num_pages + 1, (long long)INT_MAX}) {
      if (phys < INT_MIN || phys > INT_MAX) continue;
      int bits = 0;
      const bool ok = page_in_pool((int)phys, num_pages, &bits);
      const bool in_pool = phys >= 0 && phys < num_pages;
      expect(ok == in_pool, "page decision", phys, num_pages);
      expect(bits == (in_pool ? 0 : KVQ_DEVERR_PAGE_INDEX), "page bit", phys, bits);
    }
  }
  // bits accumulate: a length and a page problem in one call
  {
    int bits = 0;
    checked_len(-5, 4, page, &bits);
    page_in_pool(99, 4, &bits);
    expect(bits == (KVQ_DEVERR_SEQ_LEN | KVQ_DEVERR_PAGE_INDEX), "bits accumulate", bits, 0);
  }
  // the combine pass reads at most the splits the plan made, whatever the length says
  for (int chunk : {16, 256, 2048})
    for (int num_splits : {0, 1, 3, 64})
      for (int len : {0, 1, chunk - 1, chunk, chunk + 1, 64 * chunk, 1 << 30}) {
        const int n = splits_holding_tokens(len, chunk, num_splits);
        const long long exact = ((long long)len + chunk - 1) / chunk;
        expect(n == (exact < num_splits ? exact : num_splits), "split count", len, n);
        expect(n >= 0 && n <= num_splits, "split count bounded", n, num_splits);
      }
  // planted mistake: a checker that compared against the wrong bound would pass this page
  {
    int bits = 0;
    expect(!page_in_pool(5, 5, &bits), "page equal to num_pages rejected", 5, 5);
  }
  printf("%d failures\n", failures);
  return failures != 0;
}

// Host-side check of the decode kernels' index checks (compiled and run by
// tests/test_index_checks.py, no GPU needed): checked_len, page_in_pool and
// splits_holding_tokens from csrc/kvq_internal.cuh -- the functions every decode kernel
// calls on the lengths and block-table entries it reads from device memory -- are driven
// here with in-range and out-of-range values, which never go near a GPU; and
// slot_holds_token, the generic decode kernel's test of a lane's slot, through that
// kernel's walk over a chunk's pages for every page size up to 40 and warp step width.
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
  // the generic decode kernel's walk over one chunk's pages: warps take logical pages
  // lp = p_begin + warp, + 4, ...; in a page a warp steps s0 = 0, TPS, ... < page_size with
  // lane group gi in [0, TPS) at slot off = s0 + gi.  Every token of [t_begin, t_end) must be
  // visited exactly once, and no slot the predicate accepts may lie past its page (its row
  // would be the next (page, kv head) block's, or past the pool after the last page).
  {
    auto walk = [](int ps, int tps, int t_begin, int t_end, bool (*pred)(int, int, int, int), bool* past_page) {
      static int seen[4096];
      for (int t = 0; t < 4096; ++t) seen[t] = 0;
      *past_page = false;
      const int p_begin = t_begin / ps, p_end = (t_end + ps - 1) / ps;
      for (int warp = 0; warp < 4; ++warp)
        for (int lp = p_begin + warp; lp < p_end; lp += 4)
          for (int s0 = 0; s0 < ps; s0 += tps)
            for (int gi = 0; gi < tps; ++gi) {
              const int off = s0 + gi;
              if (!pred(lp, off, ps, t_end)) continue;
              if (off >= ps) *past_page = true;
              const int t = lp * ps + off;
              if (t >= 0 && t < 4096) ++seen[t];
            }
      bool exact = true;
      for (int t = 0; t < 4096; ++t) exact = exact && seen[t] == (t >= t_begin && t < t_end ? 1 : 0);
      return exact;
    };
    auto fixed = [](int lp, int off, int ps, int t_end) { return slot_holds_token(lp, off, ps, t_end); };
    // the form without the page bound (the predicate before the page-size fix)
    auto old_form = [](int lp, int off, int ps, int t_end) { return lp * ps + off < t_end; };
    int old_caught = 0;
    for (int tps : {1, 2, 4, 8, 16})
      for (int ps = 1; ps <= 40; ++ps)
        for (int chunk_pages : {1, 3, 8})
          for (int len : {1, ps - 1, ps, ps + 1, 5 * ps + 3, 37 * ps}) {
            if (len < 1) continue;
            const int chunk = chunk_pages * ps;
            for (int t_begin = 0; t_begin < len && t_begin + chunk <= 4096; t_begin += chunk) {
              const int t_end = t_begin + chunk < len ? t_begin + chunk : len;
              bool past = false;
              const bool exact = walk(ps, tps, t_begin, t_end, fixed, &past);
              expect(exact, "every token of the chunk once", ps * 100 + tps, t_begin);
              expect(!past, "no slot past its page", ps * 100 + tps, t_begin);
              bool past_old = false;
              if (!walk(ps, tps, t_begin, t_end, old_form, &past_old) || past_old) ++old_caught;
            }
          }
    // planted mistake: the old form goes wrong exactly where the page size is no multiple of
    // TPS and a later page of the chunk exists, so the check above must see it fail
    expect(old_caught > 0, "the check catches the predicate without the page bound", old_caught, 0);
  }
  // planted mistake: a checker that compared against the wrong bound would pass this page
  {
    int bits = 0;
    expect(!page_in_pool(5, 5, &bits), "page equal to num_pages rejected", 5, 5);
  }
  printf("%d failures\n", failures);
  return failures != 0;
}

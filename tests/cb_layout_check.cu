// Host-side check of the codebook decode kernel's shared-memory placement (compiled and run
// by tests/test_cb_layout.py, no GPU needed): for every kernel instance the library builds
// and every 16-byte-aligned start of the dynamic shared-memory window, the tables must sit
// at a multiple of their size (the lookup addresses OR lane and field bits into them), the
// warp areas must not overlap the tables or each other, and everything must end inside the
// window the launcher asks for (Layout::SMEM, at most 227 KB).
#include <cstdio>

#include "../quantized_decode_attention_rht_gb300/csrc/decode_cb.cuh"

using namespace kvq::cbk;

static int failures = 0;

template <class L>
void check(const char* name, int d, int g, int kb, int vb, int mode, int wide) {
  int worst = 0;
  for (uint32_t base = 0; base < 128 * 1024; base += 16) {
    const typename L::Placement pl = L::place(base);
    bool ok = pl.t % L::TABLE == 0 && (L::QTAB == 0 || pl.q % L::QTAB == 0) && pl.q >= base;
    ok = ok && (L::SKT == 0 || (pl.t + L::TABLE) % 1024 == 0);
    // warp areas: inside [base, end), clear of the table block [q, w), disjoint
    for (int w = 0; w < L::WARPS && ok; ++w) {
      const uint32_t a = L::area(pl, base, w), e = a + L::WSM;
      ok = a >= base && e <= pl.end && (e <= pl.q || a >= pl.w) && a % 16 == 0;
      for (int v = 0; v < w && ok; ++v) {
        const uint32_t b = L::area(pl, base, v);
        ok = e <= b || a >= b + L::WSM;
      }
    }
    ok = ok && pl.end - base <= (uint32_t)L::SMEM && L::SMEM <= 227 * 1024;
    if ((int)(pl.end - base) > worst) worst = (int)(pl.end - base);
    if (!ok) {
      printf("FAIL %s D=%d G=%d K%d V%d mode %d wide %d base %u\n", name, d, g, kb, vb, mode, wide, base);
      ++failures;
      return;
    }
  }
  printf("ok %s D=%d G=%d K%d V%d mode %d wide %d: quad %d table %d warps %d x %d, smem %d (worst use %d)\n", name,
         d, g, kb, vb, mode, wide, L::QTAB, L::TABLE, L::WARPS, L::WSM, L::SMEM, worst);
}

template <int D, int G, int KB, int VB, int MODE, bool WIDE>
void one() {
  if constexpr (G == 1 && MODE == kModePlain && D == 256)
    check<typename Path1W<D, KB, VB>::L>("Path1W", D, G, KB, VB, MODE, 0);
  else if constexpr (G == 1) check<typename Path1<D, KB, VB, MODE>::L>("Path1", D, G, KB, VB, MODE, 0);
  else check<typename PathM<D, G, KB, VB, MODE, WIDE>::L>("PathM", D, G, KB, VB, MODE, WIDE ? 1 : 0);
}
template <int D, int G, int KB, int MODE, bool WIDE>
void values() {
  one<D, G, KB, 2, MODE, WIDE>();
  one<D, G, KB, 3, MODE, WIDE>();
  one<D, G, KB, 4, MODE, WIDE>();
}
template <int D, int G, int MODE, bool WIDE>
void keys() {
  values<D, G, 2, MODE, WIDE>();
  values<D, G, 3, MODE, WIDE>();
  values<D, G, 4, MODE, WIDE>();
}
template <int D, int MODE>
void groups() {
  keys<D, 1, MODE, false>();
  keys<D, 2, MODE, false>();
  keys<D, 4, MODE, false>();
}

// A planted mistake: a layout whose launch window is 4 KB short must be reported.
template <class L>
struct Shrunk : L {
  static constexpr int SMEM = L::SMEM - 4096;
};

int main() {
  // the instances the library launches: plain codes (D 128, 256; the 16-warp tensor-core
  // variant at D 128), keys with a residual sketch (D 128), keys with an outlier stream
  groups<128, kModePlain>();
  groups<256, kModePlain>();
  keys<128, 2, kModePlain, true>();
  keys<128, 4, kModePlain, true>();
  groups<128, kModeSketch>();
  groups<128, kModeOutlier>();
  groups<256, kModeOutlier>();
  const int real = failures;
  check<Shrunk<PathM<128, 4, 3, 2, kModePlain, true>::L>>("planted", 128, 4, 3, 2, kModePlain, 1);
  const bool caught = failures == real + 1;
  failures = real;
  printf("planted mistake %s\n", caught ? "caught" : "MISSED");
  printf("%d failures\n", failures);
  return (failures || !caught) ? 1 : 0;
}

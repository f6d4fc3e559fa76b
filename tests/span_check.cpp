// span_check.cpp — CPU check of the window geometry every kernel walks (swa::Span in
// swa_kernels.h) against brute force over the visibility rule itself.
//
// For query i (at key position i + off, off = Lk - Lq) and key j, visible <=> dmin <= i + off - j
// <= dmax, with [dmin, dmax] = [0, W - 1] for a causal window and [-(W - 1), W - 1] for a two-sided
// one.  For every (Lq, Lk, W, causal) in a grid of small sizes around the tile edges this checks:
//   first_kblock / last_kblock: the key blocks holding a key visible to some query of a block;
//   first_qblock / last_qblock: the query blocks holding a query that sees some key of a block
//                               (first > last exactly when no query sees it);
//   interior: true exactly when every cell of the 128 x 128 tile is inside both sequences and
//             visible.
// Prints "ok <cases>" and exits 0, or prints the first mismatch and exits 1.
#include <cstdio>

#include "swa_kernels.h"

namespace {

bool visible(const swa::Span& sp, int i, int j) {
  const int d = i + sp.off - j;
  return d >= sp.dmin && d <= sp.dmax;
}

int fail(const char* what, const swa::Span& sp, int blk, int got, int want) {
  std::printf("mismatch %s: Lq=%d Lk=%d off=%d dmin=%d dmax=%d block %d: got %d, want %d\n", what,
              sp.Lq, sp.Lk, sp.off, sp.dmin, sp.dmax, blk, got, want);
  return 1;
}

}  // namespace

int main() {
  using swa::kBlockM;
  using swa::kBlockN;
  const int lks[] = {1, 2, 5, 127, 128, 129, 200, 255, 256, 257, 385};
  const int ws[] = {1, 2, 7, 64, 127, 128, 129, 200, 300, 1000};
  long long cases = 0;
  for (int Lk : lks) {
    for (int Lq = 1; Lq <= Lk; Lq = (Lq < 4 ? Lq + 1 : Lq * 2 + 1)) {
      const int lq_values[] = {Lq, Lk};
      for (int lq : lq_values) {
        if (lq > Lk) continue;
        for (int W : ws) {
          for (int causal = 0; causal < 2; ++causal) {
            const swa::Span sp{lq, Lk, Lk - lq, causal ? 0 : -(W - 1), W - 1};
            ++cases;
            // key blocks visited by each query block
            for (int q0 = 0; q0 < lq; q0 += kBlockM) {
              int lo = -1, hi = -1;
              for (int i = q0; i < q0 + kBlockM && i < lq; ++i)
                for (int j = 0; j < Lk; ++j)
                  if (visible(sp, i, j)) {
                    if (lo < 0 || j / kBlockN < lo) lo = j / kBlockN;
                    if (j / kBlockN > hi) hi = j / kBlockN;
                  }
              if (lo < 0) return fail("query block sees no key", sp, q0 / kBlockM, -1, 0);
              if (sp.first_kblock(q0) != lo) return fail("first_kblock", sp, q0 / kBlockM, sp.first_kblock(q0), lo);
              if (sp.last_kblock(q0) != hi) return fail("last_kblock", sp, q0 / kBlockM, sp.last_kblock(q0), hi);
            }
            // query blocks that visit each key block
            for (int k0 = 0; k0 < Lk; k0 += kBlockN) {
              int lo = -1, hi = -1;
              for (int j = k0; j < k0 + kBlockN && j < Lk; ++j)
                for (int i = 0; i < lq; ++i)
                  if (visible(sp, i, j)) {
                    if (lo < 0 || i / kBlockM < lo) lo = i / kBlockM;
                    if (i / kBlockM > hi) hi = i / kBlockM;
                  }
              const int f = sp.first_qblock(k0), l = sp.last_qblock(k0);
              if (lo < 0) {
                if (f <= l) return fail("unvisited key block has a walk", sp, k0 / kBlockN, l - f + 1, 0);
              } else {
                if (f != lo) return fail("first_qblock", sp, k0 / kBlockN, f, lo);
                if (l != hi) return fail("last_qblock", sp, k0 / kBlockN, l, hi);
              }
            }
            // interior tiles
            for (int q0 = 0; q0 < lq; q0 += kBlockM)
              for (int k0 = 0; k0 < Lk; k0 += kBlockN) {
                bool all = true;
                for (int i = q0; all && i < q0 + kBlockM; ++i)
                  for (int j = k0; all && j < k0 + kBlockN; ++j)
                    all = i < lq && j < Lk && visible(sp, i, j);
                if (sp.interior(q0, k0) != all)
                  return fail("interior", sp, (q0 / kBlockM) * 1000 + k0 / kBlockN,
                              sp.interior(q0, k0), all);
              }
          }
        }
      }
    }
  }
  std::printf("ok %lld\n", cases);
  return 0;
}

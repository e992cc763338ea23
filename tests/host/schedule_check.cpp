// Host check of the work decomposition in pa_schedule.h: every tile of every
// sequence is owned by exactly one range, the slot rule gives each (range,
// sequence) pair a distinct partial slot, and the merge side finds the same
// slots the producing side used.
#include <stdio.h>
#include <stdlib.h>

#include <vector>

#include "pa_schedule.h"

static int check(const std::vector<int>& ctx, int64_t R) {
  std::vector<int64_t> P(ctx.size() + 1, 0);
  for (size_t s = 0; s < ctx.size(); ++s) P[s + 1] = P[s] + pa::tiles_of(ctx[s]);
  const int64_t T = P.back();
  if (T == 0) return 0;
  // Ranges partition [0, T).
  for (int64_t r = 0; r < R; ++r)
    if (pa::range_start(r, T, R) > pa::range_start(r + 1, T, R)) return 1;
  if (pa::range_start(0, T, R) != 0 || pa::range_start(R, T, R) != T) return 2;
  for (int64_t x = 0; x < T; ++x) {
    const int64_t r = pa::range_of_tile(x, T, R);
    if (!(pa::range_start(r, T, R) <= x && x < pa::range_start(r + 1, T, R))) return 3;
  }
  // Producer side: slots written per range; merge side: slots read.
  std::vector<int> used(2 * R, -1);
  for (size_t s = 0; s < ctx.size(); ++s) {
    const int64_t lo = P[s], hi = P[s + 1];
    if (lo == hi) continue;
    const int64_t r0 = pa::range_of_tile(lo, T, R), r1 = pa::range_of_tile(hi - 1, T, R);
    for (int64_t r = r0; r <= r1; ++r) {
      const int64_t a = pa::range_start(r, T, R), b = pa::range_start(r + 1, T, R);
      if (a == b) continue;
      const int slot = pa::segment_slot(a, b, lo, hi);
      if (r0 == r1) {
        if (slot != -1) return 4;
        continue;
      }
      if (slot < 0) return 5;
      if (slot != pa::partial_slot_of_range(r, lo, T, R)) return 6;
      if (used[2 * r + slot] != -1) return 7;  // two sequences in one slot
      used[2 * r + slot] = (int)s;
    }
  }
  return 0;
}

int main() {
  unsigned seed = 12345;
  auto rnd = [&](int n) { seed = seed * 1103515245u + 12345u; return (int)((seed >> 8) % (unsigned)n); };
  int cases = 0;
  for (int trial = 0; trial < 3000; ++trial) {
    const int S = 1 + rnd(40);
    std::vector<int> ctx(S);
    const int kind = rnd(4);
    for (int s = 0; s < S; ++s) {
      if (kind == 0) ctx[s] = rnd(50);
      else if (kind == 1) ctx[s] = 1 + rnd(2000);
      else if (kind == 2) ctx[s] = (rnd(3) == 0) ? 0 : 1 + rnd(40);
      else ctx[s] = 16 * (1 + rnd(8));
    }
    const int64_t R = 1 + rnd(300);
    const int rc = check(ctx, R);
    if (rc) {
      printf("FAIL code %d (S=%d R=%lld kind=%d)\n", rc, S, (long long)R, kind);
      return 1;
    }
    ++cases;
  }
  // Large totals: no overflow in the 64-bit range arithmetic.
  std::vector<int> big(4096, 1 << 24);
  if (check(std::vector<int>(big.begin(), big.begin() + 8), 152)) return 1;
  printf("ok %d cases\n", cases);
  return 0;
}

// Host-side checks of the work-map arithmetic the kernels share with the
// host (moe_internal.h): the per-expert tile plan, the bound on the tile
// list every workspace and checked build relies on, the tile-entry test of
// the checked builds, and the MXFP8 per-tile scale layout.  Built and run by
// tests/test_host_logic.py with the host compiler; prints "ok" and exits 0
// when every property holds, else names the first failure and exits 1.
#include <climits>
#include <cstdint>
#include <cstdio>
#include <vector>

#include "../../precision_moe_grouped_gb300/csrc/moe_internal.h"

namespace {

int failures = 0;

void expect(bool ok, const char* what, long long a = 0, long long b = 0, long long c = 0) {
  if (!ok && failures++ < 10) std::printf("FAIL %s (%lld, %lld, %lld)\n", what, a, b, c);
}

// 64-bit linear congruential generator (Knuth's MMIX constants).
struct Lcg {
  uint64_t s;
  uint32_t next() {
    s = s * 6364136223846793005ull + 1442695040888963407ull;
    return static_cast<uint32_t>(s >> 33);
  }
};

const int kBns[] = {moe::kTinyBN, moe::kDecodeBN, moe::kW4A16BN, moe::kMidBN, moe::kPrefillBN};

void check_plan() {
  for (int bn : kBns)
    for (int c = -3; c <= 3000; ++c) {
      const int2 p = moe::expert_tile_plan(c, bn);
      if (c <= 0) {
        expect(p.x == 0, "no tiles for an empty expert", c, bn);
        continue;
      }
      const int nt = p.x, tsz = p.y;
      expect(tsz % 16 == 0 && tsz >= 16 && tsz <= bn, "tile size multiple of 16 within bn", c, bn,
             tsz);
      expect(static_cast<long long>(nt) * tsz >= c && static_cast<long long>(nt - 1) * tsz < c,
             "tiles cover the rows, last tile non-empty", c, bn, nt);
      expect(nt == (c + bn - 1) / bn, "as few tiles as bn allows", c, bn, nt);
    }
}

void check_bound() {
  Lcg g{12345};
  const int Es[] = {1, 2, 8, 64, 256, 384, 1024};
  for (int E : Es)
    for (int trial = 0; trial < 40; ++trial) {
      const int T = 1 + static_cast<int>(g.next() % 3000);
      const int k = 1 + static_cast<int>(g.next() % (E < 32 ? E : 32));
      const int64_t R = static_cast<int64_t>(T) * k;
      // counts: uniform, skewed to few experts, or rows just above a multiple of 16
      std::vector<int> cnt(E, 0);
      const int kind = trial % 3;
      for (int64_t r = 0; r < R; ++r) {
        int e;
        if (kind == 0) e = static_cast<int>(g.next() % E);
        else if (kind == 1) e = static_cast<int>((g.next() % E) * (g.next() % E) / (E > 1 ? E : 1));
        else e = static_cast<int>((r / 17) % E);
        ++cnt[e];
      }
      for (int bn : kBns) {
        int64_t tiles = 0;
        for (int e = 0; e < E; ++e) tiles += moe::expert_tile_plan(cnt[e], bn).x;
        expect(tiles <= moe::max_work_tiles(R, E, bn), "tile list within its bound", R, E, bn);
        expect(moe::max_work_tiles(R, E, bn) <= moe::max_work_tiles(R, E, moe::kTinyBN),
               "the 16-row bound covers every tile size", R, E, bn);
        // every entry of the list the plan builds passes the checked builds' test
        int64_t off = 0;
        for (int e = 0; e < E; ++e) {
          const int2 p = moe::expert_tile_plan(cnt[e], bn);
          for (int i = 0; i < p.x; ++i) {
            const int r0 = i * p.y, rows = cnt[e] - r0 < p.y ? cnt[e] - r0 : p.y;
            expect(moe::tile_entry_ok(e, static_cast<int>(off + r0), rows, 0, bn,
                                      static_cast<int>(R), E),
                   "planned entry accepted", e, off + r0, rows);
          }
          off += cnt[e];
        }
      }
    }
}

void check_entry_test() {
  const int R = 1000, E = 8, bn = 160;
  expect(moe::tile_entry_ok(0, 0, 16, 0, bn, R, E), "first tile");
  expect(moe::tile_entry_ok(7, R - 1, 1, 0, bn, R, E), "last row");
  expect(moe::tile_entry_ok(3, R - bn, bn, 0, bn, R, E), "full tile at the end");
  struct Bad { int x, y, z, w; const char* why; };
  const Bad bad[] = {{-1, 0, 16, 0, "negative expert"},      {E, 0, 16, 0, "expert E"},
                     {0, -1, 16, 0, "negative row"},         {0, 0, 0, 0, "no rows"},
                     {0, 0, -5, 0, "negative rows"},         {0, 0, bn + 1, 0, "more than bn"},
                     {0, R - 15, 16, 0, "past the last row"}, {0, R, 1, 0, "row R"},
                     {0, INT_MAX, 1, 0, "row near INT_MAX"},  {0, INT_MAX - 2, 160, 0, "sum overflow"},
                     {0, 0, INT_MIN, 0, "INT_MIN rows"},      {0, 0, 16, 1, "marked entry"}};
  for (const Bad& b : bad) expect(!moe::tile_entry_ok(b.x, b.y, b.z, b.w, bn, R, E), b.why);
}

void check_sfb_layout() {
  std::vector<int> seen(moe::kSfbTileBytes, 0);
  for (int n = 0; n < 256; ++n) {
    const uint32_t o = moe::sfb_row_offset(n);
    expect(o % 4 == 0 && o + 4 <= static_cast<uint32_t>(moe::kSfbTileBytes), "offset in the block",
           n, o);
    expect((n < 128) == (o < 512), "rows 0..127 in the first 512 bytes", n, o);
    for (int b = 0; b < 4; ++b) ++seen[o + b];
  }
  for (int i = 0; i < moe::kSfbTileBytes; ++i) expect(seen[i] == 1, "every byte used once", i);
}

}  // namespace

int main() {
  check_plan();
  check_bound();
  check_entry_test();
  check_sfb_layout();
  if (failures) {
    std::printf("%d failures\n", failures);
    return 1;
  }
  std::printf("ok\n");
  return 0;
}

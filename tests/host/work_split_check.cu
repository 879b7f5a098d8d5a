// Host-side checks of the work split shared by the attention kernels
// (work_split.cuh): the equal split of W numbered steps over C CTAs, the
// inverse map from a step to its CTA, and the split of the SMs between the
// prefill tile kernel and the decode rows of a mixed batch.  Runs on the CPU
// only; prints "ok" or the first violation.
#include <cstdio>
#include <cstdlib>

#include "work_split.cuh"

using namespace pa;

static int fail(const char* what, long long a, long long b, long long c) {
  std::printf("FAIL %s %lld %lld %lld\n", what, a, b, c);
  return 1;
}

int main() {
  // range_lo / cta_of_tile: contiguous ranges covering [0, W), sizes
  // differing by at most one, cta_of_tile the inverse.
  for (long long W = 0; W <= 400; ++W)
    for (int C = 1; C <= 48; ++C) {
      if (range_lo(W, C, 0) != 0 || range_lo(W, C, C) != W) return fail("ends", W, C, 0);
      long long mn = W, mx = 0;
      for (int c = 0; c < C; ++c) {
        const long long lo = range_lo(W, C, c), hi = range_lo(W, C, c + 1);
        if (hi < lo) return fail("order", W, C, c);
        mn = hi - lo < mn ? hi - lo : mn;
        mx = hi - lo > mx ? hi - lo : mx;
        for (long long t = lo; t < hi; ++t)
          if (cta_of_tile(W, C, t) != c) return fail("inverse", W, C, t);
      }
      if (mx - mn > 1) return fail("balance", W, C, mx - mn);
    }
  // Large totals take the 64-bit division.
  const long long big = (1ll << 40) + 12345;
  for (int C : {1, 7, 152, 456})
    for (int c = 0; c < C; c += (C / 7) + 1) {
      const long long lo = range_lo(big, C, c), hi = range_lo(big, C, c + 1);
      if (cta_of_tile(big, C, lo) != c || cta_of_tile(big, C, hi - 1) != c) return fail("big", C, c, lo);
    }
  // tile_kernel_sms: 0 without tile work, every SM without decode rows or
  // for a large tile batch, else a share in [1, num_sms] that grows with
  // the tile work and shrinks with the decode work.
  for (int sms : {1, 8, 152}) {
    if (tile_kernel_sms(0, 1000, sms, false) != 0) return fail("no tile work", sms, 0, 0);
    if (tile_kernel_sms(1000, 0, sms, false) != sms) return fail("no decode rows", sms, 0, 0);
    if (tile_kernel_sms(kSplitMaxTileNsPerSm * sms / kTileNsPerCost + 1000, 1, sms, false) != sms)
      return fail("large tile batch", sms, 0, 0);
    for (int e4m3 = 0; e4m3 < 2; ++e4m3) {
      int prev = 0;
      for (long long tc = 1; tc < 20000; tc += 97) {
        const int n = tile_kernel_sms(tc, 50000, sms, e4m3 != 0);
        if (n < 1 || n > sms || n < prev) return fail("tile share", sms, tc, n);
        prev = n;
      }
      prev = sms;
      for (long long dt = 1; dt < 400000; dt += 3001) {
        const int n = tile_kernel_sms(5000, dt, sms, e4m3 != 0);
        if (n < 1 || n > sms || n > prev) return fail("decode share", sms, dt, n);
        prev = n;
      }
    }
  }
  // decode_split_ctas: every CTA unless the tiles keep some SMs; then the
  // CTAs of the other SMs, at least one SM's worth.
  for (int sms : {2, 152})
    for (int cps : {1, 3})
      for (int t = -1; t <= sms + 1; ++t) {
        const int n = decode_split_ctas(t, sms, sms * cps, cps);
        const int want = (t <= 0 || t >= sms) ? sms * cps : (sms - t) * cps;
        if (n != want || n < cps) return fail("decode ctas", sms, cps, t);
      }
  // tile_req / tile_req_steps against unit-by-unit sums; decode_row_tiles.
  const RowLimits lim{4096, 70000, 70000, 1 << 20};
  for (int q_len = 0; q_len <= 700; q_len += 13)
    for (int ctx = 0; ctx <= 900; ctx += 37) {
      const TileReq p = tile_req(100, 100 + q_len, ctx + q_len, lim);
      if (q_len <= 1) {
        if (p.ntq != 0) return fail("not prefill rows", q_len, ctx, p.ntq);
        continue;
      }
      long long steps = 0;
      for (int u = 0; u < p.ntq; ++u) {
        const int row0 = (p.ntq - 1 - u) * 128;
        const int rows = q_len - row0 < 128 ? q_len - row0 : 128;
        steps += (ctx + row0 + rows + 127) / 128;
      }
      if (p.ntq != (q_len + 127) / 128 || tile_req_steps(p) != steps) return fail("steps", q_len, ctx, steps);
    }
  if (decode_row_tiles(5, 6, 33, lim) != 3 || decode_row_tiles(5, 7, 33, lim) != 0 ||
      decode_row_tiles(5, 6, 0, lim) != 0 || decode_row_tiles(5, 6, 70001, lim) != 0 ||
      decode_row_tiles(-1, 0, 33, lim) != 0)
    return fail("decode rows", 0, 0, 0);
  std::printf("ok\n");
  return 0;
}

// Host-side check of the decode's range arithmetic (kvq_ranges.h): builds the
// map for one configuration, enumerates the ranges in the order the decode's
// warps run them (static ranges, then tail chunks) and checks that they
// partition the block stream and that range_of / range_start invert the
// enumeration. Compiled with the system C++ compiler by test_range_map.py;
// no GPU involved.
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "kvq_ranges.h"

namespace {

struct Range {
  int64_t lo, hi, id;
};

}  // namespace

// out[0..5] = Pst, C, ntail, k, number of ranges, largest range id + 1.
// Returns 0, or the first failed property: 1 overlap or gap, 2 coverage,
// 3 range_start, 4 range_of, 5 empty range, 6 id beyond the records' room.
extern "C" int kvq_check_range_map(int tail_ok, int64_t max_ranges, int min_blocks, int tb,
                                   int groups, int64_t nwarps, int lockstep, int64_t* out) {
  const int64_t total = static_cast<int64_t>(tb) * groups;
  const int64_t even = (total + nwarps - 1) / nwarps;
  const int P = static_cast<int>(even > min_blocks ? even : min_blocks);
  const kvq::RangeMap m = kvq::make_range_map(tail_ok != 0, max_ranges, min_blocks, total, tb,
                                              groups, nwarps, P, lockstep != 0);
  std::vector<Range> rs;
  if (m.k > 0) {
    for (int64_t gw = 0; gw < static_cast<int64_t>(groups) * m.k; ++gw) {
      const int64_t hgi = gw / m.k, i = gw - hgi * m.k, lo = i * m.Pst;
      if (lo < tb) rs.push_back({hgi * tb + lo, hgi * tb + std::min<int64_t>(tb, lo + m.Pst), gw});
    }
  } else {
    const int64_t static_end = m.C == 0 ? total : nwarps * m.Pst;
    for (int64_t gw = 0; gw < nwarps; ++gw) {
      const int64_t xs = gw * m.Pst;
      if (xs < static_end) rs.push_back({xs, std::min(static_end, xs + m.Pst), gw});
    }
    for (int64_t c = 0; c < m.ntail; ++c) {
      const int64_t x0 = static_end + c * m.C;
      rs.push_back({x0, std::min(total, x0 + m.C), nwarps + c});
    }
  }
  int64_t max_id = -1;
  for (const Range& r : rs) max_id = std::max(max_id, r.id);
  out[0] = m.Pst;
  out[1] = m.C;
  out[2] = m.ntail;
  out[3] = m.k;
  out[4] = static_cast<int64_t>(rs.size());
  out[5] = max_id + 1;
  std::sort(rs.begin(), rs.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
  int64_t at = 0;
  for (const Range& r : rs) {
    if (r.hi <= r.lo) return 5;
    if (r.lo != at) return 1;
    at = r.hi;
    if (kvq::range_start(m, r.id) != r.lo) return 3;
    if (kvq::range_of(m, r.lo) != r.id || kvq::range_of(m, r.hi - 1) != r.id) return 4;
  }
  if (at != total) return 2;
  const int64_t room = m.C > 0 ? max_ranges : nwarps;
  if (max_id >= room) return 6;
  return 0;
}

// The most ranges any (q-head group, request) segment is cut into, for
// requests of nblk[b] blocks (the same in every group).
extern "C" int64_t kvq_max_pieces(int tail_ok, int64_t max_ranges, int min_blocks,
                                  const int32_t* nblk, int batch, int groups, int64_t nwarps,
                                  int lockstep) {
  std::vector<int64_t> cum(batch + 1, 0);
  for (int b = 0; b < batch; ++b) cum[b + 1] = cum[b] + nblk[b];
  const int tb = static_cast<int>(cum[batch]);
  const int64_t total = static_cast<int64_t>(tb) * groups;
  const int64_t even = (total + nwarps - 1) / nwarps;
  const int P = static_cast<int>(even > min_blocks ? even : min_blocks);
  const kvq::RangeMap m = kvq::make_range_map(tail_ok != 0, max_ranges, min_blocks, total, tb,
                                              groups, nwarps, P, lockstep != 0);
  int64_t most = 0;
  for (int h = 0; h < groups; ++h)
    for (int b = 0; b < batch; ++b) {
      if (nblk[b] == 0) continue;
      const int64_t s0 = static_cast<int64_t>(h) * tb + cum[b];
      most = std::max(most, kvq::range_of(m, s0 + nblk[b] - 1) - kvq::range_of(m, s0) + 1);
    }
  return most;
}

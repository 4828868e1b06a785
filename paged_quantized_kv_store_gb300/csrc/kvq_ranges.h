// kvq_ranges.h: how the decode cuts its block stream into ranges (static
// ranges per warp, then tail chunks handed out from a counter), and the maps
// between blocks and range ids that the decode and the combine share. Plain
// C++ so that the host tests can check the arithmetic without a GPU.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define KVQ_HD __host__ __device__ __forceinline__
#else
#define KVQ_HD inline
#endif

namespace kvq {

constexpr int kTailMinShare = 128;  // blocks per warp from which the decode has a tail

KVQ_HD int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
KVQ_HD int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// How the block stream is cut into ranges, each ending in at most two partial
// records per q head. Static part: warp w owns blocks [w Pst, (w + 1) Pst) of
// the first nwarps * Pst. Tail (C > 0): the rest in chunks of C blocks, taken
// one at a time from a counter by whichever warp is free, so that warps whose
// static part ran slower (the co-resident CTAs of an SM do not get equal
// shares of it) are not waited for. Range ids: warps 0 .. nwarps - 1, then
// nwarps + tail chunk.
struct RangeMap {
  int64_t nwarps;
  int Pst;        // blocks per static range
  int C;          // blocks per tail chunk; 0: no tail (static ranges cover all)
  int64_t ntail;  // tail chunks
  // k > 0: the static ranges are laid out per q-head group instead: group
  // hgi's tb blocks are cut into k ranges of Pst (the last one shorter),
  // ranges hgi k .. hgi k + k - 1, the same cut in every group (no tail)
  int k;
  int tb;
};

KVQ_HD int64_t range_of(const RangeMap& m, int64_t x) {
  if (m.k > 0) {
    const int64_t hgi = x / m.tb;
    return hgi * m.k + (x - hgi * m.tb) / m.Pst;
  }
  if (m.C == 0) return x / m.Pst;
  const int64_t ns = m.nwarps * m.Pst;
  return x < ns ? x / m.Pst : m.nwarps + (x - ns) / m.C;
}

KVQ_HD int64_t range_start(const RangeMap& m, int64_t r) {
  if (m.k > 0) return (r / m.k) * m.tb + (r % m.k) * m.Pst;
  if (m.C == 0 || r < m.nwarps) return r * m.Pst;
  return m.nwarps * m.Pst + (r - m.nwarps) * m.C;
}

// Static ranges cut the same way in every q-head group when the grid has at
// least a warp per group: then the warps of different kv heads read the same
// requests' blocks at the same time, and a block's token rows (the kv heads
// side by side) leave DRAM together instead of as scattered 64-256-byte
// pieces. Each group's tb blocks go to k = min(warps / groups, tb / P_min)
// ranges (rounded down, at least 1); the rest of the warps stay idle.
// Measured per kind: INT8 GQA-4 (80 blocks per warp) 6 % faster, bf16 GQA-2
// 1 %, INT4 GQA-4 3 % slower (its decode is bound by in-block latency, not
// DRAM), and nothing to gain for shares under 16 blocks; `lockstep` says
// whether to use it.
KVQ_HD RangeMap static_range_map(int64_t total, int tb, int groups, int64_t nwarps, int P,
                                 int min_blocks, bool lockstep) {
  RangeMap m{nwarps, P, 0, 0, 0, tb};
  if (!lockstep || P < 16 || tb <= 0 || groups > nwarps) return m;
  // k <= tb / P_min keeps every range at least P_min blocks long (an explicit
  // split count bounds the pieces of a request through P_min)
  const int64_t k = min64(nwarps / groups, max64(1, tb / min_blocks));
  m.k = static_cast<int>(k);
  m.Pst = static_cast<int>((tb + k - 1) / k);
  return m;
}

// The map for `total` blocks over `nwarps` warps with per-warp range length P
// (the even share, at least the plan's minimum). A tail needs a counter
// (tail_ok: an automatic split) and P >= kTailMinShare: only long ranges drift apart by
// more than a short chunk, and a chunk pays a pipeline fill and its own
// partial records. It takes about a tenth of the blocks, in at most 4 chunks
// per warp of at least 8 blocks, and is dropped when the workspace holds
// fewer than nwarps + ntail ranges (max_ranges).
KVQ_HD RangeMap make_range_map(bool tail_ok, int64_t max_ranges, int min_blocks, int64_t total,
                               int tb, int groups, int64_t nwarps, int P, bool lockstep) {
  if (!tail_ok || P < kTailMinShare)
    return static_range_map(total, tb, groups, nwarps, P, min_blocks, lockstep);
  RangeMap m{nwarps, P, 0, 0, 0, tb};
  constexpr int c0 = 8;
  const int64_t per = (9 * total) / (10 * nwarps * c0);  // static chunks per warp
  const int64_t rem = total - nwarps * per * c0;
  const int64_t c = max64(c0, (rem + 4 * nwarps - 1) / (4 * nwarps));
  const int64_t ntail = (rem + c - 1) / c;
  if (nwarps + ntail > max_ranges)
    return static_range_map(total, tb, groups, nwarps, P, min_blocks, lockstep);
  m.Pst = static_cast<int>(per * c0);
  m.C = static_cast<int>(c);
  m.ntail = ntail;
  return m;
}

}  // namespace kvq

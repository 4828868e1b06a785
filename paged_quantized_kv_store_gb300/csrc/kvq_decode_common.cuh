// kvq_decode_common.cuh: the part of the decode that does not depend on how a
// block is attended -- the block stream, its cut into ranges, and the
// shared-prefix merge -- used by both decode kernels (kvq_decode.cu and the
// grouped-query kernel in kvq_decode_gqa.cu).
//
// LMDeploy article (devpress.csdn.net) §2.2: per-sequence block tables of
// 16-token blocks. All the work of one decode call is one stream of blocks
// ordered by (q-head group, request, block); a persistent grid gives every
// warp one contiguous range of it (and, for long shares, tail chunks from a
// counter), so the split between warps is exact whatever the mix of request
// lengths.
#pragma once

#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tile.cuh"

namespace kvq {

// Dynamic shared memory: [prefix sums of the blocks per request][slack to a
// 1024-byte boundary][the stage regions of the 4 warps].
template <int KV>
__host__ __device__ constexpr size_t smem_bytes_for(int batch) {
  return align128((batch + 1) * sizeof(int32_t)) + 1024 +
         static_cast<size_t>(kWarps) * Stage<KV>::kWarpBytes;
}

// Clamped length of request b.
__device__ __forceinline__ int clamped_len(const DecodeArgs& a, int b) {
  return min(max(a.seq_lens[b], 0), a.len_cap);
}

// Leading blocks of request b attended by the shared-prefix kernel (0 in a
// plain decode).
__device__ __forceinline__ int skip_of(const DecodeArgs& a, int b) {
  return a.skip != nullptr ? a.skip[b] : 0;
}

// Blocks of request b this kernel reads.
__device__ __forceinline__ int own_blocks(const DecodeArgs& a, int b) {
  return max((clamped_len(a, b) + kBlock - 1) / kBlock - skip_of(a, b), 0);
}

// Merges the shared-prefix records of (request, q head) `row` into a state
// (max m, sum l, unnormalised output acc of the 16 dims [16 g, 16 g + 16)).
__device__ __forceinline__ void merge_prefix(const DecodeArgs& a, int64_t row, int skip, int g,
                                             float& m, float& l, float (&acc)[16]) {
  const int npc = (skip + a.pchunk - 1) / a.pchunk;
  const float* rec0 = a.ppart + row * a.pmax_chunks * kPartStride;
  float M = m;
  for (int c = 0; c < npc; ++c) M = fmaxf(M, rec0[c * kPartStride + kHeadDim]);
  if (M == -INFINITY) return;
  const float al = m == -INFINITY ? 0.f : ex2(m - M);
  l *= al;
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] *= al;
  for (int c = 0; c < npc; ++c) {
    const float* rec = rec0 + c * kPartStride;
    const float mc = rec[kHeadDim];
    const float e = mc == -INFINITY ? 0.f : ex2(mc - M);
    l += e * rec[kHeadDim + 1];
    const float4* v = reinterpret_cast<const float4*>(rec + 16 * g);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 x = v[q];
      acc[4 * q] += e * x.x;
      acc[4 * q + 1] += e * x.y;
      acc[4 * q + 2] += e * x.z;
      acc[4 * q + 3] += e * x.w;
    }
  }
  m = M;
}

// Position in the block stream: q-head group hgi (kv head * head_groups +
// group), request b, block j of nblk.
struct Cursor {
  int hgi, b, j, nblk;
};

__device__ __forceinline__ void locate(Cursor& c, int64_t x, const int32_t* cum, int batch,
                                       int tb) {
  c.hgi = static_cast<int>(x / tb);
  const int r = static_cast<int>(x - static_cast<int64_t>(c.hgi) * tb);
  int lo = 0, hi = batch - 1;  // largest b with cum[b] <= r: the non-empty request holding r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cum[mid] <= r) lo = mid; else hi = mid - 1;
  }
  c.b = lo;
  c.j = r - cum[lo];
  c.nblk = cum[lo + 1] - cum[lo];
}

// Next block of the stream (the caller knows there is one).
__device__ __forceinline__ void advance(Cursor& c, const int32_t* cum, int batch) {
  if (++c.j < c.nblk) return;
  c.j = 0;
  do {
    if (++c.b == batch) {
      c.b = 0;
      ++c.hgi;
    }
    c.nblk = cum[c.b + 1] - cum[c.b];
  } while (c.nblk == 0);
}

// The block stream of one call as every CTA sees it after its prologue.
struct StreamPlan {
  const int32_t* cum;      // [batch + 1] blocks before request b (shared memory)
  unsigned char* stages;   // the warps' stage regions follow (shared memory)
  int tb;                  // blocks of one q-head group over all requests
  int groups;              // q-head groups (kv heads x head groups)
  int64_t total;           // blocks in the stream
  int64_t nwarps;          // ranges of the static cut (warps, or CTAs, of the grid)
  int64_t static_end;      // end of the static ranges (the tail follows)
  RangeMap rm;
};

// Prologue of every decode CTA: the per-request block counts prefix-summed
// into shared memory (own_lens: followed by each request's own tokens, its
// clamped length less the shared blocks), the cut of the stream into ranges
// (TAIL: the map that can hand out tail chunks; `lockstep`: static ranges
// cut per q-head group where that pays), and, by CTA 0, the header the
// combine kernel reads and the all-zero rows of empty requests (a request
// whose only blocks are shared ones is written by the combine kernel).
// The CTA has blockDim.x threads (at most 8 warps: warp_sum holds one int per
// warp) and owns ranges_per_cta ranges of the stream (one per warp, or one).
template <bool QBF, bool TAIL>
__device__ __forceinline__ StreamPlan plan_stream(const DecodeArgs& a, unsigned char* dsmem,
                                                  int32_t* warp_sum, int cta, int ncta,
                                                  bool lockstep, bool own_lens = false,
                                                  int ranges_per_cta = kWarps) {
  int32_t* cum = reinterpret_cast<int32_t*>(dsmem);
  int32_t* lown = cum + a.batch + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nt = blockDim.x;
  {
    const int per = (a.batch + nt - 1) / nt;
    const int b0 = min(tid * per, a.batch), b1 = min(b0 + per, a.batch);
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
      sum += own_blocks(a, b);
      if (cta == 0 && a.seq_lens[b] > a.len_cap) report(a.dev_err, KVQ_DEV_ERR_LENGTH);
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_sum[w];
    int run = base + incl - sum;
    for (int b = b0; b < b1; ++b) {
      cum[b] = run;
      run += own_blocks(a, b);
      if (own_lens) lown[b] = clamped_len(a, b) - kBlock * skip_of(a, b);
    }
    if (tid == nt - 1) cum[a.batch] = base + incl;
    __syncthreads();
  }
  StreamPlan sp;
  sp.cum = cum;
  sp.stages = dsmem + align128(((own_lens ? 2 : 1) * a.batch + 1) * sizeof(int32_t));
  sp.tb = cum[a.batch];
  sp.groups = a.cta_heads > 0 ? a.kv_heads / a.cta_heads : a.kv_heads * a.head_groups;
  sp.total = static_cast<int64_t>(sp.tb) * sp.groups;
  sp.nwarps = static_cast<int64_t>(ncta) * ranges_per_cta;  // ranges of the static cut
  const int64_t even_share = (sp.total + sp.nwarps - 1) / sp.nwarps;
  const int P = static_cast<int>(even_share > a.min_blocks_per_warp ? even_share
                                                                    : a.min_blocks_per_warp);
  sp.rm = TAIL ? make_range_map(a.tail_ctr != nullptr, a.max_ranges, a.min_blocks_per_warp,
                                sp.total, sp.tb, sp.groups, sp.nwarps, P, lockstep)
               : static_range_map(sp.total, sp.tb, sp.groups, sp.nwarps, P,
                                  a.min_blocks_per_warp, lockstep);
  sp.static_end = sp.rm.C == 0 ? sp.total : sp.nwarps * sp.rm.Pst;
  if (cta == 0) {
    if (tid == 0) {
      a.hdr[0] = sp.tb;
      a.hdr[1] = sp.rm.Pst;
      a.hdr[2] = sp.rm.C;
      a.hdr[3] = static_cast<int32_t>(sp.nwarps);
      a.hdr[4] = sp.rm.k;
    }
    for (int b = tid; b <= a.batch; b += nt) a.hdr[kHdrCum + b] = cum[b];
    for (int b = 0; b < a.batch; ++b) {
      if (cum[b + 1] != cum[b] || skip_of(a, b) > 0) continue;
      for (int e = tid; e < a.q_heads * kHeadDim; e += nt)
        store_out<QBF>(a.out, static_cast<int64_t>(b) * a.q_heads * kHeadDim + e, 0.f);
    }
  }
  return sp;
}

// Runs warp gw's ranges: its static range (or its share of the per-group
// cut), then, with a tail, chunks taken from the counter while there are
// any. run_range(x0, n, rid) attends blocks [x0, x0 + n) of the stream and
// files its records under range id rid; it returns false when a copy timed
// out, and the warp stops.
template <bool TAIL, class F>
__device__ __forceinline__ void for_each_range(const DecodeArgs& a, const StreamPlan& sp,
                                               int64_t gw, int lane, F&& run_range) {
  const RangeMap& rm = sp.rm;
  if (rm.k > 0) {  // the same cut in every q-head group
    if (gw >= static_cast<int64_t>(sp.groups) * rm.k) return;
    const int64_t hgi = gw / rm.k, i = gw - hgi * rm.k;
    const int64_t lo = i * rm.Pst;
    if (lo < sp.tb)
      run_range(hgi * sp.tb + lo,
                static_cast<int>(min(sp.tb - lo, static_cast<int64_t>(rm.Pst))), gw);
    return;
  }
  const int64_t xs = gw * rm.Pst;
  if (xs < sp.static_end &&
      !run_range(xs, static_cast<int>(min(sp.static_end - xs, static_cast<int64_t>(rm.Pst))),
                 gw))
    return;
  if constexpr (TAIL) {
    if (rm.C == 0) return;
    for (;;) {
      unsigned int c = 0;
      if (lane == 0) c = atomicAdd(a.tail_ctr, 1u);
      c = __shfl_sync(kFull, c, 0);
      if (c >= rm.ntail) return;
      const int64_t x0 = sp.static_end + static_cast<int64_t>(c) * rm.C;
      if (!run_range(x0, static_cast<int>(min(sp.total - x0, static_cast<int64_t>(rm.C))),
                     sp.nwarps + c))
        return;
    }
  }
}

}  // namespace kvq

// kvq_prefix: the shared-prefix half of a cascade decode step.
//
// "pymllm Runtime Design", section "KV cache 与 prefix cache": with the radix
// prefix cache, the matched prefix of a new request is not recomputed; its KV
// slots are the ones already in the pool. LMDeploy article (devpress.csdn.net)
// §2.2: sequences of different lengths can share physical blocks (prefix
// caching). In a decode step every member of such a group attends the same
// blocks, so this kernel reads each shared block once per group and kv head
// and multiplies it with the queries of all members at once:
//   S = Q K^T   mma.m16n8k16 with M = 16 queries (members x q heads of the kv
//               head), N = 8 tokens (2 tiles per block), K = 128 dims;
//   O += P' V   M = 16 queries, N = 8 dims (16 tiles), K = 16 tokens.
// The K and V fragments are the decode kernel's (kvq_tile.cuh): the K operand
// registers of S^T = K Q^T are exactly the B operand of S = Q K^T, the V^T
// operand registers of O^T = V^T P'^T the B operand of O = P' V, and the
// scores' accumulator layout is the A operand layout of P', so nothing is
// transposed. Code offsets and the deferred scale/zero are as in the decode
// kernel.
//
// A work unit is (group, kv head, chunk of up to 32 shared blocks, tile of 16
// queries); it leaves one partial record (max, sum, unnormalised output, exp2
// domain) per query and chunk. The decode kernel merges the records of the
// requests a single warp covers; the combine kernel those of the others.
// Every CTA first scans the groups' unit counts. The units of kv head 0 also
// check their members (in range and listed once, shared blocks identical in
// every member's table, no member shorter than the shared part) and write the
// per-request count of shared blocks that the decode kernel skips.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tile.cuh"

namespace kvq {
namespace {

// [unit prefix sums per group][slack to a 1024-byte boundary][stage regions]
template <int KV>
__host__ __device__ constexpr size_t prefix_smem_bytes(int num_groups) {
  return align128((num_groups + 1) * sizeof(int32_t)) + 1024 +
         static_cast<size_t>(kWarps) * Stage<KV>::kWarpBytes;
}

struct GroupShape {
  int off, members, sb, tiles, chunks;
  bool ok;
};

// Shape of group G; ok is false (and the group does no work) when its member
// range lies outside grp_mem.
__device__ __forceinline__ GroupShape group_shape(const DecodeArgs& a, int G) {
  GroupShape s;
  s.off = a.grp_off[G];
  const int end = a.grp_off[G + 1];
  s.ok = s.off >= 0 && end >= s.off && end <= a.num_members;
  s.members = s.ok ? end - s.off : 0;
  s.sb = min(max(a.grp_shared[G], 0), a.max_shared);
  s.tiles = (s.members * a.group + 15) / 16;
  s.chunks = (s.sb + a.pchunk - 1) / a.pchunk;
  return s;
}

// Q fragments of one query row (this lane's 32 dims, permuted like the K
// dims) and its sum; zeros when the row is padding.
template <int KV, bool QBF>
__device__ __forceinline__ float load_q_row(const DecodeArgs& a, int b, int hq, bool valid, int t,
                                            uint32_t (&qr)[8][2]) {
  uint32_t qw[16];
  if (valid) {
    const uint4* qp = reinterpret_cast<const uint4*>(
        static_cast<const uint16_t*>(a.q) + (static_cast<int64_t>(b) * a.q_heads + hq) * kHeadDim +
        32 * t);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = qp[i];
      qw[4 * i] = v.x; qw[4 * i + 1] = v.y; qw[4 * i + 2] = v.z; qw[4 * i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) qw[i] = 0u;
  }
  if constexpr (KV == kI4) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int j = kk >> 1, u = kk & 1;
      qr[kk][0] = prmt(qw[4 * j + u], qw[4 * j + u + 2], 0x5410u);
      qr[kk][1] = prmt(qw[4 * j + u], qw[4 * j + u + 2], 0x7632u);
    }
  } else {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qr[kk][0] = qw[2 * kk];
      qr[kk][1] = qw[2 * kk + 1];
    }
  }
  float sum = 0.f;
  if constexpr (KvTraits<KV>::kQuant) {
#pragma unroll
    for (int i = 0; i < 16; ++i) sum += lo_to_float<QBF>(qw[i]) + hi_to_float<QBF>(qw[i]);
    sum += __shfl_xor_sync(kFull, sum, 1);
    sum += __shfl_xor_sync(kFull, sum, 2);
  }
  return sum;
}

template <int KV, bool QBF>
__global__ void __launch_bounds__(kDecodeThreads)
    prefix_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  __shared__ int32_t warp_sum[kWarps];
  using S = Stage<KV>;
  constexpr bool kQuant = KvTraits<KV>::kQuant;
  constexpr bool kPvBf = KV == kBF16;
  constexpr float kAk = CodeOffset<KV, QBF>::kK;
  constexpr float kAv = CodeOffset<KV, QBF>::kV;
  constexpr float kMid = CodeOffset<KV, QBF>::kMid;
  constexpr bool kPCorr = CodeOffset<KV, QBF>::kPCorr;
  constexpr int D = S::kDepth;

  int32_t* ucum = reinterpret_cast<int32_t*>(dsmem);  // [num_groups + 1]: units before group G
  unsigned char* stages = dsmem + align128((a.num_groups + 1) * sizeof(int32_t));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;

  // ---- work units per group, prefix-summed (every CTA) --------------------------
  {
    const int per = (a.num_groups + kDecodeThreads - 1) / kDecodeThreads;
    const int g0 = min(tid * per, a.num_groups), g1 = min(g0 + per, a.num_groups);
    int sum = 0;
    for (int G = g0; G < g1; ++G) {
      const GroupShape s = group_shape(a, G);
      sum += a.kv_heads * s.tiles * s.chunks;
      if (blockIdx.x == 0 && (!s.ok || a.grp_shared[G] > a.max_shared))
        report(a.dev_err, KVQ_DEV_ERR_PREFIX);
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
    for (int G = g0; G < g1; ++G) {
      ucum[G] = run;
      const GroupShape s = group_shape(a, G);
      run += a.kv_heads * s.tiles * s.chunks;
    }
    if (tid == kDecodeThreads - 1) ucum[a.num_groups] = base + incl;
    __syncthreads();
  }

  // ---- work units ------------------------------------------------------------------
  const int total = ucum[a.num_groups];
  const int nwarps = gridDim.x * kWarps;
  int u = blockIdx.x * kWarps + warp;
  if (u >= total) return;  // no block barrier follows
  const uint32_t region0 =
      (static_cast<uint32_t>(__cvta_generic_to_shared(stages)) + 1023u) & ~1023u;
  const uint32_t wr = region0 + static_cast<uint32_t>(warp * S::kWarpBytes);
  LaneMap<KV> lm;
  lm.init(lane, g, t, static_cast<uint32_t>(a.kv_heads * S::kRow));
  if constexpr (S::kTma) {
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < D; ++i) mbar_init(wr + S::kBarOff + 8 * i);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
  }
  uint32_t phase = 0;  // parity to wait for, per stage (TMA path)

  for (; u < total; u += nwarps) {
    int lo = 0, hi = a.num_groups - 1;  // largest G with ucum[G] <= u: a group with work
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ucum[mid] <= u) lo = mid; else hi = mid - 1;
    }
    const int G = lo;
    const GroupShape s = group_shape(a, G);
    const int r = u - ucum[G];
    const int qt = r % s.tiles;
    const int rest = r / s.tiles;
    const int c = rest % s.chunks;
    const int h = rest / s.chunks;
    const int lead = a.grp_mem[s.off];
    const int j0 = c * a.pchunk;
    const int n = min(a.pchunk, s.sb - j0);
    if (h == 0) {
      // checks, spread over the units of kv head 0: the unit of chunk c checks
      // the chunk's table entries of the members whose first query row is in
      // its tile; chunk 0's unit also records their shared block count
      const int i0 = (16 * qt + a.group - 1) / a.group;
      const int i1 = min(s.members, (16 * qt + 16 + a.group - 1) / a.group);
      const int per = n + (c == 0 ? 1 : 0);
      for (int e = lane; e < (i1 - i0) * per; e += 32) {
        const int i = i0 + e / per, k = e % per;
        const int b = a.grp_mem[s.off + i];
        uint32_t err = 0;
        if (b < 0 || b >= a.batch || lead < 0 || lead >= a.batch) {
          err = KVQ_DEV_ERR_PREFIX;
        } else if (k == n) {
          if (atomicExch(&a.skip[b], s.sb) != 0) err = KVQ_DEV_ERR_PREFIX;  // listed twice
          if (min(a.seq_lens[b], a.len_cap) < s.sb * kBlock) err = KVQ_DEV_ERR_PREFIX;
        } else if (a.block_tables[static_cast<int64_t>(b) * a.max_blocks + j0 + k] !=
                   a.block_tables[static_cast<int64_t>(lead) * a.max_blocks + j0 + k]) {
          err = KVQ_DEV_ERR_PREFIX;
        }
        report(a.dev_err, err);
      }
    }
    if (lead < 0 || lead >= a.batch) continue;

    // the two query rows of this lane: g and g + 8 of the tile
    const int nq = s.members * a.group;
    int qb_[2], qh_[2];
    bool qv_[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int i = 16 * qt + g + 8 * rr;
      qv_[rr] = i < nq;
      qb_[rr] = qv_[rr] ? a.grp_mem[s.off + i / a.group] : 0;
      qh_[rr] = h * a.group + (qv_[rr] ? i % a.group : 0);
      qv_[rr] = qv_[rr] && qb_[rr] >= 0 && qb_[rr] < a.batch;
    }
    uint32_t qa[8][4];
    float qs0, qs1;
    {
      uint32_t q0[8][2], q1[8][2];
      qs0 = load_q_row<KV, QBF>(a, qb_[0], qh_[0], qv_[0], t, q0);
      qs1 = load_q_row<KV, QBF>(a, qb_[1], qh_[1], qv_[1], t, q1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa[kk][0] = q0[kk][0];
        qa[kk][1] = q1[kk][0];
        qa[kk][2] = q0[kk][1];
        qa[kk][3] = q1[kk][1];
      }
    }

    // block ids of the chunk (the leader's table; every member's is the same)
    const int32_t win =
        lane < n ? a.block_tables[static_cast<int64_t>(lead) * a.max_blocks + j0 + lane] : -1;
    uint32_t ok_mask = 0;
    int k_issue = 0, st_issue = 0;
    auto issue_next = [&]() {
      if (k_issue < n) {
        const int32_t phys = __shfl_sync(kFull, win, k_issue);
        const uint32_t bit = 1u << st_issue;
        if (phys >= 0 && phys < a.num_blocks) {
          issue_block<KV>(wr, st_issue, a, lm, phys, h, lane);
          ok_mask |= bit;
        } else {
          ok_mask &= ~bit;
          if (lane == 0) report(a.dev_err, KVQ_DEV_ERR_BLOCK_ID);
        }
      }
      if constexpr (!S::kTma) cp_async_commit();
      ++k_issue;
      st_issue = st_issue == D - 1 ? 0 : st_issue + 1;
    };
#pragma unroll
    for (int k = 0; k < D - 1; ++k) issue_next();

    float o[16][4];
#pragma unroll
    for (int d = 0; d < 16; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;
    float r0 = 0.f, r1 = 0.f;

    int st = 0;
    for (int k = 0; k < n; ++k) {
      issue_next();
      const bool blk_ok = (ok_mask >> st) & 1u;
      if constexpr (S::kTma) {
        if (blk_ok) {
          if (!mbar_wait(wr + S::kBarOff + 8 * st, (phase >> st) & 1u)) {
            if (lane == 0) report(a.dev_err, KVQ_DEV_ERR_TIMEOUT);
            const uint32_t rest_mask = ok_mask & ~(1u << st);
            for (int i = 0; i < D; ++i)
              if ((rest_mask >> i) & 1u) mbar_wait(wr + S::kBarOff + 8 * i, (phase >> i) & 1u);
            return;
          }
          phase ^= 1u << st;
        }
      } else {
        cp_async_wait<D - 1>();
        __syncwarp();
      }
      if (blk_ok) {
        ok_mask &= ~(1u << st);
        Frag<KV> cur;
        read_frag<KV, false>(cur, wr, st, lm, g);
        // scale/zero words of tokens 2t, 2t+1 (n-tile 0) and 2t+8, 2t+9 (n-tile 1)
        uint2 ksz0, ksz1, vsz0, vsz1;
        if constexpr (kQuant) {
          const uint32_t sz = wr + S::kSzOff + 128 * st + 8 * t;
          ksz0 = lds64(sz);
          ksz1 = lds64(sz + 32);
          vsz0 = lds64(sz + 64);
          vsz1 = lds64(sz + 96);
        }
        // S = Q K^T: [n-tile][query g: tokens 2t, 2t+1 | query g+8: same]
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t ak[4];
          k_operand<KV, QBF>(cur, kk, ak);
          const uint32_t b0[2] = {ak[0], ak[2]}, b1[2] = {ak[1], ak[3]};
          mma16816<QBF>(sc[0], qa[kk], b0);
          mma16816<QBF>(sc[1], qa[kk], b1);
        }
        // scores in the exp2 domain
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          if constexpr (kQuant) {
            const uint2 w = nt ? ksz1 : ksz0;
            const float Sa = half_lo(w.x), Za = half_hi(w.x) - kAk * Sa;
            const float Sb = half_lo(w.y), Zb = half_hi(w.y) - kAk * Sb;
            sc[nt][0] = (Sa * sc[nt][0] + Za * qs0) * a.sm_scale_log2;
            sc[nt][1] = (Sb * sc[nt][1] + Zb * qs0) * a.sm_scale_log2;
            sc[nt][2] = (Sa * sc[nt][2] + Za * qs1) * a.sm_scale_log2;
            sc[nt][3] = (Sb * sc[nt][3] + Zb * qs1) * a.sm_scale_log2;
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[nt][e] *= a.sm_scale_log2;
          }
        }
        // running maximum per query row, moved only when a score exceeds it
        float bm0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        float bm1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        float mn0 = m0, mn1 = m1;
        if (__any_sync(kFull, bm0 > m0 || bm1 > m1)) {
          bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, 1));
          bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, 1));
          bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, 2));
          bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, 2));
          mn0 = fmaxf(m0, bm0);
          mn1 = fmaxf(m1, bm1);
          const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
          l0 *= al0; l1 *= al1;
          z0 *= al0; z1 *= al1;
          r0 *= al0; r1 *= al1;
#pragma unroll
          for (int d = 0; d < 16; ++d) {
            o[d][0] *= al0; o[d][1] *= al0;
            o[d][2] *= al1; o[d][3] *= al1;
          }
        }
        m0 = mn0;
        m1 = mn1;
        float p[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          p[nt][0] = ex2(sc[nt][0] - mn0);
          p[nt][1] = ex2(sc[nt][1] - mn0);
          p[nt][2] = ex2(sc[nt][2] - mn1);
          p[nt][3] = ex2(sc[nt][3] - mn1);
          l0 += p[nt][0] + p[nt][1];
          l1 += p[nt][2] + p[nt][3];
        }
        if constexpr (kQuant) {
          // P' = p S_v; sum p (Z_v + mid S_v) kept apart (as in the decode kernel)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint2 w = nt ? vsz1 : vsz0;
            const float Sa = half_lo(w.x), Za = half_hi(w.x) + kMid * Sa;
            const float Sb = half_lo(w.y), Zb = half_hi(w.y) + kMid * Sb;
            z0 += p[nt][0] * Za + p[nt][1] * Zb;
            z1 += p[nt][2] * Za + p[nt][3] * Zb;
            p[nt][0] *= Sa; p[nt][1] *= Sb;
            p[nt][2] *= Sa; p[nt][3] *= Sb;
          }
        }
        // P' as the A operand: rows g (a0, a2) and g + 8 (a1, a3)
        uint32_t pa[4], pa_lo[4];
        pa[0] = pack2<kPvBf>(p[0][0], p[0][1]);
        pa[1] = pack2<kPvBf>(p[0][2], p[0][3]);
        pa[2] = pack2<kPvBf>(p[1][0], p[1][1]);
        pa[3] = pack2<kPvBf>(p[1][2], p[1][3]);
        if constexpr (kPCorr) {
          r0 += lo_to_float<false>(pa[0]) + hi_to_float<false>(pa[0]) +
                lo_to_float<false>(pa[2]) + hi_to_float<false>(pa[2]);
          r1 += lo_to_float<false>(pa[1]) + hi_to_float<false>(pa[1]) +
                lo_to_float<false>(pa[3]) + hi_to_float<false>(pa[3]);
        }
        if constexpr (kPvBf) {
          pa_lo[0] = pack2<true>(p[0][0] - lo_to_float<true>(pa[0]),
                                 p[0][1] - hi_to_float<true>(pa[0]));
          pa_lo[1] = pack2<true>(p[0][2] - lo_to_float<true>(pa[1]),
                                 p[0][3] - hi_to_float<true>(pa[1]));
          pa_lo[2] = pack2<true>(p[1][0] - lo_to_float<true>(pa[2]),
                                 p[1][1] - hi_to_float<true>(pa[2]));
          pa_lo[3] = pack2<true>(p[1][2] - lo_to_float<true>(pa[3]),
                                 p[1][3] - hi_to_float<true>(pa[3]));
        }
        // O += P' V: dim tiles 2i and 2i + 1 from the V fragment of step i
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t av[4];
          v_operand<KV>(cur, i, av);
          const uint32_t b0[2] = {av[0], av[2]}, b1[2] = {av[1], av[3]};
          mma16816<kPvBf>(o[2 * i], pa, b0);
          mma16816<kPvBf>(o[2 * i + 1], pa, b1);
          if constexpr (kPvBf) {
            mma16816<true>(o[2 * i], pa_lo, b0);
            mma16816<true>(o[2 * i + 1], pa_lo, b1);
          }
        }
      }
      __syncwarp();
      st = st == D - 1 ? 0 : st + 1;
    }
    // every block issued was consumed: the next unit restarts the ring at
    // stage 0, and each stage's TMA phase parity carries over (every armed
    // stage was waited for exactly once)
    if constexpr (!S::kTma) cp_async_wait<0>();

    // ---- the records of rows g and g + 8 ----------------------------------------
    l0 += __shfl_xor_sync(kFull, l0, 1);
    l1 += __shfl_xor_sync(kFull, l1, 1);
    l0 += __shfl_xor_sync(kFull, l0, 2);
    l1 += __shfl_xor_sync(kFull, l1, 2);
    if constexpr (kQuant) {
      z0 += __shfl_xor_sync(kFull, z0, 1);
      z1 += __shfl_xor_sync(kFull, z1, 1);
      z0 += __shfl_xor_sync(kFull, z0, 2);
      z1 += __shfl_xor_sync(kFull, z1, 2);
      if constexpr (kPCorr) {
        r0 += __shfl_xor_sync(kFull, r0, 1);
        r1 += __shfl_xor_sync(kFull, r1, 1);
        r0 += __shfl_xor_sync(kFull, r0, 2);
        r1 += __shfl_xor_sync(kFull, r1, 2);
        z0 -= (kAv + kMid) * r0;
        z1 -= (kAv + kMid) * r1;
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      if (!qv_[rr]) continue;
      const float z = rr ? z1 : z0;
      float* rec = a.ppart + ((static_cast<int64_t>(qb_[rr]) * a.q_heads + qh_[rr]) *
                                  a.pmax_chunks + c) * kPartStride;
      // dims 32t + d (accumulator column 2t of dim tile d) and 32t + 16 + d
      float4* lo4 = reinterpret_cast<float4*>(rec + 32 * t);
      float4* hi4 = reinterpret_cast<float4*>(rec + 32 * t + 16);
#pragma unroll
      for (int d = 0; d < 16; d += 4) {
        lo4[d / 4] = make_float4(o[d][2 * rr] + z, o[d + 1][2 * rr] + z, o[d + 2][2 * rr] + z,
                                 o[d + 3][2 * rr] + z);
        hi4[d / 4] = make_float4(o[d][2 * rr + 1] + z, o[d + 1][2 * rr + 1] + z,
                                 o[d + 2][2 * rr + 1] + z, o[d + 3][2 * rr + 1] + z);
      }
      if (t == 0) {
        rec[kHeadDim] = rr ? m1 : m0;
        rec[kHeadDim + 1] = rr ? l1 : l0;
      }
    }
  }
}

template <int KV, bool QBF>
cudaError_t launch_t(const DecodeArgs& a, int grid, cudaStream_t s) {
  thread_local int opted_in_device = -1;  // per host thread: no shared state
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (opted_in_device != dev) {
    e = cudaFuncSetAttribute(prefix_kernel<KV, QBF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(prefix_smem_bytes<KV>(kMaxBatch)));
    if (e != cudaSuccess) return e;
    opted_in_device = dev;
  }
  prefix_kernel<KV, QBF><<<grid, kDecodeThreads, prefix_smem_bytes<KV>(a.num_groups), s>>>(a);
  return cudaGetLastError();
}

template <int KV, bool QBF>
int occupancy_t(int num_groups) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  // cached: a captured step (CUDA graph) repeats the call without new queries
  thread_local int cached_dev = -1, cached_groups = -1, cached_n = 0;
  if (dev == cached_dev && num_groups == cached_groups) return cached_n;
  if (cudaFuncSetAttribute(prefix_kernel<KV, QBF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(prefix_smem_bytes<KV>(kMaxBatch))) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prefix_kernel<KV, QBF>, kDecodeThreads,
                                                    prefix_smem_bytes<KV>(num_groups)) !=
      cudaSuccess)
    return 0;
  cached_dev = dev;
  cached_groups = num_groups;
  cached_n = n;
  return n;
}

}  // namespace

cudaError_t launch_prefix(const DecodeArgs& a, int kv_dtype, int q_dtype, int grid,
                          cudaStream_t s) {
  const bool qbf = q_dtype == kBF16;
  switch (kv_dtype) {
    case kF16:
      return launch_t<kF16, false>(a, grid, s);
    case kBF16:
      return launch_t<kBF16, true>(a, grid, s);
    case kI8:
      return qbf ? launch_t<kI8, true>(a, grid, s) : launch_t<kI8, false>(a, grid, s);
    case kI4:
      return qbf ? launch_t<kI4, true>(a, grid, s) : launch_t<kI4, false>(a, grid, s);
    default:
      return cudaErrorInvalidValue;
  }
}

int prefix_ctas_per_sm(int kv_dtype, int q_dtype, int num_groups) {
  const bool qbf = q_dtype == kBF16;
  switch (kv_dtype) {
    case kF16: return occupancy_t<kF16, false>(num_groups);
    case kBF16: return occupancy_t<kBF16, true>(num_groups);
    case kI8: return qbf ? occupancy_t<kI8, true>(num_groups) : occupancy_t<kI8, false>(num_groups);
    case kI4: return qbf ? occupancy_t<kI4, true>(num_groups) : occupancy_t<kI4, false>(num_groups);
    default: return 0;
  }
}

}  // namespace kvq

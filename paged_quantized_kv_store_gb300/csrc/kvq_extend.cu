// kvq_extend: extend (chunked prefill) attention over the paged, quantized pool.
//
// "pymllm Runtime Design", forward stage: an extend / prefill batch writes its
// prompt tokens into the KV cache and attends over them. LMDeploy article
// §2.3 "动态拆分与融合": a prefill longer than the 4096-token threshold is
// split into chunks prefilled in turn, so a chunk's queries attend the
// request's cached prefix and, causally, the chunk itself; §2.2 / §3.2 item 3:
// the KV is read through the block table.
//
// Request b holds kv_lens[b] tokens; its last C_b = qo_indptr[b+1] -
// qo_indptr[b] are the chunk, whose query i sits at position kv_lens[b] - C_b
// + i and attends positions 0 .. that position. The rows of the computation
// are (query, q head) pairs of one kv head, row = i * group + head, so all q
// heads of a kv head share every K/V block read. A work unit is (request, kv
// head, tile of 16 rows, part of the context); the per-block arithmetic is the
// shared-prefix kernel's (kvq_prefix.cu): S = Q K^T and O += P' V on
// mma.m16n8k16 with the 16 rows as M, the decode kernel's K/V fragments as B
// operands, scale/zero applied outside the products. Scores past a row's
// position are masked. Units are handed out by an atomic counter, longest
// tiles first. When the batch has too few tiles to fill the device, the
// context is cut into parts (pchunk blocks each) whose partial records a
// combine kernel merges; otherwise every unit writes its rows' outputs.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tile.cuh"

namespace kvq {
namespace {

// [unit prefix sums per request][slack to a 1024-byte boundary][stage regions]
template <int KV>
__host__ __device__ constexpr size_t extend_smem_bytes(int batch) {
  return align128((batch + 1) * sizeof(int32_t)) + 1024 +
         static_cast<size_t>(kWarps) * Stage<KV>::kWarpBytes;
}

struct ReqShape {
  int q0, C, L, tiles, splits;
  bool ok;
};

// Shape of request b. A request whose query rows fall outside [0, total_q),
// whose chunk is longer than its context, or whose context exceeds the
// table or the caller's bound, does no work (ok = false; reported by the
// scan).
__device__ __forceinline__ ReqShape req_shape(const ExtendArgs& a, int b) {
  ReqShape s;
  s.q0 = a.qo_indptr[b];
  const int q1 = a.qo_indptr[b + 1];
  s.C = q1 - s.q0;
  s.L = a.kv_lens[b];
  s.ok = s.q0 >= 0 && s.C >= 0 && q1 <= a.total_q && s.L >= s.C && s.L <= a.len_cap;
  if (!s.ok) {
    s.C = 0;
    s.L = 0;
  }
  s.tiles = (s.C * a.group + 15) / 16;
  const int nblk = (s.L + kBlock - 1) / kBlock;
  s.splits = a.pchunk > 0 ? max((nblk + a.pchunk - 1) / a.pchunk, 1) : 1;
  return s;
}

// Q fragments of one row (this lane's 32 dims, permuted like the K dims) and
// its sum; zeros for a padding row.
template <int KV, bool QBF>
__device__ __forceinline__ float load_q(const ExtendArgs& a, int64_t qrow, int hq, bool valid,
                                        int t, uint32_t (&qr)[8][2]) {
  uint32_t qw[16];
  if (valid) {
    const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                     (qrow * a.q_heads + hq) * kHeadDim + 32 * t);
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
    extend_kernel(const __grid_constant__ ExtendArgs a) {
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

  int32_t* ucum = reinterpret_cast<int32_t*>(dsmem);  // [batch + 1]: units before request b
  unsigned char* stages = dsmem + align128((a.batch + 1) * sizeof(int32_t));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;

  // ---- work units per request, prefix-summed (every CTA) ------------------------
  {
    const int per = (a.batch + kDecodeThreads - 1) / kDecodeThreads;
    const int b0 = min(tid * per, a.batch), b1 = min(b0 + per, a.batch);
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
      const ReqShape s = req_shape(a, b);
      sum += a.kv_heads * s.tiles * s.splits;
      if (blockIdx.x == 0 && !s.ok) report(a.dev_err, KVQ_DEV_ERR_LENGTH);
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
      ucum[b] = run;
      const ReqShape s = req_shape(a, b);
      run += a.kv_heads * s.tiles * s.splits;
    }
    if (tid == kDecodeThreads - 1) ucum[a.batch] = base + incl;
    __syncthreads();
  }
  const int total = ucum[a.batch];

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

  for (;;) {
    int u = 0;
    if (lane == 0) u = atomicAdd(a.counter, 1);
    u = __shfl_sync(kFull, u, 0);
    if (u >= total) break;
    int lo = 0, hi = a.batch - 1;  // largest b with ucum[b] <= u: a request with work
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ucum[mid] <= u) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const ReqShape s = req_shape(a, b);
    int r = u - ucum[b];
    const int c = r % s.splits;
    r /= s.splits;
    const int h = r % a.kv_heads;
    const int qt = s.tiles - 1 - r / a.kv_heads;  // the longest tiles first

    // rows g and g + 8 of the tile: (query i, q head h * group + hh)
    int qi[2], qh[2], pos[2];
    bool qv[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = 16 * qt + g + 8 * rr;
      qi[rr] = row / a.group;
      qh[rr] = h * a.group + row % a.group;
      qv[rr] = qi[rr] < s.C;
      pos[rr] = s.L - s.C + qi[rr];
    }
    const int i_max = min(s.C - 1, (16 * qt + 15) / a.group);
    const int nblk_tile = (s.L - s.C + i_max) / kBlock + 1;
    const int j_begin = a.pchunk > 0 ? c * a.pchunk : 0;
    const int j_end = a.pchunk > 0 ? min(j_begin + a.pchunk, nblk_tile) : nblk_tile;
    const int n = max(j_end - j_begin, 0);

    uint32_t qa[8][4];
    float qs0, qs1;
    {
      uint32_t q0[8][2], q1[8][2];
      qs0 = load_q<KV, QBF>(a, s.q0 + qi[0], qh[0], qv[0], t, q0);
      qs1 = load_q<KV, QBF>(a, s.q0 + qi[1], qh[1], qv[1], t, q1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa[kk][0] = q0[kk][0];
        qa[kk][1] = q1[kk][0];
        qa[kk][2] = q0[kk][1];
        qa[kk][3] = q1[kk][1];
      }
    }

    const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks;
    int32_t win = -1;  // block ids j_begin + 32 w .. + 31 of the table, one per lane
    uint32_t ok_mask = 0;
    int k_issue = 0, st_issue = 0;
    auto issue_next = [&]() {
      if (k_issue < n) {
        if ((k_issue & 31) == 0) {
          const int jj = j_begin + k_issue + lane;
          win = jj < j_end ? bt[jj] : -1;
        }
        const int32_t phys = __shfl_sync(kFull, win, k_issue & 31);
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
        uint2 ksz0, ksz1, vsz0, vsz1;
        if constexpr (kQuant) {
          const uint32_t sz = wr + S::kSzOff + 128 * st + 8 * t;
          ksz0 = lds64(sz);
          ksz1 = lds64(sz + 32);
          vsz0 = lds64(sz + 64);
          vsz1 = lds64(sz + 96);
        }
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t ak[4];
          k_operand<KV, QBF>(cur, kk, ak);
          const uint32_t b0[2] = {ak[0], ak[2]}, b1[2] = {ak[1], ak[3]};
          mma16816<QBF>(sc[0], qa[kk], b0);
          mma16816<QBF>(sc[1], qa[kk], b1);
        }
        // scores in the exp2 domain; positions past a row's own are masked
        const int tok0 = (j_begin + k) * kBlock + 2 * t;
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
          const int ta = tok0 + 8 * nt;
          if (ta > pos[0]) sc[nt][0] = -INFINITY;
          if (ta + 1 > pos[0]) sc[nt][1] = -INFINITY;
          if (ta > pos[1]) sc[nt][2] = -INFINITY;
          if (ta + 1 > pos[1]) sc[nt][3] = -INFINITY;
        }
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
          // (a maximum still -inf only happens when nothing was accumulated)
          const float al0 = mn0 == -INFINITY ? 1.f : ex2(m0 - mn0);
          const float al1 = mn1 == -INFINITY ? 1.f : ex2(m1 - mn1);
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
        // rows with every position so far masked keep p = 0
        const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
        float p[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          p[nt][0] = ex2(sc[nt][0] - ref0);
          p[nt][1] = ex2(sc[nt][1] - ref0);
          p[nt][2] = ex2(sc[nt][2] - ref1);
          p[nt][3] = ex2(sc[nt][3] - ref1);
          l0 += p[nt][0] + p[nt][1];
          l1 += p[nt][2] + p[nt][3];
        }
        if constexpr (kQuant) {
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
    // every issued block was consumed: the next unit restarts at stage 0 (the
    // TMA parities carry over, each armed stage waited for exactly once)
    if constexpr (!S::kTma) cp_async_wait<0>();

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
    const bool direct = s.splits == 1;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      if (!qv[rr]) continue;
      const float z = rr ? z1 : z0, l = rr ? l1 : l0;
      const int64_t row = (static_cast<int64_t>(s.q0) + qi[rr]) * a.q_heads + qh[rr];
      if (direct) {
        // dims 32t + d (accumulator column 2t of dim tile d) and 32t + 16 + d
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint32_t w[16];
#pragma unroll
        for (int d = 0; d < 16; d += 2) {
          w[d / 2] = pack2<QBF>((o[d][2 * rr] + z) * inv, (o[d + 1][2 * rr] + z) * inv);
          w[8 + d / 2] =
              pack2<QBF>((o[d][2 * rr + 1] + z) * inv, (o[d + 1][2 * rr + 1] + z) * inv);
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + row * kHeadDim +
                                              32 * t);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
        dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
      } else {
        float* rec = a.part + (row * a.max_splits + c) * kPartStride;
        float4* lo4 = reinterpret_cast<float4*>(rec + 32 * t);
        float4* hi4 = reinterpret_cast<float4*>(rec + 32 * t + 16);
#pragma unroll
        for (int d = 0; d < 16; d += 4) {
          lo4[d / 4] = make_float4(o[d][2 * rr] + z, o[d + 1][2 * rr] + z,
                                   o[d + 2][2 * rr] + z, o[d + 3][2 * rr] + z);
          hi4[d / 4] = make_float4(o[d][2 * rr + 1] + z, o[d + 1][2 * rr + 1] + z,
                                   o[d + 2][2 * rr + 1] + z, o[d + 3][2 * rr + 1] + z);
        }
        if (t == 0) {
          rec[kHeadDim] = rr ? m1 : m0;
          rec[kHeadDim + 1] = l;
        }
      }
    }
  }
}

// One warp per (query row, q head) of a request whose context was split:
// merges its parts' records (log-sum-exp in the exp2 domain).
template <bool QBF>
__global__ void __launch_bounds__(128) extend_combine_kernel(const __grid_constant__ ExtendArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rh = static_cast<int64_t>(blockIdx.x) * 4 + warp;
  if (rh >= static_cast<int64_t>(a.total_q) * a.q_heads) return;
  const int qrow = static_cast<int>(rh / a.q_heads);
  int lo = 0, hi = a.batch - 1;  // the request holding qrow: largest b with qo_indptr[b] <= qrow
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.qo_indptr[mid] <= qrow) lo = mid; else hi = mid - 1;
  }
  const ReqShape s = req_shape(a, lo);
  if (s.splits == 1 || qrow >= s.q0 + s.C) return;  // written by the extend kernel
  const float* rec0 = a.part + rh * a.max_splits * kPartStride;
  float mw = -INFINITY, lw = 0.f;
  if (lane < s.splits) {
    mw = rec0[lane * kPartStride + kHeadDim];
    lw = rec0[lane * kPartStride + kHeadDim + 1];
  }
  float M = mw;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
  const float e = mw == -INFINITY ? 0.f : exp2f(mw - M);
  float lsum = e * lw;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) lsum += __shfl_xor_sync(kFull, lsum, off);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = 0; i < s.splits; ++i) {
    const float ei = __shfl_sync(kFull, e, i);
    const float4 x = reinterpret_cast<const float4*>(rec0 + i * kPartStride)[lane];
    acc.x += ei * x.x; acc.y += ei * x.y; acc.z += ei * x.z; acc.w += ei * x.w;
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  uint2 w;
  w.x = pack2<QBF>(acc.x * inv, acc.y * inv);
  w.y = pack2<QBF>(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + rh * kHeadDim)[lane] = w;
}

template <int KV, bool QBF>
cudaError_t launch_t(const ExtendArgs& a, int grid, cudaStream_t s) {
  thread_local int opted_in_device = -1;  // per host thread: no shared state
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (opted_in_device != dev) {
    e = cudaFuncSetAttribute(extend_kernel<KV, QBF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(extend_smem_bytes<KV>(kMaxBatch)));
    if (e != cudaSuccess) return e;
    opted_in_device = dev;
  }
  extend_kernel<KV, QBF><<<grid, kDecodeThreads, extend_smem_bytes<KV>(a.batch), s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.pchunk == 0) return e;
  const int64_t rows = static_cast<int64_t>(a.total_q) * a.q_heads;
  if (rows == 0) return cudaSuccess;
  extend_combine_kernel<QBF><<<static_cast<unsigned>((rows + 3) / 4), 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <int KV, bool QBF>
int occupancy_t(int batch) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  thread_local int cached_dev = -1, cached_batch = -1, cached_n = 0;
  if (dev == cached_dev && batch == cached_batch) return cached_n;
  if (cudaFuncSetAttribute(extend_kernel<KV, QBF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(extend_smem_bytes<KV>(kMaxBatch))) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, extend_kernel<KV, QBF>, kDecodeThreads,
                                                    extend_smem_bytes<KV>(batch)) != cudaSuccess)
    return 0;
  cached_dev = dev;
  cached_batch = batch;
  cached_n = n;
  return n;
}

}  // namespace

cudaError_t launch_extend(const ExtendArgs& a, int kv_dtype, int q_dtype, int grid,
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

int extend_ctas_per_sm(int kv_dtype, int q_dtype, int batch) {
  const bool qbf = q_dtype == kBF16;
  switch (kv_dtype) {
    case kF16: return occupancy_t<kF16, false>(batch);
    case kBF16: return occupancy_t<kBF16, true>(batch);
    case kI8: return qbf ? occupancy_t<kI8, true>(batch) : occupancy_t<kI8, false>(batch);
    case kI4: return qbf ? occupancy_t<kI4, true>(batch) : occupancy_t<kI4, false>(batch);
    default: return 0;
  }
}

}  // namespace kvq

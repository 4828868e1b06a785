// kvq_decode: single-token decode attention over the paged, quantized pool.
//
// LMDeploy article (devpress.csdn.net) §3.2 item 3: generation attention reads
// a non-contiguous KV layout through indirect block pointers; §4.2: decoding
// has its own hand-written kernel; §2.2: per-sequence block tables of 16-token
// blocks; §2.4: INT8/INT4 KV with per-token, per-head scale and zero.
//
// Work decomposition
//   All the work is one stream of blocks ordered by (q-head group, request,
//   block), where a q-head group is a kv head with up to 8 of its q heads.
//   A persistent grid (as many CTAs as fit on the device) gives every warp
//   one contiguous range of the stream of equal length, so the split between
//   warps is exact whatever the mix of request lengths. Each CTA first scans
//   the request lengths into per-request block offsets in shared memory.
//   A warp streams its range through its own ring of shared-memory stages
//   (several blocks in flight: TMA tensor copies completing on an mbarrier
//   for INT8 tiles, per-lane cp.async otherwise), crossing request boundaries without
//   a pause: it writes the output of every request it covers entirely and,
//   for the request holding the first and the one holding the last block of
//   its range, a partial record (running max, sum, unnormalised output) that
//   the combine kernel merges with a log-sum-exp. All q heads of a kv head's
//   group are handled by the same warp, so every KV byte is read once.
//   Long shares (RangeMap) keep about nine tenths of the stream in such
//   static ranges and hand the rest out in short chunks from a counter, each
//   chunk a range of its own, so that warps that ran slower are not waited
//   for.
//
// Per-block arithmetic of one warp (16 tokens of one kv head):
//   S^T = K Q^T  with mma.m16n8k16: M = 16 tokens, N = 8 q heads (padded),
//                K = 128 dims in 8 steps (two independent accumulators).
//   O^T += V^T P'^T with M = 16 dims (8 steps over 128), N = 8 heads,
//                K = 16 tokens.
//   Quantized codes go into the tensor cores as exact 16-bit floats a + c,
//   made by writing the code into the mantissa of a constant (INT4: a shift
//   and a lop3 per two codes, a = 16, or a = 128 on the K side of bf16
//   queries; INT8 K side: one prmt per two codes, a = 1024, or a = -128
//   through fp32 for bf16 queries; INT8 V side: a
//   prmt and a packed subtract, centred, a = -128); the offset is removed
//   outside the products together with the per-token zero:
//   c S + Z = (a + c) S + Z - a S.
//     q.k = S (q.(a + c)) + (Z - a S) sum(q)
//     sum_t p_t v_t = sum_t P'_t (a + c_t) + sum_t p_t (Z_t + mid S_t)
//                     - (a + mid) sum_t P'_t,   P'_t = fp16(p_t S_t)
//   where the last sum runs over the rounded P' fed to the product, so their
//   rounding error only multiplies c - mid (mid = 2^(b-1)); for centred INT8
//   codes (a = -mid) that term vanishes. The INT4 offset of 16 keeps the P.V
//   accumulator within a few times its centred size, so its fp32
//   accumulation error stays negligible over long contexts. The P.V product is fp16 for quantized
//   pools whatever Q's type (P' = p S <= S fits fp16); bf16 pools carry P as a
//   bf16 hi + lo pair. The score fragment is transposed in registers
//   (movmatrix) to become the B operand of the second product.
//   Each lane's K and V reads are 8-64 contiguous bytes of a token row; the
//   dims are assigned to mma k-columns so that these stay contiguous (the dot
//   product does not depend on the order of the dims, and Q is permuted the
//   same way once per request).
#include <cuda_runtime.h>

#include "kvq_decode_common.cuh"
#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_store_row.cuh"
#include "kvq_tables_item.cuh"
#include "kvq_tile.cuh"

namespace kvq {
namespace {

// The decode of CTA `cta` out of `ncta` (the persistent grid); dsmem is the
// CTA's dynamic shared memory, warp_sum 4 ints of static shared memory.
// TAIL: the instantiation that can hand out tail chunks (make_range_map);
// without it a warp has one range, as the tail-free sizes want.
template <int KV, bool QBF, bool TAIL>
__device__ __forceinline__ void decode_body(const DecodeArgs& a, unsigned char* dsmem,
                                            int32_t* warp_sum, int cta, int ncta) {
  using S = Stage<KV>;
  constexpr bool kQuant = KvTraits<KV>::kQuant;
  constexpr bool kPvBf = KV == kBF16;  // P.V product type: bf16 only for bf16 pools
  constexpr float kAk = CodeOffset<KV, QBF>::kK;
  constexpr float kAv = CodeOffset<KV, QBF>::kV;
  constexpr float kMid = CodeOffset<KV, QBF>::kMid;
  constexpr bool kPCorr = CodeOffset<KV, QBF>::kPCorr;
  constexpr int D = S::kDepth;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;

  // ---- blocks per request, prefix-summed (every CTA); the cut into ranges ------
  constexpr bool kLockstep = KV != kI4;
  const StreamPlan sp = plan_stream<QBF, TAIL>(a, dsmem, warp_sum, cta, ncta, kLockstep);
  const int32_t* cum = sp.cum;
  unsigned char* stages = sp.stages;
  const int tb = sp.tb;

  // ---- this warp's ranges: its static range, then tail chunks ----------------------
  // (no block barrier follows: warps are independent from here)
  const int64_t gw = static_cast<int64_t>(cta) * kWarps + warp;
  // this warp's stage region, 1024-byte aligned (the 128-byte swizzle repeats
  // every 1024 bytes)
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

  uint32_t phase = 0;  // parity to wait for, per stage (TMA path), across ranges
  // the range [x0, x0 + n), its records filed under range id rid; false when a
  // copy timed out (the warp stops)
  auto run_range = [&](const int64_t x0, const int n, const int64_t rid) -> bool {
    // issue side: cursor, a 32-entry window of the block table, validity bits
    Cursor ic;
    locate(ic, x0, cum, a.batch, tb);
    Cursor cc = ic;  // compute side
    int win_b = -1, win_j0 = 0;
    int32_t win = -1;
    uint32_t ok_mask = 0;  // stages holding a valid block in flight
    int k_issue = 0;   // next block of the range to issue
    int st_issue = 0;  // its stage
    auto issue_next = [&]() {
      if (k_issue < n) {
        if (ic.b != win_b || ic.j >= win_j0 + 32) {
          win_b = ic.b;
          win_j0 = ic.j;
          const int jj = win_j0 + lane;
          win = jj < ic.nblk ? a.block_tables[static_cast<int64_t>(ic.b) * a.max_blocks +
                                              skip_of(a, ic.b) + jj]
                             : -1;
        }
        const int32_t phys = __shfl_sync(kFull, win, ic.j - win_j0);
        const bool ok = phys >= 0 && phys < a.num_blocks;
        const uint32_t bit = 1u << st_issue;
        if (ok) {
          issue_block<KV>(wr, st_issue, a, lm, phys, ic.hgi / a.head_groups, lane);
          ok_mask |= bit;
        } else {
          ok_mask &= ~bit;
          if (lane == 0) report(a.dev_err, KVQ_DEV_ERR_BLOCK_ID);
        }
        if (k_issue + 1 < n) advance(ic, cum, a.batch);
      }
      if constexpr (!S::kTma) cp_async_commit();
      ++k_issue;
      st_issue = st_issue == D - 1 ? 0 : st_issue + 1;
    };
  #pragma unroll
    for (int k = 0; k < D - 1; ++k) issue_next();

    // ---- per-request state ---------------------------------------------------------
    int seg_b = -1, seg_hgi = -1, hq0 = 0, nh = 0, L = 0, seg_nblk = 0, seg_skip = 0;
    int64_t seg_start = 0;
    uint32_t qb[8][2];
    float qs0 = 0.f, qs1 = 0.f;  // sum(q) of heads 2t and 2t+1
    bool hv0 = false, hv1 = false;
    float o[8][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;
    float r0 = 0.f, r1 = 0.f;  // sums of the 16-bit P' values fed to the P.V product

    // writes the finished state of request seg_b: the output if this warp
    // covered all of its blocks, else a partial record
    auto flush = [&]() {
  #pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, off);
        l1 += __shfl_xor_sync(kFull, l1, off);
        if constexpr (kQuant) {
          z0 += __shfl_xor_sync(kFull, z0, off);
          z1 += __shfl_xor_sync(kFull, z1, off);
          if constexpr (kPCorr) {
            r0 += __shfl_xor_sync(kFull, r0, off);
            r1 += __shfl_xor_sync(kFull, r1, off);
          }
        }
      }
      if constexpr (kPCorr) {
        // o = sum P'(a + c) + sum p (Z + mid S) - (a + mid) sum P'
        z0 -= (kAv + kMid) * r0;
        z1 -= (kAv + kMid) * r1;
      }
      const bool contained = seg_start >= x0 && seg_start + seg_nblk <= x0 + n;
      const int64_t row0 = static_cast<int64_t>(seg_b) * a.q_heads + hq0;
  #pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int hh = 2 * t + u;
        if (hh >= nh) continue;
        const float z = u ? z1 : z0, l = u ? l1 : l0, m = u ? m1 : m0;
        if (contained) {
          float acc[16];
  #pragma unroll
          for (int i = 0; i < 8; ++i) {
            acc[2 * i] = o[i][u] + z;
            acc[2 * i + 1] = o[i][2 + u] + z;
          }
          float mm = m, ll = l;
          if (seg_skip > 0) merge_prefix(a, row0 + hh, seg_skip, g, mm, ll, acc);
          const float inv = ll > 0.f ? 1.f / ll : 0.f;
          uint32_t w[8];
  #pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = pack2<QBF>(acc[2 * i] * inv, acc[2 * i + 1] * inv);
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) +
                                                (row0 + hh) * kHeadDim + 16 * g);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
          const int slot = seg_start <= x0 ? 0 : 1;  // the request holding x0, else the last one
          float* rec = a.part + ((rid * 2 + slot) * a.hpg + hh) * kPartStride;
          float4* ov = reinterpret_cast<float4*>(rec + 16 * g);
  #pragma unroll
          for (int i = 0; i < 8; i += 2)
            ov[i / 2] =
                make_float4(o[i][u] + z, o[i][2 + u] + z, o[i + 1][u] + z, o[i + 1][2 + u] + z);
          if (g == 0) {
            rec[kHeadDim] = m;
            rec[kHeadDim + 1] = l;
          }
        }
      }
    };

    int st = 0;  // stage of block k
    for (int k = 0; k < n; ++k) {
      issue_next();  // refills the stage block k - 1 used
      const bool blk_ok = (ok_mask >> st) & 1u;
      if constexpr (S::kTma) {
        if (blk_ok) {
          if (!mbar_wait(wr + S::kBarOff + 8 * st, (phase >> st) & 1u)) {
            // a copy did not land: report, wait (bounded) for the other copies
            // this warp started, and stop
            if (lane == 0) report(a.dev_err, KVQ_DEV_ERR_TIMEOUT);
            const uint32_t rest = ok_mask & ~(1u << st);
            for (int i = 0; i < D; ++i)
              if ((rest >> i) & 1u) mbar_wait(wr + S::kBarOff + 8 * i, (phase >> i) & 1u);
            return false;
          }
          phase ^= 1u << st;
        }
      } else {
        cp_async_wait<D - 1>();  // this lane's copies of block k have landed
        __syncwarp();            // ... and every other lane's
      }

      if (cc.b != seg_b || cc.hgi != seg_hgi) {
        if (seg_b >= 0) flush();
        // start request cc.b for q-head group cc.hgi
        seg_b = cc.b;
        seg_hgi = cc.hgi;
        seg_nblk = cc.nblk;
        seg_start = static_cast<int64_t>(cc.hgi) * tb + cum[cc.b];
        const int h = cc.hgi / a.head_groups;
        const int hg = cc.hgi - h * a.head_groups;
        hq0 = h * a.group + hg * kHeadsPerGroup;
        nh = min(kHeadsPerGroup, a.group - hg * kHeadsPerGroup);
        seg_skip = skip_of(a, cc.b);
        L = clamped_len(a, cc.b) - kBlock * seg_skip;  // tokens of this request's own blocks
        // Q fragments (B operand of S^T = K Q^T), permuted like the K dims
        uint32_t qw[16];
        if (g < nh) {
          const uint4* qp = reinterpret_cast<const uint4*>(
              static_cast<const uint16_t*>(a.q) +
              (static_cast<int64_t>(cc.b) * a.q_heads + hq0 + g) * kHeadDim + 32 * t);
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
            qb[kk][0] = prmt(qw[4 * j + u], qw[4 * j + u + 2], 0x5410u);
            qb[kk][1] = prmt(qw[4 * j + u], qw[4 * j + u + 2], 0x7632u);
          }
        } else {
  #pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            qb[kk][0] = qw[2 * kk];
            qb[kk][1] = qw[2 * kk + 1];
          }
        }
        if constexpr (kQuant) {
          float part = 0.f;
  #pragma unroll
          for (int i = 0; i < 16; ++i) part += lo_to_float<QBF>(qw[i]) + hi_to_float<QBF>(qw[i]);
          part += __shfl_xor_sync(kFull, part, 1);
          part += __shfl_xor_sync(kFull, part, 2);
          qs0 = __shfl_sync(kFull, part, (2 * t) * 4);  // lanes 4h hold sum(q) of head h
          qs1 = __shfl_sync(kFull, part, (2 * t + 1) * 4);
        }
        hv0 = 2 * t < nh;
        hv1 = 2 * t + 1 < nh;
  #pragma unroll
        for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = z0 = z1 = r0 = r1 = 0.f;
      }

      if (blk_ok) {
        ok_mask &= ~(1u << st);
        Frag<KV> cur;
        read_frag<KV>(cur, wr, st, lm, g);
        // S^T = K Q^T, even and odd k-steps in two accumulators
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
        for (int kk = 0; kk < 8; kk += 2) {
          uint32_t ak[4];
          k_operand<KV, QBF>(cur, kk, ak);
          mma16816<QBF>(sa, ak, qb[kk]);
          k_operand<KV, QBF>(cur, kk + 1, ak);
          mma16816<QBF>(sb, ak, qb[kk + 1]);
        }
        const float sc0 = sa[0] + sb[0], sc1 = sa[1] + sb[1];
        const float sc2 = sa[2] + sb[2], sc3 = sa[3] + sb[3];
        // scores of tokens g, g+8 for heads 2t, 2t+1, in the exp2 domain
        const int tok0 = cc.j * kBlock + g, tok1 = tok0 + 8;
        float s00, s01, s10, s11;
        if constexpr (kQuant) {
          // q.k = S (q.(a + c)) + (Z - a S) sum(q)
          const float S0 = half_lo(cur.ksz[0]), Z0 = half_hi(cur.ksz[0]) - kAk * S0;
          const float S1 = half_lo(cur.ksz[1]), Z1 = half_hi(cur.ksz[1]) - kAk * S1;
          s00 = (S0 * sc0 + Z0 * qs0) * a.sm_scale_log2;
          s01 = (S0 * sc1 + Z0 * qs1) * a.sm_scale_log2;
          s10 = (S1 * sc2 + Z1 * qs0) * a.sm_scale_log2;
          s11 = (S1 * sc3 + Z1 * qs1) * a.sm_scale_log2;
        } else {
          s00 = sc0 * a.sm_scale_log2;
          s01 = sc1 * a.sm_scale_log2;
          s10 = sc2 * a.sm_scale_log2;
          s11 = sc3 * a.sm_scale_log2;
        }
        if (tok0 >= L) s00 = s01 = -INFINITY;
        if (tok1 >= L) s10 = s11 = -INFINITY;
        if (!hv0) s00 = s10 = 0.f;  // padded heads: finite, never written
        if (!hv1) s01 = s11 = 0.f;
        // the running maximum moves only when some lane holds a larger score:
        // then reduce the block maximum over the 16 tokens (lanes with equal t)
        // and rescale the running state
        float bm0 = fmaxf(s00, s10), bm1 = fmaxf(s01, s11);
        float mn0 = m0, mn1 = m1;
        if (__any_sync(kFull, bm0 > m0 || bm1 > m1)) {
  #pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, off));
            bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, off));
          }
          mn0 = fmaxf(m0, bm0);
          mn1 = fmaxf(m1, bm1);
          const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
          l0 *= al0;
          l1 *= al1;
          z0 *= al0;
          z1 *= al1;
          r0 *= al0;
          r1 *= al1;
  #pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[i][0] *= al0; o[i][2] *= al0;
            o[i][1] *= al1; o[i][3] *= al1;
          }
        }
        m0 = mn0;
        m1 = mn1;
        const float p00 = ex2(s00 - mn0), p10 = ex2(s10 - mn0);
        const float p01 = ex2(s01 - mn1), p11 = ex2(s11 - mn1);
        l0 += p00 + p10;
        l1 += p01 + p11;
        float q00 = p00, q01 = p01, q10 = p10, q11 = p11;
        if constexpr (kQuant) {
          // sum_t p_t v_t = sum_t P'_t (a + c_t) + sum_t p_t (Z_t + mid S_t)
          //                 - (a + mid) sum_t P'_t,  with P'_t = p_t S_t in fp16:
          // subtracting the rounded P' actually used leaves their rounding
          // error multiplied by c - mid only, as if the codes were centred
          const float S0 = half_lo(cur.vsz[0]), Z0 = half_hi(cur.vsz[0]) + kMid * S0;
          const float S1 = half_lo(cur.vsz[1]), Z1 = half_hi(cur.vsz[1]) + kMid * S1;
          z0 += p00 * Z0 + p10 * Z1;
          z1 += p01 * Z0 + p11 * Z1;
          q00 *= S0; q01 *= S0; q10 *= S1; q11 *= S1;
        }
        // P'^T as the B operand: transpose the (token x head) fragments
        uint32_t bp[2], bp_lo[2];
        const uint32_t h0 = pack2<kPvBf>(q00, q01), h1 = pack2<kPvBf>(q10, q11);
        if constexpr (kPCorr) {
          r0 += lo_to_float<false>(h0) + lo_to_float<false>(h1);
          r1 += hi_to_float<false>(h0) + hi_to_float<false>(h1);
        }
        bp[0] = movmatrix_trans(h0);
        bp[1] = movmatrix_trans(h1);
        if constexpr (kPvBf) {
          // bf16 keeps 8 bits of P: add the rounding residual in a second
          // product so P carries ~16 bits (P = hi + lo)
          bp_lo[0] = movmatrix_trans(pack2<true>(q00 - lo_to_float<true>(h0),
                                                 q01 - hi_to_float<true>(h0)));
          bp_lo[1] = movmatrix_trans(pack2<true>(q10 - lo_to_float<true>(h1),
                                                 q11 - hi_to_float<true>(h1)));
        }
        // O^T += V^T P'^T
  #pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t av[4];
          v_operand<KV>(cur, i, av);
          mma16816<kPvBf>(o[i], av, bp);
          if constexpr (kPvBf) mma16816<true>(o[i], av, bp_lo);
        }
      }
      __syncwarp();  // all lanes are done with this stage before it is refilled
      st = st == D - 1 ? 0 : st + 1;
      if (k + 1 < n) advance(cc, cum, a.batch);
    }
    if constexpr (!S::kTma) cp_async_wait<0>();
    flush();
    return true;
  };  // run_range

  for_each_range<TAIL>(a, sp, gw, lane, run_range);
}

template <int KV, bool QBF, bool TAIL>
__global__ void __launch_bounds__(kDecodeThreads, TAIL && KV != kI4 ? 3 : 1)
    decode_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  __shared__ int32_t warp_sum[kWarps];
  // the combine kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;");
  decode_body<KV, QBF, TAIL>(a, dsmem, warp_sum, blockIdx.x, gridDim.x);
}

// The merge of one (request, q head) row that the decode did not finish
// itself, by one warp: the split-K records of the ranges its blocks were
// split between (slot 1 for the first when the request starts inside that
// range), then its shared-prefix records, if any (a request made of shared
// blocks only has nothing else). Log-sum-exp in the exp2 domain, 8 pieces
// per round of loads.
template <bool QBF>
__device__ __forceinline__ void merge_pieces(const DecodeArgs& a, int64_t bh, int hh, int lane,
                                             int64_t r_first, int64_t nd, int64_t seg_start,
                                             const RangeMap& rm, int npc) {
  auto rec_of = [&](int64_t i) -> const float* {
    if (i < nd) {
      const int slot = (i == 0 && seg_start != range_start(rm, r_first)) ? 1 : 0;
      return a.part + (((r_first + i) * 2 + slot) * a.hpg + hh) * kPartStride;
    }
    return a.ppart + (bh * a.pmax_chunks + (i - nd)) * kPartStride;
  };
  const int64_t npieces = nd + npc;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.f, M = -INFINITY;
  constexpr int kBatch = 8;  // pieces whose loads are in flight together
  for (int64_t base = 0; base < npieces; base += kBatch) {
    // every lane reads each piece's maximum and sum (one address: broadcast)
    // and its own 4 columns, all loads of the batch issued before any use;
    // through L2, as other SMs wrote the records
    float mm[kBatch], ll[kBatch];
    float4 x[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      mm[i] = -INFINITY;
      ll[i] = 0.f;
      x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (base + i < npieces) {
        const float* rec = rec_of(base + i);
        mm[i] = __ldcg(rec + kHeadDim);
        ll[i] = __ldcg(rec + kHeadDim + 1);
        x[i] = __ldcg(reinterpret_cast<const float4*>(rec) + lane);
      }
    }
    float Mb = mm[0];
#pragma unroll
    for (int i = 1; i < kBatch; ++i) Mb = fmaxf(Mb, mm[i]);
    const float Mn = fmaxf(M, Mb);
    if (Mn == -INFINITY) continue;
    if (M != Mn && M != -INFINITY) {  // this batch raised the maximum
      const float al = exp2f(M - Mn);
      lsum *= al;
      acc.x *= al; acc.y *= al; acc.z *= al; acc.w *= al;
    }
    M = Mn;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const float e = mm[i] == -INFINITY ? 0.f : exp2f(mm[i] - M);
      lsum += e * ll[i];
      acc.x += e * x[i].x; acc.y += e * x[i].y; acc.z += e * x[i].z; acc.w += e * x[i].w;
    }
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  uint2 w;
  w.x = pack2<QBF>(acc.x * inv, acc.y * inv);
  w.y = pack2<QBF>(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + bh * kHeadDim)[lane] = w;
}

template <bool QBF>
__device__ __forceinline__ void combine_row(const DecodeArgs& a, int64_t bh, int lane) {
  if (bh >= static_cast<int64_t>(a.batch) * a.q_heads) return;
  const int b = static_cast<int>(bh / a.q_heads);
  const int hq = static_cast<int>(bh - static_cast<int64_t>(b) * a.q_heads);
  const int tb = a.hdr[0];
  RangeMap rm;
  rm.Pst = a.hdr[1];
  rm.C = a.hdr[2];
  rm.nwarps = a.hdr[3];
  rm.ntail = 0;  // not needed to map blocks to ranges
  rm.k = a.hdr[4];
  rm.tb = tb;
  const int32_t* cum = a.hdr + kHdrCum;
  const int nblk = cum[b + 1] - cum[b];
  const int skip = a.skip != nullptr ? a.skip[b] : 0;
  const int npc = skip > 0 ? (skip + a.pchunk - 1) / a.pchunk : 0;
  if (nblk == 0 && npc == 0) return;  // zeroed by the decode kernel
  int hgi, hh;  // the row's q-head group in the stream, and its record row in the group
  if (a.cta_heads > 0) {  // grouped-query kernel: groups of cta_heads kv heads
    const int qpg = a.cta_heads * a.group;
    hgi = hq / qpg;
    hh = hq - hgi * qpg;
  } else {
    const int h = hq / a.group, within = hq - h * a.group;
    hgi = h * a.head_groups + within / kHeadsPerGroup;
    hh = within % kHeadsPerGroup;
  }
  const int64_t seg_start = static_cast<int64_t>(hgi) * tb + cum[b];
  int64_t r_first = 0, nd = 0;
  if (nblk > 0) {
    r_first = range_of(rm, seg_start);
    const int64_t r_last = range_of(rm, seg_start + nblk - 1);
    if (r_first == r_last) return;  // one range: written by the decode kernel
    nd = r_last - r_first + 1;
  }
  merge_pieces<QBF>(a, bh, hh, lane, r_first, nd, seg_start, rm, npc);
}

// Launched as a programmatic dependent of the decode kernel: its CTAs may
// start while the decode runs and wait here until the decode grid has
// finished and its records are visible.
template <bool QBF>
__global__ void __launch_bounds__(128) combine_kernel(const __grid_constant__ DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  combine_row<QBF>(a, static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5),
                   threadIdx.x & 31);
}

// ---- the fused step ------------------------------------------------------------

constexpr int kStepUnroll = 4;  // table entries / pool rows a half-warp has in flight

// Grid-wide barrier of a cooperative launch: thread 0 of every CTA counts in
// and waits, with acquire loads, until `target` CTAs have; the wait gives up
// after limit_ns (2 s in the step; KVQ_DEV_ERR_TIMEOUT, false: the caller
// stops).
__device__ __forceinline__ bool grid_sync(unsigned int* ctr, unsigned int target,
                                          int32_t* dev_err,
                                          uint64_t limit_ns = 2000000000ull) {
  __shared__ int ok_s;
  asm volatile("fence.proxy.async.global;" ::: "memory");  // global writes before TMA reads
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
    int ok = 1;
    const uint64_t t0 = global_ns();
    for (;;) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      if (global_ns() - t0 > limit_ns) {
        ok = 0;
        report(dev_err, KVQ_DEV_ERR_TIMEOUT);
        break;
      }
      __nanosleep(128);
    }
    __threadfence();
    ok_s = ok;
  }
  __syncthreads();
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return ok_s != 0;
}

// One decode step: (1) block tables and the quantizing store of the new
// tokens, spread over the whole grid; (2) the decode, as decode_kernel; (3)
// the combine, one warp per (request, q head). The phases are separated by
// grid barriers, so the step is one launch instead of four.
template <int KV, bool QBF, bool TAIL>
__global__ void __launch_bounds__(kDecodeThreads, KV == kI4 && !TAIL ? kMaxCtasPerSm : 3)
    step_kernel(const __grid_constant__ StepArgs s) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  __shared__ int32_t warp_sum[kWarps];
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * kWarps + (tid >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  // (1) block tables, then the store: a half-warp per table entry and per pool
  // row, kStepUnroll of them with their loads in flight together
  const int lane16 = lane & 15;
  const int64_t hw = 2 * gwarp + (lane >> 4), nhw = 2 * nwarps;
  const int64_t entries = static_cast<int64_t>(s.t.batch) * s.t.max_blocks_per_seq;
  for (int64_t i = hw; i < entries; i += kStepUnroll * nhw)
    tables_blocks<kStepUnroll>(s.t, i, nhw, lane16);
  const int64_t rows = s.st.num_tokens * 2 * s.st.kv_heads;
  for (int64_t r = hw; r < rows; r += kStepUnroll * nhw) {
    RowIn in[kStepUnroll];
#pragma unroll
    for (int u = 0; u < kStepUnroll; ++u) in[u] = load_row<KV, QBF>(s.st, r + u * nhw, lane16);
#pragma unroll
    for (int u = 0; u < kStepUnroll; ++u) write_row<KV, QBF>(s.st, in[u], lane16);
  }
  if (!grid_sync(s.barrier, gridDim.x, s.d.dev_err)) return;
  // (2) decode
  decode_body<KV, QBF, TAIL>(s.d, dsmem, warp_sum, blockIdx.x, gridDim.x);
  if (!grid_sync(s.barrier, 2 * gridDim.x, s.d.dev_err)) return;
  // (3) combine
  for (int64_t bh = gwarp; bh < static_cast<int64_t>(s.d.batch) * s.d.q_heads; bh += nwarps)
    combine_row<QBF>(s.d, bh, lane);
}

// Self-test of the step's barrier: the grid's CTAs meet at one barrier that
// waits for one CTA more than the grid has, with a limit of limit_ns, so the
// wait runs out, reports KVQ_DEV_ERR_TIMEOUT and every CTA returns.
__global__ void __launch_bounds__(kDecodeThreads) barrier_selftest_kernel(unsigned int* ctr,
                                                                         int32_t* dev_err,
                                                                         uint64_t limit_ns) {
  grid_sync(ctr, gridDim.x + 1, dev_err, limit_ns);
}

template <int KV, bool QBF, bool TAIL>
cudaError_t launch_step_t(const StepArgs& a, int grid, cudaStream_t s) {
  thread_local int opted_in_device = -1;  // per host thread: no shared state
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (opted_in_device != dev) {
    e = cudaFuncSetAttribute(step_kernel<KV, QBF, TAIL>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes_for<KV>(kMaxBatch)));
    if (e != cudaSuccess) return e;
    opted_in_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = smem_bytes_for<KV>(a.d.batch);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeCooperative;  // every CTA resident: the barriers need it
  attr.val.cooperative = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_kernel<KV, QBF, TAIL>, a);
}

template <int KV, bool QBF, bool TAIL>
int step_occupancy_t(int batch) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  thread_local int cached_dev = -1, cached_batch = -1, cached_n = 0;
  if (dev == cached_dev && batch == cached_batch) return cached_n;
  if (cudaFuncSetAttribute(step_kernel<KV, QBF, TAIL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes_for<KV>(kMaxBatch))) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, step_kernel<KV, QBF, TAIL>, kDecodeThreads,
                                                    smem_bytes_for<KV>(batch)) != cudaSuccess)
    return 0;
  cached_dev = dev;
  cached_batch = batch;
  cached_n = n;
  return n;
}

template <int KV, bool QBF, bool TAIL>
cudaError_t launch_t(const DecodeArgs& a, int grid, cudaStream_t s) {
  // allow the largest dynamic shared memory the kernel can ask for, once
  // per device
  thread_local int opted_in_device = -1;  // per host thread: no shared state
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (opted_in_device != dev) {
    e = cudaFuncSetAttribute(decode_kernel<KV, QBF, TAIL>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes_for<KV>(kMaxBatch)));
    if (e != cudaSuccess) return e;
    opted_in_device = dev;
  }
  decode_kernel<KV, QBF, TAIL><<<grid, kDecodeThreads, smem_bytes_for<KV>(a.batch), s>>>(a);
  return cudaGetLastError();
}

template <int KV, bool QBF, bool TAIL>
int occupancy_t(int batch) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  thread_local int cached_dev = -1, cached_batch = -1, cached_n = 0;
  if (dev == cached_dev && batch == cached_batch) return cached_n;
  if (cudaFuncSetAttribute(decode_kernel<KV, QBF, TAIL>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes_for<KV>(kMaxBatch))) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<KV, QBF, TAIL>,
                                                    kDecodeThreads,
                                                    smem_bytes_for<KV>(batch)) != cudaSuccess)
    return 0;
  cached_dev = dev;
  cached_batch = batch;
  cached_n = n;
  return n;
}

}  // namespace

namespace {

// f.run<KV, QBF, TAIL>() for the runtime pool kind, Q type and tail flag;
// f.fail() for a kind without a kernel.
template <typename F>
auto with_kinds(int kv_dtype, int q_dtype, bool tail, const F& f) -> decltype(f.fail()) {
  const bool qbf = q_dtype == kBF16;
  switch (kv_dtype) {
    case kF16:
      return tail ? f.template run<kF16, false, true>() : f.template run<kF16, false, false>();
    case kBF16:
      return tail ? f.template run<kBF16, true, true>() : f.template run<kBF16, true, false>();
    case kI8:
      if (qbf)
        return tail ? f.template run<kI8, true, true>() : f.template run<kI8, true, false>();
      return tail ? f.template run<kI8, false, true>() : f.template run<kI8, false, false>();
    case kI4:
      if (qbf)
        return tail ? f.template run<kI4, true, true>() : f.template run<kI4, true, false>();
      return tail ? f.template run<kI4, false, true>() : f.template run<kI4, false, false>();
    default:
      return f.fail();
  }
}

struct LaunchDecode {
  const DecodeArgs& a;
  int grid;
  cudaStream_t s;
  template <int KV, bool QBF, bool TAIL>
  cudaError_t run() const { return launch_t<KV, QBF, TAIL>(a, grid, s); }
  cudaError_t fail() const { return cudaErrorInvalidValue; }
};

struct LaunchStep {
  const StepArgs& a;
  int grid;
  cudaStream_t s;
  template <int KV, bool QBF, bool TAIL>
  cudaError_t run() const { return launch_step_t<KV, QBF, TAIL>(a, grid, s); }
  cudaError_t fail() const { return cudaErrorInvalidValue; }
};

struct DecodeOccupancy {
  int batch;
  template <int KV, bool QBF, bool TAIL>
  int run() const { return occupancy_t<KV, QBF, TAIL>(batch); }
  int fail() const { return 0; }
};

struct StepOccupancy {
  int batch;
  template <int KV, bool QBF, bool TAIL>
  int run() const { return step_occupancy_t<KV, QBF, TAIL>(batch); }
  int fail() const { return 0; }
};

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int kv_dtype, int q_dtype, int grid,
                          cudaStream_t s) {
  return with_kinds(kv_dtype, q_dtype, a.tail_ctr != nullptr, LaunchDecode{a, grid, s});
}

cudaError_t launch_combine(const DecodeArgs& a, int q_dtype, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.batch) * a.q_heads;
  if (rows == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap the decode's tail
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return q_dtype == kBF16 ? cudaLaunchKernelEx(&cfg, combine_kernel<true>, a)
                          : cudaLaunchKernelEx(&cfg, combine_kernel<false>, a);
}

cudaError_t launch_step(const StepArgs& a, int kv_dtype, int q_dtype, int grid,
                        cudaStream_t s) {
  return with_kinds(kv_dtype, q_dtype, a.d.tail_ctr != nullptr, LaunchStep{a, grid, s});
}

cudaError_t launch_barrier_selftest(unsigned int* ctr, int32_t* dev_err, int grid,
                                    uint64_t limit_ns, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeCooperative;  // as the step: every CTA resident
  attr.val.cooperative = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, barrier_selftest_kernel, ctr, dev_err, limit_ns);
}

int step_ctas_per_sm(int kv_dtype, int q_dtype, int batch, bool tail) {
  return with_kinds(kv_dtype, q_dtype, tail, StepOccupancy{batch});
}

int decode_ctas_per_sm(int kv_dtype, int q_dtype, int batch, bool tail) {
  return with_kinds(kv_dtype, q_dtype, tail, DecodeOccupancy{batch});
}

}  // namespace kvq

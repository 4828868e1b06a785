// kvq_decode_gqa: single-token decode attention over INT8 / INT4 pools for
// queries in fp16 with 4 q heads per kv head (grouped-query attention).
//
// LMDeploy article (devpress.csdn.net) §2.4: INT8/INT4 KV with a per-token,
// per-head (scale, zero); §2.2: 16-token blocks reached through block tables;
// §3.2 item 3 and §4.2: generation attention reads the paged KV through
// indirect block pointers in its own hand-written kernel.
//
// With 4 q heads per kv head a (block, kv head) unit carries 4-8 times fewer
// bytes per query than with one, and the instructions spent per unit, not
// DRAM, set the pace; the kernel is laid out to spend few.
//
// Work split. A CTA has one warp per kv head of a group of W kv heads (W = the
// pool's kv heads, or 8 of them). The work is one stream of (head group,
// request, block) units, and a persistent grid gives every CTA one contiguous
// range of it (kvq_decode_common.cuh: equal static ranges, tail chunks from a
// counter for long shares); partial records of requests a range does not
// hold whole are merged by the combine kernel. Every warp of a CTA attends the
// same blocks, each for its own kv head.
//
// Staging. One thread (warp 0, lane 0) stages a block for all W kv heads with
// two TMA tensor copies (K and V: a 4-D view of the pool ordered [block][kv
// head][token][row], so the W tiles of 16 rows land one after the other, each
// with the pool's 64- or 128-byte swizzle) and two bulk copies of the W
// heads' scale/zero runs, into a ring of kDepth stages. A stage's full
// mbarrier completes when its bytes have landed; its empty mbarrier when all W
// warps have read it, after which the next block may be staged there. The
// stage also carries the block's position (head group, request, block) for
// the consumers. Block ids come from a window of 32 located lane-parallel by
// warp 0 (binary search over the per-request block offsets in shared memory),
// one window ahead. All waits are bounded (2 s): on expiry the thread reports
// KVQ_DEV_ERR_TIMEOUT, the CTA stops staging and waits (bounded again) for
// its copies in flight before it returns.
//
// Codes as fp16 subnormals. A code c written into the low mantissa bits of an
// fp16 whose exponent field is zero is the exact value c * 2^-24 (tensor
// cores take fp16 subnormal operands exactly). So one AND (INT4: a nibble at
// bits 0-3 or 4-7 of each 16-bit half, c or 16 c units of 2^-24) or one byte
// permute with a zero source (INT8) turns two codes into one operand
// register, with no offset to remove afterwards:
//   q.k  = S 2^24 (sum_A q c 2^-24 + sum_B q 16 c 2^-24 / 16) + Z sum(q)
//   o    = 2^24 (sum_t P'_t c_t 2^-24) - mid sum_t P'_t + sum_t p_t (Z_t + mid S_t)
// with P'_t = fp16(p_t S_t), mid = 2^(b-1), and the sum of the rounded P'
// taken by one more tensor-core product against a matrix of ones, so that
// the rounding of P' only multiplies c - mid. INT4 dims whose nibble sits at
// bits 4-7 carry 16 c: on the K side they go to their own accumulator
// (class B), on the V side the output rows they produce are scaled by 1/16
// at the end.
//
// Duplicated q columns. The score product S^T = K Q^T has N = 8 columns and
// the group only 4 q heads, so columns 4-7 repeat heads 0-3. A lane of the
// mma layout holds tokens g and g + 8 for columns 2t, 2t + 1: lanes t = 0, 1
// keep token g and lanes t = 2, 3 keep token g + 8, each for heads
// 2 (t mod 2) and 2 (t mod 2) + 1, so every lane runs the softmax of two
// scores instead of four. In the P.V product columns 0-3 take tokens 0-7 and
// columns 4-7 tokens 8-15 of the same heads, so no weight changes lanes; the
// two halves are added when a request's rows are written.
//
// Running maximum. Scores live in the exp2 domain. The running maximum m of
// a q head is raised (and the state rescaled) only when a score exceeds it
// by more than 8, so weights p = 2^(s - m) stay below 2^8 and P' = p S_v
// below 2^8 S_v; a token whose V scale is above 240 (where 2^8 S_v could
// leave fp16) raises the maximum as soon as it exceeds it. The result is the
// same softmax: the maximum only bounds the exponents.
#include <cuda_runtime.h>

#include "kvq_decode_common.cuh"
#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tile.cuh"

namespace kvq {
namespace {

constexpr int kGqaGroup = 4;              // q heads per kv head served by this kernel
constexpr int kMaxCtaHeads = 8;           // warps (kv heads) per CTA
constexpr uint32_t kLoNib = 0x000F000Fu;  // nibble at bits 0-3 of each half: c
constexpr uint32_t kHiNib = 0x00F000F0u;  // nibble at bits 4-7 of each half: 16 c
constexpr float kTwo24 = 16777216.f;      // 2^24: one code unit of the subnormal encoding
constexpr uint32_t kOnes = 0x3C003C00u;   // fp16 pair (1, 1)
constexpr float kSlack = 8.f;             // the running maximum may lag the scores by this
constexpr float kSlackMaxScale = 240.f;   // ... while V scales stay below this (2^8 S_v < 2^16)
constexpr uint64_t kWaitNs = 2000000000ull;

// A stage holds one block for W kv heads: [K tiles W][V tiles W][K scale/zero
// runs W][V scale/zero runs W][position]; stages are 1024-byte aligned (the
// swizzle pattern of a tile repeats every 512 / 1024 bytes, and every tile
// starts on such a boundary).
template <int KV>
struct CtaStage {
  static constexpr int kRow = KvTraits<KV>::kRowBytes;  // 64 (INT4) or 128 (INT8)
  static constexpr int kTile = kBlock * kRow;           // one (block, kv head) tile
  static constexpr int kDepth = KV == kI4 ? 4 : 3;
  __host__ __device__ static constexpr int v_off(int w) { return w * kTile; }
  __host__ __device__ static constexpr int sz_off(int w) { return 2 * w * kTile; }
  __host__ __device__ static constexpr int info_off(int w) { return 2 * w * kTile + 2 * w * 64; }
  __host__ __device__ static constexpr int bytes(int w) {
    return (info_off(w) + 16 + 1023) / 1024 * 1024;
  }
  __host__ __device__ static constexpr uint32_t tx_bytes(int w) {
    return static_cast<uint32_t>(2 * w * kTile + 2 * w * 64);
  }
  // chunk c of row r sits at chunk c ^ swz(r): the TMA 128-byte swizzle for
  // 128-byte rows, the 64-byte swizzle for 64-byte rows
  __host__ __device__ static constexpr int at(int r, int c) {
    return r * kRow + (c ^ (kRow == 64 ? ((r >> 1) & 3) : (r & 7))) * 16;
  }
};

// Dynamic shared memory: [blocks before request b, batch + 1][own tokens of
// request b, batch][slack to 1024 bytes][kDepth stages][full and empty
// mbarriers, kDepth each].
template <int KV>
__host__ __device__ constexpr size_t gqa_smem_bytes(int batch, int w) {
  return align128((2 * batch + 1) * sizeof(int32_t)) + 1024 +
         static_cast<size_t>(CtaStage<KV>::kDepth) * CtaStage<KV>::bytes(w) +
         2 * CtaStage<KV>::kDepth * 8;
}

// Two codes as the fp16 subnormal pair selected by sel from word w's bytes
// and zero bytes (INT8): [w.b_lo, 0, w.b_hi, 0].
__device__ __forceinline__ uint32_t bytes_sub(uint32_t w, uint32_t sel) {
  return prmt(w, 0u, sel);
}

__device__ __forceinline__ void sts64(uint32_t addr, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(x), "r"(y) : "memory");
}

__device__ __forceinline__ void mbar_init_n(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Waits for the phase of parity `parity`; gives up after kWaitNs or as soon as
// *abort is set by another thread of the CTA (false either way).
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort != 0 || global_ns() - t0 > kWaitNs) return false;
  }
  return true;
}

template <int KV, bool TAIL>
__device__ __forceinline__ void gqa_body(const DecodeArgs& a, unsigned char* dsmem,
                                         int32_t* warp_sum, volatile int* abort_s,
                                         int32_t* chunk_s, int cta, int ncta) {
  using S = CtaStage<KV>;
  constexpr int D = S::kDepth;
  constexpr float kMid = KV == kI8 ? 128.f : 8.f;
  constexpr bool kLockstep = KV != kI4;

  const int W = a.cta_heads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int tsel = t >> 1;       // 0: this lane scores token g, 1: token g + 8
  const int hp = t & 1;          // ... for q heads 2 hp and 2 hp + 1 of the group
  const int tau = g + 8 * tsel;  // that token's row in the block
  const bool producer = warp == 0;

  const StreamPlan sp = plan_stream<false, TAIL>(a, dsmem, warp_sum, cta, ncta, kLockstep,
                                                 /*own_lens=*/true, /*ranges_per_cta=*/1);
  const int32_t* cum = sp.cum;
  const int32_t* lown = sp.cum + a.batch + 1;  // tokens of request b's own blocks
  const int tb = sp.tb;
  const uint32_t stage0 =
      (static_cast<uint32_t>(__cvta_generic_to_shared(sp.stages)) + 1023u) & ~1023u;
  const uint32_t SB = static_cast<uint32_t>(S::bytes(W));
  const uint32_t full0 = stage0 + D * SB, empty0 = full0 + 8 * D;
  if (tid == 0) {
    for (int i = 0; i < D; ++i) {
      mbar_init_n(full0 + 8 * i, 1);
      mbar_init_n(empty0 + 8 * i, static_cast<uint32_t>(W));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *abort_s = 0;
  }
  __syncthreads();

  // fragment offsets of this lane in its kv head's K and V tiles
  uint32_t kro[2][S::kRow / 64];  // rows g, g + 8: dims [32t, 32t + 32)
  uint32_t vro[4];                // rows 2t, 2t+1, 2t+8, 2t+9: dims [16g, 16g + 16)
#pragma unroll
  for (int i = 0; i < S::kRow / 64; ++i) {
    kro[0][i] = warp * S::kTile + S::at(g, (S::kRow / 64) * t + i);
    kro[1][i] = warp * S::kTile + S::at(g + 8, (S::kRow / 64) * t + i);
  }
  {
    const int rows[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
    for (int r = 0; r < 4; ++r)
      vro[r] = S::v_off(W) + warp * S::kTile +
               (KV == kI4 ? S::at(rows[r], g >> 1) + 8 * (g & 1) : S::at(rows[r], g));
  }
  const uint32_t szo = S::sz_off(W) + 64 * warp + 4 * tau;  // this lane's K (V: + 64 W) pair
  const float lsc = a.sm_scale_log2;  // softmax scale x log2(e)
  const uint32_t nb32 = static_cast<uint32_t>(a.num_blocks);  // valid ids are below this
  const uint32_t tx = S::tx_bytes(W);

  // blocks staged (warp 0) and consumed (every warp) by this CTA, across its
  // ranges: stage i % D, phase parity (i / D) & 1
  uint32_t n_staged = 0, n_used = 0;

  auto run_range = [&](const int64_t x0, const int n, const int64_t rid) -> bool {
    // ---- producer: windows of 32 blocks located lane-parallel by warp 0 -------------
    auto locate_window = [&](int w, int32_t& phys, uint32_t& key, int32_t& blk) {
      const int kk = 32 * w + lane;
      phys = -1;
      key = 0xFFFFFFFFu;
      blk = 0;
      if (kk < n) {
        const int64_t x = x0 + kk;
        const int hgi = static_cast<int>(x / tb);
        const int r = static_cast<int>(x - static_cast<int64_t>(hgi) * tb);
        int lo = 0, hi = a.batch - 1;  // the non-empty request holding r
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (cum[mid] <= r) lo = mid; else hi = mid - 1;
        }
        blk = r - cum[lo];
        key = (static_cast<uint32_t>(hgi) << 16) | static_cast<uint32_t>(lo);
        phys = a.block_tables[static_cast<int64_t>(lo) * a.max_blocks + skip_of(a, lo) + blk];
      }
    };
    int32_t wphys = -1, nphys = -1, wblk = 0, nblk_ = 0;
    uint32_t wkey = 0, nkey = 0;
    if (producer) {
      locate_window(0, wphys, wkey, wblk);
      locate_window(1, nphys, nkey, nblk_);
    }
    // warp 0 stages block kq of the range into the next stage; false when the
    // CTA stops (a wait ran out)
    auto stage_block = [&](const int kq) -> bool {
      const int kk = kq & 31;
      if (kk == 0 && kq > 0) {  // next window; locate the one after it
        wphys = nphys; wkey = nkey; wblk = nblk_;
        locate_window((kq >> 5) + 1, nphys, nkey, nblk_);
      }
      const int32_t phys = __shfl_sync(kFull, wphys, kk);
      const uint32_t key = __shfl_sync(kFull, wkey, kk);
      const int32_t blk = __shfl_sync(kFull, wblk, kk);
      const uint32_t s = n_staged % D;
      bool go = true;
      if (lane == 0) {
        const uint32_t st = stage0 + s * SB, full = full0 + 8 * s;
        // the stage's previous block must have been read by every warp
        if (n_staged >= D && !mbar_wait_or_abort(empty0 + 8 * s, ((n_staged / D) - 1) & 1u,
                                                 abort_s)) {
          if (*abort_s == 0) report(a.dev_err, KVQ_DEV_ERR_TIMEOUT);
          *abort_s = 1;
          go = false;
        } else {
          const bool ok = static_cast<uint32_t>(phys) < nb32;
          sts64(st + S::info_off(W), key, ok ? static_cast<uint32_t>(blk) : 0xFFFFFFFFu);
          if (ok) {
            const int h0 = static_cast<int>(key >> 16) * W;  // first kv head of the group
            const int64_t szi = (static_cast<int64_t>(phys) * a.kv_heads + h0) * kBlock;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arm(full, tx);
            tma_tile_4d(st, &a.kh_map, 0, 0, h0, phys, full);
            tma_tile_4d(st + S::v_off(W), &a.vh_map, 0, 0, h0, phys, full);
            bulk_copy(st + S::sz_off(W), a.k_sz + szi, 64 * W, full);
            bulk_copy(st + S::sz_off(W) + 64 * W, a.v_sz + szi, 64 * W, full);
          } else {
            report(a.dev_err, KVQ_DEV_ERR_BLOCK_ID);
            mbar_arrive(full);  // nothing to copy: the phase completes now
          }
        }
      }
      const bool cont = __shfl_sync(kFull, go ? 1 : 0, 0) != 0;
      if (cont) ++n_staged;
      return cont;
    };
    bool staging = producer;
    for (int k = 0; staging && k < D - 1 && k < n; ++k) staging = stage_block(k);

    // ---- per-request state of this warp's kv head -------------------------------------
    uint32_t seg_key = 0xFFFFFFFFu;
    int L = 0, seg_nblk = 0, seg_skip = 0, hq0 = 0, seg_b = 0;
    const int hh0 = warp * kGqaGroup;  // this warp's first record row in the group
    int64_t seg_start = 0;
    uint32_t qb[8][2];           // Q as the B operand of S^T = K Q^T (dims permuted like K)
    float qz0 = 0.f, qz1 = 0.f;  // sm_scale log2(e) sum(q) of this lane's two heads
    // O^T: dims (tile i, rows g / g + 8) x columns (2t, 2t + 1); columns 0-3 take
    // tokens 0-7 of every block, columns 4-7 tokens 8-15, of heads 0-3
    float o[8][4] = {};
    float R[4] = {};             // sum of the rounded P' per column
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;

    auto flush = [&]() {
      // the lanes of heads (2 hp, 2 hp + 1): t and t ^ 2, every g; columns 2t + u
      // and 2t + u + 4 hold the two token halves of head 2 hp + u
#pragma unroll
      for (int off = 2; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, off);
        l1 += __shfl_xor_sync(kFull, l1, off);
        z0 += __shfl_xor_sync(kFull, z0, off);
        z1 += __shfl_xor_sync(kFull, z1, off);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[i][c] += __shfl_xor_sync(kFull, o[i][c], 2);
      R[0] += __shfl_xor_sync(kFull, R[0], 2);
      R[1] += __shfl_xor_sync(kFull, R[1], 2);
      if (tsel != 0) return;  // lanes t = 2, 3 now hold copies
      const bool contained = seg_start >= x0 && seg_start + seg_nblk <= x0 + n;
      const int64_t row0 = static_cast<int64_t>(seg_b) * a.q_heads + hq0;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int hh = 2 * t + u;
        const float l = u ? l1 : l0, m = u ? m1 : m0;
        const float corr = (u ? z1 : z0) - kMid * R[u];
        float acc[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          // INT4 output rows fed by a nibble at bits 4-7 (odd i) carry 16 c
          const float sc = (KV == kI4 && (i & 1)) ? kTwo24 / 16.f : kTwo24;
          acc[i] = fmaf(o[i][u], sc, corr);
          acc[8 + i] = fmaf(o[i][2 + u], sc, corr);
        }
        if (contained) {
          float mm = m, ll = l;
          if (seg_skip > 0) merge_prefix(a, row0 + hh, seg_skip, g, mm, ll, acc);
          const float inv = ll > 0.f ? 1.f / ll : 0.f;
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = pack2<false>(acc[2 * i] * inv, acc[2 * i + 1] * inv);
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) +
                                                (row0 + hh) * kHeadDim + 16 * g);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
          const int slot = seg_start <= x0 ? 0 : 1;  // the request holding x0, else the last one
          float* rec = a.part + ((rid * 2 + slot) * a.hpg + hh0 + hh) * kPartStride;
          float4* ov = reinterpret_cast<float4*>(rec + 16 * g);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            ov[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
          if (g == 0) {
            rec[kHeadDim] = m;
            rec[kHeadDim + 1] = l;
          }
        }
      }
    };

    for (int k = 0; k < n; ++k) {
      if (staging && k + D - 1 < n) staging = stage_block(k + D - 1);
      const uint32_t s = n_used % D;
      const uint32_t st = stage0 + s * SB;
      if (!mbar_wait_or_abort(full0 + 8 * s, (n_used / D) & 1u, abort_s)) {
        if (lane == 0 && *abort_s == 0) {
          report(a.dev_err, KVQ_DEV_ERR_TIMEOUT);
          *abort_s = 1;
        }
        return false;
      }
      ++n_used;
      // (head group << 16 | request, block; all ones for a block id outside the pool)
      const uint2 info = lds64(st + S::info_off(W));
      const bool blk_ok = info.y != 0xFFFFFFFFu;
      const int j = static_cast<int>(info.y);

      if (info.x != seg_key) {
        if (seg_key != 0xFFFFFFFFu) flush();
        seg_key = info.x;
        const int hgi = static_cast<int>(info.x >> 16);
        seg_b = static_cast<int>(info.x & 0xFFFFu);
        seg_start = static_cast<int64_t>(hgi) * tb + cum[seg_b];
        seg_nblk = cum[seg_b + 1] - cum[seg_b];
        L = lown[seg_b];
        seg_skip = skip_of(a, seg_b);
        hq0 = (hgi * W + warp) * kGqaGroup;
        // Q of head hq0 + (g mod 4) (columns 4-7 repeat 0-3), dims [32t, 32t + 32)
        uint32_t qw[16];
        const uint4* qp = reinterpret_cast<const uint4*>(
            static_cast<const uint16_t*>(a.q) +
            (static_cast<int64_t>(seg_b) * a.q_heads + hq0 + (g & 3)) * kHeadDim + 32 * t);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = qp[i];
          qw[4 * i] = v.x; qw[4 * i + 1] = v.y; qw[4 * i + 2] = v.z; qw[4 * i + 3] = v.w;
        }
        if constexpr (KV == kI4) {
          // k-step 2j: dims (8j, 8j+4) and (8j+2, 8j+6) of the lane's 32 (nibbles at
          // bits 0-3); k-step 2j + 1: (8j+1, 8j+5) and (8j+3, 8j+7) (bits 4-7)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            qb[2 * jj][0] = prmt(qw[4 * jj], qw[4 * jj + 2], 0x5410u);
            qb[2 * jj][1] = prmt(qw[4 * jj + 1], qw[4 * jj + 3], 0x5410u);
            qb[2 * jj + 1][0] = prmt(qw[4 * jj], qw[4 * jj + 2], 0x7632u);
            qb[2 * jj + 1][1] = prmt(qw[4 * jj + 1], qw[4 * jj + 3], 0x7632u);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            qb[kk][0] = qw[2 * kk];
            qb[kk][1] = qw[2 * kk + 1];
          }
        }
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) part += half_lo(qw[i]) + half_hi(qw[i]);
        part += __shfl_xor_sync(kFull, part, 1);
        part += __shfl_xor_sync(kFull, part, 2);  // lanes 4h hold sum(q) of head h
        qz0 = lsc * __shfl_sync(kFull, part, (2 * hp) * 4);
        qz1 = lsc * __shfl_sync(kFull, part, (2 * hp + 1) * 4);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        R[0] = R[1] = R[2] = R[3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = z0 = z1 = 0.f;
      }

      if (blk_ok) {
        const uint32_t ksz = lds32(st + szo), vsz = lds32(st + szo + 64 * W);
        // ---- S^T = K Q^T: class-A k-steps into sa, class-B into sb -------------------
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (KV == kI4) {
          const uint4 k0 = lds128(st + kro[0][0]), k1 = lds128(st + kro[1][0]);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint32_t w0 = w4(k0, jj), w1 = w4(k1, jj);  // rows g, g + 8
            const uint32_t y0 = w0 >> 8, y1 = w1 >> 8;
            const uint32_t aa[4] = {w0 & kLoNib, w1 & kLoNib, y0 & kLoNib, y1 & kLoNib};
            mma16816<false>(sa, aa, qb[2 * jj]);
            const uint32_t ab[4] = {w0 & kHiNib, w1 & kHiNib, y0 & kHiNib, y1 & kHiNib};
            mma16816<false>(sb, ab, qb[2 * jj + 1]);
          }
        } else {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint4 k0 = lds128(st + kro[0][half]), k1 = lds128(st + kro[1][half]);
#pragma unroll
            for (int q2 = 0; q2 < 4; q2 += 2) {
              const int kk = 4 * half + q2;
              const uint32_t w0 = w4(k0, q2), w1 = w4(k1, q2);
              const uint32_t aa[4] = {bytes_sub(w0, 0x4140u), bytes_sub(w1, 0x4140u),
                                      bytes_sub(w0, 0x4342u), bytes_sub(w1, 0x4342u)};
              mma16816<false>(sa, aa, qb[kk]);
              const uint32_t v0 = w4(k0, q2 + 1), v1 = w4(k1, q2 + 1);
              const uint32_t ab[4] = {bytes_sub(v0, 0x4140u), bytes_sub(v1, 0x4140u),
                                      bytes_sub(v0, 0x4342u), bytes_sub(v1, 0x4342u)};
              mma16816<false>(sb, ab, qb[kk + 1]);
            }
          }
        }
        // this lane's token (row g or g + 8) and heads (2 hp, 2 hp + 1)
        const float d0a = KV == kI4 ? fmaf(sb[0], 1.f / 16.f, sa[0]) : sa[0] + sb[0];
        const float d1a = KV == kI4 ? fmaf(sb[1], 1.f / 16.f, sa[1]) : sa[1] + sb[1];
        const float d0b = KV == kI4 ? fmaf(sb[2], 1.f / 16.f, sa[2]) : sa[2] + sb[2];
        const float d1b = KV == kI4 ? fmaf(sb[3], 1.f / 16.f, sa[3]) : sa[3] + sb[3];
        const float d0 = tsel ? d0b : d0a, d1 = tsel ? d1b : d1a;
        const float sk = half_lo(ksz) * (kTwo24 * lsc), zk = half_hi(ksz);
        float s0 = fmaf(sk, d0, zk * qz0), s1 = fmaf(sk, d1, zk * qz1);
        if ((j + 1) * kBlock > L && j * kBlock + tau >= L) s0 = s1 = -INFINITY;
        const float sv = half_lo(vsz);
        // ---- online softmax: the running maximum moves when a score passes it by
        // more than the slack (by anything, for a token with a large V scale) ------
        const float slack = sv <= kSlackMaxScale ? kSlack : 0.f;
        if (__any_sync(kFull, s0 > m0 + slack || s1 > m1 + slack)) {
          float bm0 = s0, bm1 = s1;
#pragma unroll
          for (int off = 2; off < 32; off <<= 1) {
            bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, off));
            bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, off));
          }
          const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
          const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
          l0 *= al0; l1 *= al1; z0 *= al0; z1 *= al1;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[i][0] *= al0; o[i][2] *= al0;
            o[i][1] *= al1; o[i][3] *= al1;
          }
          R[0] *= al0; R[2] *= al0; R[1] *= al1; R[3] *= al1;
          m0 = mn0;
          m1 = mn1;
        }
        const float p0 = ex2(s0 - m0), p1 = ex2(s1 - m1);
        l0 += p0;
        l1 += p1;
        const float zm = fmaf(kMid, sv, half_hi(vsz));
        z0 = fmaf(p0, zm, z0);
        z1 = fmaf(p1, zm, z1);
        // P'^T as the B operand: tokens 0-7 into columns 0-3 (lanes t = 0, 1),
        // tokens 8-15 into columns 4-7 (lanes t = 2, 3); the rest zero
        const uint32_t hpk = pack2<false>(p0 * sv, p1 * sv);
        uint32_t bp[2];
        bp[0] = movmatrix_trans(tsel ? 0u : hpk);
        bp[1] = movmatrix_trans(tsel ? hpk : 0u);
        // ---- O^T += V^T P'^T over 8 tiles of 16 dims, and sum(P') ---------------------
        if constexpr (KV == kI4) {
          const uint2 v0 = lds64(st + vro[0]), v1 = lds64(st + vro[1]);  // rows 2t, 2t+1
          const uint2 v2 = lds64(st + vro[2]), v3 = lds64(st + vro[3]);  // rows 2t+8, 2t+9
          // two rows side by side: lo halves = the first row's 4 dims, hi halves
          // = the second row's
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const uint32_t sel = hf ? 0x7632u : 0x5410u;
            const uint32_t x0 = prmt(v0.x, v1.x, sel), x1 = prmt(v0.y, v1.y, sel);
            const uint32_t y0 = prmt(v2.x, v3.x, sel), y1 = prmt(v2.y, v3.y, sel);
            const uint32_t x0s = x0 >> 8, x1s = x1 >> 8, y0s = y0 >> 8, y1s = y1 >> 8;
            // tile i = 4 hf + p: output rows g -> dim 16g + i, g + 8 -> 16g + 8 + i
            {
              const uint32_t av[4] = {x0 & kLoNib, x1 & kLoNib, y0 & kLoNib, y1 & kLoNib};
              mma16816<false>(o[4 * hf + 0], av, bp);
            }
            {
              const uint32_t av[4] = {x0 & kHiNib, x1 & kHiNib, y0 & kHiNib, y1 & kHiNib};
              mma16816<false>(o[4 * hf + 1], av, bp);
            }
            {
              const uint32_t av[4] = {x0s & kLoNib, x1s & kLoNib, y0s & kLoNib, y1s & kLoNib};
              mma16816<false>(o[4 * hf + 2], av, bp);
            }
            {
              const uint32_t av[4] = {x0s & kHiNib, x1s & kHiNib, y0s & kHiNib, y1s & kHiNib};
              mma16816<false>(o[4 * hf + 3], av, bp);
            }
          }
        } else {
          const uint4 v0 = lds128(st + vro[0]), v1 = lds128(st + vro[1]);
          const uint4 v2 = lds128(st + vro[2]), v3 = lds128(st + vro[3]);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            // words hf (dims 16g + 4hf + 0..3) and 2 + hf (dims 16g + 8 + 4hf + 0..3)
            const uint32_t r0a = w4(v0, hf), r1a = w4(v1, hf);
            const uint32_t r0b = w4(v0, 2 + hf), r1b = w4(v1, 2 + hf);
            const uint32_t r2a = w4(v2, hf), r3a = w4(v3, hf);
            const uint32_t r2b = w4(v2, 2 + hf), r3b = w4(v3, 2 + hf);
#pragma unroll
            for (int pp = 0; pp < 2; ++pp) {
              // bytes (2pp, 2pp+1) of the two rows interleaved
              const uint32_t sel = pp ? 0x7362u : 0x5140u;
              const uint32_t xa = prmt(r0a, r1a, sel), xb = prmt(r0b, r1b, sel);
              const uint32_t ya = prmt(r2a, r3a, sel), yb = prmt(r2b, r3b, sel);
              {
                const uint32_t av[4] = {bytes_sub(xa, 0x4140u), bytes_sub(xb, 0x4140u),
                                        bytes_sub(ya, 0x4140u), bytes_sub(yb, 0x4140u)};
                mma16816<false>(o[4 * hf + 2 * pp], av, bp);
              }
              {
                const uint32_t av[4] = {bytes_sub(xa, 0x4342u), bytes_sub(xb, 0x4342u),
                                        bytes_sub(ya, 0x4342u), bytes_sub(yb, 0x4342u)};
                mma16816<false>(o[4 * hf + 2 * pp + 1], av, bp);
              }
            }
          }
        }
        {
          const uint32_t ones[4] = {kOnes, kOnes, kOnes, kOnes};
          mma16816<false>(R, ones, bp);
        }
      }
      __syncwarp();  // every lane is done with the stage
      if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
    if (seg_key != 0xFFFFFFFFu) flush();
    return true;
  };

  // ---- this CTA's ranges: its static range, then tail chunks ---------------------------
  const RangeMap& rm = sp.rm;
  bool alive = true;
  if (rm.k > 0) {  // the same cut in every head group
    if (cta < static_cast<int64_t>(sp.groups) * rm.k) {
      const int64_t hgi = cta / rm.k, i = cta - hgi * rm.k;
      const int64_t lo = i * rm.Pst;
      if (lo < tb)
        alive = run_range(hgi * tb + lo,
                          static_cast<int>(min(tb - lo, static_cast<int64_t>(rm.Pst))), cta);
    }
  } else {
    const int64_t xs = static_cast<int64_t>(cta) * rm.Pst;
    if (xs < sp.static_end)
      alive = run_range(
          xs, static_cast<int>(min(sp.static_end - xs, static_cast<int64_t>(rm.Pst))), cta);
    if constexpr (TAIL) {
      while (rm.C > 0) {
        __syncthreads();  // every warp is done with the previous range
        if (tid == 0) *chunk_s = *abort_s ? -1 : static_cast<int32_t>(atomicAdd(a.tail_ctr, 1u));
        __syncthreads();
        const int32_t c = *chunk_s;
        if (c < 0 || static_cast<int64_t>(c) >= rm.ntail) break;
        const int64_t x0 = sp.static_end + static_cast<int64_t>(c) * rm.C;
        alive = run_range(x0, static_cast<int>(min(sp.total - x0, static_cast<int64_t>(rm.C))),
                          sp.nwarps + c) && alive;
      }
    }
  }
  (void)alive;
  // nothing may still be copied into shared memory when the CTA exits: after a
  // timeout, the stages staged but not read are waited for (bounded)
  __syncthreads();
  if (tid == 0) {
    const int zero = 0;
    for (uint32_t i = n_used; i < n_staged; ++i)
      mbar_wait_or_abort(full0 + 8 * (i % D), (i / D) & 1u, &zero);
  }
}

template <int KV, bool TAIL>
__global__ void __launch_bounds__(kMaxCtaHeads * 32, 2)
    decode_gqa_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(1024) unsigned char dsmem[];
  __shared__ int32_t warp_sum[kMaxCtaHeads];
  __shared__ int abort_s;
  __shared__ int32_t chunk_s;
  // the combine kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;");
  gqa_body<KV, TAIL>(a, dsmem, warp_sum, &abort_s, &chunk_s, blockIdx.x, gridDim.x);
}

template <int KV, bool TAIL>
cudaError_t launch_gqa_t(const DecodeArgs& a, int grid, cudaStream_t s) {
  thread_local int opted_in_device = -1;  // per host thread: no shared state
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (opted_in_device != dev) {
    e = cudaFuncSetAttribute(decode_gqa_kernel<KV, TAIL>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(gqa_smem_bytes<KV>(kMaxBatch, kMaxCtaHeads)));
    if (e != cudaSuccess) return e;
    opted_in_device = dev;
  }
  decode_gqa_kernel<KV, TAIL>
      <<<grid, a.cta_heads * 32, gqa_smem_bytes<KV>(a.batch, a.cta_heads), s>>>(a);
  return cudaGetLastError();
}

template <int KV, bool TAIL>
int gqa_occupancy_t(int batch, int w) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  thread_local int cached_dev = -1, cached_batch = -1, cached_w = -1, cached_n = 0;
  if (dev == cached_dev && batch == cached_batch && w == cached_w) return cached_n;
  if (cudaFuncSetAttribute(decode_gqa_kernel<KV, TAIL>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(gqa_smem_bytes<KV>(kMaxBatch, kMaxCtaHeads))) !=
      cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_gqa_kernel<KV, TAIL>, w * 32,
                                                    gqa_smem_bytes<KV>(batch, w)) != cudaSuccess)
    return 0;
  cached_dev = dev;
  cached_batch = batch;
  cached_w = w;
  cached_n = n;
  return n;
}

}  // namespace

int decode_gqa_cta_heads(int kv_heads) {
  if (kv_heads <= kMaxCtaHeads) return kv_heads;
  return kv_heads % kMaxCtaHeads == 0 ? kMaxCtaHeads : 0;
}

bool decode_gqa_supported(int kv_dtype, int q_dtype, int group, int kv_heads) {
  return (kv_dtype == kI8 || kv_dtype == kI4) && q_dtype == kF16 && group == kGqaGroup &&
         decode_gqa_cta_heads(kv_heads) > 0;
}

cudaError_t launch_decode_gqa(const DecodeArgs& a, int kv_dtype, int grid, cudaStream_t s) {
  const bool tail = a.tail_ctr != nullptr;
  if (kv_dtype == kI8)
    return tail ? launch_gqa_t<kI8, true>(a, grid, s) : launch_gqa_t<kI8, false>(a, grid, s);
  if (kv_dtype == kI4)
    return tail ? launch_gqa_t<kI4, true>(a, grid, s) : launch_gqa_t<kI4, false>(a, grid, s);
  return cudaErrorInvalidValue;
}

int decode_gqa_ctas_per_sm(int kv_dtype, int batch, int w, bool tail) {
  if (kv_dtype == kI8)
    return tail ? gqa_occupancy_t<kI8, true>(batch, w) : gqa_occupancy_t<kI8, false>(batch, w);
  if (kv_dtype == kI4)
    return tail ? gqa_occupancy_t<kI4, true>(batch, w) : gqa_occupancy_t<kI4, false>(batch, w);
  return 0;
}

}  // namespace kvq

// kvq_decode_gqa: single-token decode attention over INT8 / INT4 pools for
// queries in fp16 with 4 q heads per kv head (grouped-query attention).
//
// LMDeploy article (devpress.csdn.net) §2.4: INT8/INT4 KV with a per-token,
// per-head (scale, zero); §2.2: 16-token blocks reached through block tables;
// §3.2 item 3 and §4.2: generation attention reads the paged KV through
// indirect block pointers in its own hand-written kernel.
//
// The work split is the general decode kernel's (kvq_decode_common.cuh: one
// stream of (kv head, request, block) units, a persistent grid, equal ranges
// per warp, partial records merged by the combine kernel). With 4 q heads per
// kv head a unit carries 4-8 times fewer bytes per query than with one, and
// the instructions spent per unit, not DRAM, set the pace; everything below
// is arranged to spend few.
//
// Staging. Every warp keeps a ring of kDepth stages. All 32 lanes stage a
// unit with 16-byte cp.async copies (the 16 K and the 16 V rows of one kv
// head, each row's chunks XOR-swizzled so that the fragment reads hit
// distinct banks, and the 64-byte scale/zero runs), and lane 0 leaves the
// unit's position (kv head, request, block) in the stage for the compute
// side. A tensor copy issued by one lane would move only 1-2 KB here, and
// measured costlier per unit: its operands must first be made warp-uniform.
// Physical block ids and positions come 32 units at a time: lane i of the
// warp locates unit k0 + i of its range (binary search over the per-request
// block offsets in shared memory) and loads its block id, one window ahead of
// the unit being issued.
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
// scores instead of four. One shuffle brings token g + 8's weights back to
// the lanes that feed them to the P.V product, whose columns 4-7 are zero.
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
constexpr uint32_t kLoNib = 0x000F000Fu;  // nibble at bits 0-3 of each half: c
constexpr uint32_t kHiNib = 0x00F000F0u;  // nibble at bits 4-7 of each half: 16 c
constexpr float kTwo24 = 16777216.f;      // 2^24: one code unit of the subnormal encoding
constexpr uint32_t kOnes = 0x3C003C00u;   // fp16 pair (1, 1)
constexpr float kSlack = 8.f;             // the running maximum may lag the scores by this
constexpr float kSlackMaxScale = 240.f;   // ... while V scales stay below this (2^8 S_v < 2^16)

// Per-warp ring of stages: [K tiles][V tiles][scale/zero runs][unit
// positions], 1024-byte aligned (the swizzle pattern repeats every 512 /
// 1024 bytes).
template <int KV>
struct GqaStage {
  static constexpr int kRow = KvTraits<KV>::kRowBytes;  // 64 (INT4) or 128 (INT8)
  static constexpr int kTile = kBlock * kRow;
  static constexpr int kDepth = 4;
  static constexpr int kVOff = kDepth * kTile;
  static constexpr int kSzOff = 2 * kDepth * kTile;
  static constexpr int kInfoOff = kSzOff + kDepth * 128;
  static constexpr int kWarpBytes = (kInfoOff + kDepth * 8 + 1023) / 1024 * 1024;
  static constexpr int kChunks = kRow / 16;                // 16-byte chunks per row
  static constexpr int kCopies = kBlock * kChunks / 32;    // per lane per tile
  // chunk c of row r sits at chunk c ^ swz(r): the 128-byte pattern (r mod 8)
  // for 128-byte rows, the 64-byte pattern ((r / 2) mod 4) for 64-byte rows
  __host__ __device__ static constexpr int at(int r, int c) {
    return r * kRow + (c ^ (kRow == 64 ? ((r >> 1) & 3) : (r & 7))) * 16;
  }
};

// Dynamic shared memory: [blocks before request b, batch + 1][own tokens of
// request b, batch][slack to 1024 bytes][the warps' stage rings].
template <int KV>
__host__ __device__ constexpr size_t gqa_smem_bytes(int batch) {
  return align128((2 * batch + 1) * sizeof(int32_t)) + 1024 +
         static_cast<size_t>(kWarps) * GqaStage<KV>::kWarpBytes;
}

// Two codes as the fp16 subnormal pair selected by sel from word w's bytes
// and zero bytes (INT8): [w.b_lo, 0, w.b_hi, 0].
__device__ __forceinline__ uint32_t bytes_sub(uint32_t w, uint32_t sel) {
  return prmt(w, 0u, sel);
}

__device__ __forceinline__ uint2 lds64u(uint32_t addr) { return lds64(addr); }

__device__ __forceinline__ void sts64(uint32_t addr, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(x), "r"(y) : "memory");
}

template <int KV, bool TAIL>
__device__ __forceinline__ void gqa_body(const DecodeArgs& a, unsigned char* dsmem,
                                         int32_t* warp_sum, int cta, int ncta) {
  using S = GqaStage<KV>;
  constexpr int D = S::kDepth;
  constexpr float kMid = KV == kI8 ? 128.f : 8.f;
  constexpr bool kLockstep = KV != kI4;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int tsel = t >> 1;       // 0: this lane scores token g, 1: token g + 8
  const int hp = t & 1;          // ... for q heads 2 hp and 2 hp + 1 of the group
  const int tau = g + 8 * tsel;  // that token's row in the block

  const StreamPlan sp = plan_stream<false, TAIL>(a, dsmem, warp_sum, cta, ncta, kLockstep,
                                                 /*own_lens=*/true);
  const int32_t* cum = sp.cum;
  const int32_t* lown = sp.cum + a.batch + 1;  // tokens of request b's own blocks
  const int tb = sp.tb;
  const int64_t gw = static_cast<int64_t>(cta) * kWarps + warp;

  const uint32_t region0 =
      (static_cast<uint32_t>(__cvta_generic_to_shared(sp.stages)) + 1023u) & ~1023u;
  const uint32_t wr = region0 + static_cast<uint32_t>(warp * S::kWarpBytes);
  // this lane's copies: chunk n = lane + 32 i of a tile (row n / kChunks)
  uint32_t csrc[S::kCopies], cdst[S::kCopies];
#pragma unroll
  for (int i = 0; i < S::kCopies; ++i) {
    const int n = lane + 32 * i, r = n / S::kChunks, c = n % S::kChunks;
    csrc[i] = static_cast<uint32_t>(r * a.kv_heads * S::kRow + c * 16);
    cdst[i] = S::at(r, c);
  }
  // lanes 0-3 copy the 64 bytes of K scale/zero pairs, lanes 4-7 those of V
  const uint32_t* const sz_src = (lane < 4 ? a.k_sz : a.v_sz) + 4 * (lane & 3);

  // fragment offsets of this lane in a stage's K and V tiles
  uint32_t kro[2][S::kRow / 64];  // rows g, g + 8: dims [32t, 32t + 32)
  uint32_t vro[4];                // rows 2t, 2t+1, 2t+8, 2t+9: dims [16g, 16g + 16)
#pragma unroll
  for (int i = 0; i < S::kRow / 64; ++i) {
    kro[0][i] = S::at(g, (S::kRow / 64) * t + i);
    kro[1][i] = S::at(g + 8, (S::kRow / 64) * t + i);
  }
  {
    const int rows[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
    for (int r = 0; r < 4; ++r)
      vro[r] = KV == kI4 ? S::at(rows[r], g >> 1) + 8 * (g & 1) : S::at(rows[r], g);
  }
  const float kq = a.sm_scale_log2;

  auto run_range = [&](const int64_t x0, const int n, const int64_t rid) -> bool {
    // ---- issue side: windows of 32 units located lane-parallel ---------------------
    // lane i of window w holds unit 32 w + i of the range: its block id and its
    // position packed as (kv head << 16 | request, block)
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
    int32_t wphys, nphys;
    uint32_t wkey, nkey;
    int32_t wblk, nblk_;
    locate_window(0, wphys, wkey, wblk);
    locate_window(1, nphys, nkey, nblk_);
    const uint32_t nb32 = static_cast<uint32_t>(a.num_blocks);  // valid ids are below this
    auto issue_unit = [&](const int ST, const int kq) {
      const int kk = kq & 31;
      if (kk == 0 && kq > 0) {  // next window; locate the one after it
        wphys = nphys; wkey = nkey; wblk = nblk_;
        locate_window((kq >> 5) + 1, nphys, nkey, nblk_);
      }
      const int32_t phys = __shfl_sync(kFull, wphys, kk);
      const uint32_t key = __shfl_sync(kFull, wkey, kk);
      const int32_t blk = __shfl_sync(kFull, wblk, kk);
      const bool ok = static_cast<uint32_t>(phys) < nb32;
      if (lane == 0) {
        sts64(wr + S::kInfoOff + 8 * ST, key, ok ? static_cast<uint32_t>(blk) : 0xFFFFFFFFu);
        if (!ok) report(a.dev_err, KVQ_DEV_ERR_BLOCK_ID);
      }
      if (ok) {
        // row r of the (block, head) tile: ((phys * 16 + r) * kv_heads + h) * kRow
        const int h = static_cast<int>(key >> 16);
        const int64_t ph = static_cast<int64_t>(phys) * a.kv_heads + h;
        const int64_t base = (static_cast<int64_t>(phys) * kBlock * a.kv_heads + h) * S::kRow;
        const uint8_t* kb = a.k + base;
        const uint8_t* vb = a.v + base;
        const uint32_t kd = wr + ST * S::kTile, vd = wr + S::kVOff + ST * S::kTile;
#pragma unroll
        for (int i = 0; i < S::kCopies; ++i) {
          cp_async16(kd + cdst[i], kb + csrc[i]);
          cp_async16(vd + cdst[i], vb + csrc[i]);
        }
        if (lane < 8) cp_async16(wr + S::kSzOff + 128 * ST + 16 * lane, sz_src + ph * kBlock);
      }
    };
    // stage ST receives unit kq of the range (nothing past its end); every call
    // commits one cp.async group, so that the wait below always counts kDepth - 1
    auto issue = [&](const int ST, const int kq) {
      if (kq < n) issue_unit(ST, kq);
      cp_async_commit();
    };
#pragma unroll
    for (int k = 0; k < D - 1; ++k) issue(k, k);

    // ---- per-request state -----------------------------------------------------------
    uint32_t seg_key = 0xFFFFFFFFu;
    int L = 0, seg_nblk = 0, seg_skip = 0, hq0 = 0, seg_b = 0;
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
      const bool contained = seg_start >= x0 && seg_start + seg_nblk <= x0 + n;
      const int64_t row0 = static_cast<int64_t>(seg_b) * a.q_heads + hq0;
      if (tsel == 0) {  // lanes t = 2, 3 hold copies
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
            for (int i = 0; i < 8; ++i)
              w[i] = pack2<false>(acc[2 * i] * inv, acc[2 * i + 1] * inv);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) +
                                                  (row0 + hh) * kHeadDim + 16 * g);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          } else {
            const int slot = seg_start <= x0 ? 0 : 1;  // the request holding x0, else the last
            float* rec = a.part + ((rid * 2 + slot) * a.hpg + hh) * kPartStride;
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
      }
    };

    // unit k of the range in stage ST
    auto step = [&](const int ST, const int k) {
      issue(ST == 0 ? D - 1 : ST - 1, k + D - 1);  // the stage unit k - 1 used
      cp_async_wait<D - 1>();  // this lane's copies of unit k have landed
      __syncwarp();            // ... and every other lane's
      // (kv head << 16 | request, block; all ones for a block id outside the pool)
      const uint2 info = lds64u(wr + S::kInfoOff + 8 * ST);
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
        hq0 = hgi * kGqaGroup;
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
        qz0 = kq * __shfl_sync(kFull, part, (2 * hp) * 4);
        qz1 = kq * __shfl_sync(kFull, part, (2 * hp + 1) * 4);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        R[0] = R[1] = R[2] = R[3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = z0 = z1 = 0.f;
      }

      if (blk_ok) {
        const uint32_t kKt = ST * S::kTile, kVt = S::kVOff + ST * S::kTile;
        const uint32_t szp = wr + S::kSzOff + 128 * ST + 4 * tau;
        const uint32_t ksz = lds32(szp), vsz = lds32(szp + 64);
        // ---- S^T = K Q^T: class-A k-steps into sa, class-B into sb -------------------
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (KV == kI4) {
          const uint4 k0 = lds128(wr + kKt + kro[0][0]), k1 = lds128(wr + kKt + kro[1][0]);
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
            const uint4 k0 = lds128(wr + kKt + kro[0][half]);
            const uint4 k1 = lds128(wr + kKt + kro[1][half]);
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
        const float xa0 = tsel ? sa[2] : sa[0], xa1 = tsel ? sa[3] : sa[1];
        const float xb0 = tsel ? sb[2] : sb[0], xb1 = tsel ? sb[3] : sb[1];
        const float d0 = KV == kI4 ? fmaf(xb0, 1.f / 16.f, xa0) : xa0 + xb0;
        const float d1 = KV == kI4 ? fmaf(xb1, 1.f / 16.f, xa1) : xa1 + xb1;
        const float sk = half_lo(ksz) * (kTwo24 * kq), zk = half_hi(ksz);
        float s0 = fmaf(sk, d0, zk * qz0), s1 = fmaf(sk, d1, zk * qz1);
        if (j * kBlock + tau >= L) s0 = s1 = -INFINITY;
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
          const uint2 v0 = lds64(wr + kVt + vro[0]), v1 = lds64(wr + kVt + vro[1]);
          const uint2 v2 = lds64(wr + kVt + vro[2]), v3 = lds64(wr + kVt + vro[3]);
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
          const uint4 v0 = lds128(wr + kVt + vro[0]), v1 = lds128(wr + kVt + vro[1]);
          const uint4 v2 = lds128(wr + kVt + vro[2]), v3 = lds128(wr + kVt + vro[3]);
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
      __syncwarp();  // all lanes are done with this stage before it is refilled
    };

    for (int k = 0, st = 0; k < n; ++k, st = st == D - 1 ? 0 : st + 1) step(st, k);
    cp_async_wait<0>();
    if (seg_key != 0xFFFFFFFFu) flush();
    return true;
  };

  for_each_range<TAIL>(a, sp, gw, lane, run_range);
}

template <int KV, bool TAIL>
__global__ void __launch_bounds__(kDecodeThreads, 4)
    decode_gqa_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  __shared__ int32_t warp_sum[kWarps];
  // the combine kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;");
  gqa_body<KV, TAIL>(a, dsmem, warp_sum, blockIdx.x, gridDim.x);
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
                             static_cast<int>(gqa_smem_bytes<KV>(kMaxBatch)));
    if (e != cudaSuccess) return e;
    opted_in_device = dev;
  }
  decode_gqa_kernel<KV, TAIL><<<grid, kDecodeThreads, gqa_smem_bytes<KV>(a.batch), s>>>(a);
  return cudaGetLastError();
}

template <int KV, bool TAIL>
int gqa_occupancy_t(int batch) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  thread_local int cached_dev = -1, cached_batch = -1, cached_n = 0;
  if (dev == cached_dev && batch == cached_batch) return cached_n;
  if (cudaFuncSetAttribute(decode_gqa_kernel<KV, TAIL>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(gqa_smem_bytes<KV>(kMaxBatch))) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_gqa_kernel<KV, TAIL>,
                                                    kDecodeThreads,
                                                    gqa_smem_bytes<KV>(batch)) != cudaSuccess)
    return 0;
  cached_dev = dev;
  cached_batch = batch;
  cached_n = n;
  return n;
}

}  // namespace

bool decode_gqa_supported(int kv_dtype, int q_dtype, int group) {
  return (kv_dtype == kI8 || kv_dtype == kI4) && q_dtype == kF16 && group == kGqaGroup;
}

cudaError_t launch_decode_gqa(const DecodeArgs& a, int kv_dtype, int grid, cudaStream_t s) {
  const bool tail = a.tail_ctr != nullptr;
  if (kv_dtype == kI8)
    return tail ? launch_gqa_t<kI8, true>(a, grid, s) : launch_gqa_t<kI8, false>(a, grid, s);
  if (kv_dtype == kI4)
    return tail ? launch_gqa_t<kI4, true>(a, grid, s) : launch_gqa_t<kI4, false>(a, grid, s);
  return cudaErrorInvalidValue;
}

int decode_gqa_ctas_per_sm(int kv_dtype, int batch, bool tail) {
  if (kv_dtype == kI8)
    return tail ? gqa_occupancy_t<kI8, true>(batch) : gqa_occupancy_t<kI8, false>(batch);
  if (kv_dtype == kI4)
    return tail ? gqa_occupancy_t<kI4, true>(batch) : gqa_occupancy_t<kI4, false>(batch);
  return 0;
}

}  // namespace kvq

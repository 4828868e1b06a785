// kvq_tile.cuh: shared-memory staging of 16-token (block, kv head) tiles and
// the register fragments the attention kernels feed to mma.sync.
//
// LMDeploy article (devpress.csdn.net) §2.2: 16-token blocks reached through
// per-sequence block tables; §2.4: INT8/INT4 codes with a per-token, per-head
// (scale, zero). Both the single-query decode kernel and the shared-prefix
// kernel read a block through the same stages and unpack it into the same
// operand fragments; they differ only in which operand the codes become.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

constexpr int kWarps = kDecodeThreads / 32;
constexpr int kHeadsPerGroup = 8;  // mma N
constexpr unsigned kFull = 0xFFFFFFFFu;

// ---- per-block fragments ------------------------------------------------------

// Raw bytes one lane needs from one 16-token block (K rows g, g+8; V rows
// 2t, 2t+1, 2t+8, 2t+9) plus the scale/zero words of tokens g and g+8.
template <int KV>
struct Frag;

template <>
struct Frag<kF16> {
  uint4 k[2][4];   // 64 bytes of each K row: dims [32t, 32t+32)
  uint4 v[4][2];   // 32 bytes of each V row: dims [16g, 16g+16)
  uint32_t ksz[2], vsz[2];
};
template <>
struct Frag<kBF16> : Frag<kF16> {};
template <>
struct Frag<kI8> {
  uint4 k[2][2];   // 32 bytes: dims [32t, 32t+32)
  uint4 v[4];      // 16 bytes: dims [16g, 16g+16)
  uint32_t ksz[2], vsz[2];
};
template <>
struct Frag<kI4> {
  uint4 k[2];      // 16 bytes: dims [32t, 32t+32)
  uint2 v[4];      // 8 bytes: dims [16g, 16g+16)
  uint32_t ksz[2], vsz[2];
};

// Offset a of the code encoding a + c on the K side (Q's type) and V side,
// and the middle code (2^(b-1)).
template <int KV, bool QBF>
struct CodeOffset {
  static constexpr float kK = KV == kI8 ? (QBF ? -128.f : 1024.f) : (QBF ? 128.f : 16.f);
  static constexpr float kV = KV == kI8 ? -128.f : 16.f;
  static constexpr float kMid = KV == kI8 ? 128.f : 8.f;
  // the rounded-P' correction is needed only when the V codes are not centred
  static constexpr bool kPCorr = KV == kI4;
};

// ---- shared-memory staging -------------------------------------------------------

// Every warp owns kDepth stages; stage st holds one 16-token block of one kv
// head: the K tile and the V tile (16 rows of kRow bytes) and, for quantized
// pools, the 16 (scale, zero) pairs of K and of V. The 16-byte chunks of a
// tile row are XOR-swizzled so that the fragment reads below fall on distinct
// banks. INT8 tiles arrive by TMA (one 4-D tensor copy per tile with the
// hardware's 128-byte swizzle, completion on a per-stage mbarrier); the other
// kinds by per-lane 16-byte cp.async with the same pattern (64-byte pattern
// for 64-byte rows) applied by hand.
//   per warp: [K tiles][V tiles][scale/zero][mbarriers], 1024-byte aligned
template <int KV>
struct Stage {
  static constexpr int kRow = KvTraits<KV>::kRowBytes;
  static constexpr int kChunks = kRow / 16;                // 16-byte chunks per row
  static constexpr int kTile = kBlock * kRow;
  // TMA for INT8 tiles (2 KB boxes); INT4 tiles (1 KB) stream faster through
  // per-lane cp.async (measured on the same GPU: 57 vs 64 us for the INT4
  // GQA-4 workload)
  static constexpr bool kTma = KV == kI8;
  static constexpr int kCopies = kBlock * kChunks / 32;    // cp.async chunks per lane per tile
  static constexpr int kKReads = kChunks / 4;              // 16-byte K reads per row
  static constexpr int kVReads = kChunks >= 8 ? kChunks / 8 : 1;  // V reads per row
  // blocks in flight per warp (about 8-16 KB of KV per warp)
  static constexpr int kDepth = KV == kI4 ? 4 : (KV == kI8 ? 4 : 2);
  static constexpr int kVOff = kDepth * kTile;
  static constexpr int kSzOff = 2 * kDepth * kTile;
  static constexpr int kBarOff = kSzOff + kDepth * 128;
  static constexpr int kWarpBytes = (kBarOff + kDepth * 8 + 1023) / 1024 * 1024;
  static constexpr int kTxBytes = kTma ? 2 * kTile + 128 : 0;  // bytes one TMA stage receives
  // chunk c of row r sits at chunk c ^ swz_bits(r): the 128-byte pattern
  // (r mod 8) for 128- and 256-byte rows, the 64-byte pattern ((r / 2) mod 4)
  // for 64-byte rows
  __host__ __device__ static constexpr int swz_bits(int r) {
    return kRow == 64 ? ((r >> 1) & 3) : (r & 7);
  }
  __host__ __device__ static constexpr int at(int r, int c) {
    return r * kRow + (c ^ swz_bits(r)) * 16;
  }
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 r;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(addr));
  return r;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(addr));
  return r;
}

// ---- mbarrier / TMA -------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arm(uint32_t bar, uint32_t tx_bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx_bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase of parity `parity` of the barrier; gives up after 2 s.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > 2000000000ull) return false;
  }
  return true;
}
__device__ __forceinline__ void tma_tile_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 2^x by the hardware approximation (relative error about 2^-22; tiny
// results flush to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Per-lane constants of the fragment reads from a stage (and of the cp.async
// copies into it); only the stage base and the block's address change.
template <int KV>
struct LaneMap {
  using S = Stage<KV>;
  uint32_t src[S::kTma ? 1 : S::kCopies];  // byte offset within the tile's global rows
  uint32_t dst[S::kTma ? 1 : S::kCopies];  // byte offset within the tile
  uint32_t kr[2][S::kKReads];              // K fragment reads (offset in the K tile)
  uint32_t vr[4][S::kVReads];              // V fragment reads (offset in the V tile)
  __device__ __forceinline__ void init(int lane, int g, int t, uint32_t tok_stride) {
    if constexpr (!S::kTma) {
#pragma unroll
      for (int i = 0; i < S::kCopies; ++i) {
        const int n = lane + 32 * i;
        const int r = n / S::kChunks, c = n % S::kChunks;
        src[i] = r * tok_stride + c * 16;
        dst[i] = S::at(r, c);
      }
    }
#pragma unroll
    for (int i = 0; i < S::kKReads; ++i) {
      const int c = S::kKReads * t + i;
      kr[0][i] = S::at(g, c);
      kr[1][i] = S::at(g + 8, c);
    }
    const int rows[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if constexpr (KV == kI4) {
        vr[r][0] = S::at(rows[r], g >> 1) + 8 * (g & 1);
      } else {
#pragma unroll
        for (int i = 0; i < S::kVReads; ++i) vr[r][i] = S::at(rows[r], S::kVReads * g + i);
      }
    }
  }
};

// The warp starts the copy of block `phys` of kv head h into stage st of its
// region `wr` (shared address). TMA path: lane 0 arms the stage's barrier and
// issues two tile copies and two 64-byte scale/zero copies. cp.async path:
// every lane copies its chunks; the caller commits the group.
template <int KV, class Args>
__device__ __forceinline__ void issue_block(uint32_t wr, int st, const Args& a,
                                            const LaneMap<KV>& lm, int64_t phys, int h,
                                            int lane) {
  using S = Stage<KV>;
  const uint32_t kdst = wr + st * S::kTile, vdst = wr + S::kVOff + st * S::kTile;
  if constexpr (S::kTma) {
    if (lane == 0) {
      const uint32_t bar = wr + S::kBarOff + 8 * st;
      const uint32_t sz = wr + S::kSzOff + 128 * st;
      const int64_t szi = (phys * a.kv_heads + h) * kBlock;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // after the reads of the last use
      mbar_arm(bar, S::kTxBytes);
      tma_tile_4d(kdst, &a.k_map, 0, h, 0, static_cast<int>(phys), bar);
      tma_tile_4d(vdst, &a.v_map, 0, h, 0, static_cast<int>(phys), bar);
      bulk_copy(sz, a.k_sz + szi, 64, bar);
      bulk_copy(sz + 64, a.v_sz + szi, 64, bar);
    }
  } else {
    const int64_t base = (phys * kBlock * a.kv_heads + h) * S::kRow;
    const uint8_t* kb = a.k + base;
    const uint8_t* vb = a.v + base;
#pragma unroll
    for (int i = 0; i < S::kCopies; ++i) {
      cp_async16(kdst + lm.dst[i], kb + lm.src[i]);
      cp_async16(vdst + lm.dst[i], vb + lm.src[i]);
    }
    if constexpr (KvTraits<KV>::kQuant) {
      // lanes 0-3 copy the 64 bytes of K scale/zero pairs, lanes 4-7 those of V
      if (lane < 8) {
        const uint32_t* src =
            (lane < 4 ? a.k_sz : a.v_sz) + (phys * a.kv_heads + h) * kBlock + 4 * (lane & 3);
        cp_async16(wr + S::kSzOff + 128 * st + 16 * lane, src);
      }
    }
  }
}

// This lane's fragment bytes of the block in stage st, and (kSz) the
// scale/zero words of tokens g and g+8.
template <int KV, bool kSz = true>
__device__ __forceinline__ void read_frag(Frag<KV>& f, uint32_t wr, int st,
                                          const LaneMap<KV>& lm, int g) {
  using S = Stage<KV>;
  const uint32_t kt = wr + st * S::kTile, vt = wr + S::kVOff + st * S::kTile;
  if constexpr (KV == kF16 || KV == kBF16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f.k[0][i] = lds128(kt + lm.kr[0][i]);
      f.k[1][i] = lds128(kt + lm.kr[1][i]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      f.v[r][0] = lds128(vt + lm.vr[r][0]);
      f.v[r][1] = lds128(vt + lm.vr[r][1]);
    }
  } else if constexpr (KV == kI8) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      f.k[0][i] = lds128(kt + lm.kr[0][i]);
      f.k[1][i] = lds128(kt + lm.kr[1][i]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) f.v[r] = lds128(vt + lm.vr[r][0]);
  } else {
    f.k[0] = lds128(kt + lm.kr[0][0]);
    f.k[1] = lds128(kt + lm.kr[1][0]);
#pragma unroll
    for (int r = 0; r < 4; ++r) f.v[r] = lds64(vt + lm.vr[r][0]);
  }
  if constexpr (KvTraits<KV>::kQuant && kSz) {
    const uint32_t sz = wr + S::kSzOff + 128 * st + 4 * g;
    f.ksz[0] = lds32(sz);
    f.ksz[1] = lds32(sz + 32);
    f.vsz[0] = lds32(sz + 64);
    f.vsz[1] = lds32(sz + 96);
  }
}

__device__ __forceinline__ uint32_t w4(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// A operand of S^T = K Q^T for k-step kk: rows = tokens (g, g+8),
// k-columns = this lane's dims (see the header comment).
template <int KV, bool QBF>
__device__ __forceinline__ void k_operand(const Frag<KV>& f, int kk, uint32_t (&a)[4]) {
  if constexpr (KV == kF16 || KV == kBF16) {
    a[0] = w4(f.k[0][kk >> 1], (2 * kk) & 3);
    a[2] = w4(f.k[0][kk >> 1], (2 * kk + 1) & 3);
    a[1] = w4(f.k[1][kk >> 1], (2 * kk) & 3);
    a[3] = w4(f.k[1][kk >> 1], (2 * kk + 1) & 3);
  } else if constexpr (KV == kI8) {
    const uint32_t w0 = w4(f.k[0][kk >> 2], kk & 3);
    const uint32_t w1 = w4(f.k[1][kk >> 2], kk & 3);
    if constexpr (QBF) {
      a[0] = bytes_to_bf16_pair(w0, 0, 1);
      a[2] = bytes_to_bf16_pair(w0, 2, 3);
      a[1] = bytes_to_bf16_pair(w1, 0, 1);
      a[3] = bytes_to_bf16_pair(w1, 2, 3);
    } else {
      a[0] = bytes_to_f16_offset(w0, 0x4140u);
      a[2] = bytes_to_f16_offset(w0, 0x4342u);
      a[1] = bytes_to_f16_offset(w1, 0x4140u);
      a[3] = bytes_to_f16_offset(w1, 0x4342u);
    }
  } else {
    // kk = 2 j + u: pairs of dims (8j+2u, 8j+2u+4) and (8j+2u+1, 8j+2u+5)
    const int j = kk >> 1, u = kk & 1;
    const uint32_t w0 = w4(f.k[0], j), w1 = w4(f.k[1], j);
    a[0] = nibbles_to_pair<QBF>(w0, 2 * u);
    a[2] = nibbles_to_pair<QBF>(w0, 2 * u + 1);
    a[1] = nibbles_to_pair<QBF>(w1, 2 * u);
    a[3] = nibbles_to_pair<QBF>(w1, 2 * u + 1);
  }
}

// A operand of O^T += V^T P'^T for dim step i: rows = dims (16g + 2i,
// 16g + 2i + 1), k-columns = tokens (2t, 2t+1, 2t+8, 2t+9). The product runs
// in bf16 only for bf16 pools; quantized codes always go in as fp16.
template <int KV>
__device__ __forceinline__ void v_operand(const Frag<KV>& f, int i, uint32_t (&a)[4]) {
  if constexpr (KV == kF16 || KV == kBF16) {
    const uint32_t r0 = w4(f.v[0][i >> 2], i & 3), r1 = w4(f.v[1][i >> 2], i & 3);
    const uint32_t r2 = w4(f.v[2][i >> 2], i & 3), r3 = w4(f.v[3][i >> 2], i & 3);
    a[0] = prmt(r0, r1, 0x5410u);
    a[1] = prmt(r0, r1, 0x7632u);
    a[2] = prmt(r2, r3, 0x5410u);
    a[3] = prmt(r2, r3, 0x7632u);
  } else if constexpr (KV == kI8) {
    const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;  // bytes k, k+1 of two rows, k = 2(i%2)
    const uint32_t x01 = prmt(w4(f.v[0], i >> 1), w4(f.v[1], i >> 1), sel);
    const uint32_t x23 = prmt(w4(f.v[2], i >> 1), w4(f.v[3], i >> 1), sel);
    a[0] = bytes_to_f16(x01, 0x4140u);
    a[1] = bytes_to_f16(x01, 0x4342u);
    a[2] = bytes_to_f16(x23, 0x4140u);
    a[3] = bytes_to_f16(x23, 0x4342u);
  } else {
    // i = 4 jj + 2 kk + m: bytes (2kk, 2kk+1) of word jj of the two rows,
    // nibbles 2m and 2m+1 of each half
    const int jj = i >> 2, kk = (i >> 1) & 1, m = i & 1;
    const uint32_t sel = kk ? 0x7632u : 0x5410u;
    const uint32_t r0 = jj ? f.v[0].y : f.v[0].x, r1 = jj ? f.v[1].y : f.v[1].x;
    const uint32_t r2 = jj ? f.v[2].y : f.v[2].x, r3 = jj ? f.v[3].y : f.v[3].x;
    const uint32_t x01 = prmt(r0, r1, sel), x23 = prmt(r2, r3, sel);
    a[0] = nibbles_to_pair<false>(x01, 2 * m);
    a[1] = nibbles_to_pair<false>(x01, 2 * m + 1);
    a[2] = nibbles_to_pair<false>(x23, 2 * m);
    a[3] = nibbles_to_pair<false>(x23, 2 * m + 1);
  }
}

__device__ __forceinline__ float half_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

template <bool QBF>
__device__ __forceinline__ void store_out(void* out, int64_t idx, float v) {
  if constexpr (QBF) {
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(out)[idx] = __float2half_rn(v);
  }
}

__host__ __device__ constexpr size_t align128(size_t x) { return (x + 127) / 128 * 128; }

}  // namespace kvq

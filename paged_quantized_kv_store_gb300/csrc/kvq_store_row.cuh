// kvq_store_row.cuh: the quantizing store of one pool row, shared by the
// store kernel and the fused decode step.
//
// "pymllm Runtime Design", section "KV cache 与 prefix cache": KVPool rows
// are written through a store kernel (store_cache) at the kv indices the
// allocator handed out. LMDeploy article (devpress.csdn.net) §2.4: per-head,
// per-token asymmetric INT8/INT4 quantization, min/max computed online.
// All quantizer arithmetic is explicit IEEE fp32 (__fsub_rn, __fdiv_rn,
// __float2int_rn round-half-even) and __float2half_rn, so codes, scales and
// zeros are reproducible bit for bit.
#pragma once

#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

template <bool BF>
__device__ __forceinline__ void unpack8(const uint4& w, float (&x)[8]) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = lo_to_float<BF>(v[i]);
    x[2 * i + 1] = hi_to_float<BF>(v[i]);
  }
}

// A pool row's inputs, loaded ahead of its quantization so that a caller
// can have the loads of several rows in flight at once.
struct RowIn {
  int64_t slot;  // destination kv index; < 0 for a padding token or a row past the end
  uint4 w;       // this lane's 8 input elements
  int h, which;  // kv head, 0 = K / 1 = V
  bool in_range;
};

// One (token, K-or-V, kv head) row by the 16 lanes of a half-warp (lane16 =
// lane % 16), every lane of the half-warp taking part (a row past the end
// inactive): the slot and the input elements.
template <int KV, bool IN_BF>
__device__ __forceinline__ RowIn load_row(const StoreArgs& a, int64_t row, int lane16) {
  const int64_t rows = a.num_tokens * 2 * a.kv_heads;
  RowIn in;
  in.in_range = row < rows;
  // row = (token * 2 + which) * kv_heads + head, below 2^32 (kv_store_quant
  // refuses larger stores): one 32-bit division
  const uint32_t r = in.in_range ? static_cast<uint32_t>(row) : 0u;
  const uint32_t kvh = static_cast<uint32_t>(a.kv_heads);
  const uint32_t q = r / kvh;
  in.h = static_cast<int>(r - q * kvh);
  in.which = static_cast<int>(q & 1u);
  const int64_t t = static_cast<int64_t>(q >> 1);
  in.slot = in.in_range ? a.slot_mapping[t] : -1;
  const uint16_t* src = static_cast<const uint16_t*>(in.which ? a.v_new : a.k_new) +
                        (t * a.kv_heads + in.h) * kHeadDim + lane16 * 8;
  in.w = in.in_range ? *reinterpret_cast<const uint4*>(src) : make_uint4(0, 0, 0, 0);
  return in;
}

// The row's quantization and its writes (codes, then the scale/zero pair by
// lane 0); a slot past the pool is skipped and flagged.
template <int KV, bool IN_BF>
__device__ __forceinline__ void write_row(const StoreArgs& a, const RowIn& in, int lane16) {
  const unsigned hmask = 0xFFFFu << (threadIdx.x & 16u);  // this half-warp's lanes
  const int64_t slot = in.slot;
  const bool past_pool = slot >= a.num_blocks * kBlock;
  const bool active = in.in_range && slot >= 0 && !past_pool;
  if (in.in_range && past_pool && lane16 == 0 && in.h == 0 && in.which == 0)
    report(a.dev_err, KVQ_DEV_ERR_SLOT);
  const uint4 w = active ? in.w : make_uint4(0, 0, 0, 0);
  uint8_t* pool = static_cast<uint8_t*>(in.which ? a.v_pool : a.k_pool);
  const int64_t dst_row = slot * a.kv_heads + in.h;  // slot * Hkv + h

  if constexpr (!KvTraits<KV>::kQuant) {
    if (active)
      *reinterpret_cast<uint4*>(pool + dst_row * KvTraits<KV>::kRowBytes + lane16 * 16) = w;
    return;
  } else {
    constexpr int kQmax = KV == kI8 ? 255 : 15;
    float x[8];
    unpack8<IN_BF>(w, x);
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      mn = fminf(mn, x[i]);
      mx = fmaxf(mx, x[i]);
    }
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(hmask, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(hmask, mx, off));
    }
    if (!active) return;
    mn = __fadd_rn(mn, 0.0f);  // a -0 extreme is stored as +0
    mx = __fadd_rn(mx, 0.0f);
    const float s32 = __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(kQmax));
    const __half sh = __float2half_rn(s32);
    const __half zh = __float2half_rn(mn);
    const float S = __half2float(sh);
    const float Z = __half2float(zh);
    const bool degenerate = !(S > 0.0f) || isinf(S) || !isfinite(Z);
    // code = rint(fl((x - Z) / S)) with the division's correct rounding. The
    // row's one reciprocal stands in for the eight divisions: with inv =
    // fl(1 / S), fl(d * inv) is within 1.5 * 2^-23 |d / S| of fl(d / S) (two
    // roundings of 2^-24 against one), so both round to the same integer
    // unless fl(d * inv) lies within that distance of a tie k + 1/2; there
    // (tested with the wider margin 2^-20 |q|) the correctly rounded division
    // decides. The codes are those of the division, bit for bit.
    // A degenerate row takes inv = 0: every quotient is 0 (or NaN when Z is not
    // finite), which converts to code 0 and never looks like a tie.
    const float inv = degenerate ? 0.f : __frcp_rn(S);
    uint32_t c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float d = __fsub_rn(x[i], Z);
      float qf = __fmul_rn(d, inv);
      // |qf - rint(qf)| is qf's distance to the nearest integer; qf lies within
      // 2^-20 |qf| (+ 2^-30) of a tie k + 1/2 exactly when that distance plus
      // the margin reaches 1/2
      const float r = rintf(qf);
      if (fmaf(fabsf(qf), 0x1p-20f, fabsf(__fsub_rn(qf, r))) >= 0.5f - 0x1p-30f)
        qf = rintf(__fdiv_rn(d, S));
      else
        qf = r;
      // round-half-even already done; negative codes saturate to 0
      c[i] = min(__float2uint_rn(qf), static_cast<unsigned>(kQmax));
    }
    if constexpr (KV == kI8) {
      uint2 o;
      o.x = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
      o.y = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
      *reinterpret_cast<uint2*>(pool + dst_row * KvTraits<KV>::kRowBytes + lane16 * 8) = o;
    } else {
      // two codes per byte, the even index in the low nibble
      const uint32_t o = c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12) | (c[4] << 16) |
                         (c[5] << 20) | (c[6] << 24) | (c[7] << 28);
      *reinterpret_cast<uint32_t*>(pool + dst_row * KvTraits<KV>::kRowBytes + lane16 * 4) = o;
    }
    if (lane16 == 0) {
      const int64_t blk = slot / kBlock, off = slot % kBlock;
      uint32_t* sz = static_cast<uint32_t*>(in.which ? a.v_sz : a.k_sz);
      const uint32_t pair = static_cast<uint32_t>(__half_as_ushort(sh)) |
                            (static_cast<uint32_t>(__half_as_ushort(zh)) << 16);
      sz[(blk * a.kv_heads + in.h) * kBlock + off] = pair;
    }
  }
}

// load_row then write_row.
template <int KV, bool IN_BF>
__device__ __forceinline__ void store_row(const StoreArgs& a, int64_t row, int lane16) {
  write_row<KV, IN_BF>(a, load_row<KV, IN_BF>(a, row, lane16), lane16);
}

}  // namespace kvq

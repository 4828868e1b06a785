// kvq_store: write new K/V rows into pool slots, quantizing on the way for
// INT8/INT4 pools.
//
// "pymllm Runtime Design", section "KV cache 与 prefix cache": KVPool rows
// are written through a store kernel (store_cache) at the kv indices the
// allocator handed out. LMDeploy article (devpress.csdn.net) §2.4: per-head,
// per-token asymmetric INT8/INT4 quantization, min/max computed online.
//
// Work decomposition: one (token, K-or-V, kv head) row of 128 elements per
// 16 lanes; each lane owns 8 consecutive elements (one 16-byte load). The
// row's min and max come from a 4-step xor-shuffle butterfly inside the
// half-warp. Rows of one token are adjacent in both the input and the pool,
// so a warp's two rows are contiguous reads and writes.
//
// Bit-exactness: all quantizer arithmetic is explicit IEEE fp32 (__fsub_rn,
// __fdiv_rn, __float2int_rn round-half-even) and __float2half_rn; no fused or
// approximate operation touches a code, a scale or a zero.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kStoreThreads = 256;
constexpr int kRowsPerCta = kStoreThreads / 16;

template <bool BF>
__device__ __forceinline__ void unpack8(const uint4& w, float (&x)[8]) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = lo_to_float<BF>(v[i]);
    x[2 * i + 1] = hi_to_float<BF>(v[i]);
  }
}

template <int KV, bool IN_BF>
__global__ void __launch_bounds__(kStoreThreads)
    store_kernel(StoreArgs a) {
  const int lane16 = threadIdx.x & 15;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 4);
  const int64_t rows = a.num_tokens * 2 * a.kv_heads;
  const bool in_range = row < rows;
  // row = (token * 2 + which) * kv_heads + head
  const int64_t r = in_range ? row : 0;
  const int h = static_cast<int>(r % a.kv_heads);
  const int which = static_cast<int>((r / a.kv_heads) & 1);
  const int64_t t = r / (2 * a.kv_heads);

  const int64_t slot = in_range ? a.slot_mapping[t] : -1;
  const bool past_pool = slot >= a.num_blocks * kBlock;
  const bool active = in_range && slot >= 0 && !past_pool;
  if (in_range && past_pool && lane16 == 0 && h == 0 && which == 0)
    report(a.dev_err, KVQ_DEV_ERR_SLOT);

  const uint16_t* src = static_cast<const uint16_t*>(which ? a.v_new : a.k_new) +
                        (t * a.kv_heads + h) * kHeadDim + lane16 * 8;
  uint4 w = make_uint4(0, 0, 0, 0);
  if (active) w = *reinterpret_cast<const uint4*>(src);

  uint8_t* pool = static_cast<uint8_t*>(which ? a.v_pool : a.k_pool);
  const int64_t dst_row = slot * a.kv_heads + h;  // slot * Hkv + h

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
      mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
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
    uint32_t c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int q = degenerate ? 0 : __float2int_rn(__fdiv_rn(__fsub_rn(x[i], Z), S));
      q = min(max(q, 0), kQmax);
      c[i] = static_cast<uint32_t>(q);
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
      uint32_t* sz = static_cast<uint32_t*>(which ? a.v_sz : a.k_sz);
      const uint32_t pair = static_cast<uint32_t>(__half_as_ushort(sh)) |
                            (static_cast<uint32_t>(__half_as_ushort(zh)) << 16);
      sz[(blk * a.kv_heads + h) * kBlock + off] = pair;
    }
  }
}

template <int KV, bool IN_BF>
cudaError_t launch(const StoreArgs& a, cudaStream_t s) {
  const int64_t rows = a.num_tokens * 2 * a.kv_heads;
  const int64_t ctas = (rows + kRowsPerCta - 1) / kRowsPerCta;
  if (ctas > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
  store_kernel<KV, IN_BF><<<static_cast<unsigned>(ctas), kStoreThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_store(const StoreArgs& a, cudaStream_t s) {
  if (a.num_tokens == 0) return cudaSuccess;
  const bool in_bf = a.in_dtype == kBF16;
  switch (a.kv_dtype) {
    case kF16:
      return launch<kF16, false>(a, s);
    case kBF16:
      return launch<kBF16, true>(a, s);
    case kI8:
      return in_bf ? launch<kI8, true>(a, s) : launch<kI8, false>(a, s);
    case kI4:
      return in_bf ? launch<kI4, true>(a, s) : launch<kI4, false>(a, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace kvq

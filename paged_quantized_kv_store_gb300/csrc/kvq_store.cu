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
#include "kvq_store_row.cuh"

namespace kvq {
namespace {

constexpr int kStoreThreads = 256;
constexpr int kRowsPerCta = kStoreThreads / 16;

template <int KV, bool IN_BF>
__global__ void __launch_bounds__(kStoreThreads)
    store_kernel(StoreArgs a) {
  store_row<KV, IN_BF>(a, static_cast<int64_t>(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 4),
                       threadIdx.x & 15);
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

// kvq_copy: whole-block copy between two pools by an id map.
//
// LMDeploy article (devpress.csdn.net) §4.4 "Block Manager 与缓存交换": the
// cache engine swaps blocks between the GPU and the CPU cache by a
// {dst: src} map, moving the K and V rows of each block. Within one pool the
// same copy forks a shared block before a request writes into it. A block is
// four contiguous runs in the pool layout: its K tile and V tile (16 rows x
// kv_heads x row bytes each) and, for quantized pools, its K and V
// (scale, zero) runs (kv_heads x 16 x 4 bytes each). Either pool may sit in
// pinned host memory that the GPU addresses directly (unified addressing):
// the kernel then reads or writes host memory over the CPU-GPU link.
//
// Grid: x = block pairs, y = pieces of a pair; a CTA moves up to kPiece
// 16-byte chunks of its pair, every thread kUnroll of them with all loads
// issued before the stores. Streaming cache hints: a copied block is not
// read again by this kernel.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 8;
constexpr int kPiece = kCopyThreads * kUnroll;  // 16-byte chunks per CTA

__global__ void __launch_bounds__(kCopyThreads) copy_kernel(const CopyArgs a) {
  const int64_t i = blockIdx.x;
  const int32_t s = a.src_ids[i], d = a.dst_ids[i];
  if (s < 0 || s >= a.src_blocks || d < 0 || d >= a.dst_blocks) {
    if (blockIdx.y == 0 && threadIdx.x == 0) report(a.dev_err, KVQ_DEV_ERR_BLOCK_ID);
    return;
  }
  const int64_t tile = a.tile_chunks, sz = a.sz_chunks;  // per run, in 16-byte chunks
  const int64_t per_pair = 2 * tile + 2 * sz;
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kPiece + threadIdx.x;
  uint4 v[kUnroll];
  const uint4* src[kUnroll];
  uint4* dst[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t c = c0 + static_cast<int64_t>(u) * kCopyThreads;
    src[u] = nullptr;
    dst[u] = nullptr;
    if (c < per_pair) {
      if (c < tile) {
        src[u] = a.src_k + s * tile + c;
        dst[u] = a.dst_k + d * tile + c;
      } else if (c < 2 * tile) {
        src[u] = a.src_v + s * tile + (c - tile);
        dst[u] = a.dst_v + d * tile + (c - tile);
      } else if (c < 2 * tile + sz) {
        src[u] = a.src_k_sz + s * sz + (c - 2 * tile);
        dst[u] = a.dst_k_sz + d * sz + (c - 2 * tile);
      } else {
        src[u] = a.src_v_sz + s * sz + (c - 2 * tile - sz);
        dst[u] = a.dst_v_sz + d * sz + (c - 2 * tile - sz);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u)
    if (src[u] != nullptr) v[u] = __ldcs(src[u]);
#pragma unroll
  for (int u = 0; u < kUnroll; ++u)
    if (dst[u] != nullptr) __stcs(dst[u], v[u]);
}

}  // namespace

cudaError_t launch_copy(const CopyArgs& a, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int64_t per_pair = 2 * a.tile_chunks + 2 * a.sz_chunks;
  const int64_t pieces = (per_pair + kPiece - 1) / kPiece;
  if (n > 0x7FFFFFFFll || pieces > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(n), static_cast<unsigned>(pieces));
  copy_kernel<<<grid, kCopyThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq

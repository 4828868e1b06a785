// kvq_tables_item.cuh: the block-table builder's work on one table entry
// (a request's block), shared by the tables kernel and the fused decode step.
//
// "pymllm Runtime Design", section "KV cache 与 prefix cache": the
// ReqToTokenPool maps (request slot, position) to a kv index. LMDeploy article
// (devpress.csdn.net) §2.2: each sequence keeps a table of physical block ids,
// blocks of 16 tokens. Entry j of request b is the block of its position 16 j;
// every other position of the block must sit at the matching offset of the
// same block, which is checked as it goes.
#pragma once

#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

// Table entries item, item + stride, ... (U of them; item = b *
// max_blocks_per_seq + j, those past batch * max_blocks_per_seq skipped), each
// by the 16 lanes of a half-warp: lane16 checks position 16 j + lane16, lane 0
// writes entry j. The loads of all U items are issued before any is checked.
template <int U>
__device__ __forceinline__ void tables_blocks(const TablesArgs& a, int64_t item, int64_t stride,
                                              int lane16) {
  const unsigned hmask = 0xFFFFu << (threadIdx.x & 16u);  // this half-warp's lanes
  const int64_t total = static_cast<int64_t>(a.batch) * a.max_blocks_per_seq;
  const int cap = min(a.max_context_len, a.max_blocks_per_seq * kBlock);
  int b[U], j[U], r[U], L[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t it = item + u * stride;
    const bool in = it < total;
    b[u] = in ? static_cast<int>(it / a.max_blocks_per_seq) : -1;
    j[u] = in ? static_cast<int>(it - static_cast<int64_t>(b[u]) * a.max_blocks_per_seq) : 0;
    r[u] = in ? a.req_pool_indices[b[u]] : -1;
    L[u] = in ? a.seq_lens[b[u]] : 0;
  }
  int32_t s[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const bool slot_ok = b[u] >= 0 && r[u] >= 0 && r[u] < a.num_req_slots;
    const int p = j[u] * kBlock + lane16;
    s[u] = slot_ok && p < min(max(L[u], 0), cap)
               ? a.req_to_token[static_cast<int64_t>(r[u]) * a.max_context_len + p]
               : -1;
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (b[u] < 0) continue;  // the whole half-warp: one item per half-warp
    int32_t* bt = a.block_tables + static_cast<int64_t>(b[u]) * a.max_blocks_per_seq;
    const bool req_first = j[u] == 0 && lane16 == 0;
    if (r[u] < 0 || r[u] >= a.num_req_slots) {
      if (lane16 == 0) bt[j[u]] = -1;
      if (req_first) report(a.dev_err, KVQ_DEV_ERR_REQ_SLOT);
      continue;
    }
    int Lv = max(L[u], 0);
    if (Lv > cap) {
      if (req_first) report(a.dev_err, KVQ_DEV_ERR_LENGTH);
      Lv = cap;
    }
    const int32_t first = __shfl_sync(hmask, s[u], 0, 16);  // kv index of position 16 j
    const bool block_used = j[u] * kBlock < Lv;
    uint32_t err = 0;
    if (block_used && first < 0) err |= KVQ_DEV_ERR_KV_INDEX;
    if (lane16 == 0) bt[j[u]] = block_used && first >= 0 ? first / kBlock : -1;
    if (j[u] * kBlock + lane16 < Lv) {
      if (s[u] < 0) {
        err |= KVQ_DEV_ERR_KV_INDEX;
      } else {
        const int32_t blk = first >= 0 ? first / kBlock : -1;
        if (blk < 0 || s[u] != blk * kBlock + lane16) err |= KVQ_DEV_ERR_NOT_BLOCKED;
      }
    }
    report(a.dev_err, err);
  }
}

}  // namespace kvq

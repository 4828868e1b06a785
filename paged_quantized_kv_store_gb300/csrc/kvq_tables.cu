// kvq_tables: per-request block tables from ReqToTokenPool rows.
//
// "pymllm Runtime Design", section "KV cache 与 prefix cache": the
// ReqToTokenPool maps (request slot, position) to a kv index. LMDeploy article
// (devpress.csdn.net) §2.2: each sequence keeps a table of physical block ids,
// blocks of 16 tokens. Entry j of request b is the block of its position 16 j;
// every other position of the block must sit at the matching offset of the
// same block, which this kernel checks as it goes.
//
// One CTA per request; threads stride over table entries, then positions.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kTablesThreads = 256;

__global__ void __launch_bounds__(kTablesThreads) tables_kernel(TablesArgs a) {
  const int b = blockIdx.x;
  int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
  const int r = a.req_pool_indices[b];
  uint32_t err = 0;
  if (r < 0 || r >= a.num_req_slots) {
    for (int j = threadIdx.x; j < a.max_blocks_per_seq; j += blockDim.x) bt[j] = -1;
    if (threadIdx.x == 0) report(a.dev_err, KVQ_DEV_ERR_REQ_SLOT);
    return;
  }
  int L = max(a.seq_lens[b], 0);
  const int cap = min(a.max_context_len, a.max_blocks_per_seq * kBlock);
  if (L > cap) {
    err |= (threadIdx.x == 0) ? KVQ_DEV_ERR_LENGTH : 0u;
    L = cap;
  }
  const int32_t* row = a.req_to_token + static_cast<int64_t>(r) * a.max_context_len;
  const int nblk = (L + kBlock - 1) / kBlock;
  for (int j = threadIdx.x; j < a.max_blocks_per_seq; j += blockDim.x) {
    int32_t id = -1;
    if (j < nblk) {
      const int32_t first = row[j * kBlock];
      if (first >= 0)
        id = first / kBlock;
      else
        err |= KVQ_DEV_ERR_KV_INDEX;
    }
    bt[j] = id;
  }
  for (int p = threadIdx.x; p < L; p += blockDim.x) {
    const int32_t s = row[p];
    if (s < 0) {
      err |= KVQ_DEV_ERR_KV_INDEX;
      continue;
    }
    const int32_t first = row[(p / kBlock) * kBlock];
    const int32_t blk = first >= 0 ? first / kBlock : -1;
    if (blk < 0 || s != blk * kBlock + p % kBlock) err |= KVQ_DEV_ERR_NOT_BLOCKED;
  }
  report(a.dev_err, err);
}

}  // namespace

cudaError_t launch_tables(const TablesArgs& a, cudaStream_t s) {
  if (a.batch == 0) return cudaSuccess;
  tables_kernel<<<a.batch, kTablesThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq

// kvq_tables: per-request block tables from ReqToTokenPool rows.
//
// "pymllm Runtime Design", section "KV cache 与 prefix cache": the
// ReqToTokenPool maps (request slot, position) to a kv index. LMDeploy article
// (devpress.csdn.net) §2.2: each sequence keeps a table of physical block ids,
// blocks of 16 tokens. Entry j of request b is the block of its position 16 j;
// every other position of the block must sit at the matching offset of the
// same block, which this kernel checks as it goes.
//
// One thread per (request, position): grid.x runs over requests, grid.y over
// chunks of 256 positions of the table's span, so every check is a single
// round of loads.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kTablesThreads = 256;

__global__ void __launch_bounds__(kTablesThreads) tables_kernel(TablesArgs a) {
  const int b = blockIdx.x;
  const int p = blockIdx.y * kTablesThreads + threadIdx.x;  // position in the request
  const int span = a.max_blocks_per_seq * kBlock;
  if (p >= span) return;
  int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
  const int j = p / kBlock;
  const bool entry = (p % kBlock) == 0;
  const int r = a.req_pool_indices[b];
  if (r < 0 || r >= a.num_req_slots) {
    if (entry) bt[j] = -1;
    if (p == 0) report(a.dev_err, KVQ_DEV_ERR_REQ_SLOT);
    return;
  }
  int L = max(a.seq_lens[b], 0);
  const int cap = min(a.max_context_len, span);
  if (L > cap) {
    if (p == 0) report(a.dev_err, KVQ_DEV_ERR_LENGTH);
    L = cap;
  }
  const int32_t* row = a.req_to_token + static_cast<int64_t>(r) * a.max_context_len;
  uint32_t err = 0;
  int32_t first = -1;
  if (j * kBlock < L) {
    first = row[j * kBlock];
    if (first < 0) err |= KVQ_DEV_ERR_KV_INDEX;
  }
  if (entry) bt[j] = first >= 0 ? first / kBlock : -1;
  if (p < L) {
    const int32_t s = row[p];
    if (s < 0) {
      err |= KVQ_DEV_ERR_KV_INDEX;
    } else {
      const int32_t blk = first >= 0 ? first / kBlock : -1;
      if (blk < 0 || s != blk * kBlock + p % kBlock) err |= KVQ_DEV_ERR_NOT_BLOCKED;
    }
  }
  report(a.dev_err, err);
}

}  // namespace

cudaError_t launch_tables(const TablesArgs& a, cudaStream_t s) {
  if (a.batch == 0) return cudaSuccess;
  const int span = a.max_blocks_per_seq * kBlock;
  const dim3 grid(static_cast<unsigned>(a.batch),
                  static_cast<unsigned>((span + kTablesThreads - 1) / kTablesThreads));
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
  tables_kernel<<<grid, kTablesThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq

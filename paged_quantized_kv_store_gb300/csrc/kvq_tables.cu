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
#include "kvq_tables_item.cuh"

namespace kvq {
namespace {

constexpr int kTablesThreads = 256;

__global__ void __launch_bounds__(kTablesThreads) tables_kernel(TablesArgs a) {
  const int p = blockIdx.y * kTablesThreads + threadIdx.x;  // position in the request
  const int j = p / kBlock;  // a half-warp per table entry
  if (j < a.max_blocks_per_seq)
    tables_blocks<1>(a, static_cast<int64_t>(blockIdx.x) * a.max_blocks_per_seq + j, 0,
                     p % kBlock);
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

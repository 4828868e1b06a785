// paged_decode_attn_noalloc: paged decode attention for callers that cannot
// allocate device memory.
//
// paged_decode_attn needs a scratch buffer (the split-K partial results) that
// the caller allocates and passes in. Some callers have no way to do that:
// an operator plugged into an inference engine that only hands it the input
// and output tensors, code that runs where all device memory must be reserved
// when the program is loaded, or a latency-critical loop where an allocation
// (and the device synchronization cudaMalloc can imply) is not acceptable.
// This entry point takes the scratch from a fixed array that lives in the
// library itself, so the call allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds KVQ_NOALLOC_SCRATCH_BYTES of it until the process exits. Host
// code cannot use the array's name as a device address (on the host it names
// a shadow variable), so the device address is looked up with
// cudaGetSymbolAddress, with the caller's device current, on every call. The
// address is not cached: it belongs to the module as loaded in the current
// context, and a context made anew on the same device (after
// cudaDeviceReset, or another context the caller makes current) loads the
// module again, possibly elsewhere. Once the module is loaded in a context
// the lookup is a host-side table read.
#include <cuda_runtime.h>

#include "kvq.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context, or nullptr.
void* scratch_in_current_context() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
  return p;
}

}  // namespace

extern "C" kvq_status paged_decode_attn_noalloc(
    const kvq_pool* pool, const void* q, int32_t q_dtype, void* out,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
    int32_t batch, int32_t q_heads, int32_t max_seq_len, float sm_scale, int32_t num_splits,
    int32_t* dev_err, void* stream) {
  if (pool == nullptr) return KVQ_ERR_INVALID_ARG;
  kvq_decode_plan plan;
  const kvq_status st = paged_decode_attn_plan(batch, q_heads, pool->kv_heads, pool->head_dim,
                                               max_seq_len, num_splits, 0, &plan);
  if (st != KVQ_OK) return st;
  // sizes whose static ranges need more scratch than the array holds are
  // refused by paged_decode_attn itself (KVQ_ERR_WORKSPACE, nothing launched)
  void* scratch = scratch_in_current_context();
  if (scratch == nullptr) return KVQ_ERR_CUDA;
  return paged_decode_attn(pool, q, q_dtype, out, block_tables, max_blocks_per_seq, seq_lens,
                           batch, q_heads, max_seq_len, sm_scale, num_splits, scratch,
                           static_cast<size_t>(KVQ_NOALLOC_SCRATCH_BYTES), dev_err, stream);
}

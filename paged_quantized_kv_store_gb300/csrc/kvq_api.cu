// C ABI of libkvq: argument validation, launch planning and dispatch.
// The declarations, with the passages of the source pages each entry point
// follows, are in include/kvq.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "kvq.h"
#include "kvq_internal.h"

using kvq::kBlock;
using kvq::kHeadDim;

namespace {

constexpr int kAutoMinBlocksPerWarp = 4;  // a warp's range is never shorter than this

// Decode workspace: [256 bytes: the tail-chunk counter, the fused step's
// barrier counter][header: 4 ints + batch + 1 prefix sums][partial records:
// 2 per q head of the group slot, per range; kRangesPerWarp ranges per warp of
// the plan, at least one (the static ranges alone) for a smaller workspace].
constexpr size_t kCounterBytes = 256;

size_t decode_records_offset(int32_t batch) {
  return kCounterBytes +
         (static_cast<size_t>(batch + kvq::kHdrCum + 1) * sizeof(int32_t) + 255) / 256 * 256;
}

size_t range_record_bytes(const kvq_decode_plan& p) {
  return static_cast<size_t>(2) * p.heads_per_group * kvq::kPartStride * sizeof(float);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_quant(int dt) { return dt == KVQ_INT8 || dt == KVQ_INT4; }
bool is_float16(int dt) { return dt == KVQ_F16 || dt == KVQ_BF16; }

kvq_status check_pool(const kvq_pool* p) {
  if (p == nullptr || p->k == nullptr || p->v == nullptr) return KVQ_ERR_INVALID_ARG;
  if (p->num_blocks < 0 || p->kv_heads <= 0) return KVQ_ERR_INVALID_ARG;
  if (p->block_size != kBlock || p->head_dim != kHeadDim) return KVQ_ERR_UNSUPPORTED;
  if (!is_quant(p->kv_dtype) && !is_float16(p->kv_dtype)) return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(p->k) || !aligned16(p->v)) return KVQ_ERR_INVALID_ARG;
  if (is_quant(p->kv_dtype)) {
    if (p->k_sz == nullptr || p->v_sz == nullptr) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(p->k_sz) || !aligned16(p->v_sz)) return KVQ_ERR_INVALID_ARG;
  }
  return KVQ_OK;
}

int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// cuTensorMapEncodeTiled, fetched from the driver through the runtime (no
// link-time dependency on the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  // looked up once, thread-safely (a function-local static's initializer)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// TMA view of a quantized K or V pool: [num_blocks][16][kv_heads][row bytes],
// one box = the 16 rows of one (block, head) tile, swizzled to match the
// decode kernel's reads (128-byte pattern for 128-byte rows, 64-byte pattern
// for 64-byte rows). No L2 promotion: a wider fetch would pull in the
// neighbouring head's row.
bool encode_pool_map(CUtensorMap* map, void* base, int64_t num_blocks, int kv_heads,
                     int row_bytes) {
  std::memset(map, 0, sizeof(*map));
  if (num_blocks <= 0) return true;  // no valid block id: no copy is ever issued
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(row_bytes),
                              static_cast<cuuint64_t>(kv_heads), 16,
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(row_bytes),
                                 static_cast<cuuint64_t>(kv_heads) * row_bytes,
                                 static_cast<cuuint64_t>(16) * kv_heads * row_bytes};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(row_bytes), 1, 16, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw =
      row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same pool as a 4-D view ordered [block][kv head][token][row] (token
// and head strides swapped), one box = the 16 rows of heads kv heads of one
// block, laid out head after head, each tile with the swizzle above: the
// grouped-query decode kernel stages a block for all heads of its CTA with
// one copy.
bool encode_pool_map_heads(CUtensorMap* map, void* base, int64_t num_blocks, int kv_heads,
                           int row_bytes, int heads) {
  std::memset(map, 0, sizeof(*map));
  if (num_blocks <= 0) return true;
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(row_bytes), 16,
                              static_cast<cuuint64_t>(kv_heads),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kv_heads) * row_bytes,
                                 static_cast<cuuint64_t>(row_bytes),
                                 static_cast<cuuint64_t>(16) * kv_heads * row_bytes};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(row_bytes), 16,
                             static_cast<cuuint32_t>(heads), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw =
      row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shared-prefix groups as the caller describes them.
struct PrefixDesc {
  const int32_t* offsets;
  const int32_t* members;
  const int32_t* shared_blocks;
  int num_groups;
  int num_members;
  int max_shared;
};

// Workspace of a shared-prefix decode: the plain decode's (length header and
// split-K records), then the per-request shared block counts, then one
// record per (request, q head, chunk of shared blocks).
struct SharedPrefixLayout {
  int chunk;       // shared blocks per prefix work unit
  int max_chunks;  // chunks of the longest shared prefix
  size_t skip_off, part_off, total;
};

SharedPrefixLayout shared_prefix_layout(const kvq_decode_plan& plan, int batch, int q_heads,
                                        int max_shared) {
  SharedPrefixLayout l;
  // about 8 chunks per prefix, 4 to 32 blocks each: enough units to fill the
  // device for a few dozen members, few records to merge per request
  l.chunk = std::min(kvq::kMaxPrefixChunk, std::max(4, (max_shared + 7) / 8));
  l.max_chunks = (max_shared + l.chunk - 1) / l.chunk;
  l.skip_off = align_up(plan.workspace_bytes, 256);
  l.part_off = l.skip_off + align_up(static_cast<size_t>(batch) * sizeof(int32_t), 256);
  l.total = l.part_off + static_cast<size_t>(batch) * q_heads * l.max_chunks * kvq::kPartStride *
                             sizeof(float);
  return l;
}

// Decode attention, plain (pd == nullptr) or with shared prefixes.
// The fused step's first phase (block tables and the store of the new
// tokens), when the decode runs as one launch with them.
struct StepPre {
  kvq::TablesArgs t;
  kvq::StoreArgs st;
};

// Workspace of the fused step: the decode's (its barrier counter sits in the
// counters at the start).
size_t step_workspace(const kvq_decode_plan& plan) { return plan.workspace_bytes; }

kvq_status decode_impl(const kvq_pool* pool, const void* q, int32_t q_dtype, void* out,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* seq_lens, int32_t batch, int32_t q_heads,
                       int32_t max_seq_len, float sm_scale, int32_t num_splits,
                       const PrefixDesc* pd, void* workspace, size_t workspace_bytes,
                       int32_t* dev_err, void* stream, const StepPre* pre = nullptr) {
  const kvq_status ps = check_pool(pool);
  if (ps != KVQ_OK) return ps;
  if (!is_float16(q_dtype)) return KVQ_ERR_UNSUPPORTED;
  if (is_float16(pool->kv_dtype) && q_dtype != pool->kv_dtype) return KVQ_ERR_UNSUPPORTED;
  if (batch < 0 || q_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0)
    return KVQ_ERR_INVALID_ARG;
  if (q_heads % pool->kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return KVQ_ERR_INVALID_ARG;
  kvq_decode_plan plan;
  const kvq_status st = paged_decode_attn_plan(batch, q_heads, pool->kv_heads, pool->head_dim,
                                               max_seq_len, num_splits, 0, &plan);
  if (st != KVQ_OK) return st;
  if (batch == 0) return KVQ_OK;
  if (q == nullptr || out == nullptr || block_tables == nullptr || seq_lens == nullptr)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q)) return KVQ_ERR_INVALID_ARG;
  const SharedPrefixLayout lay =
      shared_prefix_layout(plan, batch, q_heads, pd != nullptr ? pd->max_shared : 0);
  // the static ranges need one record slot per warp; the plan's size also holds
  // the tail's
  const size_t rec = range_record_bytes(plan);
  const size_t need = pd != nullptr ? lay.total
                                    : decode_records_offset(batch) + plan.warps * rec;
  if (workspace == nullptr || workspace_bytes < need) return KVQ_ERR_WORKSPACE;
  const size_t decode_bytes = pd != nullptr ? plan.workspace_bytes : workspace_bytes;
  if (!aligned16(workspace)) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(out)) return KVQ_ERR_INVALID_ARG;
  kvq::DecodeArgs a;
  std::memset(&a, 0, sizeof(a));
  // the grouped-query kernel (INT8 / INT4 pools, fp16 queries, 4 q heads per
  // kv head) serves the plain decode; the fused step keeps the general kernel
  const bool gqa = pre == nullptr && kvq::decode_gqa_supported(pool->kv_dtype, q_dtype,
                                                                q_heads / pool->kv_heads,
                                                                pool->kv_heads);
  const int cta_heads = gqa ? kvq::decode_gqa_cta_heads(pool->kv_heads) : 0;
  if (gqa) {  // one copy stages a block for the CTA's kv heads
    const int row = pool->kv_dtype == KVQ_INT8 ? kHeadDim : kHeadDim / 2;
    if (!encode_pool_map_heads(&a.kh_map, pool->k, pool->num_blocks, pool->kv_heads, row,
                               cta_heads) ||
        !encode_pool_map_heads(&a.vh_map, pool->v, pool->num_blocks, pool->kv_heads, row,
                               cta_heads))
      return KVQ_ERR_CUDA;
  }
  // the general INT8 kernels (decode, shared prefix, step) stage one tile per copy
  if (pool->kv_dtype == KVQ_INT8) {
    if (!encode_pool_map(&a.k_map, pool->k, pool->num_blocks, pool->kv_heads, kHeadDim) ||
        !encode_pool_map(&a.v_map, pool->v, pool->num_blocks, pool->kv_heads, kHeadDim))
      return KVQ_ERR_CUDA;
  } else {
    std::memset(&a.k_map, 0, sizeof(a.k_map));
    std::memset(&a.v_map, 0, sizeof(a.v_map));
  }
  a.k = static_cast<const uint8_t*>(pool->k);
  a.v = static_cast<const uint8_t*>(pool->v);
  a.k_sz = static_cast<const uint32_t*>(pool->k_sz);
  a.v_sz = static_cast<const uint32_t*>(pool->v_sz);
  a.num_blocks = pool->num_blocks;
  a.kv_heads = pool->kv_heads;
  a.q = q;
  a.out = out;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks_per_seq;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.q_heads = q_heads;
  a.group = q_heads / pool->kv_heads;
  a.head_groups = plan.head_groups;
  a.hpg = plan.heads_per_group;
  a.min_blocks_per_warp = plan.min_blocks_per_warp;
  const int nblk = std::max(1, (max_seq_len + kBlock - 1) / kBlock);
  a.len_cap = std::min(max_blocks_per_seq, nblk) * kBlock;
  a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  a.hdr = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + kCounterBytes);
  a.part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                    decode_records_offset(batch));
  a.max_ranges = std::min<int64_t>(
      static_cast<int64_t>((decode_bytes - decode_records_offset(batch)) / rec),
      static_cast<int64_t>(kvq::kRangesPerWarp) * plan.warps);
  // a tail needs an automatic split (an explicit count keeps every request to
  // num_splits + 1 pieces) and sizes whose per-range share can reach
  // kTailMinShare blocks
  int64_t max_total = static_cast<int64_t>(batch) * pool->kv_heads * plan.head_groups *
                      (a.len_cap / kBlock);
  int64_t ranges = plan.warps;
  int gqa_grid = 0;
  if (gqa) {
    // a CTA per group of cta_heads kv heads, one range each; at most
    // kMaxCtasPerSm * 4 warps per SM, as the workspace's records assume
    const int occ = kvq::decode_gqa_ctas_per_sm(pool->kv_dtype, batch, cta_heads, false);
    const int per_sm =
        std::min(occ, kvq::kMaxCtasPerSm * (kvq::kDecodeThreads / 32) / cta_heads);
    if (per_sm <= 0) return KVQ_ERR_CUDA;
    gqa_grid = plan.num_sms * per_sm;
    a.cta_heads = cta_heads;
    a.hpg = cta_heads * a.group;
    a.head_groups = 1;
    const size_t rec_g = static_cast<size_t>(2) * a.hpg * kvq::kPartStride * sizeof(float);
    a.max_ranges = std::min<int64_t>(
        static_cast<int64_t>((decode_bytes - decode_records_offset(batch)) / rec_g),
        static_cast<int64_t>(kvq::kRangesPerWarp) * gqa_grid);
    max_total = static_cast<int64_t>(batch) * (pool->kv_heads / cta_heads) * (a.len_cap / kBlock);
    ranges = gqa_grid;
  }
  const bool tail = num_splits == 0 && max_total >= int64_t{kvq::kTailMinShare} * ranges;
  a.tail_ctr = tail ? static_cast<unsigned int*>(workspace) : nullptr;
  a.dev_err = dev_err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((tail || pre != nullptr) &&
      cudaMemsetAsync(workspace, 0, 2 * sizeof(unsigned int), s) != cudaSuccess)
    return KVQ_ERR_CUDA;  // the tail counter and the step's barrier
  if (pd != nullptr && pd->num_groups > 0 && pd->max_shared > 0) {
    a.grp_off = pd->offsets;
    a.grp_mem = pd->members;
    a.grp_shared = pd->shared_blocks;
    a.num_groups = pd->num_groups;
    a.num_members = pd->num_members;
    a.max_shared = pd->max_shared;
    a.pchunk = lay.chunk;
    a.pmax_chunks = lay.max_chunks;
    a.skip = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + lay.skip_off);
    a.ppart = reinterpret_cast<float*>(static_cast<char*>(workspace) + lay.part_off);
    if (cudaMemsetAsync(a.skip, 0, static_cast<size_t>(batch) * sizeof(int32_t), s) !=
        cudaSuccess)
      return KVQ_ERR_CUDA;
    const int pper_sm = kvq::prefix_ctas_per_sm(pool->kv_dtype, q_dtype, pd->num_groups);
    if (pper_sm <= 0) return KVQ_ERR_CUDA;
    if (kvq::launch_prefix(a, pool->kv_dtype, q_dtype, plan.num_sms * pper_sm, s) != cudaSuccess)
      return KVQ_ERR_CUDA;
  }
  if (pre != nullptr) {
    // one cooperative launch: tables + store, barrier, decode, barrier, combine
    kvq::StepArgs sa;
    sa.t = pre->t;
    sa.st = pre->st;
    sa.d = a;
    sa.barrier = static_cast<unsigned int*>(workspace) + 1;  // zeroed above
    const int sper_sm = std::min(kvq::step_ctas_per_sm(pool->kv_dtype, q_dtype, batch, tail),
                                 kvq::kMaxCtasPerSm);
    if (sper_sm <= 0) return KVQ_ERR_CUDA;
    return kvq::launch_step(sa, pool->kv_dtype, q_dtype, plan.num_sms * sper_sm, s) ==
                   cudaSuccess
               ? KVQ_OK
               : KVQ_ERR_CUDA;
  }
  // persistent grid: as many CTAs as fit on the device at once (the
  // workspace has partial slots for kMaxCtasPerSm per SM)
  if (gqa) {
    if (kvq::launch_decode_gqa(a, pool->kv_dtype, gqa_grid, s) != cudaSuccess)
      return KVQ_ERR_CUDA;
  } else {
    const int per_sm = std::min(kvq::decode_ctas_per_sm(pool->kv_dtype, q_dtype, batch, tail),
                                kvq::kMaxCtasPerSm);
    if (per_sm <= 0) return KVQ_ERR_CUDA;
    if (kvq::launch_decode(a, pool->kv_dtype, q_dtype, plan.num_sms * per_sm, s) !=
        cudaSuccess)
      return KVQ_ERR_CUDA;
  }
  if (kvq::launch_combine(a, q_dtype, s) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

// Launch plan of an extend call: the context is cut into parts of pchunk
// blocks only when the batch has too few 16-row tiles to keep every warp
// busy (a short chunk over a long prefix); the workspace holds the work
// counter and, then, the parts' records.
struct ExtendPlan {
  int pchunk, max_splits;
  size_t part_off, total;
};

ExtendPlan extend_plan(int batch, int total_q, int q_heads, int kv_heads, int max_kv_len,
                       int num_sms) {
  ExtendPlan p;
  const int group = q_heads / kv_heads;
  const int64_t units = static_cast<int64_t>(kv_heads) *
                        ((static_cast<int64_t>(total_q) * group + 15) / 16 + batch);
  const int64_t warps = static_cast<int64_t>(num_sms) * 3 * (kvq::kDecodeThreads / 32);
  const int nblk = std::max(1, (max_kv_len + kBlock - 1) / kBlock);
  p.pchunk = 0;
  p.max_splits = 1;
  if (units < 2 * warps) {
    const int want = static_cast<int>(std::min<int64_t>(32, (2 * warps + units - 1) / units));
    const int chunk = std::max(8, (nblk + want - 1) / want);
    const int splits = (nblk + chunk - 1) / chunk;
    if (splits > 1) {
      p.pchunk = chunk;
      p.max_splits = splits;
    }
  }
  p.part_off = 256;  // the work counter
  p.total = p.part_off + (p.pchunk > 0 ? static_cast<size_t>(total_q) * q_heads * p.max_splits *
                                             kvq::kPartStride * sizeof(float)
                                       : 0);
  return p;
}

}  // namespace

extern "C" {

int32_t kvq_version(void) { return 101; }

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_OUT_OF_RANGE: return "device reported an out-of-range index or length";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

kvq_status kv_store_quant(const kvq_pool* pool, const void* k_new, const void* v_new,
                          int32_t in_dtype, const int64_t* slot_mapping, int64_t num_tokens,
                          int32_t* dev_err, void* stream) {
  const kvq_status ps = check_pool(pool);
  if (ps != KVQ_OK) return ps;
  if (num_tokens < 0) return KVQ_ERR_INVALID_ARG;
  if (!is_float16(in_dtype)) return KVQ_ERR_UNSUPPORTED;
  if (is_float16(pool->kv_dtype) && in_dtype != pool->kv_dtype) return KVQ_ERR_UNSUPPORTED;
  if (num_tokens == 0) return KVQ_OK;
  // the store numbers its (token, K or V, kv head) rows in 32 bits
  if (num_tokens > static_cast<int64_t>(kvq::kMaxStoreRows / (2 * pool->kv_heads)))
    return KVQ_ERR_UNSUPPORTED;
  if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_INVALID_ARG;
  kvq::StoreArgs a;
  a.k_pool = pool->k;
  a.v_pool = pool->v;
  a.k_sz = pool->k_sz;
  a.v_sz = pool->v_sz;
  a.num_blocks = pool->num_blocks;
  a.kv_heads = pool->kv_heads;
  a.kv_dtype = pool->kv_dtype;
  a.in_dtype = in_dtype;
  a.k_new = k_new;
  a.v_new = v_new;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.dev_err = dev_err;
  return kvq::launch_store(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK
                                                                                  : KVQ_ERR_CUDA;
}

kvq_status kvq_block_tables_from_req_to_token(const int32_t* req_to_token,
                                              int32_t num_req_slots, int32_t max_context_len,
                                              const int32_t* req_pool_indices,
                                              const int32_t* seq_lens, int32_t batch,
                                              int32_t max_blocks_per_seq, int32_t* block_tables,
                                              int32_t* dev_err, void* stream) {
  if (batch < 0 || num_req_slots < 0 || max_context_len < 0 || max_blocks_per_seq <= 0)
    return KVQ_ERR_INVALID_ARG;
  if (batch == 0) return KVQ_OK;
  if (req_to_token == nullptr || req_pool_indices == nullptr || seq_lens == nullptr ||
      block_tables == nullptr)
    return KVQ_ERR_INVALID_ARG;
  kvq::TablesArgs a{req_to_token, num_req_slots, max_context_len, req_pool_indices, seq_lens,
                    batch, max_blocks_per_seq, block_tables, dev_err};
  return kvq::launch_tables(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK
                                                                                  : KVQ_ERR_CUDA;
}

kvq_status paged_decode_attn_plan(int32_t batch, int32_t q_heads, int32_t kv_heads,
                                  int32_t head_dim, int32_t max_seq_len, int32_t num_splits,
                                  int32_t num_sms, kvq_decode_plan* plan) {
  if (plan == nullptr) return KVQ_ERR_INVALID_ARG;
  if (batch < 0 || q_heads <= 0 || kv_heads <= 0 || max_seq_len < 0 || num_splits < 0)
    return KVQ_ERR_INVALID_ARG;
  if (q_heads % kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return KVQ_ERR_UNSUPPORTED;
  if (batch > kvq::kMaxBatch) return KVQ_ERR_UNSUPPORTED;
  if (num_sms <= 0) num_sms = current_sm_count();
  if (num_sms <= 0) return KVQ_ERR_CUDA;
  const int group = q_heads / kv_heads;
  const int nblk = std::max(1, (max_seq_len + kBlock - 1) / kBlock);
  plan->min_blocks_per_warp =
      num_splits > 0 ? (nblk + num_splits - 1) / num_splits : kAutoMinBlocksPerWarp;
  plan->warps = num_sms * kvq::kMaxCtasPerSm * (kvq::kDecodeThreads / 32);
  plan->head_groups = (group + 7) / 8;
  plan->heads_per_group = std::min(group, 8);
  plan->num_sms = num_sms;
  plan->max_ctas_per_sm = kvq::kMaxCtasPerSm;
  plan->workspace_bytes =
      decode_records_offset(batch) +
      static_cast<size_t>(kvq::kRangesPerWarp) * plan->warps * range_record_bytes(*plan);
  return KVQ_OK;
}

size_t paged_decode_attn_workspace_size(int32_t batch, int32_t q_heads, int32_t kv_heads,
                                        int32_t head_dim, int32_t max_seq_len,
                                        int32_t num_splits) {
  kvq_decode_plan p;
  if (paged_decode_attn_plan(batch, q_heads, kv_heads, head_dim, max_seq_len, num_splits, 0,
                             &p) != KVQ_OK)
    return 0;
  return p.workspace_bytes;
}

kvq_status paged_decode_attn(const kvq_pool* pool, const void* q, int32_t q_dtype, void* out,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, int32_t batch, int32_t q_heads,
                             int32_t max_seq_len, float sm_scale, int32_t num_splits,
                             void* workspace, size_t workspace_bytes, int32_t* dev_err,
                             void* stream) {
  return decode_impl(pool, q, q_dtype, out, block_tables, max_blocks_per_seq, seq_lens, batch,
                     q_heads, max_seq_len, sm_scale, num_splits, nullptr, workspace,
                     workspace_bytes, dev_err, stream);
}

kvq_status paged_decode_attn_shared_prefix_workspace_size(
    int32_t batch, int32_t q_heads, int32_t kv_heads, int32_t head_dim, int32_t max_seq_len,
    int32_t num_splits, int32_t max_shared_blocks, size_t* bytes) {
  if (bytes == nullptr) return KVQ_ERR_INVALID_ARG;
  *bytes = 0;
  if (max_shared_blocks < 0) return KVQ_ERR_INVALID_ARG;
  kvq_decode_plan plan;
  const kvq_status st = paged_decode_attn_plan(batch, q_heads, kv_heads, head_dim, max_seq_len,
                                               num_splits, 0, &plan);
  if (st != KVQ_OK) return st;
  *bytes = shared_prefix_layout(plan, batch, q_heads, max_shared_blocks).total;
  return KVQ_OK;
}

kvq_status paged_decode_attn_shared_prefix(
    const kvq_pool* pool, const void* q, int32_t q_dtype, void* out, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch, int32_t q_heads,
    int32_t max_seq_len, float sm_scale, const int32_t* group_offsets,
    const int32_t* group_members, const int32_t* group_shared_blocks, int32_t num_groups,
    int32_t num_members, int32_t max_shared_blocks, int32_t num_splits, void* workspace,
    size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (num_groups < 0 || num_members < 0 || max_shared_blocks < 0) return KVQ_ERR_INVALID_ARG;
  if (max_shared_blocks > max_blocks_per_seq) return KVQ_ERR_INVALID_ARG;
  if (num_groups > kvq::kMaxBatch) return KVQ_ERR_UNSUPPORTED;
  if (num_groups > 0 &&
      (group_offsets == nullptr || group_shared_blocks == nullptr ||
       (num_members > 0 && group_members == nullptr)))
    return KVQ_ERR_INVALID_ARG;
  PrefixDesc pd{group_offsets, group_members, group_shared_blocks, num_groups, num_members,
                max_shared_blocks};
  return decode_impl(pool, q, q_dtype, out, block_tables, max_blocks_per_seq, seq_lens, batch,
                     q_heads, max_seq_len, sm_scale, num_splits, &pd, workspace,
                     workspace_bytes, dev_err, stream);
}

kvq_status paged_extend_attn_workspace_size(int32_t batch, int32_t total_q, int32_t q_heads,
                                            int32_t kv_heads, int32_t head_dim,
                                            int32_t max_kv_len, size_t* bytes) {
  if (bytes == nullptr) return KVQ_ERR_INVALID_ARG;
  *bytes = 0;
  if (batch < 0 || total_q < 0 || q_heads <= 0 || kv_heads <= 0 || max_kv_len < 0)
    return KVQ_ERR_INVALID_ARG;
  if (q_heads % kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return KVQ_ERR_UNSUPPORTED;
  const int sms = current_sm_count();
  if (sms <= 0) return KVQ_ERR_CUDA;
  *bytes = extend_plan(batch, total_q, q_heads, kv_heads, max_kv_len, sms).total;
  return KVQ_OK;
}

kvq_status paged_extend_attn(const kvq_pool* pool, const void* q, int32_t q_dtype, void* out,
                             const int32_t* qo_indptr, const int32_t* kv_lens,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             int32_t batch, int32_t total_q, int32_t q_heads, int32_t max_kv_len,
                             float sm_scale, int32_t variant, void* workspace,
                             size_t workspace_bytes, int32_t* dev_err, void* stream) {
  const kvq_status ps = check_pool(pool);
  if (ps != KVQ_OK) return ps;
  if (!is_float16(q_dtype)) return KVQ_ERR_UNSUPPORTED;
  if (is_float16(pool->kv_dtype) && q_dtype != pool->kv_dtype) return KVQ_ERR_UNSUPPORTED;
  if (batch < 0 || total_q < 0 || q_heads <= 0 || max_blocks_per_seq <= 0 || max_kv_len < 0)
    return KVQ_ERR_INVALID_ARG;
  if (q_heads % pool->kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return KVQ_ERR_INVALID_ARG;
  if (variant < KVQ_EXTEND_AUTO || variant > KVQ_EXTEND_TCGEN05) return KVQ_ERR_INVALID_ARG;
  // the tcgen05 kernel reads a missing block's rows from block 0 (and masks
  // them), so it needs a pool with at least one block
  const bool tc_ok = kvq::extend_tc_supported(pool->kv_dtype, q_dtype) &&
                     batch <= kvq::extend_tc_max_batch() && pool->num_blocks > 0;
  if (variant == KVQ_EXTEND_TCGEN05 && !tc_ok) return KVQ_ERR_UNSUPPORTED;
  if (batch > kvq::kMaxBatch) return KVQ_ERR_UNSUPPORTED;
  if (batch == 0 || total_q == 0) return KVQ_OK;
  if (q == nullptr || out == nullptr || qo_indptr == nullptr || kv_lens == nullptr ||
      block_tables == nullptr)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace)) return KVQ_ERR_INVALID_ARG;
  const int sms = current_sm_count();
  if (sms <= 0) return KVQ_ERR_CUDA;
  const ExtendPlan plan =
      extend_plan(batch, total_q, q_heads, pool->kv_heads, max_kv_len, sms);
  if (workspace == nullptr || workspace_bytes < plan.total) return KVQ_ERR_WORKSPACE;
  kvq::ExtendArgs a;
  std::memset(&a, 0, sizeof(a));
  if (pool->kv_dtype == KVQ_INT8) {
    if (!encode_pool_map(&a.k_map, pool->k, pool->num_blocks, pool->kv_heads, kHeadDim) ||
        !encode_pool_map(&a.v_map, pool->v, pool->num_blocks, pool->kv_heads, kHeadDim))
      return KVQ_ERR_CUDA;
  }
  a.k = static_cast<const uint8_t*>(pool->k);
  a.v = static_cast<const uint8_t*>(pool->v);
  a.k_sz = static_cast<const uint32_t*>(pool->k_sz);
  a.v_sz = static_cast<const uint32_t*>(pool->v_sz);
  a.num_blocks = pool->num_blocks;
  a.kv_heads = pool->kv_heads;
  a.q = q;
  a.out = out;
  a.qo_indptr = qo_indptr;
  a.kv_lens = kv_lens;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks_per_seq;
  a.batch = batch;
  a.q_heads = q_heads;
  a.group = q_heads / pool->kv_heads;
  a.total_q = total_q;
  a.pchunk = plan.pchunk;
  a.max_splits = plan.max_splits;
  a.len_cap = std::min(max_blocks_per_seq, std::max(1, (max_kv_len + kBlock - 1) / kBlock)) *
              kBlock;
  a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  a.counter = static_cast<int32_t*>(workspace);
  a.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.part_off);
  a.dev_err = dev_err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(a.counter, 0, sizeof(int32_t), s) != cudaSuccess) return KVQ_ERR_CUDA;
  // tcgen05 (256-row units) when the pool kind allows it and the batch has at
  // least one unit per SM; else 16-row tiles on mma.sync (which can also cut
  // the context of a short chunk into parts)
  const int64_t tc_units = static_cast<int64_t>(pool->kv_heads) *
                           ((static_cast<int64_t>(total_q) * a.group + 255) / 256);
  const bool use_tc = variant == KVQ_EXTEND_TCGEN05 ||
                      (variant == KVQ_EXTEND_AUTO && tc_ok && tc_units >= sms);
  if (use_tc) {
    // persistent CTAs, one per SM (each holds all 512 TMEM columns)
    if (kvq::extend_tc_ctas_per_sm(pool->kv_dtype, q_dtype, batch) <= 0) return KVQ_ERR_CUDA;
    return kvq::launch_extend_tc(a, pool->kv_dtype, q_dtype, sms, s) == cudaSuccess
               ? KVQ_OK
               : KVQ_ERR_CUDA;
  }
  const int per_sm = kvq::extend_ctas_per_sm(pool->kv_dtype, q_dtype, batch);
  if (per_sm <= 0) return KVQ_ERR_CUDA;
  return kvq::launch_extend(a, pool->kv_dtype, q_dtype, sms * per_sm, s) == cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

kvq_status kvq_decode_step_workspace_size(int32_t batch, int32_t q_heads, int32_t kv_heads,
                                          int32_t head_dim, int32_t max_seq_len,
                                          int32_t num_splits, size_t* bytes) {
  if (bytes == nullptr) return KVQ_ERR_INVALID_ARG;
  *bytes = 0;
  kvq_decode_plan plan;
  const kvq_status st = paged_decode_attn_plan(batch, q_heads, kv_heads, head_dim, max_seq_len,
                                               num_splits, 0, &plan);
  if (st != KVQ_OK) return st;
  *bytes = step_workspace(plan);
  return KVQ_OK;
}

kvq_status kvq_selftest_step_barrier(uint32_t* counter, int32_t grid_ctas, int32_t limit_us,
                                     int32_t* dev_err, void* stream) {
  if (counter == nullptr || dev_err == nullptr || grid_ctas < 0 || limit_us <= 0 ||
      limit_us > 1000000)
    return KVQ_ERR_INVALID_ARG;
  const int grid = grid_ctas > 0 ? grid_ctas : current_sm_count();
  if (grid <= 0) return KVQ_ERR_CUDA;
  return kvq::launch_barrier_selftest(counter, dev_err, grid,
                                      static_cast<uint64_t>(limit_us) * 1000ull,
                                      static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

int32_t kvq_decode_step_fused(int32_t batch, int64_t num_tokens) {
  return batch > 0 && num_tokens <= 2 * static_cast<int64_t>(batch) ? 1 : 0;
}

kvq_status kvq_decode_step(const kvq_pool* pool, const int32_t* req_to_token,
                           int32_t num_req_slots, int32_t max_context_len,
                           const int32_t* req_pool_indices, const int32_t* seq_lens,
                           int32_t batch, int32_t* block_tables, int32_t max_blocks_per_seq,
                           const void* k_new, const void* v_new, const int64_t* slot_mapping,
                           int64_t num_tokens, const void* q, int32_t q_dtype, void* out,
                           int32_t q_heads, int32_t max_seq_len, float sm_scale,
                           int32_t num_splits, void* workspace, size_t workspace_bytes,
                           int32_t* dev_err, void* stream) {
  const kvq_status ps = check_pool(pool);
  if (ps != KVQ_OK) return ps;
  if (num_req_slots < 0 || max_context_len < 0 || num_tokens < 0) return KVQ_ERR_INVALID_ARG;
  if (!is_float16(q_dtype)) return KVQ_ERR_UNSUPPORTED;
  if (batch > 0 && (req_to_token == nullptr || req_pool_indices == nullptr))
    return KVQ_ERR_INVALID_ARG;
  if (num_tokens > 0) {
    if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr)
      return KVQ_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_INVALID_ARG;
  }
  if (batch < 0) return KVQ_ERR_INVALID_ARG;
  if (batch == 0)  // nothing to attend: the step is the store alone
    return kv_store_quant(pool, k_new, v_new, q_dtype, slot_mapping, num_tokens, dev_err, stream);
  if (!kvq_decode_step_fused(batch, num_tokens)) {
    // a prefill chunk rides along: its store runs at full occupancy in a
    // kernel of its own, and so do the tables and the attention
    kvq_status st = kvq_block_tables_from_req_to_token(
        req_to_token, num_req_slots, max_context_len, req_pool_indices, seq_lens, batch,
        max_blocks_per_seq, block_tables, dev_err, stream);
    if (st != KVQ_OK) return st;
    st = kv_store_quant(pool, k_new, v_new, q_dtype, slot_mapping, num_tokens, dev_err, stream);
    if (st != KVQ_OK) return st;
    return decode_impl(pool, q, q_dtype, out, block_tables, max_blocks_per_seq, seq_lens, batch,
                       q_heads, max_seq_len, sm_scale, num_splits, nullptr, workspace,
                       workspace_bytes, dev_err, stream);
  }
  StepPre pre;
  pre.t = kvq::TablesArgs{req_to_token, num_req_slots, max_context_len, req_pool_indices,
                          seq_lens, batch, max_blocks_per_seq, block_tables, dev_err};
  pre.st.k_pool = pool->k;
  pre.st.v_pool = pool->v;
  pre.st.k_sz = pool->k_sz;
  pre.st.v_sz = pool->v_sz;
  pre.st.num_blocks = pool->num_blocks;
  pre.st.kv_heads = pool->kv_heads;
  pre.st.kv_dtype = pool->kv_dtype;
  pre.st.in_dtype = q_dtype;  // the new rows come in Q's dtype
  pre.st.k_new = k_new;
  pre.st.v_new = v_new;
  pre.st.slot_mapping = slot_mapping;
  pre.st.num_tokens = num_tokens;
  pre.st.dev_err = dev_err;
  return decode_impl(pool, q, q_dtype, out, block_tables, max_blocks_per_seq, seq_lens, batch,
                     q_heads, max_seq_len, sm_scale, num_splits, nullptr, workspace,
                     workspace_bytes, dev_err, stream, &pre);
}

kvq_status kvq_copy_blocks(const kvq_pool* src, const kvq_pool* dst, const int32_t* src_ids,
                           const int32_t* dst_ids, int64_t n, int32_t* dev_err, void* stream) {
  kvq_status st = check_pool(src);
  if (st != KVQ_OK) return st;
  st = check_pool(dst);
  if (st != KVQ_OK) return st;
  if (src->kv_dtype != dst->kv_dtype || src->kv_heads != dst->kv_heads) return KVQ_ERR_INVALID_ARG;
  if (n < 0) return KVQ_ERR_INVALID_ARG;
  if (n == 0) return KVQ_OK;
  if (src_ids == nullptr || dst_ids == nullptr) return KVQ_ERR_INVALID_ARG;
  const int row = is_quant(src->kv_dtype) ? (src->kv_dtype == KVQ_INT8 ? kHeadDim : kHeadDim / 2)
                                          : 2 * kHeadDim;
  kvq::CopyArgs a;
  a.src_k = static_cast<const uint4*>(src->k);
  a.src_v = static_cast<const uint4*>(src->v);
  a.src_k_sz = static_cast<const uint4*>(src->k_sz);
  a.src_v_sz = static_cast<const uint4*>(src->v_sz);
  a.dst_k = static_cast<uint4*>(dst->k);
  a.dst_v = static_cast<uint4*>(dst->v);
  a.dst_k_sz = static_cast<uint4*>(dst->k_sz);
  a.dst_v_sz = static_cast<uint4*>(dst->v_sz);
  a.src_blocks = src->num_blocks;
  a.dst_blocks = dst->num_blocks;
  a.tile_chunks = static_cast<int64_t>(kBlock) * src->kv_heads * row / 16;
  a.sz_chunks = is_quant(src->kv_dtype) ? static_cast<int64_t>(src->kv_heads) * kBlock * 4 / 16 : 0;
  a.src_ids = src_ids;
  a.dst_ids = dst_ids;
  a.dev_err = dev_err;
  return kvq::launch_copy(a, n, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK
                                                                                  : KVQ_ERR_CUDA;
}

kvq_status kvq_check_error(int32_t* dev_err, uint32_t* bits_out, void* stream) {
  if (dev_err == nullptr) return KVQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, dev_err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KVQ_ERR_CUDA;
  if (v != 0 && cudaMemset(dev_err, 0, sizeof(v)) != cudaSuccess) return KVQ_ERR_CUDA;
  if (bits_out != nullptr) *bits_out = static_cast<uint32_t>(v);
  return v == 0 ? KVQ_OK : KVQ_ERR_OUT_OF_RANGE;
}

}  // extern "C"

// Internal interface between the C-ABI layer (kvq_api.cu) and the kernels.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the encoder is fetched at run time)
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvq.h"
#include "kvq_ranges.h"

namespace kvq {

constexpr int kBlock = 16;     // tokens per block (LMDeploy article §2.2)
constexpr int kHeadDim = 128;  // head_dim supported by the kernels

struct StoreArgs {
  void* k_pool;
  void* v_pool;
  void* k_sz;
  void* v_sz;
  int64_t num_blocks;
  int kv_heads;
  int kv_dtype;
  int in_dtype;
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  int32_t* dev_err;
};

struct TablesArgs {
  const int32_t* req_to_token;
  int32_t num_req_slots;
  int32_t max_context_len;
  const int32_t* req_pool_indices;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t max_blocks_per_seq;
  int32_t* block_tables;
  int32_t* dev_err;
};

struct DecodeArgs {
  // TMA descriptors of the K and V pools (quantized pools only): 4-D views
  // [num_blocks][16][kv_heads][row bytes], one box = one (block, head) tile
  CUtensorMap k_map;
  CUtensorMap v_map;
  const uint8_t* k;
  const uint8_t* v;
  const uint32_t* k_sz;  // (scale, zero) fp16 pairs
  const uint32_t* v_sz;
  int64_t num_blocks;
  int kv_heads;
  const void* q;         // [B, Hq, D]
  void* out;             // [B, Hq, D]
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* seq_lens;
  int batch;
  int q_heads;
  int group;             // q_heads / kv_heads
  int head_groups;       // ceil(group / 8)
  int hpg;               // heads per group slot: min(group, 8)
  int min_blocks_per_warp;
  int len_cap;           // lengths are clamped to this (tokens)
  float sm_scale_log2;   // sm_scale * log2(e): scores live in the exp2 domain
  float* part;           // [ranges][2][hpg][kPartStride]: o[128], max, sum
  int64_t max_ranges;    // ranges the workspace holds records for
  unsigned int* tail_ctr;  // tail chunks handed out (zero at launch); null: no tail
  int32_t* hdr;          // [0] blocks per head group, [1] blocks per static range,
                         // [2] blocks per tail chunk (0: none), [3] warps,
                         // [4] ranges per q-head group (0: one cut of the whole stream),
                         // [kHdrCum .. kHdrCum + batch] prefix sums of the blocks per request
  int32_t* dev_err;
  // shared-prefix decode only (null / 0 otherwise): group G's members are
  // grp_mem[grp_off[G] .. grp_off[G + 1]) and share their first grp_shared[G]
  // blocks; the prefix kernel fills skip and ppart, the decode kernel reads
  // each request's blocks from skip[b] on and, with the combine kernel,
  // merges ppart
  const int32_t* grp_off;     // [num_groups + 1]
  const int32_t* grp_mem;     // [num_members]
  const int32_t* grp_shared;  // [num_groups]
  int num_groups;
  int num_members;
  int max_shared;             // bound on grp_shared (blocks)
  int pchunk;                 // shared blocks per prefix work unit (<= 32)
  int pmax_chunks;            // ceil(max_shared / pchunk): records per (request, q head)
  int32_t* skip;              // [batch] shared blocks of request b (0: none)
  float* ppart;               // [batch][q_heads][pmax_chunks][kPartStride]
  // grouped-query kernel: kv heads per CTA (one warp each; 0 for the other
  // kernels); its stream runs over (group of cta_heads kv heads, request,
  // block) and its records hold the group's cta_heads * group q heads
  int cta_heads;
  // ... and its TMA views of the K and V pools, ordered [block][kv head][token]
  // [row], one box = the 16 rows of cta_heads kv heads (k_map / v_map keep the
  // one-tile view the other INT8 kernels use)
  CUtensorMap kh_map;
  CUtensorMap vh_map;
};

struct CopyArgs {
  const uint4* src_k;
  const uint4* src_v;
  const uint4* src_k_sz;  // null for 16-bit pools (sz_chunks = 0)
  const uint4* src_v_sz;
  uint4* dst_k;
  uint4* dst_v;
  uint4* dst_k_sz;
  uint4* dst_v_sz;
  int64_t src_blocks;
  int64_t dst_blocks;
  int64_t tile_chunks;  // 16-byte chunks of one block's K (or V) tile
  int64_t sz_chunks;    // 16-byte chunks of one block's K (or V) scale/zero run
  const int32_t* src_ids;
  const int32_t* dst_ids;
  int32_t* dev_err;
};

struct ExtendArgs {
  CUtensorMap k_map;  // as in DecodeArgs (INT8 pools)
  CUtensorMap v_map;
  const uint8_t* k;
  const uint8_t* v;
  const uint32_t* k_sz;
  const uint32_t* v_sz;
  int64_t num_blocks;
  int kv_heads;
  const void* q;               // [total_q, Hq, D]
  void* out;                   // [total_q, Hq, D]
  const int32_t* qo_indptr;    // [batch + 1]
  const int32_t* kv_lens;      // [batch]
  const int32_t* block_tables;
  int max_blocks;
  int batch;
  int q_heads;
  int group;                   // q_heads / kv_heads
  int total_q;
  int pchunk;                  // blocks per work unit along the context (split), or 0: none
  int max_splits;              // records per (query row, q head) when split
  int len_cap;                 // longest context accepted (tokens)
  float sm_scale_log2;
  int32_t* counter;            // work counter (zero at launch)
  float* part;                 // [total_q][Hq][max_splits][kPartStride] when split
  int32_t* dev_err;
};

// One decode step in a single cooperative launch: block tables, the store of
// the step's new tokens, decode and combine, separated by grid barriers.
struct StepArgs {
  TablesArgs t;
  StoreArgs st;
  DecodeArgs d;
  unsigned int* barrier;  // zero at launch
};

cudaError_t launch_store(const StoreArgs& a, cudaStream_t s);
// kv_dtype / q_dtype as for launch_decode (the new rows have Q's dtype)
cudaError_t launch_step(const StepArgs& a, int kv_dtype, int q_dtype, int grid_ctas,
                        cudaStream_t s);
int step_ctas_per_sm(int kv_dtype, int q_dtype, int batch, bool tail);
// the step's grid barrier made to wait for one CTA more than the grid has
cudaError_t launch_barrier_selftest(unsigned int* ctr, int32_t* dev_err, int grid,
                                    uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_extend(const ExtendArgs& a, int kv_dtype, int q_dtype, int grid_ctas,
                          cudaStream_t s);
int extend_ctas_per_sm(int kv_dtype, int q_dtype, int batch);
// the tcgen05 version (256-row units; INT8, INT4 and fp16 pools)
bool extend_tc_supported(int kv_dtype, int q_dtype);
cudaError_t launch_extend_tc(const ExtendArgs& a, int kv_dtype, int q_dtype, int grid_ctas,
                             cudaStream_t s);
int extend_tc_ctas_per_sm(int kv_dtype, int q_dtype, int batch);
int extend_tc_max_batch();                // most requests the tcgen05 kernel takes
cudaError_t launch_copy(const CopyArgs& a, int64_t n, cudaStream_t s);
cudaError_t launch_tables(const TablesArgs& a, cudaStream_t s);
// kv_dtype / q_dtype select the template instance
cudaError_t launch_decode(const DecodeArgs& a, int kv_dtype, int q_dtype, int grid_ctas,
                          cudaStream_t s);
cudaError_t launch_combine(const DecodeArgs& a, int q_dtype, cudaStream_t s);
cudaError_t launch_prefix(const DecodeArgs& a, int kv_dtype, int q_dtype, int grid_ctas,
                          cudaStream_t s);

// CTAs of the decode kernel resident per SM (occupancy) for a dtype pair and batch
int decode_ctas_per_sm(int kv_dtype, int q_dtype, int batch, bool tail);
// The grouped-query decode kernel (kvq_decode_gqa.cu): INT8 / INT4 pools, fp16
// queries, 4 q heads per kv head, a CTA per group of cta_heads kv heads (one
// warp each); same workspace and combine, records of cta_heads * 4 q heads.
// Its kh_map / vh_map are the [block][kv head][token][row] views
// (encode_pool_map_heads).
bool decode_gqa_supported(int kv_dtype, int q_dtype, int group, int kv_heads);
int decode_gqa_cta_heads(int kv_heads);  // kv heads per CTA (0: unsupported)
cudaError_t launch_decode_gqa(const DecodeArgs& a, int kv_dtype, int grid, cudaStream_t s);
int decode_gqa_ctas_per_sm(int kv_dtype, int batch, int cta_heads, bool tail);
// the same for the shared-prefix kernel and a number of groups
int prefix_ctas_per_sm(int kv_dtype, int q_dtype, int num_groups);

constexpr int kMaxBatch = 8192;        // request lengths are scanned in shared memory
constexpr uint32_t kMaxStoreRows = 0xFFFFFFFFu;  // store rows (tokens x 2 x kv heads) per call
constexpr int kDecodeThreads = 128;
constexpr int kMaxCtasPerSm = 4;       // the workspace has slots for this many CTAs per SM
constexpr int kPartStride = kHeadDim + 4;  // floats per partial record (16-byte multiple)
constexpr int kHdrCum = 5;                 // first prefix sum in the decode's header
constexpr int kRangesPerWarp = 5;          // records the workspace holds: static + tail
constexpr int kMaxPrefixChunk = 32;    // shared blocks per prefix unit: one table window

}  // namespace kvq

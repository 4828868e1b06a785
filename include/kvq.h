/*
 * kvq.h -- C ABI of libkvq: a paged, quantized KV store and paged decode
 * attention for one GPU (NVIDIA GB300, sm_103a).
 *
 * Problem model (as the source pages describe it):
 *  - "pymllm Runtime Design", section "KV cache 与 prefix cache": a
 *    ReqToTokenPool maps (request slot, position) to an integer kv index, a
 *    free list hands those indices out, and a KVPool keeps each layer's K and
 *    V tensors on the GPU, written by a store kernel (store_cache).
 *  - LMDeploy article (devpress.csdn.net), §2.2 "分块 KV 缓存": the cache is
 *    split into blocks of 16 tokens; each sequence keeps a table of physical
 *    block ids; the per-layer shape is [num_blocks, block_size, kv_heads,
 *    head_dim].
 *  - same article, §2.4 "KV Cache 在线量化": K/V may be stored as INT8 or INT4
 *    with per-head, per-token asymmetric min/max quantization computed online
 *    (quant_policy 8 or 4).
 *  - same article, §3.2 item 3 and §4.2: decode ("generation") attention reads
 *    the non-contiguous cache through indirect block pointers in a kernel of
 *    its own.
 *
 * Conventions for every entry point:
 *  - Every pointer argument except the ones documented as host pointers is a
 *    DEVICE pointer on the current CUDA device. The caller owns all memory;
 *    the library never allocates, frees or synchronizes (except
 *    kvq_check_error, which synchronizes its stream).
 *  - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *    default stream. Work is enqueued asynchronously on it.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns a KVQ_ERR_* status and launches nothing.
 *  - Data-dependent faults (a slot past the pool, a block id outside the
 *    pool, a length past the table) are never trapped on the device: the
 *    offending access is skipped and a bit is OR-ed into the caller's device
 *    error word `dev_err` (an int32 in device memory; NULL disables the
 *    report). Read it with kvq_check_error.
 *  - Block size is 16 tokens and head_dim is 128.
 *  - Pool and tensor base pointers must be 16-byte aligned.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
  KVQ_ERR_UNSUPPORTED = 2,   /* valid but unsupported combination (dtype, head_dim...) */
  KVQ_ERR_CUDA = 3,          /* a CUDA runtime call or a launch failed */
  KVQ_ERR_OUT_OF_RANGE = 4,  /* kvq_check_error: the device error word was non-zero */
  KVQ_ERR_WORKSPACE = 5      /* workspace missing or smaller than required */
} kvq_status;

/* Element kinds. INT8/INT4 use the pages' quant_policy numbers. */
typedef enum kvq_dtype {
  KVQ_F16 = 0,
  KVQ_BF16 = 1,
  KVQ_INT4 = 4,
  KVQ_INT8 = 8
} kvq_dtype;

/* Bits of the device error word. */
#define KVQ_DEV_ERR_REQ_SLOT 1u    /* block tables: request slot outside the ReqToTokenPool */
#define KVQ_DEV_ERR_LENGTH 2u      /* a length past the pool row, the table or max_seq_len */
#define KVQ_DEV_ERR_KV_INDEX 4u    /* block tables: negative kv index in a used position */
#define KVQ_DEV_ERR_NOT_BLOCKED 8u /* block tables: row not block-contiguous */
#define KVQ_DEV_ERR_SLOT 16u       /* store: slot >= num_blocks * 16 (token skipped) */
#define KVQ_DEV_ERR_BLOCK_ID 32u   /* decode: block id outside [0, num_blocks) (block skipped) */
#define KVQ_DEV_ERR_TIMEOUT 64u    /* decode: a tile copy did not complete within 2 s (warp stopped) */
#define KVQ_DEV_ERR_PREFIX 128u    /* shared-prefix decode: a group description that does not hold */

/*
 * One layer's KV pool (KVPool of "pymllm Runtime Design"; shape from LMDeploy
 * article §2.2). slot = block_id * 16 + offset is the pool's kv index.
 *  k, v   : [num_blocks, 16, kv_heads, row] where row is head_dim 16-bit
 *           elements (F16/BF16), head_dim bytes (INT8 codes) or head_dim / 2
 *           bytes (INT4, two codes per byte, even index in the low nibble).
 *  k_sz, v_sz : INT8/INT4 only, else NULL. Pairs of fp16 (scale, zero), scale
 *           first, laid out [num_blocks, kv_heads, 16]: the 16 pairs of one
 *           (block, head) are contiguous. A code c stands for c * scale + zero
 *           (LMDeploy article §2.4: per-head, per-token asymmetric).
 */
typedef struct kvq_pool {
  void* k;
  void* v;
  void* k_sz;
  void* v_sz;
  int64_t num_blocks;
  int32_t block_size; /* must be 16 */
  int32_t kv_heads;
  int32_t head_dim;   /* must be 128 */
  int32_t kv_dtype;   /* kvq_dtype */
} kvq_pool;

/*
 * kv_store_quant -- write the K/V rows of num_tokens new tokens into the pool
 * ("pymllm Runtime Design": KVPool.set_kv through the store_cache kernel;
 * LMDeploy article §2.4 for the quantization).
 *
 *  k_new, v_new : [num_tokens, kv_heads, head_dim] elements of in_dtype
 *                 (KVQ_F16 or KVQ_BF16), contiguous.
 *  slot_mapping : [num_tokens] int64 kv indices ("out_cache_loc"); a negative
 *                 slot skips the token; a slot >= num_blocks * 16 is skipped
 *                 and reported as KVQ_DEV_ERR_SLOT.
 *  For F16/BF16 pools in_dtype must equal the pool dtype and rows are copied.
 *  For INT8/INT4 pools each (token, head) row x of K and of V is quantized:
 *    mn = min x, mx = max x (a signed zero taken as +0), in fp32
 *    scale = fp16_rne((mx - mn) / (2^b - 1)),  zero = fp16_rne(mn)
 *    code_i = clamp(rne((x_i - zero) / scale), 0, 2^b - 1)   (IEEE fp32)
 *    and all codes are 0 when scale is 0 or not finite or zero not finite.
 *  Inputs must be finite; bf16 inputs beyond the fp16 range are outside the
 *  contract (their scale/zero saturate). Tokens that share a slot race.
 *  Returns KVQ_OK, KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED or KVQ_ERR_CUDA.
 */
kvq_status kv_store_quant(const kvq_pool* pool, const void* k_new, const void* v_new,
                          int32_t in_dtype, const int64_t* slot_mapping, int64_t num_tokens,
                          int32_t* dev_err, void* stream);

/*
 * kvq_block_tables_from_req_to_token -- derive each request's block table
 * from its ReqToTokenPool row ("pymllm Runtime Design": (request slot,
 * position) -> kv index; LMDeploy article §2.2: per-sequence block table,
 * block size 16).
 *
 *  req_to_token     : [num_req_slots, max_context_len] int32, row-major.
 *  req_pool_indices : [batch] int32 request slot of each request.
 *  seq_lens         : [batch] int32 tokens of each request (device).
 *  block_tables     : [batch, max_blocks_per_seq] int32 output:
 *                     entry j = req_to_token[r][16 j] / 16 for j < ceil(L/16),
 *                     -1 after that.
 *  The row must be block-contiguous (req_to_token[r][16 j + i] == 16 * entry j
 *  + i for every position below L); violations set KVQ_DEV_ERR_NOT_BLOCKED,
 *  negative indices KVQ_DEV_ERR_KV_INDEX, a request slot out of range
 *  KVQ_DEV_ERR_REQ_SLOT (its row is left all -1) and a length past the row or
 *  the table KVQ_DEV_ERR_LENGTH (the length is clamped).
 */
kvq_status kvq_block_tables_from_req_to_token(const int32_t* req_to_token,
                                              int32_t num_req_slots, int32_t max_context_len,
                                              const int32_t* req_pool_indices,
                                              const int32_t* seq_lens, int32_t batch,
                                              int32_t max_blocks_per_seq, int32_t* block_tables,
                                              int32_t* dev_err, void* stream);

/*
 * Launch plan of paged_decode_attn (host-only arithmetic; no device access
 * when num_sms > 0). The decode work is one stream of (kv head, q-head group,
 * request, block) items; a persistent grid of warps cuts it into equal
 * contiguous ranges, at least min_blocks_per_warp blocks each. With an
 * automatic split and at least 16 blocks per warp, the static ranges cover
 * about nine tenths of the stream and the rest is cut into tail chunks of 4
 * to 8 (or more) blocks that warps take from a counter as they finish, so
 * that warps running at different speeds end together. A warp writes the
 * output of every request a range covers completely and, for the first and
 * last request of the range, a partial result (running max, sum,
 * unnormalised output) that a combine kernel merges with a log-sum-exp.
 *  num_splits : 0 = automatic; else requests are cut into at most
 *               num_splits + 1 pieces (min_blocks_per_warp =
 *               ceil(max blocks / num_splits)).
 *  num_sms    : SMs to plan for; 0 = ask the current device.
 */
typedef struct kvq_decode_plan {
  int32_t min_blocks_per_warp; /* lower bound of each warp's share, in blocks */
  int32_t warps;               /* warps the workspace has partial slots for */
  int32_t head_groups;         /* ceil((q_heads / kv_heads) / 8) */
  int32_t heads_per_group;     /* min(q_heads / kv_heads, 8) */
  int32_t num_sms;
  int32_t max_ctas_per_sm;     /* persistent CTAs per SM the workspace allows */
  size_t workspace_bytes;      /* counters, header (lengths prefix), 2 partial slots per
                                  range for 5 ranges per warp (static + tail) */
} kvq_decode_plan;

kvq_status paged_decode_attn_plan(int32_t batch, int32_t q_heads, int32_t kv_heads,
                                  int32_t head_dim, int32_t max_seq_len, int32_t num_splits,
                                  int32_t num_sms, kvq_decode_plan* plan);

/* Workspace bytes paged_decode_attn needs for these sizes on the current
 * device (0 if none). Returns 0 as well for invalid sizes. */
size_t paged_decode_attn_workspace_size(int32_t batch, int32_t q_heads, int32_t kv_heads,
                                        int32_t head_dim, int32_t max_seq_len,
                                        int32_t num_splits);

/*
 * paged_decode_attn -- single-token decode attention for a continuous batch
 * over the paged pool (LMDeploy article §3.2 item 3 and §4.2; §2.2 for the
 * block tables).
 *
 *  q            : [batch, q_heads, head_dim] of q_dtype (KVQ_F16/KVQ_BF16).
 *                 For F16/BF16 pools q_dtype must equal the pool dtype.
 *  out          : [batch, q_heads, head_dim] of q_dtype.
 *  block_tables : [batch, max_blocks_per_seq] int32 physical block ids.
 *  seq_lens     : [batch] int32 context length of each request, counting the
 *                 token just stored; 0 gives an all-zero output row.
 *  max_seq_len  : host upper bound of seq_lens (sizes the plan); longer
 *                 requests are clamped and flagged KVQ_DEV_ERR_LENGTH.
 *  sm_scale     : softmax scale (e.g. 1/sqrt(head_dim)).
 *  num_splits   : as in paged_decode_attn_plan.
 *  workspace    : device scratch of paged_decode_attn_workspace_size(...)
 *                 bytes, 16-byte aligned. A smaller one is accepted down to
 *                 one range per warp (256 bytes + the header, (batch + 6)
 *                 int32 rounded up to 256 bytes, + warps * 2 *
 *                 heads_per_group * 132 floats) and then runs without the
 *                 tail; below that KVQ_ERR_WORKSPACE.
 * For request b and q head h (kv head h / (q_heads / kv_heads)):
 *   out[b][h] = sum_t softmax_t(sm_scale * q . k_t) v_t over t < seq_lens[b],
 * with k_t, v_t read from slot block_tables[b][t / 16] * 16 + t % 16 and
 * dequantized (c * scale + zero) for INT8/INT4 pools. Accumulation is fp32,
 * the result is rounded once to q_dtype. Block ids outside the pool are
 * skipped and flagged KVQ_DEV_ERR_BLOCK_ID.
 */
kvq_status paged_decode_attn(const kvq_pool* pool, const void* q, int32_t q_dtype, void* out,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, int32_t batch, int32_t q_heads,
                             int32_t max_seq_len, float sm_scale, int32_t num_splits,
                             void* workspace, size_t workspace_bytes, int32_t* dev_err,
                             void* stream);

/*
 * paged_decode_attn_shared_prefix -- the same attention as paged_decode_attn,
 * computed as a cascade for requests that share leading blocks
 * ("pymllm Runtime Design", section "KV cache 与 prefix cache": radix prefix
 * cache hits reuse the matched prefix's KV slots; LMDeploy article §2.2:
 * sequences share physical blocks under prefix caching). Each shared block is
 * read once per group and kv head and multiplied with the queries of all the
 * group's members together; each member's own blocks then go through the
 * decode kernel, and the two parts are merged with a log-sum-exp.
 *
 * Arguments not listed here mean what they mean for paged_decode_attn.
 *  group_offsets       : device int32 [num_groups + 1], non-decreasing;
 *                        group G's members are
 *                        group_members[group_offsets[G] .. group_offsets[G + 1]).
 *  group_members       : device int32 [num_members]: request indices in
 *                        [0, batch); a request belongs to at most one group.
 *                        Requests in no group are decoded as usual.
 *  group_shared_blocks : device int32 [num_groups]: the number of leading
 *                        blocks that every member's block table holds
 *                        identically, each full (16 * shared <= seq_lens[b]
 *                        for every member b); at most max_shared_blocks.
 *  max_shared_blocks   : host bound of group_shared_blocks, at most
 *                        max_blocks_per_seq (sizes the workspace).
 *  workspace           : at least *bytes of
 *                        paged_decode_attn_shared_prefix_workspace_size.
 * A group description that does not hold (a member out of range or listed
 * twice, tables that differ within the shared blocks, a member shorter than
 * the shared part, a shared count above max_shared_blocks) sets
 * KVQ_DEV_ERR_PREFIX; the output rows of that group are then unspecified,
 * and no memory outside the arguments is touched. The result equals
 * paged_decode_attn's up to rounding order.
 */
kvq_status paged_decode_attn_shared_prefix_workspace_size(
    int32_t batch, int32_t q_heads, int32_t kv_heads, int32_t head_dim, int32_t max_seq_len,
    int32_t num_splits, int32_t max_shared_blocks, size_t* bytes);

kvq_status paged_decode_attn_shared_prefix(
    const kvq_pool* pool, const void* q, int32_t q_dtype, void* out, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch, int32_t q_heads,
    int32_t max_seq_len, float sm_scale, const int32_t* group_offsets,
    const int32_t* group_members, const int32_t* group_shared_blocks, int32_t num_groups,
    int32_t num_members, int32_t max_shared_blocks, int32_t num_splits, void* workspace,
    size_t workspace_bytes, int32_t* dev_err, void* stream);

/*
 * paged_decode_attn_noalloc -- the same computation as paged_decode_attn,
 * for callers that cannot allocate device memory (an operator inside an
 * engine that only passes it its tensors, a program that must reserve all
 * device memory when it loads, a loop where an allocation's latency or
 * implied synchronization is not acceptable). The pages have no counterpart:
 * this is a deployment convenience of this library.
 *
 * The split-K scratch comes from one array of KVQ_NOALLOC_SCRATCH_BYTES that
 * the library keeps in device memory (every GPU that loads the library holds
 * it until the process exits); nothing is allocated by the call. The caller
 * still passes inputs and outputs, with the meaning and layout of
 * paged_decode_attn.
 *  - Every call looks up the array's device address (cudaGetSymbolAddress)
 *    in the current context, so a context made anew on the device (after
 *    cudaDeviceReset, or one the caller makes current) is served at the
 *    array's address there. The first call in a context may load the
 *    library's device code into it: make that first call before any stream
 *    capture; later calls only read a host-side table.
 *  - Sizes whose static ranges alone need more than KVQ_NOALLOC_SCRATCH_BYTES
 *    are rejected with KVQ_ERR_WORKSPACE before anything is launched; sizes
 *    whose full workspace does not fit run without the tail.
 *  - All calls share the one array and it keeps the last call's contents;
 *    nothing in it needs to start at zero (every entry read is first written
 *    by the same call). Calls whose work overlaps on the GPU (other streams,
 *    other host threads) race on the array: serialize them.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

kvq_status paged_decode_attn_noalloc(const kvq_pool* pool, const void* q, int32_t q_dtype,
                                     void* out, const int32_t* block_tables,
                                     int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                     int32_t batch, int32_t q_heads, int32_t max_seq_len,
                                     float sm_scale, int32_t num_splits, int32_t* dev_err,
                                     void* stream);

/*
 * paged_extend_attn -- extend (chunked prefill) attention over the paged pool
 * ("pymllm Runtime Design", forward stage: an extend / prefill batch writes
 * its prompt tokens to the KV cache and attends over them; LMDeploy article
 * §2.3: a prefill longer than the 4096-token threshold is split into chunks
 * prefilled in turn). The chunk's K/V rows are stored first (kv_store_quant);
 * every query then reads the request's K/V through its block table,
 * dequantized in registers.
 *  q, out      : [total_q, q_heads, head_dim] of q_dtype (KVQ_F16/KVQ_BF16;
 *                equal to the pool dtype for F16/BF16 pools), 16-byte aligned.
 *  qo_indptr   : device int32 [batch + 1], non-decreasing, qo_indptr[0] = 0,
 *                qo_indptr[batch] = total_q: request b's chunk queries are
 *                rows qo_indptr[b] .. qo_indptr[b + 1] - 1.
 *  kv_lens     : device int32 [batch]: tokens of request b in the pool, its
 *                chunk included (kv_lens[b] >= its chunk length).
 *  block_tables: [batch, max_blocks_per_seq] int32 physical block ids.
 *  max_kv_len  : host upper bound of kv_lens (sizes the plan); a longer
 *                request is skipped and flagged KVQ_DEV_ERR_LENGTH.
 *  variant     : KVQ_EXTEND_AUTO, or a kernel to use:
 *                KVQ_EXTEND_MMA_SYNC (tiles of 16 rows on mma.sync; every pool
 *                kind; cuts long contexts into parts when the batch has few
 *                query tiles) or KVQ_EXTEND_TCGEN05 (units of 256 rows on
 *                tcgen05 with tensor-memory accumulators; INT8, INT4 and
 *                fp16 pools of at least one block, at most 4096 requests;
 *                KVQ_ERR_UNSUPPORTED otherwise). AUTO takes the tcgen05 kernel when it accepts
 *                the call and the batch has at least as many 256-row units
 *                as the device has SMs.
 *  workspace   : at least *bytes of paged_extend_attn_workspace_size, 16-byte
 *                aligned; nothing in it needs to start at zero.
 * Chunk query i of request b (chunk length C) sits at position
 * kv_lens[b] - C + i and attends positions 0 .. that position:
 *   out[row][h] = sum_t softmax_t(sm_scale * q . k_t) v_t, t <= position,
 * fp32 accumulation, rounded once to q_dtype. A request whose rows fall
 * outside [0, total_q), whose chunk is longer than its context or whose
 * context exceeds the table is skipped and flagged KVQ_DEV_ERR_LENGTH (its
 * rows are not written); block ids outside the pool are skipped and flagged
 * KVQ_DEV_ERR_BLOCK_ID.
 */
#define KVQ_EXTEND_AUTO 0
#define KVQ_EXTEND_MMA_SYNC 1
#define KVQ_EXTEND_TCGEN05 2

kvq_status paged_extend_attn_workspace_size(int32_t batch, int32_t total_q, int32_t q_heads,
                                            int32_t kv_heads, int32_t head_dim,
                                            int32_t max_kv_len, size_t* bytes);

kvq_status paged_extend_attn(const kvq_pool* pool, const void* q, int32_t q_dtype, void* out,
                             const int32_t* qo_indptr, const int32_t* kv_lens,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             int32_t batch, int32_t total_q, int32_t q_heads, int32_t max_kv_len,
                             float sm_scale, int32_t variant, void* workspace,
                             size_t workspace_bytes, int32_t* dev_err, void* stream);

/*
 * kvq_decode_step -- one decode step of a layer in a single launch: the
 * block tables from the ReqToTokenPool rows (as
 * kvq_block_tables_from_req_to_token), the quantizing store of the step's new
 * K/V rows (as kv_store_quant, the rows in q_dtype), then the attention (as
 * paged_decode_attn, reading the tables just built). "pymllm Runtime Design",
 * forward stage: a decode step stores each request's new token and attends
 * over its cache; one kernel instead of four, its phases (tables + store,
 * attention, split-K combine) separated by grid barriers (a cooperative
 * launch: every CTA resident; each barrier wait gives up after 2 s with
 * KVQ_DEV_ERR_TIMEOUT). Arguments mean what they mean for the three calls it
 * replaces; block_tables is written. The workspace is at least *bytes of
 * kvq_decode_step_workspace_size (the decode's; its barrier counter sits in
 * the workspace's counters).
 * The single launch is used when the step stores at most two tokens per
 * request (kvq_decode_step_fused): its first phase runs at the attention's
 * occupancy, which suits a decode batch's new tokens but not a prefill chunk
 * stored in the same step (LMDeploy article §2.3, chunked prefill beside the
 * decodes); with more tokens the same work runs as four kernels.
 */
int32_t kvq_decode_step_fused(int32_t batch, int64_t num_tokens);

kvq_status kvq_decode_step_workspace_size(int32_t batch, int32_t q_heads, int32_t kv_heads,
                                          int32_t head_dim, int32_t max_seq_len,
                                          int32_t num_splits, size_t* bytes);

kvq_status kvq_decode_step(const kvq_pool* pool, const int32_t* req_to_token,
                           int32_t num_req_slots, int32_t max_context_len,
                           const int32_t* req_pool_indices, const int32_t* seq_lens,
                           int32_t batch, int32_t* block_tables, int32_t max_blocks_per_seq,
                           const void* k_new, const void* v_new, const int64_t* slot_mapping,
                           int64_t num_tokens, const void* q, int32_t q_dtype, void* out,
                           int32_t q_heads, int32_t max_seq_len, float sm_scale,
                           int32_t num_splits, void* workspace, size_t workspace_bytes,
                           int32_t* dev_err, void* stream);

/*
 * kvq_selftest_step_barrier -- a self-test of the bounded grid barrier that
 * kvq_decode_step's single launch waits at (the pages have no counterpart:
 * it checks this library's failure handling). One cooperative launch of
 * `grid_ctas` CTAs (0: one per SM) meets at that barrier, made to wait for
 * one CTA more than the grid has, with a limit of limit_us microseconds: the
 * wait runs out, sets KVQ_DEV_ERR_TIMEOUT in *dev_err and every CTA returns,
 * leaving the context usable. counter: a device word, zero at the call (it
 * counts the arrivals). Asynchronous on `stream`; allocates nothing.
 */
kvq_status kvq_selftest_step_barrier(uint32_t* counter, int32_t grid_ctas, int32_t limit_us,
                                     int32_t* dev_err, void* stream);

/*
 * kvq_copy_blocks -- copy whole blocks from one pool to another (LMDeploy
 * article §4.4: the cache engine swaps blocks between the GPU and the CPU
 * cache by a {dst: src} map, K and V alike; inside one pool the same copy
 * forks a shared block before a request writes into it).
 *  src, dst : pools of the same kv_dtype, kv_heads and head_dim. Either may
 *             be in pinned host memory the GPU can address (cudaHostAlloc,
 *             torch pin_memory; under unified addressing the host pointers
 *             are used as they are): a swap out or in is then this one call,
 *             reading or writing host memory over the CPU-GPU link.
 *  src_ids, dst_ids : int32 [n], device-addressable.
 * For every i, block src_ids[i] of src is copied to block dst_ids[i] of dst:
 * its K and V tiles (16 x kv_heads rows each) and, for INT8/INT4 pools, its
 * K and V (scale, zero) pairs. The dst ids must be distinct and, when src and
 * dst are the same pool, none of them may also be a src id (the pairs run in
 * parallel). A pair with an id outside its pool is skipped and flagged
 * KVQ_DEV_ERR_BLOCK_ID. Asynchronous on `stream`; allocates nothing.
 */
kvq_status kvq_copy_blocks(const kvq_pool* src, const kvq_pool* dst, const int32_t* src_ids,
                           const int32_t* dst_ids, int64_t n, int32_t* dev_err, void* stream);

/*
 * kvq_check_error -- synchronize `stream`, read the device error word and
 * clear it. Returns KVQ_OK if it was 0, KVQ_ERR_OUT_OF_RANGE otherwise (the
 * bits are stored to *bits_out when bits_out is not NULL), KVQ_ERR_CUDA if the
 * stream reported an error.
 */
kvq_status kvq_check_error(int32_t* dev_err, uint32_t* bits_out, void* stream);

/* Short text for a status code (static storage). */
const char* kvq_status_string(kvq_status status);

/* Library ABI version (major * 100 + minor). */
int32_t kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */

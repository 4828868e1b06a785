// kvq_extend_tc: extend (chunked prefill) attention on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory), warp-specialised.
//
// Same computation as kvq_extend.cu ("pymllm Runtime Design", forward stage:
// extend / prefill; LMDeploy article §2.3: prefills split into chunks; §2.4:
// per-token, per-head INT8/INT4 scale and zero). A work unit is 256 rows
// (query, q head) of one kv head; the request's context is walked in tiles
// of 64 tokens (4 blocks). One CTA per SM, fourteen working warps (fifteen
// for INT8 pools) in five roles:
//   * raw-ring producer (warp 14, INT8 pools): hands out the work units (an
//     atomic counter, longest tiles first) and copies each tile's raw codes
//     and scale/zero words by TMA into a two-stage raw ring, one box per
//     (block, K or V), two tiles ahead of the staging warpgroup;
//   * staging warpgroup (warps 8-11): takes each tile's codes from the raw
//     ring (INT8) or straight from the pool (other kinds: per-thread
//     addresses fixed for the unit, the tile's four block ids fetched a tile
//     ahead; these pools' units are handed out here) and writes K in a
//     K-major 128-byte-swizzled tile and V transposed (dims as rows) into a
//     three-stage ring;
//   * two MMA warps (warps 12 and 13, one per softmax warpgroup g, on
//     different sub-partitions; one elected lane issues): S_g = Q_g K^T
//     (M 128, N 64, K 128) into the warpgroup's own TMEM columns, the next
//     tile's S_g as soon as warpgroup g has read the current one out of TMEM
//     (so it runs during that warpgroup's exponentials), and O_g += P_g V
//     (M 128, K 64, A read from TMEM) as soon as warpgroup g's P is ready;
//   * two softmax warpgroups (warps 0-3, 4-7), one thread per row: read the
//     row of S (tcgen05.ld), mask (causal, missing blocks), apply the online
//     softmax with a lazily moved maximum (a stale maximum only scales every
//     term alike; O is rescaled in TMEM when it moves), and write P to their
//     own TMEM columns (tcgen05.st).
// Numerics by query type:
//   * fp16 queries: K and V are staged dequantized, (c - mid) S + (Z + mid S)
//     in fp16 with one rounding; P = 2^(s - m) is computed as fp16 pairs, and
//     V's tile carries a row of ones, so the P V product also gives the row
//     sum over the same fp16 P. Output: O / l.
//   * bf16 queries: the codes stay exact (K as c - mid in bf16, V as c - mid
//     in fp16); s = S_k (q.(c - mid)) + (Z_k + mid S_k) sum(q) from per-token
//     arrays, P' = p S_v in fp16, and sum p and sum p (Z_v + mid S_v) in fp32
//     registers. Output: (O + z) / l.
// Roles meet only at mbarriers (no CTA-wide barrier inside the work loop);
// every wait is bounded (2 s, then KVQ_DEV_ERR_TIMEOUT and every role leaves
// its loop), and the MMA warps wait for their products in flight before the
// CTA frees its TMEM.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tile.cuh"
#include "kvq_umma.cuh"

namespace kvq {
namespace {

constexpr int kWgRows = 128;              // rows per softmax warpgroup (M, TMEM lanes)
constexpr int kUnitRows = 2 * kWgRows;    // rows per work unit
constexpr int kTcTok = 64;                // tokens per context tile (N of S, K of P V)
constexpr int kStageThreads = 128;        // staging warpgroup
constexpr int kSoftWarps = 8;             // warps 0-7: softmax warpgroups 0 and 1
constexpr int kMmaWarp = 12;              // warps 8-11 stage, warps 12 and 13 issue the MMAs
constexpr int kTcThreads = 16 * 32;       // four warpgroups; warp 14 copies the raw codes of
                                          // INT8 pools, warp 15 only holds registers
// Registers per thread after the split (setmaxnreg): the launch gives every
// thread 65536 / 512 = 128; the staging and MMA warpgroups give theirs back
// down to kLowRegs, the softmax warpgroups take them up to kHighRegs.
constexpr uint32_t kLowRegs = 120, kHighRegs = 136;
static_assert(2 * kLowRegs + 2 * kHighRegs == 4 * (65536 / kTcThreads),
              "the split must add up to the launch's registers");
// TMEM columns: S_g at 64 g (64), O_g at 128 + o_cols g, P'_g at p_col + 32 g
// (32: two fp16 per column). With fp16 queries O_g has 144 columns: the 128
// output dims, then the row sum of P (V's tile carries a row of ones).
constexpr uint32_t kTmemCols = 512;
template <bool QBF>
constexpr uint32_t o_cols() { return QBF ? 128u : 144u; }
template <bool QBF>
constexpr uint32_t p_col() { return 128u + 2u * o_cols<QBF>(); }
static_assert(p_col<false>() + 64 <= kTmemCols && p_col<true>() + 64 <= kTmemCols, "TMEM map");

// shared memory, offsets from a 1024-byte aligned base
constexpr int kStages = 3;                          // K/V ring depth (tiles)
constexpr uint32_t kQBytes = kWgRows * 256;         // 2 column blocks of 128 rows x 128 B
constexpr uint32_t kKBytes = kTcTok * 256;          // 2 column blocks of 64 rows x 128 B
constexpr int kVRows = 144;                         // 128 dims, a row of ones, 15 of zeros
constexpr uint32_t kVBytes = kVRows * kTcTok * 2;   // V^T: kVRows x 64 tokens
constexpr uint32_t kSzBytes = 4 * kTcTok * 4;       // S_k'[64] Z_k'[64] S_v[64] Z_v'[64]
constexpr uint32_t kQOff = 0;                       // Q of warpgroup g at g * kQBytes
constexpr uint32_t kKOff = kQOff + 2 * kQBytes;     // K tile of stage s at s * kKBytes
constexpr uint32_t kVOff = kKOff + kStages * kKBytes;
constexpr uint32_t kSzOff = kVOff + kStages * kVBytes;
constexpr uint32_t kInfoOff = kSzOff + kStages * kSzBytes;  // per stage: max S_v (2 halves), missing masks
// Raw ring (INT8 pools): a tile's codes as the TMA copies land them. Stage:
// the K rows of its four blocks (one box per block: 16 rows of 128 bytes,
// 128-byte swizzle, so tile token t sits at row t), the V rows likewise,
// the 64 K and 64 V scale/zero words, and the four blocks' valid bits.
constexpr int kRawStages = 2;
constexpr uint32_t kRawBox = kBlock * 128;                 // one (block, kv head) box
constexpr uint32_t kRawVOff = 4 * kRawBox;
constexpr uint32_t kRawSzOff = 8 * kRawBox;                // K words [64], then V words [64]
constexpr uint32_t kRawValidOff = kRawSzOff + 2 * kTcTok * 4;
constexpr uint32_t kRawTx = 8 * kRawBox + 2 * kTcTok * 4;  // bytes the copies of a stage bring
constexpr uint32_t kRawBytes = (kRawValidOff + 16 + 1023) / 1024 * 1024;
constexpr uint32_t kRawOff = (kInfoOff + kStages * 16 + 1023) / 1024 * 1024;
template <int KV>
constexpr bool raw_ring() { return KV == kI8; }
constexpr uint32_t kBarOff = kRawOff + kRawStages * kRawBytes;
// mbarriers (index: runs by stage or warpgroup)
constexpr uint32_t kBarKvFull = 0;                  // staging -> MMA, softmax (128 arrivals), per stage
constexpr uint32_t kBarKvEmpty = kStages;           // MMA commit: the stage's products are done
constexpr uint32_t kBarSFull = 2 * kStages;         // MMA commit: S_g is in TMEM
constexpr uint32_t kBarPFull = kBarSFull + 2;       // softmax g -> MMA (128 arrivals)
constexpr uint32_t kBarODone = kBarPFull + 2;       // MMA commit: O_g += P'_g V done
constexpr uint32_t kBarQFull = kBarODone + 2;       // softmax g -> MMA: the unit's Q rows (128 arrivals)
constexpr uint32_t kBarUnitFull = kBarQFull + 2;    // unit slot written
constexpr uint32_t kBarUnitEmpty = kBarUnitFull + 2; // unit slot read by every working warp
constexpr uint32_t kBarSRead = kBarUnitEmpty + 2;   // softmax g -> MMA: S_g read out of TMEM (128 arrivals)
constexpr uint32_t kBarDrain = kBarSRead + 2;       // MMA commit before TMEM is freed
constexpr uint32_t kBarRawFull = kBarDrain + 1;     // raw stage landed (TMA bytes), per raw stage
constexpr uint32_t kBarRawEmpty = kBarRawFull + kRawStages;  // raw stage read (128 arrivals)
constexpr uint32_t kNumBars = kBarRawEmpty + kRawStages;
constexpr uint32_t kSlotOff = kBarOff + 8 * kNumBars;  // TMEM base address
constexpr uint32_t kUnitOff = kSlotOff + 4;            // 2 unit slots
constexpr uint32_t kAbortOff = kUnitOff + 8;
constexpr uint32_t kFixedBytes = kAbortOff + 4;
// requests per launch (their unit prefix sums live in shared memory)
constexpr int kTcMaxBatch = 4096;

__host__ __device__ constexpr size_t tc_smem_bytes(int batch) {
  return 1024 + kFixedBytes + align128((batch + 1) * sizeof(int32_t));
}
// the opt-in shared-memory limit of a CTA on sm_100-class GPUs (227 KB),
// with the kernel's static shared memory (1 KB as placed)
static_assert(tc_smem_bytes(kTcMaxBatch) + 1024 <= 232448, "shared memory over the CTA limit");

struct TcReq {
  int q0, C, L, tiles;
  bool ok;
};

__device__ __forceinline__ TcReq tc_req(const ExtendArgs& a, int b) {
  TcReq s;
  s.q0 = a.qo_indptr[b];
  const int q1 = a.qo_indptr[b + 1];
  s.C = q1 - s.q0;
  s.L = a.kv_lens[b];
  s.ok = s.q0 >= 0 && s.C >= 0 && q1 <= a.total_q && s.L >= s.C && s.L <= a.len_cap;
  if (!s.ok) s.C = s.L = 0;
  s.tiles = (s.C * a.group + kUnitRows - 1) / kUnitRows;
  return s;
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// Code value c - mid as a 16-bit float of the product's type (exact).
template <bool BF>
__device__ __forceinline__ uint32_t centred_pair(int c0, int c1, int mid) {
  return pack2<BF>(static_cast<float>(c0 - mid), static_cast<float>(c1 - mid));
}

// Raw bytes of one 64-token context tile that staging thread `tid` (0..127)
// holds: K chunks (16 bytes of one token row each), V pieces (8 dims of 8
// consecutive tokens), and, for threads < 64, the scale/zero words of token
// tid and whether its block is missing.
template <int KV>
struct RawTile {
  static constexpr int kRow = KvTraits<KV>::kRowBytes;
  static constexpr int kKChunks = kTcTok * (kRow / 16) / kStageThreads;  // 4 / 2 / 8
  static constexpr int kVWords = kRow / 64;  // 32-bit words per token of an 8-dim piece: 2 / 1 / 4
  uint4 k[kKChunks];
  uint32_t v[8][kVWords];
  uint32_t ksz, vsz;
  uint32_t ksz4[KvTraits<KV>::kQuant ? kKChunks : 1];  // K scale/zero of each K chunk's token
  uint32_t kmask;  // which K chunks belong to a token in the context (block in the pool)
  uint32_t vsz8[KvTraits<KV>::kQuant ? 8 : 1];  // V scale/zero of this thread's 8 V tokens
  uint32_t vmask;  // which of those 8 tokens are in the context (block in the pool)
  bool sz_ok;  // token `tid` is in the context and its block in the pool
  bool miss;   // token `tid` of the tile is in the context but its block id is outside the pool
};

// The K chunk (16 bytes of codes: token t of the tile, chunk ch of its row)
// that staging item e (= thread + 128 i) moves. Eight neighbouring lanes take
// 2 tokens x 4 chunks (INT8), 4 x 2 (INT4) or 1 x 8 (fp16): under the 128-byte
// swizzle their 16-byte stores then land in eight different bank groups, and
// a warp still reads whole token rows. For INT8 the second token of a lane
// group takes the other half of its row, so that the group's 16-byte reads
// from the swizzled raw stage also fall in eight different bank groups.
template <int KV>
__device__ __forceinline__ void k_item(int e, int& t, int& ch) {
  constexpr int kChunks = RawTile<KV>::kRow / 16;  // 8 / 4 / 16 per token row
  constexpr int kCpg = kChunks / 2;                // chunks per lane group of 8
  constexpr int kTpg = 8 / kCpg;                   // tokens per lane group
  const int lane8 = e & 7, grp = e >> 3;
  t = kTpg * (grp >> 1) + lane8 / kCpg;
  const int half = KV == kI8 ? (grp & 1) ^ (lane8 / kCpg) : (grp & 1);
  ch = kCpg * half + lane8 % kCpg;
}

// The V piece (8 consecutive tokens 8 tg .., 8 dims 8 dc ..) that staging
// thread tid (0..127) transposes. The eight lanes of a quarter warp always
// take eight different token groups, so their 16-byte stores of V^T rows hit
// eight bank groups; for INT8 the sixteen lanes of a half warp also take the
// sixteen dim groups, so that their 8-byte reads of one token row from the
// raw stage are conflict-free.
template <int KV>
__device__ __forceinline__ void v_item(int tid, int& tg, int& dc) {
  if constexpr (KV == kI8) {
    dc = tid & 15;
    tg = ((tid & 7) + (tid >> 4)) & 7;
  } else {
    tg = tid & 7;
    dc = tid >> 3;
  }
}

// Table entries of the tile's four blocks (tokens tok0 .. tok0 + 63). The
// index is clamped to the table row, so the loads are unconditional; an entry
// of a block past the context is ignored where it is used. Staging fetches
// them a tile ahead.
__device__ __forceinline__ int4 tile_blocks(const int32_t* bt, int tok0, int max_blocks) {
  const int b0 = tok0 / kBlock, last = max_blocks - 1;
  int4 r;
  r.x = __ldg(bt + min(b0, last));
  r.y = __ldg(bt + min(b0 + 1, last));
  r.z = __ldg(bt + min(b0 + 2, last));
  r.w = __ldg(bt + min(b0 + 3, last));
  return r;
}

__device__ __forceinline__ int pick4(const int4& v, int k) {
  return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

// Per-thread constants of a staging thread's loads, fixed for a unit (kv
// head h): which tile block and token each K item reads and its byte offset
// from the block's first row; the same for the thread's 8 V tokens.
template <int KV>
struct StageMap {
  using R = RawTile<KV>;
  int kb[R::kKChunks];         // tile block (0..3) of K item i
  int kt[R::kKChunks];         // tile token of K item i
  uint32_t koff[R::kKChunks];  // bytes from the block's first row (token row, head, chunk)
  uint32_t kszo[R::kKChunks];  // scale word index within the block's words (head, token)
  int vb;                      // tile block of the V tokens 8 tg .. 8 tg + 7
  uint32_t voff, vszo;
  __device__ __forceinline__ void init(const ExtendArgs& a, int h, int tid) {
    const uint32_t head_row = static_cast<uint32_t>(a.kv_heads) * R::kRow;  // one token
#pragma unroll
    for (int i = 0; i < R::kKChunks; ++i) {
      int t, ch;
      k_item<KV>(tid + kStageThreads * i, t, ch);
      kb[i] = t / kBlock;
      kt[i] = t;
      koff[i] = (t % kBlock) * head_row + h * R::kRow + 16 * ch;
      kszo[i] = h * kBlock + t % kBlock;
    }
    int tg, dc;
    v_item<KV>(tid, tg, dc);
    const int tv = 8 * tg;
    vb = tv / kBlock;
    voff = (tv % kBlock) * head_row + h * R::kRow + dc * 4 * R::kVWords;
    vszo = h * kBlock + tv % kBlock;
  }
};

// The tile's four blocks: each id when the block is inside the context and
// the pool (bit b of *valid), else 0 -- an address that is safe to read.
// Codes read from there, and from the context's last block past its length,
// are never used: those tokens are masked (p = 0), and their scale/zero words
// are zeroed.
__device__ __forceinline__ int4 safe_blocks(const ExtendArgs& a, const int4& blks, int tok0,
                                            int L, uint32_t* valid) {
  const int e[4] = {blks.x, blks.y, blks.z, blks.w};
  int o[4];
  uint32_t v = 0u;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const bool ok = tok0 + b * kBlock < L && e[b] >= 0 && e[b] < a.num_blocks;
    o[b] = ok ? e[b] : 0;
    v |= (ok ? 1u : 0u) << b;
  }
  *valid = v;
  return make_int4(o[0], o[1], o[2], o[3]);
}

// Issues the global loads of tile tok0 into r; no instruction here waits for
// their data.
template <int KV, bool QBF>
__device__ __forceinline__ void load_tile(const ExtendArgs& a, const StageMap<KV>& m,
                                          const int4& blks, int tok0, int L, int h, int tid,
                                          RawTile<KV>& r) {
  using R = RawTile<KV>;
  uint32_t valid;
  const int4 sb = safe_blocks(a, blks, tok0, L, &valid);
  const int64_t blk_bytes = static_cast<int64_t>(kBlock) * a.kv_heads * R::kRow;
  const int64_t blk_words = static_cast<int64_t>(kBlock) * a.kv_heads;
  r.kmask = 0u;
#pragma unroll
  for (int i = 0; i < R::kKChunks; ++i) {
    const int64_t blk = pick4(sb, m.kb[i]);
    r.k[i] = __ldg(reinterpret_cast<const uint4*>(a.k + blk * blk_bytes + m.koff[i]));
    r.kmask |= ((valid >> m.kb[i]) & 1u && tok0 + m.kt[i] < L ? 1u : 0u) << i;
    if constexpr (KvTraits<KV>::kQuant && !QBF)
      r.ksz4[i] = __ldg(a.k_sz + blk * blk_words + m.kszo[i]);
  }
  // V: tokens 8 tg .. 8 tg + 7 (one block: 8 divides 16), dims 8 dc .. 8 dc + 7
  int tg, dc;
  v_item<KV>(tid, tg, dc);
  (void)dc;  // the V address is the map's
  const int tv = 8 * tg;
  const int64_t vblk = pick4(sb, m.vb);
  const uint8_t* vrow = a.v + vblk * blk_bytes + m.voff;
  const int64_t head_row = static_cast<int64_t>(a.kv_heads) * R::kRow;
  const bool vok = (valid >> m.vb) & 1u;
  r.vmask = 0u;
#pragma unroll
  for (int t = 0; t < 8; ++t) r.vmask |= (vok && tok0 + tv + t < L ? 1u : 0u) << t;
  if constexpr (KvTraits<KV>::kQuant && !QBF) {  // 8 consecutive words: two 16-byte loads
    const uint4* vs = reinterpret_cast<const uint4*>(a.v_sz + vblk * blk_words + m.vszo);
    const uint4 w0 = __ldg(vs), w1 = __ldg(vs + 1);
    r.vsz8[0] = w0.x; r.vsz8[1] = w0.y; r.vsz8[2] = w0.z; r.vsz8[3] = w0.w;
    r.vsz8[4] = w1.x; r.vsz8[5] = w1.y; r.vsz8[6] = w1.z; r.vsz8[7] = w1.w;
  }
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const uint8_t* src = vrow + t * head_row;
    if constexpr (R::kVWords == 4) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
      r.v[t][0] = w.x; r.v[t][R::kVWords > 1 ? 1 : 0] = w.y;
      r.v[t][R::kVWords > 2 ? 2 : 0] = w.z; r.v[t][R::kVWords > 3 ? 3 : 0] = w.w;
    } else if constexpr (R::kVWords == 2) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
      r.v[t][0] = w.x; r.v[t][R::kVWords > 1 ? 1 : 0] = w.y;
    } else {
      r.v[t][0] = __ldg(reinterpret_cast<const uint32_t*>(src));
    }
  }
  r.miss = false;
  r.sz_ok = false;
  r.ksz = r.vsz = 0u;
  if (tid < kTcTok) {
    const bool ok = (valid >> (tid / kBlock)) & 1u;
    r.sz_ok = ok && tok0 + tid < L;
    r.miss = tok0 + tid < L && !ok;
    if constexpr (KvTraits<KV>::kQuant && QBF) {  // the scale arrays of the exact path
      const int64_t i = pick4(sb, tid / kBlock) * blk_words + h * kBlock + tid % kBlock;
      r.ksz = __ldg(a.k_sz + i);
      r.vsz = __ldg(a.v_sz + i);
    }
    if (r.miss) report(a.dev_err, KVQ_DEV_ERR_BLOCK_ID);
  }
}

// The same registers as load_tile, for an INT8 pool, read from raw stage
// `st` (shared address) where the copies of tile tok0 have landed: row t of
// the K and V regions is tile token t, its 16-byte chunk c at c ^ (t mod 8).
template <bool QBF>
__device__ __forceinline__ void read_tile(const ExtendArgs& a, uint32_t st, int tok0, int L,
                                          int tid, RawTile<kI8>& r) {
  using R = RawTile<kI8>;
  const uint32_t valid = lds32(st + kRawValidOff);
  r.kmask = 0u;
#pragma unroll
  for (int i = 0; i < R::kKChunks; ++i) {
    int t, ch;
    k_item<kI8>(tid + kStageThreads * i, t, ch);
    r.k[i] = lds128(st + t * 128 + ((ch ^ (t & 7)) << 4));
    r.kmask |= ((valid >> (t / kBlock)) & 1u && tok0 + t < L ? 1u : 0u) << i;
    if constexpr (!QBF) r.ksz4[i] = lds32(st + kRawSzOff + 4 * t);
  }
  int tg, dc;
  v_item<kI8>(tid, tg, dc);
  const bool vok = (valid >> (tg >> 1)) & 1u;  // tokens 8 tg .. 8 tg + 7: block tg / 2
  r.vmask = 0u;
#pragma unroll
  for (int t = 0; t < 8; ++t) r.vmask |= (vok && tok0 + 8 * tg + t < L ? 1u : 0u) << t;
  if constexpr (!QBF) {
    const uint4 w0 = lds128(st + kRawSzOff + 4 * kTcTok + 32 * tg);
    const uint4 w1 = lds128(st + kRawSzOff + 4 * kTcTok + 32 * tg + 16);
    r.vsz8[0] = w0.x; r.vsz8[1] = w0.y; r.vsz8[2] = w0.z; r.vsz8[3] = w0.w;
    r.vsz8[4] = w1.x; r.vsz8[5] = w1.y; r.vsz8[6] = w1.z; r.vsz8[7] = w1.w;
  }
  // row 8 tg + t has t mod 8 = t: its chunk dc / 2 sits at (dc / 2) ^ t
  const uint32_t vrow = st + kRawVOff + 8 * tg * 128 + 8 * (dc & 1);
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const uint2 w = lds64(vrow + t * 128 + (((dc >> 1) ^ t) << 4));
    r.v[t][0] = w.x;
    r.v[t][1] = w.y;
  }
  r.miss = false;
  r.sz_ok = false;
  r.ksz = r.vsz = 0u;
  if (tid < kTcTok) {
    const bool ok = (valid >> (tid / kBlock)) & 1u;
    r.sz_ok = ok && tok0 + tid < L;
    r.miss = tok0 + tid < L && !ok;
    if constexpr (QBF) {
      r.ksz = lds32(st + kRawSzOff + 4 * tid);
      r.vsz = lds32(st + kRawSzOff + 4 * kTcTok + 4 * tid);
    }
    if (r.miss) report(a.dev_err, KVQ_DEV_ERR_BLOCK_ID);
  }
}

// 16-bit pair q (dims 2q, 2q + 1) of one token's 8-dim V piece, c - mid.
template <int KV>
__device__ __forceinline__ uint32_t piece_pair(const uint32_t (&w)[RawTile<KV>::kVWords], int q) {
  constexpr int kMid = KV == kI8 ? 128 : 8;
  if constexpr (KV == kF16) {
    return w[q];
  } else if constexpr (KV == kI8) {
    return bytes_to_f16(w[q >> 1], (q & 1) ? 0x4342u : 0x4140u);
  } else {
    const uint32_t byte = (w[0] >> (8 * q)) & 0xFF;
    return centred_pair<false>(byte & 0xF, byte >> 4, kMid);
  }
}

// Registers -> one stage of the ring: the K tile at `kt` (K-major, Q's type),
// V transposed at `vt` (fp16), the per-token S_k', Z_k', S_v, Z_v' arrays at
// `sz` (softmax scale folded into the K pair), and at `info` the largest S_v
// of each half-tile and the two 32-token masks of missing tokens. `tid` is
// the staging thread (0..127).
// fp16 pair (mid, mid) of a pool kind: 128 for INT8 codes, 8 for INT4
template <int KV>
__device__ __forceinline__ uint32_t kMidPair() {
  return KV == kI8 ? 0x58005800u : 0x48004800u;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

template <int KV, bool QBF>
__device__ __forceinline__ void store_tile(const ExtendArgs& a, const RawTile<KV>& r, uint32_t kt,
                                           uint32_t vt, uint32_t sz, uint32_t info, int tid) {
  using R = RawTile<KV>;
  constexpr int kMid = KV == kI8 ? 128 : 8;
  constexpr bool VDEQ = !QBF;  // fp16 queries: V is staged dequantized
  if (tid < kTcTok && !VDEQ) {  // whole warps: the first two of the staging group
    float Sk = a.sm_scale_log2, Zk = 0.f, Sv = 1.f, Zv = 0.f;
    if constexpr (KvTraits<KV>::kQuant) {
      const uint32_t ksz = r.sz_ok ? r.ksz : 0u, vsz = r.sz_ok ? r.vsz : 0u;
      const float s_k = half_lo(ksz), s_v = half_lo(vsz);
      Sk = s_k * a.sm_scale_log2;
      Zk = (half_hi(ksz) + kMid * s_k) * a.sm_scale_log2;
      Sv = s_v;
      Zv = half_hi(vsz) + kMid * s_v;
    }
    sts32(sz + 4 * tid, __float_as_uint(Sk));
    sts32(sz + 4 * kTcTok + 4 * tid, __float_as_uint(Zk));
    sts32(sz + 8 * kTcTok + 4 * tid, __float_as_uint(Sv));
    sts32(sz + 12 * kTcTok + 4 * tid, __float_as_uint(Zv));
    float mx = Sv;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    if ((tid & 31) == 0) sts32(info + 4 * (tid >> 5), __float_as_uint(mx));
  }
  if (tid < kTcTok) {
    const uint32_t miss = __ballot_sync(kFull, r.miss);
    if ((tid & 31) == 0) sts32(info + 8 + 4 * (tid >> 5), miss);
  }
#pragma unroll
  for (int i = 0; i < R::kKChunks; ++i) {
    int t, ch;
    k_item<KV>(tid + kStageThreads * i, t, ch);
    const uint32_t x[4] = {r.k[i].x, r.k[i].y, r.k[i].z, r.k[i].w};
    // dequantized K (fp16 queries): (c - mid) S + (Z + mid S), one rounding;
    // zero for a token outside the context
    uint32_t ks2 = 0u, kz2 = 0u;
    if constexpr (VDEQ && KvTraits<KV>::kQuant) {
      const uint32_t w = (r.kmask >> i) & 1u ? r.ksz4[i] : 0u;
      ks2 = prmt(w, w, 0x1010u);
      kz2 = hfma2(kMidPair<KV>(), ks2, prmt(w, w, 0x3232u));
    }
    auto kdeq = [&](uint32_t pair) {
      if constexpr (VDEQ && KvTraits<KV>::kQuant) return hfma2(pair, ks2, kz2);
      return pair;
    };
    if constexpr (KV == kF16) {
      sts128(kt + umma_kmajor_offset(kTcTok, t, 8 * ch), x[0], x[1], x[2], x[3]);
    } else if constexpr (KV == kI8) {
      // c - 128 exactly: fp16 by a byte permute into 1024 + c and one packed
      // subtract; bf16 through fp32
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t word = x[2 * hf + (q >> 1)];
          if constexpr (QBF) {
            v[q] = (q & 1) ? bytes_to_bf16_pair(word, 2, 3) : bytes_to_bf16_pair(word, 0, 1);
          } else {
            v[q] = kdeq(bytes_to_f16(word, (q & 1) ? 0x4342u : 0x4140u));
          }
        }
        sts128(kt + umma_kmajor_offset(kTcTok, t, 16 * ch + 8 * hf), v[0], v[1], v[2], v[3]);
      }
    } else {
#pragma unroll
      for (int qt = 0; qt < 4; ++qt) {
        uint32_t v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t byte = (x[qt] >> (8 * q)) & 0xFF;
          v[q] = kdeq(centred_pair<QBF>(byte & 0xF, byte >> 4, kMid));
        }
        sts128(kt + umma_kmajor_offset(kTcTok, t, 32 * ch + 8 * qt), v[0], v[1], v[2], v[3]);
      }
    }
  }
  // V: 8 tokens x 8 dims -> 8 rows (dims) of 8 tokens, one 16-byte store each
  int tg, dc;
  v_item<KV>(tid, tg, dc);
  // dequantized V (fp16 queries): per token pair, (S, S') and (Z + mid S, ..)
  // as fp16 pairs, zero for tokens outside the context
  uint32_t s2[4], z2[4];
  if constexpr (VDEQ && KvTraits<KV>::kQuant) {
#pragma unroll
    for (int tp = 0; tp < 4; ++tp) {
      const uint32_t wa = (r.vmask >> (2 * tp)) & 1u ? r.vsz8[2 * tp] : 0u;
      const uint32_t wb = (r.vmask >> (2 * tp + 1)) & 1u ? r.vsz8[2 * tp + 1] : 0u;
      s2[tp] = prmt(wa, wb, 0x5410u);
      z2[tp] = hfma2(kMidPair<KV>(), s2[tp], prmt(wa, wb, 0x7632u));
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int tp = 0; tp < 4; ++tp) {
      if constexpr (KV == kI8) {
        // transposed at the byte level first, [t0 d, t1 d, t0 d', t1 d'] for
        // dims d = 2q, d' = 2q + 1 of tokens t0 = 2 tp, t1 = 2 tp + 1; then
        // each half as the pair c - 128 (one permute fewer per two pairs)
        const uint32_t tb = prmt(r.v[2 * tp][q >> 1], r.v[2 * tp + 1][q >> 1],
                                 (q & 1) ? 0x7362u : 0x5140u);
        lo[tp] = bytes_to_f16(tb, 0x4140u);
        hi[tp] = bytes_to_f16(tb, 0x4342u);
      } else {
        const uint32_t p0 = piece_pair<KV>(r.v[2 * tp], q);
        const uint32_t p1 = piece_pair<KV>(r.v[2 * tp + 1], q);
        lo[tp] = prmt(p0, p1, 0x5410u);
        hi[tp] = prmt(p0, p1, 0x7632u);
      }
      if constexpr (VDEQ && KvTraits<KV>::kQuant) {  // (c - mid) S + (Z + mid S), one rounding
        lo[tp] = hfma2(lo[tp], s2[tp], z2[tp]);
        hi[tp] = hfma2(hi[tp], s2[tp], z2[tp]);
      }
    }
    sts128(vt + umma_kmajor_offset(kVRows, 8 * dc + 2 * q, 8 * tg), lo[0], lo[1], lo[2], lo[3]);
    sts128(vt + umma_kmajor_offset(kVRows, 8 * dc + 2 * q + 1, 8 * tg), hi[0], hi[1], hi[2], hi[3]);
  }
}

// 2^x of both fp16 halves, one instruction
__device__ __forceinline__ uint32_t ex2_h2(uint32_t h) {
  uint32_t r;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(r) : "r"(h));
  return r;
}

// One fp32 column of this thread's TMEM lane.
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r)
      : "r"(taddr)
      : "memory");
  return __uint_as_float(r);
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ---- waits --------------------------------------------------------------------

// One thread's bounded wait on a barrier phase that also gives up when another
// role has aborted the CTA (the flag at `abort_flag`); on its own timeout it
// sets the flag and reports KVQ_DEV_ERR_TIMEOUT. try_wait blocks in hardware
// for a while; the flag and the clock are read only after 64 such tries.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int32_t* dev_err) {
#pragma unroll 1
  for (int i = 0; i < 64; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (global_ns() - t0 > 2000000000ull) {
      *abort_flag = 1;
      report(dev_err, KVQ_DEV_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// The same for a whole warp, with one verdict for all its lanes.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* dev_err) {
  const bool ok = wait_or_abort(bar, parity, abort_flag, dev_err);
  return __all_sync(kFull, ok);
}

__device__ __forceinline__ void mbar_init_count(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_one(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 64 consecutive fp32 columns of this thread's TMEM lane: two loads, one wait;
// the second half passes through an empty asm placed after the wait so that no
// use of it can move above the wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[32 * h + 0]), "=r"(r[32 * h + 1]), "=r"(r[32 * h + 2]), "=r"(r[32 * h + 3]),
          "=r"(r[32 * h + 4]), "=r"(r[32 * h + 5]), "=r"(r[32 * h + 6]), "=r"(r[32 * h + 7]),
          "=r"(r[32 * h + 8]), "=r"(r[32 * h + 9]), "=r"(r[32 * h + 10]), "=r"(r[32 * h + 11]),
          "=r"(r[32 * h + 12]), "=r"(r[32 * h + 13]), "=r"(r[32 * h + 14]),
          "=r"(r[32 * h + 15]), "=r"(r[32 * h + 16]), "=r"(r[32 * h + 17]),
          "=r"(r[32 * h + 18]), "=r"(r[32 * h + 19]), "=r"(r[32 * h + 20]),
          "=r"(r[32 * h + 21]), "=r"(r[32 * h + 22]), "=r"(r[32 * h + 23]),
          "=r"(r[32 * h + 24]), "=r"(r[32 * h + 25]), "=r"(r[32 * h + 26]),
          "=r"(r[32 * h + 27]), "=r"(r[32 * h + 28]), "=r"(r[32 * h + 29]),
          "=r"(r[32 * h + 30]), "=r"(r[32 * h + 31])
        : "r"(taddr + 32u * h));
  }
  // the wait, tied to the first half's registers
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
        "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
        "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
  asm volatile(""
               : "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]),
                 "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]),
                 "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]),
                 "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]),
                 "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]),
                 "+r"(r[62]), "+r"(r[63])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this thread's TMEM lane, scaled by `f` in
// place (load, wait, multiply, store, wait).
__device__ __forceinline__ void tmem_scale16(uint32_t taddr, float f) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};\n"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// ---- work units -----------------------------------------------------------------

struct TcUnit {
  int b, h, qt, ntiles;
  TcReq s;
};

// Unit u: request b (by the prefix sums of units per request), kv head h and
// 256-row tile qt (longest first), with the number of 64-token context tiles
// its last query attends.
__device__ __forceinline__ TcUnit tc_unit(const ExtendArgs& a, const int32_t* ucum, int u) {
  int lo = 0, hi = a.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ucum[mid] <= u) lo = mid; else hi = mid - 1;
  }
  TcUnit w;
  w.b = lo;
  w.s = tc_req(a, lo);
  const int r = u - ucum[lo];
  w.h = r % a.kv_heads;
  w.qt = w.s.tiles - 1 - r / a.kv_heads;
  const int i_max = min(w.s.C - 1, (w.qt * kUnitRows + kUnitRows - 1) / a.group);
  const int n_tok = w.s.L - w.s.C + i_max + 1;
  w.ntiles = (n_tok + kTcTok - 1) / kTcTok;
  return w;
}

struct TcShared {
  uint32_t base, tmem;
  volatile int* abort_flag;
  volatile int* unit_slot;
  const int32_t* ucum;
  int total;
  __device__ __forceinline__ uint32_t bar(uint32_t i) const { return base + kBarOff + 8u * i; }
};

// ---- roles ------------------------------------------------------------------------

// Hands out unit k (an atomic counter) through slot k mod 2 once every
// working warp has read unit k - 2 from it. The one thread that runs it is
// the raw-ring producer's lane 0 (INT8 pools: it runs furthest ahead, so the
// copies of a unit's first tiles start while the previous unit is staged),
// else thread 0 of the staging warpgroup.
__device__ __forceinline__ void publish_unit(const ExtendArgs& a, const TcShared& c, uint32_t k) {
  const uint32_t slot = k & 1u;
  if (k < 2 || wait_or_abort(c.bar(kBarUnitEmpty + slot), ((k >> 1) - 1u) & 1u, c.abort_flag,
                             a.dev_err)) {
    c.unit_slot[slot] = atomicAdd(a.counter, 1);
    mbar_arrive_one(c.bar(kBarUnitFull + slot));
  }
}

// Staging warpgroup: fills the K/V ring (and hands out the units when there
// is no raw-ring producer).
template <int KV, bool QBF>
__device__ __forceinline__ void staging_role(const ExtendArgs& a, const TcShared& c, int tid) {
  const int lane = tid & 31;
  if constexpr (!QBF) {
    // rows 128..143 of every V stage: ones, then zeros (the B columns that give
    // each row's sum of P); published with each stage's first arrival
    for (int e = tid; e < kStages * 16 * 8; e += kStageThreads) {
      const int stg = e / 128, rr = (e / 8) % 16, ch = e % 8;
      const uint32_t v = rr == 0 ? 0x3C003C00u : 0u;
      sts128(c.base + kVOff + stg * kVBytes + umma_kmajor_offset(kVRows, 128 + rr, 8 * ch), v, v,
             v, v);
    }
    fence_async_smem();
  }
  uint32_t tc = 0;  // tiles staged so far
  uint32_t rc = 0;  // raw stages consumed so far (INT8 pools)
  for (uint32_t k = 0;; ++k) {
    const uint32_t slot = k & 1u;
    if (!raw_ring<KV>() && tid == 0) publish_unit(a, c, k);
    __syncwarp();
    if (!warp_wait(c.bar(kBarUnitFull + slot), (k >> 1) & 1u, c.abort_flag, a.dev_err)) return;
    const int u = c.unit_slot[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive_one(c.bar(kBarUnitEmpty + slot));
    if (u >= c.total) return;
    const TcUnit w = tc_unit(a, c.ucum, u);
    const int n = w.ntiles, L = w.s.L;
    // registers -> the next K/V stage
    auto store_one = [&](const RawTile<KV>& r) {
      const uint32_t st = tc % kStages, use = tc / kStages;
      if (use > 0 &&
          !warp_wait(c.bar(kBarKvEmpty + st), (use - 1u) & 1u, c.abort_flag, a.dev_err))
        return false;
      store_tile<KV, QBF>(a, r, c.base + kKOff + st * kKBytes, c.base + kVOff + st * kVBytes,
                          c.base + kSzOff + st * kSzBytes, c.base + kInfoOff + st * 16u, tid);
      fence_async_smem();
      mbar_arrive_one(c.bar(kBarKvFull + st));
      ++tc;
      return true;
    };
    if constexpr (raw_ring<KV>()) {
      // the producer warp's copies land tile j in raw stage rc mod kRawStages
      for (int j = 0; j < n; ++j) {
        const uint32_t rs = rc % kRawStages, use = rc / kRawStages;
        if (!warp_wait(c.bar(kBarRawFull + rs), use & 1u, c.abort_flag, a.dev_err)) return;
        RawTile<KV> r;
        read_tile<QBF>(a, c.base + kRawOff + rs * kRawBytes, j * kTcTok, L, tid, r);
        mbar_arrive_one(c.bar(kBarRawEmpty + rs));
        ++rc;
        if (!store_one(r)) return;
      }
    } else {
      // tile j's codes are loaded while tile j - 1 is staged, its block ids
      // a tile before that
      const int32_t* bt = a.block_tables + static_cast<int64_t>(w.b) * a.max_blocks;
      StageMap<KV> map;
      map.init(a, w.h, tid);
      RawTile<KV> r;
      int4 blk = tile_blocks(bt, 0, a.max_blocks);
      if (n > 0) load_tile<KV, QBF>(a, map, blk, 0, L, w.h, tid, r);
      blk = tile_blocks(bt, kTcTok, a.max_blocks);
      for (int j = 0; j < n; ++j) {
        if (!store_one(r)) return;
        if (j + 1 < n) {
          load_tile<KV, QBF>(a, map, blk, (j + 1) * kTcTok, L, w.h, tid, r);
          blk = tile_blocks(bt, (j + 2) * kTcTok, a.max_blocks);
        }
      }
    }
  }
}

// Raw-ring producer (INT8 pools; warp 14): hands out the units, and for each
// tile of each unit one lane writes which of the tile's four blocks are valid
// into the next raw stage and copies, for the unit's kv head, the four
// blocks' K and V rows (one TMA box per block and tensor) and their
// scale/zero words (64-byte bulk copies); a block past the context or
// outside the pool is read from block 0 and masked by the consumers. Before
// the warp leaves, every copy it issued has landed (bounded waits), so none
// is in flight when the CTA ends.
template <int KV>
__device__ __forceinline__ void producer_role(const ExtendArgs& a, const TcShared& c, int lane) {
  uint32_t rt = 0;  // tiles issued
  bool ok = true;
  for (uint32_t k = 0; ok; ++k) {
    const uint32_t slot = k & 1u;
    if (lane == 0) publish_unit(a, c, k);
    __syncwarp();
    if (!warp_wait(c.bar(kBarUnitFull + slot), (k >> 1) & 1u, c.abort_flag, a.dev_err)) break;
    const int u = c.unit_slot[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive_one(c.bar(kBarUnitEmpty + slot));
    if (u >= c.total) break;
    const TcUnit w = tc_unit(a, c.ucum, u);
    const int32_t* bt = a.block_tables + static_cast<int64_t>(w.b) * a.max_blocks;
    int4 blk = tile_blocks(bt, 0, a.max_blocks);
    for (int j = 0; j < w.ntiles; ++j) {
      const uint32_t rs = rt % kRawStages, use = rt / kRawStages;
      if (use > 0 &&
          !warp_wait(c.bar(kBarRawEmpty + rs), (use - 1u) & 1u, c.abort_flag, a.dev_err)) {
        ok = false;
        break;
      }
      uint32_t valid;
      const int4 sb = safe_blocks(a, blk, j * kTcTok, w.s.L, &valid);
      if (lane == 0) {
        const uint32_t st = c.base + kRawOff + rs * kRawBytes, bar = c.bar(kBarRawFull + rs);
        sts32(st + kRawValidOff, valid);
        fence_async_smem();  // after the consumers' reads of the stage's last use
        mbar_arm(bar, kRawTx);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int phys = pick4(sb, b);
          const int64_t szi = (static_cast<int64_t>(phys) * a.kv_heads + w.h) * kBlock;
          tma_tile_4d(st + b * kRawBox, &a.k_map, 0, w.h, 0, phys, bar);
          tma_tile_4d(st + kRawVOff + b * kRawBox, &a.v_map, 0, w.h, 0, phys, bar);
          bulk_copy(st + kRawSzOff + 64 * b, a.k_sz + szi, 64, bar);
          bulk_copy(st + kRawSzOff + 4 * kTcTok + 64 * b, a.v_sz + szi, 64, bar);
        }
      }
      __syncwarp();
      ++rt;
      blk = tile_blocks(bt, (j + 1) * kTcTok, a.max_blocks);
    }
  }
  if (lane == 0)
    for (uint32_t i = rt > kRawStages ? rt - kRawStages : 0u; i < rt; ++i)
      mbar_wait(c.bar(kBarRawFull + i % kRawStages), (i / kRawStages) & 1u);
  __syncwarp();
}

// One lane of a converged warp (elect.sync).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n .reg .pred P;\n elect.sync _|P, 0xffffffff;\n selp.b32 %0, 1, 0, P;\n}"
      : "=r"(pred));
  return pred != 0;
}

// An MMA warp, one per softmax warpgroup g (warp 12 for g = 0, 13 for g = 1,
// on different sub-partitions, so the two issue in parallel): all 32 lanes
// run the loop (the descriptors stay warp-uniform) and wait together; one
// elected lane issues each product and commit. The two warpgroups' products
// need no order between them; a K/V stage is released when both MMA warps
// have committed its products (the empty barrier takes two arrivals).
template <bool QBF>
__device__ __forceinline__ void mma_role(const ExtendArgs& a, const TcShared& c, int g,
                                         int lane) {
  constexpr uint32_t idesc_s = umma_idesc_f16(QBF, kWgRows, kTcTok);
  constexpr uint32_t idesc_o = umma_idesc_f16(false, kWgRows, o_cols<QBF>());
  // descriptors of k-step 0; a k-step adds its byte offset / 16 to the low field
  const uint64_t q_desc0 = umma_desc_sw128(c.base + kQOff + g * kQBytes, 1024);
  const uint64_t k_desc0 = umma_desc_sw128(c.base + kKOff, 1024);
  const uint64_t v_desc0 = umma_desc_sw128(c.base + kVOff, 1024);
  const uint32_t s_tmem = c.tmem + 64u * g, o_tmem = c.tmem + 128u + o_cols<QBF>() * g;
  const uint32_t p_tmem = c.tmem + p_col<QBF>() + 32u * g;
  auto issue_s = [&](uint32_t st) {
    const uint64_t kd = k_desc0 + (st * kKBytes >> 4);
    if (elect_one()) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        umma_f16(s_tmem, q_desc0 + (((k >> 2) * (kWgRows * 128) + (k & 3) * 32) >> 4),
                 kd + (((k >> 2) * (kTcTok * 128) + (k & 3) * 32) >> 4), idesc_s, k > 0);
      umma_commit(c.bar(kBarSFull + g));
    }
    __syncwarp();
  };
  auto issue_o = [&](uint32_t st, bool acc) {
    const uint64_t vd = v_desc0 + (st * kVBytes >> 4);
    if (elect_one()) {
#pragma unroll
      for (int k = 0; k < kTcTok / 16; ++k)
        umma_f16_tmem_a(o_tmem, p_tmem + 8u * k, vd + ((k * 32) >> 4), idesc_o, acc || k > 0);
      umma_commit(c.bar(kBarODone + g));
      umma_commit(c.bar(kBarKvEmpty + st));  // this warpgroup is done with the stage
    }
    __syncwarp();
  };
  auto wait = [&](uint32_t b, uint32_t parity) {
    const bool ok = warp_wait(b, parity, c.abort_flag, a.dev_err);
    tc_fence_after();
    return ok;
  };
  uint32_t tc = 0;  // tiles issued so far
  for (uint32_t k = 0;; ++k) {
    const uint32_t slot = k & 1u;
    if (!wait(c.bar(kBarUnitFull + slot), (k >> 1) & 1u)) return;
    const int u = c.unit_slot[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive_one(c.bar(kBarUnitEmpty + slot));
    if (u >= c.total) return;
    const int n = tc_unit(a, c.ucum, u).ntiles;
    if (!wait(c.bar(kBarQFull + g), k & 1u)) return;
    if (!wait(c.bar(kBarKvFull + tc % kStages), (tc / kStages) & 1u)) return;
    issue_s(tc % kStages);
    for (int j = 0; j < n; ++j, ++tc) {
      const uint32_t st = tc % kStages, nx = (tc + 1u) % kStages;
      // S of the next tile as soon as the warpgroup has read this one out of
      // TMEM: it runs while the warpgroup computes this tile's P'
      if (!wait(c.bar(kBarSRead + g), tc & 1u)) return;
      if (j + 1 < n) {
        if (!wait(c.bar(kBarKvFull + nx), ((tc + 1u) / kStages) & 1u)) return;
        issue_s(nx);
      }
      if (!wait(c.bar(kBarPFull + g), tc & 1u)) return;
      issue_o(st, j > 0);
    }
  }
}

// A softmax warpgroup: warps 4 g .. 4 g + 3, one thread per row i of the
// unit's half g.
template <int KV, bool QBF>
__device__ __forceinline__ void softmax_role(const ExtendArgs& a, const TcShared& c, int g,
                                             int i, int warp) {
  constexpr bool kQuant = KvTraits<KV>::kQuant;
  constexpr bool kVDeq = !QBF;  // K and V staged dequantized: P = p, no scale arrays
  const uint32_t lane_addr = c.tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
  const uint32_t s_addr = lane_addr + 64u * g, o_addr = lane_addr + 128u + o_cols<QBF>() * g;
  const uint32_t q_tile = c.base + kQOff + g * kQBytes;
  const uint32_t p_addr = lane_addr + p_col<QBF>() + 32u * g;
  const int lane = i & 31;
  auto wait = [&](uint32_t b, uint32_t parity) {
    return warp_wait(b, parity, c.abort_flag, a.dev_err);
  };
  uint32_t tc = 0;
  for (uint32_t k = 0;; ++k) {
    const uint32_t slot = k & 1u;
    if (!wait(c.bar(kBarUnitFull + slot), (k >> 1) & 1u)) return;
    const int u = c.unit_slot[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive_one(c.bar(kBarUnitEmpty + slot));
    if (u >= c.total) return;
    const TcUnit w = tc_unit(a, c.ucum, u);
    const int row = w.qt * kUnitRows + g * kWgRows + i;
    const int qi = row / a.group;
    const int hq = w.h * a.group + row % a.group;
    const bool valid = qi < w.s.C;
    const int pos = w.s.L - w.s.C + qi;

    // Q row of this thread into the K-major tile (zeros for a padding row)
    float qsum = 0.f;
    {
      const uint4* qp = reinterpret_cast<const uint4*>(
          static_cast<const uint16_t*>(a.q) +
          ((static_cast<int64_t>(w.s.q0) + qi) * a.q_heads + hq) * kHeadDim);
#pragma unroll 4
      for (int ch = 0; ch < 16; ++ch) {
        const uint4 x = valid ? qp[ch] : make_uint4(0u, 0u, 0u, 0u);
        sts128(q_tile + umma_kmajor_offset(kWgRows, i, 8 * ch), x.x, x.y, x.z, x.w);
        if constexpr (kQuant && !kVDeq) {
          qsum += lo_to_float<QBF>(x.x) + hi_to_float<QBF>(x.x) + lo_to_float<QBF>(x.y) +
                  hi_to_float<QBF>(x.y) + lo_to_float<QBF>(x.z) + hi_to_float<QBF>(x.z) +
                  lo_to_float<QBF>(x.w) + hi_to_float<QBF>(x.w);
        }
      }
    }
    fence_async_smem();
    mbar_arrive_one(c.bar(kBarQFull + g));

    const float2 qs2 = make_float2(qsum, qsum);
    float m = -INFINITY;
    float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // two chains each
    float2 z2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    for (int j = 0; j < w.ntiles; ++j, ++tc) {
      const uint32_t st = tc % kStages;
      if (!wait(c.bar(kBarSFull + g), tc & 1u)) return;
      // the stage's scale arrays (already complete: S was computed from it)
      if (!wait(c.bar(kBarKvFull + st), (tc / kStages) & 1u)) return;
      tc_fence_after();
      const uint32_t sz = c.base + kSzOff + st * kSzBytes;
      float x[kTcTok];
      tmem_ld64(s_addr, x);
      tc_fence_before();
      mbar_arrive_one(c.bar(kBarSRead + g));  // S_g's columns may take the next tile
      // kVDeq: K was staged dequantized; s = raw * softmax scale (log2 units).
      // A positive scale goes into the exponent's FMA below (the maximum of
      // raw scores then gives the maximum of s); any other scale is applied
      // here.
      const float cs = a.sm_scale_log2;
      if constexpr (kVDeq) {
        if (!(cs > 0.f)) {
          const float2 c2 = make_float2(cs, cs);
#pragma unroll
          for (int q = 0; q < kTcTok / 2; ++q) {
            const float2 r = __fmul2_rn(make_float2(x[2 * q], x[2 * q + 1]), c2);
            x[2 * q] = r.x;
            x[2 * q + 1] = r.y;
          }
        }
      } else {
      // s = S_k' raw + Z_k' sum(q) (softmax scale folded in), two tokens per
      // instruction
#pragma unroll
      for (int q = 0; q < kTcTok / 4; ++q) {
        const float4 sk = lds_f4(sz + 16 * q), zk = lds_f4(sz + 4 * kTcTok + 16 * q);
        const float2 b0 = __fmul2_rn(make_float2(zk.x, zk.y), qs2);
        const float2 b1 = __fmul2_rn(make_float2(zk.z, zk.w), qs2);
        const float2 r0 = __ffma2_rn(make_float2(sk.x, sk.y), make_float2(x[4 * q], x[4 * q + 1]), b0);
        const float2 r1 =
            __ffma2_rn(make_float2(sk.z, sk.w), make_float2(x[4 * q + 2], x[4 * q + 3]), b1);
        x[4 * q] = r0.x;
        x[4 * q + 1] = r0.y;
        x[4 * q + 2] = r1.x;
        x[4 * q + 3] = r1.y;
      }
      }
      // positions past the row's own, and missing tokens, are masked
      const int tok0 = j * kTcTok;
      if (tok0 + kTcTok - 1 > pos) {
#pragma unroll
        for (int t = 0; t < kTcTok; ++t)
          if (tok0 + t > pos) x[t] = -INFINITY;
      }
      const float4 info = lds_f4(c.base + kInfoOff + st * 16u);
      const uint32_t miss0 = __float_as_uint(info.z), miss1 = __float_as_uint(info.w);
      if ((miss0 | miss1) != 0u) {
#pragma unroll
        for (int t = 0; t < kTcTok; ++t)
          if (((t < 32 ? miss0 : miss1) >> (t & 31)) & 1u) x[t] = -INFINITY;
      }
      float bq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // independent chains
#pragma unroll
      for (int t = 0; t < kTcTok; t += 2) bq[(t >> 1) & 3] = max3(bq[(t >> 1) & 3], x[t], x[t + 1]);
      const float cm = (kVDeq && cs > 0.f) ? cs : 1.f;  // scale still to apply
      const float bm = fmaxf(max3(bq[0], bq[1], bq[2]), bq[3]) * cm;
      // the reference maximum moves only when a score exceeds it by more than
      // tau (log2 units): p <= 2^tau then, and P' = p S_v stays within fp16
      // when the tile's largest V scale is at most 240 (else tau = 0: exact)
      const float tau = (kVDeq || fmaxf(info.x, info.y) <= 240.f) ? 8.f : 0.f;
      const float mn = (m == -INFINITY || bm > m + tau) ? fmaxf(m, bm) : m;
      const float al = (m == -INFINITY || mn == m) ? 1.f : ex2(m - mn);
      if (j > 0) {
        // O_g of the previous tile is complete (its P' buffer is free again)
        if (!wait(c.bar(kBarODone + g), (tc - 1u) & 1u)) return;
        tc_fence_after();
        if (__any_sync(kFull, al != 1.f)) {
#pragma unroll 1
          for (int cc = 0; cc < static_cast<int>(o_cols<QBF>()) / 16; ++cc)
            tmem_scale16(o_addr + 16 * cc, al);
        }
      }
      const float2 al2 = make_float2(al, al);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        l2[e] = __fmul2_rn(l2[e], al2);
        z2[e] = __fmul2_rn(z2[e], al2);
      }
      m = mn;
      const float nref = m == -INFINITY ? 0.f : -m;
      const float2 nref2 = make_float2(nref, nref);
      uint32_t pw[kTcTok / 2];
      if constexpr (kVDeq) {
        // P = 2^(s - m) straight in fp16 pairs: the exponent pair rounded to
        // fp16 and one packed exponential; the row sum comes from the P V
        // product (V's row of ones), over the same fp16 values
        const float2 cm2 = make_float2(cm, cm);
#pragma unroll
        for (int q = 0; q < kTcTok / 2; ++q) {
          const float2 d = __ffma2_rn(make_float2(x[2 * q], x[2 * q + 1]), cm2, nref2);
          pw[q] = ex2_h2(pack2<false>(d.x, d.y));
        }
      } else {
      // P' = p S_v (quantized) or p, fp16, into this row of P'_g in TMEM
#pragma unroll
      for (int c8 = 0; c8 < kTcTok / 8; ++c8) {
        float4 sva = make_float4(1.f, 1.f, 1.f, 1.f), svb = sva, zva = sva, zvb = sva;
        if constexpr (!kVDeq) {
          sva = lds_f4(sz + 8 * kTcTok + 32 * c8);
          svb = lds_f4(sz + 8 * kTcTok + 32 * c8 + 16);
          zva = lds_f4(sz + 12 * kTcTok + 32 * c8);
          zvb = lds_f4(sz + 12 * kTcTok + 32 * c8 + 16);
        }
        const float2 sv[4] = {make_float2(sva.x, sva.y), make_float2(sva.z, sva.w),
                              make_float2(svb.x, svb.y), make_float2(svb.z, svb.w)};
        const float2 zv[4] = {make_float2(zva.x, zva.y), make_float2(zva.z, zva.w),
                              make_float2(zvb.x, zvb.y), make_float2(zvb.z, zvb.w)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int t0 = 8 * c8 + 2 * q;
          const float2 d = __fadd2_rn(make_float2(x[t0], x[t0 + 1]), nref2);
          const float2 p = make_float2(ex2(d.x), ex2(d.y));
          l2[q & 1] = __fadd2_rn(l2[q & 1], p);
          if constexpr (kQuant && !kVDeq) {
            z2[q & 1] = __ffma2_rn(p, zv[q], z2[q & 1]);
            const float2 v = __fmul2_rn(p, sv[q]);
            pw[4 * c8 + q] = pack2<false>(v.x, v.y);
          } else {
            pw[4 * c8 + q] = pack2<false>(p.x, p.y);
          }
        }
      }
      }
      tmem_st32u(p_addr, pw);
      tc_fence_before();
      mbar_arrive_one(c.bar(kBarPFull + g));
    }
    // output row: (O + z) / l (every lane takes part in the TMEM reads)
    if (!wait(c.bar(kBarODone + g), (tc - 1u) & 1u)) return;
    tc_fence_after();
    {
      float l = (l2[0].x + l2[0].y) + (l2[1].x + l2[1].y);
      const float z = (z2[0].x + z2[0].y) + (z2[1].x + z2[1].y);
      if constexpr (kVDeq) l = tmem_ld1(o_addr + kHeadDim);  // the row-sum column
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(
          static_cast<uint16_t*>(a.out) +
          ((static_cast<int64_t>(w.s.q0) + qi) * a.q_heads + hq) * kHeadDim);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        float v[32];
        tmem_ld32(o_addr + 32 * cc, v);
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t wd[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              wd[e] = pack2<QBF>((v[8 * q + 2 * e] + z) * inv, (v[8 * q + 2 * e + 1] + z) * inv);
            dst[4 * cc + q] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
          }
        }
      }
    }
    tc_fence_before();
  }
}

template <int KV, bool QBF>
__global__ void __launch_bounds__(kTcThreads, 1) extend_tc_kernel(const __grid_constant__ ExtendArgs a) {
  extern __shared__ __align__(1024) unsigned char dsmem[];
  __shared__ int32_t warp_sum[kTcThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw_base = static_cast<uint32_t>(__cvta_generic_to_shared(dsmem));
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  unsigned char* gbase = dsmem + (base - raw_base);
  int32_t* ucum = reinterpret_cast<int32_t*>(gbase + kFixedBytes);

  // ---- work units per request, prefix-summed ----------------------------------
  {
    const int per = (a.batch + kTcThreads - 1) / kTcThreads;
    const int b0 = min(tid * per, a.batch), b1 = min(b0 + per, a.batch);
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
      const TcReq s = tc_req(a, b);
      sum += a.kv_heads * s.tiles;
      if (blockIdx.x == 0 && !s.ok) report(a.dev_err, KVQ_DEV_ERR_LENGTH);
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int basec = 0;
    for (int w = 0; w < warp; ++w) basec += warp_sum[w];
    int run = basec + incl - sum;
    for (int b = b0; b < b1; ++b) {
      ucum[b] = run;
      run += a.kv_heads * tc_req(a, b).tiles;
    }
    if (tid == kTcThreads - 1) ucum[a.batch] = basec + incl;
  }
  TcShared c;
  c.base = base;
  c.abort_flag = reinterpret_cast<volatile int*>(gbase + kAbortOff);
  c.unit_slot = reinterpret_cast<volatile int*>(gbase + kUnitOff);
  c.ucum = ucum;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init_count(c.bar(kBarKvFull + s), kStageThreads);
      mbar_init_count(c.bar(kBarKvEmpty + s), 2);  // one commit per MMA warp
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init_count(c.bar(kBarSFull + s), 1);
      mbar_init_count(c.bar(kBarPFull + s), kWgRows);
      mbar_init_count(c.bar(kBarODone + s), 1);
      mbar_init_count(c.bar(kBarQFull + s), kWgRows);
      mbar_init_count(c.bar(kBarUnitFull + s), 1);
      // lane 0 of every working warp: softmax, staging, MMA (and the producer)
      mbar_init_count(c.bar(kBarUnitEmpty + s), kSoftWarps + 4 + 2 + (raw_ring<KV>() ? 1 : 0));
      mbar_init_count(c.bar(kBarSRead + s), kWgRows);
    }
    mbar_init_count(c.bar(kBarDrain), 2);  // one commit per MMA warp
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init_count(c.bar(kBarRawFull + s), 1);  // the producer's arming arrival
      mbar_init_count(c.bar(kBarRawEmpty + s), kStageThreads);
    }
    *c.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(base + kSlotOff, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(c.tmem) : "r"(base + kSlotOff));
  c.total = ucum[a.batch];

  if (warp < kSoftWarps) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kHighRegs));
    softmax_role<KV, QBF>(a, c, warp >> 2, tid & (kWgRows - 1), warp);
  } else if (warp < kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLowRegs));
    staging_role<KV, QBF>(a, c, tid - kSoftWarps * 32);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLowRegs));
    if (warp == kMmaWarp || warp == kMmaWarp + 1) {
      mma_role<QBF>(a, c, warp - kMmaWarp, lane);
      // every product either MMA warp issued completes before the TMEM is freed
      __syncwarp();
      if (elect_one()) {
        umma_commit(c.bar(kBarDrain));
        mbar_wait(c.bar(kBarDrain), 0);
      }
      __syncwarp();
    } else if (raw_ring<KV>() && warp == kMmaWarp + 2) {
      producer_role<KV>(a, c, lane);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(c.tmem, kTmemCols);
  }
}

template <int KV, bool QBF>
cudaError_t launch_tc_t(const ExtendArgs& a, int grid, cudaStream_t s) {
  thread_local int opted_in_device = -1;  // per host thread: no shared state
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (opted_in_device != dev) {
    e = cudaFuncSetAttribute(extend_tc_kernel<KV, QBF>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tc_smem_bytes(kTcMaxBatch)));
    if (e != cudaSuccess) return e;
    // two CTAs per SM need the largest shared-memory carveout
    e = cudaFuncSetAttribute(extend_tc_kernel<KV, QBF>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    opted_in_device = dev;
  }
  extend_tc_kernel<KV, QBF><<<grid, kTcThreads, tc_smem_bytes(a.batch), s>>>(a);
  return cudaGetLastError();
}

template <int KV, bool QBF>
int tc_occupancy_t(int batch) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  thread_local int cached_dev = -1, cached_batch = -1, cached_n = 0;
  if (dev == cached_dev && batch == cached_batch) return cached_n;
  if (cudaFuncSetAttribute(extend_tc_kernel<KV, QBF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(tc_smem_bytes(kTcMaxBatch))) != cudaSuccess ||
      cudaFuncSetAttribute(extend_tc_kernel<KV, QBF>,
                           cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, extend_tc_kernel<KV, QBF>, kTcThreads,
                                                    tc_smem_bytes(batch)) != cudaSuccess)
    return 0;
  cached_dev = dev;
  cached_batch = batch;
  cached_n = n;
  return n;
}

}  // namespace

int extend_tc_max_batch() { return kTcMaxBatch; }

bool extend_tc_supported(int kv_dtype, int q_dtype) {
  return kv_dtype == kI8 || kv_dtype == kI4 || (kv_dtype == kF16 && q_dtype == kF16);
}

cudaError_t launch_extend_tc(const ExtendArgs& a, int kv_dtype, int q_dtype, int grid,
                             cudaStream_t s) {
  const bool qbf = q_dtype == kBF16;
  switch (kv_dtype) {
    case kF16:
      return launch_tc_t<kF16, false>(a, grid, s);
    case kI8:
      return qbf ? launch_tc_t<kI8, true>(a, grid, s) : launch_tc_t<kI8, false>(a, grid, s);
    case kI4:
      return qbf ? launch_tc_t<kI4, true>(a, grid, s) : launch_tc_t<kI4, false>(a, grid, s);
    default:
      return cudaErrorInvalidValue;
  }
}

int extend_tc_ctas_per_sm(int kv_dtype, int q_dtype, int batch) {
  const bool qbf = q_dtype == kBF16;
  switch (kv_dtype) {
    case kF16: return tc_occupancy_t<kF16, false>(batch);
    case kI8: return qbf ? tc_occupancy_t<kI8, true>(batch) : tc_occupancy_t<kI8, false>(batch);
    case kI4: return qbf ? tc_occupancy_t<kI4, true>(batch) : tc_occupancy_t<kI4, false>(batch);
    default: return 0;
  }
}

}  // namespace kvq

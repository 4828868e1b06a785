// kvq_extend_tc: extend (chunked prefill) attention on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// Same computation as kvq_extend.cu ("pymllm Runtime Design", forward stage:
// extend / prefill; LMDeploy article §2.3: prefills split into chunks; §2.4:
// per-token, per-head INT8/INT4 scale and zero). A CTA takes 128 rows (query,
// q head) of one kv head = the 128 TMEM lanes, one thread per row, and walks
// the request's context in tiles of 64 tokens (4 blocks):
//   1. the 128 threads stage the tile: K codes become centred 16-bit values
//      c - mid (exact; Q's type) in a K-major 128-byte-swizzled tile, V codes
//      become c - mid in fp16 written transposed (dims as rows, tokens as the
//      reduction axis), so both products read K-major operands; the
//      per-token scale S and shifted zero Z + mid S go to a small table;
//   2. one thread issues S = Q K^T (M 128, N 64, K 128: 8 MMAs) into TMEM;
//   3. every thread reads its row of S (tcgen05.ld), applies
//      s = S_k (q.(c - mid)) + (Z_k + mid S_k) sum(q), the causal mask and the
//      online softmax (no shuffles: a thread owns its row); when its running
//      maximum moves by more than a threshold, the warp rescales its rows of
//      O in TMEM (a stale maximum only scales every term alike); P' = p S_v goes
//      to shared memory in fp16 and sum p (Z_v + mid S_v) stays in a register;
//   4. one thread issues O += P' V (M 128, N 128, K 64: 4 MMAs) into TMEM.
// At the end each thread reads its row of O, adds the zero term, divides by
// the softmax sum and writes the output row. Every mbarrier wait is bounded
// (2 s; then the CTA reports KVQ_DEV_ERR_TIMEOUT, frees its TMEM and stops).
// Work units (request, kv head, 128-row tile) come from an atomic counter,
// longest tiles first. Staging is not overlapped with the products in this
// version.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tile.cuh"
#include "kvq_umma.cuh"

namespace kvq {
namespace {

constexpr int kTcRows = 128;   // rows per CTA (M, TMEM lanes)
constexpr int kTcTok = 64;     // tokens per context tile (N of S, K of P V)
constexpr int kTcThreads = 128;
constexpr uint32_t kTmemCols = 256;  // S: columns 0..63, O: 64..191

// shared memory, offsets from a 1024-byte aligned base
constexpr uint32_t kQOff = 0;                       // 2 x 128 rows x 128 B
constexpr uint32_t kKOff = kQOff + 2 * 128 * 128;   // 2 x 64 rows x 128 B
constexpr uint32_t kVOff = kKOff + 2 * 64 * 128;    // 1 x 128 rows x 128 B (V^T)
constexpr uint32_t kPOff = kVOff + 128 * 128;       // 1 x 128 rows x 128 B
constexpr uint32_t kSzOff = kPOff + 128 * 128;      // 64 tokens x 4 floats
constexpr uint32_t kOkOff = kSzOff + kTcTok * 16;   // 64 token flags
constexpr uint32_t kBarOff = kOkOff + kTcTok * 4;   // 2 mbarriers
constexpr uint32_t kSlotOff = kBarOff + 16;         // TMEM base address
constexpr uint32_t kSvMaxOff = kSlotOff + 8;        // largest V scale of the tile (2 halves)
constexpr uint32_t kFixedBytes = kSlotOff + 16;

__host__ __device__ constexpr size_t tc_smem_bytes(int batch) {
  return 1024 + kFixedBytes + align128((batch + 1) * sizeof(int32_t));
}

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
  s.tiles = (s.C * a.group + kTcRows - 1) / kTcRows;
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
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float2 lds_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
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

// 16-bit pair (two consecutive tokens of one dim) for the transposed V tile.
__device__ __forceinline__ uint32_t lo_hi(uint32_t x, uint32_t y, bool hi) {
  return hi ? ((x >> 16) | (y & 0xFFFF0000u)) : ((x & 0xFFFFu) | (y << 16));
}

// Raw bytes of one 64-token context tile that this thread stages: K chunks
// (16 bytes of one token row each), V pieces (8 dims of 8 consecutive tokens),
// and, for threads < 64, the scale/zero words and validity of token tid.
template <int KV>
struct RawTile {
  static constexpr int kRow = KvTraits<KV>::kRowBytes;
  static constexpr int kKChunks = kTcTok * (kRow / 16) / kTcThreads;  // 4 / 2 / 8
  static constexpr int kVWords = kRow / 64;  // 32-bit words per token of an 8-dim piece: 2 / 1 / 4
  uint4 k[kKChunks];
  uint32_t v[8][kVWords];
  uint32_t ksz, vsz;
  bool ok;
};

// Global row (token t of the tile, kv head h) of a pool, or null when the
// token is past the context or its block id is outside the pool.
template <int KV>
__device__ __forceinline__ const uint8_t* tc_row(const ExtendArgs& a, const int32_t* bt,
                                                 const uint8_t* pool, int tt, int L, int h) {
  constexpr int kRow = KvTraits<KV>::kRowBytes;
  if (tt >= L) return nullptr;
  const int32_t blk = bt[tt / kBlock];
  if (blk < 0 || blk >= a.num_blocks) return nullptr;
  return pool + ((static_cast<int64_t>(blk) * kBlock + tt % kBlock) * a.kv_heads + h) * kRow;
}

template <int KV>
__device__ __forceinline__ void load_tile(const ExtendArgs& a, const int32_t* bt, int tok0, int L,
                                          int h, int tid, RawTile<KV>& r) {
  using R = RawTile<KV>;
  constexpr int kChunks = R::kRow / 16;
#pragma unroll
  for (int i = 0; i < R::kKChunks; ++i) {
    const int e = tid + kTcThreads * i;
    const uint8_t* src = tc_row<KV>(a, bt, a.k, tok0 + e / kChunks, L, h);
    r.k[i] = src ? __ldg(reinterpret_cast<const uint4*>(src) + e % kChunks)
                 : make_uint4(0u, 0u, 0u, 0u);
  }
  // V: tokens 8 tg .. 8 tg + 7 (one block: 8 divides 16), dims 8 dc .. 8 dc + 7
  const int tg = tid & 7, dc = tid >> 3;  // 8 token groups across lanes: no bank conflicts
  const int tv = tok0 + 8 * tg;
  const int32_t vblk = tv < L ? bt[tv / kBlock] : -1;
  const bool vok = vblk >= 0 && vblk < a.num_blocks;
  const uint8_t* vrow =
      a.v + ((static_cast<int64_t>(vok ? vblk : 0) * kBlock + tv % kBlock) * a.kv_heads + h) *
                R::kRow +
      dc * 4 * R::kVWords;
  const int64_t vstride = static_cast<int64_t>(a.kv_heads) * R::kRow;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const bool ok = vok && tv + t < L;
    const uint8_t* src = vrow + t * vstride;
    if constexpr (R::kVWords == 4) {
      const uint4 w = ok ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0u, 0u, 0u, 0u);
      r.v[t][0] = w.x; r.v[t][R::kVWords > 1 ? 1 : 0] = w.y;
      r.v[t][R::kVWords > 2 ? 2 : 0] = w.z; r.v[t][R::kVWords > 3 ? 3 : 0] = w.w;
    } else if constexpr (R::kVWords == 2) {
      const uint2 w = ok ? __ldg(reinterpret_cast<const uint2*>(src)) : make_uint2(0u, 0u);
      r.v[t][0] = w.x; r.v[t][R::kVWords > 1 ? 1 : 0] = w.y;
    } else {
      r.v[t][0] = ok ? __ldg(reinterpret_cast<const uint32_t*>(src)) : 0u;
    }
  }
  r.ok = false;
  r.ksz = r.vsz = 0u;
  if (tid < kTcTok) {
    const int tt = tok0 + tid;
    if (tt < L) {
      const int32_t blk = bt[tt / kBlock];
      r.ok = blk >= 0 && blk < a.num_blocks;
      if (r.ok && KvTraits<KV>::kQuant) {
        const int64_t i = (static_cast<int64_t>(blk) * a.kv_heads + h) * kBlock + tt % kBlock;
        r.ksz = __ldg(a.k_sz + i);
        r.vsz = __ldg(a.v_sz + i);
      }
      if (!r.ok) report(a.dev_err, KVQ_DEV_ERR_BLOCK_ID);
    }
  }
}

// The four 16-bit pairs (dims 0-1, 2-3, 4-5, 6-7) of one token's 8-dim piece.
template <int KV>
__device__ __forceinline__ void piece_pairs(const uint32_t (&w)[RawTile<KV>::kVWords],
                                            uint32_t (&p)[4]) {
  constexpr int kMid = KV == kI8 ? 128 : 8;
  if constexpr (KV == kF16) {
    p[0] = w[0]; p[1] = w[1]; p[2] = w[2]; p[3] = w[3];
  } else if constexpr (KV == kI8) {
#pragma unroll
    for (int q = 0; q < 4; ++q) p[q] = bytes_to_f16(w[q >> 1], (q & 1) ? 0x4342u : 0x4140u);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t byte = (w[0] >> (8 * q)) & 0xFF;
      p[q] = centred_pair<false>(byte & 0xF, byte >> 4, kMid);
    }
  }
}

// Registers -> shared memory: the K tile (K-major, Q's type), V transposed
// (fp16), per-token (S_k', Z_k', S_v, Z_v') with the softmax scale folded
// into the K pair, and validity flags. Returns (for the whole CTA) whether
// any token of the tile is missing.
template <int KV, bool QBF>
__device__ __forceinline__ void store_tile(const ExtendArgs& a, const RawTile<KV>& r,
                                           uint32_t base, int tid) {
  using R = RawTile<KV>;
  constexpr int kMid = KV == kI8 ? 128 : 8;
  constexpr int kChunks = R::kRow / 16;
  if (tid < kTcTok) {
    float Sk = a.sm_scale_log2, Zk = 0.f, Sv = 1.f, Zv = 0.f;
    if constexpr (KvTraits<KV>::kQuant) {
      const float s_k = half_lo(r.ksz), s_v = half_lo(r.vsz);
      Sk = s_k * a.sm_scale_log2;
      Zk = (half_hi(r.ksz) + kMid * s_k) * a.sm_scale_log2;
      Sv = s_v;
      Zv = half_hi(r.vsz) + kMid * s_v;
    }
    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(base + kSzOff + 16 * tid), "f"(Sk),
                 "f"(Zk), "f"(Sv), "f"(Zv)
                 : "memory");
    sts32(base + kOkOff + 4 * tid, r.ok ? 1u : 0u);
    float mx = Sv;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    if ((tid & 31) == 0) sts32(base + kSvMaxOff + 4 * (tid >> 5), __float_as_uint(mx));
  }
#pragma unroll
  for (int i = 0; i < R::kKChunks; ++i) {
    const int e = tid + kTcThreads * i;
    const int t = e / kChunks, ch = e % kChunks;
    const uint32_t x[4] = {r.k[i].x, r.k[i].y, r.k[i].z, r.k[i].w};
    if constexpr (KV == kF16) {
      sts128(base + kKOff + umma_kmajor_offset(kTcTok, t, 8 * ch), x[0], x[1], x[2], x[3]);
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
            v[q] = bytes_to_f16(word, (q & 1) ? 0x4342u : 0x4140u);
          }
        }
        sts128(base + kKOff + umma_kmajor_offset(kTcTok, t, 16 * ch + 8 * hf), v[0], v[1], v[2],
               v[3]);
      }
    } else {
#pragma unroll
      for (int qt = 0; qt < 4; ++qt) {
        uint32_t v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t byte = (x[qt] >> (8 * q)) & 0xFF;
          v[q] = centred_pair<QBF>(byte & 0xF, byte >> 4, kMid);
        }
        sts128(base + kKOff + umma_kmajor_offset(kTcTok, t, 32 * ch + 8 * qt), v[0], v[1], v[2],
               v[3]);
      }
    }
  }
  // V: 8 tokens x 8 dims -> 8 rows (dims) of 8 tokens, one 16-byte store each
  const int tg = tid & 7, dc = tid >> 3;  // 8 token groups across lanes: no bank conflicts
  uint32_t pr[8][4];
#pragma unroll
  for (int t = 0; t < 8; ++t) piece_pairs<KV>(r.v[t], pr[t]);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int tp = 0; tp < 4; ++tp) {
      lo[tp] = prmt(pr[2 * tp][q], pr[2 * tp + 1][q], 0x5410u);
      hi[tp] = prmt(pr[2 * tp][q], pr[2 * tp + 1][q], 0x7632u);
    }
    sts128(base + kVOff + umma_kmajor_offset(128, 8 * dc + 2 * q, 8 * tg), lo[0], lo[1], lo[2],
           lo[3]);
    sts128(base + kVOff + umma_kmajor_offset(128, 8 * dc + 2 * q + 1, 8 * tg), hi[0], hi[1],
           hi[2], hi[3]);
  }
}

// Bounded wait on an mbarrier phase by every thread, with one verdict for the
// whole CTA.
__device__ __forceinline__ bool cta_wait(uint32_t bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __syncthreads_and(ok ? 1 : 0) != 0;
}

template <int KV, bool QBF>
__global__ void __launch_bounds__(kTcThreads, 1)
    extend_tc_kernel(const __grid_constant__ ExtendArgs a) {
  extern __shared__ __align__(1024) unsigned char dsmem[];
  __shared__ int32_t warp_sum[kTcThreads / 32];
  constexpr bool kQuant = KvTraits<KV>::kQuant;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = (static_cast<uint32_t>(__cvta_generic_to_shared(dsmem)) + 1023u) & ~1023u;
  int32_t* ucum = reinterpret_cast<int32_t*>(dsmem + (base - static_cast<uint32_t>(
                                                          __cvta_generic_to_shared(dsmem))) +
                                             kFixedBytes);
  const uint32_t bar_s = base + kBarOff, bar_o = base + kBarOff + 8;

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
  if (tid == 0) {
    mbar_init(bar_s);
    mbar_init(bar_o);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(base + kSlotOff, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t tmem;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(base + kSlotOff));
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * warp) << 16);
  const int total = ucum[a.batch];
  __shared__ int unit_s;
  uint32_t ns = 0, no = 0;  // completed phases of bar_s and bar_o
  bool alive = true;
  uint32_t failed_bar = 0, failed_parity = 0;

  for (;;) {
    if (tid == 0) unit_s = atomicAdd(a.counter, 1);
    __syncthreads();
    const int u = unit_s;
    __syncthreads();
    if (u >= total) break;
    int lo = 0, hi = a.batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ucum[mid] <= u) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const TcReq s = tc_req(a, b);
    const int r = u - ucum[b];
    const int h = r % a.kv_heads;
    const int qt = s.tiles - 1 - r / a.kv_heads;  // longest tiles first
    const int row = qt * kTcRows + tid;
    const int qi = row / a.group;
    const int hq = h * a.group + row % a.group;
    const bool valid = qi < s.C;
    const int pos = s.L - s.C + qi;
    const int i_max = min(s.C - 1, (qt * kTcRows + kTcRows - 1) / a.group);
    const int n_tok = s.L - s.C + i_max + 1;  // context the tile attends
    const int ntiles = (n_tok + kTcTok - 1) / kTcTok;
    const int32_t* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks;

    // Q row of this thread into the K-major tile (zeros for a padding row)
    float qsum = 0.f;
    {
      const uint4* qp = reinterpret_cast<const uint4*>(
          static_cast<const uint16_t*>(a.q) +
          ((static_cast<int64_t>(s.q0) + qi) * a.q_heads + hq) * kHeadDim);
#pragma unroll 4
      for (int ch = 0; ch < 16; ++ch) {
        const uint4 w = valid ? qp[ch] : make_uint4(0u, 0u, 0u, 0u);
        sts128(base + kQOff + umma_kmajor_offset(kTcRows, tid, 8 * ch), w.x, w.y, w.z, w.w);
        if constexpr (kQuant) {
          qsum += lo_to_float<QBF>(w.x) + hi_to_float<QBF>(w.x) + lo_to_float<QBF>(w.y) +
                  hi_to_float<QBF>(w.y) + lo_to_float<QBF>(w.z) + hi_to_float<QBF>(w.z) +
                  lo_to_float<QBF>(w.w) + hi_to_float<QBF>(w.w);
        }
      }
    }
    float m = -INFINITY, l = 0.f, z = 0.f;

    RawTile<KV> raw;
    load_tile<KV>(a, bt, 0, s.L, h, tid, raw);
    for (int j = 0; j < ntiles && alive; ++j) {
      store_tile<KV, QBF>(a, raw, base, tid);
      // the tile's missing tokens (rare: block ids outside the pool)
      const bool holes = __syncthreads_or(tid < kTcTok && !raw.ok &&
                                          j * kTcTok + tid < s.L) != 0;
      if (j + 1 < ntiles) load_tile<KV>(a, bt, (j + 1) * kTcTok, s.L, h, tid, raw);
      fence_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t idesc_s = umma_idesc_f16(QBF, kTcRows, kTcTok);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          umma_f16(tmem, umma_desc_sw128(base + kQOff + (k >> 2) * (kTcRows * 128) + (k & 3) * 32,
                                         1024),
                   umma_desc_sw128(base + kKOff + (k >> 2) * (kTcTok * 128) + (k & 3) * 32, 1024),
                   idesc_s, k > 0);
        umma_commit(bar_s);
      }
      if (!cta_wait(bar_s, ns & 1u)) {
        alive = false;
        failed_bar = bar_s;
        failed_parity = ns & 1u;
        break;
      }
      ++ns;
      tc_fence_after();
      // this row's scores, scaled, masked, in the exp2 domain
      float sc[kTcTok];
      {
        float v[32];
        tmem_ld32(lane_base, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) sc[i] = v[i];
        tmem_ld32(lane_base + 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) sc[32 + i] = v[i];
      }
      // s = S_k' raw + Z_k' sum(q) (scale folded in); positions past the row's
      // own, and missing tokens, are masked
      float bm = -INFINITY;
      const bool diag = j * kTcTok + kTcTok - 1 > pos;
#pragma unroll
      for (int i = 0; i < kTcTok; ++i) {
        const float2 kz = lds_f2(base + kSzOff + 16 * i);
        float x = kz.x * sc[i] + kz.y * qsum;
        if (diag && j * kTcTok + i > pos) x = -INFINITY;
        sc[i] = x;
        bm = fmaxf(bm, x);
      }
      if (holes) {
        bm = -INFINITY;
#pragma unroll
        for (int i = 0; i < kTcTok; ++i) {
          if (lds_u32(base + kOkOff + 4 * i) == 0u) sc[i] = -INFINITY;
          bm = fmaxf(bm, sc[i]);
        }
      }
      // the reference maximum moves only when a score exceeds it by more than
      // tau (log2 units): p <= 2^tau then, and P' = p S_v stays within fp16
      // when the tile's largest V scale is at most 240 (else tau = 0: exact)
      const float sv_max = fmaxf(__uint_as_float(lds_u32(base + kSvMaxOff)),
                                 __uint_as_float(lds_u32(base + kSvMaxOff + 4)));
      const float tau = sv_max <= 240.f ? 8.f : 0.f;
      const float mn = (m == -INFINITY || bm > m + tau) ? fmaxf(m, bm) : m;
      const float al = (m == -INFINITY || mn == m) ? 1.f : ex2(m - mn);
      // rescale this warp's rows of O when some row's maximum moved
      if (j > 0 && __any_sync(kFull, al != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tmem_ld32(lane_base + 64 + 32 * c, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= al;
          tmem_st32(lane_base + 64 + 32 * c, v);
        }
      }
      l *= al;
      z *= al;
      m = mn;
      const float ref = m == -INFINITY ? 0.f : m;
      // P' = p S_v (quantized) or p, fp16, into this row of the P tile
#pragma unroll
      for (int c8 = 0; c8 < kTcTok / 8; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i0 = 8 * c8 + 2 * q;
          const float p0 = ex2(sc[i0] - ref), p1 = ex2(sc[i0 + 1] - ref);
          l += p0 + p1;
          float v0 = p0, v1 = p1;
          if constexpr (kQuant) {
            const float4 s0 = lds_f4(base + kSzOff + 16 * i0);
            const float4 s1 = lds_f4(base + kSzOff + 16 * i0 + 16);
            z += p0 * s0.w + p1 * s1.w;
            v0 = p0 * s0.z;
            v1 = p1 * s1.z;
          }
          w[q] = pack2<false>(v0, v1);
        }
        sts128(base + kPOff + umma_kmajor_offset(kTcRows, tid, 8 * c8), w[0], w[1], w[2], w[3]);
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t idesc_o = umma_idesc_f16(false, kTcRows, kHeadDim);
#pragma unroll
        for (int k = 0; k < kTcTok / 16; ++k)
          umma_f16(tmem + 64, umma_desc_sw128(base + kPOff + k * 32, 1024),
                   umma_desc_sw128(base + kVOff + k * 32, 1024), idesc_o, j > 0 || k > 0);
        umma_commit(bar_o);
      }
      if (!cta_wait(bar_o, no & 1u)) {
        alive = false;
        failed_bar = bar_o;
        failed_parity = no & 1u;
        break;
      }
      ++no;
      tc_fence_after();
    }
    if (!alive) break;
    // output row: (O + z) / l (every lane takes part in the TMEM reads)
    {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(
          static_cast<uint16_t*>(a.out) +
          ((static_cast<int64_t>(s.q0) + qi) * a.q_heads + hq) * kHeadDim);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(lane_base + 64 + 32 * c, v);
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack2<QBF>((v[8 * q + 2 * e] + z) * inv, (v[8 * q + 2 * e + 1] + z) * inv);
            dst[4 * c + q] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (!alive) {
    if (tid == 0) report(a.dev_err, KVQ_DEV_ERR_TIMEOUT);
    // the product still in flight: one more bounded wait before freeing TMEM
    mbar_wait(failed_bar, failed_parity);
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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
                             static_cast<int>(tc_smem_bytes(kMaxBatch)));
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
                           static_cast<int>(tc_smem_bytes(kMaxBatch))) != cudaSuccess ||
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

size_t extend_tc_smem_bytes(int batch) { return tc_smem_bytes(batch); }

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

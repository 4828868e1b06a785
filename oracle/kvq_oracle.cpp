// Oracle for the paged, quantized KV store and paged decode attention.
//
// TEST INFRASTRUCTURE ONLY. This file is a plain, slow, single-threaded CPU
// restatement of what the hot path computes. Only the tests, the smoke check
// and the benchmark's CPU-baseline leg load it. The product library never
// links, calls or reads it, and it shares no code, header, table or helper
// with the CUDA path.
//
// Sources (pages are cited by title and section):
//   * "pymllm Runtime Design", section "KV cache 与 prefix cache":
//     ReqToTokenPool maps (request slot, position) to a KV index; a free list
//     hands out integer KV slots; KVPool keeps per-layer K/V tensors and is
//     written by a store kernel (store_cache).
//   * LMDeploy article (devpress.csdn.net), §2.2 "分块 KV 缓存": the cache is
//     cut into fixed blocks of 16 tokens and each sequence keeps a logical
//     block table of physical block ids; the CacheEngine sketch there gives
//     the per-layer shape [num_blocks, block_size, num_kv_heads, head_dim].
//   * same article, §2.4 "KV Cache 在线量化": per-head, per-token asymmetric
//     INT8/INT4 quantization with min/max scale computed online, no
//     calibration (quant_policy 8 or 4).
//   * same article, §3.2 item 3 and §4.2: generation attention reads a
//     non-contiguous KV layout through indirect block pointers, in its own
//     decode kernel.
//
// Readings where the pages are silent (each is also listed in the design
// notes):
//   * scale = fp16(fp32(max - min) / (2^b - 1)); zero = fp16(min) is a float
//     offset (dequant = code * scale + zero), not an integer zero point.
//   * codes use the stored fp16 scale and zero: c = clamp(rne((x - Z) / S)).
//   * a row whose stored scale is 0 or not finite, or whose stored zero is
//     not finite, stores all-zero codes.
//   * a signed zero min or max is taken as +0 so the stored bits are unique.
//   * INT4: two codes per byte, the even index in the low nibble.
//   * scale/zero pairs are stored per (block, kv head, offset in block).
//   * q-head h reads kv head h / (Hq / Hkv).
//   * a request of length 0 produces an all-zero output row.
//   * attention is evaluated in fp64 on the exact values the stored
//     representation stands for (fp16/bf16 elements, or code * S + Z).
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fno-fast-math -shared -fPIC.
// The quantizer is IEEE fp32 (sub, div, round-half-even); -ffp-contract=off
// keeps the compiler from fusing any multiply-add.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// dtype tags, same numbers as the pages' quant_policy for the integer kinds
enum { ODT_F16 = 0, ODT_BF16 = 1, ODT_INT4 = 4, ODT_INT8 = 8 };

constexpr int kBlockSize = 16;  // tokens per block (LMDeploy article §2.2)

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// IEEE-754 binary16 and bfloat16, written from the format definitions.
// ---------------------------------------------------------------------------

// binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
float oracle_f16_to_f32(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1F;
  const int m = h & 0x3FF;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(m), -24);  // subnormal: m * 2^-24
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(1024 + m), e - 25);  // (1 + m/1024) 2^(e-15)
  }
  return static_cast<float>(sign ? -v : v);
}

// Nearest binary16 value, ties to the even fraction. The magnitude is
// divided by the spacing (quantum) of binary16 numbers at its exponent,
// rounded to an integer with nearbyint (the default rounding mode is
// round-half-even) and multiplied back. Everything here is exact in double.
uint16_t oracle_f32_to_f16(float f) {
  if (std::isnan(f)) return 0x7E00;
  const uint16_t sign = std::signbit(f) ? 0x8000 : 0;
  const double a = std::fabs(static_cast<double>(f));
  // Largest finite binary16 is 65504; halfway to the next power of two,
  // 65520, and above round to infinity.
  if (a >= 65520.0) return sign | 0x7C00;
  if (a == 0.0) return sign;
  int e2;
  std::frexp(a, &e2);                 // a = fr * 2^e2, fr in [0.5, 1)
  const int unbiased = e2 - 1;        // floor(log2 a)
  const int q_exp = (unbiased < -14) ? -24 : unbiased - 10;
  const double r = std::nearbyint(std::ldexp(a, -q_exp));  // a / quantum, RNE
  const double v = std::ldexp(r, q_exp);
  if (v == 0.0) return sign;
  if (v < std::ldexp(1.0, -14)) {     // subnormal result: code = v / 2^-24
    return sign | static_cast<uint16_t>(r);
  }
  int ev;
  const double fr = std::frexp(v, &ev);  // v = fr * 2^ev
  const int exp_field = ev - 1 + 15;
  const int frac = static_cast<int>(std::ldexp(fr, 11)) - 1024;  // (2 fr - 1) * 1024
  return sign | static_cast<uint16_t>(exp_field << 10) | static_cast<uint16_t>(frac);
}

// bfloat16 is the upper half of a binary32.
float oracle_bf16_to_f32(uint16_t b) {
  const uint32_t bits = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

static float load_elem(const uint16_t* p, int64_t i, int dtype) {
  return dtype == ODT_BF16 ? oracle_bf16_to_f32(p[i]) : oracle_f16_to_f32(p[i]);
}

// ---------------------------------------------------------------------------
// Quantizer: one (token, kv head) row of n values, K or V alike
// (LMDeploy article §2.4: per-head per-token asymmetric, online min/max).
// codes[i] receives one code per element (unpacked).
// ---------------------------------------------------------------------------
void oracle_quantize_row(const float* x, int n, int bits, uint8_t* codes,
                         uint16_t* scale_bits, uint16_t* zero_bits) {
  const int qmax = (1 << bits) - 1;
  float mn = x[0], mx = x[0];
  for (int i = 1; i < n; ++i) {
    if (x[i] < mn) mn = x[i];
    if (x[i] > mx) mx = x[i];
  }
  mn = mn + 0.0f;  // -0 becomes +0
  mx = mx + 0.0f;
  const float range = mx - mn;                         // fp32, round to nearest
  const float s32 = range / static_cast<float>(qmax);  // fp32 division
  *scale_bits = oracle_f32_to_f16(s32);
  *zero_bits = oracle_f32_to_f16(mn);
  const float S = oracle_f16_to_f32(*scale_bits);
  const float Z = oracle_f16_to_f32(*zero_bits);
  const bool degenerate = !(S > 0.0f) || std::isinf(S) || !std::isfinite(Z);
  for (int i = 0; i < n; ++i) {
    if (degenerate) {
      codes[i] = 0;
      continue;
    }
    const float d = x[i] - Z;            // fp32 subtraction
    const float t = d / S;               // fp32 division
    long c = std::lrint(t);              // round half to even (default mode)
    if (c < 0) c = 0;
    if (c > qmax) c = qmax;
    codes[i] = static_cast<uint8_t>(c);
  }
}

// Row-wise form of the quantizer: x [rows, n] fp32 -> codes [rows, n],
// scale and zero bits [rows].
void oracle_quantize_rows(const float* x, int64_t rows, int n, int bits, uint8_t* codes,
                          uint16_t* scale_bits, uint16_t* zero_bits) {
  for (int64_t r = 0; r < rows; ++r)
    oracle_quantize_row(x + r * n, n, bits, codes + r * n, scale_bits + r, zero_bits + r);
}

// Element-wise conversions over arrays.
void oracle_f32_to_f16_array(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(x[i]);
}
void oracle_f16_to_f32_array(const uint16_t* x, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f32(x[i]);
}

// Value a stored code stands for: c * S + Z, exact in double.
double oracle_dequant(int code, uint16_t scale_bits, uint16_t zero_bits) {
  const double S = oracle_f16_to_f32(scale_bits);
  const double Z = oracle_f16_to_f32(zero_bits);
  return static_cast<double>(code) * S + Z;
}

// ---------------------------------------------------------------------------
// Pool addressing. A pool holds K (or V) for num_blocks blocks of 16 slots;
// slot = block_id * 16 + offset ("kv index" of the ReqToTokenPool).
//   f16/bf16 : element (slot, h, d) at ((slot * Hkv + h) * D + d), 16-bit
//   int8     : byte    ((slot * Hkv + h) * D + d)
//   int4     : byte    ((slot * Hkv + h) * D/2 + d/2), low nibble = even d
//   scale/zero: pair   ((block * Hkv + h) * 16 + offset), two fp16 words
//               (scale first, then zero)
// ---------------------------------------------------------------------------
struct OraclePool {
  void* data;         // K or V elements / codes
  uint16_t* sz;       // scale/zero pairs (quantized kinds only)
  int64_t num_blocks;
  int kv_heads;
  int head_dim;
  int dtype;
};

static void pool_store_row(const OraclePool& P, int64_t slot, int h, const float* x,
                           const uint16_t* raw) {
  const int D = P.head_dim;
  const int64_t row = slot * P.kv_heads + h;
  if (P.dtype == ODT_F16 || P.dtype == ODT_BF16) {
    uint16_t* dst = static_cast<uint16_t*>(P.data) + row * D;
    for (int d = 0; d < D; ++d) dst[d] = raw[d];  // plain row copy
    return;
  }
  const int bits = P.dtype == ODT_INT8 ? 8 : 4;
  std::vector<uint8_t> codes(D);
  uint16_t sb, zb;
  oracle_quantize_row(x, D, bits, codes.data(), &sb, &zb);
  uint8_t* base = static_cast<uint8_t*>(P.data);
  if (bits == 8) {
    for (int d = 0; d < D; ++d) base[row * D + d] = codes[d];
  } else {
    for (int d = 0; d < D; d += 2)
      base[row * (D / 2) + d / 2] =
          static_cast<uint8_t>(codes[d] | (codes[d + 1] << 4));
  }
  const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
  const int64_t pair = (blk * P.kv_heads + h) * kBlockSize + off;
  P.sz[2 * pair + 0] = sb;
  P.sz[2 * pair + 1] = zb;
}

static double pool_load(const OraclePool& P, int64_t slot, int h, int d) {
  const int D = P.head_dim;
  const int64_t row = slot * P.kv_heads + h;
  if (P.dtype == ODT_F16 || P.dtype == ODT_BF16) {
    return load_elem(static_cast<const uint16_t*>(P.data), row * D + d, P.dtype);
  }
  const uint8_t* base = static_cast<const uint8_t*>(P.data);
  int code;
  if (P.dtype == ODT_INT8) {
    code = base[row * D + d];
  } else {
    const uint8_t byte = base[row * (D / 2) + d / 2];
    code = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
  }
  const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
  const int64_t pair = (blk * P.kv_heads + h) * kBlockSize + off;
  return oracle_dequant(code, P.sz[2 * pair + 0], P.sz[2 * pair + 1]);
}

// ---------------------------------------------------------------------------
// Store path ("pymllm Runtime Design", KVPool written by store_cache): write
// token t's K and V rows, for every kv head, into slot_mapping[t]. A negative
// slot skips the token. Returns the number of tokens whose slot is beyond the
// pool (those are skipped too).
// k_new, v_new: [num_tokens, Hkv, D] 16-bit elements of dtype in_dtype.
// ---------------------------------------------------------------------------
int64_t oracle_kv_store(void* k_pool, void* v_pool, uint16_t* k_sz, uint16_t* v_sz,
                        int64_t num_blocks, int kv_heads, int head_dim, int kv_dtype,
                        const uint16_t* k_new, const uint16_t* v_new, int in_dtype,
                        const int64_t* slot_mapping, int64_t num_tokens) {
  const OraclePool K{k_pool, k_sz, num_blocks, kv_heads, head_dim, kv_dtype};
  const OraclePool V{v_pool, v_sz, num_blocks, kv_heads, head_dim, kv_dtype};
  const int D = head_dim;
  std::vector<float> x(D);
  int64_t bad = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * kBlockSize) {
      ++bad;
      continue;
    }
    for (int h = 0; h < kv_heads; ++h) {
      const int64_t src = (t * kv_heads + h) * D;
      for (int d = 0; d < D; ++d) x[d] = load_elem(k_new, src + d, in_dtype);
      pool_store_row(K, slot, h, x.data(), k_new + src);
      for (int d = 0; d < D; ++d) x[d] = load_elem(v_new, src + d, in_dtype);
      pool_store_row(V, slot, h, x.data(), v_new + src);
    }
  }
  return bad;
}

// ---------------------------------------------------------------------------
// Block tables from ReqToTokenPool rows ("pymllm Runtime Design": the pool
// maps (request slot, position) to a kv index; LMDeploy article §2.2: each
// sequence keeps a table of physical block ids, block size 16).
//   block_tables[b][j] = req_to_token[r][16 j] / 16 for j < ceil(L_b / 16),
//   -1 for the remaining entries, where r = req_pool_indices[b].
// The rows must be block-contiguous: req_to_token[r][16 j + i] equals
// 16 * block_tables[b][j] + i for every position below L_b. Returns a bit
// mask: 1 = request slot out of range, 2 = length beyond the row or the
// table, 4 = negative kv index, 8 = row not block-contiguous.
// ---------------------------------------------------------------------------
int oracle_block_tables(const int32_t* req_to_token, int32_t num_req_slots,
                        int32_t max_context_len, const int32_t* req_pool_indices,
                        const int32_t* seq_lens, int32_t batch, int32_t max_blocks_per_seq,
                        int32_t* block_tables) {
  int err = 0;
  for (int b = 0; b < batch; ++b) {
    int32_t* bt = block_tables + static_cast<int64_t>(b) * max_blocks_per_seq;
    for (int j = 0; j < max_blocks_per_seq; ++j) bt[j] = -1;
    const int r = req_pool_indices[b];
    int L = seq_lens[b];
    if (r < 0 || r >= num_req_slots) {
      err |= 1;
      continue;
    }
    if (L < 0) L = 0;
    if (L > max_context_len || L > max_blocks_per_seq * kBlockSize) {
      err |= 2;
      L = std::min(max_context_len, max_blocks_per_seq * kBlockSize);
    }
    const int32_t* row = req_to_token + static_cast<int64_t>(r) * max_context_len;
    const int nblk = (L + kBlockSize - 1) / kBlockSize;
    for (int j = 0; j < nblk; ++j) {
      const int32_t first = row[j * kBlockSize];
      if (first < 0) {
        err |= 4;
        continue;
      }
      bt[j] = first / kBlockSize;
    }
    for (int p = 0; p < L; ++p) {
      const int32_t s = row[p];
      if (s < 0) {
        err |= 4;
        continue;
      }
      const int32_t blk = bt[p / kBlockSize];
      if (blk < 0 || s != blk * kBlockSize + p % kBlockSize) err |= 8;
    }
  }
  return err;
}

// ---------------------------------------------------------------------------
// Decode attention for one (request, q head) over the paged pool (LMDeploy
// article §3.2 item 3: KV read through indirect block pointers; §2.2 block
// tables). Definition, in fp64:
//   slot(t) = bt[t / 16] * 16 + t % 16, t < L
//   s_t = sm_scale * sum_d q[d] k_t[d]
//   p_t = exp(s_t - max s) / sum_u exp(s_u - max s)
//   out[d] = sum_t p_t v_t[d]
// probs (optional, length L) receives p_t. Returns -1 if a block id is
// outside the pool, else 0.
// ---------------------------------------------------------------------------
static int decode_one(const OraclePool& K, const OraclePool& V, const double* q,
                      const int32_t* bt, int L, int h_kv, double sm_scale, double* out,
                      double* probs) {
  const int D = K.head_dim;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (L <= 0) return 0;
  std::vector<double> s(L);
  std::vector<int64_t> slot(L);
  for (int t = 0; t < L; ++t) {
    const int32_t blk = bt[t / kBlockSize];
    if (blk < 0 || blk >= K.num_blocks) return -1;
    slot[t] = static_cast<int64_t>(blk) * kBlockSize + t % kBlockSize;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q[d] * pool_load(K, slot[t], h_kv, d);
    s[t] = sm_scale * dot;
  }
  double m = s[0];
  for (int t = 1; t < L; ++t) m = std::max(m, s[t]);
  double l = 0.0;
  for (int t = 0; t < L; ++t) {
    s[t] = std::exp(s[t] - m);
    l += s[t];
  }
  for (int t = 0; t < L; ++t) {
    const double p = s[t] / l;
    if (probs) probs[t] = p;
    for (int d = 0; d < D; ++d) out[d] += p * pool_load(V, slot[t], h_kv, d);
  }
  return 0;
}

// Single (request, q head) entry point, mainly for sampled checks.
// q: D 16-bit elements of q_dtype.
int oracle_decode_one(const void* k_pool, const void* v_pool, const uint16_t* k_sz,
                      const uint16_t* v_sz, int64_t num_blocks, int kv_heads, int head_dim,
                      int kv_dtype, const uint16_t* q, int q_dtype, const int32_t* bt_row,
                      int32_t seq_len, int32_t h_kv, double sm_scale, double* out,
                      double* probs) {
  const OraclePool K{const_cast<void*>(k_pool), const_cast<uint16_t*>(k_sz), num_blocks,
                     kv_heads, head_dim, kv_dtype};
  const OraclePool V{const_cast<void*>(v_pool), const_cast<uint16_t*>(v_sz), num_blocks,
                     kv_heads, head_dim, kv_dtype};
  std::vector<double> qd(head_dim);
  for (int d = 0; d < head_dim; ++d) qd[d] = load_elem(q, d, q_dtype);
  return decode_one(K, V, qd.data(), bt_row, seq_len, h_kv, sm_scale, out, probs);
}

// Whole batch: q [B, Hq, D], block_tables [B, max_blocks_per_seq],
// seq_lens [B] (the count includes the token just stored), out [B, Hq, D]
// fp64. q-head h uses kv head h / (Hq / Hkv). Returns 0, or -1 on a block id
// outside the pool, or -2 on a head count that does not divide.
int oracle_paged_decode(const void* k_pool, const void* v_pool, const uint16_t* k_sz,
                        const uint16_t* v_sz, int64_t num_blocks, int kv_heads, int head_dim,
                        int kv_dtype, const uint16_t* q, int q_dtype,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* seq_lens, int32_t batch, int32_t q_heads,
                        double sm_scale, double* out) {
  if (q_heads % kv_heads != 0) return -2;
  const int group = q_heads / kv_heads;
  for (int b = 0; b < batch; ++b) {
    for (int h = 0; h < q_heads; ++h) {
      const int64_t row = static_cast<int64_t>(b) * q_heads + h;
      const int rc = oracle_decode_one(
          k_pool, v_pool, k_sz, v_sz, num_blocks, kv_heads, head_dim, kv_dtype,
          q + row * head_dim, q_dtype,
          block_tables + static_cast<int64_t>(b) * max_blocks_per_seq, seq_lens[b],
          h / group, sm_scale, out + row * head_dim, nullptr);
      if (rc != 0) return rc;
    }
  }
  return 0;
}

// Extend (chunked prefill) attention: "pymllm Runtime Design", forward stage
// (an extend / prefill batch writes its prompt tokens to the KV cache and
// attends over them); LMDeploy article §2.3 "动态拆分与融合" (a prefill longer
// than the 4096-token threshold is split into chunks prefilled in turn). Request b has kv_lens[b] tokens in the pool, the last
// C_b = qo_indptr[b + 1] - qo_indptr[b] of them being the chunk whose
// queries are q rows qo_indptr[b] .. qo_indptr[b + 1] - 1. Chunk query i sits
// at position kv_lens[b] - C_b + i and attends positions 0 .. that position
// (causal): the plain paged attention of that row with seq_len = position + 1.
// q, out: [total_q, Hq, D]. Returns 0, or the first nonzero code of
// decode_one, or -3 on a chunk longer than its request.
int oracle_paged_extend(const void* k_pool, const void* v_pool, const uint16_t* k_sz,
                        const uint16_t* v_sz, int64_t num_blocks, int kv_heads, int head_dim,
                        int kv_dtype, const uint16_t* q, int q_dtype, const int32_t* qo_indptr,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* kv_lens, int32_t batch, int32_t q_heads, double sm_scale,
                        double* out) {
  if (q_heads % kv_heads != 0) return -2;
  const int group = q_heads / kv_heads;
  for (int b = 0; b < batch; ++b) {
    const int32_t c = qo_indptr[b + 1] - qo_indptr[b];
    if (c > kv_lens[b]) return -3;
    for (int32_t i = 0; i < c; ++i) {
      const int32_t pos = kv_lens[b] - c + i;
      const int64_t r = qo_indptr[b] + i;
      for (int h = 0; h < q_heads; ++h) {
        const int64_t row = r * q_heads + h;
        const int rc = oracle_decode_one(
            k_pool, v_pool, k_sz, v_sz, num_blocks, kv_heads, head_dim, kv_dtype,
            q + row * head_dim, q_dtype,
            block_tables + static_cast<int64_t>(b) * max_blocks_per_seq, pos + 1, h / group,
            sm_scale, out + row * head_dim, nullptr);
        if (rc != 0) return rc;
      }
    }
  }
  return 0;
}

// Block copy / swap (LMDeploy article §4.4 "Block Manager 与缓存交换": a
// swap map {dst: src} moves whole blocks between the GPU and CPU caches, K
// and V alike). For i = 0 .. n-1 in order, block src_ids[i] of the source
// pool is copied to block dst_ids[i] of the destination pool: its 16 rows of
// K and of V for every kv head and, for quantized kinds, its (scale, zero)
// pairs. Both pools have the same kind, kv heads and head_dim. A pair with an
// id outside its pool is skipped and counted; the count is returned.
int64_t oracle_copy_blocks(const void* src_k, const void* src_v, const uint16_t* src_k_sz,
                           const uint16_t* src_v_sz, int64_t src_blocks, void* dst_k,
                           void* dst_v, uint16_t* dst_k_sz, uint16_t* dst_v_sz,
                           int64_t dst_blocks, int kv_heads, int head_dim, int kv_dtype,
                           const int32_t* src_ids, const int32_t* dst_ids, int64_t n) {
  const int64_t row_bytes = kv_dtype == 4 ? head_dim / 2 : (kv_dtype == 8 ? head_dim : 2 * head_dim);
  const int64_t tile = 16 * kv_heads * row_bytes;  // bytes of one block of K (or V)
  const int64_t pairs = static_cast<int64_t>(kv_heads) * 16 * 2;  // fp16 words of scale/zero
  const bool quant = kv_dtype == 4 || kv_dtype == 8;
  int64_t skipped = 0;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t s = src_ids[i], d = dst_ids[i];
    if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
      ++skipped;
      continue;
    }
    std::memcpy(static_cast<uint8_t*>(dst_k) + d * tile,
                static_cast<const uint8_t*>(src_k) + s * tile, tile);
    std::memcpy(static_cast<uint8_t*>(dst_v) + d * tile,
                static_cast<const uint8_t*>(src_v) + s * tile, tile);
    if (quant) {
      std::memcpy(dst_k_sz + d * pairs, src_k_sz + s * pairs, pairs * sizeof(uint16_t));
      std::memcpy(dst_v_sz + d * pairs, src_v_sz + s * pairs, pairs * sizeof(uint16_t));
    }
  }
  return skipped;
}

}  // extern "C"

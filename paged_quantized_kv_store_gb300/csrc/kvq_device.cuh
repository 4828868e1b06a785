// Device helpers shared by the libkvq kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kvq.h"
#include "kvq_internal.h"

namespace kvq {

// element kinds as template tags
enum Kind : int { kF16 = KVQ_F16, kBF16 = KVQ_BF16, kI4 = KVQ_INT4, kI8 = KVQ_INT8 };

template <int KV>
struct KvTraits;
template <>
struct KvTraits<kF16> {
  static constexpr int kRowBytes = 2 * kHeadDim;
  static constexpr bool kQuant = false;
};
template <>
struct KvTraits<kBF16> {
  static constexpr int kRowBytes = 2 * kHeadDim;
  static constexpr bool kQuant = false;
};
template <>
struct KvTraits<kI8> {
  static constexpr int kRowBytes = kHeadDim;
  static constexpr bool kQuant = true;
};
template <>
struct KvTraits<kI4> {
  static constexpr int kRowBytes = kHeadDim / 2;
  static constexpr bool kQuant = true;
};

// ---- loads ------------------------------------------------------------------

// Streaming 16-byte load through the non-coherent path, not kept in L1.
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ldg_stream8(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(r.x), "=r"(r.y)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ldg_nc32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// ---- packed 16-bit arithmetic -------------------------------------------------

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// (a & b) | c in one LOP3
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Codes enter the tensor cores as exact 16-bit floats a + c, made by writing
// the code into the mantissa of a constant whose exponent makes one mantissa
// step worth 1; the caller removes a outside the products (with the zero).
//   INT4 as fp16: 16 + c   (0x4C00 with the code in mantissa bits 6..9)
//   INT4 as bf16: 128 + c  (0x4300 with the code in mantissa bits 0..3)
//   INT8 as fp16: 1024 + c (0x6400 with the code in mantissa bits 0..7), and
//                 c - 128 after one packed subtract
//   INT8 as bf16: c - 128  (through fp32)
// The P.V product takes INT8 codes centred exactly: with a large offset its
// accumulator would carry a constant that grows over a long context, and its
// fp32 accumulation error with it. The Q.K product starts afresh for every
// block, so the offset costs nothing there.

// Nibble s (0..3) of each 16-bit half of w as a pair a + c. s is a constant
// after unrolling, so the shift folds into one instruction or none.
template <bool BF>
__device__ __forceinline__ uint32_t nibbles_to_pair(uint32_t w, int s) {
  if constexpr (BF) {
    return and_or(w >> (4 * s), 0x000F000Fu, 0x43004300u);
  } else {
    const uint32_t x = s == 0 ? (w << 6) : s == 1 ? (w << 2) : s == 2 ? (w >> 2) : (w >> 6);
    return and_or(x, 0x03C003C0u, 0x4C004C00u);
  }
}

// Two bytes of w (selected by sel, producing [b_lo, 0x64, b_hi, 0x64]) as the
// fp16 pair 1024 + c.
__device__ __forceinline__ uint32_t bytes_to_f16_offset(uint32_t w, uint32_t sel) {
  return prmt(w, 0x64646464u, sel);
}

// Two bytes of w (selected by sel, producing [b_lo, 0x64, b_hi, 0x64], the
// fp16 pair 1024 + c) as the exact fp16 pair c - 128: one packed subtract of
// 1152 (0x6480).
__device__ __forceinline__ uint32_t bytes_to_f16(uint32_t w, uint32_t sel) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(prmt(w, 0x64646464u, sel)), "r"(0x64806480u));
  return r;
}

// Two bytes of w (byte indices i0 low, i1 high) as the exact bf16 pair
// c - 128: the bytes go through fp32 (2^23 + c, minus 2^23 + 128) and a
// paired round-to-nearest conversion, exact since |c - 128| <= 128.
__device__ __forceinline__ uint32_t bytes_to_bf16_pair(uint32_t w, int i0, int i1) {
  const float f0 = __uint_as_float(0x4B000000u | ((w >> (8 * i0)) & 0xFFu)) - 8388736.0f;
  const float f1 = __uint_as_float(0x4B000000u | ((w >> (8 * i1)) & 0xFFu)) - 8388736.0f;
  __nv_bfloat162 p = __floats2bfloat162_rn(f0, f1);
  return *reinterpret_cast<uint32_t*>(&p);
}

// ---- tensor-core fragments ----------------------------------------------------

// D = A(16x16, row) * B(16x8, col) + D, fp32 accumulate.
template <bool BF>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  if constexpr (BF) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
}

// Transpose an 8x8 matrix of 16-bit values held one row-pair per thread.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

template <bool BF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
  } else {
    __half2 p = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
  }
}

template <bool BF>
__device__ __forceinline__ float lo_to_float(uint32_t v) {
  if constexpr (BF) {
    return __uint_as_float(v << 16);
  } else {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
  }
}

template <bool BF>
__device__ __forceinline__ float hi_to_float(uint32_t v) {
  if constexpr (BF) {
    return __uint_as_float(v & 0xFFFF0000u);
  } else {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
  }
}

__device__ __forceinline__ void report(int32_t* dev_err, uint32_t bits) {
  if (dev_err != nullptr && bits != 0u) atomicOr(reinterpret_cast<unsigned int*>(dev_err), bits);
}

}  // namespace kvq

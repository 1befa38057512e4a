// Device-side helpers shared by the kvq kernels (sm_103a).
//
// Everything that decides a stored code uses the IEEE round-to-nearest
// intrinsics (__fmul_rn, __fadd_rn, ...), which the compiler never contracts
// into FMAs, so the write path is bit-reproducible against a plain float32
// restatement of its formulas.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace kvq {

enum Fmt : int { INT8 = 1, E4M3 = 2, E5M2 = 3, INT4A = 4, UINT8A = 5, BF16 = 6 };

__host__ __device__ constexpr bool is_asym(int f) { return f == INT4A || f == UINT8A; }
__host__ __device__ constexpr int row_bytes(int f, int d) {
  return f == INT4A ? d / 2 : f == BF16 ? 2 * d : d;
}
__host__ __device__ constexpr int asym_levels(int f) { return f == INT4A ? 15 : 255; }

// Per-device error word (bits KVQ_DEVERR_*), one per translation unit (no
// relocatable device code); the host ORs them all (kvq_get_device_error).
static __device__ unsigned int g_error_word = 0;
__device__ __forceinline__ void raise_error(unsigned bits) { atomicOr(&g_error_word, bits); }

// Host side: read and clear this translation unit's error word.
#define KVQ_ERROR_ACCESSOR(NAME)                                                   \
  cudaError_t NAME(unsigned* bits) {                                               \
    unsigned v = 0, zero = 0;                                                      \
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v));             \
    if (e != cudaSuccess) return e;                                                \
    *bits |= v;                                                                    \
    return v ? cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) : cudaSuccess; \
  }

// ---------------------------------------------------------------------------
// memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

template <int BYTES>
__device__ __forceinline__ void cp_async(uint32_t dst, const void* src) {
  if constexpr (BYTES == 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  } else {
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(dst), "l"(src), "n"(BYTES)
                 : "memory");
  }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// bit manipulation
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  return __byte_perm(a, b, sel);
}
// (a & b) | c
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// two E4M3 bytes (low 16 bits) -> f16x2, element order kept (exact)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t lo16) {
  uint32_t d;
  uint16_t s = static_cast<uint16_t>(lo16);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(s));
  return d;
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// D = A(16x16, f16) * B(16x8, f16) + C, fp32 accumulate
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// float -> code conversions (write path)
// ---------------------------------------------------------------------------
// two floats -> two fp8 codes (round to nearest even, saturate to max finite);
// returns lo byte = code(lo), next byte = code(hi)
template <int F>
__device__ __forceinline__ uint32_t f32x2_to_fp8x2(float lo, float hi) {
  uint16_t d;
  if constexpr (F == E4M3) {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  }
  return d;
}

// ---------------------------------------------------------------------------
// Packed float32 pairs (sm_100 and later): one instruction computes two IEEE
// float32 operations, each rounded to nearest exactly as the scalar operation
// (no flush of subnormals), so they stand in for __fadd_rn / __fsub_rn /
// __fmul_rn / __fmaf_rn pairwise without changing any result.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{ .reg .b64 pa, pb, pd; mov.b64 pa, {%2, %3}; mov.b64 pb, {%4, %5};"
      " add.rn.f32x2 pd, pa, pb; mov.b64 {%0, %1}, pd; }"
      : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{ .reg .b64 pa, pb, pd; mov.b64 pa, {%2, %3}; mov.b64 pb, {%4, %5};"
      " sub.rn.f32x2 pd, pa, pb; mov.b64 {%0, %1}, pd; }"
      : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{ .reg .b64 pa, pb, pd; mov.b64 pa, {%2, %3}; mov.b64 pb, {%4, %5};"
      " mul.rn.f32x2 pd, pa, pb; mov.b64 {%0, %1}, pd; }"
      : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// d = a * b + c, one rounding per lane
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
  asm("{ .reg .b64 pa, pb, pc, pd; mov.b64 pa, {%2, %3}; mov.b64 pb, {%4, %5};"
      " mov.b64 pc, {%6, %7}; fma.rn.f32x2 pd, pa, pb, pc; mov.b64 {%0, %1}, pd; }"
      : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// (c << 8) | (sat4(a) << 4) | sat4(b), sat4 = clamp to [0, 15]
__device__ __forceinline__ uint32_t pack_sat_u4(int a, int b, uint32_t c) {
  uint32_t d;
  asm("cvt.pack.sat.u4.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// (c << 16) | (sat8(a) << 8) | sat8(b), sat8 = clamp to [0, 255]
__device__ __forceinline__ uint32_t pack_sat_u8(int a, int b, uint32_t c) {
  uint32_t d;
  asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// Walsh-Hadamard butterfly across a group of lanes.  Each lane holds E
// consecutive elements of a row of length E * LANES (LANES consecutive lanes,
// group-aligned).  Stages h = 1, 2, ..., in increasing order; every output is
// one IEEE add / subtract of (lower-index, higher-index) elements, so the
// result does not depend on the thread mapping.
// ---------------------------------------------------------------------------
template <int E, int LANES>
__device__ __forceinline__ void fwht_lanes(float (&v)[E], int sub) {
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if ((i & h) == 0) {
        float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int lo = 1; lo < LANES; lo <<= 1) {
    const bool upper = (sub & lo) != 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      float other = __shfl_xor_sync(0xffffffffu, v[i], lo);
      v[i] = upper ? __fsub_rn(other, v[i]) : __fadd_rn(v[i], other);
    }
  }
}

}  // namespace kvq

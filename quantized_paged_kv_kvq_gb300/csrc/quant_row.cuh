// Quantization of one cache row (token, kv-head) held by a group of D/8 lanes,
// 8 consecutive elements each: shared by the cache-write kernel and the
// decode kernel's new-token append.
//
// Symmetric codes follow the INT8 per-layer-scale cache of the
// "vllm-int8-kv-cache-for-ampere-sm86" summary and the FP8 e4m3 / e5m2 cache
// with a kv_scale of vLLM PR #4893 (item 1); asymmetric codes follow vLLM issue
// #4025 'Support for 4-bit KV Cache in paged-attention op', section 'methods'
// (fp16 scale and zero point per row, int4 packed two to a byte); KVarN's
// variance normalisation and Hadamard rotation come first for the KVarN cache
// ('KVarN : le backend natif pour la quantification du cache KV', section
// 'Contexte Technique').
#pragma once

#include "kvq_device.cuh"

namespace kvq {

template <int D>
struct RowGeom {
  static constexpr int LPR = D / 8;     // lanes per row
  static constexpr int RPI = 32 / LPR;  // rows per warp-wide 16-byte load
};

__device__ __forceinline__ void unpack8(const uint4& r, float (&x)[8]) {
  x[0] = bf16_lo(r.x); x[1] = bf16_hi(r.x);
  x[2] = bf16_lo(r.y); x[3] = bf16_hi(r.y);
  x[4] = bf16_lo(r.z); x[5] = bf16_hi(r.z);
  x[6] = bf16_lo(r.w); x[7] = bf16_hi(r.w);
}

// Fixed-order float32 sum of a row: 8 values per lane left to right, then
// lane groups combined with xor offsets LPR/2, ..., 1.
template <int LPR>
__device__ __forceinline__ float tree_sum8(const float (&x)[8]) {
  float s = x[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) s = __fadd_rn(s, x[i]);
#pragma unroll
  for (int o = LPR / 2; o >= 1; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
  return s;
}

// KVarN pre-quantization of one row, in place: x <- cR * H (d . x / sigma16).
template <int D>
__device__ __forceinline__ __half varnorm_rotate(float (&x)[8], int sub, uint32_t sign_bits,
                                                 float cR) {
  constexpr int LPR = RowGeom<D>::LPR;
  const float inv_d = 1.0f / D;  // exact (power of two)
  const float mean = __fmul_rn(tree_sum8<LPR>(x), inv_d);
  float sq[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float dv = __fsub_rn(x[i], mean);
    sq[i] = __fmul_rn(dv, dv);
  }
  const float var = __fmul_rn(tree_sum8<LPR>(sq), inv_d);
  __half s16 = __float2half_rn(__fsqrt_rn(var));
  if (__half2float(s16) == 0.0f) s16 = __float2half_rn(1.0f);
  const float inv_sigma = __frcp_rn(__half2float(s16));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float y = __fmul_rn(x[i], inv_sigma);
    x[i] = ((sign_bits >> i) & 1u) ? -y : y;
  }
  fwht_lanes<8, LPR>(x, sub);
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(x[i], cR);
  return s16;
}

// Quantize one row held by the lane group and store codes (+ meta).
template <int D, int F, bool KVARN>
__device__ __forceinline__ void quantize_store(float (&x)[8], bool active, int h, int sub,
                                               size_t row, uint8_t* __restrict__ cache,
                                               __half* __restrict__ meta, float inv, int64_t blk,
                                               int off, int Hkv, int bs, uint32_t sign_bits,
                                               float cR) {
  constexpr int LPR = RowGeom<D>::LPR;
  if constexpr (F == BF16) {  // the values themselves (x holds bf16 values exactly)
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = (__float_as_uint(x[2 * i]) >> 16) | (__float_as_uint(x[2 * i + 1]) & 0xFFFF0000u);
    if (active)
      *reinterpret_cast<uint4*>(cache + row * (2 * D) + sub * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  } else if constexpr (F == INT8) {
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int c = __float2int_rn(__fmul_rn(x[i], inv));
      c = max(-128, min(127, c));
      w[i >> 2] |= (static_cast<uint32_t>(c) & 0xFFu) << (8 * (i & 3));
    }
    if (active) *reinterpret_cast<uint2*>(cache + row * D + sub * 8) = make_uint2(w[0], w[1]);
  } else if constexpr (F == E4M3 || F == E5M2) {
    uint32_t w[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t lo = f32x2_to_fp8x2<F>(__fmul_rn(x[4 * j], inv), __fmul_rn(x[4 * j + 1], inv));
      const uint32_t hi =
          f32x2_to_fp8x2<F>(__fmul_rn(x[4 * j + 2], inv), __fmul_rn(x[4 * j + 3], inv));
      w[j] = lo | (hi << 16);
    }
    if (active) *reinterpret_cast<uint2*>(cache + row * D + sub * 8) = make_uint2(w[0], w[1]);
  } else {
    static_assert(is_asym(F), "format");
    __half sig16 = __float2half_rn(1.0f);
    if constexpr (KVARN) sig16 = varnorm_rotate<D>(x, sub, sign_bits, cR);
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      mn = fminf(mn, x[i]);
      mx = fmaxf(mx, x[i]);
    }
#pragma unroll
    for (int o = LPR / 2; o >= 1; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    constexpr int L = asym_levels(F);
    __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(L)));
    if (__half2float(s16) == 0.0f) s16 = __float2half_rn(1.0f);
    const __half z16 = __float2half_rn(mn);
    const float zf = __half2float(z16);
    const float inv_s = __frcp_rn(__half2float(s16));
    int c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[i] = __float2int_rn(__fmul_rn(__fsub_rn(x[i], zf), inv_s));
      c[i] = max(0, min(L, c[i]));
    }
    if (active) {
      if constexpr (F == INT4A) {
        uint32_t w = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) w |= static_cast<uint32_t>(c[i]) << (4 * i);
        *reinterpret_cast<uint32_t*>(cache + row * (D / 2) + sub * 4) = w;
      } else {
        uint32_t w0 = 0, w1 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          w0 |= static_cast<uint32_t>(c[i]) << (8 * i);
          w1 |= static_cast<uint32_t>(c[i + 4]) << (8 * i);
        }
        *reinterpret_cast<uint2*>(cache + row * D + sub * 8) = make_uint2(w0, w1);
      }
      if (sub == 0) {
        constexpr int NF = KVARN ? 3 : 2;
        __half* m = meta + ((static_cast<size_t>(blk) * Hkv + h) * NF) * bs + off;
        m[0] = s16;
        m[bs] = z16;
        if constexpr (KVARN) m[2 * bs] = sig16;
      }
    }
  }
}

}  // namespace kvq

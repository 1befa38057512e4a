// Quantize-and-scatter into the paged cache for the asymmetric formats (INT4 /
// UINT8 codes with an fp16 scale and zero point per (token, kv-head) row), with
// or without KVarN's variance normalisation and Hadamard rotation.
//
// vLLM issue #4025 'Support for 4-bit KV Cache in paged-attention op',
// section 'methods', items 1-2 (scale and zero point, int4 storage in the
// paged-cache write); the KVarN article ('KVarN : le backend natif pour la
// quantification du cache KV', section 'Contexte Technique') for the
// normalisation and rotation before asymmetric codes.
#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "quant_row.cuh"

namespace kvq {

KVQ_ERROR_ACCESSOR(take_error_bits_write_asym)

namespace {

constexpr int kWriteWarps = 8;

// ---------------------------------------------------------------------------
// Asymmetric formats (INT4 / UINT8 with a per-row scale and zero point), with
// or without the KVarN normalisation + rotation.  Their per-row work (sigma,
// the butterfly, min / max, the fp16 scale) is ALU-heavy, so a row is held by
// only D/32 lanes, 32 consecutive elements each: five of the seven butterfly
// stages and most of each reduction stay in registers.  The arithmetic is that
// of the narrow row code (quantize_store, 8 elements per lane), in the same
// order (fixed sum tree over groups of 8, butterfly stages h = 1, 2, ...,
// D/2), so the codes are the same.
// ---------------------------------------------------------------------------
template <int D>
struct WideGeom {
  static constexpr int LPR = D / 32;    // lanes per row
  static constexpr int RPW = 32 / LPR;  // rows per warp pass
  static constexpr int GPL = 4;         // groups of 8 per lane
};

// Fixed-order float32 sum of a row: each group of 8 left to right, then every
// group sum s_j becomes s_j + s_(j xor o) for o = D/16, ..., 1 (group j of the
// row is group j % 4 of lane j / 4 of the row's lanes).
template <int D>
__device__ __forceinline__ float tree_sum32(const float (&x)[32]) {
  constexpr int LPR = WideGeom<D>::LPR;
  float g[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float t = x[8 * j];
#pragma unroll
    for (int i = 1; i < 8; ++i) t = __fadd_rn(t, x[8 * j + i]);
    g[j] = t;
  }
  // offsets D/16 .. 4 cross lanes (lane offset o / 4), then 2 and 1 are local
#pragma unroll
  for (int lo = LPR / 2; lo >= 1; lo >>= 1) {
#pragma unroll
    for (int j = 0; j < 4; ++j) g[j] = __fadd_rn(g[j], __shfl_xor_sync(0xffffffffu, g[j], lo));
  }
  const float a0 = __fadd_rn(g[0], g[2]), a1 = __fadd_rn(g[1], g[3]);
  return __fadd_rn(a0, a1);
}

// Butterfly stages h = 1 .. 16 in registers, then h = 32, 64 across the lanes
// of the row (lane bit b set: other - v, else v + other; one fma with a +-1
// factor is that same single rounding).
template <int D>
__device__ __forceinline__ void fwht32(float (&v)[32], int sub) {
  constexpr int LPR = WideGeom<D>::LPR;
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & h) == 0) {
        const float x = v[i], y = v[i + h];
        v[i] = __fadd_rn(x, y);
        v[i + h] = __fsub_rn(x, y);
      }
    }
  }
#pragma unroll
  for (int lo = 1; lo < LPR; lo <<= 1) {
    const float sgn = (sub & lo) ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float other = __shfl_xor_sync(0xffffffffu, v[i], lo);
      v[i] = __fmaf_rn(sgn, v[i], other);
    }
  }
}

// One row (token t, kv-head h) of an asymmetric format, 32 elements per lane.
template <int D, int F, bool KVARN>
__device__ __forceinline__ void quantize_row_wide(float (&x)[32], int sub, bool active,
                                                  uint8_t* __restrict__ cache,
                                                  __half* __restrict__ meta, size_t row,
                                                  int64_t blk, int off, int h, int Hkv, int bs,
                                                  uint32_t sign_bits, float cR) {
  constexpr int LPR = WideGeom<D>::LPR;
  __half sig16 = __float2half_rn(1.0f);
  if constexpr (KVARN) {
    const float inv_d = 1.0f / D;  // exact (power of two)
    const float mean = __fmul_rn(tree_sum32<D>(x), inv_d);
    float sq[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float dv = __fsub_rn(x[i], mean);
      sq[i] = __fmul_rn(dv, dv);
    }
    const float var = __fmul_rn(tree_sum32<D>(sq), inv_d);
    sig16 = __float2half_rn(__fsqrt_rn(var));
    if (__half2float(sig16) == 0.0f) sig16 = __float2half_rn(1.0f);
    const float inv_sigma = __frcp_rn(__half2float(sig16));
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float y = __fmul_rn(x[i], inv_sigma);
      // d_i = -1: flip the sign bit (the exact negation, as one logic op)
      x[i] = __uint_as_float(__float_as_uint(y) ^ ((sign_bits << (31 - i)) & 0x80000000u));
    }
    fwht32<D>(x, sub);
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __fmul_rn(x[i], cR);
  }
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int i = 1; i < 32; ++i) {
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
  // code = clamp(rne((x - z) * inv_s), 0, L): a saturating round-to-nearest-even
  // conversion to u8 is rne then clamp to [0, 255]
  uint32_t c[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float v = __fmul_rn(__fsub_rn(x[i], zf), inv_s);
    uint32_t q;
    asm("cvt.rni.sat.u8.f32 %0, %1;" : "=r"(q) : "f"(v));
    c[i] = L == 255 ? q : min(q, static_cast<uint32_t>(L));
  }
  if (active) {
    if constexpr (F == INT4A) {
      uint4 w;
      uint32_t ww[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t t = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) t |= c[8 * k + i] << (4 * i);
        ww[k] = t;
      }
      w.x = ww[0]; w.y = ww[1]; w.z = ww[2]; w.w = ww[3];
      *reinterpret_cast<uint4*>(cache + row * (D / 2) + sub * 16) = w;
    } else {
      uint32_t ww[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        ww[k] = c[4 * k] | (c[4 * k + 1] << 8) | (c[4 * k + 2] << 16) | (c[4 * k + 3] << 24);
      uint4* dst = reinterpret_cast<uint4*>(cache + row * D + sub * 32);
      dst[0] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
      dst[1] = make_uint4(ww[4], ww[5], ww[6], ww[7]);
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

template <int D, int KF, int VF, bool KVARN>
__global__ void __launch_bounds__(kWriteWarps * 32)
    write_asym_kernel(WriteArgs a) {
  constexpr int LPR = WideGeom<D>::LPR;
  constexpr int RPW = WideGeom<D>::RPW;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWriteWarps + (threadIdx.x >> 5);
  if (t >= a.num_tokens) return;
  const int64_t slot = a.slot_mapping[t];
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(a.num_blocks) * a.block_size) {
    if (lane == 0) raise_error(1u);  // KVQ_DEVERR_SLOT_RANGE
    return;
  }
  const int64_t blk = slot >> a.block_shift;
  const int off = static_cast<int>(slot & (a.block_size - 1));
  const int sub = lane % LPR, grp = lane / LPR;
  const int Hkv = a.num_kv_heads;

  uint32_t sign_bits = 0;  // bit i: element sub*32 + i of the diagonal is -1
  if constexpr (KVARN) {
    if (a.signs != nullptr) {
      const uint4* sp = reinterpret_cast<const uint4*>(a.signs + sub * 32);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 sv = sp[q];
        const uint32_t w4[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int b = 0; b < 4; ++b)
            sign_bits |= ((w4[k] >> (8 * b + 7)) & 1u) << (16 * q + 4 * k + b);
      }
    }
  }

  const uint16_t* krow = a.key + t * a.key_stride;
  const uint16_t* vrow = a.value + t * a.value_stride;
  const size_t row0 = (static_cast<size_t>(blk) * a.block_size + off) * Hkv;
  // rows of the token: K heads 0..Hkv-1, then V heads; RPW rows per pass
  for (int r0 = 0; r0 < 2 * Hkv; r0 += RPW) {
    const int r = r0 + grp;
    const bool act = r < 2 * Hkv;
    const bool is_v = r >= Hkv;
    const int h = is_v ? r - Hkv : r;
    uint4 raw[4];
    const uint16_t* src = (is_v ? vrow : krow) + h * D + sub * 32;
#pragma unroll
    for (int q = 0; q < 4; ++q) raw[q] = act ? ldg_stream16(src + 8 * q) : make_uint4(0, 0, 0, 0);
    float x[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float e[8];
      unpack8(raw[q], e);
#pragma unroll
      for (int i = 0; i < 8; ++i) x[8 * q + i] = e[i];
    }
    if (__all_sync(0xffffffffu, !is_v || !act)) {
      quantize_row_wide<D, KF, KVARN>(x, sub, act, a.k_cache, a.k_meta, row0 + h, blk, off, h,
                                      Hkv, a.block_size, sign_bits, a.cR);
    } else if (__all_sync(0xffffffffu, is_v || !act)) {
      quantize_row_wide<D, VF, KVARN>(x, sub, act, a.v_cache, a.v_meta, row0 + h, blk, off, h,
                                      Hkv, a.block_size, sign_bits, a.cR);
    } else {  // a pass with K and V rows (fewer kv-heads than rows per pass)
      quantize_row_wide<D, KF, KVARN>(x, sub, act && !is_v, a.k_cache, a.k_meta, row0 + h, blk,
                                      off, h, Hkv, a.block_size, sign_bits, a.cR);
      if constexpr (KVARN) {  // the K pass rotated x in place: the V rows start again
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float e[8];
          unpack8(act ? ldg_stream16(src + 8 * q) : make_uint4(0, 0, 0, 0), e);
#pragma unroll
          for (int i = 0; i < 8; ++i) x[8 * q + i] = e[i];
        }
      }
      quantize_row_wide<D, VF, KVARN>(x, sub, act && is_v, a.v_cache, a.v_meta, row0 + h, blk,
                                      off, h, Hkv, a.block_size, sign_bits, a.cR);
    }
  }
}

template <int D, int KF, int VF, bool KVARN>
cudaError_t launch_asym_t(const WriteArgs& a, cudaStream_t st) {
  const int64_t blocks = (a.num_tokens + kWriteWarps - 1) / kWriteWarps;
  write_asym_kernel<D, KF, VF, KVARN><<<static_cast<unsigned>(blocks), kWriteWarps * 32, 0, st>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_asym_d(const WriteArgs& a, int kf, int vf, bool kvarn, cudaStream_t st) {
#define KVQ_W(KF_, VF_, KV_) \
  if (kf == KF_ && vf == VF_ && kvarn == KV_) return launch_asym_t<D, KF_, VF_, KV_>(a, st);
  KVQ_W(INT4A, INT4A, false)
  KVQ_W(INT4A, UINT8A, false)
  KVQ_W(UINT8A, INT4A, false)
  KVQ_W(UINT8A, UINT8A, false)
  KVQ_W(INT4A, INT4A, true)
  KVQ_W(INT4A, UINT8A, true)
  KVQ_W(UINT8A, INT4A, true)
  KVQ_W(UINT8A, UINT8A, true)
#undef KVQ_W
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_write_asym(const WriteArgs& a, int head_dim, int kf, int vf, bool kvarn,
                              cudaStream_t st) {
  if (head_dim == 64) return dispatch_asym_d<64>(a, kf, vf, kvarn, st);
  if (head_dim == 128) return dispatch_asym_d<128>(a, kf, vf, kvarn, st);
  return cudaErrorNotSupported;
}

}  // namespace kvq

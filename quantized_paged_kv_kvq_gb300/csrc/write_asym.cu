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
// Resident CTAs per SM each instance is compiled for (its register budget):
// the KVarN rows need more registers.
constexpr int ctas_per_sm(bool kvarn) { return kvarn ? 3 : 4; }

// ---------------------------------------------------------------------------
// Asymmetric formats (INT4 / UINT8 with a per-row scale and zero point), with
// or without the KVarN normalisation + rotation.  Their per-row work (sigma,
// the butterfly, min / max, the fp16 scale) is ALU-heavy, so a row is held by
// only D/32 lanes, 32 consecutive elements each: five of the seven butterfly
// stages and most of each reduction stay in registers.  The arithmetic is that
// of the narrow row code (quantize_store, 8 elements per lane), in the same
// order (fixed sum tree over groups of 8, butterfly stages h = 1, 2, ...,
// D/2), so the codes are the same.  Elementwise steps run on packed float32
// pairs, and codes are packed by saturating conversions, which cuts the
// instructions per element by about a third.  One warp per token; a pass
// quantizes RPW consecutive rows of the token (its K heads, then its V heads).
// ---------------------------------------------------------------------------
template <int D>
struct WideGeom {
  static constexpr int LPR = D / 32;    // lanes per row
  static constexpr int RPW = 32 / LPR;  // rows per warp pass
};

// Fixed-order float32 sum of a row: each group of 8 left to right, then every
// group sum s_j becomes s_j + s_(j xor o) for o = D/16, ..., 1 (group j of the
// row is group j % 4 of lane j / 4 of the row's lanes).  XP: the lane's blocks
// are permuted (register block b of lane L is the lane's block b xor L, see
// bfly_blocks), so the partner lane's group sits in register block b xor o;
// each add is commutative, so every lane still forms the same sums.
template <int D, bool XP>
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
    float o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = __shfl_xor_sync(0xffffffffu, g[XP ? (j ^ lo) : j], lo);
#pragma unroll
    for (int j = 0; j < 4; ++j) g[j] = __fadd_rn(g[j], o[j]);
  }
  const float a0 = __fadd_rn(g[0], g[2]), a1 = __fadd_rn(g[1], g[3]);
  return __fadd_rn(a0, a1);
}

// A butterfly stage between register blocks b and b + hb/8 (hb = 8 or 16) whose
// roles depend on the lane: s = +1 when the lower register block holds the
// lower element of each pair, -1 when it holds the upper one.  Then
// lower + upper = s*v[lo] + v[hi] lands in the slot of the lower element and
// lower - upper in the other (-s*v[hi] + v[lo]); an fma with a +-1 factor is
// the single rounding of that sum or difference.
__device__ __forceinline__ void bfly_blocks(float (&v)[32], int hb, float s) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    if ((i & hb) == 0) {
      const float a0 = v[i], a1 = v[i + 1], b0 = v[i + hb], b1 = v[i + hb + 1];
      fma2(v[i], v[i + 1], s, s, a0, a1, b0, b1);
      fma2(v[i + hb], v[i + hb + 1], -s, -s, b0, b1, a0, a1);
    }
  }
}

// Butterfly stages h = 1 .. 16 in registers, then h = 32, 64 across the lanes
// of the row (lane bit b set: other - v, else v + other; one fma with a +-1
// factor is that same single rounding).  Elements 2m and 2m+1 travel as a
// packed pair, so every stage but h = 1 runs two butterflies per instruction.
// XP (KVarN, D = 128): register block b of lane L holds the lane's block b xor
// L, so stages h = 8, 16 pair register blocks with lane-dependent roles.
template <bool XP>
__device__ __forceinline__ void fwht32_local(float (&v)[32], int sub) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {  // h = 1: inside a pair
    const float x = v[i], y = v[i + 1];
    v[i] = __fadd_rn(x, y);
    v[i + 1] = __fsub_rn(x, y);
  }
  // h = 2, 4 inside the 8-element blocks; h = 8, 16 between them
#pragma unroll
  for (int h = 2; h < (XP ? 8 : 32); h <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      if ((i & h) == 0) {
        const float x0 = v[i], x1 = v[i + 1], y0 = v[i + h], y1 = v[i + h + 1];
        add2(v[i], v[i + 1], x0, x1, y0, y1);
        sub2(v[i + h], v[i + h + 1], x0, x1, y0, y1);
      }
    }
  }
  if constexpr (XP) {
    bfly_blocks(v, 8, (sub & 1) ? -1.0f : 1.0f);
    bfly_blocks(v, 16, (sub & 2) ? -1.0f : 1.0f);
  }
}
template <int D>
__device__ __forceinline__ void fwht32(float (&v)[32], int sub) {
  constexpr int LPR = WideGeom<D>::LPR;
  fwht32_local<false>(v, sub);
#pragma unroll
  for (int lo = 1; lo < LPR; lo <<= 1) {
    const float sgn = (sub & lo) ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float o0 = __shfl_xor_sync(0xffffffffu, v[i], lo);
      const float o1 = __shfl_xor_sync(0xffffffffu, v[i + 1], lo);
      fma2(v[i], v[i + 1], sgn, sgn, v[i], v[i + 1], o0, o1);
    }
  }
}

// Butterfly stages h = 32 and 64 of a 128-wide row held by four lanes in the
// XP layout (register block b of lane L = elements 32L + 8(b xor L) .. + 7):
// register block b (b = 1, 2, 3) of every lane goes to lane L xor b, whose
// block it is, and block 0 stays.  Afterwards register block b of lane L holds
// elements 32(L xor b) + 8L .. + 7, so both stages pair register blocks, with
// the roles of the local ones.  Same pairs, stage order and single roundings
// as across lanes; 24 shuffles.
__device__ __forceinline__ void fwht_cross_xor(float (&v)[32], int sub) {
#pragma unroll
  for (int bb = 1; bb < 4; ++bb)
#pragma unroll
    for (int t = 0; t < 8; ++t) v[8 * bb + t] = __shfl_xor_sync(0xffffffffu, v[8 * bb + t], bb);
  bfly_blocks(v, 8, (sub & 1) ? -1.0f : 1.0f);   // h = 32
  bfly_blocks(v, 16, (sub & 2) ? -1.0f : 1.0f);  // h = 64
}

// Minimum and maximum of the 32 values (exact): four groups of 8 with
// three-input operations, then the groups; short dependent chains, few live
// values.
__device__ __forceinline__ void minmax32(const float (&x)[32], float& mn, float& mx) {
  float gmn[4], gmx[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const float* v = x + 8 * g;
    gmn[g] = min3f(min3f(v[0], v[1], v[2]), min3f(v[3], v[4], v[5]), fminf(v[6], v[7]));
    gmx[g] = max3f(max3f(v[0], v[1], v[2]), max3f(v[3], v[4], v[5]), fmaxf(v[6], v[7]));
  }
  mn = fminf(min3f(gmn[0], gmn[1], gmn[2]), gmn[3]);
  mx = fmaxf(max3f(gmx[0], gmx[1], gmx[2]), gmx[3]);
}

// Shared-memory index (in pairs) of the rotation's diagonal pair m (elements
// 2m, 2m+1) of a row of D: lane sub's pairs ml = 0..15 (m = 16 sub + ml) sit
// at (ml / 2) * 2 LPR + 2 sub + ml % 2, so the 16-byte reads (two pairs) of
// the row's LPR lanes fall on distinct banks.
template <int D>
__host__ __device__ constexpr int sign_pair_index(int m) {
  constexpr int LPR = D / 32;
  return (m % 16) / 2 * 2 * LPR + 2 * (m / 16) + m % 2;
}

// One row (token t, kv-head h) of an asymmetric format, 32 elements per lane.
// sgn: the rotation's diagonal pairs (+-1.0f) in shared memory, offset to this
// lane's first pair (sign_pair_index).
template <int D, int F, bool KVARN>
__device__ __forceinline__ void quantize_row_wide(float (&x)[32], int sub, bool active,
                                                  uint8_t* __restrict__ cache,
                                                  __half* __restrict__ meta, size_t row,
                                                  int64_t blk, int off, int h, int Hkv, int bs,
                                                  const float2* sgn, float cR) {
  constexpr int LPR = WideGeom<D>::LPR;
  // KVarN at D = 128: the lane's blocks arrive permuted (register block b of
  // lane L = its block b xor L) and the last two butterfly stages exchange
  // blocks by shuffles, after which register block b of lane L holds elements
  // 32(L xor b) + 8L + t (t < 8)
  constexpr bool XP = KVARN && D == 128;
  __half sig16 = __float2half_rn(1.0f);
  if constexpr (KVARN) {
    // Every packed product below feeds a scalar add (the sum tree, the h = 1
    // butterfly) or no add at all: ptxas contracts a packed multiply and a
    // packed add of the same pairs into one FFMA2 even with .rn, which would
    // skip the product's rounding (seen on the squared deviations when the
    // tree ran on packed pairs).
    const float inv_d = 1.0f / D;  // exact (power of two)
    const float mean = __fmul_rn(tree_sum32<D, XP>(x), inv_d);
    float sq[32];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float d0, d1;
      sub2(d0, d1, x[i], x[i + 1], mean, mean);
      mul2(sq[i], sq[i + 1], d0, d1, d0, d1);
    }
    const float var = __fmul_rn(tree_sum32<D, XP>(sq), inv_d);
    sig16 = __float2half_rn(__fsqrt_rn(var));
    if (__half2float(sig16) == 0.0f) sig16 = __float2half_rn(1.0f);
    const float inv_sigma = __frcp_rn(__half2float(sig16));
    // y = d . (x * (1/sigma)) = x * (d * (1/sigma)): a product by -1 is exact and
    // rounding is symmetric in sign, so the two orders give the same bits
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 sp = *reinterpret_cast<const float4*>(sgn + (i / 4) * 2 * LPR);
      float m0, m1, m2, m3;
      mul2(m0, m1, sp.x, sp.y, inv_sigma, inv_sigma);
      mul2(m2, m3, sp.z, sp.w, inv_sigma, inv_sigma);
      mul2(x[i], x[i + 1], x[i], x[i + 1], m0, m1);
      mul2(x[i + 2], x[i + 3], x[i + 2], x[i + 3], m2, m3);
    }
    if constexpr (XP) {
      fwht32_local<true>(x, sub);
      fwht_cross_xor(x, sub);
    } else {
      fwht32<D>(x, sub);
    }
#pragma unroll
    for (int i = 0; i < 32; i += 2) mul2(x[i], x[i + 1], x[i], x[i + 1], cR, cR);
  }
  float mn, mx;
  minmax32(x, mn, mx);
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
  // code = clamp(rne((x - z) * inv_s), 0, L): rne to int32, then the pack
  // instruction's saturation to [0, L]; each word is packed as soon as its
  // codes exist
  auto code2 = [&](int i, int& c0, int& c1) {
    float v0, v1;
    sub2(v0, v1, x[i], x[i + 1], zf, zf);
    mul2(v0, v1, v0, v1, inv_s, inv_s);
    c0 = __float2int_rn(v0);
    c1 = __float2int_rn(v1);
  };
  if constexpr (F == INT4A) {  // element 2i in the low nibble of byte i
    uint32_t ww[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      int c0, c1;
      code2(8 * k + 6, c0, c1);
      uint32_t t = pack_sat_u4(c1, c0, 0u);
      code2(8 * k + 4, c0, c1);
      t = pack_sat_u4(c1, c0, t);
      code2(8 * k + 2, c0, c1);
      t = pack_sat_u4(c1, c0, t);
      code2(8 * k, c0, c1);
      ww[k] = pack_sat_u4(c1, c0, t);
    }
    if (active) {
      if constexpr (XP) {  // word b: elements 32(b xor sub) + 8 sub .. + 7
#pragma unroll
        for (int b = 0; b < 4; ++b)
          *reinterpret_cast<uint32_t*>(cache + row * (D / 2) + 16 * (b ^ sub) + 4 * sub) = ww[b];
      } else {
        *reinterpret_cast<uint4*>(cache + row * (D / 2) + sub * 16) =
            make_uint4(ww[0], ww[1], ww[2], ww[3]);
      }
    }
  } else {  // element i in byte i
    uint32_t ww[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      int c0, c1, c2, c3;
      code2(4 * k + 2, c2, c3);
      code2(4 * k, c0, c1);
      ww[k] = pack_sat_u8(c1, c0, pack_sat_u8(c3, c2, 0u));
    }
    if (active) {
      if constexpr (XP) {  // words 2b, 2b+1: elements 32(b xor sub) + 8 sub .. + 7
#pragma unroll
        for (int b = 0; b < 4; ++b)
          *reinterpret_cast<uint2*>(cache + row * D + 32 * (b ^ sub) + 8 * sub) =
              make_uint2(ww[2 * b], ww[2 * b + 1]);
      } else {
        uint4* dst = reinterpret_cast<uint4*>(cache + row * D + sub * 32);
        dst[0] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
        dst[1] = make_uint4(ww[4], ww[5], ww[6], ww[7]);
      }
    }
  }
  if (active) {
    if (sub == 0) {
      constexpr int NF = KVARN ? 3 : 2;
      __half* m = meta + ((static_cast<size_t>(blk) * Hkv + h) * NF) * bs + off;
      m[0] = s16;
      m[bs] = z16;
      if constexpr (KVARN) m[2 * bs] = sig16;
    }
  }
}

// The rows r = p * RPW + (lane / LPR) of a token (its K heads, then its V
// heads), held in x: quantized and stored.  reload(x) refills x with the
// lane's input (a pass with both K and V rows quantizes x twice, and the
// KVarN row code rotates x in place).
template <int D, int KF, int VF, bool KVARN, class Reload>
__device__ __forceinline__ void quantize_pass(float (&x)[32], const Reload& reload,
                                              const WriteArgs& a, int r, int sub, size_t row0,
                                              long long blk, int off, const float2* lane_sgn) {
  const int Hkv = a.num_kv_heads;
  const bool act = r < 2 * Hkv;
  const bool is_v = r >= Hkv;
  const int h = is_v ? r - Hkv : r;
  if (__all_sync(0xffffffffu, !is_v || !act)) {
    quantize_row_wide<D, KF, KVARN>(x, sub, act, a.k_cache, a.k_meta, row0 + h, blk, off, h, Hkv,
                                    a.block_size, lane_sgn, a.cR);
  } else if (__all_sync(0xffffffffu, is_v || !act)) {
    quantize_row_wide<D, VF, KVARN>(x, sub, act, a.v_cache, a.v_meta, row0 + h, blk, off, h, Hkv,
                                    a.block_size, lane_sgn, a.cR);
  } else {  // a pass with K and V rows (fewer kv-heads than rows per pass)
    quantize_row_wide<D, KF, KVARN>(x, sub, act && !is_v, a.k_cache, a.k_meta, row0 + h, blk, off,
                                    h, Hkv, a.block_size, lane_sgn, a.cR);
    if constexpr (KVARN) reload(x);  // the K rows were rotated in place
    quantize_row_wide<D, VF, KVARN>(x, sub, act && is_v, a.v_cache, a.v_meta, row0 + h, blk, off,
                                    h, Hkv, a.block_size, lane_sgn, a.cR);
  }
}

// The rotation's diagonal as +-1.0f pairs in shared memory (sign_pair_index),
// in the order of each lane's registers: pair ml of lane sub (m = 16 sub + ml)
// holds the signs of the elements in its registers 2 ml, 2 ml + 1, which at
// D = 128 are the lane's block (ml / 4) xor sub, offset 2 (ml % 4).
template <int D, bool KVARN>
__device__ __forceinline__ void fill_sign_pairs(float2* sgn, const int8_t* signs) {
  if constexpr (KVARN) {
    for (int m = threadIdx.x; m < D / 2; m += blockDim.x) {
      const int sub = m / 16, ml = m % 16;
      const int mg = D == 128 ? 16 * sub + 4 * ((ml / 4) ^ sub) + ml % 4 : m;
      float2 p = make_float2(1.0f, 1.0f);
      if (signs != nullptr) {
        p.x = signs[2 * mg] < 0 ? -1.0f : 1.0f;
        p.y = signs[2 * mg + 1] < 0 ? -1.0f : 1.0f;
      }
      sgn[sign_pair_index<D>(m)] = p;
    }
    __syncthreads();
  }
}

// Persistent warps, one resident wave: warp w of the grid quantizes tokens
// w, w + W, w + 2W, ... (W warps in the grid), each loading its pass's rows
// straight from global memory.  Against one CTA per 8 tokens this saves the
// launch, sign-table fill and drain of every CTA (7 % on the KVarN write, 10 %
// on INT4).
template <int D, int KF, int VF, bool KVARN>
__global__ void __launch_bounds__(kWriteWarps * 32, ctas_per_sm(KVARN))
    write_asym_kernel(WriteArgs a) {
  constexpr int LPR = WideGeom<D>::LPR, RPW = WideGeom<D>::RPW;
  __shared__ __align__(16) float2 sgn[KVARN ? D / 2 : 1];
  fill_sign_pairs<D, KVARN>(sgn, a.signs);
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR, grp = lane / LPR;
  const int Hkv = a.num_kv_heads;
  const float2* lane_sgn = sgn + (KVARN ? sign_pair_index<D>(sub * 16) : 0);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWriteWarps;
  auto row_src = [&](int64_t t, int r) {
    return (r < Hkv ? a.key + t * a.key_stride + static_cast<size_t>(r) * D
                    : a.value + t * a.value_stride + static_cast<size_t>(r - Hkv) * D) + sub * 32;
  };
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kWriteWarps + (threadIdx.x >> 5);
       t < a.num_tokens; t += stride) {
    const int64_t slot = a.slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= static_cast<int64_t>(a.num_blocks) * a.block_size) {
      if (lane == 0) raise_error(1u);  // KVQ_DEVERR_SLOT_RANGE
      continue;
    }
    const int64_t blk = slot >> a.block_shift;
    const int off = static_cast<int>(slot & (a.block_size - 1));
    const size_t row0 = (static_cast<size_t>(blk) * a.block_size + off) * Hkv;
    for (int r0 = 0; r0 < 2 * Hkv; r0 += RPW) {
      const int r = r0 + grp;
      const bool act = r < 2 * Hkv;
      const uint16_t* src = row_src(t, act ? r : 0);
      auto load = [&](float (&y)[32]) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float e[8];
          // KVarN at D = 128: register block q holds the lane's block q xor sub
          const int qb = (KVARN && D == 128) ? (q ^ sub) : q;
          unpack8(act ? ldg_stream16(src + 8 * qb) : make_uint4(0, 0, 0, 0), e);
#pragma unroll
          for (int i = 0; i < 8; ++i) y[8 * q + i] = e[i];
        }
      };
      float x[32];
      load(x);
      quantize_pass<D, KF, VF, KVARN>(x, load, a, r, sub, row0, blk, off, lane_sgn);
    }
  }
}

template <int D, int KF, int VF, bool KVARN>
cudaError_t launch_asym_t(const WriteArgs& a, cudaStream_t st) {
  const int64_t blocks = (a.num_tokens + kWriteWarps - 1) / kWriteWarps;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    sms = 152;
  const int64_t resident = static_cast<int64_t>(sms) * ctas_per_sm(KVARN);
  const int64_t grid = blocks < resident ? blocks : resident;
  write_asym_kernel<D, KF, VF, KVARN><<<static_cast<unsigned>(grid), kWriteWarps * 32, 0, st>>>(a);
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

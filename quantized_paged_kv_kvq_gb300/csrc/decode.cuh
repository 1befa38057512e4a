// Single-token paged decode attention over the quantized cache.
//
// vLLM issue #4025 'Support for 4-bit KV Cache in paged-attention op',
// section 'methods', item 3: the paged-attention op takes k_scale,
// k_zeropoint, v_scale, v_zeropoint, reads the quantized cache, converts it
// to fp16/bf16 and computes attention; PR #4893's side note runs FP8-cache
// decode through the same paged-attention kernel.
//
// Design (one GPU, HBM-bound):
//  * grid (kv-head, sequence, context partition); a CTA of kWarps warps owns
//    one (sequence, kv-head, partition of P tokens) and its G query heads;
//    each warp streams every kWarps-th 16-token tile of the partition through
//    its own cp.async ring in shared memory (lane-linear, bank-conflict
//    free), so no block-wide barrier sits in the token loop;
//  * codes become exact fp16 values in registers (byte permutes / nibble
//    masks onto the 1024.0 exponent, or the native e4m3 convert) and feed
//    mma.sync m16n8k16 with fp32 accumulation: S^T = K q^T with 16 tokens x
//    8 query heads, then O^T += V^T P^T with 16 dims x 8 heads -- the GQA
//    group is the n = 8 dimension (G = 4 pads it with zero queries);
//  * the dot-product dimension is permuted so that every lane's operands
//    come from contiguous 16-byte loads; the query is permuted to match;
//  * online softmax in the log2 domain, rescaling only when the running
//    maximum grows by more than 2^8; scales, zero points and sigma are folded
//    in after the k-sum (K) or into the probabilities (V);
//  * partitions are combined in shared memory across warps and, when a
//    sequence spans several partitions, by a second log-sum-exp kernel.
#pragma once

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

constexpr int kDecodeWarps = 4;
constexpr int kDecodeMinBlocks = 4;  // resident CTAs per SM the register budget targets

template <int D, int KF, int VF, bool KVARN>
struct DecodeCfg {
  static constexpr int KB = row_bytes(KF, D);
  static constexpr int VB = row_bytes(VF, D);
  static constexpr int KSTEPS = D / 16;
  static constexpr int DTILES = D / 16;
  static constexpr int K_LANE = KB / 4;                  // K bytes per row per lane
  static constexpr int KPS = K_LANE < 16 ? K_LANE : 16;  // cp.async piece
  static constexpr int KP = K_LANE / KPS;                // pieces per row
  static constexpr int KSTRIDE_P = KB / KP;              // bytes between pieces
  static constexpr int KW = K_LANE / 4;                  // words per row per lane
  static constexpr int VPS = VB / 8;                     // V bytes per token per lane
  static constexpr int VW = VPS / 4;
  static constexpr int KMF = is_asym(KF) ? (KVARN ? 3 : 2) : 0;
  static constexpr int VMF = is_asym(VF) ? (KVARN ? 3 : 2) : 0;
  static constexpr int K_BYTES = 2 * KP * 32 * KPS;
  static constexpr int V_BYTES = 4 * 32 * VPS;
  static constexpr int M_BYTES = (KMF + VMF) * 32;
  static constexpr int STAGE = K_BYTES + V_BYTES + M_BYTES;
  static constexpr int STAGES = STAGE >= 4096 ? 3 : STAGE >= 3072 ? 4 : STAGE >= 2048 ? 5 : 8;
  static constexpr int WARP_SMEM = STAGES * STAGE;
  static constexpr int RING = kDecodeWarps * WARP_SMEM;
  static constexpr int COMBINE = kDecodeWarps * 8 * (D + 2) * 4 + 8 * D * 4;  // warps
  static constexpr int MERGE = (8 * kMaxPartitions + 8 + 8 * D) * 4;        // partitions
  static constexpr int QAREA = 8 * D * 4;
  static constexpr int max2(int x, int y) { return x > y ? x : y; }
  // rings and the query rows live side by side; the combines reuse it all later
  static constexpr int MAIN = max2(RING + QAREA, max2(COMBINE, MERGE));
  static constexpr int SMEM = MAIN + (kMaxPartition / 16) * 4;
  static_assert(KW * 4 == K_LANE && VW * 4 == VPS, "layout");
};

// d index of the query element that meets k-slot (2c, 2c+1, 2c+8, 2c+9)[e]
// of k-step j in lane-quad position c.
template <int D, int KF>
__device__ __forceinline__ int kslot_d(int c, int j, int e) {
  using C = DecodeCfg<D, KF, INT8, false>;
  if constexpr (KF != INT4A) {
    constexpr int WPP = C::KPS / 4;
    const int piece = j / WPP, within = j % WPP;
    return piece * C::KSTRIDE_P + c * C::KPS + 4 * within + e;
  } else {
    const int eb = 2 * (c * C::KPS + 4 * (j >> 1));
    const int ev = (e == 0) ? 0 : (e == 1) ? 4 : (e == 2) ? 1 : 5;
    return eb + ((j & 1) ? ev + 2 : ev);
  }
}

// K operand (rows = tokens 2g, 2g+1; 4 k-slots per lane) for k-step j.
template <int KF, int KW>
__device__ __forceinline__ void k_frag(const uint32_t (&kw)[2][KW], int j, uint32_t& a0,
                                       uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  constexpr uint32_t K64 = 0x64646464u;
  if constexpr (KF == INT4A) {
    const int m = j >> 1, sh = (j & 1) * 8;
    a0 = and_or(kw[0][m] >> sh, 0x000F000Fu, 0x64006400u);
    a2 = and_or(kw[0][m] >> (sh + 4), 0x000F000Fu, 0x64006400u);
    a1 = and_or(kw[1][m] >> sh, 0x000F000Fu, 0x64006400u);
    a3 = and_or(kw[1][m] >> (sh + 4), 0x000F000Fu, 0x64006400u);
  } else if constexpr (KF == E4M3) {
    a0 = e4m3x2_to_f16x2(kw[0][j] & 0xFFFFu);
    a2 = e4m3x2_to_f16x2(kw[0][j] >> 16);
    a1 = e4m3x2_to_f16x2(kw[1][j] & 0xFFFFu);
    a3 = e4m3x2_to_f16x2(kw[1][j] >> 16);
  } else if constexpr (KF == E5M2) {
    a0 = prmt(kw[0][j], 0u, 0x1404);
    a2 = prmt(kw[0][j], 0u, 0x3424);
    a1 = prmt(kw[1][j], 0u, 0x1404);
    a3 = prmt(kw[1][j], 0u, 0x3424);
  } else {  // INT8 (words already offset-binary) or UINT8A: biased 1024 + byte
    a0 = prmt(kw[0][j], K64, 0x4140);
    a2 = prmt(kw[0][j], K64, 0x4342);
    a1 = prmt(kw[1][j], K64, 0x4140);
    a3 = prmt(kw[1][j], K64, 0x4342);
  }
}

// V operand (rows = dims, k = tokens 4c..4c+3) for d-tile i; exact code values.
template <int VF>
__device__ __forceinline__ void v_pair(uint32_t wa, uint32_t wb, int i, uint32_t& rg,
                                       uint32_t& rg8) {
  constexpr uint32_t K64 = 0x64646464u;
  if constexpr (VF == INT4A) {
    const uint32_t pr = (i & 2) ? prmt(wa, wb, 0x7632) : prmt(wa, wb, 0x5410);
    const int sh = (i & 1) * 8;
    rg = hsub2_u32(and_or(pr >> sh, 0x000F000Fu, 0x64006400u), 0x64006400u);
    rg8 = hsub2_u32(and_or(pr >> (sh + 4), 0x000F000Fu, 0x64006400u), 0x64006400u);
  } else {
    const uint32_t il = (i & 1) ? prmt(wa, wb, 0x7362) : prmt(wa, wb, 0x5140);
    if constexpr (VF == E4M3) {
      rg = e4m3x2_to_f16x2(il & 0xFFFFu);
      rg8 = e4m3x2_to_f16x2(il >> 16);
    } else if constexpr (VF == E5M2) {
      rg = prmt(il, 0u, 0x1404);
      rg8 = prmt(il, 0u, 0x3424);
    } else {
      constexpr uint32_t bias = VF == INT8 ? 0x64806480u : 0x64006400u;  // 1152 / 1024
      rg = hsub2_u32(prmt(il, K64, 0x4140), bias);
      rg8 = hsub2_u32(prmt(il, K64, 0x4342), bias);
    }
  }
}

template <int VF, int VW>
__device__ __forceinline__ void v_frag(const uint32_t (&vw)[4][VW], int i, uint32_t& a0,
                                       uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  const int m = (VF == INT4A) ? (i >> 2) : (i >> 1);
  v_pair<VF>(vw[0][m], vw[1][m], i, a0, a1);
  v_pair<VF>(vw[2][m], vw[3][m], i, a2, a3);
}

// In-place rotation of a row of D floats in shared memory by one warp:
// forward x <- cR*H(d.x), inverse x <- d.(cR*H x).
template <int D, bool INVERSE>
__device__ __forceinline__ void rotate_row_warp(float* row, const int8_t* signs, float cR,
                                                int lane) {
  constexpr int E = D / 32;
  float v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = row[lane * E + e];
  if (!INVERSE && signs != nullptr) {
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (signs[lane * E + e] < 0) v[e] = -v[e];
  }
  fwht_lanes<E, 32>(v, lane);
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = __fmul_rn(v[e], cR);
  if (INVERSE && signs != nullptr) {
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (signs[lane * E + e] < 0) v[e] = -v[e];
  }
  __syncwarp();
#pragma unroll
  for (int e = 0; e < E; ++e) row[lane * E + e] = v[e];
}

__device__ __forceinline__ uint16_t f2bf(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}

template <int D, int KF, int VF, bool KVARN>
__global__ void __launch_bounds__(kDecodeWarps * 32, kDecodeMinBlocks)
    decode_partition_kernel(const DecodeArgs a) {
  using C = DecodeCfg<D, KF, VF, KVARN>;
  extern __shared__ __align__(16) uint8_t smem[];
  const int h = blockIdx.x, s = blockIdx.y, p = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int G = a.gqa;
  int ctx = a.context_lens[s];
  if (ctx < 0 || ctx > a.max_context_len) {  // contract violation: clamp, flag
    if (threadIdx.x == 0 && h == 0 && p == 0) raise_error(4u);  // KVQ_DEVERR_CONTEXT_RANGE
    ctx = ctx < 0 ? 0 : a.max_context_len;
  }
  const int P = a.partition_tokens;
  const int t_begin = p * P;
  const bool direct = a.num_partitions == 1;
  const size_t out_row0 = static_cast<size_t>(s) * a.num_q_heads + static_cast<size_t>(h) * G;

  if (t_begin >= ctx) {
    if (p == 0) {  // empty context: the output is zero
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) a.out[out_row0 * D + i] = 0;
    }
    return;
  }
  const int len = min(ctx - t_begin, P);
  const int ntiles = (len + 15) >> 4;
  const int Hkv = a.num_kv_heads;
  const int bs_shift = a.block_shift, bs_mask = a.block_size - 1;

  // ---- block ids of this partition
  int* s_blk = reinterpret_cast<int*>(smem + C::MAIN);
  {
    const int nblk = (len + bs_mask) >> bs_shift;
    const int* bt = a.block_table + static_cast<size_t>(s) * a.max_blocks_per_seq + (t_begin >> bs_shift);
    for (int i = threadIdx.x; i < nblk; i += blockDim.x) {
      int b = bt[i];
      if (b < 0 || b >= a.num_blocks) {
        raise_error(2u);  // KVQ_DEVERR_BLOCK_RANGE
        b = 0;
      }
      s_blk[i] = b;
    }
  }
  __syncthreads();

  // ---- per-warp pipeline over tiles warp, warp + W, ...; the first tiles are
  // requested before the query is prepared so that the two overlap
  uint8_t* ring = smem + warp * C::WARP_SMEM;
  const uint32_t ring_s = smem_u32(ring);
  const int my_tiles = ntiles > warp ? (ntiles - warp + kDecodeWarps - 1) / kDecodeWarps : 0;
  const uint32_t rowK = static_cast<uint32_t>(Hkv) * C::KB;  // bytes from one token row to the next
  const uint32_t rowV = static_cast<uint32_t>(Hkv) * C::VB;
  const uint32_t lane_k = 2 * g * rowK + h * C::KB + c * C::KPS;
  const uint32_t lane_v = 4 * c * rowV + h * C::VB + g * C::VPS;

  auto issue = [&](int it, int stage) {
    const int tok0 = (warp + it * kDecodeWarps) * 16;
    const int blk = s_blk[tok0 >> bs_shift];
    const size_t trow = (static_cast<size_t>(blk) << bs_shift) + (tok0 & bs_mask);
    const uint8_t* kb = a.k_cache + trow * rowK + lane_k;
    const uint8_t* vb = a.v_cache + trow * rowV + lane_v;
    const uint32_t st = ring_s + stage * C::STAGE;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
#pragma unroll
      for (int pc = 0; pc < C::KP; ++pc)
        cp_async<C::KPS>(st + ((r * C::KP + pc) * 32 + lane) * C::KPS, kb + r * rowK + pc * C::KSTRIDE_P);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      cp_async<C::VPS>(st + C::K_BYTES + (u * 32 + lane) * C::VPS, vb + u * rowV);
    if constexpr (C::KMF + C::VMF > 0) {
      if (lane < 2 * (C::KMF + C::VMF)) {
        const int fidx = lane >> 1, half = lane & 1;
        const bool isk = fidx < C::KMF;
        const int f = isk ? fidx : fidx - C::KMF;
        const int nf = isk ? C::KMF : C::VMF;
        const __half* base = isk ? a.k_meta : a.v_meta;
        const __half* src = base + ((static_cast<size_t>(blk) * Hkv + h) * nf + f) * a.block_size +
                            (tok0 & bs_mask) + 8 * half;
        cp_async<16>(st + C::K_BYTES + C::V_BYTES + fidx * 32 + half * 16, src);
      }
    }
  };

#pragma unroll
  for (int i = 0; i < C::STAGES - 1; ++i) {
    if (i < my_tiles) issue(i, i);
    cp_async_commit();
  }

  // ---- query rows (fp32) of the G heads, rotated for KVarN
  float* sq = reinterpret_cast<float*>(smem + C::RING);
  for (int i = threadIdx.x; i < 8 * D; i += blockDim.x) {
    const int n = i / D;
    float v = 0.0f;
    if (n < G) v = __uint_as_float(static_cast<uint32_t>(a.query[out_row0 * D + i]) << 16);
    sq[i] = v;
  }
  __syncthreads();
  if constexpr (KVARN) {
    for (int n = warp; n < G; n += kDecodeWarps) rotate_row_warp<D, false>(sq + n * D, a.signs, a.cR, lane);
    __syncthreads();
  }
  uint32_t qf[C::KSTEPS][2];
  float qs = 0.0f;
#pragma unroll
  for (int j = 0; j < C::KSTEPS; ++j) {
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[e] = __half2float(__float2half_rn(sq[g * D + kslot_d<D, KF>(c, j, e)]));
      qs += v[e];
    }
    qf[j][0] = pack_half2(v[0], v[1]);
    qf[j][1] = pack_half2(v[2], v[3]);
  }
  qs += __shfl_xor_sync(0xffffffffu, qs, 1);
  qs += __shfl_xor_sync(0xffffffffu, qs, 2);
  const float qsum0 = __shfl_sync(0xffffffffu, qs, (2 * c) * 4);
  const float qsum1 = __shfl_sync(0xffffffffu, qs, (2 * c + 1) * 4);

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;
  float O[C::DTILES][4];
#pragma unroll
  for (int i = 0; i < C::DTILES; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;

  int stage = 0;
  for (int it = 0; it < my_tiles; ++it) {
    cp_async_wait<C::STAGES - 2>();
    __syncwarp();
    const uint8_t* st = ring + stage * C::STAGE;
    const int valid = len - (warp + it * kDecodeWarps) * 16;

    uint32_t kw[2][C::KW];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
#pragma unroll
      for (int pc = 0; pc < C::KP; ++pc) {
        const uint8_t* src = st + ((r * C::KP + pc) * 32 + lane) * C::KPS;
        if constexpr (C::KPS == 16) {
          const uint4 w = *reinterpret_cast<const uint4*>(src);
          kw[r][pc * 4 + 0] = w.x; kw[r][pc * 4 + 1] = w.y;
          kw[r][pc * 4 + 2] = w.z; kw[r][pc * 4 + 3] = w.w;
        } else {
          const uint2 w = *reinterpret_cast<const uint2*>(src);
          kw[r][pc * 2 + 0] = w.x; kw[r][pc * 2 + 1] = w.y;
        }
      }
      if constexpr (KF == INT8) {
#pragma unroll
        for (int k = 0; k < C::KW; ++k) kw[r][k] ^= 0x80808080u;
      }
    }

    // ---- S^T = K q^T (two accumulators halve the dependent mma chain)
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < C::KSTEPS; ++j) {
      uint32_t a0, a1, a2, a3;
      k_frag<KF, C::KW>(kw, j, a0, a1, a2, a3);
      if (j & 1) mma16816(sb, a0, a1, a2, a3, qf[j][0], qf[j][1]);
      else mma16816(sa, a0, a1, a2, a3, qf[j][0], qf[j][1]);
    }
    float sacc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) sacc[k] = sa[k] + sb[k];

    uint32_t vw[4][C::VW];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint8_t* src = st + C::K_BYTES + (u * 32 + lane) * C::VPS;
      if constexpr (C::VPS == 16) {
        const uint4 w = *reinterpret_cast<const uint4*>(src);
        vw[u][0] = w.x; vw[u][1] = w.y; vw[u][2] = w.z; vw[u][3] = w.w;
      } else if constexpr (C::VPS == 8) {
        const uint2 w = *reinterpret_cast<const uint2*>(src);
        vw[u][0] = w.x; vw[u][1] = w.y;
      } else {
        vw[u][0] = *reinterpret_cast<const uint32_t*>(src);
      }
      if constexpr (VF == INT8) {
#pragma unroll
        for (int k = 0; k < C::VW; ++k) vw[u][k] ^= 0x80808080u;
      }
    }
    if (valid < 16) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (4 * c + u >= valid) {
#pragma unroll
          for (int k = 0; k < C::VW; ++k) vw[u][k] = (VF == INT8) ? 0x80808080u : 0u;
        }
    }
    const uint8_t* meta = st + C::K_BYTES + C::V_BYTES;
    float sl[4];
    if constexpr (!is_asym(KF)) {
      constexpr float bias = KF == INT8 ? 1152.0f : 0.0f;
      sl[0] = (sacc[0] - bias * qsum0) * a.qk_scale;
      sl[1] = (sacc[1] - bias * qsum1) * a.qk_scale;
      sl[2] = (sacc[2] - bias * qsum0) * a.qk_scale;
      sl[3] = (sacc[3] - bias * qsum1) * a.qk_scale;
    } else {
      const float2 ks = __half22float2(*reinterpret_cast<const __half2*>(meta + 0 * 32 + 4 * g));
      const float2 kz = __half22float2(*reinterpret_cast<const __half2*>(meta + 1 * 32 + 4 * g));
      float ks0 = ks.x, ks1 = ks.y, kz0 = kz.x, kz1 = kz.y;
      if constexpr (KVARN) {
        const float2 ksg = __half22float2(*reinterpret_cast<const __half2*>(meta + 2 * 32 + 4 * g));
        ks0 *= ksg.x; kz0 *= ksg.x; ks1 *= ksg.y; kz1 *= ksg.y;
      }
      sl[0] = (ks0 * (sacc[0] - 1024.0f * qsum0) + kz0 * qsum0) * a.qk_scale;
      sl[1] = (ks0 * (sacc[1] - 1024.0f * qsum1) + kz0 * qsum1) * a.qk_scale;
      sl[2] = (ks1 * (sacc[2] - 1024.0f * qsum0) + kz1 * qsum0) * a.qk_scale;
      sl[3] = (ks1 * (sacc[3] - 1024.0f * qsum1) + kz1 * qsum1) * a.qk_scale;
    }
    const bool ok0 = 2 * g < valid, ok1 = 2 * g + 1 < valid;
    if (!ok0) sl[0] = sl[1] = -INFINITY;
    if (!ok1) sl[2] = sl[3] = -INFINITY;

    // ---- online softmax (log2 domain), lazy rescale: the running maximum m is
    // only raised (with a reduction over the tile) when some logit exceeds it
    // by more than 8, so probabilities stay <= 2^8 and most tiles skip it
    float mx0 = fmaxf(sl[0], sl[2]), mx1 = fmaxf(sl[1], sl[3]);
    if (__any_sync(0xffffffffu, (mx0 > m0 + 8.0f) || (mx1 > m1 + 8.0f))) {
#pragma unroll
      for (int o = 4; o <= 16; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float al0 = fast_exp2(m0 - n0), al1 = fast_exp2(m1 - n1);
      m0 = n0;
      m1 = n1;
      l0 *= al0; l1 *= al1; z0 *= al0; z1 *= al1;
#pragma unroll
      for (int i = 0; i < C::DTILES; ++i) {
        O[i][0] *= al0; O[i][2] *= al0;
        O[i][1] *= al1; O[i][3] *= al1;
      }
    }
    float pr[4];
    pr[0] = fast_exp2(sl[0] - m0);
    pr[1] = fast_exp2(sl[1] - m1);
    pr[2] = fast_exp2(sl[2] - m0);
    pr[3] = fast_exp2(sl[3] - m1);
    l0 += pr[0] + pr[2];
    l1 += pr[1] + pr[3];
    if constexpr (is_asym(VF)) {
      const float2 vs = __half22float2(*reinterpret_cast<const __half2*>(meta + (C::KMF + 0) * 32 + 4 * g));
      const float2 vz = __half22float2(*reinterpret_cast<const __half2*>(meta + (C::KMF + 1) * 32 + 4 * g));
      float vs0 = vs.x, vs1 = vs.y, vz0 = vz.x, vz1 = vz.y;
      if constexpr (KVARN) {
        const float2 vsg = __half22float2(*reinterpret_cast<const __half2*>(meta + (C::KMF + 2) * 32 + 4 * g));
        vs0 *= vsg.x; vz0 *= vsg.x; vs1 *= vsg.y; vz1 *= vsg.y;
      }
      if (!ok0) vs0 = vz0 = 0.f;
      if (!ok1) vs1 = vz1 = 0.f;
      z0 += pr[0] * vz0 + pr[2] * vz1;
      z1 += pr[1] * vz0 + pr[3] * vz1;
      pr[0] *= vs0; pr[1] *= vs0;
      pr[2] *= vs1; pr[3] *= vs1;
    }
    // ---- P^T operand: lane (g, c) needs head g, tokens 4c..4c+3
    const uint32_t x0 = pack_half2(pr[0], pr[2]);  // head 2c, tokens (2g, 2g+1)
    const uint32_t x1 = pack_half2(pr[1], pr[3]);  // head 2c+1
    const int src0 = (2 * c) * 4 + (g >> 1), src1 = (2 * c + 1) * 4 + (g >> 1);
    const uint32_t u0 = __shfl_sync(0xffffffffu, x0, src0);
    const uint32_t u1 = __shfl_sync(0xffffffffu, x1, src0);
    const uint32_t u2 = __shfl_sync(0xffffffffu, x0, src1);
    const uint32_t u3 = __shfl_sync(0xffffffffu, x1, src1);
    const uint32_t b0 = (g & 1) ? u1 : u0;
    const uint32_t b1 = (g & 1) ? u3 : u2;
    // ---- O^T += V^T P^T
#pragma unroll
    for (int i = 0; i < C::DTILES; ++i) {
      uint32_t a0, a1, a2, a3;
      v_frag<VF, C::VW>(vw, i, a0, a1, a2, a3);
      mma16816(O[i], a0, a1, a2, a3, b0, b1);
    }
    __syncwarp();
    const int nx = it + C::STAGES - 1;
    if (nx < my_tiles) issue(nx, stage == 0 ? C::STAGES - 1 : stage - 1);
    cp_async_commit();
    stage = stage + 1 == C::STAGES ? 0 : stage + 1;
  }
  cp_async_wait<0>();

#pragma unroll
  for (int o = 4; o <= 16; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    z0 += __shfl_xor_sync(0xffffffffu, z0, o);
    z1 += __shfl_xor_sync(0xffffffffu, z1, o);
  }
  __syncthreads();  // every ring is drained; reuse shared memory for the combine

  float* cO = reinterpret_cast<float*>(smem);        // [W][8][D]
  float* cM = cO + kDecodeWarps * 8 * D;             // [W][8]
  float* cL = cM + kDecodeWarps * 8;                 // [W][8]
  float* cRes = cL + kDecodeWarps * 8;               // [8][D] (direct KVarN output)
#pragma unroll
  for (int i = 0; i < C::DTILES; ++i) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int d = g * (D / 8) + 2 * i + r;
      cO[(warp * 8 + 2 * c) * D + d] = O[i][2 * r] + z0;
      cO[(warp * 8 + 2 * c + 1) * D + d] = O[i][2 * r + 1] + z1;
    }
  }
  if (g == 0) {
    cM[warp * 8 + 2 * c] = m0;
    cM[warp * 8 + 2 * c + 1] = m1;
    cL[warp * 8 + 2 * c] = l0;
    cL[warp * 8 + 2 * c + 1] = l1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int n = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, cM[w * 8 + n]);
    float acc = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) {
      const float mw = cM[w * 8 + n];
      if (mw == -INFINITY) continue;
      const float wt = fast_exp2(mw - M);
      acc += wt * cO[(w * 8 + n) * D + d];
      L += wt * cL[w * 8 + n];
    }
    if constexpr (!is_asym(VF)) acc *= a.v_scale;
    if (direct) {
      const float res = acc / L;
      if constexpr (KVARN) cRes[i] = res;
      else a.out[out_row0 * D + i] = f2bf(res);
    } else {
      const size_t r = (out_row0 + n) * a.num_partitions + p;
      a.ws_acc[r * D + d] = acc;
      if (d == 0) {
        a.ws_ml[2 * r] = M;
        a.ws_ml[2 * r + 1] = L;
      }
    }
  }
  if (direct) {
    if constexpr (KVARN) {
      __syncthreads();
      for (int n = warp; n < G; n += kDecodeWarps) rotate_row_warp<D, true>(cRes + n * D, a.signs, a.cR, lane);
      __syncthreads();
      for (int i = threadIdx.x; i < G * D; i += blockDim.x) a.out[out_row0 * D + i] = f2bf(cRes[i]);
    }
    return;
  }

  // ---- the last CTA to finish a (sequence, kv-head) merges its partitions
  __threadfence();
  __syncthreads();
  int* s_last = reinterpret_cast<int*>(smem + C::MAIN);  // block ids are dead by now
  const int np_s = (ctx + P - 1) / P;
  if (threadIdx.x == 0) {
    unsigned long long* ctr = a.counters + static_cast<size_t>(s) * Hkv + h;
    unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(ctr), assumed, nv = 0;
    int tries = 0;
    do {  // counters carry the call's epoch: stale contents from any earlier use are reset
      assumed = old;
      nv = ((assumed >> 16) == a.epoch) ? assumed + 1 : ((a.epoch << 16) | 1ull);
      old = atomicCAS(ctr, assumed, nv);
    } while (old != assumed && ++tries < (1 << 20));
    if (old != assumed) raise_error(8u);  // KVQ_DEVERR_COMBINE
    s_last[0] = (old == assumed) && static_cast<int>(nv & 0xFFFFull) == np_s;
  }
  __syncthreads();
  if (!s_last[0]) return;
  __threadfence();
  float* sW = reinterpret_cast<float*>(smem);  // [8][np_s] partition weights
  float* sLinv = sW + 8 * kMaxPartitions;      // [8]
  float* sRes = sLinv + 8;                     // [8][D]
  for (int n = warp; n < G; n += kDecodeWarps) {
    const size_t r0 = (out_row0 + n) * a.num_partitions;
    float M = -INFINITY;
    for (int q = lane; q < np_s; q += 32) M = fmaxf(M, __ldcg(a.ws_ml + 2 * (r0 + q)));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int q = lane; q < np_s; q += 32) {
      const float w = fast_exp2(__ldcg(a.ws_ml + 2 * (r0 + q)) - M);
      sW[n * np_s + q] = w;
      L += w * __ldcg(a.ws_ml + 2 * (r0 + q) + 1);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) sLinv[n] = 1.0f / L;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * (D / 4); i += blockDim.x) {
    const int n = i / (D / 4), d4 = (i % (D / 4)) * 4;
    const float4* src = reinterpret_cast<const float4*>(a.ws_acc + (out_row0 + n) * a.num_partitions * D + d4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int q = 0; q < np_s; ++q) {
      const float4 v = __ldcg(src + static_cast<size_t>(q) * (D / 4));
      const float w = sW[n * np_s + q];
      acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
    }
    const float li = sLinv[n];
    if constexpr (KVARN) {
      sRes[n * D + d4 + 0] = acc.x * li; sRes[n * D + d4 + 1] = acc.y * li;
      sRes[n * D + d4 + 2] = acc.z * li; sRes[n * D + d4 + 3] = acc.w * li;
    } else {
      uint16_t* o = a.out + (out_row0 + n) * D + d4;
      o[0] = f2bf(acc.x * li); o[1] = f2bf(acc.y * li);
      o[2] = f2bf(acc.z * li); o[3] = f2bf(acc.w * li);
    }
  }
  if constexpr (KVARN) {
    __syncthreads();
    for (int n = warp; n < G; n += kDecodeWarps) rotate_row_warp<D, true>(sRes + n * D, a.signs, a.cR, lane);
    __syncthreads();
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) a.out[out_row0 * D + i] = f2bf(sRes[i]);
  }
}

}  // namespace kvq

// Single-token paged decode attention over the quantized cache.
//
// vLLM issue #4025 'Support for 4-bit KV Cache in paged-attention op',
// section 'methods', item 3: the paged-attention op takes k_scale,
// k_zeropoint, v_scale, v_zeropoint, reads the quantized cache, converts it
// to fp16/bf16 and computes attention; PR #4893's side note runs FP8-cache
// decode through the same paged-attention kernel.
//
// Design (one GPU, HBM-bound):
//  * stream-K: grid (ranges, kv-head groups of <= 8 heads); the 16-token
//    tiles of all sequences, in order, are cut into equal contiguous ranges,
//    one per CTA, so every SM gets the same work whatever the context lengths;
//    one consumer warp per kv-head.  Each tile is one pipeline stage: a TMA
//    box per kv-head for K and V (cp.async.bulk.tensor, 128B/64B swizzle) plus
//    one box per metadata array, completing on the stage's "full" mbarrier;
//    warps copy the stage into registers, release it on its "empty" mbarrier
//    and one elected thread refills it at once.  A block's rows of all heads
//    stream from HBM back to back.
//  * codes become exact fp16 values in registers (byte permutes / nibble
//    masks onto the 1024.0 exponent, or the native e4m3 convert) and feed
//    mma.sync m16n8k16 with fp32 accumulation: S^T = K q^T with 16 tokens x
//    8 query heads, then O^T += V^T P^T with 16 dims x 8 heads -- the GQA
//    group is the n = 8 dimension (G = 4 pads it with zero queries).  The
//    operands come from shared memory with 16-byte loads; the dot-product
//    dimension is permuted so each lane's slice is contiguous (the query is
//    permuted to match) and tokens are assigned to mma rows so that, with the
//    swizzle, every 16-byte load of a quarter-warp hits distinct banks.
//  * online softmax in the log2 domain; the running maximum is raised (with
//    a reduction) only when a logit exceeds it by more than 8, so P <= 2^8;
//    scales, zero points and sigma are folded in after the k-sum (K) or into
//    the probabilities (V).
//  * a sequence split between ranges is merged (log-sum-exp) by the last CTA
//    to finish its part, from L2, inside the same launch.
#pragma once

#include <cuda.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "quant_row.cuh"

namespace kvq {

constexpr int kHeadsPerCta = kHeadsPerCtaHost;  // kv-heads (= consumer warps) per CTA
constexpr int kSpinLimit = 1 << 22;  // default polls of an mbarrier before giving up

template <int D_, int KF, int VF, bool KVARN>
struct DecodeCfg {
  static constexpr int D = D_;
  static constexpr int KB = row_bytes(KF, D);
  static constexpr int VB = row_bytes(VF, D);
  static constexpr int KSTEPS = D / 16;
  static constexpr int DTILES = D / 16;
  static constexpr int K_LANE = KB / 4;                  // K bytes per row per lane
  static constexpr int KPS = K_LANE < 16 ? K_LANE : 16;  // load piece
  static constexpr int KP = K_LANE / KPS;                // pieces per row
  static constexpr int KSTRIDE_P = KB / KP;              // bytes between pieces
  static constexpr int KW = K_LANE / 4;                  // words per row per lane
  static constexpr int VPS = VB / 8;                     // V bytes per token per lane
  static constexpr int VW = VPS / 4;
  static constexpr int KMF = is_asym(KF) ? (KVARN ? 3 : 2) : 0;
  static constexpr int VMF = is_asym(VF) ? (KVARN ? 3 : 2) : 0;
  static constexpr int K_HEAD = 16 * KB;  // bytes of one head's 16-token box
  static constexpr int V_HEAD = 16 * VB;
  // swizzle of the TMA boxes: 16-byte chunk index ^= address bits [7, 7+n)
  // (a 256-byte row of 16-bit values is loaded as two 128-byte halves, each a
  // swizzle row, so it takes the 128-byte swizzle too)
  static constexpr int swz_bits(int rb) { return rb >= 128 ? 3 : rb == 64 ? 2 : 0; }
  static constexpr int K_SWZ = swz_bits(KB);
  static constexpr int V_SWZ = swz_bits(VB);
  static constexpr int align(int x) { return (x + 1023) / 1024 * 1024; }
  static constexpr int align128(int x) { return (x + 127) / 128 * 128; }
  // metadata of one field set: room for two 8-token boxes (pages of 8 tokens)
  // or one 16-token box
  static constexpr int meta_half(int hpc, int f) { return align128(hpc * f * 16); }
  static constexpr int meta_room(int hpc, int f) { return 2 * meta_half(hpc, f); }
  static constexpr int stage_bytes(int hpc) {
    return align(hpc * K_HEAD) + align(hpc * V_HEAD) + align(meta_room(hpc, KMF) + meta_room(hpc, VMF));
  }
  static constexpr int STAGE_MAX = stage_bytes(kHeadsPerCta);
  // ring depth: about 96 KB of tiles per CTA with two CTAs per SM
  static constexpr int STAGES = STAGE_MAX >= 24576 ? 3 : STAGE_MAX >= 16384 ? 5 : 6;
  static constexpr int EB = KF == BF16 ? 2 : 1;  // K element bytes (INT4: see kslot_d)
  static constexpr bool KVARN_ = KVARN;
  static_assert(KW * 4 == K_LANE && VW * 4 == VPS, "layout");
  static_assert(KMF == VMF || KMF == 0 || VMF == 0, "one metadata row layout for K and V");
};

// Shared memory of a CTA (bytes): the ring; per warp its query rows (G rows of
// D bf16, filled ahead of each segment) and, with KVarN, a float row for the
// query rotation; per stage a tile header and two mbarriers; a scratch area
// with the producer's cursor and the abort flag; and 1 KB of alignment.
__host__ __device__ constexpr int q_rows_bytes(int g, int d) { return (g * d * 2 + 15) / 16 * 16; }
template <class C>
__host__ __device__ constexpr int decode_smem_bytes(int hpc, int g) {
  return C::STAGES * C::stage_bytes(hpc) + hpc * q_rows_bytes(g, C::D) + (C::KVARN_ ? hpc * C::D * 4 : 0) +
         C::STAGES * 48 + 256 + 1024;
}

// Row of mma row r (0..15) of a tile: the QK row r holds token kRow[r].  With
// V's k-slot tokens kRow[c + 8(u&1) + 4(u>>1)] this makes each quarter-warp's
// 16-byte shared loads conflict-free under the swizzle and lets lane (g, c)
// take its P operand from lanes c and c + 4.
__device__ __forceinline__ int tile_row(int r) {
  // 0,5,2,7, 8,13,10,15, 4,1,6,3, 12,9,14,11
  const int lo = r & 3, hi = (r >> 2) & 1, top = r >> 3;
  const int odd = lo & 1;
  return lo + 8 * hi + 4 * (odd ^ top);
}
__device__ __forceinline__ int v_token(int c, int u) { return tile_row(c + 8 * (u & 1) + 4 * (u >> 1)); }

// d index of the query element that meets k-slot (2c, 2c+1, 2c+8, 2c+9)[e]
// of k-step j in lane-quad position c.
template <int D, int KF>
__device__ __forceinline__ int kslot_d(int c, int j, int e) {
  using C = DecodeCfg<D, KF, INT8, false>;
  if constexpr (KF != INT4A) {  // 4 consecutive elements per k-step and lane
    constexpr int EB = C::EB;
    constexpr int WPP = C::KPS / (4 * EB);  // k-steps per load piece
    const int piece = j / WPP, within = j % WPP;
    return (piece * C::KSTRIDE_P + c * C::KPS + 4 * EB * within) / EB + e;
  } else {
    const int eb = 2 * (c * C::KPS + 4 * (j >> 1));
    const int ev = (e == 0) ? 0 : (e == 1) ? 4 : (e == 2) ? 1 : 5;
    return eb + ((j & 1) ? ev + 2 : ev);
  }
}

// K operand (rows = the lane's two tokens; 4 k-slots per lane) for k-step j.
template <int KF, int KW>
__device__ __forceinline__ void k_frag(const uint32_t (&kw)[2][KW], int j, uint32_t& a0,
                                       uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  constexpr uint32_t K64 = 0x64646464u;
  if constexpr (KF == INT4A) {
    // low nibble of each byte pair -> 1024 + c (0x6400 | c), high nibble in
    // place -> 64 + c (0x5400 | c << 4, where one fp16 step is 1/16): one shift
    // per word; the two offsets come off after the k-sum
    const int m = j >> 1;
    const uint32_t w0 = (j & 1) ? (kw[0][m] >> 8) : kw[0][m];
    const uint32_t w1 = (j & 1) ? (kw[1][m] >> 8) : kw[1][m];
    a0 = and_or(w0, 0x000F000Fu, 0x64006400u);
    a2 = and_or(w0, 0x00F000F0u, 0x54005400u);
    a1 = and_or(w1, 0x000F000Fu, 0x64006400u);
    a3 = and_or(w1, 0x00F000F0u, 0x54005400u);
  } else if constexpr (KF == E4M3) {
    a0 = e4m3x2_to_f16x2(kw[0][j] & 0xFFFFu);
    a2 = e4m3x2_to_f16x2(kw[0][j] >> 16);
    a1 = e4m3x2_to_f16x2(kw[1][j] & 0xFFFFu);
    a3 = e4m3x2_to_f16x2(kw[1][j] >> 16);
  } else if constexpr (KF == BF16) {  // the values themselves, two per word
    a0 = kw[0][2 * j];
    a2 = kw[0][2 * j + 1];
    a1 = kw[1][2 * j];
    a3 = kw[1][2 * j + 1];
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

// V operand (rows = dims, k = the lane's 4 tokens) for d-tile i; exact values.
template <int VF>
__device__ __forceinline__ void v_pair(uint32_t wa, uint32_t wb, int i, uint32_t& rg,
                                       uint32_t& rg8) {
  constexpr uint32_t K64 = 0x64646464u;
  if constexpr (VF == INT4A) {  // (1024 + c) - 1024 and (64 + c) - 64, exact
    const uint32_t pr = (i & 2) ? prmt(wa, wb, 0x7632) : prmt(wa, wb, 0x5410);
    const uint32_t w = (i & 1) ? (pr >> 8) : pr;
    rg = hsub2_u32(and_or(w, 0x000F000Fu, 0x64006400u), 0x64006400u);
    rg8 = hsub2_u32(and_or(w, 0x00F000F0u, 0x54005400u), 0x54005400u);
  } else if constexpr (VF == BF16) {  // word i holds dims 2i, 2i+1 of the token
    rg = prmt(wa, wb, 0x5410);
    rg8 = prmt(wa, wb, 0x7632);
  } else {
    const uint32_t il = (i & 1) ? prmt(wa, wb, 0x7362) : prmt(wa, wb, 0x5140);
    if constexpr (VF == E4M3) {
      rg = e4m3x2_to_f16x2(il & 0xFFFFu);
      rg8 = e4m3x2_to_f16x2(il >> 16);
    } else if constexpr (VF == E5M2) {
      rg = prmt(il, 0u, 0x1404);
      rg8 = prmt(il, 0u, 0x3424);
    } else {  // exact: subtract the 1152 / 1024 offset in fp16 (a large offset left in
              // the fp32 sum costs accuracy over long contexts)
      constexpr uint32_t bias = VF == INT8 ? 0x64806480u : 0x64006400u;
      rg = hsub2_u32(prmt(il, K64, 0x4140), bias);
      rg8 = hsub2_u32(prmt(il, K64, 0x4342), bias);
    }
  }
}

template <int VF, int VW>
__device__ __forceinline__ void v_frag(const uint32_t (&vw)[4][VW], int i, uint32_t& a0,
                                       uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  const int m = (VF == INT4A) ? (i >> 2) : (VF == BF16) ? i : (i >> 1);
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
  __syncwarp();
}

__device__ __forceinline__ uint16_t f2bf(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}

// ---------------------------------------------------------------------------
// mbarrier / TMA primitives
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for `parity` of an mbarrier, at most `limit` polls; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int limit) {
  for (int n = 0; n < limit; ++n)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// The same, giving up early once the CTA's abort flag (shared memory) is set;
// the flag is read only after the first poll has failed.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity, int limit,
                                                   const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  for (int n = 1; n < limit; ++n) {
    if ((n & 15) == 0 && *abort) return false;
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
}
// 4-D TMA tile load completing on mbarrier `bar`, with an L2 eviction policy
// (the cache stream is read once: evict-first keeps it from flushing the
// small data that is read again -- partial results, queries, block tables).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
      : "memory");
}
// The same for a 5-D tensor map (rows of 16-bit values seen as two 128-byte halves).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, int v, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v), "r"(bar),
      "l"(policy)
      : "memory");
}
// Codes of one tile: the row-major maps are 4-D (row, head, token, block) per
// head or (row, token, head, block) head-major; rows over 128 bytes add a
// leading half-row dimension (two 128-byte halves, each a swizzle row).
template <int RB>
__device__ __forceinline__ void tma_codes_head(uint32_t dst, const CUtensorMap* map, int head,
                                               int tok, int blk, uint32_t bar, uint64_t pol) {
  if constexpr (RB > 128) tma_load_5d(dst, map, 0, 0, head, tok, blk, bar, pol);
  else tma_load_4d(dst, map, 0, head, tok, blk, bar, pol);
}
template <int RB>
__device__ __forceinline__ void tma_codes_heads(uint32_t dst, const CUtensorMap* map, int tok,
                                                int head0, int blk, uint32_t bar, uint64_t pol) {
  if constexpr (RB > 128) tma_load_5d(dst, map, 0, 0, tok, head0, blk, bar, pol);
  else tma_load_4d(dst, map, 0, tok, head0, blk, bar, pol);
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Shared address of 16-byte chunk `chunk` (plus `byte` within it) of row `row`
// of a swizzled box starting at `base` (1024-byte aligned for swizzled boxes).
template <int RB, int SWZ>
__device__ __forceinline__ uint32_t swz_addr(uint32_t base, int row, int chunk, int byte = 0) {
  const uint32_t off = static_cast<uint32_t>(row * RB + chunk * 16);
  const uint32_t phys = SWZ ? (off ^ (((off >> 7) & ((1u << SWZ) - 1)) << 4)) : off;
  return base + phys + byte;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
  return r;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 r;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
  return r;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a));
  return r;
}
__device__ __forceinline__ float lds_half(uint32_t a) {
  uint16_t r;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(r) : "r"(a));
  return __half2float(__ushort_as_half(r));
}


// Walsh-Hadamard butterfly over rows of D = 8 * E values where lane (g, c) of
// a warp holds the E consecutive values g*E .. g*E+E-1 of row c (the layout of
// the PV accumulators); same stage order as fwht_lanes.
template <int E>
__device__ __forceinline__ void fwht_accum_rows(float (&v)[E], int g) {
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if ((i & h) == 0) {
        float x = v[i], y = v[i + h];
        v[i] = __fadd_rn(x, y);
        v[i + h] = __fsub_rn(x, y);
      }
    }
  }
#pragma unroll
  for (int gm = 1; gm < 8; gm <<= 1) {
    const bool upper = (g & gm) != 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float other = __shfl_xor_sync(0xffffffffu, v[i], 4 * gm);
      v[i] = upper ? __fsub_rn(other, v[i]) : __fadd_rn(v[i], other);
    }
  }
}

// mma16816 with the accumulator given as four separate floats; BF: both
// operands bf16 (the 16-bit cache), else both fp16
template <bool BF = false>
__device__ __forceinline__ void mma16816(float& c0, float& c1, float& c2, float& c3, uint32_t a0,
                                         uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  if constexpr (BF) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c0), "+f"(c1), "+f"(c2), "+f"(c3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c0), "+f"(c1), "+f"(c2), "+f"(c3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}
__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// two operands of an mma in the cache's 16-bit type (bf16 for the 16-bit
// cache, else fp16), rounded to nearest
template <bool BF>
__device__ __forceinline__ uint32_t pack_op2(float lo, float hi) {
  return BF ? pack_bf162(lo, hi) : pack_half2(lo, hi);
}

// Page modes of the decode kernel (its PAGES template argument).
constexpr int kPagesOne = 0;    // one pool, pages of 16 tokens or more
constexpr int kPages8 = 1;      // one pool of 8-token pages
constexpr int kPagesMixed = 2;  // a pool per page class, pages of 16 tokens or more

// The producer's position in the range.
struct Cursor {
  long long ps;  // global index of the first tile of sequence s
  int s, t;      // sequence and tile of the next load
  int tiles, ctx;
  int blk;         // block id of that tile (read ahead)
  int nx, nx_ctx;  // next sequence of the range with tokens (num_seqs: none)
  int i;           // loads issued
  int cls;         // page class of sequence s
  int lam;         // weighted start of sequence s (the partition's line)
};

static_assert(sizeof(Cursor) <= 48, "the cursor lives in scratch words 16..21");

// Tensor maps of each page class's codes and metadata (N classes).
template <int N>
struct DecodeMaps {
  CUtensorMap k[N], v[N], km[N], vm[N];
};
template <int PAGES>
using DecodeMapsOf = DecodeMaps<PAGES == kPagesMixed ? kMaxPageClasses : 1>;

// Page class of sequence s (0 without a class array; a class outside the
// call's raises KVQ_DEVERR_CLASS_RANGE and reads class 0).
__device__ __forceinline__ int seq_class_of(const DecodeArgs& a, int s) {
  if (a.seq_class == nullptr) return 0;
  const int c = a.seq_class[s];
  if (c < a.num_classes) return c;
  raise_error(32u);  // KVQ_DEVERR_CLASS_RANGE
  return 0;
}

// One stage's tile: which sequence / tile it is and how it ends a segment.
struct TileHeader {
  int s;       // sequence
  int t;       // 16-token tile index within the sequence
  int valid;   // valid tokens in the tile (1..16)
  int flags;   // bit 0: first tile of this CTA's segment of s; bit 1: last tile
  int ps;      // global index of the sequence's first tile
  int tiles;   // tiles of the sequence
  int next_s;  // sequence of the range's next segment (first tiles only), or -1
  int lam;     // weighted start of the sequence on the partition's line
};

__device__ __forceinline__ uint16_t lds_u16(uint32_t a) {
  uint16_t r;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(r) : "r"(a));
  return r;
}
__device__ __forceinline__ void sts_u16(uint32_t a, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int seq_tiles(const DecodeArgs& a, int s) {
  const int ctx = a.context_lens[s];
  return ctx <= 0 ? 0 : (min(ctx, a.max_context_len) + 15) >> 4;
}

// floor(n / d) for n >= 0, d > 0: a 32-bit division whenever both fit (the
// 64-bit division is a long software sequence on this part)
__device__ __forceinline__ long long div_floor(long long n, long long d) {
  if (((static_cast<unsigned long long>(n) | static_cast<unsigned long long>(d)) >> 32) == 0)
    return static_cast<unsigned>(n) / static_cast<unsigned>(d);
  return n / d;
}
// ---- Stream-K partition.  The tiles lie on a weighted line: each sequence with
// tokens takes kBoundaryWeight (the cost of starting and ending a segment),
// then kTileWeight per tile, so a range that holds a sequence boundary gets
// fewer tiles.  The line (total weight W) is cut at cut(k) = floor(W k / NC);
// a tile belongs to the range whose interval holds its weighted start.  The
// partition is a fixed function of the lengths and NC.
constexpr int kTileWeight = 4;
constexpr int kBoundaryWeight = 16;  // 4 tiles: the best of 1.5 to 7 measured on the bench shapes

__device__ __forceinline__ long long cut(const DecodeArgs& a, long long W, int k) {
  return div_floor(W * k, a.num_ctas);
}
// The range holding weighted position w < W: the largest k with cut(k) <= w.
__device__ __forceinline__ int range_of_w(const DecodeArgs& a, long long w, long long W) {
  return static_cast<int>(div_floor((w + 1) * a.num_ctas - 1, W));
}
// A sequence on the weighted line: weighted start lam, first global tile ps,
// v tiles, boundary weight c; its tile t starts at lam + c + kTileWeight * t.
struct SeqSpan {
  long long lam, ps;
  int v, c;
};
// Tiles of the sequence whose weighted start lies before w.
__device__ __forceinline__ long long tiles_before(const SeqSpan& q, long long w) {
  const long long d = w - q.lam - q.c;
  if (d <= 0) return 0;
  const long long t = (d + kTileWeight - 1) / kTileWeight;
  return t < q.v ? t : q.v;
}
// Whether ranges [k0, k1) hold a tile of the sequence.
__device__ __forceinline__ bool holds_tiles(const DecodeArgs& a, long long W, const SeqSpan& q,
                                            int k0, int k1) {
  return tiles_before(q, cut(a, W, k0)) < tiles_before(q, cut(a, W, k1));
}
// The ranges of the sequence's first and last tiles.
__device__ __forceinline__ int first_range(const DecodeArgs& a, long long W, const SeqSpan& q) {
  return range_of_w(a, q.lam + q.c, W);
}
__device__ __forceinline__ int last_range(const DecodeArgs& a, long long W, const SeqSpan& q) {
  return range_of_w(a, q.lam + q.c + static_cast<long long>(kTileWeight) * (q.v - 1), W);
}

template <int N>
__device__ __forceinline__ void store_bf16_run(uint16_t* dst, const float (&v)[N]) {
  static_assert(N % 8 == 0, "run of 16-byte pieces");
#pragma unroll
  for (int i = 0; i < N / 8; ++i) {
    uint4 w;
    w.x = static_cast<uint32_t>(f2bf(v[8 * i])) | (static_cast<uint32_t>(f2bf(v[8 * i + 1])) << 16);
    w.y = static_cast<uint32_t>(f2bf(v[8 * i + 2])) | (static_cast<uint32_t>(f2bf(v[8 * i + 3])) << 16);
    w.z = static_cast<uint32_t>(f2bf(v[8 * i + 4])) | (static_cast<uint32_t>(f2bf(v[8 * i + 5])) << 16);
    w.w = static_cast<uint32_t>(f2bf(v[8 * i + 6])) | (static_cast<uint32_t>(f2bf(v[8 * i + 7])) << 16);
    reinterpret_cast<uint4*>(dst)[i] = w;
  }
}
template <int N>
__device__ __forceinline__ void store_f16_run(__half* dst, const float (&v)[N]) {
  static_assert(N % 8 == 0, "run of 16-byte pieces");
#pragma unroll
  for (int i = 0; i < N / 8; ++i)
    reinterpret_cast<uint4*>(dst)[i] =
        make_uint4(pack_half2(v[8 * i], v[8 * i + 1]), pack_half2(v[8 * i + 2], v[8 * i + 3]),
                   pack_half2(v[8 * i + 4], v[8 * i + 5]), pack_half2(v[8 * i + 6], v[8 * i + 7]));
}

// N fp16 values of a row at p[64i + e] (i < N/8, e < 8): one 16-byte load per i.
template <int N>
__device__ __forceinline__ void ldcg_halves(const __half* p, uint4 (&v)[N / 8]) {
  static_assert(N % 8 == 0, "whole 16-byte pieces");
#pragma unroll
  for (int i = 0; i < N / 8; ++i) v[i] = __ldcg(reinterpret_cast<const uint4*>(p + 64 * i));
}
__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

constexpr int kTeam = 8;       // ranges merged together at the first level of a tree
constexpr int kTreeRanges = 32;  // sequences over more ranges than this merge in two levels

// Slot of range kk for the sequence q: the range's first segment (0) when the
// range starts inside the sequence (the previous sequence's last tile, at
// weighted start q.lam - kTileWeight, lies before the cut), else its last (1).
__device__ __forceinline__ long long slot_index(const DecodeArgs& a, long long W, const SeqSpan& q,
                                                int kk, int HG, int hg) {
  return (static_cast<long long>(kk) * HG + hg) * 2 + (cut(a, W, kk) > q.lam - kTileWeight ? 0 : 1);
}

// Log-sum-exp merge of slots, by the whole CTA (warp w merges its kv-head's G
// query heads, four at a time).  The inputs are the slots of ranges r_first +
// step*i (i < count) for the sequence q, skipping a
// range whose span of `step` ranges (clipped at r_last) holds no tile.  A slot
// holds, per query head, the normalised output acc/l in fp16 and (m, l) in
// fp32; the merge is out = sum_i 2^(m_i - M) l_i (acc_i/l_i) / sum_i 2^(m_i - M) l_i.
// The result goes to the output rows of sequence s (dst < 0; with the inverse
// rotation for KVarN) or, in the same slot format, to slot dst.  Lane (nn, r)
// owns query head nn's dims 64i + 8r + e (i < DL/8, e < 8), so each 16-byte
// load of a warp reads whole 128-byte lines; each lane reads every slot's
// (m, l) itself, and the loads of PU slots are issued together.
template <int D, bool KVARN>
__device__ __forceinline__ void merge_slots(const DecodeArgs& a, int s, const SeqSpan& q,
                                            long long W, int HG, int hg, int warp, int lane, int hpc,
                                            int r_first, int step, int count, int r_last,
                                            long long dst) {
  constexpr int LQ = 8;        // lanes per query head
  constexpr int DL = D / LQ;   // dims per lane
  constexpr int PU = 4;        // slots per batch of loads
  const int G = a.gqa, rows = hpc * G;
  const int r = lane % LQ;
  const int h = hg * hpc + warp;
#pragma unroll 1
  for (int n0 = 0; n0 < G; n0 += 32 / LQ) {  // every lane runs every pass (shuffles below)
    const int nn = n0 + lane / LQ;
    const bool act = nn < G;
    float M = -INFINITY, Lsum = 0.f;
    float acc[DL];
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[e] = 0.f;
#pragma unroll 1
    for (int c0 = 0; c0 < count; c0 += 32) {  // slots c0 .. c0+31
      // lane p: first slot row of input c0 + p, or -1 if its span holds no tile
      long long base = -1;
      if (c0 + lane < count) {
        const int kk = r_first + step * (c0 + lane);
        if (holds_tiles(a, W, q, kk, min(kk + step, r_last + 1)))
          base = slot_index(a, W, q, kk, HG, hg) * rows;
      }
      const int cn = min(32, count - c0);
#pragma unroll 1
      for (int p0 = 0; p0 < cn; p0 += PU) {
        float ml[PU][2];
        uint4 v[PU][DL / 8];
#pragma unroll
        for (int u = 0; u < PU; ++u) {
          const long long b = __shfl_sync(0xffffffffu, base, (p0 + u) & 31);
          if (act && p0 + u < cn && b >= 0) {
            const long long sl = b + warp * G + nn;
            const float2 x = __ldcg(reinterpret_cast<const float2*>(a.ws_ml + 2 * sl));
            ml[u][0] = x.x;
            ml[u][1] = x.y;
            ldcg_halves<DL>(a.ws_acc + sl * D + 8 * r, v[u]);
          } else {
            ml[u][0] = -INFINITY;
            ml[u][1] = 0.f;
#pragma unroll
            for (int i = 0; i < DL / 8; ++i) v[u][i] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        float bm = ml[0][0];
#pragma unroll
        for (int u = 1; u < PU; ++u) bm = fmaxf(bm, ml[u][0]);
        // no slot in this batch (empty ranges; more ranges than tiles): nothing to
        // add, and 2^(m - M) would be 2^(-inf + inf) while M is still -inf
        if (bm == -INFINITY) continue;
        if (bm > M) {  // raise the running maximum, rescaling what was summed so far
          const float sc = fast_exp2(M - bm);
          Lsum *= sc;
#pragma unroll
          for (int e = 0; e < DL; ++e) acc[e] *= sc;
          M = bm;
        }
#pragma unroll
        for (int u = 0; u < PU; ++u) {
          const float w = fast_exp2(ml[u][0] - M) * ml[u][1];  // 2^(m - M) l
          Lsum += w;
#pragma unroll
          for (int i = 0; i < DL / 8; ++i) {
            const uint32_t q[4] = {v[u][i].x, v[u][i].y, v[u][i].z, v[u][i].w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float2 f = half2_bits_to_float2(q[t]);
              acc[8 * i + 2 * t] += w * f.x;
              acc[8 * i + 2 * t + 1] += w * f.y;
            }
          }
        }
      }
    }
    const float il = act ? 1.0f / Lsum : 0.f;
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[e] *= il;
    if (dst >= 0) {  // an intermediate result: back into slot format
      if (act) {
        const long long sl = dst * rows + warp * G + nn;
#pragma unroll
        for (int i = 0; i < DL / 8; ++i) {
          float piece[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) piece[e] = acc[8 * i + e];
          store_f16_run<8>(a.ws_acc + sl * D + 64 * i + 8 * r, piece);
        }
        if (r == 0) *reinterpret_cast<float2*>(a.ws_ml + 2 * sl) = make_float2(M, Lsum);
      }
      continue;
    }
    if constexpr (KVARN) {  // inverse rotation x = d . (cR * H y): the Walsh-Hadamard
      // matrix is unchanged by a permutation of index bits, so the butterflies run
      // over the local index (dim bits 0-2, 6) and then across the lanes (3-5)
      fwht_lanes<DL, LQ>(acc, r);
#pragma unroll
      for (int e = 0; e < DL; ++e) {
        const int dd = 64 * (e >> 3) + 8 * r + (e & 7);
        const float sgn = (a.signs != nullptr && a.signs[dd] < 0) ? -1.f : 1.f;
        acc[e] = __fmul_rn(acc[e], a.cR) * sgn;
      }
    }
    if (act) {
      uint16_t* orow = a.out + (static_cast<size_t>(s) * a.num_q_heads + static_cast<size_t>(h) * G + nn) * D + 8 * r;
#pragma unroll
      for (int i = 0; i < DL / 8; ++i) {
        float piece[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) piece[e] = acc[8 * i + e];
        store_bf16_run<8>(orow + 64 * i, piece);
      }
    }
  }
}

// New-token append, run by every warp of a CTA before its first tile load:
// the token at position ctx-1 of each sequence whose last tile lies in
// [R0, R1) is quantized into the caches, this warp's kv-head h only, with the
// row code of the cache write (so the codes equal kvq_write_cache's for the
// slot block_table[s][(ctx-1) / bs] * bs + (ctx-1) % bs).  That tile belongs
// to this range alone, so no other CTA reads the new row.  The warps walk the
// sequences from the range's first one, 32 at a time (a lane per sequence,
// prefix sum of tile counts, ballot of those that end inside the range).
// MIXED: the row lands in the pool of the sequence's page class.
template <int D, int KF, int VF, bool KVARN, bool MIXED>
__device__ __forceinline__ void append_new_tokens(const DecodeArgs& a, long long R0, long long R1,
                                               int s0, long long ps0, int h, int lane) {
  constexpr int LPR = RowGeom<D>::LPR;
  const int sub = lane % LPR;
  uint32_t sign_bits = 0;
  if constexpr (KVARN) {
    if (a.signs != nullptr) {
      const uint2 sg = *reinterpret_cast<const uint2*>(a.signs + sub * 8);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t byte = ((i < 4 ? sg.x : sg.y) >> (8 * (i & 3))) & 0xFFu;
        sign_bits |= (byte & 0x80u) ? (1u << i) : 0u;
      }
    }
  }
  const float kinv = (!is_asym(KF) && a.k_head_scale != nullptr) ? __frcp_rn(a.k_head_scale[h]) : a.k_inv;
  const float vinv = (!is_asym(VF) && a.v_head_scale != nullptr) ? __frcp_rn(a.v_head_scale[h]) : a.v_inv;
  const int S = a.num_seqs, Hkv = a.num_kv_heads;
  long long ps = ps0;  // first tile of sequence `base`
  for (int base = s0; base < S && ps < R1; base += 32) {
    const int s = base + lane;
    const int cx = s < S ? a.context_lens[s] : 0;
    const int cc = cx <= 0 ? 0 : min(cx, a.max_context_len);
    const long long v = (cc + 15) >> 4;
    long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const long long last = ps + incl - 1;  // last tile of sequence s
    unsigned mine = __ballot_sync(0xffffffffu, v > 0 && last >= R0 && last < R1);
    while (mine != 0u) {
      const int src = __ffs(mine) - 1;
      mine &= mine - 1u;
      const int sq = base + src;
      const int pos = __shfl_sync(0xffffffffu, cc, src) - 1;
      const int cls = MIXED ? seq_class_of(a, sq) : 0;
      const int bshift = a.block_shift[cls], bsz = 1 << bshift;
      const int blk = a.block_table[static_cast<size_t>(sq) * a.max_blocks_per_seq + (pos >> bshift)];
      if (blk < 0 || blk >= a.num_blocks[cls]) {
        if (lane == 0) raise_error(2u);  // KVQ_DEVERR_BLOCK_RANGE: nothing written
        continue;
      }
      const int off = pos & (bsz - 1);
      const size_t row = (static_cast<size_t>(blk) * bsz + off) * Hkv + h;
      float x[8];
      unpack8(*reinterpret_cast<const uint4*>(a.new_key + static_cast<size_t>(sq) * a.new_key_stride +
                                              static_cast<size_t>(h) * D + sub * 8), x);
      quantize_store<D, KF, KVARN>(x, lane < LPR, h, sub, row, a.k_cache_w[cls], a.k_meta_w[cls],
                                   kinv, blk, off, Hkv, bsz, sign_bits, a.cR);
      unpack8(*reinterpret_cast<const uint4*>(a.new_value + static_cast<size_t>(sq) * a.new_value_stride +
                                              static_cast<size_t>(h) * D + sub * 8), x);
      quantize_store<D, VF, KVARN>(x, lane < LPR, h, sub, row, a.v_cache_w[cls], a.v_meta_w[cls],
                                   vinv, blk, off, Hkv, bsz, sign_bits, a.cR);
    }
    ps += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// Stream-K decode: CTA (k, hg) owns tiles [k*T/NC, (k+1)*T/NC) of the global
// tile order (sequence-major, 16 tokens of all this group's heads per tile).
// Thread 0 is also the producer that keeps the ring full.  A sequence the
// range covers only in part leaves a partial result in the range's slot,
// published with the call's tag by the group's last warp (the others never
// wait for it); after its own range, a CTA that finds the tags of every other
// range of such a sequence merges the slots.  Store-then-fence-then-load of
// the tags guarantees at least one finder; a claim word per sequence keeps it
// to one.
// PAGES: kPagesOne (one pool, pages of 16 tokens or more), kPages8 (8-token
// pages: a tile is two pages) or kPagesMixed (each sequence in the pool of its
// page class); separate instances, so that one page size keeps the one-box
// path's registers.
// Two CTAs per SM (128 registers a thread), except the 16-bit cache (its
// stages fill shared memory): one.
template <int D, int KF, int VF, bool KVARN, int PAGES>
__global__ void __launch_bounds__(kHeadsPerCta * 32, (KF == BF16) ? 1 : 2)
    decode_partition_kernel(const DecodeArgs a, const __grid_constant__ DecodeMapsOf<PAGES> maps) {
  using C = DecodeCfg<D, KF, VF, KVARN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;  // the window is padded by 1 KB
  uint8_t* smem = smem_raw + (base_s - raw_s);

  const int k = blockIdx.x, NC = gridDim.x, hg = blockIdx.y, HG = gridDim.y;
  const int hpc = a.heads_per_cta;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int G = a.gqa, S = a.num_seqs;
  const int h = hg * hpc + warp;  // this warp's kv-head
  const int pub = hpc - 1;        // the warp that publishes partial results
  const int stage_bytes = C::stage_bytes(hpc);
  const int v_off = C::align(hpc * C::K_HEAD);
  const int m_off = v_off + C::align(hpc * C::V_HEAD);  // K metadata box, then V's
  const int vm_off = m_off + C::meta_room(hpc, C::KMF);
  // 8-token pages: a 16-token tile is two pages, loaded as two boxes each
  constexpr bool split = PAGES == kPages8;
  constexpr bool mixed = PAGES == kPagesMixed;
  const uint32_t ring_end = C::STAGES * stage_bytes;
  const int qrb = q_rows_bytes(G, D);
  const uint32_t qbuf_s = base_s + ring_end + warp * qrb;  // this warp's query rows (bf16)
  const uint32_t rot_off = ring_end + hpc * qrb;           // KVarN: one float row per warp
  const uint32_t hdr_off = rot_off + (KVARN ? hpc * D * 4 : 0);
  TileHeader* hdr = reinterpret_cast<TileHeader*>(smem + hdr_off);
  const uint32_t full_s = base_s + hdr_off + C::STAGES * sizeof(TileHeader);
  const uint32_t empty_s = full_s + 8 * C::STAGES;
  long long* scratch =
      reinterpret_cast<long long*>(smem + hdr_off + C::STAGES * (sizeof(TileHeader) + 16));
  // scratch: [0] W (the partition line's length), [1] first sequence, [2] its
  // first tile, [3] R1, [4..12) scan,
  // [12..16) partial segments: (first tile, sequence << 32 | tiles) per end of the range,
  // [16..22) producer cursor, [22] second page id, [23] abort flag (int),
  // [24] withheld tile (int; test hook), [25] per end of the range: warps whose
  // rows of the partial slot are stored (two ints), [26..28) range bounds
  // (prologue), [28..30) per end of the range: the weighted start of its
  // sequence, [30] the boundary weight, [31] the first sequence's weighted start
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(scratch + 23);
  int* const done_warps = reinterpret_cast<int*>(scratch + 25);
  const int spin = a.spin_limit;

  // this warp's G query rows of sequence s -> shared memory (asynchronous)
  auto prefetch_q = [&](int s) {
    const uint16_t* src =
        a.query + (static_cast<size_t>(s) * a.num_q_heads + static_cast<size_t>(h) * G) * D;
    for (int i = lane; i < G * D / 8; i += 32) cp_async<16>(qbuf_s + 16 * i, src + 8 * i);
    cp_async_commit();
  };

  // ---- the ring's barriers and the CTA's flags (published by the barriers of
  // the range scan below)
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(full_s + 8 * i, 1);
      mbar_init(empty_s + 8 * i, hpc);
    }
    for (int i = 12; i < 16; ++i) scratch[i] = -1;
    *abort_flag = 0;
    reinterpret_cast<int*>(scratch + 24)[0] =
        (k == a.withhold_cta && hg == 0) ? a.withhold_tile : -1;
    done_warps[0] = done_warps[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }

  // ---- context checks; zero outputs of the empty sequences this CTA owns
  if (k == 0 && hg == 0) {
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
      const int ctx = a.context_lens[s];
      if (ctx < 0 || ctx > a.max_context_len) raise_error(4u);  // KVQ_DEVERR_CONTEXT_RANGE
    }
  }
  for (int s = k; s < S; s += NC) {
    if (seq_tiles(a, s) == 0) {
      uint16_t* o = a.out + (static_cast<size_t>(s) * a.num_q_heads + static_cast<size_t>(h) * G) * D;
      for (int i = lane; i < G * D; i += 32) o[i] = 0;
    }
  }

  // ---- the range [R0, R1) of global tiles and its first sequence: a block scan
  // of (sequences with tokens, tiles) gives each sequence its first tile and
  // weighted start; the sequence whose weighted span holds cut(k) gives R0
  // (and cut(k+1) R1); then the sequence holding tile R0.  With more sequences
  // than threads the chunked scan below charges no boundary weight.
  long long T = 0, Wt = 0;
  int bw = kBoundaryWeight;
  long long R0 = 0, R1 = 0;
  if (S <= static_cast<int>(blockDim.x)) {  // one pass: a sequence per thread
    const int s = threadIdx.x;
    const long long v = s < S ? seq_tiles(a, s) : 0;
    const long long pk = v > 0 ? (1ll << 40) | v : 0;  // (sequences with tokens, tiles)
    long long incl = pk;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) scratch[4 + warp] = incl;
    __syncthreads();
    long long before = 0, tot = 0;
    for (int w = 0; w < hpc; ++w) {
      const long long x = scratch[4 + w];
      tot += x;
      if (w < warp) before += x;
    }
    const long long mask = (1ll << 40) - 1;
    T = tot & mask;
    Wt = static_cast<long long>(kTileWeight) * T + bw * (tot >> 40);
    const long long ex = before + incl - pk;  // exclusive prefix
    const SeqSpan q{static_cast<long long>(kTileWeight) * (ex & mask) + bw * (ex >> 40), ex & mask,
                    static_cast<int>(v), bw};
    const long long lam_end = q.lam + kTileWeight * v + bw;
    __syncthreads();  // every thread has read the scan words
    const long long c0 = cut(a, Wt, k), c1 = cut(a, Wt, k + 1);
    if (v > 0 && q.lam <= c0 && c0 < lam_end) scratch[26] = q.ps + tiles_before(q, c0);
    if (v > 0 && q.lam <= c1 && c1 < lam_end) scratch[27] = q.ps + tiles_before(q, c1);
    if (threadIdx.x == 0) {  // a cut at the end of the line
      if (c0 >= Wt) scratch[26] = T;
      if (c1 >= Wt) scratch[27] = T;
    }
    __syncthreads();
    R0 = scratch[26];
    R1 = scratch[27];
    if (v > 0 && q.ps <= R0 && R0 < q.ps + v) {
      scratch[1] = s;
      scratch[2] = q.ps;
      scratch[31] = q.lam;  // the first sequence's weighted start (read below)
    }
    __syncthreads();
  } else {  // many sequences: total first, then a chunked scan up to the range start
    bw = 0;
    long long part = 0;
    for (int s = threadIdx.x; s < S; s += blockDim.x) part += seq_tiles(a, s);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) scratch[4 + warp] = part;
    __syncthreads();
    for (int w = 0; w < hpc; ++w) T += scratch[4 + w];
    __syncthreads();
    Wt = static_cast<long long>(kTileWeight) * T;
    // with no boundary weight the first tile at or after cut(k) is cut(k) / kTileWeight rounded up
    R0 = (cut(a, Wt, k) + kTileWeight - 1) / kTileWeight;
    R1 = (cut(a, Wt, k + 1) + kTileWeight - 1) / kTileWeight;
    long long running = 0;
    for (int base = 0; base < S && running <= R0; base += blockDim.x) {
      const int s = base + threadIdx.x;
      const long long v = s < S ? seq_tiles(a, s) : 0;
      long long incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) scratch[4 + warp] = incl;
      __syncthreads();
      long long before = running;
      for (int w = 0; w < warp; ++w) before += scratch[4 + w];
      const long long excl = before + incl - v;
      if (v > 0 && excl <= R0 && R0 < excl + v) {
        scratch[1] = s;
        scratch[2] = excl;
        scratch[31] = kTileWeight * excl;
      }
      for (int w = 0; w < hpc; ++w) running += scratch[4 + w];
      __syncthreads();
    }
  }
  if (R0 >= R1) return;
  const int n = static_cast<int>(R1 - R0);
  const int s_first = static_cast<int>(scratch[1]);
  const long long ps_first = scratch[2];
  prefetch_q(s_first);
  if (a.new_key != nullptr) {  // new-token append: codes stored before any tile is loaded
    append_new_tokens<D, KF, VF, KVARN, mixed>(a, R0, R1, s_first, ps_first, h, lane);
    // the stores (generic proxy) before the tensor loads (async proxy) the
    // barrier below lets thread 0 issue
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }

  const long long lam_first = scratch[31];
  if (threadIdx.x == 0) {  // read by thread 0 alone until the barriers after the loop
    scratch[0] = Wt;
    scratch[3] = R1;
    scratch[30] = bw;
  }
  // the append's stores before thread 0's first tensor loads (the barriers and
  // flags were set up before the range scan, whose barriers publish them)
  if (a.new_key != nullptr) __syncthreads();

  // ---- producer cursor (thread 0): walks the range tile by tile
  const uint32_t tile_bytes = hpc * (C::K_HEAD + C::V_HEAD) + hpc * (C::KMF + C::VMF) * 32;
  // The cursor lives in shared memory: only thread 0 uses it, and registers
  // held by every thread for it would be taken from the consumers.
  Cursor* cur = reinterpret_cast<Cursor*>(scratch + 16);
  // 8-token pages: block id of the cursor tile's second page (read ahead); kept
  // out of the cursor, whose copies stay as small as for the other page sizes
  int* const cur_blk2 = reinterpret_cast<int*>(scratch + 22);
  auto block_of = [&](const Cursor& u) {  // block id of the cursor's tile (in its class's pool)
    return a.block_table[static_cast<size_t>(u.s) * a.max_blocks_per_seq +
                         ((16 * u.t) >> a.block_shift[mixed ? u.cls : 0])];
  };
  auto second_half = [&](const Cursor& u) {  // 8-token pages: tokens 8..15 of the tile exist
    return split && 16 * u.t + 8 < u.ctx;
  };
  auto block2_of = [&](const Cursor& u) {  // their page (entries past the context are never read)
    return second_half(u) ? a.block_table[static_cast<size_t>(u.s) * a.max_blocks_per_seq +
                                          ((16 * u.t) >> a.block_shift[0]) + 1]
                          : 0;
  };
  auto find_next = [&](Cursor& u) {  // first sequence after u.s with tokens, if the range goes on
    u.nx = S;
    if (u.ps + u.tiles >= scratch[3]) return;
    for (int s2 = u.s + 1; s2 < S; ++s2) {
      const int cx = a.context_lens[s2];
      const int cc = cx <= 0 ? 0 : min(cx, a.max_context_len);
      if (cc > 0) {
        u.nx = s2;
        u.nx_ctx = cc;
        return;
      }
    }
  };
  if (threadIdx.x == 0) {
    Cursor u;
    u.ps = ps_first;
    u.s = s_first;
    u.t = static_cast<int>(R0 - ps_first);
    u.ctx = min(a.context_lens[s_first], a.max_context_len);
    u.tiles = (u.ctx + 15) >> 4;
    u.cls = mixed ? seq_class_of(a, u.s) : 0;
    u.lam = static_cast<int>(lam_first);
    u.blk = block_of(u);
    if constexpr (split) *cur_blk2 = block2_of(u);
    u.nx_ctx = 0;
    u.i = 0;
    find_next(u);
    *cur = u;
  }
  auto issue = [&](int st) {  // the cursor's tile into stage st, then advance the cursor
    const uint64_t pol = l2_evict_first_policy();
    Cursor u = *cur;
    TileHeader& hd = hdr[st];
    hd.s = u.s;
    hd.t = u.t;
    hd.valid = min(16, u.ctx - 16 * u.t);
    hd.flags = (u.i == 0 || u.t == 0 ? 1 : 0) | (u.i == n - 1 || u.t == u.tiles - 1 ? 2 : 0);
    hd.ps = static_cast<int>(u.ps);
    hd.tiles = u.tiles;
    hd.next_s = u.nx < S ? u.nx : -1;
    hd.lam = u.lam;
    const int tok = 16 * u.t;
    int blk = u.blk;
    const int cl = mixed ? u.cls : 0;
    if (blk < 0 || blk >= a.num_blocks[cl]) {
      raise_error(2u);  // KVQ_DEVERR_BLOCK_RANGE: read block 0 instead
      blk = 0;
    }
    const int off = tok & ((1 << a.block_shift[cl]) - 1);
    const uint32_t sb = base_s + st * stage_bytes;
    const uint32_t bar = full_s + 8 * st;
    // test hook: this tile's loads are never issued (its stage never fills)
    if (u.i == reinterpret_cast<const int*>(scratch + 24)[0]) {
    } else if constexpr (split) {  // 8-token pages: the tile is two pages, each loaded as
      // per-head 8-row boxes (rows 0-7, then 8-15 of the head's [16][row] box)
      // and [head][field][8] metadata boxes (the second meta_half bytes on)
      const bool two = second_half(u);
      int blk2 = *cur_blk2;
      if (two && (blk2 < 0 || blk2 >= a.num_blocks[0])) {
        raise_error(2u);
        blk2 = 0;
      }
      mbar_arrive_expect(bar, two ? tile_bytes : tile_bytes / 2);
      for (int hf = 0; hf < (two ? 2 : 1); ++hf) {
        const int b = hf ? blk2 : blk;
        for (int hh = 0; hh < hpc; ++hh) {
          tma_codes_head<C::KB>(sb + hh * C::K_HEAD + hf * 8 * C::KB, &maps.k[0], hg * hpc + hh, 0,
                                b, bar, pol);
          tma_codes_head<C::VB>(sb + v_off + hh * C::V_HEAD + hf * 8 * C::VB, &maps.v[0],
                                hg * hpc + hh, 0, b, bar, pol);
        }
        if constexpr (C::KMF > 0)
          tma_load_4d(sb + m_off + hf * C::meta_half(hpc, C::KMF), &maps.km[0], 0, 0, hg * hpc, b,
                      bar, pol);
        if constexpr (C::VMF > 0)
          tma_load_4d(sb + vm_off + hf * C::meta_half(hpc, C::VMF), &maps.vm[0], 0, 0, hg * hpc, b,
                      bar, pol);
      }
    } else {  // one box per tile (pages of 16 or more tokens)
      mbar_arrive_expect(bar, tile_bytes);
      if (a.one_box) {
        tma_codes_heads<C::KB>(sb, &maps.k[cl], off, hg * hpc, blk, bar, pol);
        tma_codes_heads<C::VB>(sb + v_off, &maps.v[cl], off, hg * hpc, blk, bar, pol);
      } else {
        for (int hh = 0; hh < hpc; ++hh) {
          tma_codes_head<C::KB>(sb + hh * C::K_HEAD, &maps.k[cl], hg * hpc + hh, off, blk, bar,
                                pol);
          tma_codes_head<C::VB>(sb + v_off + hh * C::V_HEAD, &maps.v[cl], hg * hpc + hh, off, blk,
                                bar, pol);
        }
      }
      if constexpr (C::KMF > 0)
        tma_load_4d(sb + m_off, &maps.km[cl], off, 0, hg * hpc, blk, bar, pol);
      if constexpr (C::VMF > 0)
        tma_load_4d(sb + vm_off, &maps.vm[cl], off, 0, hg * hpc, blk, bar, pol);
    }
    ++u.i;
    if (++u.t == u.tiles && u.i < n) {  // on to the next sequence with tokens
      u.lam += kTileWeight * u.tiles + static_cast<int>(scratch[30]);
      u.ps += u.tiles;
      u.t = 0;
      if (u.nx >= S) {  // cannot happen with the tile count T; stay in bounds
        raise_error(4u);
        u.nx = S - 1;
        u.nx_ctx = 16;
      }
      u.s = u.nx;
      u.ctx = u.nx_ctx;
      u.tiles = (u.ctx + 15) >> 4;
      if constexpr (mixed) u.cls = seq_class_of(a, u.s);
      find_next(u);
    }
    if (u.i < n) {  // prefetched: consumed by the next issue
      u.blk = block_of(u);
      if constexpr (split) *cur_blk2 = block2_of(u);
    }
    *cur = u;
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < C::STAGES && i < n; ++i) issue(i);

  // ---- per-lane shared-memory addresses inside a stage (swizzled boxes)
  const int row0 = tile_row(g), row1 = tile_row(g + 8);
  uint32_t k_addr[2][C::KP];
#pragma unroll
  for (int pc = 0; pc < C::KP; ++pc) {
    const int chunk = (pc * C::KSTRIDE_P + c * C::KPS) / 16, byte = (c * C::KPS) % 16;
    k_addr[0][pc] = swz_addr<C::KB, C::K_SWZ>(warp * C::K_HEAD, row0, chunk, byte);
    k_addr[1][pc] = swz_addr<C::KB, C::K_SWZ>(warp * C::K_HEAD, row1, chunk, byte);
  }
  uint32_t v_addr[4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
    v_addr[u] = v_off + swz_addr<C::VB, C::V_SWZ>(warp * C::V_HEAD, v_token(c, u),
                                                  (g * C::VPS) / 16, (g * C::VPS) % 16);
  // metadata rows: per warp [field][16 tokens]; with 8-token pages two boxes of
  // [warp][field][8 tokens], the second meta_half bytes on
  constexpr int fstr = split ? 16 : 32;  // bytes between a warp's fields
  const int mhalf = C::meta_half(hpc, C::KMF > 0 ? C::KMF : C::VMF);
  const uint32_t mrow0 = split ? (row0 >> 3) * mhalf + 2 * (row0 & 7) : 2 * row0;
  const uint32_t mrow1 = split ? (row1 >> 3) * mhalf + 2 * (row1 & 7) : 2 * row1;
  const uint32_t meta_k = m_off + warp * C::KMF * fstr;
  const uint32_t meta_v = vm_off + warp * C::VMF * fstr;
  // this warp's kv-head scales (per-kv-head scales, when given, replace the tensor's)
  const float vsc = is_asym(VF) ? 1.0f : (a.v_head_scale != nullptr ? a.v_head_scale[h] : a.v_scale);
  const float qks = (!is_asym(KF) && a.k_head_scale != nullptr) ? a.qk_base * a.k_head_scale[h]
                                                                : a.qk_scale;

  uint32_t qf[C::KSTEPS][2];
  float qsum0 = 0.f, qsum1 = 0.f;
  float qb0 = 0.f, qb1 = 0.f;  // int4 K: sum over k of q_k times the code offset of slot k
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;
  // PV accumulators as the output runs they become: lane (g, c) holds dims
  // g*E .. g*E+E-1 of query heads 2c (Oa) and 2c+1 (Ob)
  constexpr int E = 2 * C::DTILES;
  float Oa[E], Ob[E];
  int seg_t0 = 0;
  bool first_seg = true;  // the range's first segment (slot 0 if partial; slot 1 otherwise)

  // A wait that runs out (a tile that never lands, a warp that never arrives)
  // raises KVQ_DEVERR_TIMEOUT and the abort flag: the producer issues nothing
  // more, so every warp soon meets a wait that cannot complete, sees the flag
  // there and leaves the loop; nothing is published, and the CTA returns once
  // no copy it issued is in flight (below).
  auto give_up = [&]() {
    if (lane == 0) {
      raise_error(16u);  // KVQ_DEVERR_TIMEOUT: the results of this launch are invalid
      *abort_flag = 1;
    }
  };
  int st = 0;
  uint32_t phase = 0;
  for (int i = 0; i < n; ++i) {
    if (!__all_sync(0xffffffffu, mbar_wait_or_abort(full_s + 8 * st, phase, spin, abort_flag))) {
      give_up();
      break;
    }
    const TileHeader hd = hdr[st];
    const uint32_t sb = base_s + st * stage_bytes;
    const size_t out_row0 = static_cast<size_t>(hd.s) * a.num_q_heads + static_cast<size_t>(h) * G;

    if (hd.flags & 1) {  // a new segment: this warp's query fragment, fresh state
      cp_async_wait<0>();  // the rows were fetched during the previous segment
      __syncwarp();
      float qs = 0.0f, qh = 0.0f;  // qh: the k-slots that meet high nibbles (int4 K)
      if constexpr (KVARN) {
        // each query row of the group is rotated in a float row and written back
        // over its bf16 row as fp16 (the rounding every quantized format gives
        // the query), so the fragments below read it like any other row
        float* srow = reinterpret_cast<float*>(smem + rot_off + warp * D * 4);
        for (int nn = 0; nn < G; ++nn) {
          for (int e = lane; e < D; e += 32)
            srow[e] = __uint_as_float(static_cast<uint32_t>(lds_u16(qbuf_s + 2 * (nn * D + e))) << 16);
          __syncwarp();
          rotate_row_warp<D, false>(srow, a.signs, a.cR, lane);
          for (int e = lane; e < D; e += 32)
            sts_u16(qbuf_s + 2 * (nn * D + e), __half_as_ushort(__float2half_rn(srow[e])));
          __syncwarp();
        }
      }
#pragma unroll
      for (int j = 0; j < C::KSTEPS; ++j) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[e] = 0.0f;
          if (g < G) {
            const uint16_t bits = lds_u16(qbuf_s + 2 * (g * D + kslot_d<D, KF>(c, j, e)));
            if constexpr (KVARN) {
              v[e] = __half2float(__ushort_as_half(bits));
            } else {
              v[e] = __uint_as_float(static_cast<uint32_t>(bits) << 16);
              if constexpr (KF != BF16) v[e] = __half2float(__float2half_rn(v[e]));
            }
          }
          qs += v[e];
          if (e >= 2) qh += v[e];
        }
        qf[j][0] = pack_op2<KF == BF16>(v[0], v[1]);  // exact (bf16 or its fp16 rounding)
        qf[j][1] = pack_op2<KF == BF16>(v[2], v[3]);
      }
      __syncwarp();  // every lane has read the rows: fetch the next segment's
      if (hd.next_s >= 0) prefetch_q(hd.next_s);
      // a query value that is not finite after its conversion (beyond fp16's
      // range for the quantized formats, or an infinity or NaN in the input)
      if (__any_sync(0xffffffffu, !isfinite(qs)) && lane == 0) raise_error(64u);  // KVQ_DEVERR_QUERY_RANGE
      qs += __shfl_xor_sync(0xffffffffu, qs, 1);
      qs += __shfl_xor_sync(0xffffffffu, qs, 2);
      qsum0 = __shfl_sync(0xffffffffu, qs, (2 * c) * 4);
      qsum1 = __shfl_sync(0xffffffffu, qs, (2 * c + 1) * 4);
      if constexpr (KF == INT4A) {  // offsets 1024 (low nibbles) and 64 (high nibbles)
        qh += __shfl_xor_sync(0xffffffffu, qh, 1);
        qh += __shfl_xor_sync(0xffffffffu, qh, 2);
        qb0 = fmaf(1024.0f, qsum0, -960.0f * __shfl_sync(0xffffffffu, qh, (2 * c) * 4));
        qb1 = fmaf(1024.0f, qsum1, -960.0f * __shfl_sync(0xffffffffu, qh, (2 * c + 1) * 4));
      } else {
        qb0 = 1024.0f * qsum0;
        qb1 = 1024.0f * qsum1;
      }
      m0 = m1 = -INFINITY;
      l0 = l1 = z0 = z1 = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) Oa[e] = Ob[e] = 0.f;
      seg_t0 = hd.t;
    }
    const int valid = hd.valid;

    // ---- K rows (and K metadata) of the stage into registers
    uint32_t kw[2][C::KW];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
#pragma unroll
      for (int pc = 0; pc < C::KP; ++pc) {
        if constexpr (C::KPS == 16) {
          const uint4 w = lds128(sb + k_addr[r][pc]);
          kw[r][pc * 4 + 0] = w.x; kw[r][pc * 4 + 1] = w.y;
          kw[r][pc * 4 + 2] = w.z; kw[r][pc * 4 + 3] = w.w;
        } else {
          const uint2 w = lds64(sb + k_addr[r][pc]);
          kw[r][pc * 2 + 0] = w.x; kw[r][pc * 2 + 1] = w.y;
        }
      }
    }
    float ks0 = 1.f, ks1 = 1.f, kz0 = 0.f, kz1 = 0.f, vs0 = 1.f, vs1 = 1.f, vz0 = 0.f, vz1 = 0.f;
    if constexpr (is_asym(KF)) {
      const uint32_t mk = sb + meta_k;
      ks0 = lds_half(mk + mrow0); ks1 = lds_half(mk + mrow1);
      kz0 = lds_half(mk + fstr + mrow0); kz1 = lds_half(mk + fstr + mrow1);
      if constexpr (KVARN) {
        const float sg0 = lds_half(mk + 2 * fstr + mrow0), sg1 = lds_half(mk + 2 * fstr + mrow1);
        ks0 *= sg0; kz0 *= sg0; ks1 *= sg1; kz1 *= sg1;
      }
    }
    if constexpr (KF == INT8) {
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int q = 0; q < C::KW; ++q) kw[r][q] ^= 0x80808080u;
    }
    // ---- S^T = K q^T (two accumulators halve the dependent mma chain)
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sbb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < C::KSTEPS; ++j) {
      uint32_t a0, a1, a2, a3;
      k_frag<KF, C::KW>(kw, j, a0, a1, a2, a3);
      if (j & 1) mma16816<KF == BF16>(sbb[0], sbb[1], sbb[2], sbb[3], a0, a1, a2, a3, qf[j][0], qf[j][1]);
      else mma16816<KF == BF16>(sa[0], sa[1], sa[2], sa[3], a0, a1, a2, a3, qf[j][0], qf[j][1]);
    }
    float sl[4];
    {
      float sacc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) sacc[q] = sa[q] + sbb[q];
      if constexpr (!is_asym(KF)) {
        constexpr float bias = KF == INT8 ? 1152.0f : 0.0f;
        sl[0] = (sacc[0] - bias * qsum0) * qks;
        sl[1] = (sacc[1] - bias * qsum1) * qks;
        sl[2] = (sacc[2] - bias * qsum0) * qks;
        sl[3] = (sacc[3] - bias * qsum1) * qks;
      } else {
        sl[0] = (ks0 * (sacc[0] - qb0) + kz0 * qsum0) * a.qk_scale;
        sl[1] = (ks0 * (sacc[1] - qb1) + kz0 * qsum1) * a.qk_scale;
        sl[2] = (ks1 * (sacc[2] - qb0) + kz1 * qsum0) * a.qk_scale;
        sl[3] = (ks1 * (sacc[3] - qb1) + kz1 * qsum1) * a.qk_scale;
      }
    }
    const bool ok0 = row0 < valid, ok1 = row1 < valid;
    if (!ok0) sl[0] = sl[1] = -INFINITY;
    if (!ok1) sl[2] = sl[3] = -INFINITY;

    // ---- V rows (and V metadata), then release the stage
    uint32_t vw[4][C::VW];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if constexpr (C::VPS == 16) {
        const uint4 w = lds128(sb + v_addr[u]);
        vw[u][0] = w.x; vw[u][1] = w.y; vw[u][2] = w.z; vw[u][3] = w.w;
      } else if constexpr (C::VPS == 32) {  // 16-bit values: chunks 2g and 2g+1, whose
        // swizzled addresses differ in bit 4 only (same 128-byte row)
        const uint4 w0 = lds128(sb + v_addr[u]);
        const uint4 w1 = lds128(sb + (v_addr[u] ^ 16u));
        vw[u][0] = w0.x; vw[u][1] = w0.y; vw[u][2] = w0.z; vw[u][3] = w0.w;
        vw[u][4] = w1.x; vw[u][5] = w1.y; vw[u][6] = w1.z; vw[u][7] = w1.w;
      } else if constexpr (C::VPS == 8) {
        const uint2 w = lds64(sb + v_addr[u]);
        vw[u][0] = w.x; vw[u][1] = w.y;
      } else {
        vw[u][0] = lds32(sb + v_addr[u]);
      }
    }
    if constexpr (is_asym(VF)) {
      const uint32_t mv = sb + meta_v;
      vs0 = lds_half(mv + mrow0); vs1 = lds_half(mv + mrow1);
      vz0 = lds_half(mv + fstr + mrow0); vz1 = lds_half(mv + fstr + mrow1);
      if constexpr (KVARN) {
        const float sg0 = lds_half(mv + 2 * fstr + mrow0), sg1 = lds_half(mv + 2 * fstr + mrow1);
        vs0 *= sg0; vz0 *= sg0; vs1 *= sg1; vz1 *= sg1;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_s + 8 * st);
    __syncwarp();

    if constexpr (VF == INT8) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int q = 0; q < C::VW; ++q) vw[u][q] ^= 0x80808080u;
    }
    if (valid < 16) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v_token(c, u) >= valid) {
#pragma unroll
          for (int q = 0; q < C::VW; ++q) vw[u][q] = (VF == INT8) ? 0x80808080u : 0u;
        }
    }


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
      for (int d = 0; d < C::DTILES; ++d) {
        Oa[2 * d] *= al0; Oa[2 * d + 1] *= al0;
        Ob[2 * d] *= al1; Ob[2 * d + 1] *= al1;
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
      if (!ok0) vs0 = vz0 = 0.f;
      if (!ok1) vs1 = vz1 = 0.f;
      z0 += pr[0] * vz0 + pr[2] * vz1;
      z1 += pr[1] * vz0 + pr[3] * vz1;
      pr[0] *= vs0; pr[1] *= vs0;
      pr[2] *= vs1; pr[3] *= vs1;
    }
    // ---- P^T operand: lane (g, c) needs head g at its 4 V tokens
    const uint32_t x0 = pack_op2<VF == BF16>(pr[0], pr[2]);  // head 2c, rows (g, g+8)
    const uint32_t x1 = pack_op2<VF == BF16>(pr[1], pr[3]);  // head 2c+1
    const int src0 = c * 4 + (g >> 1), src1 = (c + 4) * 4 + (g >> 1);
    const uint32_t u0 = __shfl_sync(0xffffffffu, x0, src0);
    const uint32_t u1 = __shfl_sync(0xffffffffu, x1, src0);
    const uint32_t u2 = __shfl_sync(0xffffffffu, x0, src1);
    const uint32_t u3 = __shfl_sync(0xffffffffu, x1, src1);
    const uint32_t b0 = (g & 1) ? u1 : u0;
    const uint32_t b1 = (g & 1) ? u3 : u2;
    // ---- O^T += V^T P^T
#pragma unroll
    for (int d = 0; d < C::DTILES; ++d) {
      uint32_t a0, a1, a2, a3;
      v_frag<VF, C::VW>(vw, d, a0, a1, a2, a3);
      mma16816<VF == BF16>(Oa[2 * d], Ob[2 * d], Oa[2 * d + 1], Ob[2 * d + 1], a0, a1, a2, a3, b0,
                           b1);
    }
    // refill this stage once every warp has read it.  Thread 0 waits for that at
    // the end of its own tile, not right after its own release: waiting there
    // held warp 0 behind the slowest warp on every tile, and with it the
    // refills (the others then polled for data): 7 % on a KVarN decode of 4 x 131k tokens.
    if (threadIdx.x == 0 && cur->i < n) {
      if (mbar_wait_or_abort(empty_s + 8 * st, phase, spin, abort_flag)) {
        issue(st);
      } else {
        raise_error(16u);  // KVQ_DEVERR_TIMEOUT
        *abort_flag = 1;
      }
    }
    __syncwarp();
    if (++st == C::STAGES) {
      st = 0;
      phase ^= 1u;
    }
    if (!(hd.flags & 2)) continue;

    // ================= end of this CTA's segment of sequence hd.s =================
    float L0 = l0, L1 = l1, Z0 = z0, Z1 = z1;
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) {
      L0 += __shfl_xor_sync(0xffffffffu, L0, o);
      L1 += __shfl_xor_sync(0xffffffffu, L1, o);
      Z0 += __shfl_xor_sync(0xffffffffu, Z0, o);
      Z1 += __shfl_xor_sync(0xffffffffu, Z1, o);
    }
    const bool whole = seg_t0 == 0 && hd.t == hd.tiles - 1;
    const int j = first_seg ? 0 : 1;
    first_seg = false;
    {  // normalised output (a partial slot holds acc / l too)
      const float sc0 = vsc / L0, sc1 = vsc / L1;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        Oa[e] = (Oa[e] + Z0) * sc0;
        Ob[e] = (Ob[e] + Z1) * sc1;
      }
    }
    if (whole) {  // the whole sequence lies in this range: write the output
      if constexpr (KVARN) {  // inverse rotation: x = d . (cR * H y)
        fwht_accum_rows<E>(Oa, g);
        fwht_accum_rows<E>(Ob, g);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int dd = g * E + e;
          const float sgn = (a.signs != nullptr && a.signs[dd] < 0) ? -1.f : 1.f;
          Oa[e] = __fmul_rn(Oa[e], a.cR) * sgn;
          Ob[e] = __fmul_rn(Ob[e], a.cR) * sgn;
        }
      }
      if (2 * c < G) store_bf16_run<E>(a.out + (out_row0 + 2 * c) * D + g * E, Oa);
      if (2 * c + 1 < G) store_bf16_run<E>(a.out + (out_row0 + 2 * c + 1) * D + g * E, Ob);
      continue;
    }

    // ---- part of a sequence: (m, l, acc) into this range's slot, then publish
    const size_t slot = ((static_cast<size_t>(k) * HG + hg) * 2 + j) * (hpc * G) + warp * G;
    if (2 * c < G) store_f16_run<E>(a.ws_acc + (slot + 2 * c) * D + g * E, Oa);
    if (2 * c + 1 < G) store_f16_run<E>(a.ws_acc + (slot + 2 * c + 1) * D + g * E, Ob);
    if (g == 0) {
      if (2 * c < G) *reinterpret_cast<float2*>(a.ws_ml + 2 * (slot + 2 * c)) = make_float2(m0, L0);
      if (2 * c + 1 < G)
        *reinterpret_cast<float2*>(a.ws_ml + 2 * (slot + 2 * c + 1)) = make_float2(m1, L1);
    }
    // the last warp to store its rows publishes the slot: each warp counts
    // itself in (the warp barrier orders its lanes' stores before lane 0's
    // release), and the one that completes the count fences and stores the
    // tag.  No warp waits for another, so a warp that gave up leaves the
    // count short and the slot unpublished.
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(done_warps + j, 1) == hpc - 1) {
        __threadfence();  // every warp's slot stores (seen through the count) before the tag
        st_relaxed_u64(a.tags + (static_cast<size_t>(k) * HG + hg) * 2 + j, a.epoch);
        scratch[12 + 2 * j] = hd.ps;
        scratch[13 + 2 * j] = (static_cast<long long>(hd.s) << 32) | hd.tiles;
        scratch[28 + j] = hd.lam;
      }
    }
    __syncwarp();
  }

  // ---- merges.  A CTA with a partial segment checks the tags of the sequence's
  // other ranges (store-then-fence-then-load: at least one range sees them
  // all) and the one that swaps the call's tag into the claim word merges.
  // A sequence over more than kTreeRanges ranges merges in two levels instead:
  // teams of kTeam consecutive ranges, each merged (by its member that wins the
  // team's claim) into the slot of its first range, then the teams (by the team
  // merger that sees every team's tag and wins the sequence's claim).
  __syncthreads();
  if (*abort_flag) {  // a wait gave up: publish and merge nothing; leave once the
    // copies already issued have landed: each thread's query-row prefetch, and
    // the bulk copies of the last STAGES tiles issued (the only ones that can
    // still be in flight; a withheld tile was never issued)
    cp_async_wait<0>();
    if (threadIdx.x == 0) {
      const int issued = cur->i;
      for (int t = issued > C::STAGES ? issued - C::STAGES : 0; t < issued; ++t) {
        if (t == reinterpret_cast<const int*>(scratch + 24)[0]) continue;
        mbar_wait(full_s + 8 * (t % C::STAGES), (t / C::STAGES) & 1, spin);
      }
    }
    return;
  }
  const long long Wm = scratch[0];
  const int bwm = static_cast<int>(scratch[30]);
  if (warp == pub) {
    __threadfence();
#pragma unroll 1
    for (int jj = 0; jj < 2; ++jj) {
      const long long info = scratch[13 + 2 * jj];
      if (info < 0) continue;
      const SeqSpan q{scratch[28 + jj], scratch[12 + 2 * jj],
                      static_cast<int>(info & 0xFFFFFFFFll), bwm};
      const int ka = first_range(a, Wm, q), kb = last_range(a, Wm, q);
      const bool tree = kb - ka + 1 > kTreeRanges;
      const int lo = tree ? ka + (k - ka) / kTeam * kTeam : ka;
      const int hi = tree ? min(kb, lo + kTeam - 1) : kb;
      bool done = true;
      for (int kk = lo + lane; kk <= hi; kk += 32) {
        if (kk == k || !holds_tiles(a, Wm, q, kk, kk + 1)) continue;  // this range, or an empty one
        if (ld_relaxed_u64(a.tags + slot_index(a, Wm, q, kk, HG, hg)) != a.epoch)
          done = false;
      }
      done = __all_sync(0xffffffffu, done);
      if (lane == 0) {  // one merge per sequence (per team)
        unsigned long long* claim =
            tree ? a.team_claims + slot_index(a, Wm, q, lo, HG, hg)
                 : a.claims + static_cast<size_t>(info >> 32) * HG + hg;
        if (!done || atomicExch(claim, a.epoch) == a.epoch) scratch[13 + 2 * jj] = -1;
      }
      __syncwarp();
    }
    __threadfence();
  }
  __syncthreads();
#pragma unroll 1
  for (int pm = 0; pm < 2; ++pm) {
    const long long info = scratch[13 + 2 * pm];
    if (info < 0) continue;
    const int s = static_cast<int>(info >> 32);
    const SeqSpan q{scratch[28 + pm], scratch[12 + 2 * pm], static_cast<int>(info & 0xFFFFFFFFll),
                    bwm};
    const int ka = first_range(a, Wm, q), kb = last_range(a, Wm, q);
    if (kb - ka + 1 <= kTreeRanges) {  // one level: every range's slot, straight to the output
      merge_slots<D, KVARN>(a, s, q, Wm, HG, hg, warp, lane, hpc, ka, 1, kb - ka + 1, kb, -1);
      continue;
    }
    const int nteams = (kb - ka) / kTeam + 1;
    const int lo = ka + (k - ka) / kTeam * kTeam, hi = min(kb, lo + kTeam - 1);
    const long long rep = slot_index(a, Wm, q, lo, HG, hg);
    merge_slots<D, KVARN>(a, s, q, Wm, HG, hg, warp, lane, hpc, lo, 1, hi - lo + 1, kb, rep);
    __syncthreads();  // every warp's rows of the team result are stored
    if (warp == pub) {
      if (lane == 0) {
        __threadfence();
        st_relaxed_u64(a.team_tags + rep, a.epoch);
      }
      __syncwarp();
      __threadfence();
      bool done = true;
      for (int t = lane; t < nteams; t += 32) {
        const int lo2 = ka + t * kTeam;
        if (lo2 == lo) continue;
        if (!holds_tiles(a, Wm, q, lo2, min(lo2 + kTeam, kb + 1))) continue;  // a team of empty ranges
        if (ld_relaxed_u64(a.team_tags + slot_index(a, Wm, q, lo2, HG, hg)) != a.epoch)
          done = false;
      }
      done = __all_sync(0xffffffffu, done);
      if (lane == 0)  // one final merge per sequence
        scratch[4 + pm] =
            done && atomicExch(a.claims + static_cast<size_t>(s) * HG + hg, a.epoch) != a.epoch;
      __syncwarp();
      __threadfence();
    }
    __syncthreads();
    if (scratch[4 + pm])
      merge_slots<D, KVARN>(a, s, q, Wm, HG, hg, warp, lane, hpc, ka, kTeam, nteams, kb, -1);
  }
}

}  // namespace kvq

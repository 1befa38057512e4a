// Quantize-and-scatter into the paged cache (write_to_paged_cache) for the
// symmetric formats, plus the per-tensor and per-kv-head scale calibration.
// The asymmetric formats and KVarN are in write_asym.cu.
//
// vLLM issue #4025 'Support for 4-bit KV Cache in paged-attention op',
// section 'methods', items 1-2 (scale / zero point, int4 storage in the
// paged-cache write); the INT8 cache with per-layer scales of the
// "vllm-int8-kv-cache-for-ampere-sm86" summary; FP8 e4m3 / e5m2 with a
// kv_scale from vLLM PR #4893 (item 1); the KVarN article's variance
// normalisation + Hadamard rotation before asymmetric codes ('Contexte
// Technique').
//
// Mapping: one warp per token.  A row (token, kv-head) of D bf16 values is
// held by D/8 consecutive lanes, 8 consecutive elements (16 bytes) each, so
// a warp covers 256/D rows per 16-byte load and every load and store is
// fully coalesced.  Per-row reductions (min / max / sums) are xor-butterflies
// inside the lane group.  HBM-bound: 2*D*2 bytes read and D or D/2 bytes
// (+ meta) written per row.
#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "quant_row.cuh"

namespace kvq {

KVQ_ERROR_ACCESSOR(take_error_bits_write)

namespace {

constexpr int kWriteWarps = 8;

template <int D, int KF, int VF, bool KVARN>
__global__ void __launch_bounds__(kWriteWarps * 32)
    write_cache_kernel(WriteArgs a) {
  constexpr int LPR = RowGeom<D>::LPR;
  constexpr int RPI = RowGeom<D>::RPI;
  constexpr int U = 4;  // row groups loaded before any is processed
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

  uint32_t sign_bits = 0;
  if constexpr (KVARN) {
    if (a.signs != nullptr) {
      const uint2 s = *reinterpret_cast<const uint2*>(a.signs + sub * 8);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t byte = ((i < 4 ? s.x : s.y) >> (8 * (i & 3))) & 0xFFu;
        sign_bits |= (byte & 0x80u) ? (1u << i) : 0u;
      }
    }
  }

  const uint16_t* krow = a.key + t * a.key_stride;
  const uint16_t* vrow = a.value + t * a.value_stride;
  const size_t row0 = (static_cast<size_t>(blk) * a.block_size + off) * Hkv;

  for (int h0 = 0; h0 < Hkv; h0 += RPI * U) {
    uint4 rk[U], rv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int h = h0 + u * RPI + grp;
      rk[u] = h < Hkv ? ldg_stream16(krow + h * D + sub * 8) : make_uint4(0, 0, 0, 0);
      rv[u] = h < Hkv ? ldg_stream16(vrow + h * D + sub * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int hb = h0 + u * RPI;
      if (hb >= Hkv) break;
      const int h = hb + grp;
      const bool act = h < Hkv;
      float x[8];
      // per-kv-head scales: 1/scale[h], correctly rounded like the host's division
      const float kinv = a.k_head_scale != nullptr && act ? __frcp_rn(a.k_head_scale[h]) : a.k_inv;
      const float vinv = a.v_head_scale != nullptr && act ? __frcp_rn(a.v_head_scale[h]) : a.v_inv;
      unpack8(rk[u], x);
      quantize_store<D, KF, KVARN>(x, act, h, sub, row0 + h, a.k_cache, a.k_meta, kinv, blk,
                                   off, Hkv, a.block_size, sign_bits, a.cR);
      unpack8(rv[u], x);
      quantize_store<D, VF, KVARN>(x, act, h, sub, row0 + h, a.v_cache, a.v_meta, vinv, blk,
                                   off, Hkv, a.block_size, sign_bits, a.cR);
    }
  }
}

// ---------------------------------------------------------------------------
// per-tensor absmax calibration
// ---------------------------------------------------------------------------
__global__ void absmax_kernel(const uint16_t* __restrict__ x, int64_t n, unsigned* out) {
  float m = 0.0f;
  const int64_t nvec = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
       i += stride) {
    const uint4 r = ldg_stream16(x + i * 8);
    float v[8];
    unpack8(r, v);
#pragma unroll
    for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(v[k]));
  }
  for (int64_t i = nvec * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride)
    m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(x[i]) << 16)));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(m));  // m >= 0: uint order
}

__global__ void scale_from_absmax_kernel(float* scale, float qmax) {
  const float amax = __uint_as_float(*reinterpret_cast<unsigned*>(scale));
  *scale = amax == 0.0f ? 1.0f : __fdiv_rn(amax, qmax);
}

// absmax per kv-head of x [T, Hkv, D] (row stride `stride`): one warp per
// (token, head) row pass over 8-element pieces, atomicMax per head.
__global__ void absmax_heads_kernel(const uint16_t* __restrict__ x, int64_t T, int hkv, int d,
                                    int64_t stride, unsigned* out) {
  const int pieces = d / 8;
  const int64_t total = T * hkv * pieces;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += step) {
    const int64_t row = i / pieces;
    const int pc = static_cast<int>(i - row * pieces);
    const int64_t t = row / hkv;
    const int h = static_cast<int>(row - t * hkv);
    const uint4 r = ldg_stream16(x + t * stride + static_cast<int64_t>(h) * d + pc * 8);
    float v[8];
    unpack8(r, v);
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(v[k]));
    atomicMax(out + h, __float_as_uint(m));  // m >= 0: unsigned order is float order
  }
}

__global__ void head_scales_from_absmax_kernel(float* scales, int hkv, float qmax) {
  for (int h = threadIdx.x; h < hkv; h += blockDim.x) {
    const float amax = __uint_as_float(reinterpret_cast<unsigned*>(scales)[h]);
    scales[h] = amax == 0.0f ? 1.0f : __fdiv_rn(amax, qmax);
  }
}

template <int D, int KF, int VF, bool KVARN>
cudaError_t launch_write_t(const WriteArgs& a, cudaStream_t st) {
  const int64_t blocks = (a.num_tokens + kWriteWarps - 1) / kWriteWarps;
  write_cache_kernel<D, KF, VF, KVARN><<<static_cast<unsigned>(blocks), kWriteWarps * 32, 0, st>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_write_d(const WriteArgs& a, int kf, int vf, bool kvarn, cudaStream_t st) {
#define KVQ_W(KF_, VF_, KV_) \
  if (kf == KF_ && vf == VF_ && kvarn == KV_) return launch_write_t<D, KF_, VF_, KV_>(a, st);
  KVQ_W(INT8, INT8, false)
  KVQ_W(INT8, E4M3, false)
  KVQ_W(INT8, E5M2, false)
  KVQ_W(E4M3, INT8, false)
  KVQ_W(E4M3, E4M3, false)
  KVQ_W(E4M3, E5M2, false)
  KVQ_W(E5M2, INT8, false)
  KVQ_W(E5M2, E4M3, false)
  KVQ_W(E5M2, E5M2, false)
  KVQ_W(BF16, BF16, false)
#undef KVQ_W
  return cudaErrorNotSupported;
}

}  // namespace

bool write_supported(int kf, int vf, bool kvarn) {
  const bool sym_k = !is_asym(kf), sym_v = !is_asym(vf);
  if (kvarn) return !sym_k && !sym_v;
  return sym_k == sym_v;
}

cudaError_t launch_write(const WriteArgs& a, int head_dim, int kf, int vf, bool kvarn,
                         cudaStream_t st) {
  if (is_asym(kf) || is_asym(vf)) return launch_write_asym(a, head_dim, kf, vf, kvarn, st);
  if (head_dim == 64) return dispatch_write_d<64>(a, kf, vf, kvarn, st);
  if (head_dim == 128) return dispatch_write_d<128>(a, kf, vf, kvarn, st);
  return cudaErrorNotSupported;
}

cudaError_t launch_calibrate_heads(const uint16_t* x, int64_t num_tokens, int hkv, int d,
                                   int64_t stride, float qmax, float* scales, cudaStream_t st,
                                   int num_sms) {
  cudaError_t e = cudaMemsetAsync(scales, 0, sizeof(float) * hkv, st);
  if (e != cudaSuccess) return e;
  const int64_t total = num_tokens * hkv * (d / 8);
  if (total > 0) {
    const int64_t want = (total + 255) / 256;
    const int blocks = static_cast<int>(want < 4LL * num_sms ? want : 4LL * num_sms);
    absmax_heads_kernel<<<blocks, 256, 0, st>>>(x, num_tokens, hkv, d, stride,
                                                 reinterpret_cast<unsigned*>(scales));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  head_scales_from_absmax_kernel<<<1, 256, 0, st>>>(scales, hkv, qmax);
  return cudaGetLastError();
}

cudaError_t launch_calibrate(const uint16_t* x, int64_t n, float qmax, float* scale,
                             cudaStream_t st, int num_sms) {
  cudaError_t e = cudaMemsetAsync(scale, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  if (n > 0) {
    const int64_t want = (n / 8 + 255) / 256;
    const int blocks = static_cast<int>(want < 4LL * num_sms ? (want > 0 ? want : 1) : 4LL * num_sms);
    absmax_kernel<<<blocks, 256, 0, st>>>(x, n, reinterpret_cast<unsigned*>(scale));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  scale_from_absmax_kernel<<<1, 1, 0, st>>>(scale, qmax);
  return cudaGetLastError();
}

}  // namespace kvq

// Standalone in-place orthonormal Walsh-Hadamard rotation of rows (the
// rotation of the KVarN article, 'Contexte Technique').  A row of D values is
// held by D/8 consecutive lanes, 8 consecutive elements each (float32: two
// 16-byte loads; bf16: one); the butterfly order is the one the cache write
// uses, so the result is bit-identical to a float32 restatement.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

template <int D, bool BF16, bool INV>
__global__ void __launch_bounds__(256) hadamard_kernel(void* x, int64_t rows, const int8_t* signs,
                                                       float cR) {
  constexpr int LPR = D / 8, RPW = 32 / LPR;
  const int lane = threadIdx.x & 31, sub = lane % LPR, grp = lane / LPR;
  uint32_t sign_bits = 0;
  if (signs != nullptr) {
    const uint2 sv = *reinterpret_cast<const uint2*>(signs + sub * 8);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = ((i < 4 ? sv.x : sv.y) >> (8 * (i & 3))) & 0xFFu;
      sign_bits |= (byte & 0x80u) ? (1u << i) : 0u;
    }
  }
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       w * RPW < rows; w += warps) {
    const int64_t row = w * RPW + grp;
    const bool act = row < rows;
    float v[8];
    if constexpr (BF16) {
      uint16_t* p = static_cast<uint16_t*>(x) + row * D + sub * 8;
      uint4 r = act ? *reinterpret_cast<const uint4*>(p) : make_uint4(0, 0, 0, 0);
      v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x); v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
      v[4] = bf16_lo(r.z); v[5] = bf16_hi(r.z); v[6] = bf16_lo(r.w); v[7] = bf16_hi(r.w);
    } else {
      float* p = static_cast<float*>(x) + row * D + sub * 8;
      float4 r0 = act ? reinterpret_cast<const float4*>(p)[0] : make_float4(0, 0, 0, 0);
      float4 r1 = act ? reinterpret_cast<const float4*>(p)[1] : make_float4(0, 0, 0, 0);
      v[0] = r0.x; v[1] = r0.y; v[2] = r0.z; v[3] = r0.w;
      v[4] = r1.x; v[5] = r1.y; v[6] = r1.z; v[7] = r1.w;
    }
    if (!INV) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = ((sign_bits >> i) & 1u) ? -v[i] : v[i];
    }
    fwht_lanes<8, LPR>(v, sub);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = __fmul_rn(v[i], cR);
      if (INV) v[i] = ((sign_bits >> i) & 1u) ? -v[i] : v[i];
    }
    if (!act) continue;
    if constexpr (BF16) {
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        o[k] = *reinterpret_cast<uint32_t*>(&b);
      }
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(x) + row * D + sub * 8) =
          make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      float* p = static_cast<float*>(x) + row * D + sub * 8;
      reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
      reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

template <int D>
cudaError_t launch_d(void* x, int dtype, int64_t rows, const int8_t* signs, int inverse, float cR,
                     cudaStream_t st) {
  constexpr int RPW = 32 / (D / 8);
  const int64_t warps_needed = (rows + RPW - 1) / RPW;
  const int64_t blocks64 = (warps_needed + 7) / 8;
  const unsigned blocks = static_cast<unsigned>(blocks64 < 65536 ? blocks64 : 65536);
  if (dtype == 1) {
    if (inverse) hadamard_kernel<D, true, true><<<blocks, 256, 0, st>>>(x, rows, signs, cR);
    else hadamard_kernel<D, true, false><<<blocks, 256, 0, st>>>(x, rows, signs, cR);
  } else {
    if (inverse) hadamard_kernel<D, false, true><<<blocks, 256, 0, st>>>(x, rows, signs, cR);
    else hadamard_kernel<D, false, false><<<blocks, 256, 0, st>>>(x, rows, signs, cR);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_hadamard(void* x, int dtype, int64_t rows, int head_dim, const int8_t* signs,
                            int inverse, float cR, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  switch (head_dim) {
    case 64: return launch_d<64>(x, dtype, rows, signs, inverse, cR, st);
    case 128: return launch_d<128>(x, dtype, rows, signs, inverse, cR, st);
    case 256: return launch_d<256>(x, dtype, rows, signs, inverse, cR, st);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace kvq

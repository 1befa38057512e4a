// Launch of the decode kernel for one template instance: TMA descriptors of the
// caller's cache arrays, then one launch (the last CTA of each sequence and
// head group merges its partitions).
#pragma once

#include <cudaTypedefs.h>

#include <atomic>

#include "decode.cuh"

namespace kvq {

// cuTensorMapEncodeTiled, fetched once through the runtime (no libcuda link).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

inline CUtensorMapSwizzle swizzle_mode(int bits) {
  return bits == 3 ? CU_TENSOR_MAP_SWIZZLE_128B
                   : bits == 2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE;
}

// Codes [NB, bs, Hkv, row] bytes: dims (row, Hkv, bs, NB), box = one head's
// 16 tokens (8 with 8-token pages: one page).  A row over 128 bytes (16-bit
// values) is two 128-byte halves: dims (128, 2, Hkv, bs, NB).
inline bool encode_codes_map(CUtensorMap* m, const void* base, int row, int hkv, int bs, int nb,
                             int swz_bits) {
  if (row > 128) {
    const cuuint64_t dims[5] = {128, cuuint64_t(row / 128), cuuint64_t(hkv), cuuint64_t(bs),
                                cuuint64_t(nb)};
    const cuuint64_t strides[4] = {128, cuuint64_t(row), cuuint64_t(row) * hkv,
                                   cuuint64_t(row) * hkv * bs};
    const cuuint32_t box[5] = {128, cuuint32_t(row / 128), 1, cuuint32_t(bs < 16 ? bs : 16), 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return tensor_map_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle_mode(swz_bits), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t dims[4] = {cuuint64_t(row), cuuint64_t(hkv), cuuint64_t(bs), cuuint64_t(nb)};
  const cuuint64_t strides[3] = {cuuint64_t(row), cuuint64_t(row) * hkv,
                                 cuuint64_t(row) * hkv * bs};
  const cuuint32_t box[4] = {cuuint32_t(row), 1, cuuint32_t(bs < 16 ? bs : 16), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return tensor_map_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle_mode(swz_bits), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Codes again, dims ordered (row, bs, Hkv, NB): one box of 16 tokens x hpc heads
// lands head-major ([head][token][row]) in shared memory, the layout of hpc
// single-head boxes, with one TMA instead of hpc.  Every address it can reach is
// inside the cache; if the encoder rejects the ordering, per-head boxes are used.
inline bool encode_codes_map_headmajor(CUtensorMap* m, const void* base, int row, int hkv, int bs,
                                       int nb, int hpc, int swz_bits) {
  if (row > 128) {  // two 128-byte halves per row: dims (128, 2, bs, Hkv, NB)
    const cuuint64_t dims[5] = {128, cuuint64_t(row / 128), cuuint64_t(bs), cuuint64_t(hkv),
                                cuuint64_t(nb)};
    const cuuint64_t strides[4] = {128, cuuint64_t(row) * hkv, cuuint64_t(row),
                                   cuuint64_t(row) * hkv * bs};
    const cuuint32_t box[5] = {128, cuuint32_t(row / 128), 16, cuuint32_t(hpc), 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return tensor_map_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle_mode(swz_bits), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t dims[4] = {cuuint64_t(row), cuuint64_t(bs), cuuint64_t(hkv), cuuint64_t(nb)};
  const cuuint64_t strides[3] = {cuuint64_t(row) * hkv, cuuint64_t(row),
                                 cuuint64_t(row) * hkv * bs};
  const cuuint32_t box[4] = {cuuint32_t(row), 16, cuuint32_t(hpc), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return tensor_map_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle_mode(swz_bits), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Metadata [NB, Hkv, F, bs] fp16: dims (bs, F, Hkv, NB), box = 16 tokens x F x hpc
// (8 tokens with 8-token pages).
inline bool encode_meta_map(CUtensorMap* m, const void* base, int nf, int hkv, int bs, int nb,
                            int hpc) {
  const cuuint64_t dims[4] = {cuuint64_t(bs), cuuint64_t(nf), cuuint64_t(hkv), cuuint64_t(nb)};
  const cuuint64_t strides[3] = {cuuint64_t(bs) * 2, cuuint64_t(bs) * 2 * nf,
                                 cuuint64_t(bs) * 2 * nf * hkv};
  const cuuint32_t box[4] = {cuuint32_t(bs < 16 ? bs : 16), cuuint32_t(nf), cuuint32_t(hpc), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return tensor_map_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int KF, int VF, bool KVARN>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t st) {
  using C = DecodeCfg<D, KF, VF, KVARN>;
  if (tensor_map_encoder() == nullptr) return cudaErrorNotSupported;
  DecodeMaps<kMaxPageClasses> maps;
  memset(&maps, 0, sizeof(maps));
  const int hpc = a.heads_per_cta;
  DecodeArgs args = a;
  // one head-major box per tile when every class's codes allow it (pages of 16
  // tokens or more), else per-head boxes (8-token pages take two per head: they
  // land as one head's 16 rows)
  args.one_box = 1;
  for (int c = 0; c < a.num_classes; ++c) {
    const int bs = 1 << a.block_shift[c];
    args.one_box = args.one_box && bs >= 16 &&
                   encode_codes_map_headmajor(&maps.k[c], a.k_cache[c], C::KB, a.num_kv_heads, bs,
                                              a.num_blocks[c], hpc, C::K_SWZ) &&
                   encode_codes_map_headmajor(&maps.v[c], a.v_cache[c], C::VB, a.num_kv_heads, bs,
                                              a.num_blocks[c], hpc, C::V_SWZ);
  }
  for (int c = 0; c < a.num_classes; ++c) {
    const int bs = 1 << a.block_shift[c];
    if (!args.one_box &&
        (!encode_codes_map(&maps.k[c], a.k_cache[c], C::KB, a.num_kv_heads, bs, a.num_blocks[c],
                           C::K_SWZ) ||
         !encode_codes_map(&maps.v[c], a.v_cache[c], C::VB, a.num_kv_heads, bs, a.num_blocks[c],
                           C::V_SWZ)))
      return cudaErrorInvalidValue;
    if (C::KMF > 0 && !encode_meta_map(&maps.km[c], a.k_meta[c], C::KMF, a.num_kv_heads, bs,
                                       a.num_blocks[c], hpc))
      return cudaErrorInvalidValue;
    if (C::VMF > 0 && !encode_meta_map(&maps.vm[c], a.v_meta[c], C::VMF, a.num_kv_heads, bs,
                                       a.num_blocks[c], hpc))
      return cudaErrorInvalidValue;
  }

  auto kern_one = decode_partition_kernel<D, KF, VF, KVARN, kPagesOne>;
  auto kern_split = decode_partition_kernel<D, KF, VF, KVARN, kPages8>;
  auto kern_mixed = decode_partition_kernel<D, KF, VF, KVARN, kPagesMixed>;
  const int smem = decode_smem_bytes<C>(hpc, a.gqa);
  static std::atomic<unsigned long long> attr_done{0};  // one bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_done.load() & bit)) {
    const int most = decode_smem_bytes<C>(kHeadsPerCta, 8);
    for (const void* k : {reinterpret_cast<const void*>(kern_one),
                          reinterpret_cast<const void*>(kern_split),
                          reinterpret_cast<const void*>(kern_mixed)}) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
      if (e != cudaSuccess) return e;
    }
    attr_done.fetch_or(bit);
  }
  const dim3 grid(a.num_ctas, a.num_kv_heads / hpc, 1);
  if (a.seq_class != nullptr) {  // a class array: the mixed instance (pages of 16 or more)
    kern_mixed<<<grid, hpc * 32, smem, st>>>(args, maps);
  } else {  // one pool: class 0's maps only
    DecodeMaps<1> one;
    one.k[0] = maps.k[0];
    one.v[0] = maps.v[0];
    one.km[0] = maps.km[0];
    one.vm[0] = maps.vm[0];
    if (a.block_shift[0] < 4)
      kern_split<<<grid, hpc * 32, smem, st>>>(args, one);
    else
      kern_one<<<grid, hpc * 32, smem, st>>>(args, one);
  }
  return cudaGetLastError();
}

}  // namespace kvq

// Launch of the decode kernel for one template instance (one launch: the last
// CTA of each (sequence, kv-head) merges its partitions).
#pragma once

#include <atomic>

#include "decode.cuh"

namespace kvq {

template <int D, int KF, int VF, bool KVARN>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t st) {
  using C = DecodeCfg<D, KF, VF, KVARN>;
  auto kern = decode_partition_kernel<D, KF, VF, KVARN>;
  static std::atomic<unsigned long long> attr_done{0};  // one bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_done.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit);
  }
  const dim3 grid(a.num_kv_heads, a.num_seqs, a.num_partitions);
  kern<<<grid, kDecodeWarps * 32, C::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq

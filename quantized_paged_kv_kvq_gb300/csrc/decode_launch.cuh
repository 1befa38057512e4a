// Launch of the decode partition kernel (+ the log-sum-exp combine when a
// sequence spans several partitions) for one template instance.
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
  if (a.phase & 1) {
    const dim3 grid(a.num_kv_heads, a.num_seqs, a.num_partitions);
    kern<<<grid, kDecodeWarps * 32, C::SMEM, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if ((a.phase & 2) && a.num_partitions > 1) {
    decode_reduce_kernel<D, KVARN><<<dim3(a.num_q_heads, a.num_seqs), 256, 0, st>>>(a);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace kvq

// Decode instances: head_dim 128, INT8 keys (values INT8 / E4M3 / E5M2).
// One translation unit per group of instances keeps the build parallel.
#include "decode_launch.cuh"

namespace kvq {

KVQ_ERROR_ACCESSOR(take_error_bits_decode_d128_sym)

cudaError_t launch_decode_d128_sym(const DecodeArgs& a, int head_dim, int kf, int vf, bool kvarn,
                                   cudaStream_t st) {
  if (head_dim != 128) return cudaErrorNotSupported;
#define KVQ_D(KF_, VF_, KV_) \
  if (kf == KF_ && vf == VF_ && kvarn == KV_) return launch_decode_t<128, KF_, VF_, KV_>(a, st);
  KVQ_D(INT8, INT8, false)
  KVQ_D(INT8, E4M3, false)
  KVQ_D(INT8, E5M2, false)
#undef KVQ_D
  return cudaErrorNotSupported;
}

}  // namespace kvq

// Decode instances: head_dim 64, per-token asymmetric formats (INT4 / UINT8).
// One translation unit per group of instances keeps the build parallel.
#include "decode_launch.cuh"

namespace kvq {

KVQ_ERROR_ACCESSOR(take_error_bits_decode_d64_asym)

cudaError_t launch_decode_d64_asym(const DecodeArgs& a, int head_dim, int kf, int vf, bool kvarn,
                                   cudaStream_t st) {
  if (head_dim != 64) return cudaErrorNotSupported;
#define KVQ_D(KF_, VF_, KV_) \
  if (kf == KF_ && vf == VF_ && kvarn == KV_) return launch_decode_t<64, KF_, VF_, KV_>(a, st);
  KVQ_D(INT4A, INT4A, false)
  KVQ_D(INT4A, UINT8A, false)
  KVQ_D(UINT8A, INT4A, false)
  KVQ_D(UINT8A, UINT8A, false)
#undef KVQ_D
  return cudaErrorNotSupported;
}

}  // namespace kvq

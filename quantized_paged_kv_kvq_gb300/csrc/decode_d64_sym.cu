// Decode instances: head_dim 64, per-tensor-scale formats (INT8 / E4M3 / E5M2).
#include "decode_launch.cuh"

namespace kvq {

KVQ_ERROR_ACCESSOR(take_error_bits_decode_d64_sym)

cudaError_t launch_decode_d64_sym(const DecodeArgs& a, int kf, int vf, cudaStream_t st) {
#define KVQ_D(KF_, VF_) \
  if (kf == KF_ && vf == VF_) return launch_decode_t<64, KF_, VF_, false>(a, st);
  KVQ_D(INT8, INT8)
  KVQ_D(INT8, E4M3)
  KVQ_D(INT8, E5M2)
  KVQ_D(E4M3, INT8)
  KVQ_D(E4M3, E4M3)
  KVQ_D(E4M3, E5M2)
  KVQ_D(E5M2, INT8)
  KVQ_D(E5M2, E4M3)
  KVQ_D(E5M2, E5M2)
#undef KVQ_D
  return cudaErrorNotSupported;
}

}  // namespace kvq

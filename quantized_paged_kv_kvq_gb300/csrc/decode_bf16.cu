// Decode instances for the unquantized 16-bit cache (bf16 K and V; PR #4893
// 'Load FP8 kv-cache scaling factors from checkpoints', item 1: with
// --kv-cache-dtype auto the cache keeps the model's 16-bit values), head_dim
// 64 and 128.
#include "decode_launch.cuh"

namespace kvq {

KVQ_ERROR_ACCESSOR(take_error_bits_decode_bf16)

cudaError_t launch_decode_bf16(const DecodeArgs& a, int head_dim, int kf, int vf, bool kvarn,
                               cudaStream_t st) {
  if (kf != BF16 || vf != BF16 || kvarn) return cudaErrorNotSupported;
  if (head_dim == 64) return launch_decode_t<64, BF16, BF16, false>(a, st);
  if (head_dim == 128) return launch_decode_t<128, BF16, BF16, false>(a, st);
  return cudaErrorNotSupported;
}

}  // namespace kvq

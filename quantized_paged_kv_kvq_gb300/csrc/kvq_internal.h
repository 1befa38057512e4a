// Internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

// Most stream-K ranges (CTAs per head group) of one decode launch.
constexpr int kMaxCtas = 65535;
// Most kv-heads (consumer warps) per decode CTA.
constexpr int kHeadsPerCtaHost = 8;

struct WriteArgs {
  const uint16_t* key;    // bf16 bits
  const uint16_t* value;  // bf16 bits
  int64_t key_stride;     // elements between tokens
  int64_t value_stride;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  uint8_t* k_cache;
  uint8_t* v_cache;
  __half* k_meta;
  __half* v_meta;
  int num_kv_heads;
  int block_size;
  int block_shift;  // log2(block_size)
  int num_blocks;
  float k_inv;  // 1/k_scale (symmetric formats)
  float v_inv;
  const float* k_head_scale;  // per-kv-head scales or nullptr (then k_inv / v_inv)
  const float* v_head_scale;
  const int8_t* signs;
  float cR;  // float(1/sqrt(head_dim))
};

// Page classes of one decode call (pools of pages of one size each).
constexpr int kMaxPageClasses = 2;

struct DecodeArgs {
  // The cache: one pool per page class (its codes, metadata, page size and
  // block count); a cache of one page size has one.  seq_class[s] is the class
  // of sequence s (nullptr: class 0), whose block ids index that pool.
  const uint8_t* k_cache[kMaxPageClasses];
  const uint8_t* v_cache[kMaxPageClasses];
  const __half* k_meta[kMaxPageClasses];
  const __half* v_meta[kMaxPageClasses];
  int block_shift[kMaxPageClasses];  // log2(page size)
  int num_blocks[kMaxPageClasses];
  const uint8_t* seq_class;
  int num_classes;
  const uint16_t* query;  // bf16 [S, Hq, D]
  uint16_t* out;          // bf16 [S, Hq, D]
  const int32_t* block_table;
  const int32_t* context_lens;
  const int8_t* signs;
  __half* ws_acc;  // [NC, head groups, 2, heads per group, D]: partial outputs acc / l (fp16)
  float* ws_ml;   // [NC, head groups, 2, heads per group, 2]: partial (max, sum)
  unsigned long long* tags;    // [NC, head groups, 2]: the call's tag once a slot is written
  unsigned long long* team_tags;    // [NC, head groups, 2]: set once a team of ranges is merged
  unsigned long long* team_claims;  // [NC, head groups, 2]: claim of a team's merge
  unsigned long long* claims;       // [S, head groups]: claim of a sequence's final merge
  unsigned long long epoch;    // nonzero tag of this call
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int gqa;
  int heads_per_cta;  // kv-heads per CTA (= consumer warps), divides num_kv_heads
  int one_box;        // K / V tile loaded head-major by one TMA each (else per head)
  int max_blocks_per_seq;
  int max_context_len;
  int num_ctas;          // NC: stream-K ranges (CTAs per head group)
  float qk_scale;        // sm_scale * log2(e) [* k_scale for symmetric K]
  float v_scale;         // symmetric V: multiplies the output
  float qk_base;         // sm_scale * log2(e)
  const float* k_head_scale;  // per-kv-head scales or nullptr (then qk_scale / v_scale)
  const float* v_head_scale;
  float cR;
  // New-token append (kvq_decode_append); new_key == nullptr for a plain decode.
  // The token at position context_lens[s] - 1 of sequence s comes from row s
  // of new_key / new_value (bf16 [S, Hkv, D], row strides in elements).
  const uint16_t* new_key;
  const uint16_t* new_value;
  int64_t new_key_stride;
  int64_t new_value_stride;
  uint8_t* k_cache_w[kMaxPageClasses];  // the same pools, writable
  uint8_t* v_cache_w[kMaxPageClasses];
  __half* k_meta_w[kMaxPageClasses];
  __half* v_meta_w[kMaxPageClasses];
  float k_inv;  // 1/k_scale (symmetric formats, per-tensor scales)
  float v_inv;
  // Bounded pipeline waits: polls of an mbarrier before the CTA gives up (sets
  // KVQ_DEVERR_TIMEOUT and returns).  Test hook: CTA (withhold_cta, head group
  // 0) never issues the loads of its tile withhold_tile (-1: none), so that a
  // wait runs out with nothing in flight.
  int spin_limit;
  int withhold_cta;
  int withhold_tile;
};

cudaError_t launch_write(const WriteArgs& a, int head_dim, int kf, int vf, bool kvarn,
                         cudaStream_t st);
cudaError_t launch_write_asym(const WriteArgs& a, int head_dim, int kf, int vf, bool kvarn,
                              cudaStream_t st);
bool write_supported(int kf, int vf, bool kvarn);

// Decode launchers, one per translation unit of kernel instances: each returns
// cudaErrorNotSupported for a (head_dim, formats, KVarN) it does not hold.
using DecodeLauncher = cudaError_t (*)(const DecodeArgs& a, int head_dim, int kf, int vf,
                                       bool kvarn, cudaStream_t st);
#define KVQ_DECODE_UNITS(X) \
  X(decode_d64_sym)         \
  X(decode_d64_fp8k)        \
  X(decode_d64_asym)        \
  X(decode_d64_kvarn)       \
  X(decode_d128_sym)        \
  X(decode_d128_fp8k)       \
  X(decode_d128_asym)       \
  X(decode_d128_kvarn)      \
  X(decode_bf16)
#define KVQ_DECLARE_UNIT(U)                                                                  \
  cudaError_t launch_##U(const DecodeArgs& a, int head_dim, int kf, int vf, bool kvarn,      \
                         cudaStream_t st);                                                   \
  cudaError_t take_error_bits_##U(unsigned* bits);
KVQ_DECODE_UNITS(KVQ_DECLARE_UNIT)
#undef KVQ_DECLARE_UNIT

// read-and-clear of the write units' device error words
cudaError_t take_error_bits_write(unsigned* bits);
cudaError_t take_error_bits_write_asym(unsigned* bits);

cudaError_t launch_hadamard(void* x, int dtype, int64_t rows, int head_dim, const int8_t* signs,
                            int inverse, float cR, cudaStream_t st);

cudaError_t launch_calibrate(const uint16_t* x, int64_t n, float qmax, float* scale,
                             cudaStream_t st, int num_sms);
cudaError_t launch_calibrate_heads(const uint16_t* x, int64_t num_tokens, int hkv, int d,
                                   int64_t stride, float qmax, float* scales, cudaStream_t st,
                                   int num_sms);

}  // namespace kvq

// C ABI of libkvq.so: host-side argument validation and the stream-ordered
// launcher (kernel variant and grid from format, head_dim, GQA ratio and
// context length).  No allocation, no per-call state.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <chrono>

#include "../../include/kvq.h"
#include "kvq_device.cuh"
#include "kvq_internal.h"

using namespace kvq;

namespace {

constexpr float kLog2e = 1.4426950408889634f;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_fmt(int f) { return f >= KVQ_FMT_INT8 && f <= KVQ_FMT_BF16; }

// Families that share a kernel: per-tensor-scaled 8-bit codes, per-row
// asymmetric codes (optionally KVarN), and the 16-bit cache (K and V both).
bool pairing_ok(int kf, int vf, bool kvarn) {
  if ((kf == KVQ_FMT_BF16) != (vf == KVQ_FMT_BF16)) return false;
  const bool ak = is_asym(kf), av = is_asym(vf);
  if (kvarn) return ak && av;
  return ak == av;
}
bool scaled(int f) { return !is_asym(f) && f != KVQ_FMT_BF16; }

// Checks shared by write and decode on the cache description.
kvq_status check_cache(const kvq_cache_desc* c) {
  if (c == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (!valid_fmt(c->k_fmt) || !valid_fmt(c->v_fmt)) return KVQ_ERR_INVALID_ARGUMENT;
  if (c->num_kv_heads < 1 || c->num_blocks < 1 || c->block_size < 1 || c->head_dim < 1)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (c->flags & ~KVQ_FLAG_VARNORM_ROTATE) return KVQ_ERR_INVALID_ARGUMENT;
  if (c->head_dim != 64 && c->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  // a power of two from 8 to 128: a 16-token tile lies in one block, or in two
  // consecutive entries of the block table (8-token pages)
  if (c->block_size != 8 && c->block_size != 16 && c->block_size != 32 && c->block_size != 64 &&
      c->block_size != 128)
    return KVQ_ERR_UNSUPPORTED;
  const bool kvarn = (c->flags & KVQ_FLAG_VARNORM_ROTATE) != 0;
  if (!pairing_ok(c->k_fmt, c->v_fmt, kvarn)) return KVQ_ERR_UNSUPPORTED;
  if (scaled(c->k_fmt) && !(c->k_scale > 0.0f && isfinite(c->k_scale)))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (scaled(c->v_fmt) && !(c->v_scale > 0.0f && isfinite(c->v_scale)))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (is_asym(c->k_fmt) && (c->k_meta == nullptr || !aligned(c->k_meta, 16)))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (is_asym(c->v_fmt) && (c->v_meta == nullptr || !aligned(c->v_meta, 16)))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (kvarn && c->signs != nullptr && !aligned(c->signs, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  // per-kv-head scales: scaled symmetric formats only
  if (c->k_head_scales != nullptr && (!scaled(c->k_fmt) || !aligned(c->k_head_scales, 4)))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (c->v_head_scales != nullptr && (!scaled(c->v_fmt) || !aligned(c->v_head_scales, 4)))
    return KVQ_ERR_INVALID_ARGUMENT;
  return KVQ_OK;
}

float rotation_scale(int d) { return static_cast<float>(1.0 / sqrt(static_cast<double>(d))); }

// SM count of the current device, cached per device.
int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  int v = (dev >= 0 && dev < 64) ? cache[dev].load() : 0;
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) cache[dev].store(v);
  return v;
}

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

int heads_per_cta(int hkv) { return hkv < 8 ? hkv : 8; }

// Stream-K ranges per head group: as many as the decode kernel has resident
// CTAs (two per SM; one for the 16-bit cache, whose 64 KB stages fill an
// SM's shared memory), at most one per possible tile.
int auto_ctas(int num_seqs, int max_ctx, int head_groups, int sms, int per_sm) {
  const long long tiles_max = static_cast<long long>(num_seqs) * ((max_ctx + 15) / 16);
  long long nc =
      (static_cast<long long>(sms > 0 ? sms : 152) * per_sm + head_groups - 1) / head_groups;
  if (nc > tiles_max) nc = tiles_max;
  if (nc > kMaxCtas) nc = kMaxCtas;
  return static_cast<int>(nc < 1 ? 1 : nc);
}

// Workspace: per (range, head group, first/last segment of the range, head) a
// partial output of D fp16 (acc / l) and its (max, sum) in f32; per (range,
// head group, first/last segment) three 64-bit words (completion tag, team
// tag, team claim); per (sequence, head group) a 64-bit merge claim.  One
// range needs none.
size_t workspace_bytes_for(int num_seqs, int hq, int hkv, int d, int nc) {
  if (nc <= 1) return 0;
  const size_t rows = static_cast<size_t>(nc) * 2 * hq;
  const size_t groups = static_cast<size_t>(hkv / heads_per_cta(hkv));
  return rows * (d * 2 + 2 * sizeof(float)) + static_cast<size_t>(nc) * groups * 2 * 8 * 3 +
         static_cast<size_t>(num_seqs) * groups * 8;
}

// Test hook of the bounded pipeline waits (kvq_debug_arm_wait_timeout): armed
// for the next decode launch of the process only.
std::atomic<int> g_wait_hook_armed{0};
std::atomic<int> g_wait_hook_polls{0};
std::atomic<int> g_wait_hook_cta{-1};
std::atomic<int> g_wait_hook_tile{-1};

// Polls of an mbarrier before a decode CTA gives up (the kernel's default).
constexpr int kDefaultSpinLimit = 1 << 22;

// Nonzero 64-bit tag, different for every decode call of the process, so that
// the completion tags never need clearing between calls.
unsigned long long next_epoch() {
  static std::atomic<unsigned long long> counter{0};
  static const unsigned long long base = [] {
    unsigned long long x = static_cast<unsigned long long>(
        std::chrono::steady_clock::now().time_since_epoch().count());
    x ^= reinterpret_cast<uintptr_t>(&counter) * 0x9E3779B97F4A7C15ull;
    return x;
  }();
  const unsigned long long e = base + counter.fetch_add(1);
  return e == 0 ? 1 : e;
}

kvq_status decode_shape(const kvq_cache_desc* c, int32_t num_seqs, int32_t num_q_heads,
                        int32_t max_context_len, int32_t num_ctas, int* NC) {
  kvq_status st = check_cache(c);
  if (st != KVQ_OK) return st;
  if (num_seqs < 0 || num_q_heads < 1 || max_context_len < 0) return KVQ_ERR_INVALID_ARGUMENT;
  if (num_q_heads % c->num_kv_heads) return KVQ_ERR_INVALID_ARGUMENT;
  if (num_q_heads / c->num_kv_heads > 8) return KVQ_ERR_UNSUPPORTED;
  if (c->num_kv_heads > 8 && c->num_kv_heads % 8) return KVQ_ERR_UNSUPPORTED;
  if (num_ctas < 0 || num_ctas > kMaxCtas) return KVQ_ERR_INVALID_ARGUMENT;
  int nc = num_ctas;
  if (nc == 0) {
    const int sms = sm_count();
    if (sms <= 0) return KVQ_ERR_CUDA;
    nc = auto_ctas(num_seqs, max_context_len, c->num_kv_heads / heads_per_cta(c->num_kv_heads),
                   sms, c->k_fmt == KVQ_FMT_BF16 ? 1 : 2);
  }
  *NC = nc;
  return KVQ_OK;
}

}  // namespace

extern "C" {

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARGUMENT: return "KVQ_ERR_INVALID_ARGUMENT";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA";
  }
  return "KVQ_ERR_UNKNOWN";
}

const char* kvq_version(void) { return "kvq 0.1.0 sm_103a"; }

kvq_status kvq_write_cache(const kvq_cache_desc* cache, void* k_cache, void* v_cache,
                           const void* key, const void* value, int64_t key_stride,
                           int64_t value_stride, const int64_t* slot_mapping, int64_t num_tokens,
                           kvq_stream_t stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (num_tokens < 0) return KVQ_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return KVQ_OK;
  if (!k_cache || !v_cache || !key || !value || !slot_mapping) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(key, 16) || !aligned(value, 16) ||
      !aligned(slot_mapping, 8))
    return KVQ_ERR_INVALID_ARGUMENT;
  const int64_t row = static_cast<int64_t>(cache->num_kv_heads) * cache->head_dim;
  if (key_stride < row || value_stride < row || key_stride % 8 || value_stride % 8)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (num_tokens > (1LL << 31) * 8) return KVQ_ERR_UNSUPPORTED;
  const bool kvarn = (cache->flags & KVQ_FLAG_VARNORM_ROTATE) != 0;
  WriteArgs a;
  a.key = static_cast<const uint16_t*>(key);
  a.value = static_cast<const uint16_t*>(value);
  a.key_stride = key_stride;
  a.value_stride = value_stride;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.k_cache = static_cast<uint8_t*>(k_cache);
  a.v_cache = static_cast<uint8_t*>(v_cache);
  a.k_meta = static_cast<__half*>(cache->k_meta);
  a.v_meta = static_cast<__half*>(cache->v_meta);
  a.num_kv_heads = cache->num_kv_heads;
  a.block_size = cache->block_size;
  a.block_shift = __builtin_ctz(static_cast<unsigned>(cache->block_size));
  a.num_blocks = cache->num_blocks;
  // inv = 1/scale, one IEEE float32 division on the host
  volatile float one = 1.0f;
  a.k_inv = scaled(cache->k_fmt) ? one / cache->k_scale : 1.0f;
  a.v_inv = scaled(cache->v_fmt) ? one / cache->v_scale : 1.0f;
  a.k_head_scale = cache->k_head_scales;
  a.v_head_scale = cache->v_head_scales;
  a.signs = cache->signs;
  a.cR = rotation_scale(cache->head_dim);
  const cudaError_t e =
      launch_write(a, cache->head_dim, cache->k_fmt, cache->v_fmt, kvarn, stream);
  if (e == cudaErrorNotSupported) return KVQ_ERR_UNSUPPORTED;
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_decode_workspace_size_ex(const kvq_cache_desc* cache, int32_t num_seqs,
                                        int32_t num_q_heads, int32_t max_context_len,
                                        int32_t num_ctas, size_t* bytes) {
  if (bytes == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  int NC = 0;
  kvq_status st = decode_shape(cache, num_seqs, num_q_heads, max_context_len, num_ctas, &NC);
  if (st != KVQ_OK) return st;
  *bytes = workspace_bytes_for(num_seqs, num_q_heads, cache->num_kv_heads, cache->head_dim, NC);
  return KVQ_OK;
}

kvq_status kvq_decode_workspace_size(const kvq_cache_desc* cache, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t max_context_len,
                                     size_t* bytes) {
  return kvq_decode_workspace_size_ex(cache, num_seqs, num_q_heads, max_context_len, 0, bytes);
}

}  // extern "C"

namespace {

// The new-token rows of kvq_decode_append (nullptr key: a plain decode).
struct AppendRows {
  const void* key = nullptr;
  const void* value = nullptr;
  int64_t key_stride = 0;
  int64_t value_stride = 0;
};

// Page classes of a mixed cache: every class the same formats, kv-heads,
// head_dim, flags, scales and signs as class 0; pages of 16 tokens or more
// (an 8-token page takes its own kernel instance, one page size per call).
kvq_status check_classes(const kvq_cache_desc* classes, int32_t num_classes,
                         void* const* k_caches, void* const* v_caches, const uint8_t* seq_class) {
  if (classes == nullptr || k_caches == nullptr || v_caches == nullptr || seq_class == nullptr)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (num_classes < 1 || num_classes > kMaxPageClasses) return KVQ_ERR_UNSUPPORTED;
  const kvq_cache_desc& c0 = classes[0];
  for (int c = 0; c < num_classes; ++c) {
    const kvq_cache_desc& x = classes[c];
    kvq_status st = check_cache(&x);
    if (st != KVQ_OK) return st;
    if (x.k_fmt != c0.k_fmt || x.v_fmt != c0.v_fmt || x.num_kv_heads != c0.num_kv_heads ||
        x.head_dim != c0.head_dim || x.flags != c0.flags || x.signs != c0.signs ||
        x.k_head_scales != c0.k_head_scales || x.v_head_scales != c0.v_head_scales ||
        (scaled(x.k_fmt) && x.k_scale != c0.k_scale) || (scaled(x.v_fmt) && x.v_scale != c0.v_scale))
      return KVQ_ERR_INVALID_ARGUMENT;
    if (x.block_size < 16) return KVQ_ERR_UNSUPPORTED;
    if (k_caches[c] == nullptr || v_caches[c] == nullptr || !aligned(k_caches[c], 16) ||
        !aligned(v_caches[c], 16))
      return KVQ_ERR_INVALID_ARGUMENT;
  }
  return KVQ_OK;
}

kvq_status decode_call(const kvq_cache_desc* classes, int32_t num_classes,
                       void* const* k_caches, void* const* v_caches, const uint8_t* seq_class,
                       void* out, const void* query, int32_t num_seqs, int32_t num_q_heads,
                       const int32_t* block_table, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, int32_t max_context_len, float sm_scale,
                       int32_t num_ctas, void* workspace, size_t workspace_bytes,
                       const AppendRows& app, kvq_stream_t stream) {
  const kvq_cache_desc* cache = classes;  // class 0: formats, heads, scales of every class
  int NC = 0;
  kvq_status st = decode_shape(cache, num_seqs, num_q_heads, max_context_len, num_ctas, &NC);
  if (st != KVQ_OK) return st;
  if (num_seqs == 0) return KVQ_OK;
  if (!k_caches[0] || !v_caches[0] || !out || !query || !block_table || !context_lens)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(k_caches[0], 16) || !aligned(v_caches[0], 16) || !aligned(out, 16) ||
      !aligned(query, 16) || !aligned(block_table, 4) || !aligned(context_lens, 4))
    return KVQ_ERR_INVALID_ARGUMENT;
  int min_bs = cache->block_size;
  for (int c = 1; c < num_classes; ++c)
    min_bs = classes[c].block_size < min_bs ? classes[c].block_size : min_bs;
  if (max_blocks_per_seq < ceil_div(max_context_len, min_bs) || max_blocks_per_seq < 0)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!isfinite(sm_scale)) return KVQ_ERR_INVALID_ARGUMENT;
  const size_t need =
      workspace_bytes_for(num_seqs, num_q_heads, cache->num_kv_heads, cache->head_dim, NC);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return KVQ_ERR_WORKSPACE;
  if (need > 0 && !aligned(workspace, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  const bool kvarn = (cache->flags & KVQ_FLAG_VARNORM_ROTATE) != 0;
  DecodeArgs a;
  const bool append = app.key != nullptr;
  for (int c = 0; c < kMaxPageClasses; ++c) {
    const int cc = c < num_classes ? c : 0;
    const kvq_cache_desc& x = classes[cc];
    a.k_cache[c] = static_cast<const uint8_t*>(k_caches[cc]);
    a.v_cache[c] = static_cast<const uint8_t*>(v_caches[cc]);
    a.k_meta[c] = static_cast<const __half*>(x.k_meta);
    a.v_meta[c] = static_cast<const __half*>(x.v_meta);
    a.block_shift[c] = __builtin_ctz(static_cast<unsigned>(x.block_size));
    a.num_blocks[c] = x.num_blocks;
    a.k_cache_w[c] = append ? static_cast<uint8_t*>(k_caches[cc]) : nullptr;
    a.v_cache_w[c] = append ? static_cast<uint8_t*>(v_caches[cc]) : nullptr;
    a.k_meta_w[c] = append ? static_cast<__half*>(x.k_meta) : nullptr;
    a.v_meta_w[c] = append ? static_cast<__half*>(x.v_meta) : nullptr;
  }
  a.seq_class = seq_class;
  a.num_classes = num_classes;
  a.query = static_cast<const uint16_t*>(query);
  a.out = static_cast<uint16_t*>(out);
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.signs = cache->signs;
  const size_t rows = static_cast<size_t>(NC) * 2 * num_q_heads;
  a.ws_acc = need ? static_cast<__half*>(workspace) : nullptr;
  a.ws_ml = need ? reinterpret_cast<float*>(static_cast<__half*>(workspace) + rows * cache->head_dim)
                 : nullptr;
  a.tags = need ? reinterpret_cast<unsigned long long*>(a.ws_ml + rows * 2) : nullptr;
  const size_t slot_words = static_cast<size_t>(NC) *
                           (cache->num_kv_heads / heads_per_cta(cache->num_kv_heads)) * 2;
  a.team_tags = need ? a.tags + slot_words : nullptr;
  a.team_claims = need ? a.tags + 2 * slot_words : nullptr;
  a.claims = need ? a.tags + 3 * slot_words : nullptr;
  a.epoch = next_epoch();
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = cache->num_kv_heads;
  a.gqa = num_q_heads / cache->num_kv_heads;
  a.heads_per_cta = heads_per_cta(cache->num_kv_heads);
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_context_len = max_context_len;
  a.num_ctas = NC;
  a.qk_scale = sm_scale * kLog2e * (scaled(cache->k_fmt) ? cache->k_scale : 1.0f);
  a.v_scale = scaled(cache->v_fmt) ? cache->v_scale : 1.0f;
  a.qk_base = sm_scale * kLog2e;
  a.k_head_scale = cache->k_head_scales;
  a.v_head_scale = cache->v_head_scales;
  a.cR = rotation_scale(cache->head_dim);
  a.new_key = static_cast<const uint16_t*>(app.key);
  a.new_value = static_cast<const uint16_t*>(app.value);
  a.new_key_stride = app.key_stride;
  a.new_value_stride = app.value_stride;
  volatile float one = 1.0f;  // 1/scale, one IEEE float32 division, as kvq_write_cache
  a.k_inv = scaled(cache->k_fmt) ? one / cache->k_scale : 1.0f;
  a.v_inv = scaled(cache->v_fmt) ? one / cache->v_scale : 1.0f;
  a.spin_limit = kDefaultSpinLimit;
  a.withhold_cta = -1;
  a.withhold_tile = -1;
  if (g_wait_hook_armed.exchange(0) != 0) {
    a.spin_limit = g_wait_hook_polls.load();
    a.withhold_cta = g_wait_hook_cta.load();
    a.withhold_tile = g_wait_hook_tile.load();
  }
  // A launch recorded into a CUDA graph is replayed with the same call tag, so
  // a replay would find the tags and claims its predecessor left: while the
  // stream is capturing, the call first clears them (a memset node that runs
  // before the kernel at every replay).  Direct calls take a fresh tag instead.
  if (need > 0) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap) != cudaSuccess)
      return KVQ_ERR_CUDA;
    if (cap == cudaStreamCaptureStatusActive) {
      const size_t words = 3 * slot_words + static_cast<size_t>(num_seqs) *
                                                (cache->num_kv_heads / heads_per_cta(cache->num_kv_heads));
      if (cudaMemsetAsync(a.tags, 0, words * sizeof(unsigned long long),
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KVQ_ERR_CUDA;
    }
  }
  cudaError_t e = cudaErrorNotSupported;
  const int kf = cache->k_fmt, vf = cache->v_fmt;
#define KVQ_UNIT_LAUNCHER(U) launch_##U,
  static const DecodeLauncher launchers[] = {KVQ_DECODE_UNITS(KVQ_UNIT_LAUNCHER)};
#undef KVQ_UNIT_LAUNCHER
  for (DecodeLauncher f : launchers) {  // the unit that holds the instance launches it
    e = f(a, cache->head_dim, kf, vf, kvarn, stream);
    if (e != cudaErrorNotSupported) break;
  }
  if (e == cudaErrorNotSupported) return KVQ_ERR_UNSUPPORTED;
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// The new-token rows of kvq_decode_append, checked.
kvq_status append_rows(const kvq_cache_desc* cache, int32_t num_seqs, const void* new_key,
                       const void* new_value, int64_t key_stride, int64_t value_stride,
                       AppendRows* app) {
  if (num_seqs > 0) {
    if (!new_key || !new_value || !aligned(new_key, 16) || !aligned(new_value, 16))
      return KVQ_ERR_INVALID_ARGUMENT;
    const int64_t row = static_cast<int64_t>(cache->num_kv_heads) * cache->head_dim;
    if (key_stride < row || value_stride < row || key_stride % 8 || value_stride % 8)
      return KVQ_ERR_INVALID_ARGUMENT;
    if (!write_supported(cache->k_fmt, cache->v_fmt,
                         (cache->flags & KVQ_FLAG_VARNORM_ROTATE) != 0))
      return KVQ_ERR_UNSUPPORTED;
  }
  app->key = new_key;
  app->value = new_value;
  app->key_stride = key_stride;
  app->value_stride = value_stride;
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_paged_decode_ex(const kvq_cache_desc* cache, const void* k_cache,
                               const void* v_cache, void* out, const void* query,
                               int32_t num_seqs, int32_t num_q_heads, const int32_t* block_table,
                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                               int32_t max_context_len, float sm_scale, int32_t num_ctas,
                               void* workspace, size_t workspace_bytes, kvq_stream_t stream) {
  void* kc = const_cast<void*>(k_cache);
  void* vc = const_cast<void*>(v_cache);
  return decode_call(cache, 1, &kc, &vc, nullptr, out, query, num_seqs, num_q_heads, block_table,
                     max_blocks_per_seq, context_lens, max_context_len, sm_scale, num_ctas,
                     workspace, workspace_bytes, AppendRows{}, stream);
}

kvq_status kvq_decode_append(const kvq_cache_desc* cache, void* k_cache, void* v_cache,
                             const void* new_key, const void* new_value, int64_t key_stride,
                             int64_t value_stride, void* out, const void* query,
                             int32_t num_seqs, int32_t num_q_heads, const int32_t* block_table,
                             int32_t max_blocks_per_seq, const int32_t* context_lens,
                             int32_t max_context_len, float sm_scale, int32_t num_ctas,
                             void* workspace, size_t workspace_bytes, kvq_stream_t stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  AppendRows app;
  st = append_rows(cache, num_seqs, new_key, new_value, key_stride, value_stride, &app);
  if (st != KVQ_OK) return st;
  return decode_call(cache, 1, &k_cache, &v_cache, nullptr, out, query, num_seqs, num_q_heads,
                     block_table, max_blocks_per_seq, context_lens, max_context_len, sm_scale,
                     num_ctas, workspace, workspace_bytes, app, stream);
}

kvq_status kvq_decode_mixed(const kvq_cache_desc* classes, int32_t num_classes,
                            void* const* k_caches, void* const* v_caches,
                            const uint8_t* seq_class, const void* new_key, const void* new_value,
                            int64_t key_stride, int64_t value_stride, void* out,
                            const void* query, int32_t num_seqs, int32_t num_q_heads,
                            const int32_t* block_table, int32_t max_blocks_per_seq,
                            const int32_t* context_lens, int32_t max_context_len,
                            float sm_scale, int32_t num_ctas, void* workspace,
                            size_t workspace_bytes, kvq_stream_t stream) {
  kvq_status st = check_classes(classes, num_classes, k_caches, v_caches, seq_class);
  if (st != KVQ_OK) return st;
  AppendRows app;
  if (new_key != nullptr || new_value != nullptr) {
    st = append_rows(classes, num_seqs, new_key, new_value, key_stride, value_stride, &app);
    if (st != KVQ_OK) return st;
  }
  return decode_call(classes, num_classes, k_caches, v_caches, seq_class, out, query, num_seqs,
                     num_q_heads, block_table, max_blocks_per_seq, context_lens,
                     max_context_len, sm_scale, num_ctas, workspace, workspace_bytes, app,
                     stream);
}

kvq_status kvq_paged_decode(const kvq_cache_desc* cache, const void* k_cache,
                            const void* v_cache, void* out, const void* query, int32_t num_seqs,
                            int32_t num_q_heads, const int32_t* block_table,
                            int32_t max_blocks_per_seq, const int32_t* context_lens,
                            int32_t max_context_len, float sm_scale, void* workspace,
                            size_t workspace_bytes, kvq_stream_t stream) {
  return kvq_paged_decode_ex(cache, k_cache, v_cache, out, query, num_seqs, num_q_heads,
                             block_table, max_blocks_per_seq, context_lens, max_context_len,
                             sm_scale, 0, workspace, workspace_bytes, stream);
}

kvq_status kvq_hadamard(void* x, int32_t dtype, int64_t rows, int32_t head_dim,
                        const int8_t* signs, int32_t inverse, kvq_stream_t stream) {
  if (rows < 0 || (dtype != 0 && dtype != 1) || (inverse != 0 && inverse != 1))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  if (rows == 0) return KVQ_OK;
  if (x == nullptr || !aligned(x, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  if (signs != nullptr && !aligned(signs, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  const cudaError_t e =
      launch_hadamard(x, dtype, rows, head_dim, signs, inverse, rotation_scale(head_dim), stream);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_calibrate_scale(const void* x, int64_t n, float qmax, float* scale_out,
                               kvq_stream_t stream) {
  if (n < 0 || !(qmax > 0.0f && isfinite(qmax)) || scale_out == nullptr ||
      !aligned(scale_out, 4))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (n > 0 && (x == nullptr || !aligned(x, 16))) return KVQ_ERR_INVALID_ARGUMENT;
  const int sms = sm_count();
  if (sms <= 0) return KVQ_ERR_CUDA;
  const cudaError_t e =
      launch_calibrate(static_cast<const uint16_t*>(x), n, qmax, scale_out, stream, sms);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_calibrate_head_scales(const void* x, int64_t num_tokens, int32_t num_kv_heads,
                                     int32_t head_dim, int64_t stride, float qmax,
                                     float* scales_out, kvq_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 8 || head_dim % 8 ||
      !(qmax > 0.0f && isfinite(qmax)) || scales_out == nullptr || !aligned(scales_out, 4))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (stride < static_cast<int64_t>(num_kv_heads) * head_dim || stride % 8)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (num_tokens > 0 && (x == nullptr || !aligned(x, 16))) return KVQ_ERR_INVALID_ARGUMENT;
  const int sms = sm_count();
  if (sms <= 0) return KVQ_ERR_CUDA;
  const cudaError_t e =
      launch_calibrate_heads(static_cast<const uint16_t*>(x), num_tokens, num_kv_heads, head_dim,
                             stride, qmax, scales_out, stream, sms);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_debug_arm_wait_timeout(int32_t polls, int32_t cta, int32_t tile) {
  if (polls < 1 || cta < -1 || tile < -1) return KVQ_ERR_INVALID_ARGUMENT;
  g_wait_hook_polls.store(polls);
  g_wait_hook_cta.store(cta);
  g_wait_hook_tile.store(tile);
  g_wait_hook_armed.store(1);
  return KVQ_OK;
}

kvq_status kvq_get_device_error(kvq_stream_t stream, uint32_t* bits) {
  if (bits == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KVQ_ERR_CUDA;
  unsigned v = 0;
#define KVQ_UNIT_TAKE(U) take_error_bits_##U,
  cudaError_t (*take[])(unsigned*) = {take_error_bits_write, take_error_bits_write_asym,
                                      KVQ_DECODE_UNITS(KVQ_UNIT_TAKE)};
#undef KVQ_UNIT_TAKE
  for (auto f : take)
    if (f(&v) != cudaSuccess) return KVQ_ERR_CUDA;
  *bits = v;
  return KVQ_OK;
}

}  // extern "C"

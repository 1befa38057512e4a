// kvq_paged_decode_static: kvq_paged_decode without a caller-provided
// workspace.  The split-K scratch lives in a fixed-size array in device
// global memory that is part of the library image, so the call needs no
// allocation of any kind.
//
// Scratch: kStaticScratchBytes (16 MiB) in `g_decode_scratch`; every GPU
// that loads the library holds that much for the life of the process.
// Host code may not use the array's name as a device address (on the host it
// names a stand-in object), so its device address is looked up with
// cudaGetSymbolAddress, with the device current, on the first call made on
// the device, and cached together with the unique id of the context it was
// looked up in: a call made in another context of that device (after a
// cudaDeviceReset, the library's module is loaded again, possibly elsewhere)
// looks it up again.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/kvq.h"
#include "kvq_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Unique id of the calling thread's current context (0 if it cannot be read).
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
      ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_decode_scratch on the current device (looked up once per
// device and context).
kvq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  const unsigned long long ctx = current_context_id();
  if (g_scratch_ptr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return KVQ_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = current_context_id();  // the lookup made the context current
  }
  *out = g_scratch_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" {

size_t kvq_paged_decode_static_capacity(void) { return kStaticScratchBytes; }

kvq_status kvq_paged_decode_static(const kvq_cache_desc* cache, const void* k_cache,
                                   const void* v_cache, void* out, const void* query,
                                   int32_t num_seqs, int32_t num_q_heads,
                                   const int32_t* block_table, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int32_t max_context_len,
                                   float sm_scale, int32_t num_ctas, kvq_stream_t stream) {
  size_t need = 0;
  kvq_status st = kvq_decode_workspace_size_ex(cache, num_seqs, num_q_heads, max_context_len,
                                               num_ctas, &need);
  if (st != KVQ_OK) return st;
  if (need > kStaticScratchBytes) return KVQ_ERR_WORKSPACE;  // sizes beyond the fixed scratch
  void* scratch = nullptr;
  if (need > 0) {
    st = scratch_address(&scratch);
    if (st != KVQ_OK) return st;
  }
  return kvq_paged_decode_ex(cache, k_cache, v_cache, out, query, num_seqs, num_q_heads,
                             block_table, max_blocks_per_seq, context_lens, max_context_len,
                             sm_scale, num_ctas, scratch, need ? kStaticScratchBytes : 0,
                             stream);
}

}  // extern "C"

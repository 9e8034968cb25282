// decode_static.cu -- attn_decode_paged_static: paged split-KV decode that
// allocates nothing and takes no workspace argument.
//
// Why it exists: attn_decode_paged needs a caller-supplied workspace for the
// split partial states. Some callers have no way to obtain device memory at
// the point of the call -- for example a plugin loaded into a host program
// that owns all device memory and offers it no allocation hook, or a serving
// hot loop that must not call cudaMalloc (which can synchronise the device
// and takes allocator locks). This entry point keeps the partials in a
// fixed-size array that lives in the library's own device image instead.
//
// The scratch array below is a file-scope __device__ variable: the CUDA
// module loader reserves it on every GPU that loads this library, and it
// stays reserved until the process exits. In host code the name
// g_decode_static_scratch is only a host-side stand-in for the symbol, not a
// device address; the real address is looked up with cudaGetSymbolAddress,
// with the device current, the first time this entry point runs on a device,
// and again whenever that device's context has changed since (after a
// cudaDeviceReset the module is loaded anew and the array can move).
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace attn {

namespace {

static __device__ __align__(256) unsigned char g_decode_static_scratch[ATTN_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
struct ScratchAddr {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;  // unique id of the context the address belongs to
};
ScratchAddr g_scratch[kMaxDevices];

// Unique id of the calling thread's current context (0 when it cannot be
// read, in which case the address is looked up on every call).
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

// Device address of the current device's copy of the scratch array (nullptr
// on error, with the CUDA error in *err).
void* scratch_for_current_device(cudaError_t* err) {
  int dev = -1;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  // Before the device's first runtime call no context is current and the id
  // reads 0; the symbol lookup then creates the context, and its id is read
  // again for the next call.
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchAddr& a = g_scratch[dev];
  const unsigned long long id = current_context_id();
  if (a.ptr == nullptr || id == 0 || id != a.ctx_id) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_decode_static_scratch);
    if (*err != cudaSuccess) return nullptr;
    a.ptr = p;
    a.ctx_id = id != 0 ? id : current_context_id();
  }
  return a.ptr;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_decode_paged_static(const void* q, const void* k_cache,
                                                  const void* v_cache, const int32_t* block_table,
                                                  const int32_t* seq_lens, int B, int h, int h_kv,
                                                  int d_h, int page_size, int num_blocks,
                                                  int max_blocks_per_seq, int num_splits,
                                                  float scale, void* o, float* lse, void* stream) {
  // Same argument rules as attn_decode_paged, checked before anything else.
  if (B < 0 || h < 1 || h_kv < 1 || h % h_kv != 0 || num_blocks < 1 || max_blocks_per_seq < 1 ||
      num_splits < 1 || num_splits > ATTN_MAX_SPLITS || !std::isfinite(scale) || !(scale > 0.f))
    return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || h_kv > 65535) return ATTN_ERR_INVALID_ARG;
  const int g = h / h_kv;
  if ((d_h != 64 && d_h != 128) || page_size != 16 || (g != 1 && g != 2 && g != 4 && g != 8))
    return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * page_size > (1ll << 30))
    return ATTN_ERR_INVALID_ARG;
  if (B == 0) return ATTN_OK;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned_to(q, 16) || !aligned_to(k_cache, 16) || !aligned_to(v_cache, 16) ||
      !aligned_to(o, 16) || !aligned_to(block_table, 4) || !aligned_to(seq_lens, 4) ||
      !aligned_to(lse, 4))
    return ATTN_ERR_INVALID_ARG;

  // The partials must fit in the fixed array; larger batches are refused.
  const long long rows = static_cast<long long>(B) * h;
  const PartialLayout L = partial_layout(rows, num_splits, d_h);
  if (L.total > static_cast<size_t>(ATTN_DECODE_STATIC_SCRATCH_BYTES)) return ATTN_ERR_INVALID_ARG;

  cudaError_t e = cudaSuccess;
  uint8_t* ws = static_cast<uint8_t*>(scratch_for_current_device(&e));
  if (ws == nullptr) return ATTN_ERR_CUDA;

  // Nothing in the scratch has to start at zero: stage 1 writes every partial
  // (split < n_active of its row) before the merge reads it, and the merge
  // never reads a split at or past n_active.
  DecodeArgs a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.B = B;
  a.h = h;
  a.h_kv = h_kv;
  a.d_h = d_h;
  a.page_size = page_size;
  a.num_blocks = num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_splits = num_splits;
  a.scale = scale;
  a.o_part = reinterpret_cast<float*>(ws + L.o_off);
  a.m_part = reinterpret_cast<float*>(ws + L.m_off);
  a.l_part = reinterpret_cast<float*>(ws + L.l_off);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = launch_decode_split(a, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  e = launch_merge(a.o_part, a.m_part, a.l_part, nullptr, seq_lens, h, page_size,
                   max_blocks_per_seq * page_size, static_cast<int>(rows), num_splits, d_h, o, lse,
                   ATTN_DTYPE_BF16, s);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

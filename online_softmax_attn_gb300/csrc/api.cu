// api.cu -- the C ABI declared in include/attn.h: host-side validation,
// workspace carve-up, tensor-map encoding and kernel launches. No entry point
// here allocates, frees or synchronises (except attn_get_device_error and
// attn_get_last_device_error, synchronising queries by contract); the host-memory prefill, with its
// copy streams, lives in host_prefill.cu.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace attn {

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

attn_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

}  // namespace

CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* base,
                           const uint64_t* dims, const uint64_t* strides_bytes,
                           const uint32_t* box, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  uint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  return fn(map, dtype, rank, base, dims, strides_bytes, box, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE: return "device-side error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

int attn_version(void) { return 301; }

int attn_decode_split_plan(int seq_len, int page_size, int num_splits, int* pages_per_split) {
  if (seq_len < 0 || page_size < 1 || num_splits < 1) return -1;
  return split_plan(seq_len, page_size, num_splits, pages_per_split);
}

int attn_recommended_splits_ragged(int B, int h_kv, int max_seq_len, long long total_seq_len,
                                   int num_sms) {
  if (B < 1 || h_kv < 1 || max_seq_len < 0 || total_seq_len < 0 || num_sms < 1) return -1;
  return splits_rule(B, h_kv, max_seq_len, total_seq_len, num_sms, ATTN_MAX_SPLITS);
}

int attn_recommended_splits(int B, int h_kv, int max_seq_len, int device) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    (void)cudaGetLastError();  // leave no sticky error for the caller
    return -1;
  }
  return attn_recommended_splits_ragged(B, h_kv, max_seq_len, 0, sms);
}

size_t attn_decode_workspace_bytes(int B, int h, int num_splits, int d_h) {
  if (B < 0 || h < 1 || d_h < 1 || num_splits < 1) return 0;
  return partial_layout(static_cast<long long>(B) * h, num_splits, d_h).total;
}

size_t attn_prefill_workspace_bytes(int T, int h_kv, int d_h, attn_dtype_t dtype) {
  if (T < 0 || h_kv < 1 || (d_h != 64 && d_h != 128)) return static_cast<size_t>(-1);
  if (dtype != ATTN_DTYPE_F32 && dtype != ATTN_DTYPE_BF16) return static_cast<size_t>(-1);
  if (dtype == ATTN_DTYPE_F32 || T == 0) return 0;
  return attn::prefill_layout(T, h_kv, d_h).total;
}

attn_status_t attn_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                           int T, int h, int h_kv, int d_h, int causal, float scale,
                           attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (T < 0 || h < 1 || h_kv < 1 || h % h_kv != 0 || !std::isfinite(scale) || !(scale > 0.f))
    return ATTN_ERR_INVALID_ARG;
  if (h > 65535) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_DTYPE_F32 && dtype != ATTN_DTYPE_BF16) return ATTN_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return ATTN_ERR_UNSUPPORTED;
  if (T == 0) return ATTN_OK;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  if (workspace && (!aligned(workspace, 256) ||
                    workspace_bytes < attn_prefill_workspace_bytes(T, h_kv, d_h, dtype)))
    return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == ATTN_DTYPE_F32)
    return from_cuda(launch_prefill_f32(static_cast<const float*>(q),
                                        static_cast<const float*>(k),
                                        static_cast<const float*>(v), static_cast<float*>(o), lse,
                                        T, h, h_kv, d_h, causal != 0, scale, s));
  const cudaError_t e =
      launch_prefill_bf16(q, k, v, o, lse, T, h, h_kv, d_h, causal != 0, scale, workspace, s);
  if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
  return from_cuda(e);
}

namespace {
// Shared by attn_decode_paged (fixed_pps = 0: pages per split from
// num_splits), attn_decode_paged_deterministic (fixed_pps > 0) and
// attn_decode_paged_adaptive (adaptive: pages per split planned on the device,
// kept in the 256 bytes after the partials).
attn_status_t decode_paged_impl(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* seq_lens, int B, int h,
                                int h_kv, int d_h, int page_size, int num_blocks,
                                int max_blocks_per_seq, int num_splits, int fixed_pps, float scale,
                                void* workspace, size_t workspace_bytes, void* o, float* lse,
                                void* stream, bool adaptive = false) {
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
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !workspace || !o)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(lse, 4) ||
      !aligned(workspace, 256))
    return ATTN_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * h;
  if (rows > 0x7fffffffll) return ATTN_ERR_INVALID_ARG;  // rows index an int grid
  const PartialLayout L = partial_layout(rows, num_splits, d_h);
  if (workspace_bytes < L.total + (adaptive ? 256u : 0u)) return ATTN_ERR_INVALID_ARG;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
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
  a.fixed_pps = fixed_pps;
  int* pps_dev = adaptive ? reinterpret_cast<int*>(ws + L.total) : nullptr;
  a.pps_dev = pps_dev;
  a.o_part = reinterpret_cast<float*>(ws + L.o_off);
  a.m_part = reinterpret_cast<float*>(ws + L.m_off);
  a.l_part = reinterpret_cast<float*>(ws + L.l_off);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (adaptive) {
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = launch_decode_plan(seq_lens, nullptr, B, h_kv, max_blocks_per_seq * page_size, sms,
                             num_splits, pps_dev, s);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
  }
  e = launch_decode_split(a, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  e = launch_merge(a.o_part, a.m_part, a.l_part, nullptr, seq_lens, h, page_size,
                   max_blocks_per_seq * page_size, static_cast<int>(rows), num_splits, d_h, o, lse,
                   ATTN_DTYPE_BF16, s, fixed_pps, pps_dev);
  return from_cuda(e);
}
}  // namespace

size_t attn_prefill_paged_workspace_bytes(int B) {
  if (B < 0) return 0;
  return align256(size_t(B + 1) * sizeof(int32_t));
}

namespace {
// Layout of the larger paged-prefill workspace: tile offsets, then the V
// format flags [B, h_kv, max_tiles] int32, then the fp16 V copy
// [B, max_tiles * 128, h_kv, d_h]. Zero when the copy cannot be addressed
// (its token count must stay below 2^31) or the arguments are invalid.
struct PagedV16Layout {
  size_t flags_off = 0, v16_off = 0, total = 0;
};
PagedV16Layout paged_v16_layout(int B, int max_blocks_per_seq, int h_kv, int d_h) {
  PagedV16Layout L;
  if (B < 0 || max_blocks_per_seq < 1 || max_blocks_per_seq > (1 << 26) || h_kv < 1 ||
      h_kv > 65535 || (d_h != 64 && d_h != 128))
    return L;
  const long long max_tiles = (max_blocks_per_seq + 7) / 8;
  const long long tokens = static_cast<long long>(B) * max_tiles * 128;
  if (tokens >= (1ll << 31)) return L;
  L.flags_off = attn_prefill_paged_workspace_bytes(B);
  L.v16_off = L.flags_off + align256(size_t(B) * h_kv * max_tiles * sizeof(int32_t));
  L.total = L.v16_off + size_t(tokens) * h_kv * d_h * 2;
  return L;
}
}  // namespace

size_t attn_prefill_paged_v16_workspace_bytes(int B, int max_blocks_per_seq, int h_kv, int d_h) {
  return paged_v16_layout(B, max_blocks_per_seq, h_kv, d_h).total;
}

size_t attn_prefill_paged_decode_workspace_bytes(int B, int h, int decode_splits, int d_h) {
  if (B < 0 || h < 1 || d_h < 1 || decode_splits < 0 || decode_splits > ATTN_MAX_SPLITS) return 0;
  if (decode_splits == 0) return 0;
  // The adaptive decode's partials, then 256 bytes for its device plan.
  return partial_layout(static_cast<long long>(B) * h, decode_splits, d_h).total + 256;
}

attn_status_t attn_prefill_paged(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, const int32_t* cu_seqlens_q,
                                 const int32_t* seq_lens, int B, int total_q, int h, int h_kv,
                                 int d_h, int page_size, int num_blocks, int max_blocks_per_seq,
                                 int max_q_len, int causal, float scale, int decode_splits,
                                 void* workspace, size_t workspace_bytes, void* o, float* lse,
                                 void* stream) {
  if (B < 0 || total_q < 0 || h < 1 || h > 65535 || h_kv < 1 || h % h_kv != 0 ||
      num_blocks < 1 || max_blocks_per_seq < 1 || !std::isfinite(scale) || !(scale > 0.f) ||
      decode_splits < 0 || decode_splits > ATTN_MAX_SPLITS)
    return ATTN_ERR_INVALID_ARG;
  if ((d_h != 64 && d_h != 128) || page_size != 16) return ATTN_ERR_UNSUPPORTED;
  if (decode_splits > 0) {
    const int g = h / h_kv;
    if (g != 1 && g != 2 && g != 4 && g != 8) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535 || static_cast<long long>(B) * h > 0x7fffffffll) return ATTN_ERR_INVALID_ARG;
  }
  if (static_cast<long long>(max_blocks_per_seq) * page_size > (1ll << 30))
    return ATTN_ERR_INVALID_ARG;
  if (B == 0 || total_q == 0) return ATTN_OK;
  if (max_q_len < 1) return ATTN_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_table || !cu_seqlens_q || !seq_lens || !workspace || !o)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
      !aligned(block_table, 4) || !aligned(cu_seqlens_q, 4) || !aligned(seq_lens, 4) ||
      !aligned(lse, 4) || !aligned(workspace, 256))
    return ATTN_ERR_INVALID_ARG;
  // Workspace: the decode rows' partials first (decode_splits > 0), then the
  // prefill's own layout, small or with the fp16 V copy.
  const size_t dec_bytes = attn_prefill_paged_decode_workspace_bytes(B, h, decode_splits, d_h);
  if (workspace_bytes < dec_bytes + attn_prefill_paged_workspace_bytes(B))
    return ATTN_ERR_INVALID_ARG;
  uint8_t* const dec_ws = static_cast<uint8_t*>(workspace);
  workspace = dec_ws + dec_bytes;
  workspace_bytes -= dec_bytes;
  PagedPrefill a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.cu_q = cu_seqlens_q;
  a.seq_lens = seq_lens;
  a.tile_off = static_cast<int32_t*>(workspace);
  a.v16 = nullptr;
  a.vwide = nullptr;
  const PagedV16Layout L = paged_v16_layout(B, max_blocks_per_seq, h_kv, d_h);
  if (L.total != 0 && workspace_bytes >= L.total) {
    a.v16 = static_cast<uint8_t*>(workspace) + L.v16_off;
    a.vwide = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + L.flags_off);
  }
  a.B = B;
  a.total_q = total_q;
  a.h = h;
  a.h_kv = h_kv;
  a.d_h = d_h;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks_per_seq;
  a.max_q_len = max_q_len;
  a.causal = causal != 0;
  a.scale = scale;
  a.o = o;
  a.lse = lse;
  a.decode_rows_apart = decode_splits > 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_prefill_paged(a, s);
  if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
  if (e != cudaSuccess || decode_splits == 0) return from_cuda(e);
  // Rows of one query: the split-KV decode ([DEC] "Where GQA enters": a
  // single query row as one row of a 128-row tile wastes the rest; split the
  // key axis instead), with its split count planned on the device from those
  // rows' lengths under a grid of decode_splits, their queries and outputs at
  // token cu_seqlens_q[b].
  const PartialLayout PL = partial_layout(static_cast<long long>(B) * h, decode_splits, d_h);
  int* pps_dev = reinterpret_cast<int*>(dec_ws + PL.total);
  DecodeArgs da;
  da.q = q;
  da.k_cache = k_cache;
  da.v_cache = v_cache;
  da.block_table = block_table;
  da.seq_lens = seq_lens;
  da.B = B;
  da.h = h;
  da.h_kv = h_kv;
  da.d_h = d_h;
  da.page_size = page_size;
  da.num_blocks = num_blocks;
  da.max_blocks_per_seq = max_blocks_per_seq;
  da.num_splits = decode_splits;
  da.scale = scale;
  da.pps_dev = pps_dev;
  da.q_rows = cu_seqlens_q;
  da.o_part = reinterpret_cast<float*>(dec_ws + PL.o_off);
  da.m_part = reinterpret_cast<float*>(dec_ws + PL.m_off);
  da.l_part = reinterpret_cast<float*>(dec_ws + PL.l_off);
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = launch_decode_plan(seq_lens, cu_seqlens_q, B, h_kv, max_blocks_per_seq * page_size, sms,
                           decode_splits, pps_dev, s);
  if (e == cudaSuccess) e = launch_decode_split(da, s);
  if (e == cudaSuccess)
    e = launch_merge(da.o_part, da.m_part, da.l_part, nullptr, seq_lens, h, page_size,
                     max_blocks_per_seq * page_size, static_cast<int>(static_cast<long long>(B) * h),
                     decode_splits, d_h, o, lse, ATTN_DTYPE_BF16, s, 0, pps_dev, cu_seqlens_q);
  return from_cuda(e);
}

attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* seq_lens, int B, int h,
                                int h_kv, int d_h, int page_size, int num_blocks,
                                int max_blocks_per_seq, int num_splits, float scale,
                                void* workspace, size_t workspace_bytes, void* o, float* lse,
                                void* stream) {
  return decode_paged_impl(q, k_cache, v_cache, block_table, seq_lens, B, h, h_kv, d_h, page_size,
                           num_blocks, max_blocks_per_seq, num_splits, 0, scale, workspace,
                           workspace_bytes, o, lse, stream);
}

size_t attn_decode_adaptive_workspace_bytes(int B, int h, int max_splits, int d_h) {
  if (B < 0 || h < 1 || d_h < 1 || max_splits < 1) return 0;
  return partial_layout(static_cast<long long>(B) * h, max_splits, d_h).total + 256;
}

attn_status_t attn_decode_paged_adaptive(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_table, const int32_t* seq_lens,
                                         int B, int h, int h_kv, int d_h, int page_size,
                                         int num_blocks, int max_blocks_per_seq, int max_splits,
                                         float scale, void* workspace, size_t workspace_bytes,
                                         void* o, float* lse, void* stream) {
  return decode_paged_impl(q, k_cache, v_cache, block_table, seq_lens, B, h, h_kv, d_h, page_size,
                           num_blocks, max_blocks_per_seq, max_splits, 0, scale, workspace,
                           workspace_bytes, o, lse, stream, true);
}

attn_status_t attn_decode_paged_deterministic(const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_table,
                                              const int32_t* seq_lens, int B, int h, int h_kv,
                                              int d_h, int page_size, int num_blocks,
                                              int max_blocks_per_seq, int num_splits,
                                              int pages_per_split, float scale, void* workspace,
                                              size_t workspace_bytes, void* o, float* lse,
                                              void* stream) {
  if (pages_per_split < 1 || max_blocks_per_seq < 1) return ATTN_ERR_INVALID_ARG;
  // The grid must hold every split of the longest possible row.
  if (static_cast<long long>(num_splits) * pages_per_split < max_blocks_per_seq)
    return ATTN_ERR_INVALID_ARG;
  return decode_paged_impl(q, k_cache, v_cache, block_table, seq_lens, B, h, h_kv, d_h, page_size,
                           num_blocks, max_blocks_per_seq, num_splits, pages_per_split, scale,
                           workspace, workspace_bytes, o, lse, stream);
}

attn_status_t attn_merge_states(const float* o_part, const float* m_part, const float* l_part,
                                const int32_t* n_active, int rows, int num_splits, int d_h,
                                void* o, float* lse, attn_dtype_t out_dtype, void* stream) {
  if (rows < 0 || num_splits < 1) return ATTN_ERR_INVALID_ARG;
  if (out_dtype != ATTN_DTYPE_F32 && out_dtype != ATTN_DTYPE_BF16) return ATTN_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return ATTN_ERR_UNSUPPORTED;
  if (rows == 0) return ATTN_OK;
  if (!o_part || !m_part || !l_part || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned(o_part, 16) || !aligned(m_part, 4) || !aligned(l_part, 4) || !aligned(o, 16) ||
      !aligned(n_active, 4) || !aligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  return from_cuda(launch_merge(o_part, m_part, l_part, n_active, nullptr, 1, 16, 0, rows,
                                num_splits, d_h, o, lse, out_dtype,
                                static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_merge_lse_pair(const void* o_a, const float* lse_a, const void* o_b,
                                  const float* lse_b, int rows, int d_h, attn_dtype_t in_dtype,
                                  void* o, float* lse, attn_dtype_t out_dtype, void* stream) {
  if (rows < 0) return ATTN_ERR_INVALID_ARG;
  if ((in_dtype != ATTN_DTYPE_F32 && in_dtype != ATTN_DTYPE_BF16) ||
      (out_dtype != ATTN_DTYPE_F32 && out_dtype != ATTN_DTYPE_BF16))
    return ATTN_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return ATTN_ERR_UNSUPPORTED;
  if (rows == 0) return ATTN_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned(o_a, 16) || !aligned(o_b, 16) || !aligned(o, 16) || !aligned(lse_a, 4) ||
      !aligned(lse_b, 4) || !aligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(lse);
    const uintptr_t hi = lo + static_cast<uintptr_t>(rows) * sizeof(float);
    for (const float* in : {lse_a, lse_b}) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(in);
      const uintptr_t b = a + static_cast<uintptr_t>(rows) * sizeof(float);
      if (lo < b && a < hi) return ATTN_ERR_INVALID_ARG;
    }
  }
  return from_cuda(launch_merge_pair(o_a, lse_a, o_b, lse_b, rows, d_h, in_dtype, o, lse,
                                     out_dtype, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return ATTN_ERR_INVALID_ARG;
  return from_cuda(launch_wait_timeout_selftest(uint64_t(limit_us) * 1000ull,
                                                static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_selftest_prefill_stall(int key_tile) {
  const cudaError_t e = attn::prefill_set_stall(key_tile < 0 ? -1 : key_tile);
  if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_selftest_delayed_copy(int32_t* dst, const int32_t* src, int n,
                                         unsigned int delay_us, void* stream) {
  if (n < 0 || delay_us > 1000 || (n > 0 && (!dst || !src)) || !aligned(dst, 4) ||
      !aligned(src, 4))
    return ATTN_ERR_INVALID_ARG;
  if (n == 0) return ATTN_OK;
  return from_cuda(launch_delayed_copy(dst, src, n, uint64_t(delay_us) * 1000ull,
                                       static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_get_device_error(void* stream, unsigned int* bits) {
  if (bits == nullptr) return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e1 = cudaSuccess, e2 = cudaSuccess, e3 = cudaSuccess, e4 = cudaSuccess;
  unsigned int v = decode_read_and_clear_error(s, &e1);
  v |= merge_read_and_clear_error(s, &e2);
  v |= prefill_read_and_clear_error(s, &e3);
  v |= simt_read_and_clear_error(s, &e4);
  *bits = v;
  if (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess || e4 != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status_t attn_get_last_device_error(void* stream) {
  unsigned int bits = 0;
  const attn_status_t st = attn_get_device_error(stream, &bits);
  if (st != ATTN_OK) return st;
  if (bits & ATTN_DEVERR_WAIT_TIMEOUT) return ATTN_ERR_DEVICE_TIMEOUT;
  return bits ? ATTN_ERR_DEVICE : ATTN_OK;
}

}  // extern "C"

// internal.h -- launchers between the C-ABI layer (api.cu) and the kernel
// translation units. Arguments are already validated when these are called.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "attn.h"

namespace attn {

// Partial-state workspace carve-up: O~ [rows, S, d], m [rows, S], l [rows, S].
struct PartialLayout {
  size_t o_off, m_off, l_off, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline PartialLayout partial_layout(long long rows, int num_splits, int d_h) {
  PartialLayout L;
  L.o_off = 0;
  L.m_off = align256(size_t(rows) * num_splits * d_h * sizeof(float));
  L.l_off = L.m_off + align256(size_t(rows) * num_splits * sizeof(float));
  L.total = L.l_off + align256(size_t(rows) * num_splits * sizeof(float));
  return L;
}

// merge.cu -----------------------------------------------------------------
// n_active == nullptr and seq_lens == nullptr: all splits active.
// seq_lens != nullptr: n_active(row) = split_plan(seq_lens[row / heads_per_seq]),
// with the length clamped into [0, max_len] exactly as the decode kernel does.
// fixed_pps as in split_plan_fixed (0: pages per split from num_splits).
// q_rows != nullptr (a mixed batch's cu_seqlens_q): only rows of sequences
// with one query are merged, each written at token q_rows[row / heads_per_seq].
cudaError_t launch_merge(const float* o_part, const float* m_part, const float* l_part,
                         const int32_t* n_active, const int32_t* seq_lens, int heads_per_seq,
                         int page_size, int max_len, int rows, int num_splits, int d_h, void* o, float* lse,
                         attn_dtype_t out_dtype, cudaStream_t stream, int fixed_pps = 0,
                         const int* pps_dev = nullptr, const int32_t* q_rows = nullptr);
unsigned int merge_read_and_clear_error(cudaStream_t stream, cudaError_t* st);
// Pairwise (O, LSE) merge; arguments validated by the caller.
cudaError_t launch_merge_pair(const void* o_a, const float* lse_a, const void* o_b,
                              const float* lse_b, int rows, int d_h, attn_dtype_t in_dtype,
                              void* o, float* lse, attn_dtype_t out_dtype, cudaStream_t stream);

// decode.cu ----------------------------------------------------------------
struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int B, h, h_kv, d_h, page_size, num_blocks, max_blocks_per_seq, num_splits;
  float scale;
  float* o_part;
  float* m_part;
  float* l_part;
  int fixed_pps = 0;  // > 0: fixed pages per split (split_plan_fixed)
  const int* pps_dev = nullptr;  // non-null: pages per split read from device memory
  // Non-null (a mixed batch's cu_seqlens_q [B + 1]): only rows with one query
  // are decoded, their query and output at token q_rows[b].
  const int32_t* q_rows = nullptr;
};
// One CTA: the batch's split count by splits_rule, as pages per split of the
// longest row, written to *pps_out (adaptive decode).
cudaError_t launch_decode_plan(const int32_t* seq_lens, const int32_t* q_rows, int B, int h_kv,
                               int max_len, int num_sms, int max_splits, int* pps_out,
                               cudaStream_t stream);
cudaError_t launch_decode_split(const DecodeArgs& a, cudaStream_t stream);
unsigned int decode_read_and_clear_error(cudaStream_t stream, cudaError_t* st);
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream);
// One CTA: lets the next kernel start, waits delay_ns, copies n int32.
cudaError_t launch_delayed_copy(int32_t* dst, const int32_t* src, int n, uint64_t delay_ns,
                                cudaStream_t stream);

// prefill_simt.cu ----------------------------------------------------------
cudaError_t launch_prefill_f32(const float* q, const float* k, const float* v, float* o,
                               float* lse, int T, int h, int h_kv, int d_h, int causal,
                               float scale, cudaStream_t stream);

// prefill_tc.cu --------------------------------------------------------------
// Workspace carve-up: fp16 copy of V [h_kv, T, d_h], then one int flag per
// (KV head, 128-key tile).
struct PrefillLayout {
  size_t v16_off, flags_off, sched_off, total;
};
PrefillLayout prefill_layout(int T, int h_kv, int d_h);
// workspace == nullptr: every key tile takes the exact bf16 P_hi + P_lo path.
cudaError_t launch_prefill_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                                int T, int h, int h_kv, int d_h, int causal, float scale,
                                void* workspace, cudaStream_t stream);
// Paged, variable-length prefill (arguments validated by the caller).
struct PagedPrefill {
  const void* q;            // [total_q, h, d_h] bf16
  const void* k_cache;      // [num_blocks, 16, h_kv, d_h] bf16
  const void* v_cache;
  const int32_t* block_table;  // [B, max_blocks]
  const int32_t* cu_q;         // [B + 1]
  const int32_t* seq_lens;     // [B]
  int32_t* tile_off;           // [B + 1] workspace
  void* v16;                   // fp16 V copy [B, max_tiles * 128, h_kv, d_h] or nullptr
  int32_t* vwide;              // [B, h_kv, max_tiles] V-format flags (with v16)
  int B, total_q, h, h_kv, d_h, num_blocks, max_blocks, max_q_len, causal;
  float scale;
  void* o;                     // [total_q, h, d_h] bf16
  float* lse;                  // [total_q, h] or nullptr
  int decode_rows_apart = 0;   // nonzero: rows of one query get no query tiles
};
cudaError_t launch_prefill_paged(const PagedPrefill& a, cudaStream_t stream);
unsigned int prefill_read_and_clear_error(cudaStream_t stream, cudaError_t* st);
// Debug builds: the key tile each prefill CTA skips loading K for (-1: none);
// cudaErrorNotSupported in release builds.
cudaError_t prefill_set_stall(int key_tile);
// The fp32 SIMT prefill's error word (debug-build index checks only).
unsigned int simt_read_and_clear_error(cudaStream_t stream, cudaError_t* st);

// tensor maps ---------------------------------------------------------------
// Encodes a tiled tensor map through the driver entry point (no libcuda link).
CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* base,
                           const uint64_t* dims, const uint64_t* strides_bytes,
                           const uint32_t* box, CUtensorMapSwizzle swizzle);

}  // namespace attn

// common.cuh -- device helpers shared by the kernels of this library:
// mbarrier / TMA / tcgen05 PTX wrappers, bounded waits, bf16 unpacking.
//
// Every wait on an mbarrier is bounded: after ATTN_WAIT_LIMIT_NS of polling it
// records ATTN_DEVERR_WAIT_TIMEOUT in the module's error word and returns
// false, and the caller takes its early exit. Nothing here traps.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"

#ifndef ATTN_WAIT_LIMIT_NS
#define ATTN_WAIT_LIMIT_NS 2000000000ull  // 2 s
#endif

// Debug builds (-DATTN_DEBUG) check indices and offsets on the kernels'
// global stores and on the shared-memory offsets they compute:
//   ATTN_GUARD(cond, err)  -> cond, after recording ATTN_DEVERR_DEBUG_INDEX in
//                             *err when it is false; the caller skips the
//                             access it guards;
//   ATTN_DCHECK(cond, err) -> records the same bit for an invariant whose
//                             violation cannot be skipped locally.
// Nothing traps. Release builds compile both to nothing (the condition is not
// evaluated).
#ifdef ATTN_DEBUG
#define ATTN_GUARD(cond, err) (::attn::debug_check(static_cast<bool>(cond), (err)))
#define ATTN_DCHECK(cond, err) ((void)::attn::debug_check(static_cast<bool>(cond), (err)))
#else
#define ATTN_GUARD(cond, err) (true)
#define ATTN_DCHECK(cond, err) ((void)0)
#endif

namespace attn {

__device__ __forceinline__ bool debug_check(bool ok, unsigned int* err) {
  if (!ok) atomicOr(err, ATTN_DEVERR_DEBUG_INDEX);
  return ok;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Split plan, shared by the decode producer, its reduce and the host.
// ---------------------------------------------------------------------------
// fixed_pps > 0: every split covers fixed_pps pages (the last one the rest),
// so a row's split boundaries depend on its own length only; the caller
// guarantees num_splits >= ceil(n_pages / fixed_pps).
__host__ __device__ __forceinline__ int split_plan_fixed(int seq_len, int page_size,
                                                         int num_splits, int fixed_pps,
                                                         int* pages_per_split) {
  const int n_pages = (seq_len + page_size - 1) / page_size;
  if (n_pages <= 0) {
    if (pages_per_split) *pages_per_split = 0;
    return 0;
  }
  const int pps = fixed_pps > 0 ? fixed_pps : (n_pages + num_splits - 1) / num_splits;
  if (pages_per_split) *pages_per_split = pps;
  return (n_pages + pps - 1) / pps;
}

__host__ __device__ __forceinline__ int split_plan(int seq_len, int page_size, int num_splits,
                                                   int* pages_per_split) {
  return split_plan_fixed(seq_len, page_size, num_splits, 0, pages_per_split);
}

// Split count for a decode batch ([DEC] "The grid": fill the first wave,
// S* = ceil(N_SM / (B h_kv))). A ragged batch (longest row > 1.25x the mean,
// known from total_len > 0) is raised until the longest row's split is at
// most a quarter of the mean work per SM; every split of the longest row then
// keeps at least 32 pages. Result in [1, max_splits]. The host recommendation
// and the on-device plan of the adaptive decode use this same function.
__host__ __device__ __forceinline__ int splits_rule(long long B, long long h_kv, long long max_len,
                                                    long long total_len, long long num_sms,
                                                    long long max_splits) {
  const long long g2d = B * h_kv;
  long long s = (num_sms + g2d - 1) / g2d;  // first-wave coverage
  const long long max_pages = (max_len + 15) / 16;
  if (total_len > 0 && 4ll * max_len * B > 5ll * total_len) {
    const long long total_pages = ((total_len + 15) / 16) * h_kv;
    const long long mean_per_sm = (total_pages + num_sms - 1) / num_sms;
    const long long target = mean_per_sm / 4 > 0 ? mean_per_sm / 4 : 1;
    const long long s_bal = (max_pages + target - 1) / target;
    if (s_bal > s) s = s_bal;
  }
  const long long s_work = (max_pages + 31) / 32;
  if (s > s_work) s = s_work;
  if (s < 1) s = 1;
  if (s > max_splits) s = max_splits;
  return static_cast<int>(s);
}

// Row length as the decode kernels use it: clamped into [0, max_blocks*page].
__device__ __forceinline__ int clamp_seq_len(int seq_len, int max_len, unsigned int* err) {
  if (seq_len < 0 || seq_len > max_len) {
    atomicOr(err, ATTN_DEVERR_BAD_SEQ_LEN);
    seq_len = seq_len < 0 ? 0 : max_len;
  }
  return seq_len;
}

// ---------------------------------------------------------------------------
// Small PTX wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Maximum that returns NaN when either operand is NaN (fmaxf returns the
// other one). Running maxima use it so that a NaN logit or state reaches the
// row's result as IEEE arithmetic on the definition would carry it, instead
// of dropping out of the max.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete: false, with
// ATTN_DEVERR_WAIT_TIMEOUT raised in *err, once limit_ns have passed.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, unsigned int* err,
                                              uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(err, ATTN_DEVERR_WAIT_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int* err) {
  return mbar_wait_for(bar, parity, err, ATTN_WAIT_LIMIT_NS);
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// TMA tile loads (global -> this CTA's shared memory), completion counted in
// bytes on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const void* tmap, uint32_t bar,
                                                 int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "l"(policy)
      : "memory");
}

// Prefetch of one tile box into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_3d(const void* tmap, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// bf16 helpers (exact widening of packed pairs).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 t = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

}  // namespace attn

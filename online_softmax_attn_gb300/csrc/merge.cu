// merge.cu -- N-way merge of split partial states (the reduce stage of
// split-KV decoding, also exported on its own as attn_merge_states).
//
// Math ("Decode attention: FlashDecoding, split-K, paged kernels", stage 2 of
// the split: take the overall max, rescale each split's l_i and O~_i by
// exp(m_i - M), sum, divide once; and "Merge normalized attention without
// averaging tile outputs": branch around the all-empty case instead of
// evaluating -inf - (-inf)).
//
// Layout: WPR warps per output row (1 for many rows, 8 when there are too
// few rows to fill the GPU, 32 for fewer than 128 rows of more than 64
// splits, and always 8 for fixed-size splits); lane j owns d_h/32 consecutive output elements,
// so each split's O~ row is read as one coalesced 128-bit (d_h=128) or 64-bit
// (d_h=64) access per lane. Warp w of a row takes splits w, w + WPR, ... in
// batches (4 splits per warp, 8 with WPR = 8) whose m, l and O~ loads are
// issued together; the first batch
// is issued beside the load that gives the active-split count (it stays
// inside the partial buffers, which hold all S splits, and a split found
// inactive is skipped, never multiplied by zero), so a row costs one memory
// round trip rather than three (count, then every m for the max, then O~).
// Each warp keeps a running (max, l, O~) over its splits -- the same merge,
// taken in a different order -- and with WPR > 1 the warps' states combine in
// shared memory.
#include "common.cuh"
#include "internal.h"
#include "pdl.cuh"

namespace attn {

static __device__ unsigned int g_merge_err;

template <int D, bool kOutBf16, int WPR>
__global__ void __launch_bounds__(WPR > 8 ? WPR * 32 : 256)
    merge_states_kernel(const float* __restrict__ o_part, const float* __restrict__ m_part,
                        const float* __restrict__ l_part, const int32_t* __restrict__ n_active,
                        const int32_t* __restrict__ seq_lens, int heads_per_seq, int page_size,
                        int max_len, int rows, int S, void* __restrict__ o_out, float* __restrict__ lse_out,
                        int fixed_pps, const int* __restrict__ pps_dev,
                        const int32_t* __restrict__ q_rows) {
  constexpr int VEC = D / 32;
  static_assert(VEC == 2 || VEC == 4, "d_h must be 64 or 128");
  constexpr int RPC = WPR > 8 ? 1 : 8 / WPR;  // rows per CTA (8 warps, or WPR warps for one row)
  // Splits per warp whose loads are in flight together: with 8 warps per row
  // a first batch of 8 covers 64 splits in one round trip, with 32 warps a
  // batch of 5 (what fits the 64 registers of a 1024-thread CTA) covers 160.
  constexpr int U = WPR > 8 ? 5 : (WPR > 1 ? 8 : 4);
  __shared__ float red_acc[WPR > 1 ? WPR * D : 1];
  __shared__ float red_m[WPR], red_l[WPR];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int wr = warp % WPR;  // this warp's share of the row
  const int row = blockIdx.x * RPC + warp / WPR;
  pdl_wait();  // the partials are the previous kernel's output
  pdl_trigger();
  if (WPR == 1 && row >= rows) return;
  bool live = row < rows;  // WPR > 1: one row per CTA
  // Where the row is written: the row itself, or in a mixed batch the token
  // of its sequence's one query (rows of longer sequences are not merged).
  size_t out_row = row;
  if (q_rows != nullptr && live) {
    const int b = row / heads_per_seq;
    const int r0 = q_rows[b], r1 = q_rows[b + 1];
    live = r1 - r0 == 1;
    out_row = size_t(r0) * heads_per_seq + row % heads_per_seq;
  }
  // Debug checks: the output row lies within the output (rows, or h per
  // query token of a mixed batch); a failed check leaves the row unwritten.
  if (live && !ATTN_GUARD(out_row < (q_rows != nullptr
                                          ? size_t(q_rows[rows / heads_per_seq]) * heads_per_seq
                                          : size_t(rows)),
                          &g_merge_err))
    live = false;
  if (WPR == 1 && !live) return;

  const float* mrow = m_part + size_t(row) * S;
  const float* lrow = l_part + size_t(row) * S;
  const float* orow = o_part + size_t(row) * S * D + lane * VEC;
  float mi[U], li[U], oi[U][VEC];
  auto load_batch = [&](int base, int lim) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * WPR;
      if (i < lim) {
        mi[u] = mrow[i];
        li[u] = lrow[i];
        const float* src = orow + size_t(i) * D;
        if constexpr (VEC == 4) {
          const float4 t = __ldg(reinterpret_cast<const float4*>(src));
          oi[u][0] = t.x; oi[u][1] = t.y; oi[u][2] = t.z; oi[u][3] = t.w;
        } else {
          const float2 t = __ldg(reinterpret_cast<const float2*>(src));
          oi[u][0] = t.x; oi[u][1] = t.y;
        }
      }
    }
  };
  // First batch: in flight beside the active-split count.
  if (live) load_batch(wr, S);

  int n = 0;
  if (live) {
    if (n_active != nullptr) {
      n = n_active[row];
    } else if (seq_lens != nullptr) {
      const int len = clamp_seq_len(seq_lens[row / heads_per_seq], max_len, &g_merge_err);
      n = split_plan_fixed(len, page_size, S, pps_dev ? *pps_dev : fixed_pps, nullptr);
    } else {
      n = S;
    }
    n = max(0, min(n, S));
  }

  // Running state over this warp's splits, exp2 domain for the max.
  float Mw = -INFINITY, Lw = 0.f, acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  auto merge_batch = [&](int base) {
    float bm = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (base + u * WPR < n) bm = fmax_nan(bm, mi[u] * kLog2e);
    if (bm == -INFINITY) return;  // no active split with keys in this batch
    const float Mn = fmax_nan(Mw, bm);
    const float sc = (Mw == -INFINITY) ? 0.f : ex2_approx(Mw - Mn);
    Lw *= sc;
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] *= sc;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (base + u * WPR < n && mi[u] != -INFINITY) {
        const float w = ex2_approx(fmaf(mi[u], kLog2e, -Mn));
        Lw = fmaf(w, li[u], Lw);
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = fmaf(w, oi[u][e], acc[e]);
      }
    }
    Mw = Mn;
  };
  if (live) {
    merge_batch(wr);
    for (int base = wr + U * WPR; base < n; base += U * WPR) {
      load_batch(base, n);
      merge_batch(base);
    }
  }

  float M = Mw, L = Lw;
  if constexpr (WPR > 1) {
#pragma unroll
    for (int e = 0; e < VEC; ++e) red_acc[wr * D + lane * VEC + e] = acc[e];
    if (lane == 0) {
      red_m[wr] = Mw;
      red_l[wr] = Lw;
    }
    __syncthreads();
    if (wr != 0 || !live) return;
    M = -INFINITY;
#pragma unroll
    for (int w = 0; w < WPR; ++w) M = fmax_nan(M, red_m[w]);
    L = 0.f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < WPR; ++w) {
        const float f = (red_m[w] == -INFINITY) ? 0.f : ex2_approx(red_m[w] - M);
        L = fmaf(f, red_l[w], L);
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = fmaf(f, red_acc[w * D + lane * VEC + e], acc[e]);
      }
    }
  }

  // No active split with a key (M = -inf) is the empty row. A NaN state
  // (NaN m, l or O~ in an active split) is not: it propagates to o and lse.
  const bool empty = M == -INFINITY;
  const float inv = empty ? 0.f : 1.f / L;
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = empty ? 0.f : acc[e] * inv;

  if constexpr (kOutBf16) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(o_out) +
                                                out_row * D + lane * VEC);
    if constexpr (VEC == 4) {
      uint2 pk;
      pk.x = pack_bf16x2(acc[0], acc[1]);
      pk.y = pack_bf16x2(acc[2], acc[3]);
      *reinterpret_cast<uint2*>(dst) = pk;
    } else {
      dst[0] = pack_bf16x2(acc[0], acc[1]);
    }
  } else {
    float* dst = static_cast<float*>(o_out) + out_row * D + lane * VEC;
    if constexpr (VEC == 4) {
      *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    } else {
      *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
    }
  }
  // M is in exp2 units here; the partials' m and the LSE are natural-log.
  if (lse_out != nullptr && lane == 0) lse_out[out_row] = empty ? -INFINITY : M * kLn2 + logf(L);
}

cudaError_t launch_merge(const float* o_part, const float* m_part, const float* l_part,
                         const int32_t* n_active, const int32_t* seq_lens, int heads_per_seq,
                         int page_size, int max_len, int rows, int num_splits, int d_h, void* o, float* lse,
                         attn_dtype_t out_dtype, cudaStream_t stream, int fixed_pps,
                         const int* pps_dev, const int32_t* q_rows) {
  if (rows <= 0) return cudaSuccess;
  // Few rows and many splits: spread each row's splits over 8 warps, or over
  // 32 (one 1024-thread CTA per row) when there are more than 64 splits and
  // under 128 rows, so that every split's loads go out in the first batch.
  // With fixed-size splits (the batch-invariant mode) always 8: the order in
  // which a row's splits are summed then depends on that row's split count
  // alone, not on the batch's rows or grid width.
  const bool wide = fixed_pps > 0 || (rows < 512 && num_splits > 4);
  const bool wider = fixed_pps == 0 && rows < 128 && num_splits > 64;
  const dim3 grid(wide ? rows : (rows + 7) / 8);
  const dim3 block(wider ? 1024 : 256);
  const bool bf = out_dtype == ATTN_DTYPE_BF16;
  cudaError_t e = cudaSuccess;
#define ATTN_MERGE_LAUNCH(D, BF, W)                                                               \
  e = launch_pdl(merge_states_kernel<D, BF, W>, grid, block, 0, stream, o_part, m_part, l_part, \
                 n_active, seq_lens, heads_per_seq, page_size, max_len, rows, num_splits, o, lse, \
                 fixed_pps, pps_dev, q_rows)
  if (d_h == 128) {
    if (bf) {
      if (wider) ATTN_MERGE_LAUNCH(128, true, 32);
      else if (wide) ATTN_MERGE_LAUNCH(128, true, 8);
      else ATTN_MERGE_LAUNCH(128, true, 1);
    } else {
      if (wider) ATTN_MERGE_LAUNCH(128, false, 32);
      else if (wide) ATTN_MERGE_LAUNCH(128, false, 8);
      else ATTN_MERGE_LAUNCH(128, false, 1);
    }
  } else {
    if (bf) {
      if (wider) ATTN_MERGE_LAUNCH(64, true, 32);
      else if (wide) ATTN_MERGE_LAUNCH(64, true, 8);
      else ATTN_MERGE_LAUNCH(64, true, 1);
    } else {
      if (wider) ATTN_MERGE_LAUNCH(64, false, 32);
      else if (wide) ATTN_MERGE_LAUNCH(64, false, 8);
      else ATTN_MERGE_LAUNCH(64, false, 1);
    }
  }
#undef ATTN_MERGE_LAUNCH
  return e;
}

// ---------------------------------------------------------------------------
// Pairwise (O, LSE) merge ("The state that gets passed around is the
// log-sum-exp"): each thread owns 8 consecutive elements of one row (16-byte
// bf16 or 32-byte fp32 accesses) and forms the row's two weights itself --
// recomputing two exponentials per thread is cheaper than sharing them.
// ---------------------------------------------------------------------------
template <bool kBf16>
__device__ __forceinline__ void load8(const void* base, size_t off, float (&v)[8]) {
  if constexpr (kBf16) {
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off));
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = bf16lo(w[e]);
      v[2 * e + 1] = bf16hi(w[e]);
    }
  } else {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    const float4 a = __ldg(src), b = __ldg(src + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

template <int D, bool kInBf16, bool kOutBf16>
__global__ void __launch_bounds__(256)
    merge_pair_kernel(const void* __restrict__ o_a, const float* __restrict__ lse_a,
                      const void* __restrict__ o_b, const float* __restrict__ lse_b, int rows,
                      void* o, float* __restrict__ lse) {
  constexpr int TPR = D / 8;  // threads per row
  const long long total = static_cast<long long>(rows) * TPR;
  for (long long it = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; it < total;
       it += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(it / TPR);
    const int part = static_cast<int>(it % TPR);
    const size_t off = static_cast<size_t>(row) * D + part * 8;
    const float la = lse_a[row], lb = lse_b[row];
    float va[8], vb[8], r[8];
    load8<kInBf16>(o_a, off, va);
    load8<kInBf16>(o_b, off, vb);
    const float M = fmax_nan(la, lb);  // a NaN side is not an empty one
    float L;
    if (M == -INFINITY) {  // both sides empty: no -inf - -inf
#pragma unroll
      for (int e = 0; e < 8; ++e) r[e] = 0.f;
      L = -INFINITY;
    } else {
      const float ea = (la == -INFINITY) ? 0.f : expf(la - M);
      const float eb = (lb == -INFINITY) ? 0.f : expf(lb - M);
      const float sum = ea + eb;
      const float wa = ea / sum, wb = eb / sum;  // weights first: a convex combination
#pragma unroll
      for (int e = 0; e < 8; ++e) r[e] = fmaf(wa, va[e], wb * vb[e]);
      L = M + logf(sum);
    }
    if constexpr (kOutBf16) {
      uint4 y;
      y.x = pack_bf16x2(r[0], r[1]);
      y.y = pack_bf16x2(r[2], r[3]);
      y.z = pack_bf16x2(r[4], r[5]);
      y.w = pack_bf16x2(r[6], r[7]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(o) + off) = y;
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(o) + off);
      dst[0] = make_float4(r[0], r[1], r[2], r[3]);
      dst[1] = make_float4(r[4], r[5], r[6], r[7]);
    }
    if (lse != nullptr && part == 0) lse[row] = L;
  }
}

cudaError_t launch_merge_pair(const void* o_a, const float* lse_a, const void* o_b,
                              const float* lse_b, int rows, int d_h, attn_dtype_t in_dtype,
                              void* o, float* lse, attn_dtype_t out_dtype, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    (void)cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long items = static_cast<long long>(rows) * (d_h / 8);
  const long long blocks = (items + 255) / 256;
  const int grid = static_cast<int>(blocks < 8ll * sms ? blocks : 8ll * sms);
  const bool ib = in_dtype == ATTN_DTYPE_BF16, ob = out_dtype == ATTN_DTYPE_BF16;
#define ATTN_PAIR(D, IB, OB) \
  merge_pair_kernel<D, IB, OB><<<grid, 256, 0, stream>>>(o_a, lse_a, o_b, lse_b, rows, o, lse)
  if (d_h == 128) {
    if (ib) { if (ob) ATTN_PAIR(128, true, true); else ATTN_PAIR(128, true, false); }
    else { if (ob) ATTN_PAIR(128, false, true); else ATTN_PAIR(128, false, false); }
  } else {
    if (ib) { if (ob) ATTN_PAIR(64, true, true); else ATTN_PAIR(64, true, false); }
    else { if (ob) ATTN_PAIR(64, false, true); else ATTN_PAIR(64, false, false); }
  }
#undef ATTN_PAIR
  return cudaGetLastError();
}

unsigned int merge_read_and_clear_error(cudaStream_t stream, cudaError_t* st) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_merge_err, sizeof(v), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_merge_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (st) *st = e;
  return v;
}

}  // namespace attn

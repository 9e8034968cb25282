// decode.cu -- stage 1 of split-KV paged decode attention.
//
// "Decode attention: FlashDecoding, split-K, paged kernels": with one query
// token per row there is too little query parallelism, so the key axis is cut
// into splits ("The grid", "Segment length, and the early exit"); each
// (row, KV head, split) gets one CTA that runs the online-softmax recurrence
// over its pages for all g = h/h_kv query heads sharing the KV head ("Where
// GQA enters": one K/V page load feeds g heads) and stores the unnormalised
// partial (O~, m, l) ("What the merge costs"). Pages are found through the
// block table (paged addressing: key p of row b sits in slot p % 16 of page
// block_table[b][p / 16]).
//
// GB300 design
//   * The work is HBM-bound (4 FLOP/byte for g = 4), so the kernel is built
//     around bytes in flight: each warp owns a private ring of NST stages, and
//     each stage receives one K page and one V page of its KV head (16 tokens x
//     d_h bf16 each) through a 4-D TMA tensor map over the cache
//     [num_blocks, 16, h_kv, d_h], in 64-element halves with the 128-byte
//     swizzle (so that fragment loads hit distinct shared-memory banks). The
//     page's 16 rows are gathered by the copy engine; the SM only waits on an
//     mbarrier.
//   * Per page, the two contractions are warp-level tensor-core MMAs
//     (m16n8k16, bf16 in, fp32 accumulate) with the g query heads of the KV
//     head as the M rows (rows g..15 are zero): S = q K^T over the page's 16
//     keys, then O~ += P V over d_h. The S accumulator fragment of a lane is
//     exactly the P operand fragment of the next MMA, so scores never leave
//     registers, and the fragments of K and V come from ldmatrix (V
//     transposed). This keeps the instruction count per page an order of
//     magnitude below a SIMT dot product with cross-lane reductions, so a warp
//     spends its time waiting for bytes rather than issuing.
//   * P is the exact two-term bf16 split P_hi + P_lo (P_hi = p truncated to
//     bf16, P_lo = bf16(p - P_hi)), two MMAs per V fragment: a single bf16 P
//     loses up to 2^-8 relative per weight, which rows dominated by a few keys
//     do not average away.
//   * Softmax statistics are per page: one max and one rescale per 16 keys,
//     in base 2 (scores are scaled by scale*log2(e) in fp32 after the MMA);
//     partial m is written back in natural-log units.
//   * Warps of a CTA take pages round-robin and merge their states through
//     shared memory at the end, so a CTA writes one partial per head.
//   * Launch geometry depends only on (B, h_kv, num_splits); surplus splits of
//     short rows return at once (CUDA-graph friendly).
#include "common.cuh"
#include "internal.h"
#include "pdl.cuh"

namespace attn {

static __device__ unsigned int g_decode_err;

namespace {

constexpr int kPage = 16;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D (16x8 fp32) += A (16x16 bf16, rows 8..15 zero) * B (16x8 bf16).
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

template <int D, int G, int NW, int NST>
struct DecodeCfg {
  static constexpr int HALVES = D / 64;             // 64-element (128-byte) swizzled halves
  static constexpr int HALF_BYTES = kPage * 128;    // one half of one page: 16 rows x 128 B
  static constexpr int PAGE_BYTES = kPage * D * 2;  // K or V page
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;
  static constexpr int RING_BYTES = NW * NST * STAGE_BYTES;
  static constexpr int MERGE_BYTES = NW * G * D * 4;
  static constexpr int ML_BYTES = NW * G * 2 * 4;
  static constexpr int BAR_BYTES = NW * NST * 8;
  static constexpr int SMEM = RING_BYTES + MERGE_BYTES + ML_BYTES + BAR_BYTES + 1024;
  static_assert(G <= 8, "the g heads of a KV head fill rows 0..7 of the MMA tile");
  static_assert(NST <= 32, "ring deeper than one block-table chunk");
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
};

// Shared address of the 16-byte chunk `chunk` (8 elements, 0 .. D/8-1) of
// token row `row` in a page stored as 128-byte-swizzled halves.
__device__ __forceinline__ uint32_t page_chunk(uint32_t page, int row, int chunk) {
  return page + (chunk >> 3) * (kPage * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// TMA prefetch of a 4-D tile into L2 (nothing is written to shared memory).
__device__ __forceinline__ void tma_prefetch_l2_4d(const void* tmap, int c0, int c1, int c2,
                                                   int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

template <int D, int G, int NW, int NST>
__global__ void __launch_bounds__(NW * 32, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ block_table,
                        const int32_t* __restrict__ seq_lens, int h, int max_blocks, int num_blocks,
                        int num_splits, int fixed_pps, const int* __restrict__ pps_dev,
                        const int32_t* __restrict__ q_rows, float qscale,
                        float* __restrict__ o_part, float* __restrict__ m_part,
                        float* __restrict__ l_part) {
  using C = DecodeCfg<D, G, NW, NST>;
  constexpr int KS = D / 16;  // k-steps of S = q K^T
  constexpr int ND = D / 8;   // n-tiles of O~ += P V

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int gid = lane >> 2;  // MMA row (query head) / key / dim held by this lane
  const int tq = lane & 3;    // column pair within the fragment

  // Before the dependency wait, warm L2 with this warp's first NST pages (a
  // TMA prefetch lands nothing in this SM). The seq_len, split plan and table
  // entries read here only steer the prefetch: were an earlier kernel still
  // writing them, some other page would be warmed, and the loads after the
  // wait read the right ones (L2 is the point of coherence). Every read of
  // seq_lens, the split plan and the table in this kernel goes to L2
  // (ld.global.cg): a line cached in L1 by an early read would otherwise
  // serve a later one the old value. Only the first wave of CTAs (one per
  // SM) can start before the previous kernel ends; the later ones would only
  // request their first pages twice.
  uint32_t n_sm;
  asm("mov.u32 %0, %%nsmid;" : "=r"(n_sm));
  const uint32_t cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  if (lane == 0 && cta < n_sm && q_rows == nullptr) {
    const int sl = min(max(__ldcg(seq_lens + b), 0), max_blocks * kPage);
    const int np = (sl + kPage - 1) / kPage;  // 0 .. max_blocks
    // Pages per split as the plan takes them. A value read this early may be
    // anything (the plan kernel may not have written it yet), so it is
    // bounded before use and every table index stays in [0, np).
    const int fp = pps_dev ? __ldcg(pps_dev) : fixed_pps;
    const int pps0 = fp > 0 ? min(fp, max(np, 1)) : (np + num_splits - 1) / num_splits;
    if (pps0 >= 1 && static_cast<long long>(split) * pps0 < np) {
      const int lo = split * pps0, hi = min(lo + pps0, np);
      for (int i = 0; i < NST; ++i) {
        const int p = lo + warp + NW * i;
        if (p >= hi) break;
        const int phys = __ldcg(block_table + size_t(b) * max_blocks + p);
        if (phys < 0 || phys >= num_blocks) continue;
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          tma_prefetch_l2_4d(&tmap_k, hf * 64, kvh, 0, phys);
          tma_prefetch_l2_4d(&tmap_v, hf * 64, kvh, 0, phys);
        }
      }
    }
  }
  pdl_wait();     // q, seq_lens, the split plan and the partials' buffers are the previous kernel's
  pdl_trigger();  // the merge may be scheduled once every split CTA is running

  // A mixed batch (q_rows = its cu_seqlens_q): only the rows with one query
  // are decoded here, their query at token q_rows[b]; the others return.
  size_t q_tok = b;
  if (q_rows != nullptr) {
    const int r0 = __ldcg(q_rows + b), r1 = __ldcg(q_rows + b + 1);
    if (r1 - r0 != 1) return;
    q_tok = r0;
  }

  // q fragments first: they do not depend on the row length. A-operand
  // layout of m16n8k16: a0 = (row gid, k 2tq..2tq+1), a2 = (row gid, k+8).
  uint32_t qa0[KS], qa2[KS];
  {
    // Debug checks: the head group lies within the row's h heads, and the
    // token within the query tokens (B, or q_rows[B] in a mixed batch).
    const bool q_ok = ATTN_GUARD(
        kvh * G + G <= h &&
            q_tok < (q_rows != nullptr ? size_t(__ldcg(q_rows + gridDim.z)) : size_t(gridDim.z)),
        &g_decode_err);
    const __nv_bfloat16* qr = q + (q_tok * h + kvh * G + min(gid, G - 1)) * D + 2 * tq;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint32_t x0 = q_ok ? __ldg(reinterpret_cast<const uint32_t*>(qr + 16 * ks)) : 0u;
      const uint32_t x2 = q_ok ? __ldg(reinterpret_cast<const uint32_t*>(qr + 16 * ks + 8)) : 0u;
      qa0[ks] = gid < G ? x0 : 0u;
      qa2[ks] = gid < G ? x2 : 0u;
    }
  }

  const int seq_len = clamp_seq_len(__ldcg(seq_lens + b), max_blocks * kPage, &g_decode_err);
  int pps = 0;
  const int n_act =
      split_plan_fixed(seq_len, kPage, num_splits, pps_dev ? __ldcg(pps_dev) : fixed_pps, &pps);
  if (split >= n_act) return;  // surplus split of a short (or empty) row

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  float* merge_acc = reinterpret_cast<float*>(smem + C::RING_BYTES);  // [NW][G][D]
  float* ml_s = merge_acc + NW * G * D;                                // [NW][G][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ml_s + NW * G * 2);    // [NW][NST]

  if (tid == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    for (int i = 0; i < NW * NST; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_barrier_init();
  }
  __syncthreads();

  const int n_pages = (seq_len + kPage - 1) / kPage;
  const int p_begin = split * pps;
  const int p_end = min(p_begin + pps, n_pages);
  const int span = p_end - p_begin;
  const int nloc = span > warp ? (span - warp + NW - 1) / NW : 0;
  const int32_t* bt_row = block_table + size_t(b) * max_blocks;

  const uint32_t ring_base = smem_u32(smem) + warp * NST * C::STAGE_BYTES;
  const uint32_t bar_base = smem_u32(&bars[warp * NST]);
  const uint64_t policy = policy_evict_first();

  // Block-table entries for this warp's pages, 32 at a time (lane i holds
  // local page 32*chunk + i).
  int bt_reg = lane < nloc ? __ldcg(bt_row + p_begin + warp + NW * lane) : -1;

  auto issue = [&](int i, int phys) {
    const int st = i % NST;
    const uint32_t dst = ring_base + st * C::STAGE_BYTES;
    const uint32_t bar = bar_base + st * 8;
    if (phys < 0 || phys >= num_blocks) atomicOr(&g_decode_err, ATTN_DEVERR_BAD_PAGE);
    // An out-of-range page coordinate is filled with zeros by the copy engine.
    mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
#pragma unroll
    for (int hf = 0; hf < C::HALVES; ++hf) {
      tma_load_4d_hint(dst + hf * C::HALF_BYTES, &tmap_k, bar, hf * 64, kvh, 0, phys, policy);
      tma_load_4d_hint(dst + C::PAGE_BYTES + hf * C::HALF_BYTES, &tmap_v, bar, hf * 64, kvh, 0,
                       phys, policy);
    }
  };

  const int npro = min(NST, nloc);
  int issued = npro;
  for (int i = 0; i < npro; ++i) {
    const int phys = __shfl_sync(0xffffffffu, bt_reg, i);
    if (lane == 0) issue(i, phys);
  }

  // O~ for head gid (rows 8..15 of the tile stay zero): o[nd][0..1] are dims
  // 8nd + 2tq, +1.
  float o[ND][4];
#pragma unroll
  for (int nd = 0; nd < ND; ++nd)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nd][e] = 0.f;
  float m_run = -INFINITY;  // base-2 running max of head gid (same on the 4 lanes of a quad)
  float l_lane = 0.f;       // this lane's share of the head's normaliser

  // ldmatrix row addresses (lane -> matrix lane/8, row lane%8).
  const int lm = lane >> 3, lr = lane & 7;
  const int k_row = 8 * (lm >> 1) + lr;  // S: matrices (keys 0-7 | 8-15) x (chunk | chunk+1)
  const int k_dc = lm & 1;
  const int v_row = 8 * (lm & 1) + lr;   // P V: matrices (keys 0-7 | 8-15) x (chunk | chunk+1)
  const int v_dc = lm >> 1;

  int failed_at = -1;
  for (int i = 0; i < nloc; ++i) {
    const int st = i % NST;
    if (!mbar_wait(bar_base + st * 8, (i / NST) & 1, &g_decode_err)) {
      failed_at = i;  // error word already set; results of this CTA are void
      break;
    }
    const uint32_t kp = ring_base + st * C::STAGE_BYTES;
    const uint32_t vp = kp + C::PAGE_BYTES;
    const int page = p_begin + warp + NW * i;
    const int valid = min(kPage, seq_len - page * kPage);
    if (valid < kPage) {
      // The row's last page: its slots past seq_len hold whatever the cache
      // holds there (possibly NaN or inf). Their weights are 0, but 0 * NaN
      // is NaN in the P V product, so those V rows are zeroed first.
      constexpr int CPR = D / 8;  // 16-byte chunks per row
      for (int c = lane; c < (kPage - valid) * CPR; c += 32)
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                         page_chunk(vp, valid + c / CPR, c % CPR)),
                     "r"(0u)
                     : "memory");
      fence_proxy_async_smem();  // before the stage is refilled by the copy engine
      __syncwarp();
    }

    // ---- S = q K^T: two 8-key n-tiles, KS k-steps ----
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t b00, b01, b10, b11;
      ldsm_x4(page_chunk(kp, k_row, 2 * ks + k_dc), b00, b01, b10, b11);
      mma_bf16(sc[0], qa0[ks], qa2[ks], b00, b01);
      mma_bf16(sc[1], qa0[ks], qa2[ks], b10, b11);
    }
    // This lane holds head gid's scores of keys 2tq, 2tq+1 (tile 0) and
    // 8+2tq, 9+2tq (tile 1).
    float s[4] = {sc[0][0] * qscale, sc[0][1] * qscale, sc[1][0] * qscale, sc[1][1] * qscale};
    if (valid < kPage) {
      if (2 * tq >= valid) s[0] = -INFINITY;
      if (2 * tq + 1 >= valid) s[1] = -INFINITY;
      if (8 + 2 * tq >= valid) s[2] = -INFINITY;
      if (9 + 2 * tq >= valid) s[3] = -INFINITY;
    }

    // ---- online update (one rescale per page) ----
    float mx = fmax_nan(fmax_nan(s[0], s[1]), fmax_nan(s[2], s[3]));
    mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // Finite (every page has a valid key) unless a logit is NaN, which then
    // carries through m, alpha, p, l and O~ to the row's result.
    const float m_new = fmax_nan(m_run, mx);
    const float alpha = ex2_approx(m_run - m_new);  // 0 while m_run = -inf
    m_run = m_new;
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = ex2_approx(s[e] - m_new);
    l_lane = fmaf(l_lane, alpha, (p[0] + p[1]) + (p[2] + p[3]));
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      o[nd][0] *= alpha;
      o[nd][1] *= alpha;
    }
    // P as the A operand (keys 2tq.. in a0, keys 8+2tq.. in a2), two bf16 terms.
    uint32_t ph0, ph2, pl0, pl2;
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(ph0) : "r"(__float_as_uint(p[0])), "r"(__float_as_uint(p[1])));
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(ph2) : "r"(__float_as_uint(p[2])), "r"(__float_as_uint(p[3])));
    pl0 = pack_bf16x2(p[0] - __uint_as_float(__float_as_uint(p[0]) & 0xffff0000u),
                      p[1] - __uint_as_float(__float_as_uint(p[1]) & 0xffff0000u));
    pl2 = pack_bf16x2(p[2] - __uint_as_float(__float_as_uint(p[2]) & 0xffff0000u),
                      p[3] - __uint_as_float(__float_as_uint(p[3]) & 0xffff0000u));

    // ---- O~ += P V: ND n-tiles of 8 dims, two at a time ----
#pragma unroll
    for (int nd = 0; nd < ND; nd += 2) {
      uint32_t b00, b01, b10, b11;
      ldsm_x4_t(page_chunk(vp, v_row, nd + v_dc), b00, b01, b10, b11);
      mma_bf16(o[nd], ph0, ph2, b00, b01);
      mma_bf16(o[nd], pl0, pl2, b00, b01);
      mma_bf16(o[nd + 1], ph0, ph2, b10, b11);
      mma_bf16(o[nd + 1], pl0, pl2, b10, b11);
    }
    __syncwarp();

    // ---- refill this stage with the page NST ahead ----
    const int inext = i + NST;
    if (inext < nloc) {
      if ((inext & 31) == 0)
        bt_reg = (inext + lane < nloc) ? __ldcg(bt_row + p_begin + warp + NW * (inext + lane)) : -1;
      const int phys = __shfl_sync(0xffffffffu, bt_reg, inext & 31);
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(inext, phys);
      }
      issued = inext + 1;
    }
  }
  if (failed_at >= 0) {
    // Give this warp's copies still in flight a bounded chance to land before
    // the CTA can exit; the CTA still joins the barrier below.
    for (int j = failed_at; j < issued; ++j)
      (void)mbar_wait(bar_base + (j % NST) * 8, (j / NST) & 1, &g_decode_err);
  }

  // ---- head gid's normaliser over its quad, then merge the warps ----
  l_lane += __shfl_xor_sync(0xffffffffu, l_lane, 1);
  l_lane += __shfl_xor_sync(0xffffffffu, l_lane, 2);
  if (gid < G) {
#pragma unroll
    for (int nd = 0; nd < ND; ++nd)
      *reinterpret_cast<float2*>(merge_acc + (warp * G + gid) * D + 8 * nd + 2 * tq) =
          make_float2(o[nd][0], o[nd][1]);
    if (tq == 0) {
      ml_s[(warp * G + gid) * 2 + 0] = nloc > 0 ? m_run : -INFINITY;
      ml_s[(warp * G + gid) * 2 + 1] = nloc > 0 ? l_lane : 0.f;
    }
  }
  __syncthreads();

  const size_t row0 = size_t(b) * h + kvh * G;
  for (int idx = tid; idx < G * D; idx += NW * 32) {
    const int hh = idx / D;
    const int e = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmax_nan(M, ml_s[(w * G + hh) * 2]);
    float A = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = ml_s[(w * G + hh) * 2];
      const float wt = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
      A = fmaf(wt, merge_acc[(w * G + hh) * D + e], A);
      L = fmaf(wt, ml_s[(w * G + hh) * 2 + 1], L);
    }
    const size_t prow = (row0 + hh) * num_splits + split;
    if (!ATTN_GUARD(prow < size_t(gridDim.z) * h * num_splits, &g_decode_err)) continue;
    o_part[prow * D + e] = A;
    if (e == 0) {
      m_part[prow] = M * kLn2;
      l_part[prow] = L;
    }
  }
}

template <int D, int G, int NW, int NST>
cudaError_t launch_cfg(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t stream) {
  using C = DecodeCfg<D, G, NW, NST>;
  auto kern = decode_split_kernel<D, G, NW, NST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.num_splits, a.h_kv, a.B);
  const float qscale = a.scale * kLog2e;
  return launch_pdl(kern, grid, dim3(NW * 32), C::SMEM, stream, tk, tv,
                    static_cast<const __nv_bfloat16*>(a.q), a.block_table, a.seq_lens, a.h,
                    a.max_blocks_per_seq, a.num_blocks, a.num_splits, a.fixed_pps, a.pps_dev,
                    a.q_rows, qscale, a.o_part, a.m_part, a.l_part);
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                     cudaStream_t stream) {
  const int g = a.h / a.h_kv;
  switch (g) {
    case 1: return launch_cfg<D, 1, 8, 3>(a, tk, tv, stream);
    case 2: return launch_cfg<D, 2, 8, 3>(a, tk, tv, stream);
    case 4: return launch_cfg<D, 4, 8, 3>(a, tk, tv, stream);
    case 8: return launch_cfg<D, 8, 8, 3>(a, tk, tv, stream);
    default: return cudaErrorInvalidValue;
  }
}

// On-device split plan of the adaptive decode: the batch's longest and total
// (clamped) length, splits_rule, then pages per split of the longest row. The
// split kernel and the merge read the result, so the launch geometry (a grid
// of max_splits) never depends on the lengths. With q_rows (a mixed batch's
// cu_seqlens_q) only the rows with one query count.
__global__ void __launch_bounds__(256)
    decode_plan_kernel(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ q_rows,
                       int B, int h_kv, int max_len, int num_sms, int max_splits,
                       int* __restrict__ pps_out) {
  __shared__ long long s_tot[256];
  __shared__ int s_max[256], s_cnt[256];
  long long tot = 0;
  int mx = 0, cnt = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    if (q_rows != nullptr && q_rows[b + 1] - q_rows[b] != 1) continue;
    const int len = clamp_seq_len(seq_lens[b], max_len, &g_decode_err);
    tot += len;
    mx = max(mx, len);
    ++cnt;
  }
  s_tot[threadIdx.x] = tot;
  s_max[threadIdx.x] = mx;
  s_cnt[threadIdx.x] = cnt;
  __syncthreads();
  for (int off = blockDim.x / 2; off > 0; off >>= 1) {
    if (threadIdx.x < off) {
      s_tot[threadIdx.x] += s_tot[threadIdx.x + off];
      s_max[threadIdx.x] = max(s_max[threadIdx.x], s_max[threadIdx.x + off]);
      s_cnt[threadIdx.x] += s_cnt[threadIdx.x + off];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int s = splits_rule(max(s_cnt[0], 1), h_kv, s_max[0], s_tot[0], num_sms, max_splits);
    const int max_pages = (s_max[0] + kPage - 1) / kPage;
    *pps_out = max(1, (max_pages + s - 1) / s);
  }
}

}  // namespace

cudaError_t launch_decode_plan(const int32_t* seq_lens, const int32_t* q_rows, int B, int h_kv,
                               int max_len, int num_sms, int max_splits, int* pps_out,
                               cudaStream_t stream) {
  decode_plan_kernel<<<1, 256, 0, stream>>>(seq_lens, q_rows, B, h_kv, max_len, num_sms,
                                            max_splits, pps_out);
  return cudaGetLastError();
}

cudaError_t launch_decode_split(const DecodeArgs& a, cudaStream_t stream) {
  CUtensorMap tk, tv;
  const uint64_t dims[4] = {uint64_t(a.d_h), uint64_t(a.h_kv), uint64_t(a.page_size),
                            uint64_t(a.num_blocks)};
  const uint64_t strides[3] = {uint64_t(a.d_h) * 2, uint64_t(a.h_kv) * a.d_h * 2,
                               uint64_t(a.page_size) * a.h_kv * a.d_h * 2};
  // 64-element (128-byte) boxes: the widest the 128-byte swizzle allows.
  const uint32_t box[4] = {64u, 1u, uint32_t(a.page_size), 1u};
  if (encode_tensor_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.k_cache),
                        dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (encode_tensor_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.v_cache),
                        dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (a.d_h == 128) return launch_d<128>(a, tk, tv, stream);
  return launch_d<64>(a, tk, tv, stream);
}

// Failure-detection self-test: one thread waits, with the kernels' bounded
// wait, on an mbarrier that nothing arrives on. The wait gives up after
// limit_ns, raises ATTN_DEVERR_WAIT_TIMEOUT in this module's error word, and
// the kernel returns.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1u);
  fence_barrier_init();
  (void)mbar_wait_for(b, 0, &g_decode_err, limit_ns);
}

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 1, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

// Self-test of the reads before the dependency wait: the next kernel on the
// stream (a programmatic dependent) may start at once, and after delay_ns this
// grid copies n int32 from src to dst, so that the next kernel's reads before
// its dependency wait see the old values. The delay is a bounded spin.
__global__ void delayed_copy_kernel(int32_t* __restrict__ dst, const int32_t* __restrict__ src,
                                    int n, uint64_t delay_ns) {
  pdl_trigger();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < delay_ns) {
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}

cudaError_t launch_delayed_copy(int32_t* dst, const int32_t* src, int n, uint64_t delay_ns,
                                cudaStream_t stream) {
  delayed_copy_kernel<<<1, 256, 0, stream>>>(dst, src, n, delay_ns);
  return cudaGetLastError();
}

unsigned int decode_read_and_clear_error(cudaStream_t stream, cudaError_t* st) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_decode_err, sizeof(v), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_decode_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (st) *st = e;
  return v;
}

}  // namespace attn

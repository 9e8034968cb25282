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
//     [num_blocks, 16, h_kv, d_h]. The page's 16 rows of 2*d_h bytes are
//     gathered by the copy engine; the SM only waits on an mbarrier.
//   * Arithmetic stays fp32 SIMT (no tensor cores: the contraction per page is
//     16 x d_h x g, far too thin, and the kernel is bandwidth-bound anyway).
//     A lane owns 8 consecutive d_h elements (one 16-byte shared-memory read
//     per row), keeps q for all g heads in registers, and the per-token dot
//     products are finished with a reduce-scatter across the d_h/8 lanes of a
//     row so that each lane ends with one head's score.
//   * Softmax statistics are per page: one max and one rescale per 16 keys,
//     in base 2 (q is pre-multiplied by scale*log2(e)); partial m is written
//     back in natural-log units.
//   * Warps of a CTA take pages round-robin and merge their states through
//     shared memory at the end, so a CTA writes one partial per head.
//   * Launch geometry depends only on (B, h_kv, num_splits); surplus splits of
//     short rows return at once (CUDA-graph friendly).
#include "common.cuh"
#include "internal.h"

namespace attn {

static __device__ unsigned int g_decode_err;

namespace {

constexpr int kPage = 16;

// Reduce-scatter of N per-lane partial sums across the LPT lanes of a row:
// afterwards lane's v[0] holds the full sum for value index
// (lane & (LPT-1)) >> log2(LPT/N).
template <int N, int MASK>
struct ReduceScatter {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (N > 1) {
      constexpr int H = N / 2;
      const bool up = (lane & MASK) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = up ? v[i] : v[i + H];
        const float keep = up ? v[i + H] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
      }
      ReduceScatter<H, MASK / 2>::run(v, lane);
    } else if constexpr (MASK >= 1) {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], MASK);
      ReduceScatter<1, MASK / 2>::run(v, lane);
    }
  }
};

template <int D, int G, int NW, int NST>
struct DecodeCfg {
  static constexpr int LPT = D / 8;          // lanes per token row
  static constexpr int TPS = 32 / LPT;       // token rows per warp step
  static constexpr int RS = kPage / TPS;     // steps per page
  static constexpr int PAGE_BYTES = kPage * D * 2;
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;  // K page + V page
  static constexpr int RING_BYTES = NW * NST * STAGE_BYTES;
  static constexpr int MERGE_BYTES = NW * G * D * 4;
  static constexpr int P_BYTES = NW * kPage * G * 4;
  static constexpr int A_BYTES = NW * G * 4;
  static constexpr int ML_BYTES = NW * G * 2 * 4;
  static constexpr int BAR_BYTES = NW * NST * 8;
  static constexpr int SMEM = RING_BYTES + MERGE_BYTES + P_BYTES + A_BYTES + ML_BYTES +
                              BAR_BYTES + 1024;  // + alignment slack
  static_assert(G <= LPT, "group size must not exceed lanes per row");
  static_assert(NST <= 32, "ring deeper than one block-table chunk");
};

template <int D, int G, int NW, int NST>
__global__ void __launch_bounds__(NW * 32, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ block_table,
                        const int32_t* __restrict__ seq_lens, int h, int max_blocks, int num_blocks,
                        int num_splits, float qscale, float* __restrict__ o_part,
                        float* __restrict__ m_part, float* __restrict__ l_part) {
  using C = DecodeCfg<D, G, NW, NST>;
  constexpr int LPT = C::LPT, TPS = C::TPS, RS = C::RS;
  constexpr int REP = LPT / G;  // lanes holding the same head's score in a row

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int h_kv = gridDim.y;
  const int seq_len = clamp_seq_len(seq_lens[b], max_blocks * kPage, &g_decode_err);
  int pps = 0;
  const int n_act = split_plan(seq_len, kPage, num_splits, &pps);
  if (split >= n_act) return;  // surplus split of a short (or empty) row

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  float* merge_acc = reinterpret_cast<float*>(smem + C::RING_BYTES);         // [NW][G][D]
  float* p_s = merge_acc + NW * G * D;                                       // [NW][16][G]
  float* a_s = p_s + NW * kPage * G;                                         // [NW][G]
  float* ml_s = a_s + NW * G;                                                // [NW][G][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ml_s + NW * G * 2);           // [NW][NST]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
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

  const int c = lane % LPT;   // d_h chunk of 8 elements
  const int tg = lane / LPT;  // token row within a step
  const int my_head = (lane % LPT) / REP;
  const bool rep = (lane % REP) == 0;

  // q for the g heads of this KV head, pre-scaled into the base-2 domain.
  float qf[G][8];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(
        q + (size_t(b) * h + kvh * G + hh) * D + c * 8));
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qf[hh][2 * e] = bf16lo(w4[e]) * qscale;
      qf[hh][2 * e + 1] = bf16hi(w4[e]) * qscale;
    }
  }

  float acc[G][8];
#pragma unroll
  for (int hh = 0; hh < G; ++hh)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[hh][e] = 0.f;
  float m_run = -INFINITY;  // base-2 running max for head my_head
  float l_run = 0.f;

  const uint32_t ring_base = smem_u32(ring) + warp * NST * C::STAGE_BYTES;
  const uint32_t bar_base = smem_u32(&bars[warp * NST]);
  const uint64_t policy = policy_evict_first();

  // Block-table entries for this warp's pages, 32 at a time (lane i holds
  // local page 32*chunk + i).
  int bt_reg = lane < nloc ? bt_row[p_begin + warp + NW * lane] : -1;

  auto issue = [&](int i, int phys) {
    const int st = i % NST;
    const uint32_t dst = ring_base + st * C::STAGE_BYTES;
    const uint32_t bar = bar_base + st * 8;
    if (phys < 0 || phys >= num_blocks) atomicOr(&g_decode_err, ATTN_DEVERR_BAD_PAGE);
    // An out-of-range page coordinate is filled with zeros by the copy engine.
    mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
    tma_load_4d_hint(dst, &tmap_k, bar, 0, kvh, 0, phys, policy);
    tma_load_4d_hint(dst + C::PAGE_BYTES, &tmap_v, bar, 0, kvh, 0, phys, policy);
  };

  const int npro = min(NST, nloc);
  int issued = npro;
  for (int i = 0; i < npro; ++i) {
    const int phys = __shfl_sync(0xffffffffu, bt_reg, i);
    if (lane == 0) issue(i, phys);
  }

  float* p_w = p_s + warp * kPage * G;
  float* a_w = a_s + warp * G;
  int failed_at = -1;
  for (int i = 0; i < nloc; ++i) {
    const int st = i % NST;
    if (!mbar_wait(bar_base + st * 8, (i / NST) & 1, &g_decode_err)) {
      failed_at = i;  // error word already set; results of this CTA are void
      break;
    }
    const uint8_t* kp = ring + (warp * NST + st) * C::STAGE_BYTES;
    const uint8_t* vp = kp + C::PAGE_BYTES;
    const int page = p_begin + warp + NW * i;
    const int valid = min(kPage, seq_len - page * kPage);

    // ---- scores for this page: s[r] = head my_head, token r*TPS + tg ----
    float s[RS];
#pragma unroll
    for (int r = 0; r < RS; ++r) {
      const int t = r * TPS + tg;
      const uint4 raw = *reinterpret_cast<const uint4*>(kp + t * D * 2 + c * 16);
      const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
      float kf[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kf[2 * e] = bf16lo(w4[e]);
        kf[2 * e + 1] = bf16hi(w4[e]);
      }
      float part[G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float a0 = qf[hh][0] * kf[0];
        float a1 = qf[hh][1] * kf[1];
#pragma unroll
        for (int e = 2; e < 8; e += 2) {
          a0 = fmaf(qf[hh][e], kf[e], a0);
          a1 = fmaf(qf[hh][e + 1], kf[e + 1], a1);
        }
        part[hh] = a0 + a1;
      }
      ReduceScatter<G, LPT / 2>::run(part, lane);
      s[r] = (t < valid) ? part[0] : -INFINITY;
    }

    // ---- online update (one rescale per page) ----
    float mx = s[0];
#pragma unroll
    for (int r = 1; r < RS; ++r) mx = fmaxf(mx, s[r]);
#pragma unroll
    for (int m = LPT; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    const float m_new = fmaxf(m_run, mx);  // finite: every page has a valid key
    const float alpha = ex2_approx(m_run - m_new);  // 0 while m_run = -inf
    float psum = 0.f;
    float p[RS];
#pragma unroll
    for (int r = 0; r < RS; ++r) {
      p[r] = ex2_approx(s[r] - m_new);
      psum += p[r];
    }
#pragma unroll
    for (int m = LPT; m < 32; m <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, m);
    l_run = fmaf(l_run, alpha, psum);
    m_run = m_new;

    if (rep) {
#pragma unroll
      for (int r = 0; r < RS; ++r) p_w[(r * TPS + tg) * G + my_head] = p[r];
      if (tg == 0) a_w[my_head] = alpha;
    }
    __syncwarp();

    // ---- rescale and accumulate P V ----
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float a = a_w[hh];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[hh][e] *= a;
    }
#pragma unroll
    for (int r = 0; r < RS; ++r) {
      const int t = r * TPS + tg;
      const uint4 raw = *reinterpret_cast<const uint4*>(vp + t * D * 2 + c * 16);
      const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
      float vf[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        vf[2 * e] = bf16lo(w4[e]);
        vf[2 * e + 1] = bf16hi(w4[e]);
      }
      float pv[G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) pv[hh] = p_w[t * G + hh];
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[hh][e] = fmaf(pv[hh], vf[e], acc[hh][e]);
    }
    __syncwarp();

    // ---- refill this stage with the page NST ahead ----
    const int inext = i + NST;
    if (inext < nloc) {
      if ((inext & 31) == 0)
        bt_reg = (inext + lane < nloc) ? bt_row[p_begin + warp + NW * (inext + lane)] : -1;
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

  // ---- fold the token rows of the warp, then merge warps ----
#pragma unroll
  for (int m = LPT; m < 32; m <<= 1)
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[hh][e] += __shfl_xor_sync(0xffffffffu, acc[hh][e], m);

  if (tg == 0) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float4* dst = reinterpret_cast<float4*>(merge_acc + (warp * G + hh) * D + c * 8);
      dst[0] = make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
      dst[1] = make_float4(acc[hh][4], acc[hh][5], acc[hh][6], acc[hh][7]);
    }
    if (rep) {
      ml_s[(warp * G + my_head) * 2 + 0] = m_run;
      ml_s[(warp * G + my_head) * 2 + 1] = l_run;
    }
  }
  __syncthreads();

  const size_t row0 = size_t(b) * h + kvh * G;
  for (int idx = tid; idx < G * D; idx += NW * 32) {
    const int hh = idx / D;
    const int e = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, ml_s[(w * G + hh) * 2]);
    float A = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = ml_s[(w * G + hh) * 2];
      const float wt = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
      A = fmaf(wt, merge_acc[(w * G + hh) * D + e], A);
      L = fmaf(wt, ml_s[(w * G + hh) * 2 + 1], L);
    }
    const size_t prow = (row0 + hh) * num_splits + split;
    o_part[prow * D + e] = A;
    if (e == 0) {
      m_part[prow] = M * kLn2;
      l_part[prow] = L;
    }
  }
  (void)h_kv;
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
  kern<<<grid, NW * 32, C::SMEM, stream>>>(
      tk, tv, static_cast<const __nv_bfloat16*>(a.q), a.block_table, a.seq_lens, a.h,
      a.max_blocks_per_seq, a.num_blocks, a.num_splits, qscale, a.o_part, a.m_part, a.l_part);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                     cudaStream_t stream) {
  const int g = a.h / a.h_kv;
  switch (g) {
    case 1: return launch_cfg<D, 1, 8, 3>(a, tk, tv, stream);
    case 2: return launch_cfg<D, 2, 8, 3>(a, tk, tv, stream);
    case 4: return launch_cfg<D, 4, 8, 3>(a, tk, tv, stream);
    case 8: return launch_cfg<D, 8, 8, 2>(a, tk, tv, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_split(const DecodeArgs& a, cudaStream_t stream) {
  CUtensorMap tk, tv;
  const uint64_t dims[4] = {uint64_t(a.d_h), uint64_t(a.h_kv), uint64_t(a.page_size),
                            uint64_t(a.num_blocks)};
  const uint64_t strides[3] = {uint64_t(a.d_h) * 2, uint64_t(a.h_kv) * a.d_h * 2,
                               uint64_t(a.page_size) * a.h_kv * a.d_h * 2};
  const uint32_t box[4] = {uint32_t(a.d_h), 1u, uint32_t(a.page_size), 1u};
  if (encode_tensor_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.k_cache),
                        dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (encode_tensor_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.v_cache),
                        dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (a.d_h == 128) return launch_d<128>(a, tk, tv, stream);
  return launch_d<64>(a, tk, tv, stream);
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

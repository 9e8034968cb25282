// prefill_tc.cu -- bf16 exact-attention prefill on the sm_103a tensor cores.
//
// Method ("Naive attention and the online softmax", (3) "The online
// recurrence" and "Extending the recurrence to the output"): each query row
// streams over key tiles carrying (m, l, O~); S = Q K^T and O~ += P V are the
// two dense contractions; the row max only ever rises, and when it does the
// old l and O~ are multiplied by exp(m_old - m_new); O = O~ / l at the end,
// LSE = m + ln l. "The Online Softmax Recurrence" / "Where it breaks": the
// statistics stay fp32 while P and the operands are bf16. The pages' own
// remark that any common shift is legal ("The state that gets passed around
// is the log-sum-exp") licenses the lazy rescale used here: the reference max
// is only moved when the row max exceeds it by more than 2^8 (in exp2 units),
// so most tiles skip the O~ rescale; O~ and l always share one reference, so
// the result is unchanged.
//
// GB300 design (one CTA per (KV head, 128-query block, pair of query heads)):
//   * warp 8      : TMA producer. Q tiles of both heads once, then K and V
//                   tiles of the shared KV head through an NS-stage ring
//                   (128-byte swizzle, 64-element boxes).
//   * warp 9      : tensor-memory allocator and MMA issuer (one thread).
//                   S_t = Q_t K^T (SS MMA, M=N=128, K=d_h) into tensor memory,
//                   O_t += P_t V (TS MMA: P read from tensor memory, V from
//                   shared memory, V consumed MN-major as stored).
//   * warps 0-3, 4-7 : one softmax warpgroup per query head; thread = row
//                   (tensor-memory lane), so the row max and sum need no
//                   shuffles. P (bf16) is written over the first 64 columns
//                   of its own S tile.
//   The two heads ping-pong: while one warpgroup exponentiates its S tile,
//   the tensor core runs the other head's P V and next Q K^T.
//   Causal CTAs visit only key tiles up to the diagonal (the masked half of
//   the FLOPs is skipped) and the grid runs the longest query blocks first.
//   Every mbarrier wait is bounded; on a timeout the CTA raises the error
//   word, drains its copies and MMAs (bounded), frees tensor memory and exits.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace attn {

static __device__ unsigned int g_prefill_err;

namespace {

constexpr int kBM = 128;  // query rows per tile (tensor-memory lanes)
constexpr int kBN = 128;  // keys per tile
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when max rises > 2^8

template <int D, int NQ, int NS>
struct PfCfg {
  static constexpr int SUBS = D / 64;                // 64-element swizzle atoms along d_h
  static constexpr int SUB_BYTES = 128 * 128;        // one atom column of a 128-row tile
  static constexpr int QTILE = kBM * D * 2;
  static constexpr int KTILE = kBN * D * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NQ * QTILE;
  static constexpr int V_OFF = K_OFF + NS * KTILE;
  static constexpr int BAR_OFF = V_OFF + NS * KTILE;
  // q_full, k_full[NS], v_full[NS], kv_empty[NS], s_full[NQ], p_full[NQ],
  // o_final[NQ], mma_done
  static constexpr int NBAR = 1 + 3 * NS + 3 * NQ + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM = MISC_OFF + 16 + 1024;  // + alignment slack
  static constexpr int TMEM_COLS = NQ == 1 ? 256 : 512;
  static constexpr int THREADS = NQ * 128 + 64;
  static constexpr int PRODUCER_WARP = NQ * 4;
  static constexpr int MMA_WARP = NQ * 4 + 1;
};

struct Bars {
  uint32_t base;
  int ns, nq;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (1 + ns + s); }
  __device__ uint32_t kv_empty(int s) const { return base + 8 * (1 + 2 * ns + s); }
  __device__ uint32_t s_full(int t) const { return base + 8 * (1 + 3 * ns + t); }
  __device__ uint32_t p_full(int t) const { return base + 8 * (1 + 3 * ns + nq + t); }
  __device__ uint32_t o_final(int t) const { return base + 8 * (1 + 3 * ns + 2 * nq + t); }
  __device__ uint32_t mma_done() const { return base + 8 * (1 + 3 * ns + 3 * nq); }
};

// Bounded wait that also gives up at once when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > ATTN_WAIT_LIMIT_NS) {
      atomicOr(&g_prefill_err, ATTN_DEVERR_WAIT_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

template <int D, int NQ, int NS>
__global__ void __launch_bounds__(PfCfg<D, NQ, NS>::THREADS, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int T, int h,
                        int h_kv, int causal, float scale_log2, int n_qblk) {
  using C = PfCfg<D, NQ, NS>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  Bars bars{sbase + C::BAR_OFF, NS, NQ};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qb = causal ? (n_qblk - 1 - int(blockIdx.x)) : int(blockIdx.x);
  const int hq0 = blockIdx.y * NQ;
  const int kvh = hq0 / (h / h_kv);
  const int n_kv_all = (T + kBN - 1) / kBN;
  const int nkv = causal ? min(qb + 1, n_kv_all) : n_kv_all;

  if (threadIdx.x == 0) {
    // p_full collects one arrival per softmax thread; the others take one.
    for (int i = 0; i < C::NBAR; ++i) {
      const uint32_t bar = bars.base + 8 * i;
      const bool is_p = bar >= bars.p_full(0) && bar < bars.p_full(0) + 8 * NQ;
      mbar_init(bar, is_p ? 128u : 1u);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::MMA_WARP) tc::alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmap_q);
      prefetch_tmap(&tmap_k);
      prefetch_tmap(&tmap_v);
      mbar_arrive_expect_tx(bars.q_full(), NQ * C::QTILE);
      for (int t = 0; t < NQ; ++t)
        for (int s = 0; s < C::SUBS; ++s)
          tma_load_3d(sbase + C::Q_OFF + t * C::QTILE + s * C::SUB_BYTES, &tmap_q, bars.q_full(),
                      s * 64, qb * kBM, hq0 + t);
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int st = j % NS;
        if (j >= NS && !wait_or_abort(bars.kv_empty(st), ((j / NS) - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(bars.k_full(st), C::KTILE);
        for (int s = 0; s < C::SUBS; ++s)
          tma_load_3d(sbase + C::K_OFF + st * C::KTILE + s * C::SUB_BYTES, &tmap_k,
                      bars.k_full(st), s * 64, j * kBN, kvh);
        mbar_arrive_expect_tx(bars.v_full(st), C::KTILE);
        for (int s = 0; s < C::SUBS; ++s)
          tma_load_3d(sbase + C::V_OFF + st * C::KTILE + s * C::SUB_BYTES, &tmap_v,
                      bars.v_full(st), s * 64, j * kBN, kvh);
        issued = j + 1;
      }
      if (*abort_flag) {
        // Drain: the newest load of each stage is the only one that can still
        // be in flight. Bounded waits, error already recorded.
        (void)mbar_wait(bars.q_full(), 0, &g_prefill_err);
        for (int j = max(0, issued - NS); j < issued; ++j) {
          (void)mbar_wait(bars.k_full(j % NS), (j / NS) & 1, &g_prefill_err);
          (void)mbar_wait(bars.v_full(j % NS), (j / NS) & 1, &g_prefill_err);
        }
      }
    }
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idO = tc::idesc_bf16_f32(kBM, D, false, true);
      const uint32_t q_s = sbase + C::Q_OFF, k_s = sbase + C::K_OFF, v_s = sbase + C::V_OFF;
      auto issue_s = [&](int t, int st) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::SUB_BYTES + (kk & 3) * 32;
          const uint64_t a = tc::sw128_desc(q_s + t * C::QTILE + off, 16, 1024);
          const uint64_t b = tc::sw128_desc(k_s + st * C::KTILE + off, 16, 1024);
          tc::mma_ss(tmem + t * 256, a, b, idS, kk > 0 ? 1u : 0u);
        }
      };
      // O_t += P_hi V + P_lo V (P_hi in S columns 0-63, P_lo in 64-127).
      auto issue_pv = [&](int t, int st, bool acc) {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t b = tc::sw128_desc(v_s + st * C::KTILE + kk * 16 * 128, C::SUB_BYTES, 1024);
          tc::mma_ts(tmem + t * 256 + 128, tmem + t * 256 + kk * 8, b, idO,
                     (acc || kk > 0) ? 1u : 0u);
          tc::mma_ts(tmem + t * 256 + 128, tmem + t * 256 + 64 + kk * 8, b, idO, 1u);
        }
      };
      bool ok = wait_or_abort(bars.q_full(), 0, abort_flag) &&
                wait_or_abort(bars.k_full(0), 0, abort_flag);
      if (ok) {
        tc::fence_after();
        for (int t = 0; t < NQ; ++t) {
          issue_s(t, 0);
          tc::commit(bars.s_full(t));
        }
      }
      for (int j = 0; ok && j < nkv; ++j) {
        const int st = j % NS;
        for (int t = 0; t < NQ && ok; ++t) {
          if (!wait_or_abort(bars.p_full(t), j & 1, abort_flag)) { ok = false; break; }
          if (t == 0 && !wait_or_abort(bars.v_full(st), (j / NS) & 1, abort_flag)) { ok = false; break; }
          tc::fence_after();
          issue_pv(t, st, j > 0);
          if (j == nkv - 1) tc::commit(bars.o_final(t));
          if (j + 1 < nkv) {
            const int st1 = (j + 1) % NS;
            if (t == 0 && !wait_or_abort(bars.k_full(st1), ((j + 1) / NS) & 1, abort_flag)) { ok = false; break; }
            tc::fence_after();
            issue_s(t, st1);
            tc::commit(bars.s_full(t));
          }
        }
        if (ok) tc::commit(bars.kv_empty(st));
      }
      // Everything issued by this thread has completed once mma_done flips.
      tc::commit(bars.mma_done());
      (void)mbar_wait(bars.mma_done(), 0, &g_prefill_err);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int row = qb * kBM + r;
    const int hq = hq0 + t;
    const uint32_t tS = tmem + (uint32_t(wq * 32) << 16) + t * 256;
    const uint32_t tO = tS + 128;
    float m_ref = -INFINITY;  // exp2-domain reference max shared by l and O~
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      // Warp-uniform outcome: the tensor-memory loads below are warp-collective.
      if (!__all_sync(0xffffffffu, wait_or_abort(bars.s_full(t), j & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc::fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::ld32(tS + c * 32, sr[c]);
      tc::wait_ld();

      int lim = kBN;
      if (j * kBN + kBN > T) lim = T - j * kBN;
      if (causal && j == qb) lim = min(lim, r + 1);
      float mx = -INFINITY;
      if (lim < kBN) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c * 32 + i >= lim) sr[c][i] = __float_as_uint(-INFINITY);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(sr[c][i]));

      const float m_cand = mx * scale_log2;
      const bool need = m_cand > m_ref + kRescaleThreshold;
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx(m_ref - m_cand);  // 0 on the first tile
        m_ref = m_cand;
      }
      const float bias = (m_ref == -INFINITY) ? 0.f : m_ref;
      // P = P_hi + P_lo, both bf16: P_hi = bf16(p), P_lo = bf16(p - P_hi).
      // The pair carries ~16 significant bits, so the rounding of P no longer
      // limits the output error (a single bf16 P costs up to 2^-8 relative
      // per weight, which rows dominated by a few keys do not average away).
      // Key pair (2i, 2i+1) of chunk c lands in P column 16c + i; P_hi fills
      // columns 0-63 and P_lo columns 64-127 of the S tile just read.
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c][2 * i]), scale_log2, -bias));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c][2 * i + 1]), scale_log2, -bias));
          sum += p0 + p1;
          ph[i] = pack_bf16x2(p0, p1);
          pl[i] = pack_bf16x2(p0 - bf16lo(ph[i]), p1 - bf16hi(ph[i]));
        }
        // sr[c] is consumed: reuse it to stage [P_hi | P_lo] of this chunk.
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          sr[c][i] = ph[i];
          sr[c][16 + i] = pl[i];
        }
      }
      l = fmaf(l, alpha, sum);
      {
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            hi[16 * c + i] = sr[c][i];
            lo[16 * c + i] = sr[c][16 + i];
          }
        tc::st32(tS, hi);        // P_hi keys 0..63
        tc::st32(tS + 64, lo);   // P_lo keys 0..63
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            hi[16 * c + i] = sr[2 + c][i];
            lo[16 * c + i] = sr[2 + c][16 + i];
          }
        tc::st32(tS + 32, hi);   // P_hi keys 64..127
        tc::st32(tS + 96, lo);   // P_lo keys 64..127
      }
      if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tc::ld32(tO + c * 32, ov);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tc::st32(tO + c * 32, ov);
        }
      }
      tc::wait_st();
      tc::fence_before();
      mbar_arrive(bars.p_full(t));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(bars.o_final(t), 0, abort_flag));
    if (ok) {
      tc::fence_after();
      const bool empty = !(l > 0.f);
      const float inv = empty ? 0.f : 1.f / l;
      __nv_bfloat16* orow = o + (size_t(hq) * T + row) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tc::ld32(tO + c * 32, ov);
        tc::wait_ld();
        if (row < T) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(ov[8 * i + 0]) * inv, __uint_as_float(ov[8 * i + 1]) * inv);
            pk.y = pack_bf16x2(__uint_as_float(ov[8 * i + 2]) * inv, __uint_as_float(ov[8 * i + 3]) * inv);
            pk.z = pack_bf16x2(__uint_as_float(ov[8 * i + 4]) * inv, __uint_as_float(ov[8 * i + 5]) * inv);
            pk.w = pack_bf16x2(__uint_as_float(ov[8 * i + 6]) * inv, __uint_as_float(ov[8 * i + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + 8 * i) = pk;
          }
        }
      }
      if (row < T && lse != nullptr)
        lse[size_t(hq) * T + row] = empty ? -INFINITY : (m_ref + log2f(l)) * kLn2;
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == C::MMA_WARP) tc::dealloc(tmem, C::TMEM_COLS);
}

template <int D, int NQ, int NS>
cudaError_t launch(const void* q, const void* k, const void* v, void* o, float* lse, int T, int h,
                   int h_kv, int causal, float scale, cudaStream_t stream) {
  using C = PfCfg<D, NQ, NS>;
  CUtensorMap tq, tk, tv;
  const uint32_t box[3] = {64u, 128u, 1u};
  {
    const uint64_t dims[3] = {uint64_t(D), uint64_t(T), uint64_t(h)};
    const uint64_t strides[2] = {uint64_t(D) * 2, uint64_t(T) * D * 2};
    if (encode_tensor_map(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {uint64_t(D), uint64_t(T), uint64_t(h_kv)};
    const uint64_t strides[2] = {uint64_t(D) * 2, uint64_t(T) * D * 2};
    if (encode_tensor_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (encode_tensor_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kern = prefill_bf16_kernel<D, NQ, NS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_qblk = (T + kBM - 1) / kBM;
  const dim3 grid(n_qblk, h / NQ);
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, static_cast<__nv_bfloat16*>(o), lse, T,
                                               h, h_kv, causal, scale * kLog2e, n_qblk);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                                int T, int h, int h_kv, int d_h, int causal, float scale,
                                cudaStream_t stream) {
  const int g = h / h_kv;
  const bool pair = (g % 2) == 0;
  if (d_h == 128) {
    return pair ? launch<128, 2, 2>(q, k, v, o, lse, T, h, h_kv, causal, scale, stream)
                : launch<128, 1, 3>(q, k, v, o, lse, T, h, h_kv, causal, scale, stream);
  }
  return pair ? launch<64, 2, 3>(q, k, v, o, lse, T, h, h_kv, causal, scale, stream)
              : launch<64, 1, 4>(q, k, v, o, lse, T, h, h_kv, causal, scale, stream);
}

unsigned int prefill_read_and_clear_error(cudaStream_t stream, cudaError_t* st) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_prefill_err, sizeof(v), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_prefill_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (st) *st = e;
  return v;
}

}  // namespace attn

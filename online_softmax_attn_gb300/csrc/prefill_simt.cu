// prefill_simt.cu -- fp32 exact-attention prefill on CUDA cores.
//
// The fp32 workload (single head, d_h = 64, fp32 output within 1e-4 of the
// float64 definition) needs fp32 products: tf32 or bf16 tensor-core operands
// would round q and k to 10 or 7 mantissa bits. This path therefore runs the
// online recurrence of "Naive attention and the online softmax", (3) and
// "Extending the recurrence to the output", with fp32 FMA:
//   per key tile: m_new = max(m, tile max); alpha = exp(m - m_new) (0 while
//   m = -inf); p = exp(s - m_new); l = alpha l + sum p; O~ = alpha O~ + P V;
// and divides once at the end (o = O~ / l, LSE = m + ln l; o = 0 and
// LSE = -inf for a row with no allowed key).
//
// CTA: 64 query rows x 4 threads per row (256 threads). Each tile of 32 keys
// and values is staged in shared memory (rows padded by one word against bank
// conflicts); thread c of a row computes scores for keys c, c+4, ... and owns
// output columns c, c+4, ... . Causal CTAs stop at their last allowed tile.
#include "common.cuh"
#include "internal.h"

namespace attn {

namespace {

constexpr int kRows = 64;
constexpr int kKeys = 32;

template <int D>
struct SimtCfg {
  static constexpr int LD = D + 1;
  static constexpr int SMEM = (kRows * LD + 2 * kKeys * LD + kRows * (kKeys + 1)) * 4;
};

template <int D>
__global__ void __launch_bounds__(256)
    prefill_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                       const float* __restrict__ v, float* __restrict__ o,
                       float* __restrict__ lse, int T, int h, int h_kv, int causal, float scale) {
  using C = SimtCfg<D>;
  constexpr int LD = C::LD;
  extern __shared__ float sm[];
  float* q_s = sm;                       // [64][LD]
  float* k_s = q_s + kRows * LD;         // [32][LD]
  float* v_s = k_s + kKeys * LD;         // [32][LD]
  float* p_s = v_s + kKeys * LD;         // [64][33]

  const int hq = blockIdx.y;
  const int kvh = hq / (h / h_kv);
  const int q0 = blockIdx.x * kRows;
  const int tid = threadIdx.x;
  const int r = tid >> 2;
  const int c = tid & 3;
  const int row = q0 + r;

  const float* qh = q + size_t(hq) * T * D;
  const float* kh = k + size_t(kvh) * T * D;
  const float* vh = v + size_t(kvh) * T * D;

  for (int i = tid; i < kRows * D; i += 256) {
    const int rr = i / D, e = i % D;
    q_s[rr * LD + e] = (q0 + rr < T) ? qh[size_t(q0 + rr) * D + e] : 0.f;
  }

  float acc[D / 4];
#pragma unroll
  for (int e = 0; e < D / 4; ++e) acc[e] = 0.f;
  float m = -INFINITY, l = 0.f;

  const int kend = causal ? min(T, q0 + kRows) : T;
  for (int k0 = 0; k0 < kend; k0 += kKeys) {
    __syncthreads();
    for (int i = tid; i < kKeys * D; i += 256) {
      const int j = i / D, e = i % D;
      const bool in = k0 + j < T;
      k_s[j * LD + e] = in ? kh[size_t(k0 + j) * D + e] : 0.f;
      v_s[j * LD + e] = in ? vh[size_t(k0 + j) * D + e] : 0.f;
    }
    __syncthreads();

    float s[kKeys / 4];
    float mx = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < kKeys / 4; ++jj) {
      const int j = c + 4 * jj;
      float a = 0.f;
#pragma unroll 16
      for (int e = 0; e < D; ++e) a = fmaf(q_s[r * LD + e], k_s[j * LD + e], a);
      const int key = k0 + j;
      const bool ok = key < T && row < T && (!causal || key <= row);
      s[jj] = ok ? a * scale : -INFINITY;
      mx = fmaxf(mx, s[jj]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m, mx);
    // A tile with no allowed key for this row leaves the state unchanged
    // (and avoids -inf - -inf).
    const bool any = m_new != -INFINITY;
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    float psum = 0.f;
#pragma unroll
    for (int jj = 0; jj < kKeys / 4; ++jj) {
      const float p = (any && s[jj] != -INFINITY) ? expf(s[jj] - m_new) : 0.f;
      p_s[r * (kKeys + 1) + c + 4 * jj] = p;
      psum += p;
    }
    psum += __shfl_xor_sync(0xffffffffu, psum, 1);
    psum += __shfl_xor_sync(0xffffffffu, psum, 2);
    __syncwarp();
    if (any) {
      l = l * alpha + psum;
      m = m_new;
#pragma unroll
      for (int e = 0; e < D / 4; ++e) acc[e] *= alpha;
#pragma unroll 4
      for (int j = 0; j < kKeys; ++j) {
        const float p = p_s[r * (kKeys + 1) + j];
#pragma unroll
        for (int e = 0; e < D / 4; ++e) acc[e] = fmaf(p, v_s[j * LD + c + 4 * e], acc[e]);
      }
    }
    __syncwarp();
  }

  if (row < T) {
    const bool empty = !(l > 0.f);
    const float inv = empty ? 0.f : 1.f / l;
    float* orow = o + (size_t(hq) * T + row) * D;
#pragma unroll
    for (int e = 0; e < D / 4; ++e) orow[c + 4 * e] = acc[e] * inv;
    if (lse != nullptr && c == 0) lse[size_t(hq) * T + row] = empty ? -INFINITY : m + logf(l);
  }
}

template <int D>
cudaError_t launch(const float* q, const float* k, const float* v, float* o, float* lse, int T,
                   int h, int h_kv, int causal, float scale, cudaStream_t stream) {
  auto kern = prefill_f32_kernel<D>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SimtCfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid((T + kRows - 1) / kRows, h);
  kern<<<grid, 256, SimtCfg<D>::SMEM, stream>>>(q, k, v, o, lse, T, h, h_kv, causal, scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_f32(const float* q, const float* k, const float* v, float* o,
                               float* lse, int T, int h, int h_kv, int d_h, int causal,
                               float scale, cudaStream_t stream) {
  if (d_h == 128) return launch<128>(q, k, v, o, lse, T, h, h_kv, causal, scale, stream);
  return launch<64>(q, k, v, o, lse, T, h, h_kv, causal, scale, stream);
}

}  // namespace attn

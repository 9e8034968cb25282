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
// CTA: 16 query rows x 16 threads per row (256 threads). A thread holds its
// row of q in registers; per tile of 32 keys and values staged in shared
// memory (rows padded by one word, so the 16 threads of a row read 16 banks),
// thread c of a row scores keys c and c+16 -- one shared-memory read per FMA,
// shared by the warp's two rows -- and owns output columns c, c+16, c+32, ...
// Row maxima and sums use 16-lane shuffles; the next tile's K and V are
// fetched into registers while this tile computes. Causal CTAs stop at their
// last allowed tile.
//
// Short sequences (too few query blocks to fill the SMs) split the key range
// over a thread-block cluster of S CTAs: each CTA runs the recurrence over its
// own run of key tiles, leaves its (m, l, O~) rows in shared memory, and after
// a cluster barrier each CTA finishes 16/S of the rows by reading all S states
// through distributed shared memory and applying the merge identity of
// "Merge normalized attention without averaging tile outputs" (new max =
// max m_i, l = sum exp(m_i - max) l_i, O~ likewise; all-empty rows give 0
// and -inf). The single-head 256 x 256 workload runs as 16 clusters of 8.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace attn {

// Device error word of this module (debug-build index checks).
static __device__ unsigned int g_simt_err;

namespace {

constexpr int kRows = 16;
constexpr int kTPR = 16;  // threads per row
constexpr int kKeys = 32;

template <int D>
struct SimtCfg {
  static constexpr int LD = D + 1;
  static constexpr int SMEM = (2 * kKeys * LD + kRows * (kKeys + 1)) * 4;
};

template <int D>
__global__ void __launch_bounds__(256)
    prefill_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                       const float* __restrict__ v, float* __restrict__ o,
                       float* __restrict__ lse, int T, int h, int h_kv, int causal, float scale,
                       int S) {
  using C = SimtCfg<D>;
  constexpr int LD = C::LD;
  constexpr int OC = D / kTPR;  // output columns per thread
  extern __shared__ float sm[];
  float* k_s = sm;               // [32][LD]
  float* v_s = k_s + kKeys * LD;  // [32][LD]
  float* p_s = v_s + kKeys * LD;  // [16][33]

  const int hq = blockIdx.y;
  const int kvh = hq / (h / h_kv);
  const int split = blockIdx.x % S;  // rank in the cluster (cluster dims S x 1 x 1)
  const int q0 = (blockIdx.x / S) * kRows;
  const int tid = threadIdx.x;
  const int r = tid / kTPR;
  const int c = tid % kTPR;
  const int row = q0 + r;

  const float* qh = q + size_t(hq) * T * D;
  const float* kh = k + size_t(kvh) * T * D;
  const float* vh = v + size_t(kvh) * T * D;

  float qr[D];
  {
    const float4* src = reinterpret_cast<const float4*>(qh + size_t(min(row, T - 1)) * D);
#pragma unroll
    for (int e = 0; e < D / 4; ++e) {
      const float4 x = __ldg(src + e);
      qr[4 * e] = x.x;
      qr[4 * e + 1] = x.y;
      qr[4 * e + 2] = x.z;
      qr[4 * e + 3] = x.w;
    }
  }

  float acc[OC];
#pragma unroll
  for (int e = 0; e < OC; ++e) acc[e] = 0.f;
  float m = -INFINITY, l = 0.f;

  // The next tile's K and V are fetched into registers while this tile
  // computes, so the global-load latency stays off the per-tile chain.
  constexpr int NV = kKeys * D / 4 / 256;  // float4s of K (and of V) per thread
  float4 kn[NV], vn[NV];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = tid + 256 * i, j = idx / (D / 4), e4 = idx % (D / 4);
      const bool in = k0 + j < T;
      kn[i] = in ? __ldg(reinterpret_cast<const float4*>(kh + size_t(k0 + j) * D) + e4)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
      vn[i] = in ? __ldg(reinterpret_cast<const float4*>(vh + size_t(k0 + j) * D) + e4)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };

  // This CTA's run of key tiles: [t_lo, t_hi) of the block's allowed tiles.
  const int kend = causal ? min(T, q0 + kRows) : T;
  const int n_tiles = (kend + kKeys - 1) / kKeys;
  const int per = (n_tiles + S - 1) / S;
  const int t_lo = min(n_tiles, split * per), t_hi = min(n_tiles, t_lo + per);
  const int k_hi = t_hi * kKeys;
  if (t_lo < t_hi) fetch(t_lo * kKeys);
  for (int k0 = t_lo * kKeys; k0 < k_hi; k0 += kKeys) {
    __syncthreads();  // every row is done with the previous tile
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = tid + 256 * i, j = idx / (D / 4), e4 = idx % (D / 4);
      float* kd = k_s + j * LD + 4 * e4;
      float* vd = v_s + j * LD + 4 * e4;
      kd[0] = kn[i].x; kd[1] = kn[i].y; kd[2] = kn[i].z; kd[3] = kn[i].w;
      vd[0] = vn[i].x; vd[1] = vn[i].y; vd[2] = vn[i].z; vd[3] = vn[i].w;
    }
    __syncthreads();
    if (k0 + kKeys < k_hi) fetch(k0 + kKeys);

    float s[2];
    float mx = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = c + kTPR * jj;
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < D; ++e) a = fmaf(qr[e], k_s[j * LD + e], a);
      const int key = k0 + j;
      const bool ok = key < T && row < T && (!causal || key <= row);
      s[jj] = ok ? a * scale : -INFINITY;
      mx = fmax_nan(mx, s[jj]);
    }
#pragma unroll
    for (int off = 1; off < kTPR; off <<= 1) mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmax_nan(m, mx);  // NaN once a logit is NaN: it then reaches O and the LSE
    // A tile with no allowed key for this row leaves the state unchanged
    // (and avoids -inf - -inf).
    const bool any = m_new != -INFINITY;
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    float psum = 0.f;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const float p = (any && s[jj] != -INFINITY) ? expf(s[jj] - m_new) : 0.f;
      p_s[r * (kKeys + 1) + c + kTPR * jj] = p;
      psum += p;
    }
#pragma unroll
    for (int off = 1; off < kTPR; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    __syncwarp();  // a row's 16 threads share one warp
    if (any) {
      l = l * alpha + psum;
      m = m_new;
#pragma unroll
      for (int e = 0; e < OC; ++e) acc[e] *= alpha;
      // Only the keys this row may attend: a masked key's weight is 0, but
      // 0 * NaN (or inf) in its V row would still reach the sum.
      const int j_end = min(kKeys, (causal ? min(row + 1, T) : T) - k0);
#pragma unroll 4
      for (int j = 0; j < j_end; ++j) {
        const float p = p_s[r * (kKeys + 1) + j];
#pragma unroll
        for (int e = 0; e < OC; ++e) acc[e] = fmaf(p, v_s[j * LD + c + kTPR * e], acc[e]);
      }
    }
    __syncwarp();
  }

  if (S == 1) {
    if (row < T) {
      const bool empty = l == 0.f;  // no allowed key; a NaN l is not empty
      const float inv = empty ? 0.f : 1.f / l;
      float* orow = o + (size_t(hq) * T + row) * D;
      if (ATTN_GUARD(hq < h, &g_simt_err)) {
#pragma unroll
        for (int e = 0; e < OC; ++e) orow[c + kTPR * e] = acc[e] * inv;
        if (lse != nullptr && c == 0) lse[size_t(hq) * T + row] = empty ? -INFINITY : m + logf(l);
      }
    }
    return;
  }

  // Cluster merge. The K tile's space holds this CTA's states:
  // m_s[16], l_s[16], a_s[16][D].
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __syncthreads();
  float* m_s = sm;
  float* l_s = m_s + kRows;
  float* a_s = l_s + kRows;
  if (c == 0) {
    m_s[r] = m;
    l_s[r] = l;
  }
#pragma unroll
  for (int e = 0; e < OC; ++e) a_s[r * D + c + kTPR * e] = acc[e];
  cluster.sync();  // every CTA's states are visible cluster-wide
  {
    const int R = kRows / S;  // rows this CTA finishes
    const int tpr = 256 / R;  // threads per finished row
    const int rl = split * R + tid / tpr;
    const int col0 = tid % tpr;
    const int grow = q0 + rl;
    float mi[8], w[8];
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      mi[i] = i < S ? *cluster.map_shared_rank(m_s + rl, i) : -INFINITY;
      M = fmax_nan(M, mi[i]);
    }
    float L = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      w[i] = (M != -INFINITY && mi[i] != -INFINITY) ? expf(mi[i] - M) : 0.f;
      if (w[i] != 0.f) L += w[i] * *cluster.map_shared_rank(l_s + rl, i);
    }
    const bool empty = M == -INFINITY;  // no CTA saw an allowed key; NaN states propagate
    if (grow < T && ATTN_GUARD(hq < h, &g_simt_err)) {
      float* orow = o + (size_t(hq) * T + grow) * D;
      for (int col = col0; col < D; col += tpr) {
        float x = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (w[i] != 0.f) x += w[i] * *cluster.map_shared_rank(a_s + rl * D + col, i);
        orow[col] = empty ? 0.f : x / L;
      }
      if (lse != nullptr && col0 == 0) lse[size_t(hq) * T + grow] = empty ? -INFINITY : M + logf(L);
    }
  }
  cluster.sync();  // no CTA leaves while another still reads its states
}

// Cluster size for the key split: doubled while the grid stays within two
// CTAs per SM and every CTA keeps at least one key tile.
int split_count(int T, int h) {
  const long blocks = long((T + kRows - 1) / kRows) * h;
  const int tiles = (T + kKeys - 1) / kKeys;
  int S = 1;
  while (S < 8 && blocks * 2 * S <= 2 * 152 && tiles >= 2 * S) S *= 2;
  return S;
}

template <int D>
cudaError_t launch(const float* q, const float* k, const float* v, float* o, float* lse, int T,
                   int h, int h_kv, int causal, float scale, cudaStream_t stream) {
  // Under the 48 KB default: no shared-memory attribute call per launch.
  static_assert(SimtCfg<D>::SMEM <= 48 * 1024, "fp32 prefill tile exceeds default shared memory");
  static_assert((kRows + kRows + kRows * D) <= kKeys * SimtCfg<D>::LD, "states exceed the K tile");
  const int S = split_count(T, h);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((T + kRows - 1) / kRows) * S, h);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = SimtCfg<D>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_f32_kernel<D>, q, k, v, o, lse, T, h, h_kv, causal, scale,
                            S);
}

}  // namespace

unsigned int simt_read_and_clear_error(cudaStream_t stream, cudaError_t* st) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_simt_err, sizeof(v), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_simt_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (st) *st = e;
  return v;
}

cudaError_t launch_prefill_f32(const float* q, const float* k, const float* v, float* o,
                               float* lse, int T, int h, int h_kv, int d_h, int causal,
                               float scale, cudaStream_t stream) {
  if (d_h == 128) return launch<128>(q, k, v, o, lse, T, h, h_kv, causal, scale, stream);
  return launch<64>(q, k, v, o, lse, T, h, h_kv, causal, scale, stream);
}

}  // namespace attn

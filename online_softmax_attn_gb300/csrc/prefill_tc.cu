// prefill_tc.cu -- bf16 exact-attention prefill on the sm_103a tensor cores.
//
// Method ("Naive attention and the online softmax", (3) "The online
// recurrence" and "Extending the recurrence to the output"): each query row
// streams over key tiles carrying (m, l, O~); S = Q K^T and O~ += P V are the
// two dense contractions; the row max only ever rises, and when it does the
// old l and O~ are multiplied by exp(m_old - m_new); O = O~ / l at the end,
// LSE = m + ln l. "The Online Softmax Recurrence" / "Where it breaks": the
// statistics stay fp32 while the operands are 16-bit. The pages' remark that
// any common shift is legal ("The state that gets passed around is the
// log-sum-exp") licenses the reference used here: l, O~ and each tile's
// weights P share one exp2-domain reference m_ref, which need not be the row
// max. Every tile takes its row max; the reference moves only when that max
// passes it by more than 15 (weights then still fit fp16), and it moves to 8
// above the max, so O~ is rescaled rarely; the rescale runs after P is
// stored, in the registers S held. O = O~ / l and LSE are independent of the
// reference.
//
// GB300 design (work item: a 128-query block of a pair of query heads that
// share a KV head; contiguous rows run a persistent grid of one CTA per SM,
// paged rows one CTA per item):
//   * softmax warpgroups (warps 0-3, 4-7), one per query head; thread = row
//     (tensor-memory lane), so row sums and maxima need no shuffles. P is
//     written over the first columns of its own S tile: fp16 for a V tile
//     that converts to fp16 exactly, else bf16 P_hi and P_lo.
//   * control warpgroup: warp 8 is the TMA producer (Q of both heads per item,
//     then K and V of the shared KV head through rings of their own, 128-byte
//     swizzle, 64-element boxes); warp 9 allocates tensor memory and issues
//     the MMAs as a whole warp (elect.sync picks the issuing lane):
//     S_t = Q_t K^T (SS, M=N=128, K=d_h) and O_t += P_t V (TS: P from tensor
//     memory, V from shared memory, MN-major as stored); warps 10-11 idle.
//   * before it, v_to_f16_kernel converts V once per KV head into an fp16
//     copy (exact for |v| < 2^16) and flags each 128-key tile holding a value
//     fp16 cannot carry; flagged tiles are read as bf16 and take P_hi + P_lo.
//   The two heads ping-pong: while one warpgroup exponentiates its S tile,
//   the tensor core runs the other head's P V and next Q K^T.
//   Causal items visit only key tiles up to the diagonal (the masked half of
//   the FLOPs is skipped); the longest query blocks are handed out first.
//   A persistent CTA claims its next item as it issues the current one's last
//   loads, loads the next Q once the current item's last S MMA is done, and
//   runs the next item's first S MMAs while its softmax warps store O (staged
//   in two V stages, not in Q), so set-up and drain overlap work.
//   Every mbarrier wait is bounded; on a timeout the CTA raises the error
//   word, drains its copies and MMAs (bounded), frees tensor memory and exits.
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "pdl.cuh"
#include "tc.cuh"

namespace attn {

static __device__ unsigned int g_prefill_err;
#ifdef ATTN_DEBUG
// Self-test of the abort path: the key tile (counted over a CTA's items) whose
// K each CTA does not load, or -1.
static __device__ int g_prefill_stall_tile = -1;
#endif

namespace {

constexpr int kBM = 128;  // query rows per tile (tensor-memory lanes)
constexpr int kBN = 128;  // keys per tile
// The reference moves only when the row max exceeds it by more than this (log2
// units): weights stay at most 2^15, below fp16's largest finite value (65504).
constexpr float kRescaleBits = 15.0f;
// When it moves, the reference goes this far above the row max, so the max
// may grow by kRescaleBits + kRefHeadroom before the next move (on logits with
// a standard deviation of 9 that cuts the 32-row warps that move per tile from
// about 23% to 6%). Weights under 2^-14 are then fp16 subnormals: absolute
// error at most 2^-25 against a row sum of at least 2^-kRefHeadroom, i.e. at
// most 2^-17 of the sum per key.
constexpr float kRefHeadroom = 8.0f;

template <int D, int NQ, int NSK, int NSV>
struct PfCfg {
  static constexpr int SUBS = D / 64;                // 64-element swizzle atoms along d_h
  static constexpr int SUB_BYTES = 128 * 128;        // one atom column of a 128-row tile
  static constexpr int QTILE = kBM * D * 2;
  static constexpr int KTILE = kBN * D * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NQ * QTILE;
  static constexpr int V_OFF = K_OFF + NSK * KTILE;
  static constexpr int BAR_OFF = V_OFF + NSV * KTILE;
  // q_full, k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full[NQ],
  // p_full[NQ], o_final[NQ], mma_done, q_empty, stage_free[2], item_full[2]
  static constexpr int NBAR = 1 + 2 * NSK + 2 * NSV + 3 * NQ + 1 + 5;
  static_assert(NSV >= 3, "the epilogue stages O in two V stages the next item does not load first");
  static_assert(NBAR <= 32, "one warp initialises the barriers, one per lane");
  // tensor-memory slot, abort flag, tail tile (2 ints), item slots (2 ints)
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM = MISC_OFF + 32 + 1024;  // + alignment slack
  static constexpr int TMEM_COLS = NQ == 1 ? 256 : 512;
  // NQ softmax warpgroups + one control warpgroup (TMA warp, MMA warp, two
  // idle warps: setmaxnreg moves registers per whole warpgroup).
  static constexpr int THREADS = NQ * 128 + 128;
  static constexpr int PRODUCER_WARP = NQ * 4;
  static constexpr int MMA_WARP = NQ * 4 + 1;
  // Register split (NQ = 2): launched at 168/thread (384 x 168 = 64512);
  // control warpgroup drops to 120, softmax warpgroups rise to 192:
  // 2 x 128 x 192 + 128 x 120 = 64512, the whole launch allocation. (With
  // the O~ rescale after the P store the softmax fits 192; 88 registers
  // spilled in the control warps, and 112 spilled a few words once the
  // producer claimed items.)
  static constexpr int REG_LAUNCH = 168;
  static constexpr int REG_CONTROL = 120;
  static constexpr int REG_SOFTMAX = 192;
  static_assert(NQ != 2 || 2 * 128 * REG_SOFTMAX + 128 * REG_CONTROL <= THREADS * REG_LAUNCH,
                "register split exceeds the launch allocation");
};

template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed fp32 pairs (two lanes of one 64-bit register pair).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

struct Bars {
  uint32_t base;
  int nsk, nsv, nq;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t k_full(int s) const { return base + 8 * (1 + s); }
  __device__ uint32_t k_empty(int s) const { return base + 8 * (1 + nsk + s); }
  __device__ uint32_t v_full(int s) const { return base + 8 * (1 + 2 * nsk + s); }
  __device__ uint32_t v_empty(int s) const { return base + 8 * (1 + 2 * nsk + nsv + s); }
  __device__ uint32_t s_full(int t) const { return base + 8 * (1 + 2 * nsk + 2 * nsv + t); }
  __device__ uint32_t p_full(int t) const { return base + 8 * (1 + 2 * nsk + 2 * nsv + nq + t); }
  __device__ uint32_t o_final(int t) const {
    return base + 8 * (1 + 2 * nsk + 2 * nsv + 2 * nq + t);
  }
  __device__ uint32_t mma_done() const { return base + 8 * (1 + 2 * nsk + 2 * nsv + 3 * nq); }
  // Q's shared memory is free: the item's last S MMA has completed.
  __device__ uint32_t q_empty() const { return base + 8 * (2 + 2 * nsk + 2 * nsv + 3 * nq); }
  // An item's O rows have left the V stages they were staged in; items
  // alternate between the two barriers.
  __device__ uint32_t stage_free(int i) const {
    return base + 8 * (3 + 2 * nsk + 2 * nsv + 3 * nq + i);
  }
  // The producer has written the index of the CTA's next item (or -1: none
  // left) into item slot i; items alternate between the two.
  __device__ uint32_t item_full(int i) const {
    return base + 8 * (5 + 2 * nsk + 2 * nsv + 3 * nq + i);
  }
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

// Paged, variable-length rows (PAGED kernels): queries are packed token-major
// [total_q, h, d_h]; row b's queries are tokens cu_q[b] .. cu_q[b+1]-1 and
// sit at the last q_len positions of its seq_lens[b] keys, which live in the
// paged cache [num_blocks, 16, h_kv, d_h] through block_table row b.
// tile_off[b] is row b's first 128-query tile (tile_off[B]: all tiles).
struct PagedArgs {
  const int32_t* block_table;
  const int32_t* cu_q;
  const int32_t* seq_lens;
  const int32_t* tile_off;
  int B, max_blocks, num_blocks;
  int max_tiles;  // 128-key tiles per row in the fp16 V copy: ceil(max_blocks / 8)
};

// One work item: a 128-query block of NQ query heads that share a KV head.
struct Work {
  int hq0;       // first query head
  int kvh;       // their KV head
  int qb;        // query block (paged rows: the block within row pb)
  int nkv;       // key tiles the block visits
  int n_kv_all;  // key tiles of the KV head (contiguous) or row (paged)
  int pb, q_tok0, q_len, ctx, n_pages;  // paged rows only
};

// P of a key tile whose V stays bf16 (a value of magnitude 2^16 or more, an
// inf or a NaN): P = P_hi + P_lo, both bf16, P_hi in columns 0-63 of the S
// tile and P_lo in columns 64-127. Such tiles are rare, so this runs out of
// line, which keeps the softmax loop's code small. It reads the S tile again
// from tensor memory (the caller's registers hold it only up to the row max),
// masks keys from lim on to -inf as the caller did, and returns the row sum of
// the weights, added up in the same order as the fp16 path. Warp-collective.
__device__ __noinline__ float softmax_p_two_term(uint32_t tS, int lim, float scale_log2,
                                                 float bias) {
  uint32_t sr[4][32];
#pragma unroll
  for (int c = 0; c < 4; ++c) tc::ld32(tS + c * 32, sr[c]);
  tc::wait_ld();
  if (lim < kBN) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (c * 32 + i >= lim) sr[c][i] = __float_as_uint(-INFINITY);
  }
  const uint64_t c2 = f2(scale_log2, scale_log2);
  const uint64_t nb2 = f2(-bias, -bias);
  uint64_t sumA = f2(0.f, 0.f), sumB = f2(0.f, 0.f);
  // P = P_hi + P_lo, both bf16. P_hi is p truncated to bf16 (its upper
  // 16 bits), P_lo = bf16(p - P_hi) (the difference is exact in fp32),
  // so the pair carries ~16 significant bits (a single bf16 P costs up
  // to 2^-8 relative per weight, which rows dominated by a few keys do
  // not average away). Within chunk c, sr[c][2i] is reused for the
  // P_hi pair of keys (2i, 2i+1), sr[c][2i+1] for P_lo.
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float y0, y1;
      unf2(fma2(f2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), c2,
                nb2),
           y0, y1);
      const float p0 = ex2_approx(y0);
      const float p1 = ex2_approx(y1);
      const uint64_t pp = f2(p0, p1);
      if (i & 1) sumB = add2(sumB, pp); else sumA = add2(sumA, pp);
      const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
      uint32_t hi;
      asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(hi) : "r"(u0), "r"(u1));
      float d0, d1;
      unf2(sub2(pp, f2(__uint_as_float(u0 & 0xffff0000u), __uint_as_float(u1 & 0xffff0000u))),
           d0, d1);
      sr[c][2 * i] = hi;
      sr[c][2 * i + 1] = pack_bf16x2(d0, d1);
    }
  }
  // P_hi fills columns 0-63 and P_lo columns 64-127.
  uint32_t hi[32], lo[32];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        hi[16 * c + i] = sr[2 * half + c][2 * i];
        lo[16 * c + i] = sr[2 * half + c][2 * i + 1];
      }
    tc::st32(tS + 32 * half, hi);       // P_hi keys 64*half .. +63
    tc::st32(tS + 64 + 32 * half, lo);  // P_lo keys 64*half .. +63
  }
  float sa0, sa1;
  unf2(add2(sumA, sumB), sa0, sa1);
  return sa0 + sa1;
}

// PAGED: variable-length rows over a paged cache. PCOPY (paged only): V is
// read from the workspace copy that paged_v_to_f16_kernel made (fp16 bits
// for normal tiles, bf16 bits for flagged ones), else from the cache itself.
template <int D, int NQ, int NSK, int NSV, bool PAGED, bool PCOPY>
__global__ void __launch_bounds__(PfCfg<D, NQ, NSK, NSV>::THREADS, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ CUtensorMap tmap_v16,
                        const int* __restrict__ vwide, __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int T, int h,
                        int h_kv, int causal, float scale_log2, int n_qblk,
                        int* __restrict__ sched, const PagedArgs pa) {
  using C = PfCfg<D, NQ, NSK, NSV>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  Bars bars{sbase + C::BAR_OFF, NSK, NSV, NQ};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  // Paged rows read from the cache whose last page is partial: the key tile
  // holding that page, then (packed) the first slot past the row's last key
  // within the tile and the number of such slots up to the page's end. Kept
  // in shared memory so that no warp holds registers for it.
  int* tail_info = reinterpret_cast<int*>(smem + C::MISC_OFF + 8);
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 16);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_hp = h / NQ;
  // Work items. Contiguous rows: the grid is persistent (one CTA per SM at
  // most); item i is head group i % n_hp of the query block with the
  // (i / n_hp)-th most key tiles (causal: the longest blocks first). CTA c
  // starts with item c; the producer claims each next item from the counter
  // *sched (the V pass zeroes it), which hands out G, G + 1, ... in order, so
  // the CTA that runs out of work first takes the longest item left. Without
  // a counter the CTA takes round r's item c (rounds of G = gridDim.x items)
  // when r is even and item G - 1 - c when r is odd. The producer publishes
  // each item in an item slot; the other roles read it there. Paged rows:
  // one item, the CTA's own (grid: head groups x the rows' query tiles, each
  // row's longest tile first).
  const int G = PAGED ? 1 : int(gridDim.x);
  const int n_items = PAGED ? 1 : n_hp * n_qblk;
  auto item_of_round = [&](int rr) {
    return rr * G + ((rr & 1) ? G - 1 - int(blockIdx.x) : int(blockIdx.x));
  };
  Work pw{};
  if constexpr (PAGED) {
    const int tile = int(blockIdx.y);
    if (tile >= pa.tile_off[pa.B]) return;  // surplus CTA of the fixed grid
    int lo = 0, hi = pa.B - 1;              // last row whose first tile <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pa.tile_off[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    pw.hq0 = int(blockIdx.x) * NQ;
    pw.kvh = pw.hq0 / (h / h_kv);
    pw.pb = lo;
    pw.qb = pa.tile_off[lo + 1] - 1 - tile;  // longest tile of the row first
    pw.q_tok0 = pa.cu_q[lo];
    pw.q_len = pa.cu_q[lo + 1] - pw.q_tok0;
    int ctx = pa.seq_lens[lo];
    if (ctx < pw.q_len || ctx > pa.max_blocks * 16) {
      if (threadIdx.x == 0) atomicOr(&g_prefill_err, ATTN_DEVERR_BAD_SEQ_LEN);
      ctx = ctx < pw.q_len ? pw.q_len : pa.max_blocks * 16;
    }
    pw.ctx = ctx;
    pw.n_pages = (ctx + 15) / 16;
    const int q_hi = min(pw.qb * kBM + kBM, pw.q_len);  // end of this tile's queries
    const int key_end = causal ? ctx - pw.q_len + q_hi : ctx;
    pw.nkv = (key_end + kBN - 1) / kBN;
    pw.n_kv_all = pw.nkv;
  }
  auto work_at = [&](int i) -> Work {
    if constexpr (PAGED) {
      return pw;
    } else {
      Work w{};
      const int hp = i % n_hp;
      const int rank = i / n_hp;
      w.hq0 = hp * NQ;
      w.kvh = w.hq0 / (h / h_kv);
      w.qb = causal ? (n_qblk - 1 - rank) : rank;
      w.n_kv_all = (T + kBN - 1) / kBN;
      w.nkv = causal ? min(w.qb + 1, w.n_kv_all) : w.n_kv_all;
      return w;
    }
  };
  // Per key tile of a KV head: nonzero -> V stays bf16 (exact P_hi + P_lo
  // product); zero -> V is read from its fp16 copy (fp16 P). No flags: all
  // tiles bf16. Paged rows: flags [B, h_kv, max_tiles].
  auto wide_flags = [&](const Work& w) -> const int* {
    return !vwide ? nullptr
                  : vwide + (PAGED ? (size_t(w.pb) * h_kv + w.kvh) * pa.max_tiles
                                   : size_t(w.kvh) * w.n_kv_all);
  };
  auto is_wide = [&](const int* tile_wide, int j) {
    return tile_wide ? (__ldg(tile_wide + j) != 0) : true;
  };
  // The flags of key tiles j0 .. j0 + 31 (below n) as one bit each, for a
  // whole warp: one load per lane every 32 tiles instead of a load on every
  // tile's path to its MMAs and exponentials. Warp-collective.
  auto wide_bits = [&](const int* tile_wide, int j0, int n) -> uint32_t {
    if (!tile_wide) return 0xffffffffu;
    const int jj = j0 + (threadIdx.x & 31);
    return __ballot_sync(0xffffffffu, jj < n && __ldg(tile_wide + jj) != 0);
  };
  // Whether any of key tiles 0 .. n-1 is wide. Warp-collective.
  auto item_has_wide = [&](const int* tile_wide, int n) -> bool {
    uint32_t any = 0;
    for (int j0 = 0; j0 < n; j0 += 32) any |= wide_bits(tile_wide, j0, n);
    return any != 0;
  };

  // The tensor maps' descriptors are fetched while the CTA sets up, not on
  // the first TMA issue (any thread may issue the prefetch).
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    if (vwide) prefetch_tmap(&tmap_v16);
  }
  if (warp == 0) {
    // One barrier per lane. p_full collects one arrival per softmax thread,
    // stage_free one per softmax warp; the others take one.
    if (lane < C::NBAR) {
      const uint32_t bar = bars.base + 8 * lane;
      const bool is_p = bar >= bars.p_full(0) && bar < bars.p_full(0) + 8 * NQ;
      const bool is_stage = bar == bars.stage_free(0) || bar == bars.stage_free(1);
      mbar_init(bar, is_p ? 128u : is_stage ? uint32_t(NQ * 4) : 1u);
      fence_barrier_init();
    }
    if (lane == 0) {
      *abort_flag = 0;
      if constexpr (PAGED && !PCOPY) {
        tail_info[0] = pw.ctx % 16 != 0 ? pw.ctx / kBN : -1;
        tail_info[1] = (pw.ctx % kBN) | ((16 - pw.ctx % 16) << 8);
      }
    }
  }
  if (warp == C::MMA_WARP) tc::alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  // Item it of this CTA as the producer published it: -1 when none is left,
  // -2 on an abort. Warp-uniform (the wait's outcome is).
  auto next_item = [&](int it) -> int {
    if constexpr (PAGED) {
      return it == 0 ? 0 : -1;
    } else {
      if (!__all_sync(0xffffffffu,
                      wait_or_abort(bars.item_full(it & 1), (it >> 1) & 1, abort_flag)))
        return -2;
      return __shfl_sync(0xffffffffu, item_slot[it & 1], 0);
    }
  };

  // Register shares move per warpgroup: every warp of a warpgroup executes
  // the same setmaxnreg, at the top of its role's code.
  if (warp >= C::PRODUCER_WARP) {
  if constexpr (NQ == 2) regs_dec<C::REG_CONTROL>();
  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Loads issued so far (K and V tiles counted over all of this CTA's
      // items: tile g uses stage g % NS, phase (g / NS) & 1).
      int k_issued = 0, v_issued = 0, q_issued = 0;
      // An item's epilogue stages O in the V stages of its last two tiles;
      // the load of V tile (its last tile + 2) is the first to reuse one, so
      // it waits for that item's stage_free. stage_waited items have been
      // waited for; the last tiles of the (at most two) others are kept.
      int stage_waited = 0, gl_even = 0, gl_odd = 0;
#ifdef ATTN_DEBUG
      const int stall = g_prefill_stall_tile;
#else
      constexpr int stall = -1;
#endif
      int g0 = 0, it = 0, rr = 0;
      bool ok = true;
      int cur = PAGED ? 0 : int(blockIdx.x);  // this item (grid size <= n_items)
      for (;; ++it) {
        if constexpr (!PAGED) {
          // Q of the next item once the last S MMA of the previous one is
          // done; that S also follows every role's read of item slot
          // (it & 1) for item it - 2, so the slot can take item it.
          if (it > 0 && !wait_or_abort(bars.q_empty(), (it - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          item_slot[it & 1] = cur;
          mbar_arrive(bars.item_full(it & 1));
        }
        if (cur < 0) break;
        const Work w = work_at(cur);
        const int* tile_wide = wide_flags(w);
        mbar_arrive_expect_tx(bars.q_full(), NQ * C::QTILE);
        for (int t = 0; t < NQ; ++t)
          for (int s = 0; s < C::SUBS; ++s) {
            if constexpr (PAGED)
              tma_load_3d(sbase + C::Q_OFF + t * C::QTILE + s * C::SUB_BYTES, &tmap_q,
                          bars.q_full(), s * 64, w.hq0 + t, w.q_tok0 + w.qb * kBM);
            else
              tma_load_3d(sbase + C::Q_OFF + t * C::QTILE + s * C::SUB_BYTES, &tmap_q,
                          bars.q_full(), s * 64, w.qb * kBM, w.hq0 + t);
          }
        q_issued = it + 1;
        // Paged rows: the 8 pages of key tile j (a page past the row's end, or
        // an invalid entry, is read at coordinate -1 and arrives as zeros).
        int pg[8];
        auto fetch_pages = [&](int j) {
          if constexpr (PAGED) {
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              const int page = j * 8 + p;
              int phys = -1;
              if (page < w.n_pages) {
                phys = pa.block_table[size_t(w.pb) * pa.max_blocks + page];
                if (phys < 0 || phys >= pa.num_blocks) {
                  atomicOr(&g_prefill_err, ATTN_DEVERR_BAD_PAGE);
                  phys = -1;
                }
              }
              pg[p] = phys;
            }
          }
        };
        auto load_tile = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar, int j) {
          if constexpr (PAGED) {
#pragma unroll
            for (int s = 0; s < C::SUBS; ++s)
#pragma unroll
              for (int p = 0; p < 8; ++p)
                tma_load_4d(dst + s * C::SUB_BYTES + p * 16 * 128, map, bar, s * 64, w.kvh, 0,
                            pg[p]);
          } else {
            for (int s = 0; s < C::SUBS; ++s)
              tma_load_3d(dst + s * C::SUB_BYTES, map, bar, s * 64, j * kBN, w.kvh);
          }
        };
        // K and V have rings of their own: a K stage frees as soon as the last
        // head's S MMA on it completes, a V stage after the last P V MMA.
        for (int j = 0; j < w.nkv; ++j) {
          const int g = g0 + j;
          const int sk = g % NSK, sv = g % NSV;
          fetch_pages(j);
          if (g >= NSK && !wait_or_abort(bars.k_empty(sk), ((g / NSK) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          if (g != stall) {  // (the abort-path self-test requests nothing for one tile)
            mbar_arrive_expect_tx(bars.k_full(sk), C::KTILE);
            load_tile(sbase + C::K_OFF + sk * C::KTILE, &tmap_k, bars.k_full(sk), j);
          }
          k_issued = g + 1;
          if (g >= NSV && !wait_or_abort(bars.v_empty(sv), ((g / NSV) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          while (!PAGED && ok && stage_waited < it &&
                 ((stage_waited & 1) ? gl_odd : gl_even) + 2 <= g) {
            ok = wait_or_abort(bars.stage_free(stage_waited & 1), (stage_waited >> 1) & 1,
                               abort_flag);
            ++stage_waited;
          }
          if (!ok) break;
          // Q and K are older than the V pass, so they load before this wait;
          // the fp16 V copy and the tile flags are the V pass's output.
          if (g == 0) pdl_wait();
          mbar_arrive_expect_tx(bars.v_full(sv), C::KTILE);
          if (PAGED && PCOPY) {
            // The row's copy is token-contiguous: one 128-token box per
            // 64-element column block instead of one box per page. It holds
            // fp16 bits, or bf16 bits for a flagged tile (a byte copy: the map's
            // fp16 type only sets the element size).
            const int tok = w.pb * pa.max_tiles * kBN + j * kBN;
            for (int s = 0; s < C::SUBS; ++s)
              tma_load_3d(sbase + C::V_OFF + sv * C::KTILE + s * C::SUB_BYTES, &tmap_v16,
                          bars.v_full(sv), s * 64, w.kvh, tok);
          } else {
            load_tile(sbase + C::V_OFF + sv * C::KTILE,
                      is_wide(tile_wide, j) ? &tmap_v : &tmap_v16, bars.v_full(sv), j);
          }
          v_issued = g + 1;
        }
        if (!ok) break;
        if (it & 1) gl_odd = g0 + w.nkv - 1; else gl_even = g0 + w.nkv - 1;
        g0 += w.nkv;
        // The next item, claimed as this one's loads are all issued (a few
        // key tiles before it ends); its Q and first K tile go to L2 now, so
        // that its Q load, issued once this item's last S MMA is done, is
        // served from there.
        if constexpr (PAGED) {
          cur = -1;
        } else {
          int nxt;
          if (sched != nullptr) {
            nxt = G + atomicAdd(sched, 1);
          } else {
            ++rr;
            nxt = rr * G < n_items ? item_of_round(rr) : n_items;
          }
          cur = nxt < n_items ? nxt : -1;
          if (cur >= 0) {
            const Work wn = work_at(cur);
            for (int t = 0; t < NQ; ++t)
              for (int s = 0; s < C::SUBS; ++s)
                tma_prefetch_l2_3d(&tmap_q, s * 64, wn.qb * kBM, wn.hq0 + t);
            for (int s = 0; s < C::SUBS; ++s) tma_prefetch_l2_3d(&tmap_k, s * 64, 0, wn.kvh);
          }
        }
      }
      if (*abort_flag) {
        // Drain: the newest load of each stage is the only one that can still
        // be in flight. Bounded waits, error already recorded.
        if (q_issued > 0) (void)mbar_wait(bars.q_full(), (q_issued - 1) & 1, &g_prefill_err);
        for (int g = max(0, k_issued - NSK); g < k_issued; ++g)
          if (g != stall) (void)mbar_wait(bars.k_full(g % NSK), (g / NSK) & 1, &g_prefill_err);
        for (int g = max(0, v_issued - NSV); g < v_issued; ++g)
          (void)mbar_wait(bars.v_full(g % NSV), (g / NSV) & 1, &g_prefill_err);
      }
    }
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (operands warp-uniform); elect.sync picks
    // the lane that issues each MMA / commit. Wait outcomes are made
    // warp-uniform before any warp-collective instruction.
    {
      constexpr uint32_t idS = tc::idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idO = tc::idesc_bf16_f32(kBM, D, false, true);
      // Base descriptors once; per MMA only the start-address field (address
      // >> 4, 14 bits) advances. Shared addresses stay below 256 KB, so the
      // field never carries into its neighbour.
      const uint64_t dq0 = tc::sw128_desc(sbase + C::Q_OFF, 16, 1024);
      const uint64_t dk0 = tc::sw128_desc(sbase + C::K_OFF, 16, 1024);
      const uint64_t dv0 = tc::sw128_desc(sbase + C::V_OFF, C::SUB_BYTES, 1024);
      auto issue_s = [&](int t, int st) {
        const uint64_t da = dq0 + uint64_t((t * C::QTILE) >> 4);
        const uint64_t db = dk0 + uint64_t((st * C::KTILE) >> 4);
        const uint32_t dS = tmem + t * 256;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off16 = ((kk >> 2) * C::SUB_BYTES + (kk & 3) * 32) >> 4;
          tc::mma_ss_elect(dS, da + off16, db + off16, idS, kk > 0 ? 1u : 0u);
        }
      };
      constexpr uint32_t idO16 = tc::idesc_f16_f32(kBM, D, false, true);
      // O_t += P V. Normal tiles: P fp16 (S columns 0-63) times the fp16 copy
      // of V. Wide tiles (some |v| >= 2^16, kept bf16): O_t += P_hi V + P_lo V
      // with P_hi in columns 0-63, P_lo in columns 64-127.
      auto issue_pv = [&](int t, int st, bool acc, bool wide) {
        const uint64_t dvb = dv0 + uint64_t((st * C::KTILE) >> 4);
        const uint32_t dO = tmem + t * 256 + 128;
        const uint32_t aP = tmem + t * 256;
        if (!wide) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint64_t b = dvb + uint64_t((kk * 16 * 128) >> 4);
            tc::mma_ts_elect(dO, aP + kk * 8, b, idO16, (acc || kk > 0) ? 1u : 0u);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint64_t b = dvb + uint64_t((kk * 16 * 128) >> 4);
            tc::mma_ts_elect(dO, aP + kk * 8, b, idO, (acc || kk > 0) ? 1u : 0u);
            tc::mma_ts_elect(dO, aP + 64 + kk * 8, b, idO, 1u);
          }
        }
      };
      auto wait = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag));
      };
      // Order per key tile j: P_0 V_j, S_0(j+1), P_1 V_j, S_1(j+1): each head's
      // next QK^T follows its own P V (P aliases S in tensor memory), and the
      // other head's softmax runs while these MMAs execute. An item's first S
      // MMAs follow the previous item's last P V, so they run while its
      // softmax warps store O; its first P V waits for their first P, which
      // they write after reading O out.
      bool ok = true;
      int g0 = 0;
      for (int it = 0; ok; ++it) {
        const int item = next_item(it);
        if (item < 0) break;
        const Work w = work_at(item);
        const int* tile_wide = wide_flags(w);
        ok = wait(bars.q_full(), it & 1) && wait(bars.k_full(g0 % NSK), (g0 / NSK) & 1);
        if (!ok) break;
        tc::fence_after();
        for (int t = 0; t < NQ; ++t) {
          issue_s(t, g0 % NSK);
          tc::commit_elect(bars.s_full(t));
        }
        tc::commit_elect(bars.k_empty(g0 % NSK));
        if (w.nkv == 1) tc::commit_elect(bars.q_empty());
        if (it == 0) pdl_wait();  // the tile flags below are the V pass's output
        // The loop is instantiated twice: for items without a wide tile (the
        // common case) it has no per-tile format branch at all.
        auto tiles = [&](auto any_wide) {
        constexpr bool MAYBE_WIDE = decltype(any_wide)::value;
        uint32_t wbits = 0;
        for (int j = 0; ok && j < w.nkv; ++j) {
          const int g = g0 + j;
          const int sv = g % NSV;
          const int sk1 = (g + 1) % NSK;
          bool wide = false;
          if constexpr (MAYBE_WIDE) {
            if ((j & 31) == 0) wbits = wide_bits(tile_wide, j, w.nkv);
            wide = (wbits >> (j & 31)) & 1u;
          }
          for (int t = 0; t < NQ && ok; ++t) {
            if (!wait(bars.p_full(t), g & 1)) { ok = false; break; }
            if (t == 0 && !wait(bars.v_full(sv), (g / NSV) & 1)) { ok = false; break; }
            tc::fence_after();
            issue_pv(t, sv, j > 0, wide);
            if (j == w.nkv - 1) tc::commit_elect(bars.o_final(t));
            if (t == NQ - 1) tc::commit_elect(bars.v_empty(sv));
            if (j + 1 < w.nkv) {
              if (t == 0 && !wait(bars.k_full(sk1), ((g + 1) / NSK) & 1)) { ok = false; break; }
              tc::fence_after();
              issue_s(t, sk1);
              tc::commit_elect(bars.s_full(t));
              if (t == NQ - 1) {
                tc::commit_elect(bars.k_empty(sk1));
                if (j + 2 == w.nkv) tc::commit_elect(bars.q_empty());  // Q's last reader
              }
            }
          }
        }
        };
        if (item_has_wide(tile_wide, w.nkv)) tiles(std::true_type{}); else tiles(std::false_type{});
        g0 += w.nkv;
      }
      // Everything issued has completed once mma_done flips.
      tc::commit_elect(bars.mma_done());
      (void)__all_sync(0xffffffffu, mbar_wait(bars.mma_done(), 0, &g_prefill_err));
    }
  }
  } else {
    // ------------------------------------------------------------ softmax
    if constexpr (NQ == 2) regs_inc<C::REG_SOFTMAX>();
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t tS = tmem + (uint32_t(wq * 32) << 16) + t * 256;
    const uint32_t tO = tS + 128;
    bool ok = true;
    int g0 = 0;
    pdl_wait();  // the tile flags are the V pass's output
    for (int it = 0; ok; ++it) {
    const int item = next_item(it);
    if (item < 0) break;
    const Work w = work_at(item);
    ATTN_DCHECK(w.hq0 + NQ <= h && w.kvh < h_kv && w.nkv >= 1 &&
                    w.nkv <= (PAGED ? pa.max_tiles : w.n_kv_all) &&
                    (PAGED || w.qb < n_qblk),
                &g_prefill_err);
    const int* tile_wide = wide_flags(w);
    const int row = w.qb * kBM + r;  // query index within the row (paged) or the sequence
    const int hq = w.hq0 + t;
    // Paged rows: keys [0, key_end) are visible to this query (none for the
    // padding rows of a row's last tile).
    const bool row_valid = PAGED ? row < w.q_len : row < T;
    const int key_end =
        !PAGED ? 0 : (!row_valid ? 0 : (causal ? w.ctx - w.q_len + row + 1 : w.ctx));
    // m_ref: exp2-domain reference that l, O~ and this tile's P are relative
    // to (the row max of some tile seen so far, within 2^15 of the running
    // max).
    float m_ref = -INFINITY;
    float l = 0.f;
    // Instantiated twice, as the MMA warp's loop: without a wide tile in the
    // item, no tile takes the format branch.
    auto tiles = [&](auto any_wide) {
    constexpr bool MAYBE_WIDE = decltype(any_wide)::value;
    uint32_t wbits = 0;
    for (int j = 0; j < w.nkv; ++j) {
      const int g = g0 + j;
      // The format of P follows the format of this key tile's V.
      bool wide = false;
      if constexpr (MAYBE_WIDE) {
        if ((j & 31) == 0) wbits = wide_bits(tile_wide, j, w.nkv);
        wide = (wbits >> (j & 31)) & 1u;
      }
      // Warp-uniform outcome: the tensor-memory loads below are warp-collective.
      if (!__all_sync(0xffffffffu, wait_or_abort(bars.s_full(t), g & 1, abort_flag))) {
        ok = false;
        break;
      }
      if constexpr (PAGED && !PCOPY) {
        if (t == 0 && j == tail_info[0]) {
          // Slots of the row's last page past its last key hold whatever the
          // cache holds (possibly NaN or inf). Their weights are 0, but 0 * NaN
          // is NaN in the P V product, so they are zeroed in the V tile before
          // this head's arrival lets the MMA warp issue the tile's P V (the
          // workspace copy, when there is one, has them zeroed already). The tile's V phase cannot
          // move on before that P V, so the wait sees this tile's copy. Done
          // before the S tile is loaded, while few registers are live.
          const int sv = g % NSV;
          if (wait_or_abort(bars.v_full(sv), (g / NSV) & 1, abort_flag)) {
            // Thread r clears 16-byte chunk r % 8 of slot r / 8 past the last
            // key, in every 64-column block (16 slots x 8 chunks = 128 threads).
            if ((r >> 3) < (tail_info[1] >> 8)) {
              const uint32_t a = sbase + C::V_OFF + sv * C::KTILE +
                                 ((tail_info[1] & 0xff) + (r >> 3)) * 128 + (r & 7) * 16;
#pragma unroll
              for (int sub = 0; sub < C::SUBS; ++sub)
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a + sub * C::SUB_BYTES),
                             "r"(0u)
                             : "memory");
            }
            fence_proxy_async_smem();  // the MMA reads V through the async proxy
          }
        }
      }
      tc::fence_after();
      int lim = kBN;
      if constexpr (PAGED) {
        lim = min(kBN, key_end - j * kBN);
      } else {
        if (j * kBN + kBN > T) lim = T - j * kBN;
        if (causal && j == w.qb) lim = min(lim, r + 1);
      }
      const uint64_t c2 = f2(scale_log2, scale_log2);
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::ld32(tS + c * 32, sr[c]);
      tc::wait_ld();
      if (lim < kBN) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c * 32 + i >= lim) sr[c][i] = __float_as_uint(-INFINITY);
      }
      // Row max: per 32-column chunk a tree of 3-input maxima (11 -> 4 -> 1),
      // then the four chunk maxima. Then the lazy reference rule: the
      // reference moves (to kRefHeadroom above the row max) only when the row
      // max exceeds it by more than kRescaleBits, so every weight stays at
      // most 2^15 and fits fp16; otherwise l and O~ keep their scale.
      float cm[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        auto x = [&](int i) { return __uint_as_float(sr[c][i]); };
        float a[11];
#pragma unroll
        for (int i = 0; i < 10; ++i) a[i] = max3f(x(3 * i), x(3 * i + 1), x(3 * i + 2));
        a[10] = fmaxf(x(30), x(31));
        cm[c] = fmaxf(max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), max3f(a[6], a[7], a[8])),
                      fmaxf(a[9], a[10]));
      }
      const float mx = fmaxf(max3f(cm[0], cm[1], cm[2]), cm[3]);
      const float m_cand = mx * scale_log2;
      float alpha = 1.f;
      if (m_cand > m_ref + kRescaleBits) {
        const float m_new = m_cand + kRefHeadroom;
        alpha = ex2_approx(m_ref - m_new);  // 0 on the first tile
        l *= alpha;
        m_ref = m_new;
      }
      // O~ holds the P V of tiles < j (complete: this tile's S was issued
      // after them) and is scaled by alpha before this tile's P V adds to it.
      // That happens after P is stored, in the registers S occupied, so that
      // the exponent loop carries no extra live state for it.
      const bool rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
      const float bias = (m_ref == -INFINITY) ? 0.f : m_ref;
      const uint64_t nb2 = f2(-bias, -bias);
      float psum;  // row sum of this tile's weights
      if (!wide) {
        uint64_t sumA = f2(0.f, 0.f), sumB = f2(0.f, 0.f);
        // P in fp16 (11 significant bits). Key pair (2i, 2i+1) of chunk c
        // goes to P column 16c + i, i.e. the first 64 columns of the S tile
        // just read; sr[c][i] is reused to stage that pair (its S values
        // were consumed at step i/2).
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float y0, y1;
            unf2(fma2(f2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), c2,
                      nb2),
                 y0, y1);
            const float p0 = ex2_approx(y0);
            const float p1 = ex2_approx(y1);
            if (i & 1) sumB = add2(sumB, f2(p0, p1)); else sumA = add2(sumA, f2(p0, p1));
            sr[c][i] = pack_f16x2(p0, p1);
          }
        }
        uint32_t pw[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int i = 0; i < 16; ++i) pw[16 * c + i] = sr[2 * half + c][i];
          tc::st32(tS + 32 * half, pw);  // P keys 64*half .. +63
        }
        float sa0, sa1;
        unf2(add2(sumA, sumB), sa0, sa1);
        psum = sa0 + sa1;
      } else {
        psum = softmax_p_two_term(tS, lim, scale_log2, bias);
      }
      if (rescale) {
        // sr is free once P is stored (tcgen05.st reads its registers at
        // issue): all of O~ at once, one load latency.
        const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tc::ld32(tO + c * 32, sr[c]);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            unf2(mul2(f2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), a2),
                 x0, x1);
            sr[c][2 * i] = __float_as_uint(x0);
            sr[c][2 * i + 1] = __float_as_uint(x1);
          }
          tc::st32(tO + c * 32, sr[c]);
        }
      }
      l += psum;
      tc::wait_st();
      tc::fence_before();
      mbar_arrive(bars.p_full(t));
    }
    };
    if (item_has_wide(tile_wide, w.nkv)) tiles(std::true_type{}); else tiles(std::false_type{});
    if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(bars.o_final(t), it & 1, abort_flag));
    if (!ok) break;
    {
      tc::fence_after();
      // A row with no allowed key has l = 0 exactly (every weight is ex2 of
      // -inf). A NaN l (a NaN logit, or 0 * inf) is not empty: it reaches O
      // and the LSE.
      const bool empty = l == 0.f;
      const float inv = empty ? 0.f : 1.f / l;
      const size_t orow_idx = PAGED ? size_t(w.q_tok0 + row) * h + hq : size_t(hq) * T + row;
      // Output rows (debug checks): h * T, or h per packed query token.
      auto out_rows = [&]() -> size_t {
        return PAGED ? size_t(pa.cu_q[pa.B]) * h : size_t(h) * T;
      };
      (void)out_rows;
      // O leaves through this warp's quarter of a V stage: head 0 uses the
      // stage of the item's second-to-last key tile, head 1 that of the last
      // (every P V MMA on the first completed before head 0's o_final, on the
      // second before head 1's; the producer's next load into either waits
      // for stage_free). Q stays untouched, so the next item's Q can load
      // meanwhile. Paged rows (one item per CTA) use the head's Q tile, whose
      // last reader, the head's last S MMA, completed before o_final. Each
      // thread writes its row there in 16-byte chunks, chunk index XOR (row
      // mod 8) so the 8 rows of a store phase hit distinct banks; then the
      // warp stores whole rows, 256 (d_h = 128) or 128 contiguous bytes per
      // row, instead of 32 rows x 16 bytes per instruction.
      constexpr int RB = D * 2;    // bytes per O row
      constexpr int CH = RB / 16;  // 16-byte chunks per row
      constexpr int RPI = 32 / CH; // rows per warp store instruction
      const int gl = g0 + w.nkv - 1;
      // With one key tile, head 0's stage (that of tile gl - 1) is the one
      // head 1 of the previous item staged in; it may still be reading it.
      if (!PAGED && t == 0 && w.nkv == 1 && it > 0 &&
          !__all_sync(0xffffffffu,
                      wait_or_abort(bars.stage_free((it - 1) & 1), ((it - 1) >> 1) & 1, abort_flag)))
        break;
      uint8_t* stage =
          PAGED ? smem + C::Q_OFF + t * C::QTILE + wq * (32 * RB)
                : smem + C::V_OFF + ((t == 0 ? gl - 1 + NSV : gl) % NSV) * C::KTILE + wq * (32 * RB);
      ATTN_DCHECK(stage >= smem + (PAGED ? C::Q_OFF : C::V_OFF) &&
                      stage + 32 * RB <= smem + (PAGED ? C::K_OFF : C::BAR_OFF),
                  &g_prefill_err);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tc::ld32(tO + c * 32, ov);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 pk;
          pk.x = pack_bf16x2(__uint_as_float(ov[8 * i + 0]) * inv, __uint_as_float(ov[8 * i + 1]) * inv);
          pk.y = pack_bf16x2(__uint_as_float(ov[8 * i + 2]) * inv, __uint_as_float(ov[8 * i + 3]) * inv);
          pk.z = pack_bf16x2(__uint_as_float(ov[8 * i + 4]) * inv, __uint_as_float(ov[8 * i + 5]) * inv);
          pk.w = pack_bf16x2(__uint_as_float(ov[8 * i + 6]) * inv, __uint_as_float(ov[8 * i + 7]) * inv);
          const int ch = c * 4 + i;
          *reinterpret_cast<uint4*>(stage + lane * RB + ((ch ^ (lane & 7)) << 4)) = pk;
        }
      }
      __syncwarp();
      {
        const int ch = lane % CH;
#pragma unroll
        for (int it = 0; it < 32 / RPI; ++it) {
          const int rr = it * RPI + lane / CH;  // row within this warp's 32
          const int qrow = w.qb * kBM + wq * 32 + rr;
          if (PAGED ? qrow < w.q_len : qrow < T) {
            const uint4 x =
                *reinterpret_cast<const uint4*>(stage + rr * RB + ((ch ^ (rr & 7)) << 4));
            const size_t oi = PAGED ? size_t(w.q_tok0 + qrow) * h + hq : size_t(hq) * T + qrow;
            if (ATTN_GUARD(oi < out_rows(), &g_prefill_err))
              *reinterpret_cast<uint4*>(o + oi * D + ch * 8) = x;
          }
        }
      }
      if (row_valid && lse != nullptr && ATTN_GUARD(orow_idx < out_rows(), &g_prefill_err))
        lse[orow_idx] = empty ? -INFINITY : (m_ref + log2f(l)) * kLn2;
      // The warp's rows have left the stage (each lane's loads completed
      // before its stores issued); the fence orders these generic accesses
      // before the producer's next TMA write there.
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.stage_free(it & 1));
    }
    g0 += w.nkv;
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == C::MMA_WARP) tc::dealloc(tmem, C::TMEM_COLS);
}

// V (bf16 [h_kv, T, d_h]) -> fp16 copy with the same layout, and one flag per
// (KV head, 128-key tile): 1 when the tile holds a value with |v| >= 2^16
// (or inf / NaN), which fp16 cannot carry; such tiles are read from the bf16
// original by the attention kernel. bf16 -> fp16 is exact for
// 2^-14 <= |v| < 2^16 (8 significant bits fit in 11); smaller values round
// with an absolute error below 2^-25. One CTA per tile, 16-byte accesses.
__global__ void __launch_bounds__(256)
    v_to_f16_kernel(const uint4* __restrict__ v, uint4* __restrict__ v16, int* __restrict__ vwide,
                    int* __restrict__ sched, int T, int chunks_per_row, int n_tiles) {
  const int tile = blockIdx.x, kvh = blockIdx.y;
  // The attention kernel's item counter starts from zero for every call; it
  // reads the counter only after waiting for this grid.
  if (sched != nullptr && tile == 0 && kvh == 0 && threadIdx.x == 0) *sched = 0;
  // The attention kernel (a programmatic dependent) may start its CTAs'
  // set-up and Q, K loads now; it waits for this grid before touching V.
  pdl_trigger();
  const int rows = min(kBN, T - tile * kBN);
  const size_t base = (size_t(kvh) * T + size_t(tile) * kBN) * chunks_per_row;
  const int n = rows * chunks_per_row;
  uint32_t mx = 0;
  // All of a thread's loads (8 at d_h = 128) are in flight before the first
  // conversion: the pass is latency-bound at small T otherwise.
  constexpr int kU = 8;
  for (int i0 = threadIdx.x; i0 < n; i0 += kU * blockDim.x) {
    uint4 x[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < n) x[u] = v[base + i];
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < n) {
        uint32_t m2;
        asm("max.u16x2 %0, %1, %2;" : "=r"(m2) : "r"(x[u].x & 0x7fff7fffu), "r"(x[u].y & 0x7fff7fffu));
        asm("max.u16x2 %0, %0, %1;" : "+r"(m2) : "r"(x[u].z & 0x7fff7fffu));
        asm("max.u16x2 %0, %0, %1;" : "+r"(m2) : "r"(x[u].w & 0x7fff7fffu));
        asm("max.u16x2 %0, %0, %1;" : "+r"(mx) : "r"(m2));
        uint4 y;
        y.x = pack_f16x2(bf16lo(x[u].x), bf16hi(x[u].x));
        y.y = pack_f16x2(bf16lo(x[u].y), bf16hi(x[u].y));
        y.z = pack_f16x2(bf16lo(x[u].z), bf16hi(x[u].z));
        y.w = pack_f16x2(bf16lo(x[u].w), bf16hi(x[u].w));
        if (ATTN_GUARD(base + i < size_t(gridDim.y) * T * chunks_per_row, &g_prefill_err))
          v16[base + i] = y;
      }
    }
  }
  // bf16 bits 0x4780 = 2^16: the first magnitude fp16 cannot hold.
  const int wide = __syncthreads_or((mx & 0xffffu) >= 0x4780u || (mx >> 16) >= 0x4780u);
  if (threadIdx.x == 0 && ATTN_GUARD(tile < n_tiles && kvh < int(gridDim.y), &g_prefill_err))
    vwide[size_t(kvh) * n_tiles + tile] = wide;
}

// Paged V -> a copy of the keys each row uses, token-contiguous per row:
// [B, max_tiles * 128, h_kv, d_h] (row b's key t at token b * max_tiles * 128
// + t), and flags [B, h_kv, max_tiles] with v_to_f16_kernel's meaning. A tile
// is written as fp16 when every value converts exactly, else (flagged) as
// the bf16 values themselves, so the attention kernel reads every V tile of
// the row from this copy. Keys from the row's last key to the end of its last
// 128-key tile, and pages whose block-table entry lies outside the cache, are
// written as zeros, whatever the cache holds there. Rows the attention kernel
// skips (query count above the row's capacity) are left alone. The key count
// is clamped as the attention kernel clamps it. One CTA per (tile, row, KV
// head); each thread holds its CPR / 2 chunks of 16 bytes between the range
// check and the store.
template <int CPR>
__global__ void __launch_bounds__(256)
    paged_v_to_f16_kernel(const uint4* __restrict__ vc, const int32_t* __restrict__ block_table,
                          const int32_t* __restrict__ cu_q, const int32_t* __restrict__ seq_lens,
                          int max_blocks, int num_blocks, int h_kv, int max_tiles,
                          int skip_single, uint4* __restrict__ v16, int* __restrict__ vwide) {
  constexpr int PER = kBN * CPR / 256;  // chunks per thread
  const int jt = blockIdx.x, b = blockIdx.y, kvh = blockIdx.z;
  const int cap = max_blocks * 16;
  const int q_len = cu_q[b + 1] - cu_q[b];
  if (q_len < 0 || q_len > cap || (skip_single && q_len == 1)) return;
  int ctx = seq_lens[b];
  if (ctx < q_len || ctx > cap) ctx = ctx < q_len ? q_len : cap;
  const int n_pages = (ctx + 15) / 16;
  if (jt * 8 >= n_pages) return;
  uint4 x[PER];
  uint32_t mx = 0;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int i = threadIdx.x + 256 * u;
    const int tok = i / CPR, c = i % CPR;
    const int page = jt * 8 + (tok >> 4), slot = tok & 15;
    int phys = -1;
    if (jt * kBN + tok < ctx) {
      phys = __ldg(block_table + size_t(b) * max_blocks + page);
      if (phys >= num_blocks) phys = -1;
    }
    x[u] = make_uint4(0u, 0u, 0u, 0u);
    if (phys >= 0) x[u] = vc[((size_t(phys) * 16 + slot) * h_kv + kvh) * CPR + c];
    uint32_t m2;
    asm("max.u16x2 %0, %1, %2;" : "=r"(m2) : "r"(x[u].x & 0x7fff7fffu), "r"(x[u].y & 0x7fff7fffu));
    asm("max.u16x2 %0, %0, %1;" : "+r"(m2) : "r"(x[u].z & 0x7fff7fffu));
    asm("max.u16x2 %0, %0, %1;" : "+r"(m2) : "r"(x[u].w & 0x7fff7fffu));
    asm("max.u16x2 %0, %0, %1;" : "+r"(mx) : "r"(m2));
  }
  // bf16 bits 0x4780 = 2^16: the first magnitude fp16 cannot hold.
  const int wide = __syncthreads_or((mx & 0xffffu) >= 0x4780u || (mx >> 16) >= 0x4780u);
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int i = threadIdx.x + 256 * u;
    const int tok = i / CPR, c = i % CPR;
    uint4 y = x[u];
    if (!wide) {
      y.x = pack_f16x2(bf16lo(x[u].x), bf16hi(x[u].x));
      y.y = pack_f16x2(bf16lo(x[u].y), bf16hi(x[u].y));
      y.z = pack_f16x2(bf16lo(x[u].z), bf16hi(x[u].z));
      y.w = pack_f16x2(bf16lo(x[u].w), bf16hi(x[u].w));
    }
    const size_t vi = ((size_t(b) * max_tiles * kBN + size_t(jt) * kBN + tok) * h_kv + kvh) * CPR + c;
    if (ATTN_GUARD(tok < kBN && vi < size_t(gridDim.y) * max_tiles * kBN * h_kv * CPR,
                   &g_prefill_err))
      v16[vi] = y;
  }
  if (threadIdx.x == 0 &&
      ATTN_GUARD(jt < max_tiles && b < int(gridDim.y) && kvh < h_kv, &g_prefill_err))
    vwide[(size_t(b) * h_kv + kvh) * max_tiles + jt] = wide;
}

template <int D, int NQ, int NSK, int NSV>
cudaError_t launch(const void* q, const void* k, const void* v, const void* v16, const int* vwide,
                   int* sched, void* o, float* lse, int T, int h, int h_kv, int causal,
                   float scale, cudaStream_t stream) {
  using C = PfCfg<D, NQ, NSK, NSV>;
  static_assert(C::SMEM <= 232448, "shared memory budget");
  CUtensorMap tq, tk, tv, tv16;
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
    // Without the fp16 copy the map is a duplicate of the bf16 one, never used.
    if (encode_tensor_map(&tv16, v16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          3, const_cast<void*>(v16 ? v16 : v), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kern = prefill_bf16_kernel<D, NQ, NSK, NSV, false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_qblk = (T + kBM - 1) / kBM;
  // Persistent grid: one CTA per SM (the shared memory admits one), each
  // walking its share of the (head group, query block) items.
  const long long n_items = static_cast<long long>(h / NQ) * n_qblk;
  if (n_items <= 0) return cudaSuccess;
  if (n_items > INT_MAX / 2) return cudaErrorNotSupported;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(n_items < sms ? n_items : sms));
  // After the V pass the kernel is its programmatic dependent (it waits for
  // that grid before reading V or the flags); without one it follows
  // whatever precedes it on the stream in plain order.
  if (v16)
    return launch_pdl(kern, grid, dim3(C::THREADS), C::SMEM, stream, tq, tk, tv, tv16, vwide,
                      static_cast<__nv_bfloat16*>(o), lse, T, h, h_kv, causal, scale * kLog2e,
                      n_qblk, sched, PagedArgs{});
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tv16, nullptr,
                                               static_cast<__nv_bfloat16*>(o), lse, T, h, h_kv,
                                               causal, scale * kLog2e, n_qblk, nullptr,
                                               PagedArgs{});
  return cudaGetLastError();
}

// Row b's query tiles: tile_off[b+1] = tile_off[b] + ceil(q_len_b / 128). A
// query count below 0 or above max_q_len (the grid's bound) is an error:
// that row gets no tiles and its outputs are not written. With skip_single,
// rows of one query get no tiles either (the split-KV decode takes them).
__global__ void paged_tiles_kernel(const int32_t* __restrict__ cu_q, int B, int max_q_len,
                                   int max_blocks, int skip_single, int32_t* __restrict__ tile_off) {
  if (threadIdx.x != 0) return;
  int acc = 0;
  tile_off[0] = 0;
  for (int b = 0; b < B; ++b) {
    int n = cu_q[b + 1] - cu_q[b];
    if (n < 0 || n > max_q_len || n > max_blocks * 16) {
      atomicOr(&g_prefill_err, ATTN_DEVERR_BAD_SEQ_LEN);
      n = 0;
    }
    if (skip_single && n == 1) n = 0;  // a decode row, handled by the split-KV decode
    acc += (n + kBM - 1) / kBM;
    tile_off[b + 1] = acc;
  }
}

template <int D, int NQ, int NSK, int NSV>
cudaError_t launch_paged(const PagedPrefill& a, cudaStream_t stream) {
  using C = PfCfg<D, NQ, NSK, NSV>;
  CUtensorMap tq, tk, tv;
  {
    // Q and O token-major [total_q, h, d_h]: a 128-token box of one head.
    const uint64_t dims[3] = {uint64_t(D), uint64_t(a.h), uint64_t(a.total_q)};
    const uint64_t strides[2] = {uint64_t(D) * 2, uint64_t(a.h) * D * 2};
    const uint32_t box[3] = {64u, 1u, 128u};
    if (encode_tensor_map(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // Cache [num_blocks, 16, h_kv, d_h]: one page of one KV head per box.
    const uint64_t dims[4] = {uint64_t(D), uint64_t(a.h_kv), 16u, uint64_t(a.num_blocks)};
    const uint64_t strides[3] = {uint64_t(D) * 2, uint64_t(a.h_kv) * D * 2,
                                 uint64_t(16) * a.h_kv * D * 2};
    const uint32_t box[4] = {64u, 1u, 16u, 1u};
    if (encode_tensor_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.k_cache),
                          dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (encode_tensor_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.v_cache),
                          dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int max_tiles = (a.max_blocks + 7) / 8;
  CUtensorMap tv16 = tv;
  if (a.v16 != nullptr) {
    // fp16 copy [B * max_tiles * 128 tokens, h_kv, d_h]: a 128-token box of one head.
    const uint64_t dims[3] = {uint64_t(D), uint64_t(a.h_kv),
                              uint64_t(a.B) * uint64_t(max_tiles) * kBN};
    const uint64_t strides[2] = {uint64_t(D) * 2, uint64_t(a.h_kv) * D * 2};
    const uint32_t box[3] = {64u, 1u, 128u};
    if (encode_tensor_map(&tv16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.v16, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    paged_v_to_f16_kernel<D / 8><<<dim3(max_tiles, a.B, a.h_kv), 256, 0, stream>>>(
        static_cast<const uint4*>(a.v_cache), a.block_table, a.cu_q, a.seq_lens, a.max_blocks,
        a.num_blocks, a.h_kv, max_tiles, a.decode_rows_apart, static_cast<uint4*>(a.v16), a.vwide);
    const cudaError_t e0 = cudaGetLastError();
    if (e0 != cudaSuccess) return e0;
  }
  paged_tiles_kernel<<<1, 32, 0, stream>>>(a.cu_q, a.B, a.max_q_len, a.max_blocks,
                                           a.decode_rows_apart, a.tile_off);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = a.v16 ? prefill_bf16_kernel<D, NQ, NSK, NSV, true, true>
                    : prefill_bf16_kernel<D, NQ, NSK, NSV, true, false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // At most one partial tile per row beyond ceil(total_q / 128), and no row
  // has more than ceil(max_q_len / 128) tiles.
  const long long by_total = (static_cast<long long>(a.total_q) + kBM - 1) / kBM + a.B;
  const long long by_row = static_cast<long long>(a.B) * ((a.max_q_len + kBM - 1) / kBM);
  const long long tiles = by_total < by_row ? by_total : by_row;
  if (tiles <= 0) return cudaSuccess;
  if (tiles > 65535) return cudaErrorNotSupported;  // query tiles index grid y
  const dim3 grid(a.h / NQ, static_cast<unsigned>(tiles));
  PagedArgs pa{a.block_table, a.cu_q,      a.seq_lens,   a.tile_off,
               a.B,           a.max_blocks, a.num_blocks, max_tiles};
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tv16, a.v16 ? a.vwide : nullptr,
                                               static_cast<__nv_bfloat16*>(a.o), a.lse, 0, a.h,
                                               a.h_kv, a.causal, a.scale * kLog2e, 0, nullptr,
                                               pa);
  return cudaGetLastError();
}

}  // namespace

PrefillLayout prefill_layout(int T, int h_kv, int d_h) {
  PrefillLayout L;
  L.v16_off = 0;
  L.flags_off = align256(size_t(h_kv) * T * d_h * 2);
  L.sched_off = L.flags_off + align256(size_t(h_kv) * ((T + kBN - 1) / kBN) * sizeof(int));
  L.total = L.sched_off + 256;  // the attention kernel's item counter
  return L;
}

cudaError_t launch_prefill_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                                int T, int h, int h_kv, int d_h, int causal, float scale,
                                void* workspace, cudaStream_t stream) {
  const int g = h / h_kv;
  const bool pair = (g % 2) == 0;
  void* v16 = nullptr;
  int* vwide = nullptr;
  int* sched = nullptr;
  if (workspace) {
    const PrefillLayout L = prefill_layout(T, h_kv, d_h);
    v16 = static_cast<uint8_t*>(workspace) + L.v16_off;
    vwide = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + L.flags_off);
    sched = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + L.sched_off);
    const int n_tiles = (T + kBN - 1) / kBN;
    v_to_f16_kernel<<<dim3(n_tiles, h_kv), 256, 0, stream>>>(
        static_cast<const uint4*>(v), static_cast<uint4*>(v16), vwide, sched, T, d_h / 8,
        n_tiles);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // Stage counts fill the shared memory next to the Q tiles (<= 227 KB).
  if (d_h == 128) {
    return pair ? launch<128, 2, 2, 3>(q, k, v, v16, vwide, sched, o, lse, T, h, h_kv, causal, scale, stream)
                : launch<128, 1, 3, 3>(q, k, v, v16, vwide, sched, o, lse, T, h, h_kv, causal, scale, stream);
  }
  return pair ? launch<64, 2, 4, 4>(q, k, v, v16, vwide, sched, o, lse, T, h, h_kv, causal, scale, stream)
              : launch<64, 1, 4, 4>(q, k, v, v16, vwide, sched, o, lse, T, h, h_kv, causal, scale, stream);
}

cudaError_t launch_prefill_paged(const PagedPrefill& a, cudaStream_t stream) {
  const bool pair = ((a.h / a.h_kv) % 2) == 0;
  if (a.d_h == 128)
    return pair ? launch_paged<128, 2, 2, 3>(a, stream) : launch_paged<128, 1, 3, 3>(a, stream);
  return pair ? launch_paged<64, 2, 4, 4>(a, stream) : launch_paged<64, 1, 4, 4>(a, stream);
}

cudaError_t prefill_set_stall(int key_tile) {
#ifdef ATTN_DEBUG
  return cudaMemcpyToSymbol(g_prefill_stall_tile, &key_tile, sizeof(key_tile));
#else
  (void)key_tile;
  return cudaErrorNotSupported;
#endif
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

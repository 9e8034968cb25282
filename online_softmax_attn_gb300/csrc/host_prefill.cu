// host_prefill.cu -- attn_prefill_host: the prefill of attn_prefill with Q, K
// and V read from host memory and O, LSE written back to host memory, in one
// call.
//
// The layer is cut into groups of KV heads, each with its query heads (heads
// are the outermost dimension, so a group is one contiguous slice of every
// tensor). Group c+1's inputs copy in while group c computes and group c-1's
// outputs copy out: the copies run on two copy streams (the caller's, or a
// pair the library creates on first use), the attention on the caller's
// stream, ordered by events (fork from and join back to the caller's stream,
// which CUDA graph capture follows). Each group
// is an independent prefill over its heads ("Naive attention and the online
// softmax": every query row's recurrence reads only its own head's Q and its
// KV head's K, V), so results are bitwise those of attn_prefill.
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

constexpr int kMaxChunks = 64;
constexpr int kMaxDevices = 64;

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The streams and events one call orders its work with. An event is re-recorded
// once the wait on its previous record has been enqueued: a stream wait binds
// to the record that precedes it, so five events serve any number of groups.
struct Pipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t ev[ATTN_HOST_PIPE_EVENTS] = {};
};
enum { kEvStart = 0, kEvIn = 1, kEvCmp = 2, kEvInDone = 3, kEvOutDone = 4 };

// Library-owned pipes, one per device, created on the first call that passes
// no pipe of its own, and kept for the life of the process. Each has its own
// lock, held while a call enqueues on it.
struct OwnedPipe {
  Pipe p;
  bool ready = false;
  std::mutex mu;
};
OwnedPipe g_pipes[kMaxDevices];

void destroy_pipe(Pipe& p) {
  for (cudaEvent_t& e : p.ev)
    if (e) (void)cudaEventDestroy(e), e = nullptr;
  if (p.in) (void)cudaStreamDestroy(p.in), p.in = nullptr;
  if (p.out) (void)cudaStreamDestroy(p.out), p.out = nullptr;
}

// Called with the device's lock held.
cudaError_t ensure_owned_pipe(OwnedPipe& op) {
  if (op.ready) return cudaSuccess;
  Pipe& p = op.p;
  cudaError_t e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
  for (int i = 0; e == cudaSuccess && i < ATTN_HOST_PIPE_EVENTS; ++i)
    e = cudaEventCreateWithFlags(&p.ev[i], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    destroy_pipe(p);
    return e;
  }
  op.ready = true;
  return cudaSuccess;
}

// Device scratch: q, k, v, o, lse copies, then the prefill workspace (fp16 V
// copy and tile flags), each region 256-byte aligned.
struct HostScratch {
  size_t q, k, v, o, lse, ws, total;
};
HostScratch host_scratch(int T, int h, int h_kv, int d_h, size_t elem, size_t ws_bytes) {
  HostScratch L;
  const size_t qn = size_t(h) * T * d_h * elem, kn = size_t(h_kv) * T * d_h * elem;
  L.q = 0;
  L.k = L.q + align256(qn);
  L.v = L.k + align256(kn);
  L.o = L.v + align256(kn);
  L.lse = L.o + align256(qn);
  L.ws = L.lse + align256(size_t(h) * T * sizeof(float));
  L.total = L.ws + ws_bytes;
  return L;
}

// KV heads per group. n_chunks > 0: equal groups. n_chunks == 0 and
// h_kv >= 4: four groups in the proportions 3 : 2 : 2 : 1 (a large first
// group computes while the rest copies in; the small last group keeps short
// the compute and copy-out that nothing overlaps). Measured with 8 KV heads
// (T = 8192): 3,2,2,1 ran 0.75 ms against 0.79 for four equal groups, 0.77
// for 1,2,2,2,1 and 0.80 for 1,3,3,1. With h_kv < 4: 2 equal groups when
// h_kv is even, else 1. Returns the group count.
int chunk_plan(int h_kv, int n_chunks, int* sizes) {
  if (n_chunks == 0 && h_kv >= 4) {
    const int w[4] = {3, 2, 2, 1};
    int rest = 0;
    for (int i = 1; i < 4; ++i) {
      sizes[i] = (h_kv * w[i] + 4) / 8 > 1 ? (h_kv * w[i] + 4) / 8 : 1;
      rest += sizes[i];
    }
    sizes[0] = h_kv - rest;  // >= 1 for h_kv >= 4
    return 4;
  }
  int c = n_chunks;
  if (c == 0) c = (h_kv % 2 == 0) ? 2 : 1;
  for (int i = 0; i < c; ++i) sizes[i] = h_kv / c;
  return c;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

size_t attn_prefill_host_scratch_bytes(int T, int h, int h_kv, int d_h, attn_dtype_t dtype) {
  if (T < 0 || h < 1 || h_kv < 1 || h % h_kv != 0 || (d_h != 64 && d_h != 128))
    return static_cast<size_t>(-1);
  if (dtype != ATTN_DTYPE_F32 && dtype != ATTN_DTYPE_BF16) return static_cast<size_t>(-1);
  if (T == 0) return 0;
  const size_t elem = dtype == ATTN_DTYPE_F32 ? 4 : 2;
  const size_t ws = dtype == ATTN_DTYPE_BF16 ? prefill_layout(T, h_kv, d_h).total : 0;
  return host_scratch(T, h, h_kv, d_h, elem, ws).total;
}

attn_status_t attn_prefill_host(const void* q, const void* k, const void* v, void* o, float* lse,
                                int T, int h, int h_kv, int d_h, int causal, float scale,
                                attn_dtype_t dtype, int n_chunks, void* scratch,
                                size_t scratch_bytes, const attn_host_pipe_t* pipe,
                                void* stream) {
  if (T < 0 || h < 1 || h_kv < 1 || h % h_kv != 0 || h > 65535 || !std::isfinite(scale) ||
      !(scale > 0.f))
    return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_DTYPE_F32 && dtype != ATTN_DTYPE_BF16) return ATTN_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return ATTN_ERR_UNSUPPORTED;
  if (n_chunks < 0 || n_chunks > kMaxChunks || (n_chunks > 0 && h_kv % n_chunks != 0))
    return ATTN_ERR_INVALID_ARG;
  if (T == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !scratch) return ATTN_ERR_INVALID_ARG;
  if (!aligned_to(scratch, 256) ||
      scratch_bytes < attn_prefill_host_scratch_bytes(T, h, h_kv, d_h, dtype))
    return ATTN_ERR_INVALID_ARG;
  if (pipe != nullptr) {
    if (!pipe->copy_in || !pipe->copy_out || pipe->copy_in == pipe->copy_out ||
        pipe->copy_in == stream || pipe->copy_out == stream)
      return ATTN_ERR_INVALID_ARG;
    for (int i = 0; i < ATTN_HOST_PIPE_EVENTS; ++i)
      if (!pipe->events[i]) return ATTN_ERR_INVALID_ARG;
  }
  // The attention kernels' own limits, checked before anything is queued.
  if (dtype == ATTN_DTYPE_BF16 && (static_cast<long long>(T) + 127) / 128 > 65535)
    return ATTN_ERR_UNSUPPORTED;
  int sizes[kMaxChunks];
  const int chunks = chunk_plan(h_kv, n_chunks, sizes);
  const size_t elem = dtype == ATTN_DTYPE_F32 ? 4 : 2;
  const size_t ws_bytes = dtype == ATTN_DTYPE_BF16 ? prefill_layout(T, h_kv, d_h).total : 0;
  const HostScratch L = host_scratch(T, h, h_kv, d_h, elem, ws_bytes);
  uint8_t* base = static_cast<uint8_t*>(scratch);
  uint8_t *dq = base + L.q, *dk = base + L.k, *dv = base + L.v, *dO = base + L.o;
  float* dl = reinterpret_cast<float*>(base + L.lse);
  void* dws = dtype == ATTN_DTYPE_BF16 ? base + L.ws : nullptr;

  const int g = h / h_kv;
  const size_t q_head = size_t(T) * d_h * elem;  // one head's Q (and O) or K (and V)
  const size_t l_head = size_t(T) * sizeof(float);
  const auto* hq = static_cast<const uint8_t*>(q);
  const auto* hk = static_cast<const uint8_t*>(k);
  const auto* hv = static_cast<const uint8_t*>(v);
  auto* ho = static_cast<uint8_t*>(o);
  auto* hl = reinterpret_cast<uint8_t*>(lse);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  Pipe P;
  std::unique_lock<std::mutex> lock;
  if (pipe != nullptr) {
    P.in = static_cast<cudaStream_t>(pipe->copy_in);
    P.out = static_cast<cudaStream_t>(pipe->copy_out);
    for (int i = 0; i < ATTN_HOST_PIPE_EVENTS; ++i)
      P.ev[i] = static_cast<cudaEvent_t>(pipe->events[i]);
  } else {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    lock = std::unique_lock<std::mutex>(g_pipes[dev].mu);
    if (ensure_owned_pipe(g_pipes[dev]) != cudaSuccess) return ATTN_ERR_CUDA;
    P = g_pipes[dev].p;
  }
  // Both copy streams start after the work already queued on the caller's
  // stream (which may still be using the scratch).
  cudaError_t e = cudaEventRecord(P.ev[kEvStart], s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.in, P.ev[kEvStart], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.ev[kEvStart], 0);
  for (int c = 0, kv0 = 0; e == cudaSuccess && c < chunks; kv0 += sizes[c], ++c) {
    cudaEvent_t ev_in = P.ev[kEvIn], ev_cmp = P.ev[kEvCmp];
    const int kvc = sizes[c], hc = kvc * g;
    const size_t oq = size_t(kv0) * g * q_head, okv = size_t(kv0) * q_head;
    const size_t ol = size_t(kv0) * g * l_head;
    const size_t q_bytes = size_t(hc) * q_head, kv_bytes = size_t(kvc) * q_head;
    const size_t l_bytes = size_t(hc) * l_head;
    e = cudaMemcpyAsync(dk + okv, hk + okv, kv_bytes, cudaMemcpyHostToDevice, P.in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dv + okv, hv + okv, kv_bytes, cudaMemcpyHostToDevice, P.in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dq + oq, hq + oq, q_bytes, cudaMemcpyHostToDevice, P.in);
    if (e == cudaSuccess) e = cudaEventRecord(ev_in, P.in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_in, 0);
    if (e == cudaSuccess) {
      if (dtype == ATTN_DTYPE_F32)
        e = launch_prefill_f32(reinterpret_cast<const float*>(dq + oq),
                               reinterpret_cast<const float*>(dk + okv),
                               reinterpret_cast<const float*>(dv + okv),
                               reinterpret_cast<float*>(dO + oq),
                               reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dl) + ol), T, hc,
                               kvc, d_h, causal != 0, scale, s);
      else
        e = launch_prefill_bf16(dq + oq, dk + okv, dv + okv, dO + oq,
                                reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dl) + ol), T,
                                hc, kvc, d_h, causal != 0, scale, dws, s);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev_cmp, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, ev_cmp, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ho + oq, dO + oq, q_bytes, cudaMemcpyDeviceToHost, P.out);
    if (e == cudaSuccess && hl)
      e = cudaMemcpyAsync(hl + ol, reinterpret_cast<uint8_t*>(dl) + ol, l_bytes,
                          cudaMemcpyDeviceToHost, P.out);
  }
  // Join: the caller's stream continues after the last copy of both copy
  // streams. Done even after an error, so that nothing queued on them can
  // still read or write the caller's buffers once the stream moves on.
  cudaError_t ej = cudaEventRecord(P.ev[kEvInDone], P.in);
  if (ej == cudaSuccess) ej = cudaStreamWaitEvent(s, P.ev[kEvInDone], 0);
  if (ej == cudaSuccess) ej = cudaEventRecord(P.ev[kEvOutDone], P.out);
  if (ej == cudaSuccess) ej = cudaStreamWaitEvent(s, P.ev[kEvOutDone], 0);
  if (e == cudaSuccess) e = ej;
  if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"

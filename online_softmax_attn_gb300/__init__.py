"""Thin Python binding of the GB300 exact-attention C ABI (``include/attn.h``).

Every function here only marshals arguments: it checks tensor shapes/dtypes,
allocates outputs with PyTorch (device memory is PyTorch's job), and calls the
C entry point of the same name on the current CUDA stream. All arithmetic runs
in the library's CUDA kernels; there is no CPU fallback. If the compiled
library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from .build import LIB_PATH

__all__ = [
    "AttnError",
    "attn_prefill",
    "attn_decode_paged",
    "attn_merge_states",
    "attn_decode_split_plan",
    "attn_recommended_splits",
    "attn_recommended_splits_ragged",
    "attn_decode_workspace_bytes",
    "attn_get_device_error",
    "attn_get_last_device_error",
    "attn_selftest_prefill_stall",
    "attn_status_string",
    "library",
    "ATTN_MAX_SPLITS",
]

(ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_DEVICE,
 ATTN_ERR_DEVICE_TIMEOUT) = range(6)
ATTN_DTYPE_F32, ATTN_DTYPE_BF16 = 0, 1
ATTN_MAX_SPLITS = 1024
# Device error bits (attn_get_device_error), as in attn.h.
(ATTN_DEVERR_WAIT_TIMEOUT, ATTN_DEVERR_BAD_PAGE, ATTN_DEVERR_TMEM, ATTN_DEVERR_BAD_SEQ_LEN,
 ATTN_DEVERR_DEBUG_INDEX) = (0x1, 0x2, 0x4, 0x8, 0x10)
DEVERR_NAMES = {0x1: "wait timeout", 0x2: "page index outside cache",
                0x4: "tensor-memory allocation", 0x8: "seq_len outside table row",
                0x10: "index check failed (debug build)"}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {attn_status_string(status)} (status {status})")


def library() -> ctypes.CDLL:
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"CUDA library not built: {LIB_PATH} is missing "
            "(run `python -m online_softmax_attn_gb300.build`)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, S, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_longlong
    lib.attn_status_string.argtypes = [I]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_version.restype = I
    lib.attn_prefill_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_prefill_workspace_bytes.restype = S
    lib.attn_prefill.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, P, S, P]
    lib.attn_prefill.restype = I
    lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint, P]
    lib.attn_selftest_wait_timeout.restype = I
    lib.attn_prefill_host_scratch_bytes.argtypes = [I, I, I, I, I]
    lib.attn_prefill_host_scratch_bytes.restype = S
    lib.attn_prefill_host.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I, P, S, P, P]
    lib.attn_prefill_host.restype = I
    lib.attn_prefill_paged_workspace_bytes.argtypes = [I]
    lib.attn_prefill_paged_workspace_bytes.restype = S
    lib.attn_prefill_paged_v16_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_prefill_paged_v16_workspace_bytes.restype = S
    lib.attn_prefill_paged_decode_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_prefill_paged_decode_workspace_bytes.restype = S
    lib.attn_prefill_paged.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, I, P, S, P, P,
                                       P]
    lib.attn_prefill_paged.restype = I
    lib.attn_decode_split_plan.argtypes = [I, I, I, ctypes.POINTER(I)]
    lib.attn_decode_split_plan.restype = I
    lib.attn_recommended_splits.argtypes = [I, I, I, I]
    lib.attn_recommended_splits.restype = I
    lib.attn_recommended_splits_ragged.argtypes = [I, I, I, Z, I]
    lib.attn_recommended_splits_ragged.restype = I
    lib.attn_decode_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_decode_workspace_bytes.restype = S
    lib.attn_decode_paged.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, P, S, P, P, P]
    lib.attn_decode_paged.restype = I
    lib.attn_decode_adaptive_workspace_bytes.argtypes = [I, I, I, I]
    lib.attn_decode_adaptive_workspace_bytes.restype = S
    lib.attn_decode_paged_adaptive.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, P, S, P, P, P]
    lib.attn_decode_paged_adaptive.restype = I
    lib.attn_decode_paged_deterministic.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, S, P,
                                                     P, P]
    lib.attn_decode_paged_deterministic.restype = I
    lib.attn_merge_states.argtypes = [P, P, P, P, I, I, I, P, P, I, P]
    lib.attn_merge_states.restype = I
    lib.attn_merge_lse_pair.argtypes = [P, P, P, P, I, I, I, P, P, I, P]
    lib.attn_merge_lse_pair.restype = I
    lib.attn_selftest_delayed_copy.argtypes = [P, P, I, ctypes.c_uint, P]
    lib.attn_selftest_delayed_copy.restype = I
    lib.attn_selftest_prefill_stall.argtypes = [I]
    lib.attn_selftest_prefill_stall.restype = I
    lib.attn_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint)]
    lib.attn_get_device_error.restype = I
    lib.attn_get_last_device_error.argtypes = [P]
    lib.attn_get_last_device_error.restype = I
    _lib = lib
    return lib


def attn_status_string(status: int) -> str:
    return library().attn_status_string(int(status)).decode()


def _check(fn, status):
    if status != ATTN_OK:
        raise AttnError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def attn_prefill_workspace_bytes(T: int, h_kv: int, d_h: int, dtype=torch.bfloat16) -> int:
    """Bytes of scratch attn_prefill uses (fp16 copy of V + per-tile flags)."""
    dt = ATTN_DTYPE_BF16 if dtype == torch.bfloat16 else ATTN_DTYPE_F32
    n = library().attn_prefill_workspace_bytes(T, h_kv, d_h, dt)
    if n == (1 << 64) - 1:
        raise ValueError("invalid arguments to attn_prefill_workspace_bytes")
    return n


def attn_prefill(q, k, v, causal: bool, scale: float | None = None, o=None, lse=None,
                 return_lse: bool = True, stream=None, workspace="auto"):
    """Exact attention prefill. q [h,T,d], k/v [h_kv,T,d] (bf16 or fp32, CUDA,
    contiguous). Returns (o [h,T,d] in q's dtype, lse [h,T] fp32 or None).

    workspace: a uint8 CUDA tensor of at least attn_prefill_workspace_bytes()
    bytes, "auto" (allocated here through torch), or None (no scratch: every
    P V product of the bf16 path takes the exact two-term bf16 form)."""
    _need(q.is_cuda and k.is_cuda and v.is_cuda, "tensors must be on a CUDA device")
    _need(q.dim() == 3 and k.dim() == 3 and v.shape == k.shape, "expected q [h,T,d], k/v [h_kv,T,d]")
    _need(q.dtype == k.dtype == v.dtype and q.dtype in (torch.bfloat16, torch.float32),
          "q, k, v must share dtype bf16 or fp32")
    _need(q.is_contiguous() and k.is_contiguous() and v.is_contiguous(), "tensors must be contiguous")
    h, T, d = q.shape
    h_kv = k.shape[0]
    _need(k.shape[1] == T and k.shape[2] == d, "q and k/v disagree in T or d")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((h, T), dtype=torch.float32, device=q.device)
    dt = ATTN_DTYPE_BF16 if q.dtype == torch.bfloat16 else ATTN_DTYPE_F32
    if isinstance(workspace, str):
        _need(workspace == "auto", 'workspace must be a tensor, "auto" or None')
        n = attn_prefill_workspace_bytes(T, h_kv, d, q.dtype) if T > 0 else 0
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
    ws_bytes = 0
    if workspace is not None:
        _need(workspace.is_cuda and workspace.dtype == torch.uint8 and workspace.is_contiguous(),
              "workspace must be a contiguous uint8 CUDA tensor")
        ws_bytes = workspace.numel()
    st = library().attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), T, h, h_kv, d,
                                int(bool(causal)), scale, dt, _ptr(workspace), ws_bytes,
                                _stream(stream))
    _check("attn_prefill", st)
    return o, lse


def attn_prefill_host_scratch_bytes(T: int, h: int, h_kv: int, d_h: int, dtype=torch.bfloat16) -> int:
    """Device scratch bytes of attn_prefill_host."""
    dt = ATTN_DTYPE_BF16 if dtype == torch.bfloat16 else ATTN_DTYPE_F32
    n = library().attn_prefill_host_scratch_bytes(T, h, h_kv, d_h, dt)
    _need(n != (1 << 64) - 1, "invalid prefill shape")
    return int(n)


ATTN_HOST_PIPE_EVENTS = 5


class HostPipe(ctypes.Structure):
    """attn_host_pipe_t: the caller's two copy streams and five events."""
    _fields_ = [("copy_in", ctypes.c_void_p), ("copy_out", ctypes.c_void_p),
                ("events", ctypes.c_void_p * ATTN_HOST_PIPE_EVENTS)]


def make_host_pipe(copy_in, copy_out, events):
    """A HostPipe from two torch.cuda.Stream and five torch.cuda.Event
    (created without timing). The events are recorded once here, which makes
    torch create them; keep the torch objects alive while the pipe is used."""
    _need(len(events) == ATTN_HOST_PIPE_EVENTS, f"need {ATTN_HOST_PIPE_EVENTS} events")
    for e in events:
        e.record(copy_in)
    hp = HostPipe()
    hp.copy_in = copy_in.cuda_stream
    hp.copy_out = copy_out.cuda_stream
    for i, e in enumerate(events):
        hp.events[i] = e.cuda_event
    hp._keep = (copy_in, copy_out, tuple(events))
    return hp


def attn_prefill_host(q, k, v, causal: bool, scale: float | None = None, o=None, lse=None,
                      return_lse: bool = True, scratch=None, n_chunks: int = 0, stream=None,
                      pipe: HostPipe | None = None):
    """attn_prefill on host tensors: q [h,T,d], k/v [h_kv,T,d] (bf16 or fp32,
    CPU, contiguous; pinned memory lets the copies overlap the compute). The
    copies in and out run inside the call, pipelined over groups of KV heads
    on the current CUDA device, on the copy streams of ``pipe`` (a HostPipe;
    None: the library's own). Returns host (o, lse); they are complete once
    ``stream`` (default: the current stream) has run the queued work."""
    for t in (q, k, v):
        _need(t.device.type == "cpu" and t.is_contiguous(), "q, k, v must be contiguous CPU tensors")
    _need(q.dim() == 3 and k.dim() == 3 and v.shape == k.shape, "expected q [h,T,d], k/v [h_kv,T,d]")
    _need(q.dtype == k.dtype == v.dtype and q.dtype in (torch.bfloat16, torch.float32),
          "q, k, v must share dtype bf16 or fp32")
    h, T, d = q.shape
    h_kv = k.shape[0]
    _need(k.shape[1] == T and k.shape[2] == d, "q and k/v disagree in T or d")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if o is None:
        o = torch.empty(q.shape, dtype=q.dtype, pin_memory=q.is_pinned())
    if lse is None and return_lse:
        lse = torch.empty((h, T), dtype=torch.float32, pin_memory=q.is_pinned())
    for t in (o, lse):
        _need(t is None or (t.device.type == "cpu" and t.is_contiguous()), "o, lse must be contiguous CPU tensors")
    if scratch is None:
        scratch = torch.empty(max(attn_prefill_host_scratch_bytes(T, h, h_kv, d, q.dtype), 256),
                              dtype=torch.uint8, device=torch.cuda.current_device())
    _need(scratch.is_cuda and scratch.dtype == torch.uint8 and scratch.is_contiguous(),
          "scratch must be a contiguous uint8 CUDA tensor")
    dt = ATTN_DTYPE_BF16 if q.dtype == torch.bfloat16 else ATTN_DTYPE_F32
    st = library().attn_prefill_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), T, h, h_kv, d,
                                     int(bool(causal)), scale, dt, int(n_chunks), _ptr(scratch),
                                     scratch.numel(), None if pipe is None else ctypes.byref(pipe),
                                     _stream(stream))
    _check("attn_prefill_host", st)
    return o, lse


def attn_prefill_paged_workspace_bytes(B: int, max_blocks: int = 0, h_kv: int = 0, d_h: int = 0,
                                       v16: bool = False) -> int:
    """Workspace bytes of attn_prefill_paged: the small form (tile offsets),
    or with ``v16`` the form that also holds the fp16 V copy (0 if that copy
    cannot be used for these sizes)."""
    if v16:
        return int(library().attn_prefill_paged_v16_workspace_bytes(B, max_blocks, h_kv, d_h))
    return int(library().attn_prefill_paged_workspace_bytes(B))


def attn_prefill_paged_decode_workspace_bytes(B: int, h: int, decode_splits: int, d_h: int) -> int:
    """Bytes at the front of attn_prefill_paged's workspace for its decode rows."""
    return int(library().attn_prefill_paged_decode_workspace_bytes(B, h, decode_splits, d_h))


def attn_prefill_paged(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, max_q_len: int,
                       causal: bool = True, scale: float | None = None, workspace="auto", o=None,
                       lse=None, return_lse: bool = True, stream=None, decode_splits=None):
    """Variable-length query rows over a paged cache. q [total_q, h, d] bf16
    (rows packed back to back), caches [num_blocks, 16, h_kv, d] bf16,
    block_table [B, max_blocks] int32, cu_seqlens_q [B+1] int32, seq_lens [B]
    int32 (all CUDA). Row b's queries are its last q_len_b key positions.
    ``decode_splits``: rows of one query go to the split-KV decode with at
    most this many splits (0: they run as 1-row query tiles); None means 32
    when the workspace is allocated here and 0 for a caller's workspace.
    ``workspace``: "auto" allocates the fp16-V form when it is available,
    None the small form (all V tiles bf16), or a caller's uint8 CUDA tensor
    (the decode part first, then the prefill's).
    Returns (o [total_q, h, d] bf16, lse [total_q, h] fp32 or None)."""
    for t in (q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens):
        _need(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    _need(q.dtype == k_cache.dtype == v_cache.dtype == torch.bfloat16, "q and caches must be bf16")
    _need(block_table.dtype == cu_seqlens_q.dtype == seq_lens.dtype == torch.int32,
          "block_table, cu_seqlens_q and seq_lens must be int32")
    total_q, h, d = q.shape
    nb, page, h_kv, d2 = k_cache.shape
    _need(d2 == d and v_cache.shape == k_cache.shape, "cache shape mismatch")
    B = seq_lens.shape[0]
    _need(cu_seqlens_q.shape == (B + 1,) and block_table.dim() == 2 and block_table.shape[0] == B,
          "cu_seqlens_q [B+1], block_table [B, max_blocks] and seq_lens [B] expected")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if decode_splits is None:
        decode_splits = 0 if isinstance(workspace, torch.Tensor) else 32
    dec = attn_prefill_paged_decode_workspace_bytes(B, h, decode_splits, d)
    if isinstance(workspace, str):
        _need(workspace == "auto", 'workspace must be "auto", None or a tensor')
        n = attn_prefill_paged_workspace_bytes(B, block_table.shape[1], h_kv, d, v16=True)
        if n == 0:
            n = attn_prefill_paged_workspace_bytes(B)
        workspace = torch.empty(max(dec + n, 256), dtype=torch.uint8, device=q.device)
    elif workspace is None:
        workspace = torch.empty(max(dec + attn_prefill_paged_workspace_bytes(B), 256),
                                dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((total_q, h), dtype=torch.float32, device=q.device)
    st = library().attn_prefill_paged(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(cu_seqlens_q), _ptr(seq_lens),
        B, total_q, h, h_kv, d, page, nb, block_table.shape[1], int(max_q_len), int(bool(causal)),
        scale, int(decode_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(o), _ptr(lse), _stream(stream))
    _check("attn_prefill_paged", st)
    return o, lse


def attn_decode_split_plan(seq_len: int, num_splits: int, page_size: int = 16):
    """(active splits, pages per split) for one row; pure host logic."""
    pps = ctypes.c_int(0)
    n = library().attn_decode_split_plan(int(seq_len), int(page_size), int(num_splits),
                                         ctypes.byref(pps))
    if n < 0:
        raise ValueError("invalid split-plan arguments")
    return n, pps.value


def attn_recommended_splits(B: int, h_kv: int, max_seq_len: int, device: int | None = None) -> int:
    """Split count filling the first wave of `device` (default: the current one)."""
    if device is None:
        device = torch.cuda.current_device()
    s = library().attn_recommended_splits(int(B), int(h_kv), int(max_seq_len), int(device))
    if s < 1:
        raise ValueError("invalid arguments to attn_recommended_splits")
    return s


def attn_recommended_splits_ragged(B: int, h_kv: int, max_seq_len: int, total_seq_len: int,
                                   num_sms: int | None = None) -> int:
    """Split count for a ragged batch (total_seq_len known); pure host logic."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    s = library().attn_recommended_splits_ragged(int(B), int(h_kv), int(max_seq_len),
                                                 int(total_seq_len), int(num_sms))
    if s < 1:
        raise ValueError("invalid arguments to attn_recommended_splits_ragged")
    return s


def attn_decode_workspace_bytes(B: int, h: int, num_splits: int, d_h: int) -> int:
    return int(library().attn_decode_workspace_bytes(int(B), int(h), int(num_splits), int(d_h)))


def attn_decode_paged(q, k_cache, v_cache, block_table, seq_lens, num_splits: int,
                      scale: float | None = None, workspace=None, o=None, lse=None,
                      return_lse: bool = True, stream=None):
    """Split-KV paged decode. q [B,h,d] bf16; caches [num_blocks,16,h_kv,d] bf16;
    block_table [B,max_blocks] int32; seq_lens [B] int32 (all CUDA, contiguous).
    Returns (o [B,h,d] bf16, lse [B,h] fp32 or None)."""
    for t in (q, k_cache, v_cache, block_table, seq_lens):
        _need(t.is_cuda and t.is_contiguous(), "decode tensors must be contiguous CUDA tensors")
    _need(q.dtype == k_cache.dtype == v_cache.dtype == torch.bfloat16, "q and caches must be bf16")
    _need(block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32,
          "block_table and seq_lens must be int32")
    B, h, d = q.shape
    nb, page, h_kv, d2 = k_cache.shape
    _need(d2 == d and v_cache.shape == k_cache.shape, "cache shape mismatch")
    _need(block_table.dim() == 2 and block_table.shape[0] == B and seq_lens.shape == (B,),
          "block_table [B,max_blocks] and seq_lens [B] expected")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    need = attn_decode_workspace_bytes(B, h, num_splits, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, h), dtype=torch.float32, device=q.device)
    st = library().attn_decode_paged(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), B, h, h_kv, d,
        page, nb, block_table.shape[1], int(num_splits), scale, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(o), _ptr(lse), _stream(stream))
    _check("attn_decode_paged", st)
    return o, lse


def attn_decode_adaptive_workspace_bytes(B: int, h: int, max_splits: int, d_h: int) -> int:
    """Partials for max_splits plus 256 bytes for the on-device plan."""
    return library().attn_decode_adaptive_workspace_bytes(B, h, max_splits, d_h)


def attn_decode_paged_adaptive(q, k_cache, v_cache, block_table, seq_lens, max_splits: int,
                               scale: float | None = None, workspace=None, o=None, lse=None,
                               return_lse: bool = True, stream=None):
    """Paged decode whose split count is planned on the device from seq_lens
    (launch geometry fixed by max_splits: capturable in a CUDA graph)."""
    for t in (q, k_cache, v_cache, block_table, seq_lens):
        _need(t.is_cuda and t.is_contiguous(), "decode tensors must be contiguous CUDA tensors")
    _need(q.dtype == k_cache.dtype == v_cache.dtype == torch.bfloat16, "q and caches must be bf16")
    _need(block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32,
          "block_table and seq_lens must be int32")
    B, h, d = q.shape
    nb, page, h_kv, d2 = k_cache.shape
    _need(d2 == d and v_cache.shape == k_cache.shape, "cache shape mismatch")
    _need(block_table.dim() == 2 and block_table.shape[0] == B and seq_lens.shape == (B,),
          "block_table [B,max_blocks] and seq_lens [B] expected")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    need = attn_decode_adaptive_workspace_bytes(B, h, max_splits, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, h), dtype=torch.float32, device=q.device)
    st = library().attn_decode_paged_adaptive(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), B, h, h_kv, d,
        page, nb, block_table.shape[1], int(max_splits), scale, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(o), _ptr(lse), _stream(stream))
    _check("attn_decode_paged_adaptive", st)
    return o, lse


def attn_decode_paged_deterministic(q, k_cache, v_cache, block_table, seq_lens, pages_per_split: int,
                                    scale: float | None = None, num_splits: int | None = None,
                                    workspace=None, o=None, lse=None, return_lse: bool = True,
                                    stream=None):
    """attn_decode_paged with fixed-length splits (pages_per_split pages each):
    each row's result is independent of the rest of the batch. num_splits
    defaults to the smallest grid that covers the block table."""
    for t in (q, k_cache, v_cache, block_table, seq_lens):
        _need(t.is_cuda and t.is_contiguous(), "decode tensors must be contiguous CUDA tensors")
    _need(q.dtype == k_cache.dtype == v_cache.dtype == torch.bfloat16, "q and caches must be bf16")
    _need(block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32,
          "block_table and seq_lens must be int32")
    _need(pages_per_split >= 1, "pages_per_split must be >= 1")
    B, h, d = q.shape
    nb, page, h_kv, d2 = k_cache.shape
    _need(d2 == d and v_cache.shape == k_cache.shape, "cache shape mismatch")
    _need(block_table.dim() == 2 and block_table.shape[0] == B and seq_lens.shape == (B,),
          "block_table [B,max_blocks] and seq_lens [B] expected")
    max_blocks = block_table.shape[1]
    if num_splits is None:
        num_splits = -(-max_blocks // pages_per_split)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    need = attn_decode_workspace_bytes(B, h, num_splits, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, h), dtype=torch.float32, device=q.device)
    st = library().attn_decode_paged_deterministic(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), B, h, h_kv, d,
        page, nb, max_blocks, int(num_splits), int(pages_per_split), scale, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(o), _ptr(lse), _stream(stream))
    _check("attn_decode_paged_deterministic", st)
    return o, lse


def attn_merge_states(o_part, m_part, l_part, n_active=None, out_dtype=torch.bfloat16, o=None,
                      lse=None, return_lse: bool = True, stream=None):
    """N-way merge of split partials: o_part [rows,S,d] fp32, m_part/l_part
    [rows,S] fp32, n_active [rows] int32 or None. Returns (o [rows,d], lse [rows])."""
    for t in (o_part, m_part, l_part):
        _need(t.is_cuda and t.is_contiguous() and t.dtype == torch.float32,
              "partials must be contiguous fp32 CUDA tensors")
    rows, S, d = o_part.shape
    _need(m_part.shape == (rows, S) and l_part.shape == (rows, S), "m/l must be [rows, S]")
    if n_active is not None:
        _need(n_active.is_cuda and n_active.dtype == torch.int32 and n_active.shape == (rows,),
              "n_active must be int32 [rows] on the device")
    _need(out_dtype in (torch.bfloat16, torch.float32), "out_dtype must be bf16 or fp32")
    if o is None:
        o = torch.empty((rows, d), dtype=out_dtype, device=o_part.device)
    if lse is None and return_lse:
        lse = torch.empty((rows,), dtype=torch.float32, device=o_part.device)
    dt = ATTN_DTYPE_BF16 if out_dtype == torch.bfloat16 else ATTN_DTYPE_F32
    st = library().attn_merge_states(_ptr(o_part), _ptr(m_part), _ptr(l_part), _ptr(n_active),
                                     rows, S, d, _ptr(o), _ptr(lse), dt, _stream(stream))
    _check("attn_merge_states", st)
    return o, lse


def attn_merge_lse_pair(o_a, lse_a, o_b, lse_b, out_dtype=torch.bfloat16, o=None, lse=None,
                        return_lse: bool = True, stream=None):
    """Merge two normalised results over disjoint key sets: o_a, o_b [rows, d]
    (bf16 or fp32, same dtype), lse_a, lse_b [rows] fp32. Returns (o [rows, d]
    in out_dtype, lse [rows] fp32 or None). Leading dims are flattened."""
    _need(o_a.shape == o_b.shape and o_a.dtype == o_b.dtype, "o_a and o_b must match")
    _need(o_a.dtype in (torch.bfloat16, torch.float32), "o_a/o_b must be bf16 or fp32")
    for t in (o_a, lse_a, o_b, lse_b):
        _need(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    _need(lse_a.dtype == lse_b.dtype == torch.float32, "lse must be fp32")
    d = o_a.shape[-1]
    rows = o_a.numel() // d
    _need(lse_a.numel() == rows and lse_b.numel() == rows, "lse must hold one value per row")
    if o is None:
        o = torch.empty(o_a.shape, dtype=out_dtype, device=o_a.device)
    if lse is None and return_lse:
        lse = torch.empty(lse_a.shape, dtype=torch.float32, device=o_a.device)
    dt_in = ATTN_DTYPE_BF16 if o_a.dtype == torch.bfloat16 else ATTN_DTYPE_F32
    dt_out = ATTN_DTYPE_BF16 if o.dtype == torch.bfloat16 else ATTN_DTYPE_F32
    st = library().attn_merge_lse_pair(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), rows, d,
                                       dt_in, _ptr(o), _ptr(lse), dt_out, _stream(stream))
    _check("attn_merge_lse_pair", st)
    return o, lse


def attn_selftest_wait_timeout(limit_us: int = 1000, stream=None) -> None:
    """Run a kernel whose bounded wait runs out (nothing arrives on its
    barrier) after ``limit_us`` microseconds: it raises the wait-timeout bit
    of the device error word and returns. For failure-detection tests."""
    _check("attn_selftest_wait_timeout", library().attn_selftest_wait_timeout(int(limit_us), _stream(stream)))


def attn_selftest_delayed_copy(dst, src, delay_us: int = 20, stream=None) -> None:
    """Test aid: let the next kernel on the stream start at once, then after
    delay_us copy src into dst (int32 CUDA tensors of the same size)."""
    _need(dst.is_cuda and src.is_cuda and dst.dtype == src.dtype == torch.int32, "int32 CUDA tensors")
    _need(dst.is_contiguous() and src.is_contiguous() and dst.numel() == src.numel(), "same-size contiguous")
    _check("attn_selftest_delayed_copy",
           library().attn_selftest_delayed_copy(_ptr(dst), _ptr(src), dst.numel(), int(delay_us),
                                                _stream(stream)))


def attn_selftest_prefill_stall(key_tile: int) -> None:
    """Debug builds only: make every CTA of the next contiguous bf16 prefills
    skip loading K for its key_tile-th key tile, so that a bounded wait gives
    up and the kernel takes its abort path (key_tile < 0: off). Raises
    AttnError (UNSUPPORTED) on a release build."""
    _check("attn_selftest_prefill_stall", library().attn_selftest_prefill_stall(int(key_tile)))


def attn_get_device_error(stream=None) -> int:
    """Synchronise the stream; return and clear the device error bits."""
    bits = ctypes.c_uint(0)
    st = library().attn_get_device_error(_stream(stream), ctypes.byref(bits))
    _check("attn_get_device_error", st)
    return bits.value


def attn_get_last_device_error(stream=None) -> int:
    """Synchronise the stream, clear the device error bits, and return them as
    a status: ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT (a bounded wait gave up) or
    ATTN_ERR_DEVICE (any other bit). A failed synchronisation raises."""
    st = library().attn_get_last_device_error(_stream(stream))
    if st == ATTN_ERR_CUDA:
        _check("attn_get_last_device_error", st)
    return st


ATTN_DECODE_STATIC_SCRATCH_BYTES = 16 * 1024 * 1024
_static_ready = False


def attn_decode_paged_static(q, k_cache, v_cache, block_table, seq_lens, num_splits: int,
                             scale: float | None = None, o=None, lse=None, return_lse: bool = True,
                             stream=None):
    """attn_decode_paged without a workspace, for callers that cannot allocate
    device memory at the call site: the split partials live in a fixed
    ATTN_DECODE_STATIC_SCRATCH_BYTES array inside the library on each GPU.
    Calls on one device share that array, so they must not overlap on the GPU
    (issue them on one stream). The first call on a device resolves the
    array's address; make it before any stream capture. Outputs are allocated
    here only when o / lse are not given."""
    global _static_ready
    lib = library()
    if not _static_ready:
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.attn_decode_paged_static.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, P, P, P]
        lib.attn_decode_paged_static.restype = I
        _static_ready = True
    for t in (q, k_cache, v_cache, block_table, seq_lens):
        _need(t.is_cuda and t.is_contiguous(), "decode tensors must be contiguous CUDA tensors")
    B, h, d = q.shape
    nb, page, h_kv, _ = k_cache.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, h), dtype=torch.float32, device=q.device)
    st = lib.attn_decode_paged_static(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), B, h, h_kv, d,
        page, nb, block_table.shape[1], int(num_splits), scale, _ptr(o), _ptr(lse), _stream(stream))
    _check("attn_decode_paged_static", st)
    return o, lse

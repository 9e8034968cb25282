"""Seeded synthetic inputs for the attention workloads.

This module is shared by the tests, the benchmark and the smoke check. It holds
no attention arithmetic: it only draws random numbers, rounds them to the
storage dtype, and lays out a paged KV pool. Both the CUDA path and the float64
oracle consume the tensors it returns; neither side imports the other.

Workload shapes follow the Llama-3-8B layer used throughout "Naive attention and
the online softmax" (h = 32 query heads, h_kv = 8 KV heads, d_h = 128) and the
decode shapes of "Decode attention: FlashDecoding, split-K, paged kernels"
(§"The grid": one query token per sequence, 16-token KV pages).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

PAGE_SIZE = 16


@dataclass(frozen=True)
class PrefillShape:
    name: str
    h: int
    h_kv: int
    d_h: int
    T: int
    dtype: torch.dtype
    causal: bool
    qk_mult: float = 1.0  # Q and K are multiplied by this before rounding

    @property
    def scale(self) -> float:
        return 1.0 / (self.d_h ** 0.5)


@dataclass(frozen=True)
class DecodeShape:
    name: str
    h: int
    h_kv: int
    d_h: int
    seq_lens: tuple = field(default=())  # explicit lengths, or empty for random
    B_random: int = 0  # number of random-length rows
    max_len: int = 0  # random lengths drawn uniform in [1, max_len]
    n_empty: int = 0  # extra zero-length rows inserted at seeded positions

    @property
    def scale(self) -> float:
        return 1.0 / (self.d_h ** 0.5)


# Single-head exact attention, fp32, no mask.
SINGLE_HEAD_T256 = PrefillShape("single_head_fp32_T256_d64", 1, 1, 64, 256, torch.float32, False)
# Llama-3-8B-shaped GQA prefill layer.
GQA_T2048_CAUSAL = PrefillShape("gqa_bf16_T2048_causal", 32, 8, 128, 2048, torch.bfloat16, True)
GQA_T8192_CAUSAL = PrefillShape("gqa_bf16_T8192_causal_x3", 32, 8, 128, 8192, torch.bfloat16, True, 3.0)
GQA_T8192_FULL = PrefillShape("gqa_bf16_T8192_noncausal_x3", 32, 8, 128, 8192, torch.bfloat16, False, 3.0)

# Split-KV decode over one contiguous 32k sequence.
DECODE_S32K = DecodeShape("decode_B1_h32_hkv8_s32768", 32, 8, 128, seq_lens=(32768,))
DECODE_70B_TP8 = DecodeShape("decode_B1_h8_hkv1_s32768", 8, 1, 128, seq_lens=(32768,))
# Paged batched decode: 64 random lengths in [1, 16384] plus 2 empty rows.
DECODE_PAGED_B64 = DecodeShape("paged_decode_B64p2_h32_hkv8", 32, 8, 128,
                               B_random=64, max_len=16384, n_empty=2)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, seed: int, dtype: torch.dtype, device="cpu", mult: float = 1.0) -> torch.Tensor:
    """i.i.d. N(0,1) samples (times ``mult``) drawn in fp32, then rounded to ``dtype``."""
    x = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    if mult != 1.0:
        x.mul_(mult)
    return x.to(dtype)


def prefill_inputs(shape: PrefillShape, seed: int = 0, device="cpu", T: int | None = None):
    """Q [h,T,d_h], K and V [h_kv,T,d_h], contiguous, in ``shape.dtype``.

    For the widened-logit workloads Q and K (not V) are multiplied by ``qk_mult``
    before rounding, which scales the logits' standard deviation by qk_mult**2.
    """
    T = shape.T if T is None else T
    q = normal((shape.h, T, shape.d_h), seed * 3 + 0, shape.dtype, device, shape.qk_mult)
    k = normal((shape.h_kv, T, shape.d_h), seed * 3 + 1, shape.dtype, device, shape.qk_mult)
    v = normal((shape.h_kv, T, shape.d_h), seed * 3 + 2, shape.dtype, device)
    return q, k, v


def decode_seq_lens(shape: DecodeShape, seed: int = 0) -> list[int]:
    """Per-row KV lengths; zero-length rows go to seeded interior positions."""
    if shape.seq_lens:
        lens = list(shape.seq_lens)
    else:
        g = _gen(seed * 7 + 5, "cpu")
        lens = torch.randint(1, shape.max_len + 1, (shape.B_random,), generator=g).tolist()
    if shape.n_empty:
        g = _gen(seed * 7 + 6, "cpu")
        for _ in range(shape.n_empty):
            pos = int(torch.randint(1, len(lens), (1,), generator=g).item())
            lens.insert(pos, 0)
    return lens


def paged_layout(seq_lens: list[int], seed: int = 0, page_size: int = PAGE_SIZE,
                 spare_pages: int = 0):
    """Block table for ``seq_lens`` over a shuffled pool of physical pages.

    Returns (block_table int32 [B, max_blocks], num_blocks). Logical page p of
    row b lives at physical page block_table[b, p]; unused slots hold -1. The
    physical pages are a seeded random permutation of the pool.
    """
    need = [(s + page_size - 1) // page_size for s in seq_lens]
    total = sum(need) + spare_pages
    max_blocks = max(1, max(need) if need else 1)
    perm = torch.randperm(max(total, 1), generator=_gen(seed * 7 + 3, "cpu")).to(torch.int32)
    table = torch.full((len(seq_lens), max_blocks), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, max(total, 1)


def decode_inputs(shape: DecodeShape, seed: int = 0, device="cpu", seq_lens=None,
                  contiguous: bool = False):
    """q [B,h,d_h], K/V caches [num_blocks, 16, h_kv, d_h] (bf16), table, lengths.

    With ``contiguous`` the block table is the identity, so each row's keys are
    one contiguous run of the cache ([s, h_kv, d_h] token-major).
    """
    lens = decode_seq_lens(shape, seed) if seq_lens is None else list(seq_lens)
    B = len(lens)
    if contiguous:
        need = [(s + PAGE_SIZE - 1) // PAGE_SIZE for s in lens]
        max_blocks = max(1, max(need))
        table = torch.full((B, max_blocks), -1, dtype=torch.int32)
        off = 0
        for b, n in enumerate(need):
            table[b, :n] = torch.arange(off, off + n, dtype=torch.int32)
            off += n
        num_blocks = max(off, 1)
    else:
        table, num_blocks = paged_layout(lens, seed)
    q = normal((B, shape.h, shape.d_h), seed * 11 + 0, torch.bfloat16, device)
    kc = normal((num_blocks, PAGE_SIZE, shape.h_kv, shape.d_h), seed * 11 + 1, torch.bfloat16, device)
    vc = normal((num_blocks, PAGE_SIZE, shape.h_kv, shape.d_h), seed * 11 + 2, torch.bfloat16, device)
    seq = torch.tensor(lens, dtype=torch.int32)
    return q, kc, vc, table, seq


def partial_inputs(rows: int, num_splits: int, d_h: int, seed: int = 0, n_active=None,
                   m_spread: float = 30.0):
    """Random split partial states (o~ fp32 [rows,S,d], m, l fp32 [rows,S]).

    The states are synthetic but consistent in kind: l > 0 and m finite for
    active splits; inactive splits (index >= n_active[row]) are filled with NaN
    so that reading them would show. A row with n_active == 0 is empty.
    """
    g = _gen(seed * 13 + 1, "cpu")
    o = torch.randn((rows, num_splits, d_h), generator=g, dtype=torch.float32) * 4.0
    m = torch.randn((rows, num_splits), generator=g, dtype=torch.float32) * m_spread
    l = torch.rand((rows, num_splits), generator=g, dtype=torch.float32) * 100.0 + 1.0
    if n_active is not None:
        na = torch.as_tensor(n_active, dtype=torch.int32)
        idx = torch.arange(num_splits)[None, :]
        dead = idx >= na[:, None].long()
        o[dead[:, :, None].expand_as(o)] = float("nan")
        m[dead] = float("nan")
        l[dead] = float("nan")
    return o, m, l

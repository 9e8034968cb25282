"""attn_decode_paged_static: the decode entry point that allocates nothing.

It serves callers that cannot allocate device memory where they call decode
(for example a plugin inside a host program that owns all device memory, or a
hot loop that must not call cudaMalloc). It keeps the split partials in a
fixed array inside the library instead of a caller workspace. These tests
call it through the C ABI and compare it with attn_decode_paged on the same
inputs, and both with the float64 oracle, for two calls in a row with
different batches (the array keeps the previous call's contents, which must
not leak into the next result).
"""
import ctypes

import pytest
import torch

import online_softmax_attn_gb300 as attn
import oracle
import workloads as W
from parity import check_lse, check_out, to_np

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 * 1024 * 1024


@pytest.fixture(scope="module")
def lib():
    from online_softmax_attn_gb300 import build

    build.build()
    lib = attn.library()
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_decode_paged_static.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, P, P, P]
    lib.attn_decode_paged_static.restype = I
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def call_static(lib, q, kc, vc, table, seq, S, scale, o, lse):
    B, h, d = q.shape
    nb, page, h_kv, _ = kc.shape
    return lib.attn_decode_paged_static(
        _p(q), _p(kc), _p(vc), _p(table), _p(seq), B, h, h_kv, d, page, nb, table.shape[1], S,
        scale, _p(o), _p(lse), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_scratch_matches_workspace_entry_point_twice(lib):
    shape = W.DecodeShape("static", 32, 8, 128)
    cases = [(0, [0, 1, 17, 300, 1000, 5000], 8), (1, [4000, 16, 0, 2500, 77], 3)]
    for seed, lens, S in cases:
        q, kc, vc, table, seq = (t.cuda() for t in W.decode_inputs(shape, seed=seed, seq_lens=lens))
        assert attn.attn_decode_workspace_bytes(len(lens), shape.h, S, shape.d_h) <= SCRATCH_BYTES
        o_ref, lse_ref = attn.attn_decode_paged(q, kc, vc, table, seq, S, shape.scale)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((len(lens), shape.h), float("nan"), device="cuda")
        assert call_static(lib, q, kc, vc, table, seq, S, shape.scale, o, lse) == 0
        torch.cuda.synchronize()
        check_out(o, to_np(o_ref), torch.bfloat16, f"static o (seed {seed})")
        check_lse(lse, to_np(lse_ref), f"static lse (seed {seed})")
        O_or, L_or = oracle.decode_paged_ref(q.cpu(), kc.cpu(), vc.cpu(), table.cpu(), seq.cpu(),
                                             shape.scale)
        check_out(o, O_or, torch.bfloat16, f"static o vs oracle (seed {seed})")
        check_lse(lse, L_or, f"static lse vs oracle (seed {seed})")
    assert attn.attn_get_device_error() == 0


def test_static_scratch_refuses_oversized_request(lib):
    # 64 rows x 32 heads x 64 splits of partials need ~68 MB > 16 MiB: refused
    # on the host before any launch.
    B, h, h_kv, d, S = 64, 32, 8, 128, 64
    assert attn.attn_decode_workspace_bytes(B, h, S, d) > SCRATCH_BYTES
    q = torch.zeros((B, h, d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 16, h_kv, d), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    seq = torch.zeros((B,), dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, h), device="cuda")
    assert call_static(lib, q, kc, kc, table, seq, S, 0.088, o, lse) == attn.ATTN_ERR_INVALID_ARG

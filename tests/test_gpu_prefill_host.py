"""attn_prefill_host: the prefill with host inputs and outputs, copies
pipelined over groups of KV heads inside the call. Heads are independent
("Naive attention and the online softmax": a row's recurrence reads only its
head's Q and its KV head's K, V), so every grouping gives the bits of
attn_prefill on the same inputs; one small case also goes to the oracle."""
import pytest
import torch

import online_softmax_attn_gb300 as attn
import oracle
import workloads as W
from parity import check_lse, check_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_softmax_attn_gb300 import build

    build.build()


def device_result(q, k, v, causal, scale):
    o, lse = attn.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("n_chunks", [0, 1, 2, 4])
def test_bitwise_equal_to_device_call(causal, n_chunks):
    shape = W.PrefillShape("host_gqa", 8, 4, 128, 333, torch.bfloat16, causal)
    q, k, v = W.prefill_inputs(shape, 5)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = attn.attn_prefill_host(hq, hk, hv, causal, shape.scale, n_chunks=n_chunks)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    o_ref, l_ref = device_result(q, k, v, causal, shape.scale)
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_tapered_groups_bitwise():
    """n_chunks = 0 with 8 KV heads: unequal groups of 3, 2, 2 and 1 KV heads."""
    shape = W.PrefillShape("host_taper", 16, 8, 64, 257, torch.bfloat16, True)
    q, k, v = W.prefill_inputs(shape, 6)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = attn.attn_prefill_host(hq, hk, hv, True, shape.scale, n_chunks=0)
    torch.cuda.synchronize()
    o_ref, l_ref = device_result(q, k, v, True, shape.scale)
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_matches_oracle_and_pageable_memory():
    shape = W.PrefillShape("host_gqa_small", 4, 2, 64, 200, torch.bfloat16, True)
    q, k, v = W.prefill_inputs(shape, 6)  # pageable host memory
    o, lse = attn.attn_prefill_host(q, k, v, True, shape.scale, n_chunks=2)
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, True)
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)


def test_fp32_single_head():
    shape = W.SINGLE_HEAD_T256
    q, k, v = W.prefill_inputs(shape, 2)
    o, lse = attn.attn_prefill_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), False, shape.scale)
    torch.cuda.synchronize()
    o_ref, l_ref = device_result(q, k, v, False, shape.scale)
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_captured_in_a_cuda_graph():
    """The call forks onto its copy streams and joins back, so a capture on
    the caller's stream records all of it; replays rewrite the host outputs."""
    shape = W.PrefillShape("host_graph", 8, 2, 128, 300, torch.bfloat16, True)
    q, k, v = W.prefill_inputs(shape, 7)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    ho = torch.empty_like(hq).pin_memory()
    hl = torch.empty((8, 300), dtype=torch.float32).pin_memory()
    scratch = torch.empty(attn.attn_prefill_host_scratch_bytes(300, 8, 2, 128), dtype=torch.uint8,
                          device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # first call creates the library's copy streams, outside the capture
        attn.attn_prefill_host(hq, hk, hv, True, shape.scale, o=ho, lse=hl, scratch=scratch)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            attn.attn_prefill_host(hq, hk, hv, True, shape.scale, o=ho, lse=hl, scratch=scratch)
    torch.cuda.synchronize()
    ho.zero_()
    hl.zero_()
    g.replay()
    torch.cuda.synchronize()
    o_ref, l_ref = device_result(q, k, v, True, shape.scale)
    assert torch.equal(ho, o_ref) and torch.equal(hl, l_ref)


def test_bad_chunk_count_is_rejected():
    q, k, v = W.prefill_inputs(W.PrefillShape("host_bad", 8, 4, 64, 64, torch.bfloat16, True), 1)
    with pytest.raises(RuntimeError):
        attn.attn_prefill_host(q, k, v, True, n_chunks=3)


def _caller_pipe():
    ins, outs = torch.cuda.Stream(), torch.cuda.Stream()
    evs = [torch.cuda.Event() for _ in range(attn.ATTN_HOST_PIPE_EVENTS)]
    return attn.make_host_pipe(ins, outs, evs)


@pytest.mark.parametrize("n_chunks", [0, 8])
def test_caller_pipe_bitwise(n_chunks):
    """The caller's copy streams and events: the library creates nothing, the
    five events are reused across the groups (8 groups here), and the result
    is bitwise that of attn_prefill."""
    shape = W.PrefillShape("host_pipe", 16, 8, 128, 333, torch.bfloat16, True)
    q, k, v = W.prefill_inputs(shape, 8)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    pipe = _caller_pipe()
    o, lse = attn.attn_prefill_host(hq, hk, hv, True, shape.scale, n_chunks=n_chunks, pipe=pipe)
    torch.cuda.synchronize()
    o_ref, l_ref = device_result(q, k, v, True, shape.scale)
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_caller_pipe_captured_without_a_prior_call():
    """With the caller's pipe nothing is created inside the call, so its very
    first call may be inside a stream capture."""
    shape = W.PrefillShape("host_pipe_graph", 8, 4, 64, 200, torch.bfloat16, False)
    q, k, v = W.prefill_inputs(shape, 9)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    ho = torch.empty_like(hq).pin_memory()
    hl = torch.empty((8, 200), dtype=torch.float32).pin_memory()
    scratch = torch.empty(attn.attn_prefill_host_scratch_bytes(200, 8, 4, 64), dtype=torch.uint8,
                          device="cuda")
    pipe = _caller_pipe()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            attn.attn_prefill_host(hq, hk, hv, False, shape.scale, o=ho, lse=hl, scratch=scratch,
                                   pipe=pipe)
    g.replay()
    torch.cuda.synchronize()
    o_ref, l_ref = device_result(q, k, v, False, shape.scale)
    assert torch.equal(ho, o_ref) and torch.equal(hl, l_ref)

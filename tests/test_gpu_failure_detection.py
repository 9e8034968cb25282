"""Failure detection without a fault: a kernel's bounded wait on an mbarrier
that nothing arrives on gives up, the host reads the wait-timeout bit, and the
context keeps working (a decode after it is exact)."""
import time

import pytest
import torch

import online_softmax_attn_gb300 as attn
import oracle
import workloads as W
from parity import check_lse, check_out

pytestmark = pytest.mark.gpu

WAIT_TIMEOUT = 0x1


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_softmax_attn_gb300 import build

    build.build()


def test_wait_runs_out_and_is_reported():
    assert attn.attn_get_device_error() == 0
    t0 = time.perf_counter()
    attn.attn_selftest_wait_timeout(2000)  # 2 ms
    bits = attn.attn_get_device_error()  # synchronises
    elapsed = time.perf_counter() - t0
    assert bits & WAIT_TIMEOUT
    assert elapsed >= 0.002
    assert attn.attn_get_device_error() == 0  # read clears


def test_timeout_as_status():
    """The status form of the query: ATTN_ERR_DEVICE_TIMEOUT after a wait ran
    out, ATTN_OK once read."""
    assert attn.attn_get_last_device_error() == attn.ATTN_OK
    attn.attn_selftest_wait_timeout(300)
    assert attn.attn_get_last_device_error() == attn.ATTN_ERR_DEVICE_TIMEOUT
    assert attn.attn_get_last_device_error() == attn.ATTN_OK


def test_context_usable_after_timeout():
    attn.attn_selftest_wait_timeout(500)
    assert attn.attn_get_device_error() & WAIT_TIMEOUT
    shape = W.DECODE_PAGED_B64
    lens = [300, 0, 17, 2048]
    q, kc, vc, table, seq = W.decode_inputs(shape, 4, seq_lens=lens)
    o, lse = attn.attn_decode_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), seq.cuda(), 4, shape.scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, table, seq, shape.scale)
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)

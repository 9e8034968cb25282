"""attn_decode_paged_deterministic: fixed-length splits make a row's result
independent of the batch it is in ([DEC] "Split-K breaks bitwise
reproducibility"): bit-identical alone and inside different batches, and
within tolerance of the oracle."""
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


@pytest.mark.parametrize("pps", [8, 128])
def test_row_bitwise_identical_across_batches(pps):
    shape = W.DECODE_PAGED_B64
    row_len = 3001
    pool_lens = [row_len, 4000, 17, 2500, 1, 3999, 640, 1200]
    q_all, kc, vc, table, seq = W.decode_inputs(shape, 3, seq_lens=pool_lens)
    dq, dk, dv = q_all.cuda(), kc.cuda(), vc.cuda()
    # alone: row 0 of the pool, grid just wide enough
    o1, l1 = attn.attn_decode_paged_deterministic(dq[:1].contiguous(), dk, dv, table[:1].cuda(),
                                                  seq[:1].cuda(), pps)
    # in the whole pool, with a wider grid than needed
    o8, l8 = attn.attn_decode_paged_deterministic(dq, dk, dv, table.cuda(), seq.cuda(), pps,
                                                  num_splits=64)
    # in a different batch: the row moved to the end, two other rows
    idx = torch.tensor([5, 2, 0])
    o3, l3 = attn.attn_decode_paged_deterministic(dq[idx].contiguous(), dk, dv,
                                                  table[idx].contiguous().cuda(),
                                                  seq[idx].contiguous().cuda(), pps, num_splits=40)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    assert torch.equal(o1[0], o8[0]) and torch.equal(l1[0], l8[0])
    assert torch.equal(o1[0], o3[2]) and torch.equal(l1[0], l3[2])
    O_ref, L_ref = oracle.decode_paged_ref(q_all, kc, vc, table, seq, shape.scale)
    check_out(o8, O_ref, torch.bfloat16)
    check_lse(l8, L_ref)


def test_deterministic_empty_and_short_rows():
    shape = W.DECODE_PAGED_B64
    lens = [0, 1, 16, 17, 300]
    q, kc, vc, table, seq = W.decode_inputs(shape, 4, seq_lens=lens)
    o, lse = attn.attn_decode_paged_deterministic(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(),
                                                  seq.cuda(), 4)
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, table, seq, shape.scale)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)

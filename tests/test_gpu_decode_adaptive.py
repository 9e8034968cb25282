"""attn_decode_paged_adaptive: the split count is planned on the device from
seq_lens under a fixed launch geometry ([DEC] "SGLang: a split count computed
per sequence, on device", "CUDA graphs need the split count pinned")."""
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


def expected_pps(lens, h_kv, max_splits):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s = attn.attn_recommended_splits_ragged(len(lens), h_kv, max(lens), sum(lens), sms)
    s = min(s, max_splits)
    max_pages = (max(lens) + 15) // 16
    return max(1, -(-max_pages // s))


def plan_of(ws, B, h, d, max_splits):
    off = attn.attn_decode_workspace_bytes(B, h, max_splits, d)
    return int(ws[off:off + 4].view(torch.int32).item())


@pytest.mark.parametrize("lens,max_splits", [
    ([1, 6000, 0, 17, 3000, 4096, 255, 1], 32),   # ragged, with an empty row
    ([32768], 64),                                 # one long row
    ([32768], 7),                                  # grid narrower than the rule asks
    ([100] * 12, 16),                              # uniform short rows
])
def test_adaptive_matches_oracle_and_host_rule(lens, max_splits):
    shape = W.DECODE_PAGED_B64
    q, kc, vc, table, seq = W.decode_inputs(shape, 8, seq_lens=lens)
    B = len(lens)
    ws = torch.empty(attn.attn_decode_adaptive_workspace_bytes(B, shape.h, max_splits, shape.d_h),
                     dtype=torch.uint8, device="cuda")
    o, lse = attn.attn_decode_paged_adaptive(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), seq.cuda(),
                                             max_splits, shape.scale, workspace=ws)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    assert plan_of(ws, B, shape.h, shape.d_h, max_splits) == expected_pps(lens, shape.h_kv, max_splits)
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, table, seq, shape.scale)
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)


def test_graph_replay_adapts_to_new_lengths():
    """One capture; new seq_lens written on the device between replays; the
    plan and the results follow the new lengths without a recapture."""
    shape = W.DECODE_PAGED_B64
    lens_a = [4000, 16, 2500, 700, 3999, 1]
    lens_b = [16, 4000, 1, 0, 900, 3100]
    table_lens = [max(a, b) for a, b in zip(lens_a, lens_b)]
    q, kc, vc, table, _ = W.decode_inputs(shape, 9, seq_lens=table_lens)
    B, S = len(lens_a), 48
    dq, dk, dv, dt = q.cuda(), kc.cuda(), vc.cuda(), table.cuda()
    seq = torch.tensor(lens_a, dtype=torch.int32, device="cuda")
    ws = torch.empty(attn.attn_decode_adaptive_workspace_bytes(B, shape.h, S, shape.d_h),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty_like(dq)
    lse = torch.empty(B, shape.h, device="cuda")
    attn.attn_decode_paged_adaptive(dq, dk, dv, dt, seq, S, shape.scale, workspace=ws, o=o, lse=lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            attn.attn_decode_paged_adaptive(dq, dk, dv, dt, seq, S, shape.scale, workspace=ws, o=o, lse=lse)
    torch.cuda.synchronize()
    for lens in (lens_a, lens_b, lens_a):
        seq.copy_(torch.tensor(lens, dtype=torch.int32))
        o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert attn.attn_get_device_error() == 0
        assert plan_of(ws, B, shape.h, shape.d_h, S) == expected_pps(lens, shape.h_kv, S)
        O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, table, torch.tensor(lens, dtype=torch.int32),
                                               shape.scale)
        check_out(o, O_ref, torch.bfloat16)
        check_lse(lse, L_ref)

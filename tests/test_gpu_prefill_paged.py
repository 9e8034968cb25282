"""attn_prefill_paged (variable-length query rows over a paged cache: chunked
prefill and mixed prefill/decode batches) against the oracle."""
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


def paged_batch(q_lens, ctx_lens, h, h_kv, d, seed):
    page = W.PAGE_SIZE
    table, nblk = W.paged_layout(ctx_lens, seed)
    cu = torch.zeros(len(q_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int32), 0)
    q = W.normal((int(cu[-1]), h, d), seed * 5 + 1, torch.bfloat16)
    kc = W.normal((nblk, page, h_kv, d), seed * 5 + 2, torch.bfloat16)
    vc = W.normal((nblk, page, h_kv, d), seed * 5 + 3, torch.bfloat16)
    return q, kc, vc, table, cu, torch.tensor(ctx_lens, dtype=torch.int32)


MIXED = ([1, 128, 200, 77, 5, 300, 1, 129],
         [300, 128, 1000, 77, 4096, 813, 1, 129])


@pytest.mark.parametrize("h,h_kv,d", [(8, 2, 128), (6, 2, 128), (4, 2, 64)])
@pytest.mark.parametrize("causal", [True, False])
def test_mixed_batch_matches_oracle(h, h_kv, d, causal):
    q_lens, ctx = MIXED
    q, kc, vc, table, cu, seq = paged_batch(q_lens, ctx, h, h_kv, d, 3)
    scale = 1.0 / d ** 0.5
    o, lse = attn.attn_prefill_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cu.cuda(), seq.cuda(),
                                     max(q_lens), causal, scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    O_ref, L_ref = oracle.prefill_paged_ref(q, kc, vc, table, cu, seq, scale, causal)
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)


def test_chunked_prefill_equals_whole_row():
    """A 700-token row prefilled in chunks of 256 / 256 / 188 (each chunk's
    queries are the last positions of the keys written so far) gives the
    same outputs as the whole row at once, which is the square causal case."""
    h, h_kv, d, T = 8, 2, 128, 700
    q, kc, vc, table, _, _ = paged_batch([T], [T], h, h_kv, d, 4)
    scale = 1.0 / d ** 0.5
    dq, dk, dv, dt = q.cuda(), kc.cuda(), vc.cuda(), table.cuda()
    whole, wl = attn.attn_prefill_paged(dq, dk, dv, dt, torch.tensor([0, T], dtype=torch.int32).cuda(),
                                        torch.tensor([T], dtype=torch.int32).cuda(), T, True, scale)
    parts, lparts, done = [], [], 0
    for n in (256, 256, 188):
        o, l = attn.attn_prefill_paged(dq[done:done + n].contiguous(), dk, dv, dt,
                                       torch.tensor([0, n], dtype=torch.int32).cuda(),
                                       torch.tensor([done + n], dtype=torch.int32).cuda(), n, True, scale)
        parts.append(o)
        lparts.append(l)
        done += n
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.prefill_paged_ref(q, kc, vc, table, torch.tensor([0, T]), torch.tensor([T]),
                                            scale, True)
    check_out(whole, O_ref, torch.bfloat16)
    check_out(torch.cat(parts), O_ref, torch.bfloat16)
    check_lse(torch.cat(lparts), L_ref)


def test_bad_page_sets_error_without_fault():
    h, h_kv, d = 4, 2, 128
    q, kc, vc, table, cu, seq = paged_batch([40, 3], [300, 20], h, h_kv, d, 5)
    table = table.clone()
    table[0, 5] = kc.shape[0] + 7   # outside the cache: read as zeros, flagged
    attn.attn_prefill_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cu.cuda(), seq.cuda(), 40, True,
                            1.0 / d ** 0.5)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() & 0x2  # page index outside the cache
    assert attn.attn_get_device_error() == 0  # read clears

"""attn_merge_lse_pair (pairwise (O, LSE) merge) against the oracle, and the
cascade form: a shared prefix and per-row suffixes decoded separately, then
merged, against one decode of the whole row."""
import numpy as np
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


def pair_inputs(rows, d, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    oa = torch.randn(rows, d, generator=g)
    ob = torch.randn(rows, d, generator=g)
    la = torch.randn(rows, generator=g) * 20
    lb = torch.randn(rows, generator=g) * 20
    idx = torch.arange(rows)
    la[idx % 7 == 3] = -float("inf")        # empty left side
    lb[idx % 11 == 5] = -float("inf")       # empty right side
    both = idx % 13 == 6
    la[both] = -float("inf")
    lb[both] = -float("inf")                # both empty
    la[idx % 17 == 1] = lb[idx % 17 == 1]   # equal masses
    return oa.to(dtype), la, ob.to(dtype), lb


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("in_dtype,out_dtype", [(torch.bfloat16, torch.bfloat16),
                                                (torch.float32, torch.float32),
                                                (torch.bfloat16, torch.float32)])
@pytest.mark.parametrize("rows", [1, 333, 4099])
def test_pair_merge_matches_oracle(d, in_dtype, out_dtype, rows):
    oa, la, ob, lb = pair_inputs(rows, d, rows + d, in_dtype)
    O_ref, L_ref = oracle.merge_lse_pair_ref(oa, la, ob, lb)
    o, lse = attn.attn_merge_lse_pair(oa.cuda(), la.cuda(), ob.cuda(), lb.cuda(), out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert not torch.isnan(o).any()
    check_out(o, O_ref, out_dtype)
    check_lse(lse, L_ref)
    both = (np.isneginf(la.numpy()) & np.isneginf(lb.numpy()))
    assert torch.all(o[torch.from_numpy(both).cuda()] == 0)


def test_pair_merge_in_place():
    oa, la, ob, lb = pair_inputs(256, 128, 3, torch.float32)
    O_ref, L_ref = oracle.merge_lse_pair_ref(oa, la, ob, lb)
    ga = oa.cuda()
    o, lse = attn.attn_merge_lse_pair(ga, la.cuda(), ob.cuda(), lb.cuda(), out_dtype=torch.float32, o=ga)
    torch.cuda.synchronize()
    assert o.data_ptr() == ga.data_ptr()
    check_out(o, O_ref, torch.float32)
    check_lse(lse, L_ref)


def cascade_layout(B, prefix_pages, suffix_lens, seed):
    """Block tables over one pool: the prefix pages are shared by every row."""
    page = W.PAGE_SIZE
    sfx_pages = [(s + page - 1) // page for s in suffix_lens]
    pool = prefix_pages + sum(sfx_pages)
    perm = torch.randperm(pool, generator=torch.Generator().manual_seed(seed)).to(torch.int32)
    pre = perm[:prefix_pages]
    max_sfx = max(1, max(sfx_pages))
    full = torch.full((B, prefix_pages + max_sfx), -1, dtype=torch.int32)
    sfx = torch.full((B, max_sfx), -1, dtype=torch.int32)
    off = prefix_pages
    for b, n in enumerate(sfx_pages):
        full[b, :prefix_pages] = pre
        full[b, prefix_pages:prefix_pages + n] = perm[off:off + n]
        sfx[b, :n] = perm[off:off + n]
        off += n
    pre_tab = pre.unsqueeze(0).expand(B, prefix_pages).contiguous()
    return pool, full, pre_tab, sfx


@pytest.mark.parametrize("prefix_pages", [64, 1])
def test_cascade_prefix_suffix_equals_full_decode(prefix_pages):
    """[NA] cascade: attend to the shared prefix once per row, to each row's
    own suffix separately, merge the two (O, LSE) results; equals the
    attention over prefix + suffix. Rows with an empty suffix are included."""
    shape = W.DECODE_S32K  # h=32, h_kv=8, d_h=128
    B = 6
    g = torch.Generator().manual_seed(11)
    suffix = torch.randint(1, 700, (B,), generator=g).tolist()
    suffix[2] = 0
    pre_len = prefix_pages * W.PAGE_SIZE
    pool, full, pre_tab, sfx_tab = cascade_layout(B, prefix_pages, suffix, 5)
    q = W.normal((B, shape.h, shape.d_h), 40, torch.bfloat16)
    kc = W.normal((pool, W.PAGE_SIZE, shape.h_kv, shape.d_h), 41, torch.bfloat16)
    vc = W.normal((pool, W.PAGE_SIZE, shape.h_kv, shape.d_h), 42, torch.bfloat16)
    full_len = torch.tensor([pre_len + s for s in suffix], dtype=torch.int32)
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, full, full_len, shape.scale)

    dq, dk, dv = q.cuda(), kc.cuda(), vc.cuda()
    S = 4
    op, lp = attn.attn_decode_paged(dq, dk, dv, pre_tab.cuda(),
                                    torch.full((B,), pre_len, dtype=torch.int32).cuda(), S, shape.scale)
    os_, ls = attn.attn_decode_paged(dq, dk, dv, sfx_tab.cuda(),
                                     torch.tensor(suffix, dtype=torch.int32).cuda(), S, shape.scale)
    o, lse = attn.attn_merge_lse_pair(op, lp, os_, ls)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    assert torch.isneginf(ls[2]).all()  # the empty suffix
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)


@pytest.mark.parametrize("prefix_pages", [64, 1])
def test_cascade_shared_prefix_on_tensor_cores(prefix_pages):
    """The shared prefix attended once for all rows: the B decode queries form
    one row of attn_prefill_paged (q_len = B, non-causal, the prefix pages as
    its cache), so the prefix K/V are read once and the B queries are MMA
    rows; each row's own suffix goes through the decode kernel; the pair merge
    joins them. Equals the attention over prefix + suffix."""
    shape = W.DECODE_S32K  # h=32, h_kv=8, d_h=128
    B = 6
    g = torch.Generator().manual_seed(12)
    suffix = torch.randint(1, 700, (B,), generator=g).tolist()
    suffix[4] = 0
    pre_len = prefix_pages * W.PAGE_SIZE
    pool, full, pre_tab, sfx_tab = cascade_layout(B, prefix_pages, suffix, 6)
    q = W.normal((B, shape.h, shape.d_h), 50, torch.bfloat16)
    kc = W.normal((pool, W.PAGE_SIZE, shape.h_kv, shape.d_h), 51, torch.bfloat16)
    vc = W.normal((pool, W.PAGE_SIZE, shape.h_kv, shape.d_h), 52, torch.bfloat16)
    full_len = torch.tensor([pre_len + s for s in suffix], dtype=torch.int32)
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, full, full_len, shape.scale)

    dq, dk, dv = q.cuda(), kc.cuda(), vc.cuda()
    op, lp = attn.attn_prefill_paged(dq, dk, dv, pre_tab[:1].contiguous().cuda(),
                                     torch.tensor([0, B], dtype=torch.int32).cuda(),
                                     torch.tensor([pre_len], dtype=torch.int32).cuda(), B,
                                     causal=False, scale=shape.scale)
    os_, ls = attn.attn_decode_paged(dq, dk, dv, sfx_tab.cuda(),
                                     torch.tensor(suffix, dtype=torch.int32).cuda(), 4, shape.scale)
    o, lse = attn.attn_merge_lse_pair(op, lp, os_, ls)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)

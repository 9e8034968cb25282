"""Inputs holding NaN or inf, every kernel against the oracle.

Policy ("Naive attention and the online softmax", "The base case is a NaN
factory", on how a NaN spreads through the weighted sums): IEEE arithmetic on
the definition over each row's allowed keys. A NaN logit (a NaN in q or in an
attended k) makes the row's output and LSE NaN; a NaN or +-inf in an attended
v_j[e] makes column e of the row NaN or +-inf (which of the two for an
infinity is not promised); keys a row does not attend never reach it -- in
particular the slots of a row's last page past its length, which in a real
cache hold whatever was there before. One stated exception: in the causal
tensor-core prefill a non-finite V value at key j also makes column e NaN in
the rows of j's 128-query diagonal tile that precede j, because the tile's
P V product multiplies their zero weights by it (0 * NaN = NaN).
"""
import math

import numpy as np
import pytest
import torch

import online_softmax_attn_gb300 as attn
import oracle
import workloads as W
from parity import check_lse_nonfinite, check_nonfinite

pytestmark = pytest.mark.gpu

NAN, INF = math.nan, math.inf


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_softmax_attn_gb300 import build

    build.build()


def prefill(q, k, v, causal, scale, workspace="auto"):
    o, lse = attn.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal, scale, workspace=workspace)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("workspace", ["auto", None], ids=["fp16V", "bf16V"])
def test_prefill_nan_in_k(causal, workspace):
    shape = W.PrefillShape("nf_k", 4, 2, 128, 520, torch.bfloat16, causal)
    q, k, v = W.prefill_inputs(shape, 31)
    k[0, 200, 17] = NAN  # KV head 0: query heads 0 and 1, every row that attends key 200
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, causal)
    o, lse = prefill(q, k, v, causal, shape.scale, workspace)
    n = check_nonfinite(o, O_ref, torch.bfloat16, "nan in k")
    check_lse_nonfinite(lse, L_ref)
    assert n == 2 * (shape.T - 200 if causal else shape.T) * shape.d_h
    assert attn.attn_get_device_error() == 0


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("workspace", ["auto", None], ids=["fp16V", "bf16V"])
@pytest.mark.parametrize("value", [NAN, INF, -INF], ids=["nan", "inf", "-inf"])
def test_prefill_nonfinite_v(causal, workspace, value):
    """At the first key of a 128-key tile every row of the tile's diagonal
    query tile attends it, so the result is exactly the oracle's."""
    shape = W.PrefillShape("nf_v", 4, 2, 128, 520, torch.bfloat16, causal)
    q, k, v = W.prefill_inputs(shape, 32)
    v[1, 256, 5] = value
    v[0, 384, 9] = value
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, causal)
    o, lse = prefill(q, k, v, causal, shape.scale, workspace)
    n = check_nonfinite(o, O_ref, torch.bfloat16, "non-finite v")
    check_lse_nonfinite(lse, L_ref)
    rows = (shape.T - 256) + (shape.T - 384) if causal else 2 * shape.T
    assert n == 2 * rows


@pytest.mark.parametrize("workspace", ["auto", None], ids=["fp16V", "bf16V"])
def test_prefill_nonfinite_v_inside_causal_tile(workspace):
    """The stated exception: NaN at key 300 (inside the diagonal tile of query
    rows 256-383) also reaches column 5 of rows 256-299 of the two query heads
    of that KV head, which do not attend key 300. Everything else is exact."""
    shape = W.PrefillShape("nf_band", 4, 2, 128, 520, torch.bfloat16, True)
    q, k, v = W.prefill_inputs(shape, 33)
    v[1, 300, 5] = NAN
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, True)
    o, lse = prefill(q, k, v, True, shape.scale, workspace)
    band = np.zeros(O_ref.shape, bool)
    band[2:4, 256:300, 5] = True
    check_nonfinite(o, O_ref, torch.bfloat16, "band", extra=band)
    check_lse_nonfinite(lse, L_ref)


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_fp32_nonfinite(causal):
    """The fp32 SIMT path is exact: a masked key's values never enter a sum."""
    shape = W.PrefillShape("nf_f32", 2, 2, 64, 256, torch.float32, causal)
    q, k, v = W.prefill_inputs(shape, 34)
    k[0, 200, 3] = NAN  # head 0
    v[1, 150, 7] = INF  # head 1
    v[1, 37, 1] = NAN   # head 1, inside a 32-key tile: rows 32-36 do not attend it
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, causal)
    o, lse = prefill(q, k, v, causal, shape.scale)
    check_nonfinite(o, O_ref, torch.float32, "fp32")
    check_lse_nonfinite(lse, L_ref)


def paged_rows(q_lens, ctx, h, h_kv, d, seed):
    table, nblk = W.paged_layout(ctx, seed)
    cu = torch.zeros(len(q_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int32), 0)
    q = W.normal((int(cu[-1]), h, d), seed * 5 + 1, torch.bfloat16)
    kc = W.normal((nblk, W.PAGE_SIZE, h_kv, d), seed * 5 + 2, torch.bfloat16)
    vc = W.normal((nblk, W.PAGE_SIZE, h_kv, d), seed * 5 + 3, torch.bfloat16)
    return q, kc, vc, table, cu, torch.tensor(ctx, dtype=torch.int32)


def fill_tail(cache, table, lens, value):
    """Write `value` into the slots of each row's last page past its length
    (what an uninitialised cache may hold there)."""
    for b, s in enumerate(lens):
        if s % W.PAGE_SIZE:
            cache[int(table[b, s // W.PAGE_SIZE]), s % W.PAGE_SIZE:] = value


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("workspace", ["auto", None], ids=["fp16V", "bf16V"])
def test_paged_prefill_nonfinite(causal, workspace):
    h, h_kv, d = 8, 2, 128
    q_lens, ctx = [200, 64, 1, 30], [1000, 600, 300, 37]
    q, kc, vc, table, cu, seq = paged_rows(q_lens, ctx, h, h_kv, d, 12)
    P = W.PAGE_SIZE
    kc[int(table[0, 300 // P]), 300 % P, 1, 4] = NAN   # row 0 (queries at 800-999 attend key 300)
    vc[int(table[1, 100 // P]), 100 % P, 0, 9] = NAN   # row 1 (queries at 536-599)
    vc[int(table[1, 200 // P]), 200 % P, 1, 3] = INF
    vc[int(table[3, 0]), 3, 0, 0] = -INF               # row 3, key 3 (queries at 7-36)
    fill_tail(kc, table, ctx, NAN)
    fill_tail(vc, table, ctx, NAN)
    O_ref, L_ref = oracle.prefill_paged_ref(q, kc, vc, table, cu, seq, 1.0 / d ** 0.5, causal)
    o, lse = attn.attn_prefill_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cu.cuda(),
                                     seq.cuda(), max(q_lens), causal, 1.0 / d ** 0.5,
                                     workspace=workspace)
    torch.cuda.synchronize()
    n = check_nonfinite(o.cpu(), O_ref, torch.bfloat16, "paged prefill")
    check_lse_nonfinite(lse.cpu(), L_ref)
    assert n > 0
    assert attn.attn_get_device_error() == 0


@pytest.mark.parametrize("S", [1, 4, 16])
def test_decode_nonfinite(S):
    shape = W.DecodeShape("nf_dec", 32, 8, 128)
    lens = [40, 300, 17, 1000, 0]
    q, kc, vc, table, seq = W.decode_inputs(shape, seed=13, seq_lens=lens)
    P = W.PAGE_SIZE
    kc[int(table[0, 20 // P]), 20 % P, 3, 50] = NAN    # row 0, KV head 3
    vc[int(table[1, 299 // P]), 299 % P, 2, 7] = NAN   # row 1, its last key
    vc[int(table[1, 0]), 0, 5, 100] = -INF
    vc[int(table[3, 512 // P]), 512 % P, 0, 0] = INF
    fill_tail(kc, table, lens, NAN)
    fill_tail(vc, table, lens, INF)
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, table, seq, shape.scale)
    o, lse = attn.attn_decode_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), seq.cuda(), S)
    torch.cuda.synchronize()
    n = check_nonfinite(o.cpu(), O_ref, torch.bfloat16, f"decode S={S}")
    check_lse_nonfinite(lse.cpu(), L_ref)
    assert n == 4 * 128 + 3 * 4
    assert torch.all(o[4] == 0) and torch.all(torch.isneginf(lse[4]))
    assert attn.attn_get_device_error() == 0


def test_merge_states_nan_partials():
    """A NaN in an active split's m, l or O~ reaches the row (all of it for m
    and l, one column for O~); splits past n_active are never read."""
    rows, S, d = 5, 6, 128
    o, m, l = W.partial_inputs(rows, S, d, seed=3, n_active=[6, 6, 3, 0, 6])
    m[0, 2] = NAN
    l[1, 4] = NAN
    o[2, 1, 5] = NAN
    m[4, :] = -INF   # every split of row 4 empty: the empty row, not NaN
    l[4, :] = 0.0
    na = torch.tensor([6, 6, 3, 0, 6], dtype=torch.int32)
    O_ref, L_ref = oracle.merge_partials_ref(o, m, l, na)
    out, lse = attn.attn_merge_states(o.cuda(), m.cuda(), l.cuda(), na.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    n = check_nonfinite(out.cpu(), O_ref, torch.float32, "merge states")
    check_lse_nonfinite(lse.cpu(), L_ref)
    assert n == 2 * d + 1
    assert torch.all(out[3] == 0) and torch.all(out[4] == 0) and torch.isneginf(lse[3:]).all()


def test_merge_pair_nan_side():
    """A NaN LSE on one side is not an empty side, whichever side it is."""
    rows, d = 4, 128
    g = torch.Generator().manual_seed(5)
    oa = torch.randn(rows, d, generator=g)
    ob = torch.randn(rows, d, generator=g)
    la = torch.tensor([NAN, -INF, 0.3, NAN])
    lb = torch.tensor([-INF, NAN, NAN, NAN])
    O_ref, L_ref = oracle.merge_lse_pair_ref(oa, la, ob, lb)
    o, lse = attn.attn_merge_lse_pair(oa.cuda(), la.cuda(), ob.cuda(), lb.cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.isnan(o).all() and torch.isnan(lse).all()
    check_nonfinite(o.cpu(), O_ref, torch.float32, "merge pair")

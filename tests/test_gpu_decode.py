"""attn_decode_paged (CUDA split-KV decode + merge) against the oracle."""
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


def run_decode(q, kc, vc, table, lens, S, **kw):
    o, lse = attn.attn_decode_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), lens.cuda(), S, **kw)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("g,h_kv", [(1, 4), (2, 2), (4, 2), (8, 1)])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_small_edges(g, h_kv, d):
    """Lengths that are empty, one key, and end before / at / after a page edge."""
    shape = W.DecodeShape("t", g * h_kv, h_kv, d)
    lens = [0, 1, 15, 16, 17, 40, 333, 1000]
    q, kc, vc, table, seq = W.decode_inputs(shape, seed=g * 10 + d, seq_lens=lens)
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, table, seq, shape.scale)
    for S in (1, 3, 16, 70):
        o, lse = run_decode(q, kc, vc, table, seq, S)
        check_out(o, O_ref, torch.bfloat16, f"o S={S}")
        check_lse(lse, L_ref, f"lse S={S}")
    assert attn.attn_get_device_error() == 0


@pytest.mark.parametrize("shape,splits", [(W.DECODE_S32K, (16, 17, 64)),
                                          (W.DECODE_70B_TP8, (16, 132))])
def test_decode_contiguous_32k_split_independent(shape, splits):
    """Contiguous 32k-token KV (identity table): every split count matches the
    oracle, and the results for different split counts agree."""
    q, kc, vc, table, seq = W.decode_inputs(shape, seed=1, contiguous=True)
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, table, seq, shape.scale)
    outs = []
    for S in splits:
        o, lse = run_decode(q, kc, vc, table, seq, S)
        check_out(o, O_ref, torch.bfloat16, f"o S={S}")
        check_lse(lse, L_ref, f"lse S={S}")
        outs.append(o.float().cpu().numpy())
    for o in outs[1:]:
        check_out(torch.from_numpy(o), outs[0].astype(np.float64), torch.bfloat16, "split independence")


@pytest.mark.parametrize("which", ["recommended", "other"])
def test_decode_paged_batch_every_row(which):
    """The 66-row paged batch the benchmark times (64 lengths U[1, 16384],
    2 empty rows, shuffled pages): every row and head against the oracle, at
    the benchmark's split count and at a quarter of it plus one."""
    shape = W.DECODE_PAGED_B64
    q, kc, vc, table, seq = W.decode_inputs(shape, seed=0)
    lens = seq.tolist()
    S = attn.attn_recommended_splits_ragged(len(lens), shape.h_kv, max(lens), sum(lens))
    if which == "other":
        S = S // 4 + 1
    o, lse = run_decode(q, kc, vc, table, seq, S)
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, table, seq, shape.scale)
    check_out(o, O_ref, torch.bfloat16, f"bench paged decode o S={S}")
    check_lse(lse, L_ref, f"bench paged decode lse S={S}")
    for r in (i for i, s in enumerate(lens) if s == 0):
        assert torch.all(o[r] == 0) and torch.all(torch.isneginf(lse[r]))
    assert attn.attn_get_device_error() == 0


def test_decode_paged_batch_full_size_sampled_rows():
    """Paged batch of 64 random lengths in [1, 16384] plus 2 empty rows, shuffled
    physical pages; the split count the benchmark uses; oracle on sampled rows."""
    shape = W.DECODE_PAGED_B64
    q, kc, vc, table, seq = W.decode_inputs(shape, seed=0)
    lens = seq.tolist()
    S = attn.attn_recommended_splits_ragged(len(lens), shape.h_kv, max(lens), sum(lens))
    o, lse = run_decode(q, kc, vc, table, seq, S)
    empty = [i for i, s in enumerate(lens) if s == 0]
    assert len(empty) == 2
    order = np.argsort(lens)
    rows = sorted(set(empty) | {int(order[2]), int(order[-1]), int(order[len(order) // 2])} |
                  set(np.random.default_rng(0).choice(len(lens), 5, replace=False).tolist()))
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, table, seq, shape.scale, rows=rows)
    check_out(o[rows], O_ref[rows], torch.bfloat16)
    check_lse(lse[rows], L_ref[rows])
    for r in empty:
        assert torch.all(o[r] == 0) and torch.all(torch.isneginf(lse[r]))
    # Independent of the split count.
    o2, _ = run_decode(q, kc, vc, table, seq, max(1, S // 2) + 1)
    check_out(o2[rows], O_ref[rows], torch.bfloat16, "o other S")
    assert attn.attn_get_device_error() == 0


def test_decode_late_outlier_forces_rescale():
    """The row max sits in the last page: a missing accumulator rescale would
    show (tests that put the max first pass either way)."""
    shape = W.DecodeShape("t", 32, 8, 128)
    lens = [900, 901]
    q, kc, vc, table, seq = W.decode_inputs(shape, seed=4, seq_lens=lens)
    phys = table[0, (lens[0] - 1) // 16].item()
    kc[phys, (lens[0] - 1) % 16] = (q[0].view(8, 4, 128)[:, 0, :] * 4).to(torch.bfloat16)
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, table, seq, shape.scale)
    for S in (1, 4):
        o, lse = run_decode(q, kc, vc, table, seq, S)
        check_out(o, O_ref, torch.bfloat16)
        check_lse(lse, L_ref)


def test_decode_bad_page_and_length_flagged_without_fault():
    """A table entry outside the cache reads zeros and raises a device error
    bit; a seq_len beyond the table row is clamped and flagged."""
    shape = W.DecodeShape("t", 8, 2, 128)
    lens = [40, 20]
    q, kc, vc, table, seq = W.decode_inputs(shape, seed=9, seq_lens=lens)
    attn.attn_get_device_error()  # clear
    bad = table.clone()
    bad[0, 1] = kc.shape[0] + 5
    o, lse = run_decode(q, kc, vc, bad, seq, 2)
    assert attn.attn_get_device_error() & 0x2
    assert torch.all(torch.isfinite(o.float()))
    long = seq.clone()
    long[1] = table.shape[1] * 16 + 100
    o, lse = run_decode(q, kc, vc, table, long, 2)
    assert attn.attn_get_device_error() & 0x8
    assert torch.all(torch.isfinite(o.float()))


def test_decode_output_guard_bands_untouched():
    shape = W.DecodeShape("t", 32, 8, 128)
    lens = [5, 0, 300]
    q, kc, vc, table, seq = W.decode_inputs(shape, seed=2, seq_lens=lens)
    B, h, d = q.shape
    buf = torch.full((B * h * d + 2048,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = buf[1024:1024 + B * h * d].view(B, h, d)
    attn.attn_decode_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), seq.cuda(), 4, o=o)
    torch.cuda.synchronize()
    assert torch.all(torch.isnan(buf[:1024].float())) and torch.all(torch.isnan(buf[-1024:].float()))
    O_ref, _ = oracle.decode_paged_ref(q, kc, vc, table, seq, shape.scale)
    check_out(o, O_ref, torch.bfloat16)


def test_decode_max_split_count():
    """The largest split count the API accepts (1024) on a 32k-key row: two
    pages per split, 1024 partial states per head merged by the 8-warp merge."""
    shape = W.DECODE_70B_TP8
    q, kc, vc, table, seq = W.decode_inputs(shape, seed=3, contiguous=True)
    O_ref, L_ref = oracle.decode_paged_ref(q, kc, vc, table, seq, shape.scale)
    o, lse = run_decode(q, kc, vc, table, seq, attn.ATTN_MAX_SPLITS)
    assert attn.attn_get_device_error() == 0
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)


def test_recommended_splits_reads_the_device():
    """The device form equals the pure rule with that device's SM count and
    no total length."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for B, h_kv, s in [(1, 8, 32768), (1, 1, 32768), (66, 8, 16384), (4, 8, 256)]:
        assert attn.attn_recommended_splits(B, h_kv, s, 0) == \
            attn.attn_recommended_splits_ragged(B, h_kv, s, 0, sms)

"""attn_prefill (CUDA: tcgen05 bf16 path and fp32 SIMT path) against the oracle."""
import os

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


def run(q, k, v, causal, scale):
    o, lse = attn.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    torch.cuda.synchronize()
    return o, lse


def test_single_head_fp32_T256():
    """The fp32 single-head workload, exactly as specified (seeds 0-4), full comparison."""
    shape = W.SINGLE_HEAD_T256
    for seed in range(5):
        q, k, v = W.prefill_inputs(shape, seed)
        O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, causal=False)
        o, lse = run(q, k, v, False, shape.scale)
        check_out(o, O_ref, torch.float32)
        check_lse(lse, L_ref)


@pytest.mark.parametrize("h,h_kv,d,T,causal", [
    (4, 2, 128, 300, True),
    (4, 2, 64, 257, False),
    (2, 2, 128, 129, True),
    (3, 1, 64, 64, True),
    (8, 2, 64, 1000, True),   # enough query blocks: no key split
    (1, 1, 128, 96, False),   # 3 key tiles over a cluster of 2
])
def test_fp32_path_shapes(h, h_kv, d, T, causal):
    shape = W.PrefillShape("t", h, h_kv, d, T, torch.float32, causal)
    q, k, v = W.prefill_inputs(shape, 7)
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, causal)
    o, lse = run(q, k, v, causal, shape.scale)
    check_out(o, O_ref, torch.float32)
    check_lse(lse, L_ref)


@pytest.mark.parametrize("h,h_kv,d,T,causal", [
    (8, 2, 128, 640, True),    # GQA g=4, several tiles, head pairs
    (8, 2, 128, 333, True),    # ragged tail
    (8, 2, 128, 333, False),
    (2, 2, 128, 300, True),    # g=1: one head per CTA
    (6, 2, 128, 200, False),   # g=3: one head per CTA
    (4, 2, 64, 257, True),     # d_h = 64
    (4, 4, 64, 130, False),
    (4, 1, 128, 1, True),      # T = 1
    (4, 1, 128, 127, True),
    (4, 1, 128, 128, False),
    (4, 1, 128, 129, True),
    (8, 1, 128, 300, True),    # g=8: four head pairs share a KV head
])
def test_bf16_tc_shapes(h, h_kv, d, T, causal):
    shape = W.PrefillShape("t", h, h_kv, d, T, torch.bfloat16, causal)
    q, k, v = W.prefill_inputs(shape, 11)
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, causal)
    o, lse = run(q, k, v, causal, shape.scale)
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)
    assert attn.attn_get_device_error() == 0


def test_bf16_late_outlier_forces_rescale():
    """A key near the end of the row dominates: the running max jumps late."""
    shape = W.PrefillShape("t", 4, 2, 128, 512, torch.bfloat16, False)
    q, k, v = W.prefill_inputs(shape, 3)
    k[:, 500] = (q[0, :1].float() * 3).to(torch.bfloat16)
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, False)
    o, lse = run(q, k, v, False, shape.scale)
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)


@pytest.mark.parametrize("d", [128, 64])
def test_bf16_wide_values_keep_exact_path(d):
    """Key tiles whose V holds a value beyond fp16's range (|v| >= 2^16) stay
    bf16 and use the P_hi + P_lo product; the other tiles of the same rows use
    fp16. The output matches the oracle either way."""
    shape = W.PrefillShape("t", 4, 2, d, 400, torch.bfloat16, True)
    q, k, v = W.prefill_inputs(shape, 21)
    v[0, 130, 5] = 3.0e5     # key tile 1 of KV head 0
    v[1, 300, 7] = -7.0e4    # key tile 2 of KV head 1
    v[1, 20, 0] = 65280.0    # largest bf16 below 2^16 (fits fp16): tile 0 stays fp16
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, True)
    mag, _ = oracle.attention_ref(q, k, v.abs(), shape.scale, True)  # weighted |v|
    o, lse = run(q, k, v, True, shape.scale)
    check_out(o, O_ref, torch.bfloat16, mag=mag)
    check_lse(lse, L_ref)


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_bf16_without_workspace(d, causal):
    """No scratch: every key tile takes the exact two-term bf16 P V product."""
    shape = W.PrefillShape("t", 8, 2, d, 333, torch.bfloat16, causal)
    q, k, v = W.prefill_inputs(shape, 9)
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, causal)
    o, lse = attn.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal, shape.scale, workspace=None)
    torch.cuda.synchronize()
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)


@pytest.mark.parametrize("causal", [True, False])
def test_bf16_extreme_logits(causal):
    """Logits far outside fp32's exponent range relative to the carried
    reference: one key 2^10 (log2 units) above the rest of its row (the
    reference must move to that tile's row max, which every tile takes before
    it exponentiates, or its weight overflows), and query rows whose first key
    tile lies 2^10 below zero (weights taken against that tile's own max, not
    against zero, or they all underflow)."""
    shape = W.PrefillShape("t", 4, 2, 128, 300, torch.bfloat16, causal)
    q, k, v = W.prefill_inputs(shape, 13)
    ones = torch.ones(128, dtype=torch.bfloat16)
    q[0, 270] = 8 * ones
    k[0, 260] = 8 * ones          # q.k * scale * log2(e) ~ +1045 for (head 0, row 270)
    q[2, 0:128] = -8 * ones
    k[1, 0:128] = 8 * ones        # heads 2-3, first key tile ~ -1045 for rows 0-127
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, causal)
    o, lse = run(q, k, v, causal, shape.scale)
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)
    assert attn.attn_get_device_error() == 0


def _oracle_threads():
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(8, n))


def test_gqa_T2048_causal_full():
    """The Llama-3-8B GQA layer at T = 2048, causal; every element of O and
    LSE against the oracle."""
    shape = W.GQA_T2048_CAUSAL
    q, k, v = W.prefill_inputs(shape, 0)
    O_ref, L_ref = oracle.attention_heads_ref(q, k, v, shape.scale, True, range(shape.h),
                                              threads=_oracle_threads())
    o, lse = run(q, k, v, True, shape.scale)
    check_out(o, O_ref, torch.bfloat16, "bench T2048 causal o")
    check_lse(lse, L_ref, "bench T2048 causal lse")


@pytest.mark.parametrize("causal", [True, False])
def test_more_items_than_sms_without_workspace(causal):
    """Without a workspace the persistent kernel has no work counter: its CTAs
    take the layer's items in fixed rounds (in order, then in reverse). With
    16 head pairs x 16 query blocks = 256 items on at most 152 CTAs, several
    CTAs run a second round, reversed. Every third head against the oracle,
    and the whole output bitwise against the counter-ordered call (the order
    in which CTAs take items changes nothing in an item's arithmetic)."""
    shape = W.PrefillShape("t", 32, 8, 128, 2048, torch.bfloat16, causal)
    q, k, v = W.prefill_inputs(shape, 17)
    o, lse = attn.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal, shape.scale, workspace=None)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    heads = list(range(0, shape.h, 3))  # every third head: each KV head, both heads of a pair
    O_ref, L_ref = oracle.attention_heads_ref(q, k, v, shape.scale, causal, heads,
                                              threads=_oracle_threads())
    check_out(o[heads], O_ref, torch.bfloat16, f"no-workspace T2048 {'causal' if causal else 'full'}")
    check_lse(lse[heads], L_ref)
    # With every key tile flagged wide, the call with a workspace runs the
    # same per-item arithmetic (two-term bf16 P against the bf16 V) in the
    # counter's order: the results are bitwise those of the fixed rounds.
    ws = torch.empty(attn.attn_prefill_workspace_bytes(shape.T, shape.h_kv, shape.d_h),
                     dtype=torch.uint8, device="cuda")
    v_wide = v.clone()
    v_wide[:, ::128, 0] = 1e5  # one value fp16 cannot hold in every 128-key tile
    o1, _ = attn.attn_prefill(q.cuda(), k.cuda(), v_wide.cuda(), causal, shape.scale, workspace=None)
    o2, _ = attn.attn_prefill(q.cuda(), k.cuda(), v_wide.cuda(), causal, shape.scale, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert attn.attn_get_device_error() == 0


@pytest.mark.parametrize("h,h_kv,d,T,causal", [
    (16, 4, 64, 4096, True),    # d_h = 64: four V stages; 8 x 32 = 256 items
    (6, 2, 128, 4096, True),    # g = 3: one head per item; 6 x 32 = 192 items
    (3, 1, 64, 8192, False),    # d_h = 64, one head per item, equal items; 3 x 64 = 192
])
def test_persistent_walk_other_instances(h, h_kv, d, T, causal):
    """More items than SMs in the kernel instances the benchmark layers do not
    use (d_h = 64 with four V stages; groups of odd size, one head per item):
    CTAs take several items each, so the rings, the O staging in V stages and
    the item hand-over run across items. Every element of every other head
    against the oracle."""
    shape = W.PrefillShape("t", h, h_kv, d, T, torch.bfloat16, causal)
    q, k, v = W.prefill_inputs(shape, 21)
    o, lse = run(q, k, v, causal, shape.scale)
    assert attn.attn_get_device_error() == 0
    heads = list(range(0, h, 2))
    O_ref, L_ref = oracle.attention_heads_ref(q, k, v, shape.scale, causal, heads,
                                              threads=_oracle_threads())
    check_out(o[heads], O_ref, torch.bfloat16, f"persistent h{h} kv{h_kv} d{d} T{T}")
    check_lse(lse[heads], L_ref)


def test_graph_replays_with_new_inputs():
    """A CUDA graph of one prefill call (V pass, which also zeroes the work
    counter, then the persistent kernel), replayed after new inputs are copied
    into its buffers: every replay equals an ordinary call on those inputs,
    bitwise."""
    shape = W.PrefillShape("t", 32, 8, 128, 2048, torch.bfloat16, True)
    q, k, v = (t.cuda() for t in W.prefill_inputs(shape, 5))
    ws = torch.empty(attn.attn_prefill_workspace_bytes(shape.T, shape.h_kv, shape.d_h),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((shape.h, shape.T), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        attn.attn_prefill(q, k, v, True, shape.scale, o=o, lse=lse, workspace=ws)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            attn.attn_prefill(q, k, v, True, shape.scale, o=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    for seed in (6, 7, 8):
        q2, k2, v2 = (t.cuda() for t in W.prefill_inputs(shape, seed))
        q.copy_(q2), k.copy_(k2), v.copy_(v2)
        g.replay()
        torch.cuda.synchronize()
        o_ref, lse_ref = attn.attn_prefill(q2, k2, v2, True, shape.scale)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref), seed
        assert torch.equal(lse, lse_ref), seed
    assert attn.attn_get_device_error() == 0


@pytest.mark.parametrize("shape", [W.GQA_T8192_CAUSAL, W.GQA_T8192_FULL], ids=lambda s: s.name)
def test_gqa_T8192_every_element(shape):
    """The T = 8192 layer the benchmark times (Q, K x3), causal and not:
    every element of O and LSE, all 32 heads x 8192 rows, against the oracle,
    head by head on the host cores."""
    q, k, v = W.prefill_inputs(shape, 0)
    o, lse = run(q, k, v, shape.causal, shape.scale)
    o, lse = o.cpu(), lse.cpu()
    tag = "causal" if shape.causal else "non-causal"
    # Eight heads (two KV-head groups) per oracle call bounds the host memory.
    for h0 in range(0, shape.h, 8):
        heads = list(range(h0, h0 + 8))
        O_ref, L_ref = oracle.attention_heads_ref(q, k, v, shape.scale, shape.causal, heads,
                                                  threads=_oracle_threads())
        check_out(o[h0:h0 + 8], O_ref, torch.bfloat16, f"bench T8192 {tag} o heads {h0}-{h0 + 7}")
        check_lse(lse[h0:h0 + 8], L_ref, f"bench T8192 {tag} lse heads {h0}-{h0 + 7}")
    assert attn.attn_get_device_error() == 0


@pytest.mark.parametrize("shape", [W.GQA_T8192_CAUSAL, W.GQA_T8192_FULL], ids=lambda s: s.name)
def test_gqa_T8192_sampled_rows(shape):
    """T = 8192 with logits widened (Q, K x3); oracle on sampled rows that
    include the first and last rows and rows in the last tile (a quick check;
    the every-element comparison follows)."""
    q, k, v = W.prefill_inputs(shape, 0)
    o, lse = run(q, k, v, shape.causal, shape.scale)
    rng = np.random.default_rng(1)
    rows = [0, 1, 127, 128, 4095, 8063, 8191] + rng.integers(0, shape.T, 25).tolist()
    heads = [(i * 7) % shape.h for i in range(len(rows))]
    O_ref, L_ref = oracle.attention_rows_ref(q, k, v, shape.scale, shape.causal, heads, rows)
    check_out(o[heads, rows], O_ref, torch.bfloat16)
    check_lse(lse[heads, rows], L_ref)


@pytest.mark.parametrize("causal", [True, False])
def test_widened_logits_every_row(causal):
    """Q and K x3 (logit standard deviation 9): rows move their reference
    often and many of their keys sit 6-20 log2 units below the row max, where
    the kernel's reference headroom makes the fp16 weights subnormal. Every
    row of a 12-tile sequence with a ragged tail against the oracle."""
    shape = W.PrefillShape("widened_T1500", 8, 2, 128, 1500, torch.bfloat16, causal, 3.0)
    q, k, v = W.prefill_inputs(shape, 9)
    o, lse = run(q, k, v, causal, shape.scale)
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, causal)
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)


def test_bf16_output_guard_bands_untouched():
    shape = W.PrefillShape("t", 4, 2, 128, 200, torch.bfloat16, True)
    q, k, v = W.prefill_inputs(shape, 5)
    n = q.numel()
    buf = torch.full((n + 4096,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = buf[2048:2048 + n].view_as(q)
    lbuf = torch.full((4 * 200 + 256,), float("nan"), device="cuda")
    lse = lbuf[128:128 + 800].view(4, 200)
    attn.attn_prefill(q.cuda(), k.cuda(), v.cuda(), True, shape.scale, o=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(torch.isnan(buf[:2048].float())) and torch.all(torch.isnan(buf[-2048:].float()))
    assert torch.all(torch.isnan(lbuf[:128])) and torch.all(torch.isnan(lbuf[-128:]))
    O_ref, L_ref = oracle.attention_ref(q, k, v, shape.scale, True)
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)


def test_bf16_long_sequence_sampled_rows():
    """T = 32768 (four times the benchmark length, 256 query tiles per head):
    sampled rows, including the first, the last and rows around tile edges."""
    shape = W.PrefillShape("long_T32768", 4, 1, 128, 32768, torch.bfloat16, True)
    q, k, v = W.prefill_inputs(shape, 13)
    o, lse = run(q, k, v, True, shape.scale)
    rows = [0, 1, 127, 128, 16383, 16384, 32639, 32640, 32767]
    heads = [i % shape.h for i in range(len(rows))]
    O_ref, L_ref = oracle.attention_rows_ref(q, k, v, shape.scale, True, heads, rows)
    check_out(o[heads, rows], O_ref, torch.bfloat16)
    check_lse(lse[heads, rows], L_ref)
    assert attn.attn_get_device_error() == 0

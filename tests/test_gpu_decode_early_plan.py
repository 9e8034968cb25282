"""The split-KV decode kernel's reads before its dependency wait: it reads
seq_lens and the block table early to warm L2 with its first pages, then
again after the wait for the values it computes with. Here the kernel before
it (attn_selftest_delayed_copy) lets it start at once and rewrites the
lengths or the table 50 us later, so the early reads see the old values; the
result must be that of the new ones ("Decode attention: FlashDecoding,
split-K, paged kernels", paged addressing), against the oracle. Every read of
those arrays goes to L2, so a line an early read left in L1 cannot serve the
late one."""
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


def decode_after_rewrite(q, kc, vc, table_dev, seq_dev, dst, src, S, scale, mode="plain"):
    B, h, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, h), dtype=torch.float32, device="cuda")
    if mode == "deterministic":
        pps = 8
        n = -(-table_dev.shape[1] // pps)
        ws = torch.empty(attn.attn_decode_workspace_bytes(B, h, n, d), dtype=torch.uint8, device="cuda")
    else:
        ws = torch.empty(attn.attn_decode_workspace_bytes(B, h, S, d), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    attn.attn_selftest_delayed_copy(dst, src, delay_us=50)
    if mode == "deterministic":
        attn.attn_decode_paged_deterministic(q, kc, vc, table_dev, seq_dev, pps, scale, workspace=ws,
                                             o=o, lse=lse)
    else:
        attn.attn_decode_paged(q, kc, vc, table_dev, seq_dev, S, scale, workspace=ws, o=o, lse=lse)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("S,mode", [(1, "plain"), (4, "plain"), (16, "plain"), (64, "plain"),
                                    (0, "deterministic")])
def test_lengths_rewritten_after_the_early_read(S, mode):
    shape = W.DecodeShape("early_len", 32, 8, 128)
    old = [5000, 0, 300, 17, 4096]
    new = [40, 4000, 300, 2000, 0]
    cap = [max(a, b) for a, b in zip(old, new)]
    q, kc, vc, table, _ = (t.cuda() for t in W.decode_inputs(shape, seed=23, seq_lens=cap))
    seq_dev = torch.tensor(old, dtype=torch.int32, device="cuda")
    src = torch.tensor(new, dtype=torch.int32, device="cuda")
    o, lse = decode_after_rewrite(q, kc, vc, table, seq_dev, seq_dev, src, S, shape.scale, mode)
    assert attn.attn_get_device_error() == 0
    O_ref, L_ref = oracle.decode_paged_ref(q.cpu(), kc.cpu(), vc.cpu(), table.cpu(), src.cpu(),
                                           shape.scale)
    check_out(o, O_ref, torch.bfloat16, f"early plan lengths S={S} {mode}")
    check_lse(lse, L_ref)


@pytest.mark.parametrize("S", [1, 16])
def test_table_rewritten_after_the_early_read(S):
    """Same lengths, another mapping of every row's pages (the pool's pages
    taken in reverse), rewritten after the early read."""
    shape = W.DecodeShape("early_table", 32, 8, 128)
    lens = [3000, 700, 16, 4097]
    q, kc, vc, table, seq = (t.cuda() for t in W.decode_inputs(shape, seed=29, seq_lens=lens))
    used = table >= 0
    new_table = table.clone()
    new_table[used] = table[used].flip(0)
    table_dev = table.clone()
    o, lse = decode_after_rewrite(q, kc, vc, table_dev, seq, table_dev.view(-1), new_table.view(-1),
                                  S, shape.scale)
    assert attn.attn_get_device_error() == 0
    O_ref, L_ref = oracle.decode_paged_ref(q.cpu(), kc.cpu(), vc.cpu(), new_table.cpu(), seq.cpu(),
                                           shape.scale)
    check_out(o, O_ref, torch.bfloat16, f"early plan table S={S}")
    check_lse(lse, L_ref)


def test_delayed_copy_arguments_checked():
    a = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(attn.AttnError):
        attn.attn_selftest_delayed_copy(a, a, delay_us=5000)  # above the 1000 us bound
    attn.attn_selftest_delayed_copy(a, a + 1, delay_us=0)
    torch.cuda.synchronize()
    assert torch.all(a == 1)

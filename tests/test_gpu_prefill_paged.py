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
@pytest.mark.parametrize("workspace", ["auto", None], ids=["fp16V", "bf16V"])
@pytest.mark.parametrize("decode_splits", [0, 32], ids=["decode_rows_as_tiles", "decode_rows_split"])
def test_mixed_batch_matches_oracle(h, h_kv, d, causal, workspace, decode_splits):
    """Rows of 1, 5, 77-300 queries; the one-query rows either as 1-row query
    tiles or through the split-KV decode (g = 3 has no decode kernel, so
    h = 6 keeps the tiles)."""
    if decode_splits and (h // h_kv) not in (1, 2, 4, 8):
        decode_splits = 0
    q_lens, ctx = MIXED
    q, kc, vc, table, cu, seq = paged_batch(q_lens, ctx, h, h_kv, d, 3)
    scale = 1.0 / d ** 0.5
    o, lse = attn.attn_prefill_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cu.cuda(), seq.cuda(),
                                     max(q_lens), causal, scale, workspace=workspace,
                                     decode_splits=decode_splits)
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


def v16_layout(B, max_blocks, h_kv, d):
    tiles = (max_blocks + 7) // 8
    flags_off = attn.attn_prefill_paged_workspace_bytes(B)
    v16_off = flags_off + -(-(B * h_kv * tiles * 4) // 256) * 256
    return tiles, flags_off, v16_off


def test_fp16_copy_layout_and_flags():
    """The workspace's fp16 copy holds each row's keys token-contiguously
    (row b's key t at token b * tiles * 128 + t), zeros from the row's last key
    to the end of its last 128-key tile (the slots of the last page past the
    row's length included, whatever the cache holds there), and a zero flag
    for tiles fp16 holds."""
    h, h_kv, d = 4, 2, 64
    q_lens, ctx = [5, 40, 1], [300, 40, 129]
    q, kc, vc, table, cu, seq = paged_batch(q_lens, ctx, h, h_kv, d, 6)
    B, mb = len(ctx), table.shape[1]
    n = attn.attn_prefill_paged_workspace_bytes(B, mb, h_kv, d, v16=True)
    ws = torch.full((n,), 0x7f, dtype=torch.uint8, device="cuda")  # fp16 NaN pattern if left unwritten
    attn.attn_prefill_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cu.cuda(), seq.cuda(),
                            max(q_lens), True, 1.0 / d ** 0.5, workspace=ws)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    tiles, flags_off, v16_off = v16_layout(B, mb, h_kv, d)
    flags = ws[flags_off:flags_off + B * h_kv * tiles * 4].view(torch.int32).view(B, h_kv, tiles).cpu()
    v16 = ws[v16_off:].view(torch.float16).view(B, tiles * 128, h_kv, d).cpu()
    for b in range(B):
        pages = -(-ctx[b] // 16)
        used_tiles = -(-pages // 8)
        assert (flags[b, :, :used_tiles] == 0).all()
        keys = torch.stack([vc[table[b, t // 16], t % 16] for t in range(ctx[b])])
        assert torch.equal(v16[b, :ctx[b]], keys.to(torch.float16))
        assert (v16[b, ctx[b]:used_tiles * 128] == 0).all()


@pytest.mark.parametrize("causal", [True, False])
def test_wide_v_tiles_match_oracle(causal):
    """Pages holding values fp16 cannot carry (|v| >= 2^16) flag their 128-key
    tile, which then takes the bf16 P_hi + P_lo path; the other tiles of the
    same rows take fp16 P. Outputs match the oracle either way."""
    h, h_kv, d = 8, 2, 128
    q_lens, ctx = [200, 64, 1], [1000, 600, 300]
    q, kc, vc, table, cu, seq = paged_batch(q_lens, ctx, h, h_kv, d, 7)
    vc = vc.clone()
    vc[table[0, 3], 5, 1, 7] = 3.0e5      # row 0, tile 0, head 1
    vc[table[1, 20], 0, 0, 100] = -7.0e4  # row 1, tile 2, head 0
    vc[table[2, 9], 2, 1, 0] = 65280.0    # largest bf16 below 2^16, fits fp16: tile stays fp16
    B, mb = len(ctx), table.shape[1]
    n = attn.attn_prefill_paged_workspace_bytes(B, mb, h_kv, d, v16=True)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    scale = 1.0 / d ** 0.5
    o, lse = attn.attn_prefill_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cu.cuda(), seq.cuda(),
                                     max(q_lens), causal, scale, workspace=ws)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    tiles, flags_off, _ = v16_layout(B, mb, h_kv, d)
    flags = ws[flags_off:flags_off + B * h_kv * tiles * 4].view(torch.int32).view(B, h_kv, tiles).cpu()
    wide = {(b, k, t) for b in range(B) for k in range(h_kv) for t in range(-(-ctx[b] // 128))
            if flags[b, k, t] != 0}
    assert wide == {(0, 1, 0), (1, 0, 2)}
    O_ref, L_ref = oracle.prefill_paged_ref(q, kc, vc, table, cu, seq, scale, causal)
    mag, _ = oracle.prefill_paged_ref(q, kc, vc.abs(), table, cu, seq, scale, causal)  # weighted |v|
    check_out(o, O_ref, torch.bfloat16, mag=mag)
    check_lse(lse, L_ref)


@pytest.mark.parametrize("workspace", ["auto", None], ids=["fp16V", "bf16V"])
def test_row_beyond_capacity_is_skipped(workspace):
    """A row with more queries than its block-table row can hold keys is
    skipped (outputs untouched) and flagged; the other rows are exact."""
    h, h_kv, d = 4, 2, 64
    q, kc, vc, table, cu, seq = paged_batch([40, 3, 1], [300, 20, 300], h, h_kv, d, 8)
    cap = table.shape[1] * 16                      # 19 pages -> 304 keys
    q_lens = [40, 3, cap + 6]
    cu = torch.zeros(4, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int32), 0)
    q = W.normal((int(cu[-1]), h, d), 81, torch.bfloat16)
    scale = 1.0 / d ** 0.5
    o = torch.full((int(cu[-1]), h, d), 7.0, dtype=torch.bfloat16, device="cuda")
    attn.attn_prefill_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cu.cuda(), seq.cuda(),
                            max(q_lens), True, scale, workspace=workspace, o=o)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() & 0x8  # ATTN_DEVERR_BAD_SEQ_LEN
    assert (o[int(cu[2]):] == 7.0).all()
    O_ref, _ = oracle.prefill_paged_ref(q[:int(cu[2])], kc, vc, table[:2], cu[:3], seq[:2], scale, True)
    check_out(o[:int(cu[2])], O_ref, torch.bfloat16)


@pytest.mark.parametrize("workspace", ["auto", None], ids=["fp16V", "bf16V"])
def test_widened_logits_mixed_batch(workspace):
    """Q and K x3 (logit standard deviation 9) through the paged kernel:
    frequent reference moves and fp16-subnormal weights, every row checked."""
    q_lens, ctx = MIXED
    h, h_kv, d = 8, 2, 128
    q, kc, vc, table, cu, seq = paged_batch(q_lens, ctx, h, h_kv, d, 10)
    q = (q.float() * 3).to(torch.bfloat16)
    kc = (kc.float() * 3).to(torch.bfloat16)
    scale = 1.0 / d ** 0.5
    o, lse = attn.attn_prefill_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cu.cuda(), seq.cuda(),
                                     max(q_lens), True, scale, workspace=workspace)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    O_ref, L_ref = oracle.prefill_paged_ref(q, kc, vc, table, cu, seq, scale, True)
    check_out(o, O_ref, torch.bfloat16)
    check_lse(lse, L_ref)


@pytest.mark.parametrize("decode_splits", [1, 5, 32])
@pytest.mark.parametrize("workspace", ["auto", None], ids=["fp16V", "bf16V"])
def test_decode_heavy_mixed_batch(decode_splits, workspace):
    """The shape of a serving step: 3 chunked-prefill rows and 40 decode rows
    over 1-5000 keys (lengths crossing page edges), every row against the
    oracle, whatever the decode rows' split bound."""
    h, h_kv, d = 32, 8, 128
    g = torch.Generator().manual_seed(17)
    dec_ctx = torch.randint(1, 5000, (40,), generator=g).tolist()
    dec_ctx[:4] = [1, 15, 16, 17]
    q_lens = [300, 128, 1] + [1] * 40
    ctx = [1000, 128, 4097] + dec_ctx
    q, kc, vc, table, cu, seq = paged_batch(q_lens, ctx, h, h_kv, d, 19)
    scale = 1.0 / d ** 0.5
    o, lse = attn.attn_prefill_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cu.cuda(), seq.cuda(),
                                     max(q_lens), True, scale, workspace=workspace,
                                     decode_splits=decode_splits)
    torch.cuda.synchronize()
    assert attn.attn_get_device_error() == 0
    O_ref, L_ref = oracle.prefill_paged_ref(q, kc, vc, table, cu, seq, scale, True)
    check_out(o, O_ref, torch.bfloat16, f"mixed decode_splits={decode_splits}")
    check_lse(lse, L_ref)


def test_caller_workspace_with_decode_part():
    """A caller's workspace holding the decode part and the fp16-V form."""
    h, h_kv, d = 8, 2, 128
    q_lens, ctx = MIXED
    q, kc, vc, table, cu, seq = paged_batch(q_lens, ctx, h, h_kv, d, 5)
    B, mb = len(ctx), table.shape[1]
    n = (attn.attn_prefill_paged_decode_workspace_bytes(B, h, 7, d) +
         attn.attn_prefill_paged_workspace_bytes(B, mb, h_kv, d, v16=True))
    ws = torch.full((n,), 0x7f, dtype=torch.uint8, device="cuda")
    o, lse = attn.attn_prefill_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cu.cuda(), seq.cuda(),
                                     max(q_lens), True, 1.0 / d ** 0.5, workspace=ws, decode_splits=7)
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.prefill_paged_ref(q, kc, vc, table, cu, seq, 1.0 / d ** 0.5, True)
    check_out(o, O_ref, torch.bfloat16, "caller workspace with decode part")
    check_lse(lse, L_ref)
    with pytest.raises(attn.AttnError):  # one byte short of the decode part plus the small form
        small = attn.attn_prefill_paged_decode_workspace_bytes(B, h, 7, d) + attn.attn_prefill_paged_workspace_bytes(B)
        attn.attn_prefill_paged(q.cuda(), kc.cuda(), vc.cuda(), table.cuda(), cu.cuda(), seq.cuda(),
                                max(q_lens), True, workspace=ws[:small - 1], decode_splits=7)

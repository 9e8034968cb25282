"""The C-ABI library builds, loads and exports what include/attn.h declares;
host-only logic (split plan, split sizing, workspace size, argument
validation) checked without a GPU."""
import ctypes
import os
import re

import pytest

import online_softmax_attn_gb300 as attn
from online_softmax_attn_gb300 import build as attn_build
from pins import golden

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    attn_build.build()
    return attn.library()


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(attn_\w+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "attn_prefill" in names and "attn_decode_paged" in names and "attn_merge_states" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_exports_nothing_undeclared(lib):
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", attn_build.LIB_PATH],
                         capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T attn_" in l}
    assert exported == set(declared_functions())


def test_status_strings(lib):
    for s in range(6):
        assert attn.attn_status_string(s) != "unknown status"
    assert attn.attn_status_string(99) == "unknown status"


def test_split_plan_matches_pages():
    g = golden("split_sizing.json")
    for seg in g["segments"]:
        n, pps = attn.attn_decode_split_plan(seg["seq_len"], seg["max_splits"])
        assert n == seg["active"]
        if "pages_per_split" in seg:
            assert pps == seg["pages_per_split"]
            first = (0, pps * 16 - 1)
            last = ((n - 1) * pps * 16, seg["seq_len"] - 1)
            assert list(first) == seg["first_split_keys"]
            assert list(last) == seg["last_split_keys"]


def test_split_plan_covers_every_page_once():
    for s in [0, 1, 15, 16, 17, 255, 256, 257, 2560, 32768, 16384]:
        for S in [1, 2, 3, 16, 17, 64, 132, 1024]:
            n, pps = attn.attn_decode_split_plan(s, S)
            pages = (s + 15) // 16
            assert n <= S
            if pages == 0:
                assert n == 0
                continue
            covered = [p for i in range(n) for p in range(i * pps, min((i + 1) * pps, pages))]
            assert covered == list(range(pages))
            assert all(i * pps < pages for i in range(n))  # every active split has work


def test_workspace_bytes_match_pages():
    g = golden("split_sizing.json")
    p = g["partial_bytes_B1_h32"]
    assert attn.attn_decode_workspace_bytes(p["B"], p["h"], p["S"], p["d_h"]) == p["bytes"]
    per = g["partial_bytes_per_token_head"]
    assert attn.attn_decode_workspace_bytes(1, 1, per["S"], per["d_h"]) >= per["bytes"]
    assert attn.attn_decode_workspace_bytes(0, 1, 1, 128) == 0


def test_first_wave_split_count():
    g = golden("split_sizing.json")
    for case in g["first_wave_splits"]:
        # G_2D = B * h_kv at B = 1
        assert attn.attn_recommended_splits_ragged(1, case["g2d"], 1 << 20, 0, case["n_sm"]) == case["splits"]


def test_recommended_splits_ragged_batch_balances():
    s = attn.attn_recommended_splits_ragged(66, 8, 16384, 64 * 8192, 152)
    assert s >= 2
    # Longest row's split is at most a quarter of the mean work per SM.
    pages_max = 16384 // 16
    mean_per_sm = (64 * 8192 // 16) * 8 / 152
    assert pages_max / s <= mean_per_sm / 4 + 1


def test_invalid_arguments_rejected_before_launch(lib):
    P = ctypes.c_void_p
    dummy = P(256)  # never dereferenced: validation fails first
    S = attn.attn_status_string
    bad = attn.ATTN_ERR_INVALID_ARG
    # h not a multiple of h_kv
    assert lib.attn_prefill(dummy, dummy, dummy, dummy, None, 64, 6, 4, 128, 1, 0.1, 1, None, 0, None) == bad
    # negative T, non-positive scale, NaN scale
    assert lib.attn_prefill(dummy, dummy, dummy, dummy, None, -1, 4, 4, 128, 1, 0.1, 1, None, 0, None) == bad
    assert lib.attn_prefill(dummy, dummy, dummy, dummy, None, 64, 4, 4, 128, 1, 0.0, 1, None, 0, None) == bad
    assert lib.attn_prefill(dummy, dummy, dummy, dummy, None, 64, 4, 4, 128, 1, float("nan"), 1, None, 0, None) == bad
    # misaligned pointer
    assert lib.attn_prefill(P(258), dummy, dummy, dummy, None, 64, 4, 4, 128, 1, 0.1, 1, None, 0, None) == bad
    # unsupported head size
    assert lib.attn_prefill(dummy, dummy, dummy, dummy, None, 64, 4, 4, 96, 1, 0.1, 1, None, 0, None) == \
        attn.ATTN_ERR_UNSUPPORTED
    # T = 0 is a no-op
    assert lib.attn_prefill(None, None, None, None, None, 0, 4, 4, 128, 1, 0.1, 1, None, 0, None) == 0
    # prefill workspace: misaligned, or smaller than attn_prefill_workspace_bytes
    need = lib.attn_prefill_workspace_bytes(64, 4, 128, 1)
    assert lib.attn_prefill(dummy, dummy, dummy, dummy, None, 64, 4, 4, 128, 1, 0.1, 1, P(272), need,
                            None) == bad
    assert lib.attn_prefill(dummy, dummy, dummy, dummy, None, 64, 4, 4, 128, 1, 0.1, 1, dummy, need - 1,
                            None) == bad
    # decode: workspace too small, page size, group size, split count
    args = [dummy, dummy, dummy, dummy, dummy, 2, 32, 8, 128, 16, 100, 10, 16, 0.1, dummy, 16,
            dummy, None, None]
    assert lib.attn_decode_paged(*args) == bad
    a2 = list(args); a2[9] = 32
    assert lib.attn_decode_paged(*a2) == attn.ATTN_ERR_UNSUPPORTED
    a3 = list(args); a3[6] = 3
    assert lib.attn_decode_paged(*a3) == bad  # 32 % 3 != 0
    a4 = list(args); a4[12] = 0
    assert lib.attn_decode_paged(*a4) == bad
    a5 = list(args); a5[12] = attn.ATTN_MAX_SPLITS + 1
    assert lib.attn_decode_paged(*a5) == bad
    a6 = list(args); a6[5] = 0
    assert lib.attn_decode_paged(*a6) == 0  # B = 0 is a no-op
    # merge: bad dtype, bad d_h, rows 0
    assert lib.attn_merge_states(dummy, dummy, dummy, None, 4, 2, 128, dummy, None, 7, None) == bad
    assert lib.attn_merge_states(dummy, dummy, dummy, None, 4, 2, 80, dummy, None, 1, None) == \
        attn.ATTN_ERR_UNSUPPORTED
    assert lib.attn_merge_states(None, None, None, None, 0, 2, 128, None, None, 1, None) == 0
    assert S(bad) == "invalid argument"


def test_prefill_host_scratch_bytes(lib):
    """Device copies of q, k, v, o, lse, then the prefill workspace, each region 256-byte aligned."""
    lib.attn_prefill_host_scratch_bytes.argtypes = [ctypes.c_int] * 5
    lib.attn_prefill_host_scratch_bytes.restype = ctypes.c_size_t
    lib.attn_prefill_workspace_bytes.argtypes = [ctypes.c_int] * 4
    lib.attn_prefill_workspace_bytes.restype = ctypes.c_size_t
    f = lib.attn_prefill_host_scratch_bytes
    a = lambda x: -(-x // 256) * 256
    T, h, h_kv, d = 333, 8, 2, 64
    qb, kb, lb = h * T * d * 2, h_kv * T * d * 2, h * T * 4
    ws = lib.attn_prefill_workspace_bytes(T, h_kv, d, 1)
    assert ws == 85248 + 256 + 256  # V copy, tile flags, work counter
    assert f(T, h, h_kv, d, 1) == a(qb) + 2 * a(kb) + a(qb) + a(lb) + ws
    assert f(256, 1, 1, 64, 0) == 2 * a(256 * 64 * 4) + 2 * a(256 * 64 * 4) + a(256 * 4)  # fp32: no workspace
    assert f(0, h, h_kv, d, 1) == 0
    none = (1 << 64) - 1
    for bad in [(-1, 8, 2, 64, 1), (64, 8, 3, 64, 1), (64, 8, 2, 96, 1), (64, 8, 2, 64, 7), (64, 0, 1, 64, 1)]:
        assert f(*bad) == none, bad


def test_prefill_paged_v16_workspace_bytes(lib):
    """Tile offsets, then flags [B, h_kv, ceil(max_blocks/8)] int32, then the fp16 V copy
    [B, ceil(max_blocks/8) * 128, h_kv, d_h], each region 256-byte aligned."""
    lib.attn_prefill_paged_v16_workspace_bytes.argtypes = [ctypes.c_int] * 4
    lib.attn_prefill_paged_v16_workspace_bytes.restype = ctypes.c_size_t
    f = lib.attn_prefill_paged_v16_workspace_bytes
    assert f(8, 512, 8, 128) == 256 + 16384 + 8 * 64 * 128 * 8 * 128 * 2
    # 3 rows, 19 pages -> 3 tiles per row: offsets 256, flags 3*2*3*4=72 -> 256, copy 3*384*2*64*2
    assert f(3, 19, 2, 64) == 256 + 256 + 3 * 384 * 2 * 64 * 2
    assert f(0, 19, 2, 64) == 256 + 0 + 0
    for bad in [(-1, 19, 2, 64), (3, 0, 2, 64), (3, 19, 0, 64), (3, 19, 2, 96), (3, 1 << 27, 2, 64)]:
        assert f(*bad) == 0, bad
    # the copy's token index must fit int32: 2^13 rows x 2^11 tiles x 128 = 2^31
    assert f(1 << 13, 1 << 14, 1, 64) == 0
    assert f((1 << 13) - 1, 1 << 14, 1, 64) != 0


def test_prefill_workspace_bytes(lib):
    """fp16 copy of V (256-byte aligned), one int per (KV head, 128-key tile),
    then 256 bytes for the work counter."""
    assert lib.attn_prefill_workspace_bytes(8192, 8, 128, 1) == 8 * 8192 * 128 * 2 + 2048 + 256  # 8 x 64 ints
    assert lib.attn_prefill_workspace_bytes(333, 2, 64, 1) == 85248 + 256 + 256  # 2*333*64*2, then 6 ints
    assert lib.attn_prefill_workspace_bytes(8192, 8, 128, 0) == 0  # fp32 SIMT path: none
    assert lib.attn_prefill_workspace_bytes(0, 8, 128, 1) == 0
    none = (1 << 64) - 1
    assert lib.attn_prefill_workspace_bytes(-1, 8, 128, 1) == none
    assert lib.attn_prefill_workspace_bytes(64, 0, 128, 1) == none
    assert lib.attn_prefill_workspace_bytes(64, 8, 96, 1) == none
    assert lib.attn_prefill_workspace_bytes(64, 8, 128, 7) == none


def test_recommended_splits_uniform_rows_and_minimum_work():
    """Rows of one length take the first-wave count; no split of the longest
    row gets fewer than 32 pages; the ragged rule needs a row well above the mean."""
    assert attn.attn_recommended_splits_ragged(1, 8, 32768, 32768, 152) == 19   # ceil(152 / 8)
    assert attn.attn_recommended_splits_ragged(1, 1, 32768, 32768, 152) == 64   # 2048 pages / 32
    assert attn.attn_recommended_splits_ragged(1, 8, 256, 256, 152) == 1        # 16 pages: one split
    assert attn.attn_recommended_splits_ragged(4, 8, 8192, 4 * 8192, 152) == 5  # uniform batch: ceil(152 / 32)
    # ragged: one long row among short ones raises the count above the first wave
    assert attn.attn_recommended_splits_ragged(8, 8, 16384, 16384 + 7 * 512, 152) > 3


def test_merge_lse_pair_arguments(lib):
    P = ctypes.c_void_p
    dummy = P(256)
    bad = attn.ATTN_ERR_INVALID_ARG
    lib.attn_merge_lse_pair.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                                        ctypes.c_int, P]
    ok_args = [dummy, P(4096), P(512), P(8192), 4, 128, 1, P(1024), P(12288), 1, None]
    # rows == 0 is a no-op even with NULL pointers
    assert lib.attn_merge_lse_pair(None, None, None, None, 0, 128, 1, None, None, 1, None) == 0
    a = list(ok_args); a[4] = -1
    assert lib.attn_merge_lse_pair(*a) == bad
    a = list(ok_args); a[5] = 96
    assert lib.attn_merge_lse_pair(*a) == attn.ATTN_ERR_UNSUPPORTED
    a = list(ok_args); a[6] = 7
    assert lib.attn_merge_lse_pair(*a) == bad
    a = list(ok_args); a[0] = P(264)  # o_a not 16-byte aligned
    assert lib.attn_merge_lse_pair(*a) == bad
    a = list(ok_args); a[2] = None
    assert lib.attn_merge_lse_pair(*a) == bad
    a = list(ok_args); a[8] = P(4100)  # output LSE overlaps lse_a
    assert lib.attn_merge_lse_pair(*a) == bad


def test_decode_deterministic_arguments(lib):
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_decode_paged_deterministic.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P,
                                                    ctypes.c_size_t, P, P, P]
    d = P(256)
    bad = attn.ATTN_ERR_INVALID_ARG
    base = [d, d, d, d, d, 2, 32, 8, 128, 16, 100, 64, 4, 16, 0.1, d, 1 << 30, d, None, None]
    # 4 splits x 16 pages cover a 64-page table; arguments otherwise valid up to the launch
    a = list(base); a[13] = 0                   # pages_per_split < 1
    assert lib.attn_decode_paged_deterministic(*a) == bad
    a = list(base); a[12] = 3                   # 3 x 16 < 64 pages: a row would not fit
    assert lib.attn_decode_paged_deterministic(*a) == bad
    a = list(base); a[5] = 0                    # B = 0 is a no-op
    assert lib.attn_decode_paged_deterministic(*a) == 0


def test_decode_adaptive_workspace(lib):
    """The adaptive decode needs the partials for max_splits plus 256 bytes."""
    need = attn.attn_decode_workspace_bytes(3, 32, 16, 128)
    assert attn.attn_decode_adaptive_workspace_bytes(3, 32, 16, 128) == need + 256
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_decode_paged_adaptive.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, P,
                                               ctypes.c_size_t, P, P, P]
    d = P(256)
    assert lib.attn_decode_paged_adaptive(d, d, d, d, d, 3, 32, 8, 128, 16, 100, 64, 16, 0.1, d, need,
                                          d, None, None) == attn.ATTN_ERR_INVALID_ARG


def test_selftest_wait_timeout_arguments(lib):
    """The limit is checked on the host before any launch."""
    lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint, ctypes.c_void_p]
    lib.attn_selftest_wait_timeout.restype = ctypes.c_int
    assert lib.attn_selftest_wait_timeout(0, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_selftest_wait_timeout(1000001, None) == attn.ATTN_ERR_INVALID_ARG


def test_version(lib):
    lib.attn_version.restype = ctypes.c_int
    assert lib.attn_version() == 301


def test_prefill_host_checks_limits_before_queueing(lib):
    """attn_prefill_host refuses a bf16 layer with more than 65535 query tiles
    of 128, and a pipe with a missing member, before it touches any pointer or
    queues anything: the pointers here are placeholders no GPU could use, and
    no GPU is needed."""
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    f = lib.attn_prefill_host
    f.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I, P, S, P, P]
    f.restype = I
    fake = ctypes.c_void_p(4096)
    big_T = 65536 * 128
    st = f(fake, fake, fake, fake, None, big_T, 1, 1, 64, 1, 0.125, attn.ATTN_DTYPE_BF16, 1, fake,
           ctypes.c_size_t(-1).value, None, None)
    assert st == attn.ATTN_ERR_UNSUPPORTED
    pipe = attn.HostPipe()
    pipe.copy_in, pipe.copy_out = 4096, 8192
    for i in range(attn.ATTN_HOST_PIPE_EVENTS - 1):
        pipe.events[i] = 4096 * (i + 3)
    st = f(fake, fake, fake, fake, None, 256, 1, 1, 64, 1, 0.125, attn.ATTN_DTYPE_BF16, 1, fake,
           ctypes.c_size_t(-1).value, ctypes.byref(pipe), None)
    assert st == attn.ATTN_ERR_INVALID_ARG
    pipe.copy_out = pipe.copy_in
    pipe.events[attn.ATTN_HOST_PIPE_EVENTS - 1] = 4096 * 99
    st = f(fake, fake, fake, fake, None, 256, 1, 1, 64, 1, 0.125, attn.ATTN_DTYPE_BF16, 1, fake,
           ctypes.c_size_t(-1).value, ctypes.byref(pipe), None)
    assert st == attn.ATTN_ERR_INVALID_ARG


def declared_signatures():
    """Parameter names of every function declared in include/*.h."""
    sigs = {}
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for name, params in re.findall(r"\b(attn_\w+)\s*\(([^)]*)\)\s*;", src):
            names = [] if params.strip() in ("", "void") else \
                [re.findall(r"(\w+)\s*$", p.strip())[0] for p in params.split(",")]
            sigs[name] = names
    return sigs


# The core calls' minimal signatures, and what the header adds to them (each
# addition explained in the header's "Signatures" note).
MINIMAL = {
    "attn_prefill": ["q", "k", "v", "o", "lse", "T", "h", "h_kv", "d_h", "causal", "scale", "dtype",
                     "stream"],
    "attn_decode_paged": ["q", "k_cache", "v_cache", "block_table", "seq_lens", "B", "h", "h_kv", "d_h",
                          "page_size", "max_blocks_per_seq", "num_splits", "scale", "workspace",
                          "workspace_bytes", "o", "lse", "stream"],
    "attn_merge_states": ["o_part", "m_part", "l_part", "n_active", "rows", "num_splits", "d_h", "o", "lse",
                          "out_dtype", "stream"],
    "attn_decode_workspace_bytes": ["B", "h", "num_splits", "d_h"],
    "attn_recommended_splits": ["B", "h_kv", "max_seq_len", "device"],
    "attn_get_last_device_error": ["stream"],
    "attn_status_string": ["status"],
}
ADDED = {"attn_prefill": ["workspace", "workspace_bytes"], "attn_decode_paged": ["num_blocks"]}


def test_core_signatures_are_the_minimal_ones_plus_documented_additions():
    sigs = declared_signatures()
    for name, minimal in MINIMAL.items():
        assert name in sigs, name
        got = sigs[name]
        extra = ADDED.get(name, [])
        assert sorted(set(got) - set(minimal)) == sorted(extra), (name, got)
        # the minimal parameters keep their order
        assert [p for p in got if p not in extra] == minimal, (name, got)
    # The header's note names exactly these additions, one entry per call:
    # "<call>   <param>, <param> (after ...)".
    note = open(os.path.join(ROOT, "include", "attn.h")).read().replace("\n *", " ")
    for name, extra in ADDED.items():
        m = re.search(rf"{name}\s+([\w, ]+?)\s*\(after", note)
        assert m, name
        assert [x.strip() for x in m.group(1).split(",")] == extra, (name, m.group(1))


def test_device_error_bits_match_the_header():
    """The binding's ATTN_DEVERR_* constants are the header's #defines."""
    import re

    import online_softmax_attn_gb300 as attn

    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    bits = dict(re.findall(r"#define (ATTN_DEVERR_\w+) (0x[0-9a-fA-F]+)u", text))
    assert bits, "no ATTN_DEVERR_* bits in attn.h"
    for name, value in bits.items():
        assert getattr(attn, name) == int(value, 16), name
    assert set(attn.DEVERR_NAMES) == {int(v, 16) for v in bits.values()}


def test_prefill_stall_selftest_is_debug_only(lib):
    """The release library refuses the abort-path self-test without touching
    the device."""
    lib.attn_selftest_prefill_stall.argtypes = [ctypes.c_int]
    lib.attn_selftest_prefill_stall.restype = ctypes.c_int
    assert lib.attn_selftest_prefill_stall(2) == 2  # ATTN_ERR_UNSUPPORTED
    assert lib.attn_selftest_prefill_stall(-1) == 2

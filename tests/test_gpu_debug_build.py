"""The small-shape GPU cases of the other test modules, run once more against
the -DATTN_DEBUG build of the library. In that build every kernel checks the
indices of its global stores and the shared-memory offsets it computes; a
failed check sets ATTN_DEVERR_DEBUG_INDEX in the device error word and skips
the access (nothing traps). Each case must still match the oracle, as in its
own module, and leave no error bit set beyond those the case itself expects
and clears.

The debug library is built here, on first use, into the package directory
(libattn_gb300_debug.so), and swapped into the Python binding for this module
only."""
import itertools

import pytest
import torch

import online_softmax_attn_gb300 as attn
import test_gpu_decode as D
import test_gpu_decode_adaptive as DA
import test_gpu_decode_deterministic as DD
import test_gpu_merge as M
import test_gpu_merge_pair as MP
import test_gpu_nonfinite as NF
import test_gpu_prefill as P
import test_gpu_prefill_paged as PP

pytestmark = pytest.mark.gpu

# (module, test function): every parameter combination of each runs. Only
# small shapes: the full-size benchmark checks have their own modules.
CASES = [
    (P, "test_single_head_fp32_T256"),
    (P, "test_fp32_path_shapes"),
    (P, "test_bf16_tc_shapes"),
    (P, "test_bf16_late_outlier_forces_rescale"),
    (P, "test_bf16_wide_values_keep_exact_path"),
    (P, "test_bf16_without_workspace"),
    (P, "test_bf16_extreme_logits"),
    (P, "test_bf16_output_guard_bands_untouched"),
    (D, "test_decode_small_edges"),
    (D, "test_decode_late_outlier_forces_rescale"),
    (D, "test_decode_bad_page_and_length_flagged_without_fault"),
    (D, "test_decode_output_guard_bands_untouched"),
    (D, "test_decode_max_split_count"),
    (DA, "test_adaptive_matches_oracle_and_host_rule"),
    (DD, "test_deterministic_empty_and_short_rows"),
    (PP, "test_mixed_batch_matches_oracle"),
    (PP, "test_chunked_prefill_equals_whole_row"),
    (PP, "test_bad_page_sets_error_without_fault"),
    (PP, "test_wide_v_tiles_match_oracle"),
    (PP, "test_row_beyond_capacity_is_skipped"),
    (PP, "test_decode_heavy_mixed_batch"),
    (M, "test_merge_random_partials"),
    (M, "test_merge_all_active_when_no_counts"),
    (M, "test_merge_empty_rows_give_zero_not_nan"),
    (MP, "test_pair_merge_matches_oracle"),
    (NF, "test_prefill_nan_in_k"),
    (NF, "test_prefill_nonfinite_v"),
    (NF, "test_prefill_nonfinite_v_inside_causal_tile"),
    (NF, "test_prefill_fp32_nonfinite"),
    (NF, "test_paged_prefill_nonfinite"),
    (NF, "test_decode_nonfinite"),
    (NF, "test_merge_states_nan_partials"),
    (NF, "test_merge_pair_nan_side"),
]


def _combinations(fn):
    """Keyword sets of a test function's stacked parametrize marks."""
    axes = []
    for mark in getattr(fn, "pytestmark", []):
        if mark.name != "parametrize":
            continue
        names = mark.args[0]
        names = [n.strip() for n in names.split(",")] if isinstance(names, str) else list(names)
        values = []
        for v in mark.args[1]:
            v = v.values if hasattr(v, "values") else v  # pytest.param
            values.append(dict(zip(names, v if len(names) > 1 else (v,))))
        axes.append(values)
    out = []
    for combo in itertools.product(*axes):
        kw = {}
        for part in combo:
            kw.update(part)
        out.append(kw)
    return out


def _case_list():
    out = []
    for mod, name in CASES:
        fn = getattr(mod, name)
        for i, kw in enumerate(_combinations(fn)):
            out.append(pytest.param(fn, kw, id=f"{mod.__name__}.{name}[{i}]"))
    return out


@pytest.fixture(scope="module", autouse=True)
def debug_library():
    from online_softmax_attn_gb300 import build

    path = build.build(debug=True)
    saved_lib, saved_path = attn._lib, attn.LIB_PATH
    attn._lib, attn.LIB_PATH = None, path
    try:
        lib = attn.library()
        assert lib._name == path
        attn.attn_get_device_error()  # start from a clear error word
        yield lib
    finally:
        attn._lib, attn.LIB_PATH = saved_lib, saved_path


@pytest.mark.parametrize("fn,kw", _case_list())
def test_case_under_debug_checks(fn, kw):
    fn(**kw)
    bits = attn.attn_get_device_error()
    assert bits & attn.ATTN_DEVERR_DEBUG_INDEX == 0, f"debug index check failed (bits {bits:#x})"
    assert bits == 0, f"device error bits {bits:#x}"


def test_debug_build_is_the_library_in_use(debug_library):
    assert attn.library() is debug_library
    assert attn.library()._name.endswith("libattn_gb300_debug.so")


@pytest.mark.parametrize("h,T,key_tile", [
    (8, 1024, 2),     # 32 items: one per CTA, the stall in its only item
    (32, 4096, 40),   # 512 items: the stall in a CTA's second or later item
])
def test_prefill_abort_path_after_a_stalled_load(debug_library, h, T, key_tile):
    """The bf16 prefill's abort path, without a fault: with one key tile's K
    never requested in every CTA, the MMA warp's bounded wait gives up after
    2 s and raises ATTN_DEVERR_WAIT_TIMEOUT; every role stops (including roles
    waiting for the next item or for a stage), drains what it issued, frees
    tensor memory and exits. The next call on the same context, with the stall
    off, is exact."""
    import oracle
    import workloads as W
    from parity import check_lse, check_out

    shape = W.PrefillShape("t", h, h // 4, 128, T, torch.bfloat16, True)
    q, k, v = W.prefill_inputs(shape, 31)
    attn.attn_selftest_prefill_stall(key_tile)
    try:
        attn.attn_prefill(q.cuda(), k.cuda(), v.cuda(), True, shape.scale)
        bits = attn.attn_get_device_error()
    finally:
        attn.attn_selftest_prefill_stall(-1)
    assert bits & attn.ATTN_DEVERR_WAIT_TIMEOUT, f"bits {bits:#x}"
    assert bits & attn.ATTN_DEVERR_DEBUG_INDEX == 0
    o, lse = P.run(q, k, v, True, shape.scale)
    assert attn.attn_get_device_error() == 0
    heads = list(range(0, h, max(1, h // 8)))
    O_ref, L_ref = oracle.attention_heads_ref(q, k, v, shape.scale, True, heads, threads=8)
    check_out(o[heads], O_ref, torch.bfloat16, "after the abort")
    check_lse(lse[heads], L_ref)

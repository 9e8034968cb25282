"""Float64 CPU oracle for exact scaled dot-product attention.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the tests, the smoke check
of the CUDA library and the benchmark's CPU-baseline / reference legs may import
this package. It shares no code with the CUDA path and imports nothing from it.

Contents (each function cites the passage it follows):

* ``attention_ref``        - the definition: materialise S = scale * Q K^T per
                             head, mask by index sets, safe (max-shifted)
                             softmax, P V.  Returns O and the natural-log LSE.
* ``attention_rows_ref``   - the same definition evaluated for chosen rows only.
* ``attention_heads_ref``  - the same definition for chosen query heads, every
                             row, each row's allowed keys taken as a prefix
                             slice (whole long layers, head by head).
* ``decode_paged_ref``     - the definition for one query token per row over
                             keys gathered through a page table.
* ``block_state`` / ``merge_states`` / ``finalize_state`` - the (m, l, a)
                             partial-state algebra and its two-state merge.
* ``online_softmax_attention`` - the streaming recurrence over key blocks.
* ``merge_partials_ref``   - the N-way reduce of split partial states.
* ``merge_lse_pair_ref``   - the symmetric (O, LSE) merge of two results.
* ``prefill_paged_ref``    - variable-length query rows over a paged cache
                             (queries are a row's last key positions).
"""
from .attention import (  # noqa: F401
    EMPTY_M,
    attention_heads_ref,
    attention_ref,
    attention_rows_ref,
    block_state,
    decode_paged_ref,
    empty_state,
    finalize_state,
    merge_lse_pair_ref,
    merge_partials_ref,
    merge_states,
    online_softmax_attention,
    prefill_paged_ref,
    to_f64,
)

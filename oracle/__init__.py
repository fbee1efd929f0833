"""fp64 CPU oracle for the decode step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. The CUDA library never does, and
this package never loads the CUDA library: the two share no code. Inputs come
from the ``synthetic`` package, which both sides use.

Every function is pinned by a test in ``tests/test_oracle_pins.py`` against
values the pages print, closed forms, special cases and independent library
routines. No function here is "parity unpinned".
"""

from .decode import (
    append_contiguous,
    append_paged,
    attention_partial,
    causal_attention,
    decode_step_contiguous,
    decode_step_multi,
    decode_step_multi_e5m2,
    decode_step_multi_u8,
    decode_step_paged,
    decode_step_e5m2,
    decode_step_u8,
    dequantize_e5m2,
    dequantize_u8,
    quantize_e5m2,
    quantize_u8,
    decode_unit,
    gather_paged,
    gqa_attention,
    lse_combine,
    mha_attention,
    mqa_attention,
    page_slot,
    rope_inv_freq,
    rope_rotate,
    round_bf16,
    round_to,
    run_cached_sequence,
    run_uncached_sequence,
    window_start,
)
from .accounting import (
    expected_tokens_per_verify,
    kv_bytes_per_token,
    kv_cache_bytes,
    layer_cache_scalars,
    projection_counts_closed_form,
)

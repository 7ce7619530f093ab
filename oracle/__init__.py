"""fp64 CPU oracle for grouped-query decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import,
call or execute anything in this package.  The product (the CUDA library and its Python binding
in ``gqa_decode_attention_03_gb300``) never imports it, and this package imports nothing from
the product: the two share no code.  Inputs reach both sides from the seeded generators in
``gqa_decode_attention_03_gb300.workloads``, which hold none of the method's arithmetic.

Every function is pinned by the CPU tests in ``tests/test_oracle_pins.py`` (brute force at 40
decimal digits, closed forms under ``tests/golden/``, invariants, and planted mistakes that the
pins must catch).  No function here is "parity unpinned".
"""

from .gqa_oracle import (  # noqa: F401
    attend_positions,
    decode_f16,
    decode_q8,
    decode_tq,
    hadamard,
    dequant_f16,
    dequant_q8,
    gated_merge,
    lse_merge,
    order_key,
    output_gate,
    quantize_q8,
    select_topk_cells,
    selected_positions,
    split_partials_f16,
    split_partials_q8,
    unpack_polar,
    unpack_signs,
)

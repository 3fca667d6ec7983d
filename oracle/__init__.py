"""CPU oracle for the paged KV cache hot path -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, fp64 statement of what the CUDA library must
compute. It shares no code with the CUDA path: no kernels, headers, helpers or
tables, and neither side imports the other. Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference legs
may import it; the product path fails loudly when its CUDA extension is
missing and never routes through here.

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
the pages print, closed forms and brute force; none is "parity unpinned".
"""

from .paged_oracle import (  # noqa: F401
    bf16_bits_to_f64,
    blocks_for_tokens,
    last_block_fill,
    kv_bytes_per_token,
    slot_of,
    slot_mapping,
    kv_write,
    copy_blocks,
    gather_request_kv,
    attend_rows,
    paged_attention,
    partial_attention,
    combine_partials,
)

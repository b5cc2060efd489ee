"""CPU oracle for lightning-indexer sparse attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package.  The product path (the CUDA library and its Python
binding) never imports it and shares no code with it.

Two independent implementations of the method's definition on the source
pages, with no blocking, fusion or reordering beyond what that definition
states; each function names the passage it follows:

* ``lidx_oracle.py`` (imported here): plain numpy in float64;
* ``lidx_oracle.cpp`` (``oracle.cpp``): plain C++17 in double, OpenMP over
  query rows, reading large caches in their storage type; it is the one the
  full-size parity tests and the bench's CPU baseline use.

Pins (tests that tie this code to something other than itself) live in
``tests/test_oracle_pins.py`` and run against both implementations; they also
check the two against each other.  Every function is pinned; none is
"parity unpinned".
"""

from .lidx_oracle import (  # noqa: F401
    round_to_storage,
    hadamard_matrix,
    hadamard_rotate,
    visible_count,
    indexer_scores,
    topk_select,
    block_pool,
    block_pool_update,
    quantize_rows,
    dequantize_rows,
    block_select,
    block_select_expanded,
    attention_over,
    sparse_attention_mla,
    sparse_attention_gqa,
    dense_attention_gqa,
    dense_attention_mla,
    decode_pipeline_mla,
)

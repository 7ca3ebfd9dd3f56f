"""Plain, slow CPU oracle for paged-KV grouped-query decode attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

It shares no code with the CUDA path (``paged_kv_cache_45_gb300``): it takes
bfloat16 data as raw ``uint16`` bit patterns in NumPy arrays, widens them to
float64 and computes every result in float64 from the plain definitions the
source pages give. Each function names the page and section it follows.

``prefix_cache`` models the block pool with a prefix cache and copy-on-write
(pinned by ``tests/test_oracle_prefix.py``).

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
the pages or mathematics fix (printed table values, closed forms, invariances,
an independent library routine and brute force); none is "parity unpinned".
"""

from .paged_attention import (  # noqa: F401
    bf16_bits_to_f64,
    kv_bytes_per_token,
    kv_append,
    kv_append_inplace,
    gather_sequence,
    decode,
    decode_online,
    decode_split_partials,
    lse_merge,
    decode_pseudocode_loops,
    decode_multi,
    e4m3_value,
    e4m3_encode,
    e4m3_decode,
    quantize_rows_e4m3,
    kv_append_fp8_inplace,
    dequantize_pool,
    decode_fp8,
    decode_multi_fp8,
)
from .prefix_cache import PrefixCacheModel, CapacityError, copy_blocks  # noqa: F401

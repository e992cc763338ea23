"""fp64 CPU oracle for paged decode attention (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library never does.
"""

from .paged_attention import (  # noqa: F401
    attention,
    attention_weights,
    decode,
    decode_multi,
    decode_partials,
    decode_split,
    gather_sequence,
    merge_partials,
    write_cache,
)

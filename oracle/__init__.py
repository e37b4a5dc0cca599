"""fp64 CPU oracle for sparse MLA decode (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg and reference arm may import this package.  The CUDA path never does.
"""

from .smla_oracle import *  # noqa: F401,F403
from .smla_oracle import (  # noqa: F401
    LATENT_DIM, QK_DIM, RECORD_BYTES, ROPE_DIM, ROPE_OFFSET, SCALE_BLOCK, SCALE_OFFSET,
    bf16_to_f64, combine, e4m3_encode_rne, e4m3_table, e4m3_value, f64_to_bf16_bits_exact,
    pack_records, pow2ceil, row_positions, sparse_mla_decode, split_partials, unpack_records,
    writer_scales,
)

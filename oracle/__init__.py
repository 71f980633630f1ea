"""fp64 CPU oracle for the kvi8r, kvf8s and kvfp4 stores and attention (test
infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm use this package.  It shares no code with the CUDA
path and imports nothing from it.
"""
from .kvi8r import (  # noqa: F401
    HEAD_DIM, as_f64, hadamard, rotate, unrotate, fp16_round, row_scales, quantize,
    encode_rows, build_store, dequant, default_scale, softmax_attention, attend,
    attend_exact, attend_blockwise, rel_rms, group_scales, encode_rows_grouped, build_store_grouped,
)
from . import kvf8s  # noqa: F401
from . import kvfp4  # noqa: F401

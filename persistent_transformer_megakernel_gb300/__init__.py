"""GB300 persistent decode megakernel: Python binding of ``libmk.so``.

The binding only marshals arguments; every step of decode runs in the CUDA
library (``csrc/``).  PyTorch supplies device memory and streams.  Importing
this package does not load the library; the first handle does, and fails
loudly if it is missing or if no CUDA device is present.
"""
from ._binding import (  # noqa: F401
    MK_DECODE_PER_OP,
    MKError,
    Decoder,
    embed_sum,
    embed_sum_noalloc,
    error_string,
    lib_path,
    load_library,
    plan_for,
)

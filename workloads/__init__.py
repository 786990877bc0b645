"""Seeded synthetic inputs for the paged-attention hot path.

This package is shared by the tests, the bench and the CPU oracle's callers.
It draws random numbers and lays out input data (query/key/value tensors,
request lengths, physical block placements, request arrival traces).  It holds
none of the method's arithmetic: no slot computation, no block accounting, no
attention.  Those live separately in the CUDA library and in the oracle.
"""

from .generators import (  # noqa: F401
    PooledRows,
    randn_fp32,
    random_block_placement,
    uniform_int,
)
from .configs import (  # noqa: F401
    DecodeBatch,
    MixedStep,
    TinyCase,
    TraceSpec,
    decode_batch_llama8b,
    long_decode_llama70b,
    mixed_chunked_step,
    tiny_fp32_case,
    trace_spec,
)
from .trace import Arrival, PrefixArrival, generate_arrivals, generate_prefix_arrivals  # noqa: F401

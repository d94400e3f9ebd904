"""fp64 CPU oracle for GGD-BAM attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never calls it and
shares no code with it: the C++ source ``bam_oracle.cpp`` states the method
from the published formulas (GGD-BAM bias, SSMax convention, softmax
attention, chain-rule backward), and this module only marshals numpy arrays
into it.  Every function takes float64 arrays; callers widen their bf16
inputs exactly before calling.

Parity pins (tests/test_oracle_pins.py) tie this oracle to what the pages fix:
the ALiBi worked example, ALiBi and NoPE as special cases, the GGD prior as
``scipy.stats.gennorm``, the softmax-weight ratio invariant, closed-form rows,
decode as the last prefill row, and central finite differences for every
gradient.  No function here is "parity unpinned".
"""

from .oracle import (  # noqa: F401
    build,
    lib_path,
    bias,
    bias_grad,
    fwd,
    fwd_rows,
    decode,
    bwd,
)

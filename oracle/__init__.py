"""Plain CPU oracle for sub-byte KV-cache quantisation and packed-cache decode attention.

TEST INFRASTRUCTURE ONLY. This package is the independent check on the CUDA library: only
the test suite, the smoke check and the benchmark's CPU-baseline leg may import it. The
product path never calls it and there is no CPU fallback through it.

It is written to be read against the pages, not to be fast:
  * quantizers (`oracle.quant`) work in IEEE float32 with round-half-to-even, one operation
    at a time in the order the method states, so that the packed bytes and scales they emit
    are the exact expected values;
  * attention (`oracle.attention`) accumulates in float64 from exactly-dequantised values.

It shares no code with the CUDA path (no headers, tables or helpers) and imports nothing
from it. Readings of points the pages leave open are listed in each function's docstring.
"""
from . import quant, attention  # noqa: F401

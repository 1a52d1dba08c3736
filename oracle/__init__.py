"""CPU FP64 oracle (test infrastructure only; see q4_oracle.py)."""
from .q4_oracle import (  # noqa: F401
    GROUP, ZERO_POINT, k_pad, weight_bytes, fp16_bits_to_f64, bf16_bits_to_f64,
    unpack_codes, dequantize, linear, linear_loops, rms, within_tolerance, check,
    REL_TOL, RMS_TOL,
)
from . import sibling_formats  # noqa: F401,E402
from . import fused_ops  # noqa: F401,E402

"""GB300 (sm_103a) MXFP8 MoE hot path: quantizer -> permute -> grouped GEMM.

The compute lives in the CUDA library ``libmxmoe.so`` (sources in ``csrc/``,
C ABI in ``include/mxmoe.h``); ``binding`` is its thin Python binding and
``synth`` holds the seeded input generators.  Importing the package loads
nothing; the first binding call loads the library and raises if it is missing.
"""
from . import binding, synth  # noqa: F401
from .binding import (MX_COLWISE, MX_ROWWISE, MxError, grouped_gemm_mxfp8_dgrad,  # noqa: F401
                      grouped_gemm_mxfp8_fwd, grouped_gemm_mxfp8_wgrad, moe_gather_rows, moe_permute,
                      mxfp8_quantize)

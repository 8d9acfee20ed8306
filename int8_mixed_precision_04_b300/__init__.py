"""LLM.int8() mixed-precision decomposition linear for B300 (sm_103a).

The compute lives in the CUDA library ``libbnbint8.so`` behind the C ABI of
``include/bnb_int8.h``.  This package only marshals arguments to it
(:mod:`.binding`); torch is used for device memory and streams.  There is no
CPU fallback: without the built library every entry point raises.
"""

from .binding import (BnbError, Lib, Status, linear, linear_bias, linear_debug, load,
                      quantize_weight, workspace_bytes)
from .linear8bit import Linear8bitLt

__all__ = ["BnbError", "Lib", "Linear8bitLt", "Status", "linear", "linear_bias", "linear_debug",
           "load", "quantize_weight", "workspace_bytes"]

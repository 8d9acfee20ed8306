"""LLM.int8() mixed-precision decomposition linear for B300 (sm_103a).

The compute lives in the CUDA library ``libbnbint8.so`` behind the C ABI of
``include/bnb_int8.h``.  This package only marshals arguments to it
(:mod:`.binding`); torch is used for device memory and streams.  There is no
CPU fallback: without the built library every entry point raises.

Forms of the layer: fp16 or bf16 X / W16 / bias / Y (picked from the
tensors' dtype), with or without a bias, with the 16-bit weight as the source
of the outlier columns or with only the int8 weight kept
(:func:`linear_wq_only`); :class:`Linear8bitLt` wraps them as a module in
place of ``torch.nn.Linear``.  The blockwise 8-bit codec of optimizer states
is :func:`quantize_blockwise` / :func:`dequantize_blockwise`.
"""

from .binding import (BnbError, Lib, Status, dequantize_blockwise, linear, linear_bias,
                      linear_debug, linear_ex, linear_from_host, linear_wq_only, load,
                      quantize_blockwise, quantize_weight, workspace_bytes)
from .linear8bit import Linear8bitLt

__all__ = ["BnbError", "Lib", "Linear8bitLt", "Status", "dequantize_blockwise", "linear",
           "linear_bias", "linear_debug", "linear_ex", "linear_from_host", "linear_wq_only",
           "load", "quantize_blockwise", "quantize_weight", "workspace_bytes"]

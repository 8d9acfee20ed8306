"""``Linear8bitLt``: an inference layer in place of ``torch.nn.Linear``.

The LLM.int8() layer is a drop-in replacement for PyTorch's Linear
(bitsandbytes GPU page, section "How LLM.int8() quantizes weights and
activations"): the weight is quantized row-wise once, at construction, and
every forward call runs the mixed-precision decomposition (outlier columns of
X with |x| >= threshold in fp16, the rest in 8 bits) in the CUDA library,
bias included.  This class only keeps the tensors, reshapes the input to
[T, K] and caches a workspace per (row count, CUDA stream); it computes
nothing itself.

Concurrency: a call's workspace must not be shared with a call that may run
at the same time on the GPU.  Forward calls on one stream are ordered, so
they share one workspace; calls on different streams get different ones.
The cache grows with the distinct (row count, stream) pairs seen; ``clear_
workspaces()`` drops it.
"""

from __future__ import annotations

import torch

from . import binding


class Linear8bitLt(torch.nn.Module):
    """y = x W^T + b through ``bnb_int8_linear_ex``, in the weight's dtype.

    weight: [N, K] fp16 or bf16 on a CUDA device (K a multiple of 16); the
    inputs are cast to its dtype and the output has it (bf16 is the compute
    dtype the pages prefer where the hardware has it).  bias: [N] of the
    weight's dtype or None; threshold: the outlier threshold tau (6.0 in the pages'
    experiments; ``math.inf`` turns the decomposition off, 0 sends every
    column to 16-bit).  keep_fp16_weight: keep the 16-bit weight as the
    source of the outlier columns, or keep only the int8 weight, half of its
    bytes, and take the outlier columns from the codes dequantized (W16 NULL).  Inference only: no gradient flows
    through the layer.
    """

    def __init__(self, weight: torch.Tensor, bias: torch.Tensor | None = None,
                 threshold: float = 6.0, keep_fp16_weight: bool = True):
        super().__init__()
        if (weight.dim() != 2 or weight.dtype not in (torch.float16, torch.bfloat16)
                or not weight.is_cuda):
            raise ValueError("weight must be a 2-D fp16 or bf16 CUDA tensor")
        N, K = weight.shape
        if bias is not None and (bias.shape != (N,) or bias.dtype != weight.dtype
                                 or bias.device != weight.device):
            raise ValueError("bias must be an [N] tensor of the weight's dtype and device")
        self.dtype = weight.dtype
        self.in_features, self.out_features = K, N
        self.threshold = float(threshold)
        W16 = weight.detach().contiguous()
        Wq, sw = binding.quantize_weight(W16)
        self.register_buffer("W16", W16 if keep_fp16_weight else None)
        self.register_buffer("Wq", Wq)
        self.register_buffer("Wscale", sw)
        self.register_buffer("bias", None if bias is None else bias.detach().contiguous())
        self._ws: dict[tuple[int, int], torch.Tensor] = {}

    @classmethod
    def from_linear(cls, layer: torch.nn.Linear, threshold: float = 6.0,
                    keep_fp16_weight: bool = True,
                    dtype: torch.dtype = torch.float16) -> "Linear8bitLt":
        """The int8 layer for an existing ``nn.Linear`` (weights cast to
        ``dtype``, fp16 or bf16, on the current CUDA device if they are not
        there yet)."""
        dev = layer.weight.device if layer.weight.is_cuda else torch.device("cuda")
        w = layer.weight.detach().to(dev, dtype)
        b = None if layer.bias is None else layer.bias.detach().to(dev, dtype)
        return cls(w, b, threshold, keep_fp16_weight)

    def _workspace(self, T: int) -> torch.Tensor:
        # one workspace per (T, stream): calls on one stream are ordered and
        # may share it, calls on different streams may overlap and may not
        key = (T, torch.cuda.current_stream(self.Wq.device).cuda_stream)
        ws = self._ws.get(key)
        if ws is None:
            ws = torch.empty((binding.workspace_bytes(T, self.out_features, self.in_features),),
                             dtype=torch.uint8, device=self.Wq.device)
            self._ws[key] = ws
        return ws

    def clear_workspaces(self) -> None:
        """Drop the cached workspaces (after the streams that used them are done)."""
        self._ws.clear()

    @torch.no_grad()
    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.shape[-1] != self.in_features:
            raise ValueError(f"expected {self.in_features} input features, got {x.shape[-1]}")
        lead = x.shape[:-1]
        X = x.reshape(-1, self.in_features).to(self.dtype).contiguous()
        T = X.shape[0]
        Y = torch.empty((T, self.out_features), dtype=self.dtype, device=X.device)
        if T > 0:
            binding.linear_ex(X, self.Wq, self.Wscale, self.W16, self.bias, self.threshold,
                              Y=Y, workspace=self._workspace(T))
        return Y.reshape(*lead, self.out_features)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"bias={self.bias is not None}, dtype={self.dtype}, threshold={self.threshold}, "
                f"keep_fp16_weight={self.W16 is not None}")

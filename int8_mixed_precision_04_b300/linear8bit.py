"""``Linear8bitLt``: an inference layer in place of ``torch.nn.Linear``.

The LLM.int8() layer is a drop-in replacement for PyTorch's Linear
(bitsandbytes GPU page, section "How LLM.int8() quantizes weights and
activations"): the weight is quantized row-wise once, at construction, and
every forward call runs the mixed-precision decomposition (outlier columns of
X with |x| >= threshold in fp16, the rest in 8 bits) in the CUDA library,
bias included.  This class only keeps the tensors, reshapes the input to
[T, K] and caches a workspace per row count; it computes nothing itself.
"""

from __future__ import annotations

import torch

from . import binding


class Linear8bitLt(torch.nn.Module):
    """y = x W^T + b through ``bnb_int8_linear_bias`` (fp16 in, fp16 out).

    weight: [N, K] fp16 on a CUDA device (K a multiple of 16); bias: [N] fp16
    or None; threshold: the outlier threshold tau (6.0 in the pages'
    experiments; ``math.inf`` turns the decomposition off, 0 sends every
    column to fp16).  keep_fp16_weight: keep W16 as the source of the outlier
    columns (``bnb_int8_linear_bias``), or keep only the int8 weight, half of
    fp16's bytes, and take the outlier columns from the codes dequantized
    (``bnb_int8_linear_wq_only``).  Inference only: no gradient flows
    through the layer.
    """

    def __init__(self, weight: torch.Tensor, bias: torch.Tensor | None = None,
                 threshold: float = 6.0, keep_fp16_weight: bool = True):
        super().__init__()
        if weight.dim() != 2 or weight.dtype != torch.float16 or not weight.is_cuda:
            raise ValueError("weight must be a 2-D fp16 CUDA tensor")
        N, K = weight.shape
        if bias is not None and (bias.shape != (N,) or bias.dtype != torch.float16
                                 or bias.device != weight.device):
            raise ValueError("bias must be an fp16 [N] tensor on the weight's device")
        self.in_features, self.out_features = K, N
        self.threshold = float(threshold)
        W16 = weight.detach().contiguous()
        Wq, sw = binding.quantize_weight(W16)
        self.register_buffer("W16", W16 if keep_fp16_weight else None)
        self.register_buffer("Wq", Wq)
        self.register_buffer("Wscale", sw)
        self.register_buffer("bias", None if bias is None else bias.detach().contiguous())
        self._ws: dict[int, torch.Tensor] = {}

    @classmethod
    def from_linear(cls, layer: torch.nn.Linear, threshold: float = 6.0,
                    keep_fp16_weight: bool = True) -> "Linear8bitLt":
        """The int8 layer for an existing ``nn.Linear`` (weights cast to fp16
        on the current CUDA device if they are not there yet)."""
        dev = layer.weight.device if layer.weight.is_cuda else torch.device("cuda")
        w = layer.weight.detach().to(dev, torch.float16)
        b = None if layer.bias is None else layer.bias.detach().to(dev, torch.float16)
        return cls(w, b, threshold, keep_fp16_weight)

    def _workspace(self, T: int) -> torch.Tensor:
        ws = self._ws.get(T)
        if ws is None:
            ws = torch.empty((binding.workspace_bytes(T, self.out_features, self.in_features),),
                             dtype=torch.uint8, device=self.Wq.device)
            self._ws[T] = ws
        return ws

    @torch.no_grad()
    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.shape[-1] != self.in_features:
            raise ValueError(f"expected {self.in_features} input features, got {x.shape[-1]}")
        lead = x.shape[:-1]
        X = x.reshape(-1, self.in_features).to(torch.float16).contiguous()
        T = X.shape[0]
        Y = torch.empty((T, self.out_features), dtype=torch.float16, device=X.device)
        if T > 0 and self.W16 is not None:
            binding.linear_bias(X, self.Wq, self.Wscale, self.W16, self.bias, self.threshold,
                                Y=Y, workspace=self._workspace(T))
        elif T > 0:
            binding.linear_wq_only(X, self.Wq, self.Wscale, self.bias, self.threshold, Y=Y,
                                   workspace=self._workspace(T))
        return Y.reshape(*lead, self.out_features)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"bias={self.bias is not None}, threshold={self.threshold}, "
                f"keep_fp16_weight={self.W16 is not None}")

"""The NVFP4 linear layer of the pretraining recipe as a PyTorch autograd
Function ("NVIDIA Introduces a 4-Bit Pretraining Methodology Using NVFP4",
"Method"): all three GEMMs of a linear layer in NVFP4 with FP32 accumulation.

    fprop  Y  = X W^T        X: 1D blocks, RNE;  W: 2D 16x16 blocks, RNE
    dgrad  dX = dY W         dY: 1D blocks, stochastic rounding;  W^T: the
                             forward quantization of W, repacked (no re-encode)
    wgrad  dW = dY^T X       both operands transposed so that K = tokens,
                             16x16 Random Hadamard Transform along the tokens
                             with one sign vector for both, dY^T with
                             stochastic rounding, X^T with RNE

Every step runs in the library's kernels through the C ABI; this module only
orders the calls, keeps the quantized weight for the backward pass and
advances the Philox stream.  ``enabled=False`` keeps a layer in BF16 (the
recipe leaves some layers in higher precision); that path is torch's own
matmul and does not touch the library.

Shapes: tokens, out_features and in_features each a multiple of 64 (each of
them is the K of one of the three GEMMs, whose K steps by 64); the 2D weight
blocks and the Hadamard chunks (16) divide that.
"""
from __future__ import annotations

import torch

from . import gemm, quantize, rht_quantize, transpose_2d


def _check_shapes(tokens: int, n_out: int, n_in: int):
    for name, v in (("tokens", tokens), ("out_features", n_out), ("in_features", n_in)):
        if v % 64:
            raise ValueError(f"{name} = {v} must be a multiple of 64 (it is the K of one of the layer's GEMMs)")


class NVFP4LinearFunction(torch.autograd.Function):
    """y = x @ weight^T with NVFP4 operands in all three GEMMs.

    seed: Philox key of the gradient rounding; offset: this call's stream
    position (dgrad draws with offset 2*offset, wgrad with 2*offset + 1, so
    the two gradient quantizations never share draws).  rht_seed: sign
    vector of the wgrad Hadamard transform."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, weight: torch.Tensor, seed: int, offset: int, rht_seed: int):
        T, n_in = x.shape
        n_out = weight.shape[0]
        _check_shapes(T, n_out, n_in)
        qx = quantize(x)
        qw = quantize(weight, block="2d")
        y = gemm(qx, qw, out_dtype=x.dtype if x.dtype in (torch.bfloat16, torch.float32) else torch.bfloat16)
        ctx.save_for_backward(x)
        ctx.qw = qw
        ctx.cfg = (seed, offset, rht_seed, weight.dtype)
        return y

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        (x,) = ctx.saved_tensors
        seed, offset, rht_seed, wdtype = ctx.cfg
        dy = dy.contiguous()
        dx = dw = None
        if ctx.needs_input_grad[0]:
            qdy = quantize(dy, rounding="stochastic", seed=seed, offset=2 * offset)
            qwt = transpose_2d(ctx.qw)
            dx = gemm(qdy, qwt, out_dtype=x.dtype)
        if ctx.needs_input_grad[1]:
            qdyt, _ = rht_quantize(dy, rht_seed=rht_seed, transpose=True, rounding="stochastic", seed=seed,
                                   offset=2 * offset + 1)
            qxt, _ = rht_quantize(x, rht_seed=rht_seed, transpose=True)
            dw = gemm(qdyt, qxt, out_dtype=torch.float32)
            if wdtype != torch.float32:
                dw = dw.to(wdtype)
        ctx.qw = None
        return dx, dw, None, None, None


class NVFP4Linear(torch.nn.Module):
    """Bias-free linear layer whose three GEMMs run in NVFP4.

    enabled=False runs the layer in BF16 with torch.matmul (per-layer
    opt-out).  Every forward call advances the gradient-rounding stream by
    one position."""

    def __init__(self, in_features: int, out_features: int, *, enabled: bool = True, seed: int = 0,
                 rht_seed: int = 1, device=None, dtype=torch.bfloat16):
        super().__init__()
        self.weight = torch.nn.Parameter(torch.empty((out_features, in_features), device=device, dtype=dtype))
        torch.nn.init.normal_(self.weight, std=0.02)
        self.enabled = enabled
        self.seed = seed
        self.rht_seed = rht_seed
        self.calls = 0

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if not self.enabled:
            return x @ self.weight.t()
        offset = self.calls
        self.calls += 1
        return NVFP4LinearFunction.apply(x, self.weight, self.seed, offset, self.rht_seed)

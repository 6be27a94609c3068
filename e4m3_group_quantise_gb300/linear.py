"""FP8 linear layer: the unified precision flow of one GEMM layer.

Jet-RL (technical summaries on gist.science, "Architecture Centrale" and
"Schéma de Quantification"):
  * rollout and the training forward use the same FP8 quantisation flow, so
    the inference graph is a subgraph of the training forward graph -- here
    both call ``quantize_act`` + ``gemm_fprop`` on the same cached weight
    codes and produce bit-identical outputs;
  * master weights stay BF16; their FP8 codes (128x128 blocks) are derived
    once per weight update (cached against the tensor's version counter);
  * activations saved for backward are kept in FP8: the forward stores the
    128x1-grouped transposed codes of X (``quantize_act_transposed``), never
    the BF16 X;
  * gradients between operators are BF16; dY is quantised at the GEMM
    boundary (1x128 for DGrad, 128x1 for WGrad), and DGrad / WGrad run in FP8.
Only tensor allocation and autograd wiring live here; every arithmetic step
is a call into the CUDA library.

Errors: the calls raise on any argument or launch error.  A kernel whose
bounded wait on an asynchronous copy or a tensor-core barrier gives up does
not hang: it records the failure in the device's error word and leaves its
output incomplete.  Reading that word needs a synchronisation, so these layers
never read it themselves; a training or rollout loop that must not continue
on incomplete results calls ``jetfp8_poll_device_error()`` once per step
(after the backward, or after a rollout batch) and stops on a non-zero status.
"""
from __future__ import annotations

import torch

from . import jetfp8 as _j


class QuantizedWeight:
    """FP8 codes of a BF16 master weight, refreshed when the weight changes."""

    def __init__(self):
        self._key = None
        self.q = self.s = self.qt = None

    def get(self, w: torch.Tensor):
        key = (w.data_ptr(), w._version, tuple(w.shape), w.device)
        if key != self._key:
            self.q, self.s, self.qt = _j.quantize_weight(w.detach(), transposed=True)
            self._key = key
        return self.q, self.s, self.qt


_SIDE_STREAMS = {}


def _side_stream(device) -> torch.cuda.Stream:
    """One extra stream per device for the backward's Wgrad."""
    key = torch.device(device).index
    if key not in _SIDE_STREAMS:
        _SIDE_STREAMS[key] = torch.cuda.Stream(device=device)
    return _SIDE_STREAMS[key]


class FP8LinearFunction(torch.autograd.Function):
    """y = x W^T with FP8 Fprop; FP8 Dgrad and Wgrad in backward."""

    @staticmethod
    def forward(ctx, x2d: torch.Tensor, weight: torch.Tensor, cache: QuantizedWeight):
        q, s, qt = cache.get(weight)
        if ctx.needs_input_grad[1]:
            # one read of X: 1x128 codes for Fprop + the transposed 128x1 codes
            # saved (in FP8) for Wgrad; the former are bit-identical to rollout's
            qx, sx, qxt, sxt = _j.quantize_act_dual(x2d)
        else:
            qx, sx = _j.quantize_act(x2d)
            qxt = sxt = None
        y = _j.gemm_fprop(qx, sx, q, s)
        ctx.save_for_backward(qt, s, qxt, sxt)
        return y

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        qt, s, qxt, sxt = ctx.saved_tensors
        dy = dy.contiguous()
        dx = dw = None
        if ctx.needs_input_grad[0] and ctx.needs_input_grad[1]:
            qdy, sdy, qdyt, sdyt = _j.quantize_act_dual(dy)
        elif ctx.needs_input_grad[0]:
            qdy, sdy = _j.quantize_act(dy)
        elif ctx.needs_input_grad[1]:
            qdyt, sdyt = _j.quantize_act_transposed(dy)
        if ctx.needs_input_grad[0] and ctx.needs_input_grad[1]:
            # Dgrad and Wgrad are independent: Wgrad runs on a side stream so
            # that each GEMM's last partial wave of tiles is filled by the other
            main = torch.cuda.current_stream(dy.device)
            side = _side_stream(dy.device)
            side.wait_stream(main)
            with torch.cuda.stream(side):
                dw = _j.gemm_wgrad(qdyt, sdyt, qxt, sxt)
            for t in (qdyt, sdyt, qxt, sxt):
                t.record_stream(side)
            dx = _j.gemm_dgrad(qdy, sdy, qt, s)
            main.wait_stream(side)
            dw.record_stream(main)
            return dx, dw, None
        if ctx.needs_input_grad[0]:
            dx = _j.gemm_dgrad(qdy, sdy, qt, s)
        if ctx.needs_input_grad[1]:
            dw = _j.gemm_wgrad(qdyt, sdyt, qxt, sxt)
        return dx, dw, None


class FP8Linear(torch.nn.Module):
    """Bias-free linear layer with a BF16 master weight [out, in] and the FP8
    path for every product.  ``in_features`` and ``out_features`` must be
    multiples of 128; in training the token count must be one too (WGrad
    groups 128 tokens)."""

    def __init__(self, in_features: int, out_features: int, device=None):
        super().__init__()
        if in_features % 128 or out_features % 128:
            raise ValueError("FP8Linear needs in/out features that are multiples of 128")
        self.weight = torch.nn.Parameter(torch.empty(out_features, in_features, dtype=torch.bfloat16,
                                                     device=device))
        self._cache = QuantizedWeight()

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        shape = x.shape
        x2d = x.reshape(-1, shape[-1]).contiguous()
        if torch.is_grad_enabled() and (x.requires_grad or self.weight.requires_grad):
            y = FP8LinearFunction.apply(x2d, self.weight, self._cache)
        else:
            q, s, _ = self._cache.get(self.weight)
            qx, sx = _j.quantize_act(x2d)
            y = _j.gemm_fprop(qx, sx, q, s)
        return y.reshape(*shape[:-1], y.shape[-1])

    def forward_quantized(self, qx: torch.Tensor, sx: torch.Tensor) -> torch.Tensor:
        """Rollout Fprop on an input that is already FP8 (1x128 codes qx
        [M, in], scales sx [in/128, M]), e.g. from a fused RMSNorm or SwiGLU
        producer; no autograd.  Bit-identical to ``forward`` on the bf16 value
        those codes quantise."""
        q, s, _ = self._cache.get(self.weight)
        return _j.gemm_fprop(qx, sx, q, s)

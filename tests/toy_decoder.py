"""A 2-layer toy decoder whose every linear layer (LM head included) runs the
FP8 path -- test fixture for the unified rollout/training precision flow.

Per layer: RMSNorm -> QKV -> causal softmax attention (4 heads x 128, fp32
softmax, no positional encoding) -> O -> residual -> RMSNorm -> gate_up
(2 x 1536) -> SiLU(gate) * up -> down -> residual.  Then a final RMSNorm and
the LM head [vocab 4096, hidden 512].  Weights ~ N(0, 0.02), seed 0.
The non-linear ops use plain PyTorch (they are not on the FP8 GEMM path).
``forward(tokens, bf16_linears=True)`` runs every linear layer as a plain
PyTorch bf16 matmul on the same master weights instead: the BF16 reference
whose mismatch against the FP8 path the pages describe.

``producers="jetfp8"`` computes RMSNorm and SwiGLU with the library's own
kernels (their backward recomputes in plain PyTorch).  With ``fused=True``
(rollout, no autograd) the FP8 inputs of the qkv, gate_up, down and head
projections come straight from the fused RMSNorm / SwiGLU producers; without
it the producers write bf16 and the linear layers quantise -- the same codes.
"""
import torch

import e4m3_group_quantise_gb300 as jf
from e4m3_group_quantise_gb300 import FP8Linear

HIDDEN, HEADS, HEAD_DIM, INTER, VOCAB, LAYERS = 512, 4, 128, 1536, 4096, 2


def rmsnorm(x, w, eps=1e-6):
    xf = x.float()
    return (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + eps) * w.float()).to(torch.bfloat16)


EPS = 1e-6


def rmsnorm_ref(xf, wf, eps=EPS):
    return xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + eps) * wf


class RMSNormJ(torch.autograd.Function):
    """Forward: the library's RMSNorm kernel (bf16 output only).  Backward:
    plain PyTorch on the saved input."""

    @staticmethod
    def forward(ctx, x, w):
        ctx.save_for_backward(x, w)
        x2d = x.reshape(-1, x.shape[-1]).contiguous()
        return jf.rmsnorm_quantize_act(x2d, w, EPS, quantize=False)[2].reshape(x.shape)

    @staticmethod
    def backward(ctx, dy):
        x, w = ctx.saved_tensors
        with torch.enable_grad():
            xf = x.float().requires_grad_()
            wf = w.float().requires_grad_()
            dx, dw = torch.autograd.grad(rmsnorm_ref(xf, wf), (xf, wf), dy.float())
        return dx.to(x.dtype), dw.to(w.dtype)


class SwiGLUJ(torch.autograd.Function):
    """Forward: the library's SwiGLU kernel on gate_up [.., 2I] (bf16 output).
    Backward: plain PyTorch."""

    @staticmethod
    def forward(ctx, gu):
        ctx.save_for_backward(gu)
        g2d = gu.reshape(-1, gu.shape[-1]).contiguous()
        return jf.swiglu_quantize_act(g2d, quantize=False)[2].reshape(*gu.shape[:-1], gu.shape[-1] // 2)

    @staticmethod
    def backward(ctx, dy):
        (gu,) = ctx.saved_tensors
        with torch.enable_grad():
            f = gu.float().requires_grad_()
            g, u = f.chunk(2, dim=-1)
            (d,) = torch.autograd.grad(torch.nn.functional.silu(g) * u, (f,), dy.float())
        return d.to(gu.dtype)


class ToyDecoder(torch.nn.Module):
    def __init__(self, device="cuda", seed=0):
        super().__init__()
        g = torch.Generator(device="cpu").manual_seed(seed)
        self.embed = torch.nn.Parameter((torch.randn(VOCAB, HIDDEN, generator=g) * 0.02).to(torch.bfloat16).to(device))
        self.layers = torch.nn.ModuleList()
        for _ in range(LAYERS):
            lyr = torch.nn.Module()
            lyr.qkv = FP8Linear(HIDDEN, 3 * HEADS * HEAD_DIM, device=device)
            lyr.o = FP8Linear(HEADS * HEAD_DIM, HIDDEN, device=device)
            lyr.gate_up = FP8Linear(HIDDEN, 2 * INTER, device=device)
            lyr.down = FP8Linear(INTER, HIDDEN, device=device)
            lyr.n1 = torch.nn.Parameter(torch.ones(HIDDEN, dtype=torch.bfloat16, device=device))
            lyr.n2 = torch.nn.Parameter(torch.ones(HIDDEN, dtype=torch.bfloat16, device=device))
            self.layers.append(lyr)
        self.norm = torch.nn.Parameter(torch.ones(HIDDEN, dtype=torch.bfloat16, device=device))
        self.head = FP8Linear(HIDDEN, VOCAB, device=device)
        with torch.no_grad():
            for m in self.modules():
                if isinstance(m, FP8Linear):
                    m.weight.copy_((torch.randn(m.weight.shape, generator=g) * 0.02).to(torch.bfloat16))

    def forward(self, tokens, bf16_linears: bool = False, producers: str = "torch", fused: bool = False):
        def lin(m, x):
            return torch.nn.functional.linear(x, m.weight) if bf16_linears else m(x)

        def norm_lin(m, x, w):
            """m(rmsnorm(x, w)), through the fused FP8 producer when asked."""
            if producers == "torch":
                return lin(m, rmsnorm(x, w))
            if fused:
                q, s, _ = jf.rmsnorm_quantize_act(x.reshape(-1, x.shape[-1]).contiguous(), w, EPS)
                return m.forward_quantized(q, s).reshape(*x.shape[:-1], m.weight.shape[0])
            return lin(m, RMSNormJ.apply(x, w))

        def mlp_down(m, gu):
            if producers == "torch":
                gate, up = gu.float().chunk(2, dim=-1)
                return lin(m, (torch.nn.functional.silu(gate) * up).to(torch.bfloat16))
            if fused:
                q, s, _ = jf.swiglu_quantize_act(gu.reshape(-1, gu.shape[-1]).contiguous())
                return m.forward_quantized(q, s).reshape(*gu.shape[:-1], m.weight.shape[0])
            return lin(m, SwiGLUJ.apply(gu))

        if fused and (producers == "torch" or torch.is_grad_enabled()):
            raise ValueError("the fused path is the rollout path: jetfp8 producers, no autograd")
        B, T = tokens.shape
        h = self.embed[tokens]                                  # [B, T, H] bf16
        mask = torch.ones(T, T, dtype=torch.bool, device=tokens.device).tril()
        for lyr in self.layers:
            a = norm_lin(lyr.qkv, h, lyr.n1)                    # [B, T, 3*H]
            q, k, v = a.float().view(B, T, 3, HEADS, HEAD_DIM).unbind(2)
            q, k, v = (t.transpose(1, 2) for t in (q, k, v))     # [B, heads, T, d]
            att = (q @ k.transpose(-1, -2)) / HEAD_DIM ** 0.5
            att = att.masked_fill(~mask, float("-inf")).softmax(-1)
            ctx = (att @ v).transpose(1, 2).reshape(B, T, HEADS * HEAD_DIM).to(torch.bfloat16)
            h = h + lin(lyr.o, ctx)
            h = h + mlp_down(lyr.down, norm_lin(lyr.gate_up, h, lyr.n2))
        return norm_lin(self.head, h, self.norm)                # logits [B, T, V] bf16

"""Unified precision flow on a 2-layer toy decoder (hidden 512, vocab 4096,
seq 128, batch 2): the rollout forward (no autograd) and the training forward
(autograd, saving FP8 transposed activations for WGrad) must produce
bit-identical logits, because both run the same FP8 kernels on the same
codes (Jet-RL, "Architecture Centrale": the inference graph is a subgraph of
the training forward graph, same granularity and precision)."""
import pytest
import torch

import e4m3_group_quantise_gb300 as jf
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def model():
    require_gpu()
    from toy_decoder import ToyDecoder
    torch.manual_seed(0)
    return ToyDecoder(device="cuda", seed=0)


def tokens(seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 4096, (2, 128), generator=g).cuda()


def test_rollout_vs_training_logits_bit_identical(model):
    t = tokens()
    with torch.no_grad():
        rollout = model(t)
    train = model(t)                 # autograd on: FP8Linear.apply saves FP8 X^T
    assert train.requires_grad
    assert rollout.dtype == torch.bfloat16 and rollout.shape == (2, 128, 4096)
    assert torch.equal(rollout, train.detach())
    # and again after another rollout (no hidden state between calls)
    with torch.no_grad():
        again = model(t)
    assert torch.equal(rollout, again)


def test_training_step_backward(model):
    t = tokens(1)
    logits = model(t)
    loss = torch.nn.functional.cross_entropy(logits.float().view(-1, 4096), t.view(-1))
    loss.backward()
    for name, p in model.named_parameters():
        if p.grad is not None:
            assert torch.isfinite(p.grad.float()).all(), name
    w = model.layers[0].qkv.weight
    assert w.grad is not None and w.grad.abs().sum() > 0
    assert jf.jetfp8_poll_device_error() == 0


def test_weight_update_refreshes_codes(model):
    t = tokens(2)
    with torch.no_grad():
        before = model(t)
        model.head.weight.mul_(0.5)          # an optimiser step on the master weight
        after = model(t)
        model.head.weight.mul_(2.0)
    assert not torch.equal(before, after)


@pytest.mark.parametrize("T", [128, 512, 2048])
def test_bf16_vs_fp8_mismatch_by_length(model, T):
    """The mismatch the unified flow removes, measured without RL: next-token
    log-probabilities of a BF16 forward (every linear a bf16 matmul) against
    the FP8 forward, on the same weights, at growing sequence length.  The
    FP8 rollout and the FP8 training forward stay bit-identical at every
    length (mismatch exactly 0); BF16 against FP8 differs.  The figures are
    printed (pytest -s) for the record."""
    g = torch.Generator().manual_seed(100 + T)
    t = torch.randint(0, 4096, (1, T), generator=g).cuda()
    with torch.no_grad():
        lp_rollout = torch.log_softmax(model(t).float(), -1)
        lp_bf16 = torch.log_softmax(model(t, bf16_linears=True).float(), -1)
    lp_train = torch.log_softmax(model(t).detach().float(), -1)
    assert torch.equal(lp_rollout, lp_train)
    # log-prob of the observed next token, as an RL objective would use it
    nxt = t[0, 1:]
    a = lp_rollout[0, :-1].gather(-1, nxt[:, None])[:, 0]
    b = lp_bf16[0, :-1].gather(-1, nxt[:, None])[:, 0]
    dlp = (a - b).abs()
    kl = (lp_bf16.exp() * (lp_bf16 - lp_rollout)).sum(-1)[0]      # KL(bf16 || fp8) per position
    top1 = (lp_bf16.argmax(-1) == lp_rollout.argmax(-1)).float().mean().item()
    print(f"\nT={T}: |dlogp| mean {dlp.mean().item():.3e} max {dlp.max().item():.3e}; "
          f"KL mean {kl.mean().item():.3e} max {kl.max().item():.3e}; top-1 agreement {top1:.4f}")
    assert torch.isfinite(dlp).all() and dlp.max() > 0


def test_fused_producers_rollout_equals_training(model):
    """Rollout with the fused RMSNorm -> FP8 and SwiGLU -> FP8 producers
    feeding the GEMMs directly gives the same logits, bit for bit, as the
    training forward that writes the producers' bf16 outputs and lets the
    linear layers quantise them (and that backpropagates)."""
    t = tokens(3)
    with torch.no_grad():
        rollout = model(t, producers="jetfp8", fused=True)
        unfused = model(t, producers="jetfp8")
    train = model(t, producers="jetfp8")
    assert torch.equal(rollout, unfused)
    assert torch.equal(rollout, train.detach())
    loss = torch.nn.functional.cross_entropy(train.float().view(-1, 4096), t.view(-1))
    loss.backward()
    assert model.layers[0].n1.grad is not None and torch.isfinite(model.layers[0].n1.grad.float()).all()
    assert model.layers[1].gate_up.weight.grad.abs().sum() > 0
    # the producers' forward stays close to the PyTorch reference operators
    with torch.no_grad():
        ref = model(t)
    assert (rollout.float() - ref.float()).abs().max() < 0.25
    assert jf.jetfp8_poll_device_error() == 0

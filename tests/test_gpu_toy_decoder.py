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

"""The C-ABI calls inside CUDA graphs (the way a decode loop or a training
step is replayed without per-call host cost): a captured sequence of
quantisers and GEMMs, replayed on new inputs written into the captured
buffers, gives bit for bit what the same calls give eagerly.  The library
allocates nothing and synchronises nothing inside these calls, so capture
works on any stream."""
import pytest
import torch

import e4m3_group_quantise_gb300 as jf
from e4m3_group_quantise_gb300 import synthetic as syn
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def layer_buffers(M, N, K):
    u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
    e = lambda *s, dt=u8: torch.empty(*s, dtype=dt, device=DEV)  # noqa: E731
    return {
        "x": e(M, K, dt=bf), "w": e(N, K, dt=bf), "dy": e(M, N, dt=bf),
        "qw": e(N, K), "sw": e(N // 128, K // 128, dt=f32), "qwt": e(K, N),
        "qx": e(M, K), "sx": e(K // 128, M, dt=f32), "qxt": e(K, M), "sxt": e(M // 128, K, dt=f32),
        "qdy": e(M, N), "sdy": e(N // 128, M, dt=f32), "qdyt": e(N, M), "sdyt": e(M // 128, N, dt=f32),
        "y": e(M, N, dt=bf), "dx": e(M, K, dt=bf), "dw": e(N, K, dt=bf),
    }


def layer_step(d):
    jf.jetfp8_quantize_weight(d["w"], d["qw"], d["sw"], d["qwt"])
    jf.jetfp8_quantize_act_dual(d["x"], d["qx"], d["sx"], d["qxt"], d["sxt"])
    jf.jetfp8_quantize_act_dual(d["dy"], d["qdy"], d["sdy"], d["qdyt"], d["sdyt"])
    jf.jetfp8_gemm_fprop(d["qx"], d["sx"], d["qw"], d["sw"], d["y"])
    jf.jetfp8_gemm_dgrad(d["qdy"], d["sdy"], d["qwt"], d["sw"], d["dx"])
    jf.jetfp8_gemm_wgrad(d["qdyt"], d["sdyt"], d["qxt"], d["sxt"], d["dw"])


def fill(d, seed, M, N, K):
    d["x"].copy_(syn.activation(M, K, seed=seed, outlier_scale=20.0, device=DEV))
    d["w"].copy_(syn.weight(N, K, seed=seed, device=DEV))
    d["dy"].copy_(syn.grad_output(M, N, seed=seed, device=DEV))


@pytest.mark.parametrize("M,N,K", [(512, 768, 640), (4096, 6144, 4096)])
def test_training_step_graph_replay_matches_eager(M, N, K):
    d = layer_buffers(M, N, K)
    fill(d, 1, M, N, K)
    layer_step(d)                                   # warm-up (module loading, attributes)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side), torch.cuda.graph(g, stream=side):
        layer_step(d)
    for seed in (2, 3):
        fill(d, seed, M, N, K)
        g.replay()
        torch.cuda.synchronize()
        got = {k: d[k].clone() for k in ("qx", "sx", "qxt", "qdyt", "y", "dx", "dw")}
        layer_step(d)                               # eager, same inputs
        torch.cuda.synchronize()
        for k, v in got.items():
            assert torch.equal(v, d[k]), (seed, k)
    assert jf.jetfp8_poll_device_error() == 0


@pytest.mark.parametrize("M", [1, 64])
def test_decode_graph_replay(M):
    """A decode-sized Fprop (narrow tiles) replayed from a graph."""
    N, K = syn.PROJ_8B["qkv"]
    w = syn.weight(N, K, seed=5, device=DEV)
    qw, sw, _ = jf.quantize_weight(w, transposed=False)
    x = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
    qx = torch.empty(M, K, dtype=torch.uint8, device=DEV)
    sx = torch.empty(K // 128, M, dtype=torch.float32, device=DEV)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)

    def step():
        jf.jetfp8_quantize_act(x, qx, sx)
        jf.jetfp8_gemm_fprop(qx, sx, qw, sw, y)

    x.copy_(syn.activation(M, K, seed=6, device=DEV))
    step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side), torch.cuda.graph(g, stream=side):
        step()
    for seed in (7, 8, 9):
        x.copy_(syn.activation(M, K, seed=seed, device=DEV))
        g.replay()
        torch.cuda.synchronize()
        got = y.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(got, y), seed

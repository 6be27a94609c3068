"""The conversion every quantiser ends in (cvt.rn.satfinite.e4m3x2.f32 inside
the kernels) against the oracle's encoder for all 2^32 fp32 bit patterns:
round to nearest even, saturation to +-448 (infinities included), NaN to the
NaN code, signed zeros and subnormal E4M3 results.  The GPU converts 2^28
patterns per chunk; the oracle compares each chunk on the host while the GPU
converts the next."""
from concurrent.futures import ThreadPoolExecutor

import pytest
import torch

import oracle
import e4m3_group_quantise_gb300 as jf
from gpu_util import ORACLE_THREADS, require_gpu

pytestmark = pytest.mark.gpu
CHUNK = 1 << 28
SLICE = 1 << 24


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_every_fp32_pattern():
    bufs = [torch.empty(CHUNK, dtype=torch.uint8, device="cuda") for _ in range(2)]
    host = [torch.empty(CHUNK, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    checks = [[], []]                             # futures still reading each host buffer
    with ThreadPoolExecutor(max_workers=max(2, ORACLE_THREADS)) as pool:
        for c in range((1 << 32) // CHUNK):
            first, i = c * CHUNK, c % 2
            for f in checks[i]:                   # the buffer's previous chunk is checked
                f.result()
            jf.jetfp8_e4m3_encode_range(first, bufs[i])
            host[i].copy_(bufs[i])                # synchronous: the codes are on the host
            codes = host[i].numpy()
            checks[i] = [pool.submit(_check, first + lo, codes[lo:lo + SLICE])
                         for lo in range(0, CHUNK, SLICE)]
        for fs in checks:
            for f in fs:
                f.result()
    assert jf.jetfp8_poll_device_error() == 0


def _check(first, codes):
    # one C call per slice (the GIL is released while it runs)
    bad, where = oracle.e4m3_encode_check_range(first, codes)
    assert bad == 0, (hex(first + where), int(codes[where]))


def test_ragged_range_tail():
    """A count that is not a multiple of eight, starting mid-way: the tail
    codes are written and nothing past them."""
    out = torch.full((64,), 0xAB, dtype=torch.uint8, device="cuda")
    first = 0x3F7FFFF0                            # just below 1.0f
    jf.jetfp8_e4m3_encode_range(first, out[:45].view(-1))
    got = out.cpu().numpy()
    want = oracle.e4m3_encode(
        torch.arange(first, first + 45, dtype=torch.int64).to(torch.int32).numpy().view("float32"))
    assert (got[:45] == want).all()
    assert (got[45:] == 0xAB).all()

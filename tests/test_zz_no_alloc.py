"""nvfp4_quantize_noalloc: the quantizer for callers that cannot allocate
device memory (a plugin inside a host program that owns all device memory,
a deployment that reserves the device up front, a path where an allocation
could stall).  It keeps its scratch in a static device array of the library
rather than a caller workspace.  Its codes, scale bytes and tensor scale must
equal nvfp4_quantize's bit for bit, call after call, since both run the same
kernel.  This file sorts last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

import nvfp4_bit_quantized_quantize_gb300 as nv
from nvfp4_bit_quantized_quantize_gb300 import synth

pytestmark = pytest.mark.gpu


def _dev(x_bits):
    return torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)


def _existing(x, rows, cols, mode, seed):
    q, sf, g = nv.alloc_quantized(rows, cols)
    ws = nv.alloc_workspace()
    nv.nvfp4_quantize(x, rows, cols, cols, mode, seed, q, sf, g, ws)
    assert nv.nvfp4_device_status(ws) == 0
    return q, sf, g


def _noalloc(x, rows, cols, mode, seed):
    q, sf, g = nv.alloc_quantized(rows, cols)
    q.fill_(0xEE)
    sf.fill_(0xEE)
    g.fill_(-1.0)
    nv.nvfp4_quantize_noalloc(x, rows, cols, cols, mode, seed, q, sf, g)
    torch.cuda.synchronize()
    return q, sf, g


@pytest.mark.parametrize("mode", [nv.RN, nv.SR])
def test_noalloc_matches_quantize_on_consecutive_calls(mode):
    shapes = [(300, 1040), (256, 256), (300, 1040)]
    for call, (rows, cols) in enumerate(shapes):
        xb = synth.normal_bf16((rows, cols), 40 + call, 0, 1.0, 0.0, 0.005, 50.0)
        x = _dev(xb)
        q1, sf1, g1 = _existing(x, rows, cols, mode, 99)
        q2, sf2, g2 = _noalloc(x, rows, cols, mode, 99)
        assert torch.equal(q1, q2), f"codes differ on call {call}"
        assert torch.equal(sf1, sf2), f"scales differ on call {call}"
        assert torch.equal(g1, g2), f"tensor scale differs on call {call}"


def test_noalloc_rejects_bad_shapes_before_launch():
    x = torch.zeros((16, 32), dtype=torch.bfloat16, device="cuda")
    q, sf, g = nv.alloc_quantized(16, 32)
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_quantize_noalloc(x, 16, 24, 32, nv.RN, 0, q, sf, g)
    assert e.value.status == 2

"""Quantization-noise meter parity ("FP4 All the Way", section "Describir":
the sqrt(3) rule compares the gradient norm with the quantization noise).

The CUDA meter forms each difference in binary32 with one fused multiply-add
and sums blocks of 16 in binary32 before binary64 totals; the oracle sums in
binary64.  Per term the binary32 path is off by a few units in 2^-24 relative
(the decode scale product, the difference, 16 partial sums), so the totals
agree to well within RTOL = 2e-5."""
import numpy as np
import pytest

import oracle as O
import nvfp4_bit_quantized_quantize_gb300 as nv
from nvfp4_bit_quantized_quantize_gb300 import synth

from gpu_helpers import quant_noise, quantize, quantize_2d

pytestmark = pytest.mark.gpu
RTOL = 2e-5


def _same(gpu, ref):
    assert gpu[0] == pytest.approx(ref[0], rel=RTOL)
    assert gpu[1] == pytest.approx(ref[1], rel=RTOL)


@pytest.mark.parametrize("mode", [nv.RN, nv.SR])
@pytest.mark.parametrize("shape", [(1, 16), (48, 80), (200, 1040), (1024, 384), (130, 2064)])
def test_noise_meter_parity(shape, mode):
    x = synth.normal_bf16(shape, 61, shape[0] % 3, 1.0, 0.0, 0.01, 30.0)
    q, sf, g, st = quantize(x, mode, seed=8)
    assert st == 0
    _same(quant_noise(x, q, sf, g), O.quant_noise(x, q, sf, g))


def test_noise_meter_leading_dimension_and_2d_form():
    w = synth.normal_bf16((160, 96), 62, 0, 0.02)
    q, sf, _, _, g, st = quantize_2d(w, transpose=False)
    assert st == 0
    _same(quant_noise(w, q, sf, g, ld=104), O.quant_noise(w, q, sf, g))


def test_noise_meter_zero_and_sqrt3_rule_inputs():
    # exactly representable tensor: zero noise on both sides
    vals = np.array([v * 0.875 for v in (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)], np.float32)
    x = np.random.default_rng(4).choice(vals, size=(64, 128)).astype(np.float32)
    x[:, ::16] = 5.25
    xb = synth.f32_to_bf16_bits(x)
    q, sf, g, _ = quantize(xb)
    se, sx = quant_noise(xb, q, sf, g)
    assert se == 0.0 and sx == pytest.approx(float((x.astype(np.float64) ** 2).sum()), rel=1e-6)


def test_noise_meter_full_size_activation():
    """The MLP input X [8192, 4096] (outlier channels), forward RN form."""
    x = synth.make_workload("mlp7b_fwd_bwd_h4096_f11008_t8192", only={"X"})["X"]
    q, sf, g, st = quantize(x)
    assert st == 0
    _same(quant_noise(x, q, sf, g), O.quant_noise(x, q, sf, g))

"""Device element encoders (the exact code paths the quantizers use) against
the oracle's nearest/stochastic rounding, on every transition point of both
formats and on random inputs."""
import numpy as np
import pytest
import torch

import oracle as O
import nvfp4_bit_quantized_quantize_gb300 as nv

pytestmark = pytest.mark.gpu


def _probe(v, r=None):
    vt = torch.from_numpy(np.ascontiguousarray(v, np.float32)).cuda()
    rt = torch.from_numpy(np.ascontiguousarray(r, np.uint16).view(np.int16)).cuda() if r is not None else None
    n = v.size
    e4 = torch.empty(n, dtype=torch.uint8, device="cuda")
    rn = torch.empty(n, dtype=torch.uint8, device="cuda")
    sr = torch.empty(n, dtype=torch.uint8, device="cuda")
    nv.nvfp4_encode_probe(vt, rt, n, e4, rn, sr)
    torch.cuda.synchronize()
    return e4.cpu().numpy(), rn.cpu().numpy(), sr.cpu().numpy()


def _around(points, k=4):
    pts = np.asarray(points, np.float32)
    out = [pts]
    lo, hi = pts.copy(), pts.copy()
    for _ in range(k):
        lo = np.nextafter(lo, np.float32(-np.inf))
        hi = np.nextafter(hi, np.float32(np.inf))
        out += [lo, hi]
    return np.concatenate(out)


def test_e4m3_encoder_matches_oracle():
    finite = np.array([O.e4m3_value(c) for c in range(0x7F)], np.float64)
    mids = (finite[1:] + finite[:-1]) / 2
    rng = np.random.default_rng(1)
    v = np.concatenate([_around(mids), _around(finite), _around([448, 464, 480, 1e30]),
                        rng.uniform(0, 500, 300000), np.exp(rng.uniform(-30, 7, 300000)),
                        np.array([0.0, np.inf, 2.0 ** -149, 2.0 ** -10, 3.4e38])]).astype(np.float32)
    v = np.abs(v)
    e4, _, _ = _probe(v)
    assert np.array_equal(e4, O.e4m3_rn_sat_many(v))


def test_e2m1_rn_encoder_matches_oracle():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    rng = np.random.default_rng(2)
    base = np.concatenate([_around(mags + mids + [6.5, 7.0, 1e6, 3e38]), rng.uniform(0, 8, 200000),
                           np.exp(rng.uniform(-20, 3, 100000)), [np.inf]]).astype(np.float32)
    v = np.concatenate([base, -base, np.array([-0.0, 0.0], np.float32)])
    _, rn, _ = _probe(v)
    assert np.array_equal(rn, O.e2m1_rn_many(v))


def test_e2m1_sr_encoder_matches_oracle():
    # every 16-bit random value on grid points, ties, near-threshold and random
    # inputs; then random (value, random value) pairs
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.uniform(-7, 7, 40), [0.25, 0.75, 1.0 + 1 / 512, 2.0, 5.9999, 6.0, -0.0, 0.0,
                                                   0.001, 3.5, 4.0 + 1 / 64, 1e9, -np.inf, 1.0 + 2 ** -17,
                                                   0.5 - 2 ** -25]]).astype(np.float32)
    v = np.repeat(vals, 65536)
    r = np.tile(np.arange(65536, dtype=np.uint16), vals.size)
    _, _, sr = _probe(v, r)
    assert np.array_equal(sr, O.e2m1_sr_many(v, r))
    v2 = rng.uniform(-6.5, 6.5, 2_000_000).astype(np.float32)
    r2 = rng.integers(0, 65536, v2.size).astype(np.uint16)
    _, _, sr2 = _probe(v2, r2)
    assert np.array_equal(sr2, O.e2m1_sr_many(v2, r2))

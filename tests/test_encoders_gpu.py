"""Device element encoders (the exact code paths the quantizers use) against
the oracle's nearest/stochastic rounding: on every transition point of both
formats and on random inputs, then on every binary32 input up to infinity."""
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


# ---------------------------------------------------------------------------
# Every binary32 input.  Each encoder below is, for a fixed random value, a
# non-decreasing function of |x| onto consecutive codes (nearest rounding with
# a fixed tie rule; stochastic rounding with a fixed random value, whose carry
# point moves up with the fraction and resets to the next grid value), and for
# non-negative binary32 the bit patterns order like the values.  So the
# oracle's whole graph over the 2^31 non-negative patterns up to +inf is the
# step function given by the first pattern of each code, found below by
# bisection on the oracle; the device is then compared with that step function
# on every pattern, and on the negative patterns (E2M1) with the sign code
# added.  NaN is left out: the quantizers report a non-finite tensor before
# anything reaches an encoder.
# ---------------------------------------------------------------------------

_INF = 0x7F800000
_CHUNK = 1 << 27


def _code_starts(fn, ncodes):
    """First pattern in [0, +inf] at which fn (patterns -> codes, the oracle)
    reaches each code 1..ncodes-1."""
    target = np.arange(1, ncodes, dtype=np.int64)
    lo = np.zeros(target.size, np.int64)
    hi = np.full(target.size, _INF, np.int64)
    assert np.all(fn(lo) < target) and np.all(fn(hi) >= target)
    while np.any(hi - lo > 1):
        mid = (lo + hi) // 2
        up = fn(mid) >= target
        hi, lo = np.where(up, mid, hi), np.where(up, lo, mid)
    # consecutive codes: each start lies below the next, and the oracle just
    # below a start gives the previous code
    assert np.all(np.diff(hi) > 0)
    assert np.array_equal(fn(hi - 1), target - 1) and np.array_equal(fn(hi), target)
    return hi


def _as_f32(patterns):
    return np.asarray(patterns, np.int64).astype(np.uint32).view(np.float32)


def _sweep(starts, probe, signed):
    """Compare probe(v) with the step function on every pattern in [0, +inf],
    and on its negation with code | 8 when signed.  Returns the number of
    patterns checked."""
    starts_t = torch.from_numpy(starts).cuda()
    done = 0
    for base in range(0, _INF + 1, _CHUNK):
        n = min(_CHUNK, _INF + 1 - base)
        pat = torch.arange(base, base + n, dtype=torch.int64, device="cuda")
        want = torch.searchsorted(starts_t, pat, right=True).to(torch.uint8)
        v = pat.to(torch.int32).view(torch.float32)
        del pat
        got = probe(v)
        bad = torch.nonzero(got != want)
        assert bad.numel() == 0, f"pattern {base + int(bad[0]):#010x}: {int(got[bad[0]])} != {int(want[bad[0]])}"
        if signed:
            got = probe(torch.neg(v))
            bad = torch.nonzero(got != (want | 8))
            assert bad.numel() == 0, f"pattern -{base + int(bad[0]):#010x}"
        done += n * (2 if signed else 1)
    torch.cuda.synchronize()
    return done


def _probe_dev(v, which, R=None):
    n = v.numel()
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    r = None if R is None else torch.full((n,), R - ((R & 0x8000) << 1), dtype=torch.int16, device="cuda")
    outs = {"e4m3": None, "rn": None, "sr": None}
    outs[which] = out
    nv.nvfp4_encode_probe(v, r, n, outs["e4m3"], outs["rn"], outs["sr"])
    return out


def test_e4m3_encoder_on_every_nonnegative_binary32():
    starts = _code_starts(lambda p: O.e4m3_rn_sat_many(_as_f32(p)), 0x7F)
    assert _sweep(starts, lambda v: _probe_dev(v, "e4m3"), signed=False) == _INF + 1


def test_e2m1_rn_encoder_on_every_binary32():
    starts = _code_starts(lambda p: O.e2m1_rn_many(_as_f32(p)), 8)
    assert _sweep(starts, lambda v: _probe_dev(v, "rn"), signed=True) == 2 * (_INF + 1)


@pytest.mark.parametrize("R", [0x0000, 0x0001, 0x7FFF, 0x8000, 0xA5C3, 0xFFFF])
def test_e2m1_sr_encoder_on_every_binary32_for_one_random_value(R):
    def oracle(p):
        v = _as_f32(p)
        return O.e2m1_sr_many(v, np.full(v.size, R, np.uint16))
    starts = _code_starts(oracle, 8)
    assert _sweep(starts, lambda v: _probe_dev(v, "sr", R), signed=True) == 2 * (_INF + 1)

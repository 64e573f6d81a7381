"""Pins for the CPU oracle, checked against what the pages and mathematics fix.

Each test ties an oracle function to something other than itself: the values
the pages print (the E2M1 value list), hand-worked examples under the stated
readings (tests/golden/worked_examples.json), an independent library
implementation of the same format (torch's float8_e4m3fn cast), closed forms,
invariants, and brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from nvfp4_bit_quantized_quantize_gb300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))

# E2M1 values listed on 'Entrenamiento de Modelos de Lenguaje con 4 Bits de
# Precision', section 'Caracteristicas del Formato NVFP4'.
PAGE_E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ------------------------------------------------------------------ E2M1 ----

def test_e2m1_value_set_is_the_pages_list():
    vals = sorted({O.e2m1_value(c) for c in range(16)})
    page = sorted({s * m for m in PAGE_E2M1_MAGNITUDES for s in (1, -1)})
    assert vals == page
    # sign is bit 3, the 8 magnitude codes are monotone
    for c in range(8):
        assert O.e2m1_value(c | 8) == -O.e2m1_value(c)
    assert [O.e2m1_value(c) for c in range(8)] == PAGE_E2M1_MAGNITUDES
    assert math.copysign(1.0, O.e2m1_value(8)) == -1.0


def test_e2m1_structure_1_sign_2_exponent_1_mantissa():
    # 1 sign, 2 exponent, 1 mantissa bit: within each exponent the two codes
    # differ by the mantissa bit and the binades double.
    for e in (1, 2, 3):
        lo = O.e2m1_value(e << 1)
        hi = O.e2m1_value((e << 1) | 1)
        assert hi == lo * 1.5
        assert O.e2m1_value((e << 1)) == 2.0 ** (e - 1)


def test_e2m1_roundtrip_all_16_codes():
    for c in range(16):
        assert O.e2m1_rn(O.e2m1_value(c)) == c
    assert O.e2m1_rn(-0.0) == 8


def test_e2m1_rn_is_nearest_on_a_sweep():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.uniform(-8, 8, 200000), rng.normal(0, 1, 100000)]).astype(np.float32)
    codes = O.e2m1_rn_many(v)
    dec = np.array([O.e2m1_value(c) for c in range(16)], np.float64)[codes]
    grid = np.array(sorted({s * m for m in PAGE_E2M1_MAGNITUDES for s in (1, -1)}))
    best = np.min(np.abs(v.astype(np.float64)[:, None] - grid[None, :]), axis=1)
    assert np.all(np.abs(dec - v) <= best + 0.0)
    # sign is kept
    assert np.all(((codes & 8) != 0) == np.signbit(v))


def test_e2m1_rn_ties_table():
    for s, code in GOLD["e2m1_rn_ties"]["cases"]:
        assert O.e2m1_rn(np.float32(float(s))) == int(code, 16), s


def test_e2m1_rn_monotone():
    v = np.linspace(0, 7, 70001, dtype=np.float32)
    mags = np.array([O.e2m1_value(c) for c in range(16)])[O.e2m1_rn_many(v)]
    assert np.all(np.diff(mags) >= 0)


# ------------------------------------------------------------ E2M1 SR ----

def _closed_form_sr_mean(a):
    """E[SR(a)] = lo + gap * floor(2^16 f) / 2^16 with f = (a - lo) / gap: the
    up-probability is the fraction kept to 16 bits."""
    grid = PAGE_E2M1_MAGNITUDES
    if a >= 6:
        return 6.0
    lo = max(g for g in grid if g <= a)
    hi = grid[grid.index(lo) + 1]
    f16 = math.floor((a - lo) / (hi - lo) * 65536)
    return lo + (hi - lo) * f16 / 65536


ALL_R = np.arange(65536, dtype=np.uint16)


def test_e2m1_sr_exact_distribution_over_all_random_values():
    # Over all 2^16 random values the up-probability is exact: the mean equals
    # the closed form, only the two neighbours occur, and on the grid nothing
    # moves.
    rng = np.random.default_rng(3)
    for a in list(rng.uniform(0, 6.5, 200)) + PAGE_E2M1_MAGNITUDES + [0.25, 0.75, 1.0 + 1 / 512, 5.999]:
        a = float(np.float32(a))
        codes = O.e2m1_sr_many(np.full(65536, a, np.float32), ALL_R)
        vals = np.array([O.e2m1_value(c) for c in np.unique(codes)])
        counts = np.array([np.sum(codes == c) for c in np.unique(codes)])
        mean = float(np.sum(vals * counts) / 65536)
        assert mean == pytest.approx(_closed_form_sr_mean(a), abs=1e-12), a
        assert len(vals) <= 2
    for m in PAGE_E2M1_MAGNITUDES:
        codes = O.e2m1_sr_many(np.full(65536, m, np.float32), ALL_R)
        assert set(O.e2m1_value(c) for c in np.unique(codes)) == {m}


def test_e2m1_sr_unbiased_where_the_fraction_has_16_bits():
    # f exact in 16 bits -> exactly unbiased: E[q] == a; and the bias never
    # exceeds one 2^-16 step of the gap
    for a in [0.25, 0.125, 1.25, 1.0 + 3 / 512, 2.5, 3.0 + 17 / 256, 5.0, 4.0 + 2 * 100 / 256, 1.0 + 2 ** -17]:
        codes = O.e2m1_sr_many(np.full(65536, a, np.float32), ALL_R)
        mean = float(np.mean([O.e2m1_value(c) for c in codes]))
        gap = 0.5 if a < 2 else (1.0 if a < 4 else 2.0)
        assert a - gap * 2 ** -16 <= mean <= a + 1e-12
        if (a * 65536 / gap) % 1 == 0:
            assert mean == pytest.approx(a, abs=1e-12)


def test_e2m1_sr_carry_rule_hand_cases():
    # 1.25 lies half way from 1 to 1.5: up exactly for R >= 2^15
    assert O.e2m1_sr(1.25, 0x7FFF) == 0x2 and O.e2m1_sr(1.25, 0x8000) == 0x3
    # 5 lies half way from 4 to 6
    assert O.e2m1_sr(5.0, 0x7FFF) == 0x6 and O.e2m1_sr(5.0, 0x8000) == 0x7
    # below 0.5 the grid step is 0.5 (from 0): 0.125 is a quarter of the way
    assert O.e2m1_sr(0.125, 0xBFFF) == 0x0 and O.e2m1_sr(0.125, 0xC000) == 0x1
    # signs are kept, also on the way to zero; 6 and beyond saturate
    assert O.e2m1_sr(-0.125, 0x0000) == 0x8 and O.e2m1_sr(-0.125, 0xFFFF) == 0x9
    assert O.e2m1_sr(7.5, 0xFFFF) == 0x7 and O.e2m1_sr(-100.0, 0) == 0xF


def test_sr_values_are_uniform_16_bit_and_use_each_word_twice():
    # every element draws 16 bits; over many blocks each element's values are
    # uniform (chi-square on 256 bins of the high byte) and the four values of
    # one word use its 32 bits exactly twice (bit counts add up)
    n = 4096
    vals = np.array([O.sr_values(11, b) for b in range(n)], np.int64)
    assert vals.max() < 65536
    for j in range(16):
        hist = np.bincount(vals[:, j] >> 8, minlength=256)
        chi2 = float(np.sum((hist - n / 256) ** 2 / (n / 256)))
        assert chi2 < 400, (j, chi2)
    pop = lambda x: bin(int(x)).count("1")
    for b in range(64):
        v = vals[b]
        w = O.philox4x32_10([b, 0, 0, 0], [11, 0])
        for m in range(4):
            assert sum(pop(v[4 * m + i]) for i in range(4)) == 2 * pop(w[m])


def test_sr_values_of_block_0_seed_0_by_hand():
    # Philox4x32-10, key (0, 0), counter (0, 0, 0, 0) is the first published
    # known-answer vector: words 6627E8D5 E169C58D BC57AC4C 9B00DBD8.  Word 0's
    # bytes, least significant first, are b0 = D5, b1 = E8, b2 = 27, b3 = 66.
    # The reading pairs them as
    #   element 0: b2 b0            = 27 D5 = 10197
    #   element 1: rev(b0) rev(b2)  = AB E4 = 44004   (rev(D5) = AB, rev(27) = E4)
    #   element 2: b3 b1            = 66 E8 = 26344
    #   element 3: rev(b1) rev(b3)  = 17 66 = 5990    (rev(E8) = 17, rev(66) = 66)
    # and word 1 = E169C58D (b0 = 8D, b1 = C5, b2 = 69, b3 = E1) gives
    #   element 4: 69 8D = 27021, element 5: B1 96 = 45462,
    #   element 6: E1 C5 = 57797, element 7: A3 87 = 41863.
    R = O.sr_values(0, 0)
    assert [int(v) for v in R[:8]] == [0x27D5, 0xABE4, 0x66E8, 0x1766, 0x698D, 0xB196, 0xE1C5, 0xA387]
    # the block index is the counter: block (2^32 + 3) uses counter (3, 1, 0, 0)
    w = O.philox4x32_10([3, 1, 0, 0], [9, 0])
    b = [(int(w[2]) >> (8 * i)) & 0xFF for i in range(4)]
    rev = lambda x: int(f"{x:08b}"[::-1], 2)
    assert [int(v) for v in O.sr_values(9, (1 << 32) + 3)[8:12]] == [
        b[2] * 256 + b[0], rev(b[0]) * 256 + rev(b[2]), b[3] * 256 + b[1], rev(b[1]) * 256 + rev(b[3])]


def test_sr_paired_elements_round_independently():
    # Elements 4m and 4m+1 (and 4m+2, 4m+3) draw their 16-bit values from the
    # same two bytes of one Philox word, once in each order and bit-reversed.
    # Their up/down decisions must still be uncorrelated: over 2^17 blocks of
    # the full quantizer, with fractions of 16 significant bits, the
    # covariance of the decisions of each such pair is within 4 sigma of 0.
    n = 1 << 17
    # block max 5.5 under tensor max 6: scale byte 416, f = rn(448/416) is not
    # a power of two, so every scaled element carries a fraction with (at
    # least) 16 significant bits between its grid neighbours
    row = np.array([5.5, 1.25, 0.75, 3.0, 1.75, 2.5, 0.375, 4.5,
                    1.125, 0.625, 2.25, 3.5, 0.875, 1.375, 2.75, 5.0], np.float32)
    x = np.tile(row, (n, 1))
    x[0, :] = 6.0
    xb = synth.f32_to_bf16_bits(x)
    q, sf, g = O.quantize(xb, O.SR, 12345)
    assert sf[O.sf_offset(1, 0, 1)] == O.e4m3_rn_sat(416.0)
    f = np.float32(448.0) / np.float32(416.0)
    v = (row * f).astype(np.float32)
    lo = np.array([max(m for m in PAGE_E2M1_MAGNITUDES if m <= a) for a in v])
    gap = np.array([0.5 if a < 2 else (1.0 if a < 4 else 2.0) for a in v])
    t = np.floor((v - lo) / gap * 65536.0)
    # strictly between grid points, and not on a 2^-8 step of the gap: the
    # decisions depend on both bytes of each element's random value
    assert np.all((t > 0) & (t < 65536) & (t % 256 != 0)), t
    codes = np.empty((n, 16), np.int64)
    codes[:, 0::2] = q & 15
    codes[:, 1::2] = q >> 4
    mags = np.array(PAGE_E2M1_MAGNITUDES)[codes[1:] & 7]
    up = (mags > lo).astype(np.float64)
    # marginal probability is the kept fraction (16 bits) of the gap
    p = up.mean(axis=0)
    sig_p = np.sqrt(t / 65536 * (1 - t / 65536) / (n - 1))
    assert np.all(np.abs(p - t / 65536) <= 4 * sig_p + 1e-12), (p, t / 65536)
    for a, b in [(4 * m + i, 4 * m + i + 1) for m in range(4) for i in (0, 2)]:
        cov = np.mean((up[:, a] - p[a]) * (up[:, b] - p[b]))
        sigma = math.sqrt(p[a] * (1 - p[a]) * p[b] * (1 - p[b]) / (n - 1))
        assert abs(cov) <= 4 * sigma, (a, b, cov, sigma)


def test_sr_unbiased_over_seeds_through_quantize():
    # Statistical pin through the full quantizer: the mean over many seeds of
    # the dequantized SR result matches the closed form within 4 sigma.
    x = np.full((1, 16), 0.0, np.float32)
    x[0, 0] = 6.0      # fixes the scales: s_enc = 448, block scale 448, f = 1
    x[0, 1:] = [0.3, 1.2, 2.7, 4.9, 0.1, 1.7, 3.3, 5.5, 0.45, 2.2, 0.8, 1.45, 3.9, 5.9, 0.6]
    xb = synth.f32_to_bf16_bits(x)
    xf = synth.bf16_bits_to_f32(xb)[0]
    n = 4000
    acc = np.zeros(16)
    sq = np.zeros(16)
    for seed in range(n):
        q, sf, g = O.quantize(xb, O.SR, seed)
        d = O.dequantize(q, sf, g, 1, 16)[0]
        acc += d
        sq += d * d
    mean = acc / n
    std = np.sqrt(np.maximum(sq / n - mean ** 2, 0)) / math.sqrt(n)
    g = 6.0 / 2688.0
    for j in range(1, 16):
        expect = _closed_form_sr_mean(float(xf[j])) * float(np.float32(g)) * 448.0
        assert abs(mean[j] - expect) <= 4 * std[j] + 1e-12, j


# ------------------------------------------------------------------ E4M3 ----

def test_e4m3_decode_matches_library_format():
    lib_vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        v = O.e4m3_value(c)
        if np.isnan(lib_vals[c]):
            assert math.isnan(v), c
        else:
            assert v == lib_vals[c], c
    assert O.e4m3_value(0x7E) == 448.0


def test_e4m3_encode_matches_library_rn_below_saturation():
    # torch's fp32 -> float8_e4m3fn cast is an independent RN-even
    # implementation; below 464 no saturation rule is involved.
    rng = np.random.default_rng(11)
    finite = np.array([O.e4m3_value(c) for c in range(0x7F)], np.float64)
    mids = (finite[1:] + finite[:-1]) / 2
    near = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9), finite])
    samples = np.concatenate([near, rng.uniform(0, 463.9, 200000),
                              np.exp(rng.uniform(-16, 6.1, 200000))]).astype(np.float32)
    samples = samples[samples < 464]
    ours = O.e4m3_rn_sat_many(samples)
    ref = torch.from_numpy(samples).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturation_and_golden():
    for s, code in GOLD["e4m3_rn_sat"]["cases"]:
        assert O.e4m3_rn_sat(float(s)) == int(code, 16), s
    big = np.array([464, 480, 1e5, 3.0e38, np.inf], np.float32)
    assert np.all(O.e4m3_rn_sat_many(big) == 0x7E)


# --------------------------------------------------------------- Philox ----

# Known-answer vectors of Philox4x32 with 10 rounds, as published with the
# method (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1,
# 2, 3", SC'11): (counter words, key words) -> output words.
PHILOX4x32_10_KAT = [
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF), (0xFFFFFFFF, 0xFFFFFFFF),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,out", PHILOX4x32_10_KAT)
def test_philox_known_answer_vectors(ctr, key, out):
    # the generator's exact bit stream: round multipliers, Weyl key schedule,
    # word order and the number of rounds all show in these three vectors
    assert [int(w) for w in O.philox4x32_10(list(ctr), list(key))] == list(out)


def test_philox_statistics():
    # uniformity and counter/key sensitivity of the bytes used for stochastic
    # rounding (the exact stream is pinned by the known-answer vectors above)
    words = np.array([O.philox4x32_10([i, 0, 0, 0], [1234, 0]) for i in range(20000)], np.uint32)
    b = words.view(np.uint8).ravel()
    counts = np.bincount(b, minlength=256)
    exp = b.size / 256
    chi2 = float(np.sum((counts - exp) ** 2 / exp))
    assert chi2 < 255 + 6 * math.sqrt(2 * 255)
    bits = np.unpackbits(words.view(np.uint8))
    assert abs(bits.mean() - 0.5) < 0.005
    a = O.philox4x32_10([5, 0, 0, 0], [1, 0])
    assert not np.array_equal(a, O.philox4x32_10([5, 0, 0, 0], [2, 0]))
    assert not np.array_equal(a, O.philox4x32_10([6, 0, 0, 0], [1, 0]))
    assert not np.array_equal(a, O.philox4x32_10([5, 0, 1, 0], [1, 0]))
    # avalanche: flipping one counter bit flips ~half the output bits
    flips = []
    for i in range(200):
        x = O.philox4x32_10([i, 7, 9, 11], [3, 4])
        y = O.philox4x32_10([i ^ 1, 7, 9, 11], [3, 4])
        flips.append(np.unpackbits((x ^ y).view(np.uint8)).sum())
    assert 56 < np.mean(flips) < 72


# ------------------------------------------------------------------ RHT ----

def _sylvester(n):
    h = np.array([[1.0]])
    while h.shape[0] < n:
        h = np.kron(np.array([[1.0, 1.0], [1.0, -1.0]]), h)
    return h


def _rht_matrix(signs):
    return np.stack([O.rht16(np.eye(16, dtype=np.float32)[j], signs) for j in range(16)], axis=1)


def test_rht_hadamard_orthogonality_and_entries():
    M = _rht_matrix(0).astype(np.float64) * 4.0          # = H16
    assert np.array_equal(np.abs(M), np.ones((16, 16)))
    assert np.array_equal(M @ M.T, 16 * np.eye(16))
    assert np.array_equal(M, _sylvester(16))            # Sylvester by Kronecker products


def test_rht_worked_examples_and_dense_equivalence():
    e0 = np.zeros(16, np.float32)
    e0[0] = 1
    assert np.array_equal(O.rht16(e0, 0), np.full(16, 0.25, np.float32))
    assert np.array_equal(O.rht16(np.ones(16, np.float32), 0), np.array([4] + [0] * 15, np.float32))
    H = _sylvester(16)
    rng = np.random.default_rng(5)
    for trial in range(200):
        s = int(rng.integers(0, 1 << 16))
        v = rng.integers(-100, 100, 16).astype(np.float32)    # exact in binary32
        D = np.diag([-1.0 if (s >> i) & 1 else 1.0 for i in range(16)])
        assert np.array_equal(O.rht16(v, s).astype(np.float64), 0.25 * H @ D @ v.astype(np.float64))


def test_rht_involution_and_norm():
    rng = np.random.default_rng(6)
    for _ in range(100):
        v = rng.normal(size=16).astype(np.float32)
        y = O.rht16(O.rht16(v, 0), 0)                      # (H/4)^2 = I
        assert np.allclose(y, v, rtol=0, atol=4e-6 * np.abs(v).max() + 1e-7)
        s = int(rng.integers(0, 1 << 16))
        assert np.linalg.norm(O.rht16(v, s)) == pytest.approx(np.linalg.norm(v), rel=1e-6)


def test_rht_signs_use_16_bits():
    seen = {O.rht_signs(s) for s in range(64)}
    assert all(0 <= x < (1 << 16) for x in seen)
    assert len(seen) > 60


def test_rht_signs_are_the_low_16_bits_of_word_0_at_counter_0010():
    # Reading: the sign diagonal of seed s is bits 0..15 of word 0 of
    # Philox4x32-10 with key (s lo, s hi) and counter (0, 0, 1, 0); a set bit
    # i negates input i.  The generator itself is pinned by the known-answer
    # vectors, so this fixes the word, the bit range and the counter.
    for seed in (0, 1, 5, 0xDEADBEEF, (7 << 32) | 3):
        w = O.philox4x32_10([0, 0, 1, 0], [seed & 0xFFFFFFFF, seed >> 32])
        assert O.rht_signs(seed) == int(w[0]) & 0xFFFF, seed
        # not word 1, not the high half, not counter (0, 0, 0, 0)
        assert O.rht_signs(seed) != int(w[1]) & 0xFFFF or O.rht_signs(seed) == 0
    # seed 0: word 0 is 0x????15E1 -> inputs 0, 5, 6, 7, 8, 10 and 12 are negated
    assert O.rht_signs(0) == 0x15E1
    assert O.rht_signs(0) != int(O.philox4x32_10([0, 0, 0, 0], [0, 0])[0]) & 0xFFFF
    e = np.eye(16, dtype=np.float32)
    cols = np.stack([O.rht16(e[i], 0x15E1) for i in range(16)])
    plain = np.stack([O.rht16(e[i], 0) for i in range(16)])
    negated = [i for i in range(16) if np.array_equal(cols[i], -plain[i])]
    assert negated == [0, 5, 6, 7, 8, 10, 12]


# --------------------------------------------------------- swizzled layout ----

@pytest.mark.parametrize("rows,cols", [(128, 64), (256, 256), (300, 80), (1, 16), (129, 1008)])
def test_sf_layout_is_a_bijection_with_512_byte_atoms(rows, cols):
    kb = cols // 16
    rp = -(-rows // 128) * 128
    kp = -(-kb // 4) * 4
    offs = np.array([[O.sf_offset(r, k, kb) for k in range(kp)] for r in range(rp)])
    assert offs.size == O.sf_bytes(rows, cols)
    assert np.array_equal(np.sort(offs.ravel()), np.arange(offs.size))
    # each 128-row x 4-block atom is one contiguous 512-byte run
    for r0 in range(0, rp, 128):
        for k0 in range(0, kp, 4):
            a = offs[r0:r0 + 128, k0:k0 + 4]
            assert a.max() - a.min() == 511
    # four consecutive blocks of one row are four consecutive bytes
    assert np.all(np.diff(offs[:, :4], axis=1) == 1)


def test_sf_layout_hand_worked_offsets():
    # 128x4 atom: row r at (r % 32) * 16 + (r // 32) * 4, block at +k
    assert O.sf_offset(0, 0, 8) == 0
    assert O.sf_offset(1, 0, 8) == 16
    assert O.sf_offset(32, 0, 8) == 4
    assert O.sf_offset(33, 3, 8) == 16 + 4 + 3
    assert O.sf_offset(0, 4, 8) == 512          # next atom along K
    assert O.sf_offset(128, 0, 8) == 1024       # next atom along rows (2 groups)
    assert O.sf_offset(127, 7, 8) == 512 + 31 * 16 + 3 * 4 + 3


# ------------------------------------------------------ worked examples ----

def _bf16(strings):
    return synth.f32_to_bf16_bits(np.array([float(s) for s in strings], np.float32))


def test_worked_example_E1():
    e = GOLD["E1"]
    x = _bf16(e["x"]).reshape(1, 16)
    assert [f"{v:04x}" for v in x[0]] == e["x_bf16_hex"]
    q, sf, g = O.quantize(x, O.RN)
    assert q.tobytes().hex() == e["packed_hex"]
    assert sf[0] == int(e["scale_byte"], 16)
    assert np.float32(g).view(np.uint32) == int(e["g_f32_hex"], 16)
    assert np.all(sf[1:] == 0)  # padding


def test_worked_example_E2():
    e1, e2 = GOLD["E1"], GOLD["E2"]
    x = np.concatenate([_bf16(e1["x"]), _bf16(e2["x"])]).reshape(1, 32)
    q, sf, g = O.quantize(x, O.RN)
    assert q[0, 8:].tobytes().hex() == e2["packed_hex"]
    assert q[0, :8].tobytes().hex() == e1["packed_hex"]
    assert sf[O.sf_offset(0, 1, 2)] == int(e2["scale_byte"], 16)


def test_worked_example_E4_gemm_closed_form():
    e1 = GOLD["E1"]
    x = _bf16(e1["x"]).reshape(1, 16)
    qa, sfa, ga = O.quantize(x, O.RN)
    qb = np.full((1, 8), 0x22, np.uint8)
    sfb = np.zeros(O.sf_bytes(1, 16), np.uint8)
    sfb[0] = 0x38
    d, dabs = O.gemm_f64(qa, sfa, ga, qb, sfb, 1.0, 1, 1, 16)
    assert d[0, 0] == float(np.float32(ga)) * 448.0 * GOLD["E4"]["sum_codes"]


def test_amax_zero_and_signed_zero():
    x = synth.f32_to_bf16_bits(np.array([[0.0] * 8 + [-0.0] * 8], np.float32))
    for mode in (O.RN, O.SR):
        q, sf, g = O.quantize(x, mode, 5)
        assert g == 0.0
        assert np.all(sf == 0)
        assert q.tobytes().hex() == "0000000088888888"


def test_nonfinite_is_an_error():
    x = synth.f32_to_bf16_bits(np.array([[1.0] * 15 + [np.inf]], np.float32))
    with pytest.raises(O.OracleError) as e:
        O.quantize(x)
    assert e.value.status == O.ERR_NONFINITE
    x[0, 15] = 0x7FC0  # NaN
    with pytest.raises(O.OracleError):
        O.quantize(x)


def test_amax_is_the_largest_magnitude():
    # max |x| by hand: the extreme is negative, in the last row and column
    x = synth.f32_to_bf16_bits(np.array([[0.5, -1.0, 2.0], [0.0, 3.0, -7.5]], np.float32))
    assert O.amax(x) == 7.5
    assert O.amax(np.zeros((2, 16), np.uint16)) == 0.0
    x[1, 2] = 0x7F80  # +Inf
    with pytest.raises(O.OracleError) as e:
        O.amax(x)
    assert e.value.status == O.ERR_NONFINITE


def test_amax_sets_the_quantizers_tensor_scale():
    # g = rn(amax / 2688) with the amax the quantizers use
    x = synth.normal_bf16((64, 48), 3, 0, 1.0, 0.0, 0.01, 50.0)
    assert O.quantize(x)[2] == float(np.float32(np.float32(O.amax(x)) / np.float32(2688.0)))
    for seed in (1, 9):
        assert O.rht_quantize(x, seed)[2] == float(np.float32(np.float32(O.rht_amax(x, seed)) / np.float32(2688.0)))


def test_rht_amax_one_hot_columns():
    # one non-zero token v_i per 16-token chunk: every output of (1/4) H16 D v
    # has magnitude |v_i| / 4 whatever the signs
    x = np.zeros((32, 3), np.float32)
    x[5, 0], x[17, 1], x[31, 2] = -12.0, 3.0, 0.5
    xb = synth.f32_to_bf16_bits(x)
    for seed in range(5):
        assert O.rht_amax(xb, seed) == 3.0


def test_rht_amax_dense_matrix_form():
    # the transform as the dense product (1/4) H16 D v in binary64 (Sylvester
    # H16, D from the seed's sign bits): the butterflies' binary32 roundings
    # stay within 2^-20 of the largest input magnitude per block
    H = _sylvester(16)
    for seed in (0, 2, 77):
        x = synth.normal_bf16((48, 5), seed, 4, 1.0)
        v = synth.bf16_bits_to_f32(x).astype(np.float64)
        s = O.rht_signs(seed)
        D = np.array([-1.0 if (s >> i) & 1 else 1.0 for i in range(16)])
        y = np.concatenate([0.25 * (H @ (D * v[16 * k:16 * k + 16, c])) for k in range(3) for c in range(5)])
        got = O.rht_amax(x, seed)
        assert abs(got - np.abs(y).max()) <= 2.0 ** -20 * np.abs(v).max() * 16


def test_single_outlier_block_scales():
    # A single outlier sets amax; its block scale is 448 and it maps to +-6.
    x = np.zeros((4, 64), np.float32)
    x[2, 37] = -1000.0
    x[0, :16] = 0.5
    xb = synth.f32_to_bf16_bits(x)
    q, sf, g = O.quantize(xb)
    lin = O.unswizzle_sf(sf, 4, 4)
    assert lin[2, 2] == 0x7E
    code = (q[2, 18] >> 4) & 15
    assert code == 0xF
    # the small block's scale: rn(rn(0.5/6) * rn(2688/1000)) -> E4M3
    s_enc = np.float32(2688) / np.float32(1000)
    sbf = (np.float32(0.5) / np.float32(6)) * s_enc
    assert lin[0, 0] == O.e4m3_rn_sat(float(sbf))


def test_all_equal_blocks_round_to_six():
    # A block of equal values c has bamax = |c|; when its E4M3 scale is a
    # normal number (448 |c| / amax >= 2^-6) the scale is within 1/16 of
    # bamax/6 (times s_enc), so c lands within [6/1.0625, 6] or above 6
    # before rounding, which round-to-nearest (midpoint 5 below, 6 the
    # largest code) always takes to +-6.  Blocks whose scale falls below the
    # E4M3 normals are left out (coarser subnormal scales, or zero).
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.uniform(-50, 50, 60), [1.0, -1.0, 2.0 ** -20, 3.0e4]]).astype(np.float32)
    x = np.repeat(vals, 16).reshape(len(vals), 16)
    x = np.concatenate([x, np.full((4, 16), 7.0e4, np.float32)])  # the tensor amax
    xb = synth.f32_to_bf16_bits(x)
    xs = synth.bf16_bits_to_f32(xb).astype(np.float64)
    q, sf, g = O.quantize(xb, O.RN)
    codes = np.stack([q & 15, (q >> 4) & 15], -1).reshape(x.shape)
    normal = np.abs(xs) * 448.0 / np.abs(xs).max() >= 2.0 ** -6 * 1.01
    expect = np.where(np.signbit(xs), 0xF, 0x7)
    assert normal.sum() > 16 * 40
    assert np.array_equal(codes[normal], expect[normal])


def test_quantize_error_bound_and_nearest():
    # The RN result is the nearest grid point to x*f (|.| <= 6) and the
    # dequantized error obeys the half-gap bound of each block.
    x = synth.normal_bf16((64, 128), 1, 0, 1.0, 0.0, 0.01, 100.0)
    q, sf, g = O.quantize(x)
    deq = O.dequantize(q, sf, g, 64, 128)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    lin = O.unswizzle_sf(sf, 64, 8)
    scale = np.array([[O.e4m3_value(b) for b in row] for row in lin]) * g   # per block
    step = np.repeat(scale, 16, axis=1)  # value of one E2M1 unit
    # largest E2M1 gap is 2 -> error <= 1 unit, plus saturation slack of the
    # block scale rounding (<= 1/16 relative of 6 units)
    assert np.all(np.abs(deq - xf) <= step * (1.0 + 6.0 / 16) + 1e-30)
    rel = np.abs(deq - xf).sum() / np.abs(xf).sum()
    assert rel < 0.12


# ------------------------------------------------------------------- 2-D ----

def test_2d_transpose_and_replicated_scales():
    w = synth.normal_bf16((48, 80), 9, 0, 0.02)
    q, sf, qT, sfT, g = O.quantize_2d(w)
    lin = O.unswizzle_sf(sf, 48, 5)
    linT = O.unswizzle_sf(sfT, 80, 3)
    for tr in range(3):
        blk = lin[tr * 16:(tr + 1) * 16]
        assert np.all(blk == blk[0])
    assert np.array_equal(linT, np.repeat(np.repeat(lin[::16].T, 16, axis=0), 1, axis=1)[:80, :3])
    # codes: qT is the exact transpose of q
    def unpack(a, cols):
        lo = a & 15
        hi = a >> 4
        return np.stack([lo, hi], axis=-1).reshape(a.shape[0], cols)
    assert np.array_equal(unpack(qT, 48), unpack(q, 80).T)


def test_2d_equals_1x16_when_rows_of_each_tile_are_equal():
    base = synth.normal_bf16((3, 64), 4, 0)
    w = np.repeat(base, 16, axis=0)         # 48 x 64, each 16-row tile constant
    q2, sf2, _, _, g2 = O.quantize_2d(w, transpose=False)
    q1, sf1, g1 = O.quantize(w)
    assert g1 == g2 and np.array_equal(q1, q2) and np.array_equal(sf1, sf2)


# ------------------------------------------------------------ RHT quantize ----

def test_rht_quantize_preserves_wgrad_product():
    # (Q dY)^T (Q X) = dY^T X for the orthogonal per-chunk transform Q; after
    # NVFP4 quantization of both transformed operands the product stays within
    # the quantization error.
    T, C1, C2 = 64, 32, 48
    dy = synth.normal_bf16((T, C1), 3, 0, 1e-3)
    x = synth.normal_bf16((T, C2), 3, 1, 1.0)
    qa, sfa, ga = O.rht_quantize(dy, 17, O.RN)
    qb, sfb, gb = O.rht_quantize(x, 17, O.RN)
    d, dabs = O.gemm_f64(qa, sfa, ga, qb, sfb, gb, C1, C2, T)
    exact = synth.bf16_bits_to_f32(dy).astype(np.float64).T @ synth.bf16_bits_to_f32(x).astype(np.float64)
    err = np.abs(d - exact).sum() / np.abs(exact).sum()
    assert err < 0.25
    # without the same signs on both sides the product is destroyed
    qb2, sfb2, gb2 = O.rht_quantize(x, 18, O.RN)
    d2, _ = O.gemm_f64(qa, sfa, ga, qb2, sfb2, gb2, C1, C2, T)
    assert np.abs(d2 - exact).sum() / np.abs(exact).sum() > 0.5


def test_rht_quantize_with_identity_signs_matches_transformed_1x16():
    # Find a seed whose sign diagonal is the identity on no lane: instead,
    # transform explicitly and compare on inputs whose transform is exact in
    # bf16 (integer inputs with few bits): RHT-quantize equals 1x16 quantize
    # of the transposed transformed tensor.
    rng = np.random.default_rng(2)
    T, C = 32, 16
    v = rng.integers(-8, 9, (T, C)).astype(np.float32)
    xb = synth.f32_to_bf16_bits(v)
    seed = 99
    s = O.rht_signs(seed)
    y = np.zeros((C, T), np.float32)
    for c in range(C):
        for k in range(T // 16):
            y[c, k * 16:(k + 1) * 16] = O.rht16(v[k * 16:(k + 1) * 16, c], s)
    yb = synth.f32_to_bf16_bits(y)
    assert np.array_equal(synth.bf16_bits_to_f32(yb), y)   # exact: quarter-integers, small
    q1, sf1, g1 = O.quantize(yb, O.RN)
    q2, sf2, g2 = O.rht_quantize(xb, seed, O.RN)
    assert g1 == g2 and np.array_equal(q1, q2) and np.array_equal(sf1, sf2)


# ------------------------------------------------------------------ GEMM ----

def test_gemm_brute_force_matches_dense_matmul_of_dequantized():
    M, N, K = 24, 40, 96
    a = synth.normal_bf16((M, K), 5, 0, 1.0, 0.0, 0.02, 50.0)
    b = synth.normal_bf16((N, K), 5, 1, 0.02)
    qa, sfa, ga = O.quantize(a)
    qb, sfb, gb = O.quantize(b)
    A = O.dequantize(qa, sfa, ga, M, K)
    B = O.dequantize(qb, sfb, gb, N, K)
    d, dabs = O.gemm_f64(qa, sfa, ga, qb, sfb, gb, M, N, K)
    ref = np.matmul(A, B.T)
    assert np.allclose(d, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.allclose(dabs, np.abs(A) @ np.abs(B).T, rtol=1e-12)
    # transposed-operand mistake would show: D^T from swapped operands
    d2, _ = O.gemm_f64(qb, sfb, gb, qa, sfa, ga, N, M, K)
    assert np.allclose(d2, d.T, rtol=1e-12)
    ms = np.array([0, 5, 23, 11])
    ns = np.array([39, 0, 7, 20])
    ds, dsa = O.gemm_f64_sampled(qa, sfa, ga, qb, sfb, gb, M, N, K, ms, ns)
    assert np.array_equal(ds, d[ms, ns]) and np.array_equal(dsa, dabs[ms, ns])


def test_gemm_quantization_error_is_small():
    M, N, K = 16, 16, 256
    a = synth.normal_bf16((M, K), 6, 0)
    b = synth.normal_bf16((N, K), 6, 1)
    qa, sfa, ga = O.quantize(a)
    qb, sfb, gb = O.quantize(b)
    d, _ = O.gemm_f64(qa, sfa, ga, qb, sfb, gb, M, N, K)
    exact = synth.bf16_bits_to_f32(a).astype(np.float64) @ synth.bf16_bits_to_f32(b).astype(np.float64).T
    assert np.abs(d - exact).max() / np.abs(exact).max() < 0.2


# ------------------------------------------------ quantization-noise meter ----
# "FP4 All the Way", section "Describir": quantized training loses efficiency
# once the gradient norm falls below about sqrt(3) times the quantization
# noise.  The meter returns (sum (Q(x) - x)^2, sum x^2).

_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_noise_meter_worked_example_E1():
    """Hand-computed from E1's printed codes, scale byte 0x7E (448) and g: the
    meter must sum the squared differences element by element."""
    e = GOLD["E1"]
    x = _bf16(e["x"]).reshape(1, 16)
    q = np.frombuffer(bytes.fromhex(e["packed_hex"]), np.uint8).reshape(1, 8)
    sf = np.zeros(O.sf_bytes(1, 16), np.uint8)
    sf[0] = int(e["scale_byte"], 16)
    g = float(np.uint32(int(e["g_f32_hex"], 16)).view(np.float32))
    xs = synth.bf16_bits_to_f32(x[0]).astype(np.float64)
    expect_e = expect_x = 0.0
    for j, c in enumerate(e["codes"]):
        c = int(c, 16)
        val = (-1.0 if c & 8 else 1.0) * _E2M1[c & 7] * 448.0 * g
        expect_e += (val - xs[j]) ** 2
        expect_x += xs[j] ** 2
    se, sx = O.quant_noise(x, q, sf, g)
    assert se == pytest.approx(expect_e, rel=1e-12)
    assert sx == pytest.approx(expect_x, rel=1e-12)
    # by hand, with 448 g taken as 1: 0.10009765625^2 + 0.2001953125^2
    # + 0.19921875^2 (0.3 -> 0.5) + 4 * 0.25^2 (0.75, 1.25, -1.75, 0.25 ties)
    # + 2 * 0.5^2 (2.5, 3.5 ties) + 1 (5 -> 4) = 1.8397858142...
    assert se == pytest.approx(1.839785814285278, rel=1e-6)


def test_noise_meter_zero_on_representable_tensor():
    """x = E2M1 value * 0.875 with amax 5.25: s_enc = 512, g = 2^-9 and every
    block scale 448 are exact, so Q(x) = x and the noise is exactly 0."""
    vals = np.array([v * 0.875 for v in _E2M1] + [-v * 0.875 for v in _E2M1], np.float32)
    rng = np.random.default_rng(3)
    x = rng.choice(vals, size=(32, 64)).astype(np.float32)
    x[:, ::16] = 5.25  # every block holds the tensor max
    xb = synth.f32_to_bf16_bits(x)
    q, sf, g = O.quantize(xb)
    assert g == 2.0 ** -9
    se, sx = O.quant_noise(xb, q, sf, g)
    assert se == 0.0
    assert sx == pytest.approx(float((x.astype(np.float64) ** 2).sum()), rel=1e-15)


def test_noise_meter_power_of_two_equivariance_and_rn_below_sr():
    """Scaling x by 2^k scales Q(x) - x by 2^k exactly (tensor scale, block
    scales and codes are unchanged), so both sums scale by 4^k exactly; and
    nearest rounding never has more noise than stochastic rounding on the same
    block scales."""
    x = synth.normal_bf16((48, 80), 9, 0, 1.0, 0.0, 0.01, 30.0)
    xf = synth.bf16_bits_to_f32(x)
    q, sf, g = O.quantize(x, O.RN)
    base = O.quant_noise(x, q, sf, g)
    for k in (-6, 3):
        xk = synth.f32_to_bf16_bits(xf * np.float32(2.0 ** k))
        qk, sfk, gk = O.quantize(xk, O.RN)
        sk = O.quant_noise(xk, qk, sfk, gk)
        assert sk[0] == base[0] * 4.0 ** k and sk[1] == base[1] * 4.0 ** k
    qs, sfs, gs = O.quantize(x, O.SR, 5)
    assert np.array_equal(sfs, sf) and gs == g
    assert O.quant_noise(x, qs, sfs, gs)[0] > base[0]
    # NVFP4 of N(0,1) data: ||x|| / ||Q(x) - x|| is well above sqrt(3)
    assert math.sqrt(base[1] / base[0]) > 5.0


# ------------------------------------------------------------------ MXFP4 ----
# The comparison format ("I ricercatori di Nvidia sbloccano ...", section
# "Come funziona NVFP4?"); conversion per the OCP Microscaling v1.0 spec.

def _mx_row_from_golden():
    e = GOLD["MX1"]
    x = np.zeros(128, np.float32)
    for b, blk in enumerate(e["blocks"]):
        for j, v in enumerate(blk["x"]):
            x[b * 32 + j] = float(v)
    return synth.f32_to_bf16_bits(x).reshape(1, 128), e


def test_mx_worked_example():
    x, e = _mx_row_from_golden()
    q, sf = O.mx_quantize(x)
    for b, blk in enumerate(e["blocks"]):
        assert q[0, b * 16:b * 16 + 8].tobytes().hex() == blk["packed_hex_first8"], b
        assert not q[0, b * 16 + 8:b * 16 + 16].any()
        assert sf[e["scale_offsets_row0"][b]] == int(blk["scale_byte"], 16), b
        assert O.mx_sf_offset(0, b, 4) == e["scale_offsets_row0"][b]
    used = set(e["scale_offsets_row0"])
    assert all(sf[i] == 0 for i in range(sf.size) if i not in used)  # padding
    d = O.mx_dequantize(q, sf, 1, 128)
    assert d[0, :7].tolist() == [6.0, -6.0, 1.0, 0.0, 4.0, 2.0, -0.0]
    assert math.copysign(1.0, d[0, 6]) == -1.0
    assert d[0, 32:35].tolist() == [0.75, 0.125, -0.25]
    assert d[0, 96] == 384.0


def test_mx_e8m0_and_layout():
    assert O.e8m0_value(127) == 1.0 and O.e8m0_value(0) == 2.0 ** -127 and O.e8m0_value(254) == 2.0 ** 127
    assert math.isnan(O.e8m0_value(255))
    # 128-row x 4-word atoms, two block scales per word in bytes 0 and 1
    offs = {O.mx_sf_offset(r, kb, 6) for r in range(256) for kb in range(6)}
    assert len(offs) == 256 * 6 and max(offs) < O.sf_bytes(256, 192)
    assert all(o % 4 in (0, 1) for o in offs)
    assert O.mx_sf_offset(33, 3, 6) == (0 * 3 + 1) * 512 + 1 * 16 + 1 * 4 + 1
    assert O.mx_sf_offset(130, 4, 6) == (1 * 3 + 2) * 512 + 2 * 16 + 0 * 4 + 0


def test_mx_power_of_two_equivariance_and_error_bound():
    """x -> 2^k x leaves the codes alone and adds k to every scale byte; every
    element not saturated is within half an E2M1 step of its block grid."""
    x = synth.normal_bf16((40, 96), 12, 0, 1.0, 0.0, 0.02, 40.0)
    q, sf = O.mx_quantize(x)
    xf = synth.bf16_bits_to_f32(x)
    for k in (-9, 5):
        qk, sfk = O.mx_quantize(synth.f32_to_bf16_bits(xf * np.float32(2.0 ** k)))
        assert np.array_equal(qk, q)
        used = np.array([O.mx_sf_offset(r, kb, 3) for r in range(40) for kb in range(3)])
        assert np.array_equal(sfk[used].astype(int), sf[used].astype(int) + k)
    d = O.mx_dequantize(q, sf, 40, 96)
    for r in range(40):
        for kb in range(3):
            blk = xf[r, kb * 32:(kb + 1) * 32].astype(np.float64)
            X = 2.0 ** math.floor(math.log2(np.abs(blk).max())) / 4.0
            v = blk / X
            got = d[r, kb * 32:(kb + 1) * 32]
            step = np.where(np.abs(v) < 2, 0.5, np.where(np.abs(v) < 4, 1.0, 2.0)) * X
            ok = np.abs(v) <= 6
            assert np.all(np.abs(got - blk)[ok] <= step[ok] / 2 + 1e-30)
            assert np.all(np.abs(got[~ok]) == 6 * X)


def test_mx_gemm_brute_force_and_nonfinite():
    M, N, K = 16, 24, 96
    a = synth.normal_bf16((M, K), 13, 0, 1.0)
    b = synth.normal_bf16((N, K), 13, 1, 0.02)
    qa, sfa = O.mx_quantize(a)
    qb, sfb = O.mx_quantize(b)
    d, dabs = O.mx_gemm_f64(qa, sfa, qb, sfb, M, N, K)
    A = O.mx_dequantize(qa, sfa, M, K)
    B = O.mx_dequantize(qb, sfb, N, K)
    assert np.allclose(d, A @ B.T, rtol=1e-12, atol=1e-15)
    assert np.allclose(dabs, np.abs(A) @ np.abs(B).T, rtol=1e-12)
    bad = a.copy()
    bad[3, 40] = 0x7FC0  # NaN
    with pytest.raises(O.OracleError):
        O.mx_quantize(bad)

"""Pins of the oracle's arithmetic building blocks against things other than itself:
IEEE formats as numpy / torch implement them, published generator outputs, exact
integer Hadamard identities, dense fp64 products, and exact rational brute force.

Passages: "Beyond Compression Ratio: High-Throughput KV Compression for
Disaggregated LLM Serving" §4.1 (randomized Hadamard, min-max quantization,
reconstruction); "KVServe: ..." §5.1 (Hadamard transformer, KIVI quantizer).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- formats
def test_f16_decode_all_patterns(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_decode_all_patterns(oracle):
    bits = np.arange(65536, dtype=np.int32).astype(np.int16)
    ref = torch.from_numpy(bits).view(torch.bfloat16).float().numpy()
    got = np.array([oracle.bf16_to_f32(int(b) & 0xFFFF) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _probe_floats(n=20000, seed=0):
    rng = np.random.default_rng(seed)
    u = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    # values around the fp16 range, subnormals, ties and the overflow edge
    extra = np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e6, -1e6,
                      2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 1.5 * 2.0 ** -24, 1.0 + 2.0 ** -11,
                      1.0 + 3 * 2.0 ** -11, 0.1, -0.1, 3.14159], np.float32)
    y = (rng.standard_normal(n) * rng.choice([1e-6, 1e-3, 1, 100, 3e4], size=n)).astype(np.float32)
    return np.concatenate([x, extra, y])


def test_f16_round_nearest_matches_numpy(oracle):
    xs = _probe_floats()
    ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16(float(x), 0) for x in xs], np.uint16)
    assert np.array_equal(got, ref)


def test_f16_directed_rounding_brackets(oracle):
    """round-down is the largest binary16 <= x, round-up the smallest >= x."""
    xs = _probe_floats(5000, 1)
    xs = xs[np.abs(xs) < 6e4]
    for x in xs:
        d = np.uint16(oracle.f32_to_f16(float(x), 1)).view(np.float16)
        u = np.uint16(oracle.f32_to_f16(float(x), 2)).view(np.float16)
        xd = float(x)
        assert float(d) <= xd <= float(u)
        assert float(np.nextafter(d, np.float16(np.inf))) > xd or float(d) == xd
        assert float(np.nextafter(u, np.float16(-np.inf))) < xd or float(u) == xd


def test_f16_directed_overflow(oracle):
    assert oracle.f32_to_f16(70000.0, 1) == 0x7BFF      # toward -inf: largest finite
    assert oracle.f32_to_f16(70000.0, 2) == 0x7C00      # toward +inf: infinity
    assert oracle.f32_to_f16(-70000.0, 1) == 0xFC00
    assert oracle.f32_to_f16(-70000.0, 2) == 0xFBFF
    assert oracle.f32_to_f16(65520.0, 0) == 0x7C00      # IEEE: the tie at 65520 rounds to infinity


def test_bf16_round_nearest_matches_torch(oracle):
    xs = _probe_floats(20000, 2)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- signs
def test_splitmix64_published_outputs(oracle):
    # SplitMix64 seeded with 0 (S. Vigna's reference generator): first three outputs
    assert oracle.splitmix64_output(0, 0) == 0xE220A8397B1DCDAF
    assert oracle.splitmix64_output(0, 1) == 0x6E789E6AA1B965F4
    assert oracle.splitmix64_output(0, 2) == 0x06C45D188009454F


def test_signs_follow_top_bit(oracle):
    s = oracle.signs(0, 3)
    assert list(s) == [-1.0, 1.0, 1.0]  # top bits of the outputs above: 1, 0, 0
    s = oracle.signs(12345, 128)
    assert set(np.unique(s)) <= {-1.0, 1.0}
    assert 40 < int((s < 0).sum()) < 88  # a fair coin over 128 draws


# ---------------------------------------------------------------- Hadamard
def _sylvester(D):
    i = np.arange(D)[:, None]
    j = np.arange(D)[None, :]
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


@pytest.mark.parametrize("D", [2, 4, 8, 16, 64, 128, 256])
def test_fwht_of_unit_vectors_is_sylvester(oracle, D):
    H = _sylvester(D)
    rows = np.stack([oracle.fwht(np.eye(D, dtype=np.float32)[i]) for i in range(D)]).astype(np.int64)
    assert np.array_equal(rows, H)
    assert np.array_equal(rows @ rows.T, D * np.eye(D, dtype=np.int64))


def test_hadamard_scale_bits(oracle):
    c = np.float32(oracle.hadamard_scale(128))
    assert c.view(np.uint32) == 0x3DB504F3
    assert abs(float(c) - 1 / math.sqrt(128)) <= 2.0 ** -28  # half an ulp at 0.088


@pytest.mark.parametrize("seed", [0, 7, 2**40 + 3])
def test_hadamard_forward_against_dense_fp64(oracle, seed):
    rng = np.random.default_rng(seed)
    D = 128
    sigma = oracle.signs(seed, D)
    H = _sylvester(D).astype(np.float64) / math.sqrt(D)
    for _ in range(20):
        x = (rng.standard_normal(D) * rng.choice([1e-3, 1, 50])).astype(np.float32)
        y = oracle.hadamard_forward(x, sigma)
        ref = H @ (sigma.astype(np.float64) * x.astype(np.float64))
        assert np.linalg.norm(y - ref) <= 1e-6 * np.linalg.norm(ref)
        # orthonormal: the norm is kept
        assert abs(np.linalg.norm(y.astype(np.float64)) - np.linalg.norm(x.astype(np.float64))) <= \
            1e-6 * np.linalg.norm(x)
        back = oracle.hadamard_inverse(y, sigma)
        assert np.linalg.norm(back - x) <= 1e-6 * np.linalg.norm(x)


def test_hadamard_inverse_against_dense_fp64(oracle):
    rng = np.random.default_rng(3)
    D = 128
    sigma = oracle.signs(99, D)
    H = _sylvester(D).astype(np.float64) / math.sqrt(D)
    y = rng.standard_normal(D).astype(np.float32)
    x = oracle.hadamard_inverse(y, sigma)
    ref = sigma.astype(np.float64) * (H @ y.astype(np.float64))
    assert np.linalg.norm(x - ref) <= 1e-6 * np.linalg.norm(ref)


# ---------------------------------------------------------------- smoothing exponent
def test_ceil_log2(oracle):
    rng = np.random.default_rng(4)
    vals = list(np.float32(2.0) ** np.arange(-126, 127, dtype=np.float64).astype(np.float32))
    vals += [float(np.nextafter(np.float32(v), np.float32(np.inf))) for v in vals[:200]]
    vals += list((rng.random(500) * 10.0 ** rng.integers(-30, 30, 500)).astype(np.float32))
    for r in vals:
        r = float(np.float32(r))
        if r <= 0:
            continue
        e = oracle.ceil_log2(r)
        assert Fraction(2) ** e >= Fraction(r)
        assert e == -126 or Fraction(2) ** (e - 1) < Fraction(r)
    assert oracle.ceil_log2(0.0) == 0
    assert oracle.ceil_log2(2.0 ** -140) == -126  # clamped to the normal range
    assert oracle.ceil_log2(3e38) == 127  # 2^128 is not finite: clamped


# ---------------------------------------------------------------- quantization
def _f16(bits):
    return float(np.uint16(bits).view(np.float16))


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_quantize_group_bounds(oracle, bits):
    rng = np.random.default_rng(bits)
    Q = 2 ** bits - 1
    for trial in range(300):
        n = int(rng.choice([1, 2, 7, 32, 64, 128]))
        y = (rng.standard_normal(n) * rng.choice([1e-4, 1e-2, 1, 30, 300]) + rng.standard_normal()).astype(np.float32)
        s_b, z_b, codes, flags = oracle.quantize_group(y, bits)
        s, z = _f16(s_b), _f16(z_b)
        mn, mx = float(y.min()), float(y.max())
        assert flags == 0
        assert codes.max() <= Q
        # z: the largest binary16 <= min
        assert z <= mn and float(np.nextafter(np.float16(z), np.float16(np.inf))) > mn
        # s: the smallest binary16 >= RN32(RN32(max - z) / Q)
        v = float(np.float32(np.float32(np.float32(mx) - np.float32(z)) / np.float32(Q)))
        assert s >= v and (s == 0 or float(np.nextafter(np.float16(s), np.float16(0))) < v)
        # the grid covers [mn, mx] and every element is within half a step (+ rounding)
        assert Fraction(z) + Q * Fraction(s) >= Fraction(mx)
        # q*s + z is exact in binary64 (8 + 11 significant bits), so one rounding to binary32 = fma
        yhat = np.array([np.float32(float(q) * s + z) for q in codes], np.float32)
        err = np.abs(yhat.astype(np.float64) - y.astype(np.float64))
        ulp = np.spacing(np.abs(y)).astype(np.float64)
        assert np.all(err <= s / 2 * (1 + 2.0 ** -20) + 2 * ulp)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_quantize_group_bruteforce_exact(oracle, bits):
    """On a dyadic grid no rounding can tip a decision, so the code must be the
    exact nearest grid point (ties to the even code), found by exhaustive search."""
    rng = np.random.default_rng(10 + bits)
    Q = 2 ** bits - 1
    for trial in range(400):
        n = int(rng.integers(2, 9))
        y = (rng.integers(-64, 64, n) / 16.0).astype(np.float32)
        s_b, z_b, codes, _ = oracle.quantize_group(y, bits)
        s, z = Fraction(_f16(s_b)), Fraction(_f16(z_b))
        for yi, qi in zip(y, codes):
            if s == 0:
                assert qi == 0
                continue
            dist = [abs(Fraction(float(yi)) - (z + q * s)) for q in range(Q + 1)]
            best = min(dist)
            cands = [q for q in range(Q + 1) if dist[q] == best]
            want = cands[0] if len(cands) == 1 else [q for q in cands if q % 2 == 0][0]
            assert qi == want, (y, yi, qi, want)


def test_signed_zero_extremes_do_not_depend_on_order(oracle):
    """A group whose minimum (or maximum) is zero gets the same metadata whichever
    signed zero comes first: the zero point of a zero minimum is +0."""
    a = np.array([-0.0, 0.0, 1.5, 0.25], np.float32)
    b = np.array([0.0, -0.0, 1.5, 0.25], np.float32)
    for bits in (2, 4):
        ra, rb = oracle.quantize_group(a, bits), oracle.quantize_group(b, bits)
        assert ra[0] == rb[0] and ra[1] == rb[1] and ra[1] == 0x0000 and np.array_equal(ra[2], rb[2])
    c = np.array([-1.0, -0.0, -2.0], np.float32)   # maximum is -0
    d = np.array([-1.0, 0.0, -2.0], np.float32)
    rc, rd = oracle.quantize_group(c, 4), oracle.quantize_group(d, 4)
    assert rc[:3][0] == rd[0] and rc[1] == rd[1] and np.array_equal(rc[2], rd[2])


def test_quantize_constant_and_range(oracle):
    s_b, z_b, codes, flags = oracle.quantize_group(np.full(16, 0.5, np.float32), 4)
    assert s_b == 0 and _f16(z_b) == 0.5 and not codes.any() and flags == 0
    _, z_b, _, flags = oracle.quantize_group(np.array([-70000.0, 1.0], np.float32), 4)
    assert flags & oracle.FLAG_RANGE and z_b == 0xFBFF
    s_b, _, codes, flags = oracle.quantize_group(np.array([0.0, 3e9], np.float32), 2)
    assert flags & oracle.FLAG_RANGE and s_b == 0x7BFF and codes[1] == 3


# ---------------------------------------------------------------- packing
def test_pack_golden(oracle):
    with open(os.path.join(GOLDEN, "pack_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = oracle.pack(np.array(c["codes"], np.uint8), c["bits"])
        assert got.tobytes().hex() == c["bytes"], c
        back = oracle.unpack(got, len(c["codes"]), c["bits"])
        assert list(back) == c["codes"]


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_pack_is_little_endian_integer(oracle, bits):
    rng = np.random.default_rng(bits)
    for n in (8, 32, 64, 128):
        codes = rng.integers(0, 2 ** bits, n).astype(np.uint8)
        val = sum(int(c) << (i * bits) for i, c in enumerate(codes))
        want = val.to_bytes(n * bits // 8, "little")
        got = oracle.pack(codes, bits)
        assert got.tobytes() == want
        assert np.array_equal(oracle.unpack(got, n, bits), codes)

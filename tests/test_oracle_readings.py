"""Hand-worked pins of two readings that change stream bytes:

* the rounding of the key-smoothing centre (binary16 round-to-nearest-even of the
  fp32 midrange, including ties both ways and negative centres), and the
  exponent that follows from it, in a block that is full and in a last block of
  40 valid rows ("KVServe" §5.1 Affine transformer, §7.3; "Beyond Compression
  Ratio" §4.1 normalization);
* the statistics of a token group that runs past the last token: minimum and
  maximum over the valid tokens only, codes past the end 0 ("Beyond Compression
  Ratio" §4.1, channel-wise key groups and the min-max rule).

Expected bytes live in tests/golden/readings_examples.json with their
derivations; they were worked out by hand, not produced by any implementation.
The GPU half runs the same inputs through the CUDA library.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "readings_examples.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _f16_bits(s):
    x = np.float16(float(Fraction(s)))
    assert float(x) == float(Fraction(s)), f"{s} is not a binary16 value"
    return np.uint16(x.view(np.uint16))


def _inputs(case):
    sh = case["shape"]
    L, T, H, D = sh["layers"], sh["tokens"], sh["kv_heads"], sh["head_dim"]
    k = np.zeros((L, T, H, D), np.uint16)
    v = np.zeros((L, T, H, D), np.uint16)
    x = k if case["tensor"] == "k" else v
    for t0, t1, h, c, val in case["fill"]:
        x[0, t0:t1, h, c] = _f16_bits(val)
    for t, h, c, val in case["set"]:
        x[0, t, h, c] = _f16_bits(val)
    if case.get("cycle"):
        t0, t1, h, c, vals = case["cycle"]
        for i, t in enumerate(range(t0, t1)):
            x[0, t, h, c] = _f16_bits(vals[i % len(vals)])
    return k, v


def _profile_kw(case):
    p = dict(case["profile"])
    p.setdefault("axis_k", 0)
    p.setdefault("axis_v", 1)
    return p


def _check_payload(case, Q, off, size):
    """Compare a payload (uint8) against the case's expected bytes; off/size = the six sections."""
    mu_sec = Q[off[4]:off[4] + size[4]].view(np.uint16)
    e_sec = Q[off[5]:off[5] + size[5]].view(np.int8)
    if "expect_mu_f16" in case:
        want_mu = np.zeros_like(mu_sec)
        want_e = np.zeros_like(e_sec)
        for cell, hx in case["expect_mu_f16"].items():
            want_mu[int(cell)] = int(hx, 16)
        for cell, e in case["expect_e"].items():
            want_e[int(cell)] = e
        bad = np.flatnonzero(mu_sec != want_mu)
        assert bad.size == 0, f"centres differ at cells {bad[:8]}: got {[hex(int(mu_sec[i])) for i in bad[:8]]}"
        bad = np.flatnonzero(e_sec != want_e)
        assert bad.size == 0, f"exponents differ at cells {bad[:8]}: got {e_sec[bad[:8]].tolist()}"
    if "expect_records" in case:
        p = case["profile"]
        rec = p["group_k"] * p["bits_k"] // 8
        codes = Q[off[0]:off[0] + size[0]]
        meta = Q[off[1]:off[1] + size[1]].view(np.uint16).reshape(-1, 2)
        for g, hx in case["expect_records"].items():
            g = int(g)
            got = codes[g * rec:(g + 1) * rec].tobytes().hex()
            assert got == hx, f"record {g}: {got} != {hx}"
        for g, (s, z) in case["expect_meta"].items():
            g = int(g)
            assert (int(meta[g, 0]), int(meta[g, 1])) == (int(s, 16), int(z, 16)), \
                f"meta {g}: {hex(int(meta[g, 0]))} {hex(int(meta[g, 1]))}"


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_oracle_matches_hand_worked_reading(oracle, case):
    sh = case["shape"]
    prof = oracle.make_profile(**_profile_kw(case))
    shape = oracle.make_shape(sh["layers"], sh["tokens"], sh["kv_heads"], sh["head_dim"], sh["dtype"])
    k, v = _inputs(case)
    Q, flags = oracle.quantize(prof, shape, k, v)
    assert flags == 0
    lay = oracle.layout(prof, shape)
    _check_payload(case, Q, list(lay.off), list(lay.size))


@pytest.mark.gpu
@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_gpu_matches_hand_worked_reading(case):
    import torch

    from kv_cache_compression_encode_gb300 import kvc
    from kv_cache_compression_encode_gb300.codec import Codec

    sh = case["shape"]
    codec = Codec(kvc.make_profile(**_profile_kw(case)),
                  kvc.make_shape(sh["layers"], sh["tokens"], sh["kv_heads"], sh["head_dim"], kvc.F16))
    k, v = _inputs(case)
    kt = [torch.from_numpy(k[0].view(np.int16)).view(torch.float16).cuda()]
    vt = [torch.from_numpy(v[0].view(np.int16)).view(torch.float16).cuda()]
    Qg = codec.quantize(kt, vt)
    st, _, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    Q = Qg.cpu().numpy().view(np.uint8)[:codec.plan.payload_bytes]
    off, size = zip(*[codec.plan.section(i) for i in range(6)])
    _check_payload(case, Q, list(off), list(size))

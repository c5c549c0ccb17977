"""Pins of the oracle's lossless stages and stream container: hand-worked examples,
exact round trips at edge lengths, permutation invariants and size closed forms.

Passage: "Beyond Compression Ratio: High-Throughput KV Compression for
Disaggregated LLM Serving", §4.2 (tuple reordering TUPL8_1, bit shuffling BIT_8,
zero-oriented encoding RZE_2; device bitstream with a compressed-size scalar).
The byte formats are format v1's readings.
"""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LENGTHS = [0, 1, 7, 8, 9, 15, 16, 17, 255, 1000, 16383, 16384, 16385]


def _payloads(n, rng):
    yield "random", rng.integers(0, 256, n, dtype=np.uint8)
    yield "zeros", np.zeros(n, np.uint8)
    yield "ones", np.full(n, 0xFF, np.uint8)
    yield "const_word", np.resize(np.array([0x12, 0x00, 0x34, 0x00], np.uint8), n)
    codes = np.clip(np.round(rng.standard_normal(n) * 1.5 + 7.5), 0, 15).astype(np.uint8)
    yield "nibbles", (codes | (np.roll(codes, 1) << 4)).astype(np.uint8)
    sparse = np.where(rng.random(n) < 0.1, rng.integers(1, 256, n), 0).astype(np.uint8)
    yield "sparse", sparse


def test_stage_golden(oracle):
    with open(os.path.join(GOLDEN, "lossless_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        data = np.frombuffer(bytes.fromhex(c["in"]), np.uint8)
        got = oracle.stage_encode(c["kind"], c["param"], data)
        assert got.tobytes().hex() == c["out"], c
        back = oracle.stage_decode(c["kind"], c["param"], got, data.size)
        assert back.tobytes() == data.tobytes(), c


STAGES = [(1, 2), (1, 4), (1, 8), (2, 8), (3, 1), (3, 2), (3, 4), (4, 1), (4, 2), (4, 4)]


@pytest.mark.parametrize("kind,param", STAGES)
def test_stage_roundtrip(oracle, kind, param):
    rng = np.random.default_rng(kind * 10 + param)
    for n in LENGTHS:
        for name, data in _payloads(n, rng):
            enc = oracle.stage_encode(kind, param, data)
            if kind != 4:
                assert enc.size == n  # length-preserving stages
            back = oracle.stage_decode(kind, param, enc, n)
            assert back is not None and back.tobytes() == data.tobytes(), (kind, param, n, name)


@pytest.mark.parametrize("k", [2, 4, 8])
def test_tupl_is_a_byte_permutation(oracle, k):
    rng = np.random.default_rng(k)
    data = rng.integers(0, 256, 1003, dtype=np.uint8)
    enc = oracle.stage_encode(1, k, data)
    assert np.array_equal(np.sort(enc), np.sort(data))
    m = data.size // k
    # column j of the tuple matrix is contiguous in the output
    for j in range(k):
        assert np.array_equal(enc[j * m:(j + 1) * m], data[:m * k].reshape(m, k)[:, j])


def test_bit_shuffle_is_a_bit_permutation(oracle):
    rng = np.random.default_rng(5)
    data = rng.integers(0, 256, 4099, dtype=np.uint8)
    enc = oracle.stage_encode(2, 8, data)
    assert int(np.unpackbits(enc).sum()) == int(np.unpackbits(data).sum())
    n8 = data.size // 8 * 8
    planes = np.unpackbits(enc[:n8].reshape(8, -1), axis=1, bitorder="little")
    bits = np.unpackbits(data[:n8, None], axis=1, bitorder="little")  # [byte][plane]
    assert np.array_equal(planes, bits.T)


@pytest.mark.parametrize("w", [1, 2, 4])
def test_rze_size_closed_form(oracle, w):
    rng = np.random.default_rng(w)
    for n in [0, 5, 64, 1001, 16384]:
        for name, data in _payloads(n, rng):
            m = n // w
            words = data[:m * w].reshape(m, w) if m else np.zeros((0, w), np.uint8)
            nz = words.any(axis=1)
            B = np.packbits(nz, bitorder="little")
            nb = (m + 7) // 8
            B = B[:nb]
            nb2 = (nb + 7) // 8
            want = nb2 + int((B != 0).sum()) + w * int(nz.sum()) + (n - m * w)
            assert oracle.stage_encode(4, w, data).size == want, (name, n)


def test_rze_all_zero_chunk_is_minimal(oracle):
    out = oracle.stage_encode(4, 1, np.zeros(16384, np.uint8))
    assert out.size == 256 and not out.any()  # only B2 remains (2048 bitmap bytes -> 256)
    out = oracle.stage_encode(4, 2, np.zeros(16384, np.uint8))
    assert out.size == 128 and not out.any()


def test_rze_rejects_inconsistent_input(oracle):
    data = np.frombuffer(bytes.fromhex("0005000007000000000000000000000009"), np.uint8)
    enc = oracle.stage_encode(4, 1, data)
    assert oracle.stage_decode(4, 1, enc[:-1], data.size) is None   # truncated
    assert oracle.stage_decode(4, 1, np.concatenate([enc, [0]]).astype(np.uint8), data.size) is None  # trailing
    bad = enc.copy()
    bad[0] |= 0x02  # claims a nonzero bitmap byte that is not there
    assert oracle.stage_decode(4, 1, bad, data.size) is None


PIPELINES = [((1, 8), (4, 1)), ((1, 8), (2, 8), (4, 2)), ((1, 8), (2, 8), (3, 1), (4, 2)), ((3, 2), (4, 2)),
             ((1, 4),), ((2, 8), (3, 4))]


@pytest.mark.parametrize("stages", PIPELINES)
def test_chunk_roundtrip_and_raw_fallback(oracle, stages):
    prof = oracle.make_profile(stages=stages)
    rng = np.random.default_rng(len(stages))
    for n in [1, 8, 16, 1024, 16384]:
        for name, data in _payloads(n, rng):
            stored, raw = oracle.chunk_encode(prof, data)
            assert stored.size <= n
            if raw:
                assert stored.tobytes() == data.tobytes()
            else:
                assert stored.size < n
            back = oracle.chunk_decode(prof, stored, raw, n)
            assert back is not None and back.tobytes() == data.tobytes(), (name, n)
    stored, raw = oracle.chunk_encode(prof, rng.integers(0, 256, 16384, dtype=np.uint8))
    assert raw  # random bytes do not compress
    if stages[-1][0] == 4:
        stored, raw = oracle.chunk_encode(prof, np.zeros(16384, np.uint8))
        assert not raw and stored.size < 300


def _shape(oracle, L, T, H=2, D=128, dtype=2):
    return oracle.make_shape(L, T, H, D, dtype)


@pytest.mark.parametrize("stages,chunk", [((), 16384), (((1, 8), (4, 1)), 16384),
                                          (((1, 8), (2, 8), (4, 2)), 1024), (((1, 8), (2, 8), (3, 1), (4, 2)), 4096)])
def test_stream_roundtrip_and_container(oracle, stages, chunk):
    prof = oracle.make_profile(stages=stages, chunk_bytes=chunk)
    shape = _shape(oracle, 2, 200)
    lay = oracle.layout(prof, shape)
    rng = np.random.default_rng(chunk)
    Q = np.where(rng.random(lay.payload_bytes) < 0.3, rng.integers(0, 256, lay.payload_bytes), 0).astype(np.uint8)
    stream = oracle.lossless_encode(prof, shape, Q)
    assert stream[:4].tobytes() == b"KVC1"
    assert stream.size <= lay.max_stream_bytes
    Q2, flags = oracle.lossless_decode(prof, shape, stream)
    assert flags == 0 and np.array_equal(Q2, Q)
    if stages:
        n = lay.n_chunks
        assert n == -(-lay.payload_bytes // chunk)
        table = stream[64:64 + 4 * n].view(np.uint32)
        sizes = table & 0x7FFFFFFF
        total = lay.data_start + int(((sizes + 15) // 16 * 16).sum())
        assert stream.size == total
        assert lay.data_start == (64 + 4 * n + 15) // 16 * 16
    else:
        assert stream.size == 64 + lay.payload_bytes
        assert np.array_equal(stream[64:], Q)


def test_stream_corruption_is_detected(oracle):
    prof = oracle.make_profile(stages=((1, 8), (2, 8), (4, 2)), chunk_bytes=1024)
    shape = _shape(oracle, 1, 300)
    lay = oracle.layout(prof, shape)
    rng = np.random.default_rng(1)
    Q = np.where(rng.random(lay.payload_bytes) < 0.2, 7, 0).astype(np.uint8)
    stream = oracle.lossless_encode(prof, shape, Q)
    assert oracle.lossless_decode(prof, shape, stream)[1] == 0
    for mutate in ("magic", "bits", "truncate", "table_grow", "table_raw", "body"):
        s = stream.copy()
        if mutate == "magic":
            s[0] = ord("X")
        elif mutate == "bits":
            s[22] = 3
        elif mutate == "truncate":
            s = s[:-17]
        elif mutate == "table_grow":
            s[64:68] = np.frombuffer(np.uint32(s[64:68].view(np.uint32)[0] + 1).tobytes(), np.uint8)
        elif mutate == "table_raw":
            s[67] ^= 0x80
        elif mutate == "body":
            s[lay.data_start] ^= 0x01  # the first B2 byte now lists a bitmap byte that is missing
        assert oracle.lossless_decode(prof, shape, s)[1] & oracle.FLAG_CORRUPT, mutate

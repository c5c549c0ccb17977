"""Pins of the oracle's whole path (BS = C(Q(T(X))), "KVServe: ..." §5.1):
payload size closed forms (including the 2-bit KIVI ceiling of 16/3 in "KVServe"
§7.3), layout index pins with single planted elements, reconstruction error
bounds in the original domain, paged = contiguous, ragged and empty inputs, and
invariance to the oracle's thread count.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from kv_cache_compression_encode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits_to_f32(a, dtype):
    a = np.asarray(a, np.uint16)
    if dtype == 1:
        return a.view(np.float16).astype(np.float32)
    return (a.astype(np.uint32) << 16).view(np.float32)


def _f32_to_bits(x, dtype):
    x = np.asarray(x, np.float32)
    if dtype == 1:
        return x.astype(np.float16).view(np.uint16)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rand_kv(L, T, H, D, dtype, seed, scale=1.0, offset=0.0):
    rng = np.random.default_rng(seed)
    k = (rng.standard_normal((L, T, H, D)) * scale + offset).astype(np.float32)
    v = rng.standard_normal((L, T, H, D)).astype(np.float32)
    return _f32_to_bits(k, dtype), _f32_to_bits(v, dtype)


# ----------------------------------------------------------------- sizes
@pytest.mark.parametrize("T", [32, 256, 4096])
def test_kivi_2bit_group32_ratio_is_16_over_3(oracle, T):
    prof = oracle.make_profile(smooth_keys=False, bits_k=2, bits_v=2, group_k=32, group_v=32)
    shape = oracle.make_shape(2, T, 8, 128, 1)
    lay = oracle.layout(prof, shape)
    raw = 2 * 2 * T * 8 * 128 * 2
    assert raw * 3 == lay.payload_bytes * 16  # CR = 16 / 3 = 5.33x exactly


def test_payload_closed_form_llama8b(oracle):
    # 32 layers x 4096 tokens x 8 heads x 128, 4-bit group 128, smoothing on
    prof = oracle.make_profile(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128)
    shape = oracle.make_shape(32, 4096, 8, 128, 2)
    lay = oracle.layout(prof, shape)
    codes = 32 * 4096 * 8 * 128 // 2                 # 4 bits per element, K and V each
    meta = 32 * 4096 * 8 * 128 // 128 * 4            # 4 bytes per group of 128
    smooth = 32 * 8 * (4096 // 128) * 128 * 3        # centre (2 B) + exponent (1 B) per cell
    assert list(lay.size) == [codes, meta, codes, meta, smooth // 3 * 2, smooth // 3, 0, 0]
    assert lay.payload_bytes == 2 * codes + 2 * meta + smooth


def test_sections_are_16_byte_aligned_and_ordered(oracle):
    prof = oracle.make_profile(bits_k=3, bits_v=3, group_k=32, group_v=32)
    shape = oracle.make_shape(1, 37, 3, 128, 2)
    lay = oracle.layout(prof, shape)
    for i in range(8):
        assert lay.off[i] % 16 == 0
        if i:
            assert lay.off[i] == lay.off[i - 1] + (lay.size[i - 1] + 15) // 16 * 16
    assert lay.size[0] == 1 * 3 * 2 * 128 * 12      # ceil(37/32) token groups, 12-byte records
    assert lay.size[2] == 1 * 37 * 3 * 4 * 12       # 4 channel groups per row
    assert lay.size[4] == 3 * 1 * 128 * 2 and lay.size[5] == 3 * 128


# ----------------------------------------------------------------- index pins
def test_key_record_order_layer_head_tokengroup_channel(oracle):
    L, T, H, D = 2, 96, 3, 128
    prof = oracle.make_profile(smooth_keys=False, hadamard=False, bits_k=4, bits_v=4, group_k=32, group_v=32)
    shape = oracle.make_shape(L, T, H, D, 2)
    k = np.zeros((L, T, H, D), np.uint16)
    v = np.zeros((L, T, H, D), np.uint16)
    k[1, 37, 2, 5] = _f32_to_bits(np.float32(1.0), 2)
    Q, flags = oracle.quantize(prof, shape, k, v)
    lay = oracle.layout(prof, shape)
    assert flags == 0
    nTG = 3
    g = ((1 * H + 2) * nTG + 1) * D + 5             # [l][h][tg][c]
    meta = Q[lay.off[1]:lay.off[1] + lay.size[1]].view(np.uint16).reshape(-1, 2)
    nz = np.nonzero(meta.any(axis=1))[0]
    assert list(nz) == [g]
    assert float(np.uint16(meta[g, 1]).view(np.float16)) == 0.0          # zero point
    codes = Q[lay.off[0]:lay.off[0] + lay.size[0]].reshape(-1, 16)
    rec = oracle.unpack(codes[g], 32, 4)
    assert rec[37 - 32] == 15 and rec.sum() == 15
    assert np.count_nonzero(codes) == 1


def test_value_record_order_layer_token_head_channelgroup(oracle):
    L, T, H, D = 2, 10, 3, 128
    prof = oracle.make_profile(smooth_keys=False, hadamard=False, bits_k=4, bits_v=2, group_k=32, group_v=32)
    shape = oracle.make_shape(L, T, H, D, 2)
    k = np.zeros((L, T, H, D), np.uint16)
    v = np.zeros((L, T, H, D), np.uint16)
    v[0, 3, 1, 70] = _f32_to_bits(np.float32(-2.0), 2)
    Q, _ = oracle.quantize(prof, shape, k, v)
    lay = oracle.layout(prof, shape)
    g = ((0 * T + 3) * H + 1) * (D // 32) + 2       # [l][t][h][cg]
    meta = Q[lay.off[3]:lay.off[3] + lay.size[3]].view(np.uint16).reshape(-1, 2)
    assert list(np.nonzero(meta.any(axis=1))[0]) == [g]
    assert float(np.uint16(meta[g, 1]).view(np.float16)) == -2.0
    rec = oracle.unpack(Q[lay.off[2] + g * 8:lay.off[2] + g * 8 + 8], 32, 2)
    assert rec[6] == 0 and all(rec[i] == 3 for i in range(32) if i != 6)


def test_smoothing_cells_order(oracle):
    L, T, H, D = 1, 300, 2, 128
    prof = oracle.make_profile(smooth_keys=True, bits_k=8, bits_v=8, group_k=32, group_v=32)
    shape = oracle.make_shape(L, T, H, D, 2)
    k = np.zeros((L, T, H, D), np.uint16)
    v = np.zeros((L, T, H, D), np.uint16)
    k[0, 260, 1, 9] = _f32_to_bits(np.float32(6.0), 2)    # block 2 of head 1, channel 9
    Q, _ = oracle.quantize(prof, shape, k, v)
    lay = oracle.layout(prof, shape)
    mu = Q[lay.off[4]:lay.off[4] + lay.size[4]].view(np.uint16)
    e = Q[lay.off[5]:lay.off[5] + lay.size[5]].view(np.int8)
    cell = ((0 * H + 1) * 3 + 2) * D + 9
    assert list(np.nonzero(mu)[0]) == [cell] and float(np.uint16(mu[cell]).view(np.float16)) == 3.0
    assert list(np.nonzero(e)[0]) == [cell] and e[cell] == 2    # r = 3 -> 2^2 >= 3


# ----------------------------------------------------------------- error bounds
def _meta(Q, lay, sec):
    m = Q[lay.off[sec]:lay.off[sec] + lay.size[sec]].view(np.uint16).reshape(-1, 2)
    return m[:, 0].view(np.float16).astype(np.float64), m[:, 1].view(np.float16).astype(np.float64)


@pytest.mark.parametrize("dtype", [1, 2])
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_reconstruction_bound_plain(oracle, dtype, bits):
    """No transform: every element within half a step of its group (+ output rounding)."""
    L, T, H, D, G = 1, 70, 2, 128, 32
    prof = oracle.make_profile(smooth_keys=False, hadamard=False, bits_k=bits, bits_v=bits, group_k=G, group_v=G)
    shape = oracle.make_shape(L, T, H, D, dtype)
    k, v = _rand_kv(L, T, H, D, dtype, bits)
    stream, flags = oracle.encode(prof, shape, k, v)
    assert flags == 0
    ok, ov = np.zeros_like(k), np.zeros_like(v)
    assert oracle.decode(prof, shape, stream, ok, ov) == 0
    Q, _ = oracle.quantize(prof, shape, k, v)
    lay = oracle.layout(prof, shape)
    half_ulp = 2.0 ** -11 if dtype == 1 else 2.0 ** -8
    # keys: groups over tokens, records [l][h][tg][c]
    sk, _ = _meta(Q, lay, 1)
    sk = sk.reshape(L, H, -1, D)
    xk, rk = _bits_to_f32(k, dtype), _bits_to_f32(ok, dtype)
    for t in range(T):
        bound = sk[:, :, t // G, :] / 2 * (1 + 2.0 ** -20)
        err = np.abs(rk[:, t].astype(np.float64) - xk[:, t])
        assert np.all(err <= bound + np.abs(rk[:, t]) * half_ulp * 1.01 + 1e-7)  # output rounding of y^
    sv, _ = _meta(Q, lay, 3)
    sv = np.repeat(sv.reshape(L, T, H, D // G), G, axis=3)
    xv, rv = _bits_to_f32(v, dtype), _bits_to_f32(ov, dtype)
    err = np.abs(rv.astype(np.float64) - xv)
    assert np.all(err <= sv / 2 * (1 + 2.0 ** -20) + np.abs(rv) * half_ulp * 1.01 + 1e-7)


def test_reconstruction_bound_hadamard_and_smoothing(oracle):
    """With the rotation the row error is bounded in the 2-norm (orthonormality); with
    smoothing each channel's error is scaled by its 2^e."""
    L, T, H, D, G = 1, 130, 2, 128, 64
    dtype = 2
    prof = oracle.make_profile(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=G, group_v=G,
                               stages=((1, 8), (2, 8), (4, 2)))
    shape = oracle.make_shape(L, T, H, D, dtype)
    k, v = _rand_kv(L, T, H, D, dtype, 77, scale=3.0, offset=1.5)
    stream, flags = oracle.encode(prof, shape, k, v)
    assert flags == 0
    ok, ov = np.zeros_like(k), np.zeros_like(v)
    assert oracle.decode(prof, shape, stream, ok, ov) == 0
    Q, _ = oracle.quantize(prof, shape, k, v)
    lay = oracle.layout(prof, shape)
    # values: groups of G channels per token after the rotation
    sv, _ = _meta(Q, lay, 3)
    sv = np.repeat(sv.reshape(L, T, H, D // G), G, axis=3)
    xv, rv = _bits_to_f32(v, dtype).astype(np.float64), _bits_to_f32(ov, dtype).astype(np.float64)
    row_err = np.linalg.norm(rv - xv, axis=-1)
    row_bound = np.sqrt(((sv / 2) ** 2).sum(axis=-1)) * 1.0001 + np.linalg.norm(rv, axis=-1) * 2.0 ** -8
    assert np.all(row_err <= row_bound)
    # keys: rotate back the per-channel step bound, then scale per channel by 2^e
    sk, _ = _meta(Q, lay, 1)
    sk = sk.reshape(L, H, -1, D)
    e = Q[lay.off[5]:lay.off[5] + lay.size[5]].view(np.int8).reshape(L, H, -1, D).astype(np.float64)
    xk, rk = _bits_to_f32(k, dtype).astype(np.float64), _bits_to_f32(ok, dtype).astype(np.float64)
    for t in range(T):
        step = sk[:, :, t // G, :] / 2                 # per rotated channel
        scale = 2.0 ** e[:, :, t // 128, :]
        rot = np.sqrt((step ** 2).sum(axis=-1, keepdims=True))   # 2-norm of the rotated-domain error
        bound = rot * scale * 1.0001 + np.abs(rk[:, t]) * 2.0 ** -8 + scale * 1e-6
        assert np.all(np.abs(rk[:, t] - xk[:, t]) <= bound)


# ----------------------------------------------------------------- structure
def test_paged_equals_contiguous(oracle):
    L, T, H, D, P = 2, 100, 2, 128, 16
    prof = oracle.make_profile(hadamard=True, bits_k=4, bits_v=3, group_k=32, group_v=64, stages=((1, 8), (2, 8), (4, 2)))
    k, v = _rand_kv(L, T, H, D, 2, 5)
    shape = oracle.make_shape(L, T, H, D, 2)
    ref, f0 = oracle.encode(prof, shape, k, v)
    n_pages = -(-T // P)
    bt = np.random.default_rng(0).permutation(n_pages).astype(np.int32)
    kp = np.zeros((L, n_pages, P, H, D), np.uint16)
    vp = np.zeros_like(kp)
    for lp in range(n_pages):
        n = min(P, T - lp * P)
        kp[:, bt[lp], :n] = k[:, lp * P:lp * P + n]
        vp[:, bt[lp], :n] = v[:, lp * P:lp * P + n]
    pshape = oracle.make_shape(L, T, H, D, 2, page_size=P, page_stride=P * H * D * 2)
    got, f1 = oracle.encode(prof, pshape, kp, vp, block_table=bt)
    assert f0 == f1 == 0 and np.array_equal(got, ref)
    ok, ov = np.zeros_like(kp), np.zeros_like(vp)
    assert oracle.decode(prof, pshape, got, ok, ov, block_table=bt) == 0
    ck, cv = np.zeros_like(k), np.zeros_like(v)
    assert oracle.decode(prof, shape, ref, ck, cv) == 0
    for lp in range(n_pages):
        n = min(P, T - lp * P)
        assert np.array_equal(ok[:, bt[lp], :n], ck[:, lp * P:lp * P + n])


@pytest.mark.parametrize("T", [0, 1, 33, 129])
def test_ragged_and_empty(oracle, T):
    L, H, D = 1, 2, 128
    prof = oracle.make_profile(hadamard=True, bits_k=3, bits_v=4, group_k=64, group_v=32, stages=((1, 8), (4, 1)))
    shape = oracle.make_shape(L, T, H, D, 1)
    k, v = _rand_kv(L, T, H, D, 1, T)
    stream, flags = oracle.encode(prof, shape, k, v)
    assert flags == 0 and stream[:4].tobytes() == b"KVC1"
    ok, ov = np.zeros_like(k), np.zeros_like(v)
    assert oracle.decode(prof, shape, stream, ok, ov) == 0
    if T:
        err = np.abs(_bits_to_f32(ov, 1) - _bits_to_f32(v, 1))
        assert err.max() < 1.0


def test_nonfinite_input_flag(oracle):
    L, T, H, D = 1, 40, 1, 128
    prof = oracle.make_profile()
    shape = oracle.make_shape(L, T, H, D, 2)
    k, v = _rand_kv(L, T, H, D, 2, 1)
    v[0, 5, 0, 3] = 0x7FC0  # NaN
    _, flags = oracle.encode(prof, shape, k, v)
    assert flags & oracle.FLAG_NONFINITE


def test_thread_count_does_not_change_bytes(oracle):
    L, T, H, D = 3, 300, 4, 128
    prof = oracle.make_profile(hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128,
                               stages=((1, 8), (2, 8), (3, 1), (4, 2)), chunk_bytes=2048)
    shape = oracle.make_shape(L, T, H, D, 2)
    k, v = _rand_kv(L, T, H, D, 2, 9)
    old = oracle.set_threads(0)
    try:
        oracle.set_threads(1)
        a, _ = oracle.encode(prof, shape, k, v)
        oracle.set_threads(4)
        b, _ = oracle.encode(prof, shape, k, v)
    finally:
        oracle.set_threads(old)
    assert np.array_equal(a, b)


def test_tiny_workload_digest(oracle):
    """Regression pin across machines: the digests were written by
    tests/golden/make_oracle_digests.py, which calls only the oracle."""
    import hashlib
    from tests.golden.make_oracle_digests import digest_cases
    with open(os.path.join(GOLDEN, "oracle_digests.json")) as f:
        want = json.load(f)["digests"]
    got = digest_cases()
    assert got == want

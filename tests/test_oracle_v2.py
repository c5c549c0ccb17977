"""Pins of the oracle's format-v2 features, checked against things other than the
oracle itself:

* per-(layer, head) code widths ("KVServe" §5.1: mixed precision at layer and
  head granularity; "Beyond Compression Ratio" §4.1: head-importance-aware mixed
  precision): every (layer, head)'s records in a mixed payload equal that head's
  records in a payload quantized with its width everywhere (relocated by the
  layout's closed-form offsets, written out here); the size closed form; a
  hand-worked header with its 2-bit width map;
* the token-delta transformer ("KVServe" §5.1 "Delta", after CacheGen): anchor
  cells hold the element bits of each block's first token; small-integer inputs
  whose deltas span exactly [0, 255] give codes equal to the deltas (which fixes
  the sign x - anchor) and reconstruct exactly; with smoothing and Hadamard the
  reconstruction stays within the quantization bound.
"""
import numpy as np
import pytest

D = 128


def _f16(x):
    return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def _rand_bits(shape, seed, dtype=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32) * 2.0 + 0.5
    if dtype == 1:
        return x.astype(np.float16).view(np.uint16)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _v1_record(Q, lay, tensor, axis, L, T, H, G, b, l, h, idx):
    """Records of (l, h) in a uniform-width (v1) payload, by the v1 index formulas."""
    sec = Q[lay.off[2 * tensor]:lay.off[2 * tensor] + lay.size[2 * tensor]]
    rec = G * b // 8
    if axis == 0:
        ntg = -(-T // G)
        g = ((l * H + h) * ntg + idx[0]) * D + idx[1]
    else:
        g = ((l * T + idx[0]) * H + h) * (D // G) + idx[1]
    return sec[g * rec:(g + 1) * rec]


def _v2_record(Q, lay, tensor, axis, T, H, G, widths, l, h, idx):
    """Records of (l, h) in a mixed payload by the v2 layout written out: blocks of
    (layer, head) back to back (groups over tokens), or rows whose heads have their
    own widths (groups over channels)."""
    sec = Q[lay.off[2 * tensor]:lay.off[2 * tensor] + lay.size[2 * tensor]]
    b = int(widths[l, h])
    rec = G * b // 8
    if axis == 0:
        ntg = -(-T // G)
        block = lambda w: ntg * D * G * int(w) // 8  # noqa: E731
        base = sum(block(widths[l2, h2]) for l2 in range(widths.shape[0]) for h2 in range(H) if (l2, h2) < (l, h))
        o = base + (idx[0] * D + idx[1]) * rec
    else:
        rowb = lambda l2: sum(D * int(w) // 8 for w in widths[l2])  # noqa: E731
        base = sum(T * rowb(l2) for l2 in range(l)) + idx[0] * rowb(l) + sum(D * int(w) // 8 for w in widths[l, :h])
        o = base + idx[1] * rec
    return sec[o:o + rec]


@pytest.mark.parametrize("axis_k,axis_v", [(0, 1), (1, 0)])
@pytest.mark.parametrize("smooth,had", [(False, False), (True, True)])
def test_mixed_widths_equal_uniform_per_head(oracle, axis_k, axis_v, smooth, had):
    L, T, H, G = 2, 200, 4, 32
    rng = np.random.default_rng(5)
    wk = rng.choice([2, 3, 4, 8], size=(L, H)).astype(np.uint8)
    wv = rng.choice([2, 3, 4, 8], size=(L, H)).astype(np.uint8)
    wk[0, 0], wk[0, 1], wv[1, 2], wv[1, 3] = 2, 8, 8, 2  # both extremes in one layer / one token row
    k = _rand_bits((L, T, H, D), 1)
    v = _rand_bits((L, T, H, D), 2)
    shape = oracle.make_shape(L, T, H, D, 2)
    kw = dict(smooth_keys=smooth, hadamard=had, group_k=G, group_v=G, axis_k=axis_k, axis_v=axis_v)
    pm = oracle.make_profile(bits_k=4, bits_v=4, bits_map_k=wk, bits_map_v=wv, **kw)
    Qm, fm = oracle.quantize(pm, shape, k, v)
    lm = oracle.layout(pm, shape)
    assert fm == 0
    uni = {}
    for b in (2, 3, 4, 8):
        pu = oracle.make_profile(bits_k=b, bits_v=b, **kw)
        uni[b] = (oracle.quantize(pu, shape, k, v)[0], oracle.layout(pu, shape))
    for tensor, axis, W in ((0, axis_k, wk), (1, axis_v, wv)):
        for l in range(L):
            for h in range(H):
                b = int(W[l, h])
                Qb, lb = uni[b]
                idxs = [(tg, c) for tg in range(-(-T // G)) for c in (0, 37, 127)] if axis == 0 else \
                       [(t, cg) for t in (0, 1, 99, T - 1) for cg in range(D // G)]
                for idx in idxs:
                    got = _v2_record(Qm, lm, tensor, axis, T, H, G, W, l, h, idx)
                    want = _v1_record(Qb, lb, tensor, axis, L, T, H, G, b, l, h, idx)
                    assert np.array_equal(got, want), (tensor, l, h, idx)
                # metadata words sit where v1 puts them (4 bytes per group, whatever the width)
                mm = Qm[lm.off[2 * tensor + 1]:lm.off[2 * tensor + 1] + lm.size[2 * tensor + 1]].view(np.uint32)
                mb = Qb[lb.off[2 * tensor + 1]:lb.off[2 * tensor + 1] + lb.size[2 * tensor + 1]].view(np.uint32)
                if axis == 0:
                    ntg = -(-T // G)
                    sl = slice((l * H + h) * ntg * D, (l * H + h + 1) * ntg * D)
                    assert np.array_equal(mm[sl], mb[sl]), (tensor, l, h)
                else:
                    grid_m = mm.reshape(L, T, H, D // G)
                    grid_b = mb.reshape(L, T, H, D // G)
                    assert np.array_equal(grid_m[l, :, h], grid_b[l, :, h]), (tensor, l, h)
    # the smoothing sections do not depend on the widths
    Qb, lb = uni[4]
    for sec in (4, 5):
        assert np.array_equal(Qm[lm.off[sec]:lm.off[sec] + lm.size[sec]],
                              Qb[lb.off[sec]:lb.off[sec] + lb.size[sec]]), sec


def test_mixed_width_sizes_closed_form(oracle):
    L, T, H, G = 3, 300, 8, 64
    wk = np.array([[2, 8, 4, 4, 3, 3, 2, 8]] * L, np.uint8)
    wv = np.full((L, H), 3, np.uint8)
    wv[2] = 8
    p = oracle.make_profile(smooth_keys=True, bits_map_k=wk, bits_map_v=wv, group_k=G, group_v=G)
    lay = oracle.layout(p, oracle.make_shape(L, T, H, D, 2))
    ntg = -(-T // G)
    assert lay.size[0] == sum(ntg * D * G * int(b) // 8 for b in wk.flat)
    assert lay.size[2] == sum(T * D * int(b) // 8 for b in wv.flat)
    assert lay.size[1] == L * H * ntg * D * 4 and lay.size[3] == L * T * H * (D // G) * 4
    assert lay.header_bytes == 64 + 16   # 2 * 24 entries * 2 bits = 12 bytes -> 16
    assert lay.size[6] == lay.size[7] == 0


def test_width_map_header_hand_worked(oracle):
    # L = 1, H = 4: K widths 2 3 4 8 -> codes 0 1 2 3 -> byte 0b11100100 = 0xE4;
    # V widths 8 8 2 2 -> codes 3 3 0 0 -> byte 0b00001111 = 0x0F.
    p = oracle.make_profile(smooth_keys=False, bits_map_k=[[2, 3, 4, 8]], bits_map_v=[[8, 8, 2, 2]], group_k=32,
                            group_v=32, stages=((1, 8), (4, 2)), chunk_bytes=1024)
    shape = oracle.make_shape(1, 40, 4, D, 2)
    k = _rand_bits((1, 40, 4, D), 3)
    v = _rand_bits((1, 40, 4, D), 4)
    s, f = oracle.encode(p, shape, k, v)
    assert f == 0
    assert bytes(s[0:4]) == b"KVC1"
    assert int(s[4]) | int(s[5]) << 8 == 2        # version 2
    assert int(s[6]) | int(s[7]) << 8 == 80       # 64 + 16 header bytes
    assert s[21] == 8 and s[22] == 0 and s[23] == 0
    assert s[64] == 0xE4 and s[65] == 0x0F and not s[66:80].any()
    lay = oracle.layout(p, shape)
    assert lay.data_start == ((80 + 4 * lay.n_chunks) + 15) // 16 * 16
    # a v1 profile keeps the v1 header
    p1 = oracle.make_profile(smooth_keys=False, bits_k=4, bits_v=4, group_k=32, group_v=32)
    s1, _ = oracle.encode(p1, shape, k, v)
    assert int(s1[4]) == 1 and int(s1[6]) == 64 and s1[22] == 4


def test_mixed_round_trip_and_corruption(oracle):
    L, T, H = 2, 150, 3
    wk = np.array([[2, 8, 4], [3, 4, 8]], np.uint8)
    wv = np.array([[8, 2, 3], [4, 4, 2]], np.uint8)
    p = oracle.make_profile(hadamard=True, bits_map_k=wk, bits_map_v=wv, group_k=64, group_v=64,
                            stages=((1, 8), (2, 8), (4, 2)), chunk_bytes=2048)
    shape = oracle.make_shape(L, T, H, D, 2)
    k = _rand_bits((L, T, H, D), 7)
    v = _rand_bits((L, T, H, D), 8)
    s, f = oracle.encode(p, shape, k, v)
    assert f == 0
    ok, ov = np.zeros_like(k), np.zeros_like(v)
    assert oracle.decode(p, shape, s, ok, ov) == 0
    # per head: the reconstruction error shrinks with the width (8-bit heads far tighter than 2-bit)
    kf = (k.astype(np.uint32) << 16).view(np.float32)
    rf = (ok.astype(np.uint32) << 16).view(np.float32)
    err = np.abs(rf - kf).max(axis=(1, 3))   # [L, H]
    assert err[0, 1] * 8 < err[0, 0]          # 8-bit vs 2-bit head of layer 0
    # the same stream under a plan with one width changed is rejected (the map is in the header)
    wk2 = wk.copy()
    wk2[1, 2] = 4
    p2 = oracle.make_profile(hadamard=True, bits_map_k=wk2, bits_map_v=wv, group_k=64, group_v=64,
                             stages=((1, 8), (2, 8), (4, 2)), chunk_bytes=2048)
    assert oracle.decode(p2, shape, s, ok, ov) & oracle.FLAG_CORRUPT


# ----------------------------------------------------------------- token delta
def test_delta_anchor_cells_hold_block_first_tokens(oracle):
    L, T, H = 2, 300, 3
    k = _rand_bits((L, T, H, D), 11, dtype=1)
    v = _rand_bits((L, T, H, D), 12, dtype=1)
    p = oracle.make_profile(token_delta=True, bits_k=4, bits_v=4, group_k=64, group_v=64)
    shape = oracle.make_shape(L, T, H, D, 1)
    Q, f = oracle.quantize(p, shape, k, v)
    lay = oracle.layout(p, shape)
    nab = 3  # blocks of 128 tokens: 0, 128, 256
    for tensor, x in ((0, k), (1, v)):
        sec = Q[lay.off[6 + tensor]:lay.off[6 + tensor] + lay.size[6 + tensor]].view(np.uint16)
        assert sec.size == L * H * nab * D
        cells = sec.reshape(L, H, nab, D)
        for ab in range(nab):
            assert np.array_equal(cells[:, :, ab, :], x[:, 128 * ab, :, :]), (tensor, ab)
    s, _ = oracle.encode(p, shape, k, v)
    assert int(s[4]) == 2 and s[21] == 1 | 4


def test_delta_small_integers_code_exactly_and_reconstruct_exactly(oracle):
    """x = anchor + d, d integer in [0, 255] with 0 and 255 in every key channel group
    and every value row: z = 0 and s = 1 exactly, so each code is its delta (the
    sign is x - anchor) and decode restores x exactly."""
    L, T, H = 1, 256, 2
    rng = np.random.default_rng(21)
    anchors = rng.integers(-300, 300, size=(L, 2, H, D))          # per block
    d = rng.integers(1, 255, size=(L, T, H, D))
    for t0 in (0, 128):
        d[:, t0] = 0                                             # the anchor's own delta
        for t in range(t0 + 1, t0 + 128):                        # every value row: 0 and 255 present
            d[:, t, :, (t * 7) % D] = 0
            d[:, t, :, (t * 7 + 1) % D] = 255
        for c in range(D):                                       # every key channel group: 255 present
            d[:, t0 + 1 + (c % 127), :, c] = 255
    x = np.concatenate([anchors[:, 0:1] + d[:, :128], anchors[:, 1:2] + d[:, 128:]], axis=1).astype(np.float32)
    assert np.abs(x).max() < 2048                                # integers exact in binary16
    k = _f16(x)
    v = _f16(x[:, :, ::-1, :].copy())
    dv = d[:, :, ::-1, :]
    p = oracle.make_profile(token_delta=True, smooth_keys=False, bits_k=8, bits_v=8, group_k=128, group_v=128)
    shape = oracle.make_shape(L, T, H, D, 1)
    Q, f = oracle.quantize(p, shape, k, v)
    assert f == 0
    lay = oracle.layout(p, shape)
    kc = Q[lay.off[0]:lay.off[0] + lay.size[0]].reshape(L, H, 2, D, 128)   # [l][h][tg][c] records of 128 codes
    for tg in range(2):
        assert np.array_equal(kc[0, :, tg].transpose(2, 0, 1), d[0, 128 * tg:128 * (tg + 1)].astype(np.uint8))
    vc = Q[lay.off[2]:lay.off[2] + lay.size[2]].reshape(L, T, H, D)         # [l][t][h] rows of 128 codes
    assert np.array_equal(vc[0], dv[0].astype(np.uint8))
    s, _ = oracle.encode(p, shape, k, v)
    ok, ov = np.zeros_like(k), np.zeros_like(v)
    assert oracle.decode(p, shape, s, ok, ov) == 0
    assert np.array_equal(ok, k) and np.array_equal(ov, v)


@pytest.mark.parametrize("dtype", [1, 2])
def test_delta_with_smoothing_and_hadamard_within_bound(oracle, dtype):
    L, T, H = 1, 260, 2
    k = _rand_bits((L, T, H, D), 31, dtype)
    v = _rand_bits((L, T, H, D), 32, dtype)
    p = oracle.make_profile(token_delta=True, smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=64,
                            group_v=64, stages=((1, 8), (2, 8), (3, 1), (4, 2)), chunk_bytes=4096)
    shape = oracle.make_shape(L, T, H, D, dtype)
    s, f = oracle.encode(p, shape, k, v)
    assert f == 0
    ok, ov = np.zeros_like(k), np.zeros_like(v)
    assert oracle.decode(p, shape, s, ok, ov) == 0
    Q, _ = oracle.quantize(p, shape, k, v)
    lay = oracle.layout(p, shape)

    def f32(a):
        a = np.asarray(a, np.uint16)
        return a.view(np.float16).astype(np.float64) if dtype == 1 else \
            (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    for tensor, x, r in ((0, k, ok), (1, v, ov)):
        m = Q[lay.off[2 * tensor + 1]:lay.off[2 * tensor + 1] + lay.size[2 * tensor + 1]].view(np.uint16)
        smax = float(np.abs(m.reshape(-1, 2)[:, 0].view(np.float16).astype(np.float64)).max())
        scale = 1.0
        if tensor == 0:
            e = Q[lay.off[5]:lay.off[5] + lay.size[5]].view(np.int8)
            scale = 2.0 ** int(e.max())
        # orthonormal transform: per element at most sqrt(D) * s/2 in the transformed domain
        bound = np.sqrt(D) * smax / 2 * scale
        xe, re = f32(x), f32(r)
        tol = bound * (1 + 1e-5) + np.abs(xe) * 2.0 ** -7 + 1e-6
        assert np.all(np.abs(re - xe) <= tol), (tensor, float(np.abs(re - xe).max()), bound)

"""GPU (sm_103a) versus oracle, element by element, through the C ABI.

Small seeded cases spanning several tiles, chunks and ragged tails; every code
width, group size, axis, transform on/off, both element types, paged input, and
the degenerate shapes.  Payload bytes, stream bytes and sizes must be identical;
reconstructions must be within 1e-3 relative or one quantization step of the
oracle's (and are expected to be identical, checked in a separate test)."""
import itertools

import numpy as np
import pytest
import torch

from kv_cache_compression_encode_gb300 import kvc
from kv_cache_compression_encode_gb300.codec import Codec
from oracle import oracle as O
from tests import parity_util as U

pytestmark = pytest.mark.gpu

LC = ((1, 8), (2, 8), (4, 2))
FULL = ((1, 8), (2, 8), (3, 1), (4, 2))


def _step_bound(case, Qo):
    """Largest quantization step of the case in the original domain."""
    lay = O.layout(U.oracle_profile(case.profile), case.oracle_shape())
    steps = []
    for sec in (1, 3):
        m = Qo[lay.off[sec]:lay.off[sec] + lay.size[sec]].view(np.uint16).reshape(-1, 2)
        if m.size:
            steps.append(float(np.abs(m[:, 0].view(np.float16).astype(np.float64)).max()))
    s = max(steps) if steps else 0.0
    if case.profile.get("hadamard"):
        s *= np.sqrt(128)
    if case.profile.get("smooth_keys", True) and lay.size[5]:
        e = Qo[lay.off[5]:lay.off[5] + lay.size[5]].view(np.int8)
        s *= 2.0 ** int(e.max())
    return s + 1e-30


def _run_full(case, check_exact_recon=True):
    case.materialize()
    codec, sg, nbytes, sg_np, so, fg, fo = U.encode_both(case)
    assert fg == fo, (fg, fo)
    assert nbytes == so.size, (nbytes, so.size)
    assert np.array_equal(sg_np, so), f"stream differs at {np.flatnonzero(sg_np != so)[:8]}"
    # quantized payload on its own
    Qg = codec.quantize(case.k, case.v, case.block_table)
    codec.query()
    Qo, _ = O.quantize(U.oracle_profile(case.profile), case.oracle_shape(), case.host_bits(case.k),
                       case.host_bits(case.v), case.bt_host())
    Qg_np = U.to_np(Qg, codec.plan.payload_bytes)
    assert np.array_equal(Qg_np, Qo), f"payload differs at {np.flatnonzero(Qg_np != Qo)[:8]}"
    # decode (GPU) vs decode (oracle) of the same stream
    ok, ov = case.empty_like_kv()
    codec.decode(sg, nbytes, ok, ov, case.block_table)
    st, _, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    hk, hv = [np.zeros_like(a) for a in case.host_bits(case.k)], [np.zeros_like(a) for a in case.host_bits(case.v)]
    assert O.decode(U.oracle_profile(case.profile), case.oracle_shape(), so, hk, hv, case.bt_host()) == 0
    gk, gv = case.host_bits(ok), case.host_bits(ov)
    if case.page_size:  # only the pages the block table maps hold tokens
        bt = case.bt_host()
        used = sorted(set(bt[:-(-case.T // case.page_size)].tolist()))
        gk = [g[used] for g in gk]; gv = [g[used] for g in gv]
        hk = [h[used] for h in hk]; hv = [h[used] for h in hv]
        # the last logical page may be partly filled
        if case.T % case.page_size:
            last = int(bt[case.T // case.page_size])
            j = used.index(last)
            n = case.T % case.page_size
            for arrs in (gk, gv, hk, hv):
                for a in arrs:
                    a[j, n:] = 0
    bound = _step_bound(case, Qo)
    for g, h in zip(gk + gv, hk + hv):
        U.assert_recon_close(g, h, case.dtype, bound)
        if check_exact_recon:
            assert np.array_equal(g, h), f"{int((g != h).sum())} reconstructed elements differ"
    return codec


# --------------------------------------------------------------------------- matrix
BITS_GROUPS = list(itertools.product([2, 3, 4, 8], [32, 64, 128]))


@pytest.mark.parametrize("bits,group", BITS_GROUPS)
@pytest.mark.parametrize("had", [False, True])
def test_bits_groups_transform(bits, group, had):
    prof = dict(smooth_keys=True, hadamard=had, bits_k=bits, bits_v=bits, group_k=group, group_v=group, stages=LC,
                chunk_bytes=4096)
    _run_full(U.Case(L=2, T=300, H=3, dtype="bf16", dist="llama", seed=bits * 10 + group, profile=prof))


@pytest.mark.parametrize("stages", [(), ((1, 8), (4, 1)), FULL, ((3, 2), (4, 2)), ((1, 4), (2, 8), (4, 4)),
                                    ((1, 2), (3, 4), (4, 1)), ((2, 8),), ((1, 8), (3, 1))])
def test_stage_lists(stages):
    prof = dict(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=64, group_v=64, stages=stages,
                chunk_bytes=2048)
    _run_full(U.Case(L=2, T=260, H=2, dtype="bf16", dist="llama_sink", seed=3, profile=prof))


@pytest.mark.parametrize("axis_k,axis_v,smooth", [(1, 0, True), (1, 0, False), (0, 0, False), (1, 1, True),
                                                  (0, 1, False)])
def test_axes_and_smoothing(axis_k, axis_v, smooth):
    for had in (False, True):
        prof = dict(smooth_keys=smooth, hadamard=had, bits_k=3, bits_v=4, group_k=32, group_v=64, axis_k=axis_k,
                    axis_v=axis_v, stages=LC, chunk_bytes=1024)
        _run_full(U.Case(L=1, T=200, H=2, dtype="f16", dist="gauss_outlier", seed=11, profile=prof))


@pytest.mark.parametrize("T", [1, 7, 31, 33, 127, 128, 129, 257])
def test_ragged_token_counts(T):
    prof = dict(smooth_keys=True, hadamard=True, bits_k=4, bits_v=2, group_k=64, group_v=32, stages=FULL,
                chunk_bytes=1024)
    _run_full(U.Case(L=2, T=T, H=1, dtype="bf16", dist="llama", seed=T, profile=prof))


@pytest.mark.parametrize("L", [128, 129, 256])
def test_layer_counts_up_to_the_limit(L):
    """Up to 128 layers the key tiles arrive by TMA (one tensor map per layer in the
    launch's parameters); past that the same kernel loads them with cp.async; 256 is
    the most a plan takes (KVC_MAX_LAYERS)."""
    prof = dict(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=LC,
                chunk_bytes=4096)
    _run_full(U.Case(L=L, T=130, H=1, dtype="bf16", dist="llama", seed=L, profile=prof))


@pytest.mark.parametrize("had", [False, True])
def test_paged_gather_and_scatter(had):
    prof = dict(smooth_keys=True, hadamard=had, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=LC,
                chunk_bytes=4096)
    _run_full(U.Case(L=3, T=1000, H=8, dtype="bf16", dist="llama", seed=5, page_size=16, profile=prof))


def test_tiny_workload_full():
    from kv_cache_compression_encode_gb300.workloads import PROFILES
    _run_full(U.Case(L=1, T=256, H=8, dtype="f16", dist="gauss_outlier", seed=1234, profile=PROFILES["tiny"]))


def test_empty_tokens():
    prof = dict(stages=LC)
    case = U.Case(L=2, T=0, H=8, profile=prof)
    codec = Codec(kvc.make_profile(**prof), case.kvc_shape())
    dummy = [torch.zeros(16, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    sg = codec.encode(dummy, dummy)
    st, nbytes, flags = codec.query()
    so, _ = O.encode(O.make_profile(**prof), case.oracle_shape(), [np.zeros(1, np.uint16)] * 2,
                     [np.zeros(1, np.uint16)] * 2)
    assert st == kvc.KVC_OK and nbytes == so.size == 64
    assert np.array_equal(U.to_np(sg, nbytes), so)
    codec.decode(sg, nbytes, dummy, dummy)
    assert codec.query()[0] == kvc.KVC_OK


# --------------------------------------------------------------------------- quantization ties
def test_exact_ties_take_the_even_code():
    """Rows whose values sit exactly on (and one ulp around) the half-steps of their
    group: the encoders' corrected quotient must land exactly on each tie and round
    it to the even code, as the division does."""
    T, H = 64, 1
    base = np.arange(32, dtype=np.float32)
    rows = []
    for t in range(T):
        r = np.zeros(128, np.float32)
        r[0], r[1] = 0.0, 15.0                        # group 0: z = 0, s = 1 (4-bit)
        r[2:17] = np.arange(15) + 0.5                 # exact ties
        r[17:32] = np.nextafter(np.arange(15) + 0.5, np.float32(t % 2 and 1e9 or -1e9))
        r[32], r[33] = -1.0, 2.0                      # group 1: z = -1, s = 0.2 (rounded up)
        r[34:64] = -1.0 + (base[:30] % 16) * 0.2 + 0.1
        r[64:128] = np.float32(t) * 0.25 + base.repeat(2) * 0.125
        rows.append(r)
    x = np.stack(rows).reshape(1, T, H, 128)
    kbits = x.astype(np.float16).view(np.uint16)
    prof = dict(smooth_keys=False, hadamard=False, bits_k=4, bits_v=4, group_k=32, group_v=32, stages=())
    case = U.Case(L=1, T=T, H=H, dtype="f16", profile=prof)
    case.k = [torch.from_numpy(kbits[0].view(np.int16)).view(torch.float16).cuda()]
    case.v = [torch.from_numpy(kbits[0].view(np.int16).copy()).view(torch.float16).cuda()]
    codec, Qg, Qo, fg, fo = U.quantize_both(case)
    assert fg == fo == 0
    assert np.array_equal(Qg, Qo)


@pytest.mark.parametrize("had", [False, True])
def test_wide_smoothing_ranges_match_oracle(had):
    """Key channels whose 128-token block spans more than 2^100 (bf16 reaches 3e38):
    the key-tile encoder applies the smoothing with one fma per pair only where
    every exponent of the tile is at most 100 and with the two roundings as
    written elsewhere; both kinds of tile, side by side, must give the oracle's
    bytes.  One channel is symmetric around 0 (centre 0, exponent 104), one is
    large and positive only (the centre saturates: the RANGE flag)."""
    prof = dict(bits_k=4, bits_v=4, group_k=128, group_v=128, hadamard=had, stages=())
    case = U.Case(L=1, T=384, H=2, dtype="bf16", profile=prof, seed=5).materialize()
    sgn = torch.where(torch.arange(128, device="cuda") % 2 == 0, 1.0, -1.0)
    case.k[0][128:256, 0, 7] = (sgn * 1e31).to(torch.bfloat16)      # tile (h 0, block 1): e = 104
    case.k[0][128:256, 0, 9] = (sgn * 3.0 + 1.5).to(torch.bfloat16)  # an ordinary channel of the same tile
    case.k[0][256:384, 1, 40] = 1e36                                 # tile (h 1, block 2): centre saturates
    codec, Qg, Qo, fg, fo = U.quantize_both(case)
    assert fg == fo and fg != 0, (fg, fo)  # the saturated centre raises RANGE on both sides
    assert np.array_equal(Qg, Qo), f"payload differs at {np.flatnonzero(Qg != Qo)[:8]}"


# --------------------------------------------------------------------------- status words
def test_nonfinite_and_range_flags_match_oracle():
    prof = dict(bits_k=4, bits_v=4, group_k=32, group_v=32, stages=LC, chunk_bytes=1024)
    for kind in ("nan", "inf", "range"):
        case = U.Case(L=1, T=64, H=2, dtype="bf16", profile=prof, seed=2).materialize()
        if kind == "nan":
            case.v[0][5, 1, 3] = float("nan")
        elif kind == "inf":
            case.k[0][9, 0, 100] = float("inf")
        else:
            case.v[0][7, 0, :] = 3e9   # a value group whose scale overflows fp16
            case.k[0][:, 1, 2] = -1e6  # a key channel whose zero point overflows fp16
        codec, sg, nbytes, _, so, fg, fo = U.encode_both(case)
        assert fg == fo and fg != 0, (kind, fg, fo)
        st, _, _ = codec.query()
        want = {"nan": kvc.KVC_ERR_NONFINITE, "inf": kvc.KVC_ERR_NONFINITE, "range": kvc.KVC_ERR_RANGE}[kind]
        assert st == want
        if kind == "range":  # saturated metadata is still deterministic: bytes match too
            assert np.array_equal(U.to_np(sg, nbytes), so)


@pytest.mark.parametrize("chunk", [1024, 4096, 256])
def test_corrupt_streams_are_rejected_and_outputs_untouched(chunk):
    """1 KiB chunks decode through the generic stage functions, 4 KiB chunks through
    the fast chunk decoder; both must reject the same corruptions.  With 256-byte
    chunks the table has more than 16384 entries, so the stream and table checks
    run in the separate prepare launch instead of inside the decoder."""
    prof = dict(bits_k=4, bits_v=4, group_k=64, group_v=64, hadamard=True, stages=LC, chunk_bytes=chunk)
    big = chunk == 256
    case = U.Case(L=2 if big else 1, T=2048 if big else 300, H=8 if big else 2, dtype="bf16", dist="llama_sink",
                  profile=prof, seed=4).materialize()
    codec, sg, nbytes, sg_np, so, _, _ = U.encode_both(case)
    lay = O.layout(U.oracle_profile(prof), case.oracle_shape())
    table = so[64:64 + 4 * lay.n_chunks].view(np.uint32)
    first_rze = int(np.flatnonzero((table >> 31) == 0)[0])
    start = lay.data_start + sum(((int(e) & 0x7FFFFFFF) + 15) // 16 * 16 for e in table[:first_rze])
    mutations = {
        "magic": lambda s: s.__setitem__(0, ord("X")),
        "seed": lambda s: s.__setitem__(48, s[48] ^ 1),
        "truncate": None,
        "table_size": lambda s: s.__setitem__(64 + 4 * first_rze, s[64 + 4 * first_rze] ^ 0x10),
        "table_raw": lambda s: s.__setitem__(64 + 4 * first_rze + 3, s[64 + 4 * first_rze + 3] ^ 0x80),
        "bitmap": lambda s: s.__setitem__(start, s[start] ^ 0xFF),
    }
    for name, mut in mutations.items():
        s = so.copy()
        if mut is None:
            s = s[:-32]
        else:
            mut(s)
        fo = O.decode(U.oracle_profile(prof), case.oracle_shape(), s,
                      [np.zeros_like(a) for a in case.host_bits(case.k)],
                      [np.zeros_like(a) for a in case.host_bits(case.v)])
        dev = torch.from_numpy(np.concatenate([s, np.zeros(64, np.uint8)])).cuda()
        ok, ov = case.empty_like_kv(fill=0x1234)
        kvc.kvc_timing_enable(codec.plan, True)
        codec.decode(dev, s.size, ok, ov)
        st, _, fg = codec.query()
        names = [n for n, _ in kvc.kvc_timing_read(codec.plan)]
        kvc.kvc_timing_enable(codec.plan, False)
        assert ("kvc_decode_prepare" in names) == big, (name, names)
        assert fo & O.FLAG_CORRUPT, name
        assert st == kvc.KVC_ERR_CORRUPT and (fg & kvc.FLAG_CORRUPT), name
        for t in ok + ov:  # nothing written
            assert bool((t.view(torch.int16) == 0x1234).all()), name


@pytest.mark.parametrize("chunk", [1024, 4096])
def test_lookback_wait_is_bounded(chunk):
    """A chunk that never publishes its size: the successor's wait runs out,
    the status says TIMEOUT, and the GPU stays usable.  1 KiB chunks run the
    generic encoder, 4 KiB chunks the worker/publisher encoder."""
    prof = dict(bits_k=4, bits_v=4, group_k=64, group_v=64, stages=LC, chunk_bytes=chunk)
    case = U.Case(L=1, T=256 if chunk == 1024 else 512, H=2, profile=prof, seed=6).materialize()
    codec = Codec(kvc.make_profile(**prof), case.kvc_shape())
    kvc.kvc_debug_lookback(codec.plan, 3, 2000)
    codec.encode(case.k, case.v)
    st, _, flags = codec.query()
    assert st == kvc.KVC_ERR_TIMEOUT and flags & kvc.FLAG_TIMEOUT
    kvc.kvc_debug_lookback(codec.plan, -1, 0)
    sg = codec.encode(case.k, case.v)
    st, nbytes, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    so, _ = O.encode(U.oracle_profile(prof), case.oracle_shape(), case.host_bits(case.k), case.host_bits(case.v))
    assert np.array_equal(U.to_np(sg, nbytes), so)


def test_bad_block_table_entry_is_flagged():
    prof = dict(bits_k=4, bits_v=4, group_k=64, group_v=64, stages=())
    case = U.Case(L=1, T=64, H=2, profile=prof, page_size=16, seed=8).materialize()
    case.block_table[2] = 1 << 20
    codec = Codec(kvc.make_profile(**prof), case.kvc_shape())
    codec.encode(case.k, case.v, case.block_table)
    st, _, flags = codec.query()
    assert st == kvc.KVC_ERR_INVALID_ARG and flags & kvc.FLAG_BAD_PAGE


@pytest.mark.parametrize("had", [False, True])
def test_bad_block_table_entry_on_decode(had):
    """Decoding through a block table with one out-of-range entry flags BAD_PAGE,
    writes every row of the valid pages exactly as a clean decode does, and
    leaves the page the bad entry replaced untouched (both decoders: keys in
    128-token tiles, values row by row)."""
    prof = dict(hadamard=had, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=LC, chunk_bytes=4096)
    case = U.Case(L=2, T=256, H=2, profile=prof, page_size=16, seed=11).materialize()
    codec = Codec(kvc.make_profile(**prof), case.kvc_shape())
    sg = codec.encode(case.k, case.v, case.block_table)
    st, nbytes, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    rk, rv = case.empty_like_kv()
    codec.decode(sg, nbytes, rk, rv, case.block_table)
    st, _, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    bad_entry = 3
    bt = case.block_table.clone()
    lost = int(bt[bad_entry])
    bt[bad_entry] = 1 << 20
    ok, ov = case.empty_like_kv()
    codec.decode(sg, nbytes, ok, ov, bt)
    st, _, flags = codec.query()
    assert st == kvc.KVC_ERR_INVALID_ARG and flags & kvc.FLAG_BAD_PAGE
    canary = case.empty_like_kv()[0][0][lost]
    for got, ref in zip(ok + ov, rk + rv):
        for pg in range(case.n_pages):
            if pg == lost:
                assert torch.equal(got[pg], canary), "a row landed in the page of the bad entry"
            else:
                assert torch.equal(got[pg], ref[pg]), f"page {pg} differs from the clean decode"


def test_strided_layers_writes_stay_in_their_rows():
    """Strided token rows (256 padding bytes after each token) inside one buffer
    with guard bytes between the layers: encode reads only the rows, decode writes
    only the rows (both decoders' row copies), and the rows match a decode into a
    dense layout."""
    prof = dict(hadamard=True, bits_k=4, bits_v=4, group_k=64, group_v=128, stages=FULL, chunk_bytes=4096)
    from kv_cache_compression_encode_gb300 import synth
    L, T, H, D = 2, 300, 3, 128
    row, ts, guard = H * D * 2, H * D * 2 + 256, 4096
    span = T * ts

    def carve(fill):
        buf = torch.full((guard + L * (span + guard),), fill, dtype=torch.uint8, device="cuda")
        views = [buf[guard + l * (span + guard): guard + l * (span + guard) + span] for l in range(L)]
        return buf, views

    kbuf, kin = carve(0x7E)
    vbuf, vin = carve(0x7E)
    dense_k, dense_v = [], []
    for l in range(L):
        k, v = synth.layer_kv("llama", l, T, H, D, "bf16", 31, "cuda")
        dense_k.append(k.contiguous()); dense_v.append(v.contiguous())
        for dst, src in ((kin[l], k), (vin[l], v)):
            dst.view(T, ts)[:, :row].copy_(src.contiguous().view(torch.uint8).view(T, row))
    strided = kvc.make_shape(L, T, H, D, kvc.BF16, token_stride=ts)
    codec = Codec(kvc.make_profile(**prof), strided)
    sg = codec.encode(kin, vin)
    st, nbytes, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    # the same stream from the dense layout
    dcodec = Codec(kvc.make_profile(**prof), kvc.make_shape(L, T, H, D, kvc.BF16))
    sd = dcodec.encode(dense_k, dense_v)
    _, nd, _ = dcodec.query()
    assert nd == nbytes and torch.equal(sg[:nbytes], sd[:nd])
    # decode into strided rows surrounded by canary bytes
    okbuf, kout = carve(0x5A)
    ovbuf, vout = carve(0x5A)
    codec.decode(sg, nbytes, kout, vout)
    st, _, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    rk = [torch.empty_like(x) for x in dense_k]
    rv = [torch.empty_like(x) for x in dense_v]
    dcodec.decode(sd, nd, rk, rv)
    assert dcodec.query()[0] == kvc.KVC_OK
    for buf, outs, refs in ((okbuf, kout, rk), (ovbuf, vout, rv)):
        mask = torch.ones_like(buf, dtype=torch.bool)  # True: bytes nothing may write
        for l in range(L):
            base = guard + l * (span + guard)
            mask[base: base + span].view(T, ts)[:, :row] = False
            assert torch.equal(outs[l].view(T, ts)[:, :row], refs[l].view(torch.uint8).view(T, row)), f"layer {l}"
        assert bool((buf[mask] == 0x5A).all()), "a decoder wrote outside the token rows"


@pytest.mark.parametrize("stages", [FULL, LC, ((1, 2), (3, 4), (4, 1))])
def test_step_outputs_stay_inside_their_sizes(stages):
    """Each step writes exactly its output's bytes: the payload's payload_bytes
    (quantize, lossless decode) and the stream's reported size (lossless encode);
    the bytes after them (canary) are untouched."""
    prof = dict(hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=stages, chunk_bytes=4096)
    case = U.Case(L=2, T=300, H=3, profile=prof, seed=41).materialize()
    codec = Codec(kvc.make_profile(**prof), case.kvc_shape())
    n, cap, guard = codec.plan.payload_bytes, codec.plan.max_stream_bytes, 4096
    payload = torch.full((n + guard,), 0xA5, dtype=torch.uint8, device="cuda")
    codec.quantize(case.k, case.v, out=payload)
    assert codec.query()[0] == kvc.KVC_OK
    assert bool((payload[n:] == 0xA5).all()), "quantize wrote past the payload"
    stream = torch.full((cap + guard,), 0xA5, dtype=torch.uint8, device="cuda")
    codec.lossless_encode(payload, out=stream)
    st, nbytes, _ = codec.query()
    assert st == kvc.KVC_OK and nbytes <= cap
    assert bool((stream[nbytes:] == 0xA5).all()), "the encoder wrote past the stream's size"
    back = torch.full((n + guard,), 0xA5, dtype=torch.uint8, device="cuda")
    codec.lossless_decode(stream, nbytes, out=back)
    assert codec.query()[0] == kvc.KVC_OK
    assert torch.equal(back[:n], payload[:n])
    assert bool((back[n:] == 0xA5).all()), "the decoder wrote past the payload"


def test_repeatable_and_independent_streams():
    prof = dict(bits_k=4, bits_v=4, group_k=128, group_v=128, hadamard=True, stages=FULL, chunk_bytes=2048)
    case = U.Case(L=2, T=512, H=4, profile=prof, seed=9).materialize()
    a = Codec(kvc.make_profile(**prof), case.kvc_shape())
    b = Codec(kvc.make_profile(**prof), case.kvc_shape())
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        x = a.encode(case.k, case.v)
    with torch.cuda.stream(s2):
        y = b.encode(case.k, case.v)
    with torch.cuda.stream(s1):
        _, na, _ = a.query()
    with torch.cuda.stream(s2):
        _, nb, _ = b.query()
    torch.cuda.synchronize()
    assert na == nb and torch.equal(x[:na], y[:nb])

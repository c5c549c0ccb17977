"""kvc_decode with the codes of stored chunks read in place from the stream
(kvc_decode_codes_in_place; "Beyond Compression Ratio" §3 design goal G1, §4.2):
the reconstruction must be bit for bit the oracle's decode of the same stream, and
bit for bit the decode with the choice off.  Which path ran is read from the launch
timings: the lossless decoder is named ..._inplace when some tensor's code chunks
stay in the stream.  Cases: both tensors, one, none; 2-, 4- and 8-bit codes; keys
grouped over channels; a table large enough for the separate prepare step; a
generic stage list; compressible chunks among the in-place ones; paged output; the
token delta; profiles that must not take the path; corrupt chunk tables; more chunks
per decoder CTA than it has threads."""
import numpy as np
import pytest
import torch

from kv_cache_compression_encode_gb300 import kvc
from oracle import oracle as O
from tests import parity_util as U

pytestmark = pytest.mark.gpu

FULL = ((1, 8), (2, 8), (3, 1), (4, 2))
LC = ((1, 8), (2, 8), (4, 2))


def _expected(case):
    """Which tensors' code chunks the rule leaves in the stream, from the oracle's
    layout: uniform width 2/4/8, chunks of a power of two bytes, the code section on
    a chunk boundary with at least one whole chunk; keys-style tiles (groups over
    tokens) need ceil(T/G) G a multiple of 128 and 2048 bits dividing the chunk;
    rows (groups over channels, no smoothing) need 256 bits dividing it."""
    p = case.profile
    cb = p.get("chunk_bytes", 16384)
    if not p.get("stages") or p.get("bits_map_k") or p.get("bits_map_v") or cb & (cb - 1):
        return (False, False)
    lay = O.layout(U.oracle_profile(p), case.oracle_shape())
    out = []
    for t in (0, 1):
        bits = p.get("bits_v" if t else "bits_k", 4)
        G = p.get("group_v" if t else "group_k", 64)
        axis = p.get("axis_v" if t else "axis_k", 1 if t else 0)
        smooth = t == 0 and p.get("smooth_keys", True)
        off, size = lay.off[2 * t], lay.size[2 * t]
        ok = bits in (2, 4, 8) and off % cb == 0 and (off + size) // cb > off // cb
        if axis == 0:
            ok = ok and (-(-case.T // G) * G) % 128 == 0 and cb % (2048 * bits) == 0
        else:
            ok = ok and not smooth and cb % (256 * bits) == 0
        out.append(ok)
    return tuple(out)


def _decode(codec, case, sg, nbytes, in_place):
    kvc.kvc_decode_codes_in_place(codec.plan, in_place)
    ok, ov = case.empty_like_kv()
    kvc.kvc_timing_enable(codec.plan, True)
    codec.decode(sg, nbytes, ok, ov, case.block_table)
    st, _, flags = codec.query()
    names = {n for n, _ in kvc.kvc_timing_read(codec.plan)}
    kvc.kvc_timing_enable(codec.plan, False)
    kvc.kvc_decode_codes_in_place(codec.plan, True)
    assert st == kvc.KVC_OK and flags == 0, (st, flags)
    return case.host_bits(ok), case.host_bits(ov), names


def _check(case, materialized=False):
    if not materialized:
        case.materialize()
    codec, sg, nbytes, sg_np, so, fg, fo = U.encode_both(case)
    assert fg == fo and np.array_equal(sg_np, so)
    gk, gv, names = _decode(codec, case, sg, nbytes, True)
    want = any(_expected(case))
    assert any(n.endswith("_inplace") for n in names) == want, (sorted(names), _expected(case))
    rk, rv, names_off = _decode(codec, case, sg, nbytes, False)
    assert not any(n.endswith("_inplace") for n in names_off), sorted(names_off)
    hk = [np.zeros_like(a) for a in case.host_bits(case.k)]
    hv = [np.zeros_like(a) for a in case.host_bits(case.v)]
    assert O.decode(U.oracle_profile(case.profile), case.oracle_shape(), so, hk, hv, case.bt_host()) == 0
    if case.page_size:  # only the pages the block table maps hold tokens; zero the rest of the last one
        bt = case.bt_host()
        used = sorted(set(bt[:-(-case.T // case.page_size)].tolist()))
        arrs = [[a[used] for a in x] for x in (gk, gv, rk, rv, hk, hv)]
        if case.T % case.page_size:
            j = used.index(int(bt[case.T // case.page_size]))
            for x in arrs:
                for a in x:
                    a[j, case.T % case.page_size:] = 0
        gk, gv, rk, rv, hk, hv = arrs
    for g, r, h in zip(gk + gv, rk + rv, hk + hv):
        assert np.array_equal(g, h), f"{int((g != h).sum())} elements differ from the oracle's decode"
        assert np.array_equal(g, r), "in-place and payload decodes differ"
    return names


CASES = [
    # (bits_k, bits_v, group_k, group_v, stages, chunk, L, T, H, dtype, had, page, extra)
    (4, 4, 128, 128, FULL, 16384, 2, 512, 8, "bf16", True, 0, {}),            # both tensors
    (2, 2, 32, 32, LC, 4096, 2, 640, 4, "bf16", True, 0, {}),                 # 2-bit, 4 KiB tiles = chunks
    (8, 8, 128, 64, FULL, 16384, 2, 256, 8, "f16", False, 0, {}),             # 8-bit: one tile per chunk
    (4, 4, 32, 64, LC, 8192, 2, 400, 8, "bf16", True, 0, {}),                 # keys: 13 x 32 tokens, not whole tiles
    (4, 4, 128, 128, FULL, 16384, 2, 500, 8, "bf16", True, 0, {}),            # a partial last tile of 116 tokens
    (4, 4, 64, 64, LC, 8192, 2, 1000, 8, "bf16", True, 16, {}),               # paged output
    (4, 4, 128, 128, ((1, 4), (4, 1)), 8192, 2, 512, 8, "bf16", True, 0, {}),  # generic stage list
    (4, 4, 128, 128, FULL, 16384, 2, 512, 8, "bf16", True, 0, {"token_delta": True}),
    (4, 2, 64, 32, LC, 4096, 2, 512, 8, "bf16", True, 0,
     {"smooth_keys": False, "axis_k": 1}),                                     # keys over channels: rows decoder
    (4, 4, 128, 128, FULL, 12288, 2, 512, 8, "bf16", True, 0, {}),            # 12 KiB chunks: not a power of two
    (3, 3, 128, 128, FULL, 16384, 2, 512, 8, "bf16", True, 0, {}),            # 3-bit units cross chunks
    (4, 4, 128, 128, (), 16384, 2, 512, 8, "bf16", True, 0, {}),              # no lossless stages
]


@pytest.mark.parametrize("bk,bv,gk,gv,stages,chunk,L,T,H,dtype,had,page,extra", CASES)
def test_in_place_decode_matches_oracle(bk, bv, gk, gv, stages, chunk, L, T, H, dtype, had, page, extra):
    prof = dict(smooth_keys=True, hadamard=had, bits_k=bk, bits_v=bv, group_k=gk, group_v=gv, stages=stages,
                chunk_bytes=chunk)
    prof.update(extra)
    case = U.Case(L=L, T=T, H=H, dtype=dtype, dist="llama", seed=bk * 13 + T, page_size=page, profile=prof)
    _check(case)


def test_in_place_decode_mixed_widths_take_the_payload():
    bm = [[2, 8, 4, 4], [8, 2, 4, 2]]
    prof = dict(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=FULL,
                chunk_bytes=16384, bits_map_k=bm, bits_map_v=bm)
    case = U.Case(L=2, T=512, H=4, dtype="bf16", dist="llama", seed=5, profile=prof)
    assert _expected(case) == (False, False)
    _check(case)


def test_in_place_decode_with_the_prepare_step():
    """More than 16384 chunks (512-byte chunks, 2-bit codes): the stream checks and
    chunk offsets come from the separate prepare launch, and the lossless decoder
    replaces a chunk's offset word by the address of its bytes."""
    prof = dict(smooth_keys=True, hadamard=True, bits_k=2, bits_v=2, group_k=64, group_v=64, stages=LC,
                chunk_bytes=512)
    case = U.Case(L=4, T=4096, H=8, dtype="bf16", dist="llama", seed=6, profile=prof)
    assert _expected(case) == (False, True)
    names = _check(case)
    assert "kvc_decode_prepare" in names and "kvc_lossless_dec_inplace" in names, sorted(names)


def test_in_place_decode_with_compressible_chunks():
    """Keys and values that repeat in the first half of the tokens: their code chunks
    compress and are restored into the payload, the others stay in the stream; the
    decoders take each unit from where its chunk is."""
    prof = dict(smooth_keys=True, hadamard=False, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=FULL,
                chunk_bytes=16384)
    case = U.Case(L=1, T=1024, H=8, dtype="bf16", dist="llama", seed=3, profile=prof).materialize()
    pattern = torch.tensor([0.5, -1.25, 3.0, 0.0], dtype=torch.float32, device="cuda")
    rows = pattern[torch.arange(512, device="cuda") % 4]
    case.v[0][:512] = rows[:, None, None].expand(512, 8, 128).to(torch.bfloat16)
    case.k[0][:512] = rows[:, None, None].expand(512, 8, 128).to(torch.bfloat16)
    assert _expected(case) == (True, True)
    lay = O.layout(U.oracle_profile(prof), case.oracle_shape())
    names = _check(case, materialized=True)
    assert "kvc_lossless_dec_fast_inplace" in names
    # both kinds of chunk inside the code sections
    so, _ = O.encode(U.oracle_profile(prof), case.oracle_shape(), case.host_bits(case.k), case.host_bits(case.v))
    table = so[lay.header_bytes:lay.header_bytes + 4 * lay.n_chunks].view(np.uint32)
    kinds = set()
    for t in (0, 1):
        c0, c1 = lay.off[2 * t] // 16384, (lay.off[2 * t] + lay.size[2 * t]) // 16384
        kinds |= {int(e >> 31) for e in table[c0:c1]}
    assert kinds == {0, 1}, kinds


def test_in_place_is_on_by_default_and_lossless_decode_writes_the_payload():
    """kvc_lossless_decode on its own restores every chunk, in-place or not."""
    prof = dict(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=FULL,
                chunk_bytes=16384)
    case = U.Case(L=2, T=512, H=8, dtype="bf16", dist="llama", seed=7, profile=prof).materialize()
    codec, sg, nbytes, sg_np, so, _, _ = U.encode_both(case)
    kvc.kvc_timing_enable(codec.plan, True)
    ok, ov = case.empty_like_kv()
    codec.decode(sg, nbytes, ok, ov)
    codec.query()
    names = {n for n, _ in kvc.kvc_timing_read(codec.plan)}
    kvc.kvc_timing_enable(codec.plan, False)
    assert "kvc_lossless_dec_fast_inplace" in names
    Qg = codec.lossless_decode(sg, nbytes)
    codec.query()
    Qo, _ = O.quantize(U.oracle_profile(prof), case.oracle_shape(), case.host_bits(case.k), case.host_bits(case.v))
    assert np.array_equal(U.to_np(Qg, codec.plan.payload_bytes), Qo)


@pytest.mark.parametrize("path", ["in_decoder", "prepare"])
def test_in_place_decode_rejects_corrupt_tables_and_writes_nothing(path):
    """Chunk-table corruptions of a chunk whose codes are read in place (its stored
    flag cleared, its size changed) and a truncated stream: the decoder reports
    CORRUPT, as the oracle does, and the reconstruction kernels write nothing.  The
    table is checked inside the decoder for small tables, by the prepare step for
    large ones (512-byte chunks, more than 16384 of them)."""
    if path == "in_decoder":
        prof = dict(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=LC,
                    chunk_bytes=8192)
        case = U.Case(L=1, T=512, H=4, dtype="bf16", dist="llama", seed=11, profile=prof).materialize()
        assert _expected(case) == (True, True)
    else:
        prof = dict(smooth_keys=True, hadamard=True, bits_k=2, bits_v=2, group_k=64, group_v=64, stages=LC,
                    chunk_bytes=512)
        case = U.Case(L=4, T=4096, H=8, dtype="bf16", dist="llama", seed=12, profile=prof).materialize()
        assert _expected(case) == (False, True)
    cb = prof["chunk_bytes"]
    codec, sg, nbytes, sg_np, so, _, _ = U.encode_both(case)
    lay = O.layout(U.oracle_profile(prof), case.oracle_shape())
    table = so[lay.header_bytes:lay.header_bytes + 4 * lay.n_chunks].view(np.uint32)
    c = lay.off[2] // cb + 1  # a whole value-code chunk, stored raw
    assert table[c] >> 31 == 1 and (table[c] & 0x7FFFFFFF) == cb
    e = lay.header_bytes + 4 * c
    mutations = {
        "stored_flag": lambda s: s.__setitem__(e + 3, s[e + 3] ^ 0x80),
        "size": lambda s: s.__setitem__(e, s[e] ^ 0x10),
        "truncate": None,
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
        assert fo & O.FLAG_CORRUPT, name
        dev = torch.from_numpy(np.concatenate([s, np.zeros(64, np.uint8)])).cuda()
        ok, ov = case.empty_like_kv(fill=0x1234)
        kvc.kvc_timing_enable(codec.plan, True)
        codec.decode(dev, s.size, ok, ov)
        st, _, fg = codec.query()
        names = {n for n, _ in kvc.kvc_timing_read(codec.plan)}
        kvc.kvc_timing_enable(codec.plan, False)
        assert any(n.endswith("_inplace") for n in names), (name, sorted(names))
        assert ("kvc_decode_prepare" in names) == (path == "prepare"), (name, sorted(names))
        assert st == kvc.KVC_ERR_CORRUPT and (fg & kvc.FLAG_CORRUPT), (name, st, fg)
        for t in ok + ov:  # nothing written
            assert bool((t.view(torch.int16) == 0x1234).all()), name
    # and the plan decodes the intact stream afterwards
    gk, gv, _ = _decode(codec, case, sg, nbytes, True)
    hk = [np.zeros_like(a) for a in case.host_bits(case.k)]
    hv = [np.zeros_like(a) for a in case.host_bits(case.v)]
    assert O.decode(U.oracle_profile(prof), case.oracle_shape(), so, hk, hv) == 0
    for g, h in zip(gk + gv, hk + hv):
        assert np.array_equal(g, h)


def test_in_place_decode_with_more_chunks_per_cta_than_threads():
    """A chunk table of 405,504 entries (2-bit codes in 512-byte chunks): each CTA of
    the lossless decoder owns more chunks than it has threads, so it settles them in
    several batches of one chunk per thread.  The reconstruction must equal, element
    for element, the decode that restores every chunk into the payload first (whose
    parity with the oracle the tests above check)."""
    prof = dict(smooth_keys=True, hadamard=True, bits_k=2, bits_v=2, group_k=32, group_v=32, stages=LC,
                chunk_bytes=512)
    case = U.Case(L=8, T=32768, H=8, dtype="bf16", dist="llama", seed=13, profile=prof, gen_device="cuda")
    case.materialize()
    assert _expected(case) == (False, True)
    codec = U.Codec(U.kvc_profile(prof), case.kvc_shape())
    n_ctas = torch.cuda.get_device_properties(0).multi_processor_count * 4  # at most 4 of 512 threads per SM
    assert codec.plan.n_chunks > 512 * n_ctas
    sg = codec.encode(case.k, case.v)
    st, nbytes, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    outs = {}
    for in_place in (True, False):
        kvc.kvc_decode_codes_in_place(codec.plan, in_place)
        ok, ov = case.empty_like_kv()
        kvc.kvc_timing_enable(codec.plan, True)
        codec.decode(sg, nbytes, ok, ov)
        st, _, flags = codec.query()
        names = {n for n, _ in kvc.kvc_timing_read(codec.plan)}
        kvc.kvc_timing_enable(codec.plan, False)
        assert st == kvc.KVC_OK and flags == 0, (in_place, st, flags)
        assert "kvc_decode_prepare" in names
        assert ("kvc_lossless_dec_inplace" in names) == in_place, sorted(names)
        outs[in_place] = (ok, ov)
    kvc.kvc_decode_codes_in_place(codec.plan, True)
    for a, b in zip(outs[True][0] + outs[True][1], outs[False][0] + outs[False][1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))

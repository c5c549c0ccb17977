"""The split encode: the value encoder writes the whole lossless chunks of the
value-code section into the stream itself ("Beyond Compression Ratio" §3 G1, §4.1,
§4.2), between a lossless launch over the chunks before them and one over the
rest (an execution choice, kvc_fuse_value_chunks).  The stream must be byte for
byte the oracle's; which path ran is read from the library's launch timings.  Cases: incompressible and compressible chunks, a
section whose last chunk is partial, 2-, 4- and 8-bit values, each stage list of
the fast path with BIT_8, the Hadamard rotation on and off, both element types,
paged input; and profiles that must not take the split path."""
import numpy as np
import pytest
import torch

from kv_cache_compression_encode_gb300 import kvc
from oracle import oracle as O
from tests import parity_util as U

pytestmark = pytest.mark.gpu

FULL = ((1, 8), (2, 8), (3, 1), (4, 2))
LC = ((1, 8), (2, 8), (4, 2))
LC1 = ((1, 8), (2, 8), (4, 1))


def _fusable(case):
    """The split path's rule, from the oracle's layout: values grouped over channels
    without smoothing, widths 2/4/8, a fast stage list with BIT_8, chunks holding a
    multiple of 128 rows, the value-code section starting on a chunk boundary with
    at least one whole chunk, and a chunk after it."""
    p = case.profile
    st = tuple(tuple(x) for x in p.get("stages", ()))
    cb = p.get("chunk_bytes", 16384)
    bits = p.get("bits_v", 4)
    if st not in (FULL, LC, LC1, ((1, 8), (2, 8), (3, 1), (4, 1))) or cb % 4096 or cb > 16384:
        return False
    if p.get("axis_v", 1) != 1 or bits not in (2, 4, 8) or p.get("token_delta") or p.get("bits_map_v"):
        return False
    rec = 16 * bits
    if cb % rec or (cb // rec) % 128:
        return False
    lay = O.layout(U.oracle_profile(p), case.oracle_shape())
    off2, size2 = lay.off[2], lay.size[2]
    return off2 % cb == 0 and size2 // cb >= 1


def _run(case):
    case.materialize()
    codec = U.Codec(U.kvc_profile(case.profile), case.kvc_shape())
    kvc.kvc_fuse_value_chunks(codec.plan, True)
    kvc.kvc_timing_enable(codec.plan, True)
    sg = codec.encode(case.k, case.v, case.block_table)
    st, nbytes, flags_g = codec.query()
    names = {n for n, _ in kvc.kvc_timing_read(codec.plan)}
    kvc.kvc_timing_enable(codec.plan, False)
    so, flags_o = O.encode(U.oracle_profile(case.profile), case.oracle_shape(), case.host_bits(case.k),
                           case.host_bits(case.v), case.bt_host())
    assert flags_g == flags_o, (flags_g, flags_o)
    assert nbytes == so.size, (nbytes, so.size)
    g = U.to_np(sg, nbytes)
    assert np.array_equal(g, so), f"stream differs at {np.flatnonzero(g != so)[:8]}"
    return names


SPLIT_CASES = [
    # (bits_v, group_v, stages, chunk, T, H, dtype, hadamard, paged)
    (4, 128, FULL, 16384, 512, 8, "bf16", True, False),    # whole chunks only
    (4, 128, FULL, 16384, 500, 8, "bf16", True, False),    # a partial last chunk (160 rows)
    (4, 64, LC, 8192, 512, 8, "f16", False, False),
    (2, 32, LC, 4096, 640, 4, "bf16", True, False),
    (2, 128, LC1, 8192, 1000, 8, "bf16", False, True),     # paged input
    (8, 128, LC, 16384, 256, 8, "bf16", True, False),
    (8, 64, FULL, 16384, 300, 2, "f16", True, False),
]


@pytest.mark.parametrize("bits_v,group_v,stages,chunk,T,H,dtype,had,paged", SPLIT_CASES)
def test_split_encode_matches_oracle(bits_v, group_v, stages, chunk, T, H, dtype, had, paged):
    prof = dict(smooth_keys=True, hadamard=had, bits_k=4, bits_v=bits_v, group_k=128, group_v=group_v,
                stages=stages, chunk_bytes=chunk)
    case = U.Case(L=2, T=T, H=H, dtype=dtype, dist="llama", seed=bits_v * 7 + T, page_size=16 if paged else 0,
                  profile=prof)
    want = _fusable(case)
    names = _run(case)
    assert ("kvc_enc_rows_lc" in names) == want, (names, want)


def test_split_encode_compressible_chunks():
    """Value rows that repeat (constant within each row, a few distinct rows): their
    code chunks compress, so the value encoder runs the stage transform itself."""
    prof = dict(smooth_keys=True, hadamard=False, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=FULL,
                chunk_bytes=16384)
    case = U.Case(L=1, T=1024, H=8, dtype="bf16", dist="llama", seed=3, profile=prof).materialize()
    pattern = torch.tensor([0.5, -1.25, 3.0, 0.0], dtype=torch.float32, device="cuda")
    rows = pattern[torch.arange(512, device="cuda") % 4]
    case.v[0][:512] = rows[:, None, None].expand(512, 8, 128).to(torch.bfloat16)
    case.materialize = lambda: case  # keep the planted rows
    assert _fusable(case)
    names = _run(case)
    assert "kvc_enc_rows_lc" in names


def test_split_is_off_by_default():
    prof = dict(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=FULL,
                chunk_bytes=16384)
    case = U.Case(L=2, T=512, H=8, dtype="bf16", dist="llama", seed=4, profile=prof).materialize()
    assert _fusable(case)
    codec = U.Codec(U.kvc_profile(prof), case.kvc_shape())
    kvc.kvc_timing_enable(codec.plan, True)
    codec.encode(case.k, case.v)
    codec.query()
    names = {n for n, _ in kvc.kvc_timing_read(codec.plan)}
    assert "kvc_enc_rows_lc" not in names and "kvc_enc_rows" in names


@pytest.mark.parametrize("prof", [
    dict(bits_v=3, group_v=128, stages=FULL, chunk_bytes=16384),       # 3-bit rows do not fill a chunk evenly
    dict(bits_v=4, group_v=128, stages=((1, 8), (4, 2)), chunk_bytes=16384),  # no BIT_8
    dict(bits_v=4, group_v=128, stages=FULL, chunk_bytes=1024),        # not a fast chunk size
    dict(bits_v=4, group_v=128, stages=FULL, chunk_bytes=16384, token_delta=True),
])
def test_profiles_outside_the_split_path(prof):
    prof = dict(smooth_keys=True, hadamard=True, bits_k=4, group_k=128, **prof)
    case = U.Case(L=1, T=512, H=8, dtype="bf16", dist="llama", seed=9, profile=prof)
    names = _run(case)
    assert "kvc_enc_rows_lc" not in names


@pytest.mark.parametrize("ticket", [3, 37])
def test_split_encode_lookback_wait_is_bounded(ticket):
    """A chunk that never publishes (before the value codes, or one of the value
    encoder's own): the look-backs that meet it run out, the status says TIMEOUT,
    and the next encode on the same plan is clean and matches the oracle."""
    prof = dict(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=FULL,
                chunk_bytes=16384)
    case = U.Case(L=2, T=512, H=8, dtype="bf16", dist="llama", seed=8, profile=prof).materialize()
    assert _fusable(case)
    lay = O.layout(U.oracle_profile(prof), case.oracle_shape())
    c0, nfull = lay.off[2] // 16384, lay.size[2] // 16384
    assert ticket < c0 or c0 <= ticket < c0 + nfull
    codec = U.Codec(U.kvc_profile(prof), case.kvc_shape())
    kvc.kvc_fuse_value_chunks(codec.plan, True)
    kvc.kvc_debug_lookback(codec.plan, ticket, 2000)
    codec.encode(case.k, case.v)
    st, _, flags = codec.query()
    assert st == kvc.KVC_ERR_TIMEOUT and flags & kvc.FLAG_TIMEOUT
    kvc.kvc_debug_lookback(codec.plan, -1, 0)
    sg = codec.encode(case.k, case.v)
    st, nbytes, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    so, _ = O.encode(U.oracle_profile(prof), case.oracle_shape(), case.host_bits(case.k), case.host_bits(case.v))
    assert np.array_equal(U.to_np(sg, nbytes), so)

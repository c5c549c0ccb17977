"""The rule for which code chunks kvc_decode reads in place, as bench.py restates
it to count the lossless decoder's bytes, agrees with the GPU tests' restatement
(which the GPU tests check against the library's launches) on every profile those
tests use and on a few more; every unit the in-place kernels read through one chunk
lookup lies inside one chunk under it; and the two execution-choice entry points
reject a null plan.  No GPU needed: plans are host objects."""
import numpy as np
import pytest

import bench
from kv_cache_compression_encode_gb300 import kvc
from oracle import oracle as O
from tests import parity_util as U
from tests.test_gpu_inplace import CASES, FULL, LC, _expected

MORE = [
    # (bits_k, bits_v, group_k, group_v, stages, chunk, L, T, H, dtype, had, page, extra)
    (2, 2, 64, 64, LC, 512, 4, 4096, 8, "bf16", True, 0, {}),        # V only: a 2-bit key tile is 4 KiB
    (4, 4, 128, 128, LC, 8192, 1, 512, 4, "bf16", True, 0, {}),
    (4, 4, 64, 64, LC, 1024, 1, 300, 2, "bf16", True, 0, {}),         # the corrupt-stream tests' profile
    (8, 8, 128, 128, LC, 16384, 80, 16384, 8, "bf16", True, 0, {}),   # Llama-70B's
    (2, 2, 32, 32, FULL, 16384, 32, 32768, 8, "bf16", False, 0, {}),  # 8B at 32K's
    (4, 4, 128, 128, FULL, 16384, 2, 512, 8, "bf16", True, 0, {"axis_v": 0}),  # values over tokens: key-tile decoder
]


@pytest.mark.parametrize("bk,bv,gk,gv,stages,chunk,L,T,H,dtype,had,page,extra", CASES + MORE)
def test_bench_rule_matches_the_tests_rule(bk, bv, gk, gv, stages, chunk, L, T, H, dtype, had, page, extra):
    prof = dict(smooth_keys=True, hadamard=had, bits_k=bk, bits_v=bv, group_k=gk, group_v=gv, stages=stages,
                chunk_bytes=chunk)
    prof.update(extra)
    case = U.Case(L=L, T=T, H=H, dtype=dtype, page_size=page, profile=prof)
    if page:
        case.n_pages = -(-T // page)
    plan = kvc.Plan(U.kvc_profile(prof), case.kvc_shape())
    lay = O.layout(U.oracle_profile(prof), case.oracle_shape())
    want = [(lay.off[2 * t] // chunk, (lay.off[2 * t] + lay.size[2 * t]) // chunk)
            for t, ok in enumerate(_expected(case)) if ok]
    assert bench.in_place_ranges(plan, T) == want


def test_mixed_widths_are_outside_the_rule():
    bm = [[2, 8, 4, 4], [8, 2, 4, 2]]
    prof = dict(bits_k=4, bits_v=4, group_k=128, group_v=128, stages=FULL, chunk_bytes=16384, bits_map_k=bm,
                bits_map_v=bm)
    plan = kvc.Plan(kvc.make_profile(**prof), kvc.make_shape(2, 512, 4, 128, kvc.BF16))
    assert bench.in_place_ranges(plan, 512) == []


def test_execution_choices_reject_a_null_plan():
    lib = kvc.load()
    assert lib.kvc_decode_codes_in_place(None, 1) == kvc.KVC_ERR_INVALID_ARG
    assert lib.kvc_fuse_value_chunks(None, 1) == kvc.KVC_ERR_INVALID_ARG
    plan = kvc.Plan(kvc.make_profile(stages=FULL), kvc.make_shape(1, 128, 2, 128, kvc.BF16))
    kvc.kvc_decode_codes_in_place(plan, False)
    kvc.kvc_decode_codes_in_place(plan, True)
    kvc.kvc_fuse_value_chunks(plan, True)
    assert plan.launches == 0


@pytest.mark.parametrize("bk,bv,gk,gv,stages,chunk,L,T,H,dtype,had,page,extra", CASES + MORE)
def test_units_read_in_place_stay_inside_one_chunk(bk, bv, gk, gv, stages, chunk, L, T, H, dtype, had, page,
                                                   extra):
    """What the in-place kernels rely on: each unit they read through one chunk
    lookup -- a key-style tile (2048 bits bytes from its first record) or a value
    step (the codes of 16 consecutive rows) -- lies inside one chunk wherever the
    rule reads that tensor in place.  Every unit of every accepted profile, from the
    oracle's layout."""
    prof = dict(smooth_keys=True, hadamard=had, bits_k=bk, bits_v=bv, group_k=gk, group_v=gv, stages=stages,
                chunk_bytes=chunk)
    prof.update(extra)
    case = U.Case(L=L, T=T, H=H, dtype=dtype, page_size=page, profile=prof)
    if page:
        case.n_pages = -(-T // page)
    plan = kvc.Plan(U.kvc_profile(prof), case.kvc_shape())
    lay = O.layout(U.oracle_profile(prof), case.oracle_shape())
    ranges = bench.in_place_ranges(plan, T)
    for t, ok in enumerate(_expected(case)):
        if not ok:
            continue
        bits = bv if t else bk
        G = gv if t else gk
        off, size = lay.off[2 * t], lay.size[2 * t]
        assert (off // chunk, (off + size) // chunk) in ranges
        if prof.get("axis_v" if t else "axis_k", 1 if t else 0) == 0:  # tiles over tokens
            n_tg, ng, rec = -(-T // G), 128 // G, G * bits // 8
            lh = np.arange(L * H, dtype=np.int64)[:, None]
            sb = np.arange(-(-T // 128), dtype=np.int64)[None, :]
            start = off + (lh * n_tg + sb * ng) * 128 * rec
            length = np.minimum(ng, n_tg - sb * ng) * 128 * rec  # the tile's groups
            assert (length == 2048 * bits).all()
        else:  # value steps of 16 rows
            NR = L * T * H
            itn = np.arange(-(-NR // 16), dtype=np.int64)
            start = off + itn * 256 * bits
            length = np.minimum(16, NR - 16 * itn) * 16 * bits
        end = start + length
        assert (start // chunk == (end - 1) // chunk).all()
        assert end.max() <= off + size

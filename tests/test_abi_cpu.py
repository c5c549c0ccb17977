"""Host-side checks of the C ABI (no GPU needed, no compute calls):
the library builds for sm_103a and loads, exports every entry point declared in
include/kvc.h, the ctypes mirrors match the C struct layouts, and plan validation
and the payload layout agree with the oracle's layout."""
import ctypes as C
import os
import re
import subprocess

import pytest

from kv_cache_compression_encode_gb300 import build, kvc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvc.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kvc.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 19
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (kvc_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert set(kvc.EXPORTS) <= exported
    for n in names:
        assert hasattr(lib, n)


def test_struct_layouts_match_c(tmp_path):
    src = tmp_path / "sz.c"
    src.write_text(f"""
#include <stdio.h>
#include <stddef.h>
#include "{HEADER}"
int main(void) {{
  printf("%zu %zu %zu %zu\\n", sizeof(kvc_profile), sizeof(kvc_shape), sizeof(kvc_kv), sizeof(kvc_timing));
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %d\\n", offsetof(kvc_profile, group_k), offsetof(kvc_profile, stages),
         offsetof(kvc_profile, chunk_bytes), offsetof(kvc_profile, hadamard_seed), offsetof(kvc_profile, n_stages),
         offsetof(kvc_profile, token_delta), offsetof(kvc_profile, bits_map_k), offsetof(kvc_profile, bits_map_v),
         KVC_PROFILE_V1_SIZE);
  printf("%zu %zu %zu\\n", offsetof(kvc_shape, num_pages), offsetof(kvc_shape, token_stride),
         offsetof(kvc_shape, page_stride));
  return 0;
}}""")
    exe = tmp_path / "sz"
    subprocess.check_call(["gcc", "-std=c11", str(src), "-o", str(exe)])
    lines = subprocess.check_output([str(exe)], text=True).split("\n")
    assert [int(x) for x in lines[0].split()] == [C.sizeof(kvc.Profile), C.sizeof(kvc.Shape), C.sizeof(kvc.KV),
                                                    C.sizeof(kvc.Timing)]
    P = kvc.Profile
    assert [int(x) for x in lines[1].split()] == [P.group_k.offset, P.stages.offset, P.chunk_bytes.offset,
                                                    P.hadamard_seed.offset, P.n_stages.offset, P.token_delta.offset,
                                                    P.bits_map_k.offset, P.bits_map_v.offset, kvc.PROFILE_V1_SIZE]
    assert P.token_delta.offset == kvc.PROFILE_V1_SIZE  # the v2 fields extend the v1 struct
    S = kvc.Shape
    assert [int(x) for x in lines[2].split()] == [S.num_pages.offset, S.token_stride.offset, S.page_stride.offset]


CASES = [
    (dict(bits_k=4, bits_v=4, group_k=128, group_v=128, hadamard=True, stages=((1, 8), (2, 8), (3, 1), (4, 2))),
     (32, 4096, 8)),
    (dict(bits_k=2, bits_v=2, group_k=32, group_v=32, stages=((1, 8), (2, 8), (4, 2))), (32, 32768, 8)),
    (dict(bits_k=8, bits_v=8, group_k=128, group_v=128, hadamard=True, stages=((1, 8), (2, 8), (4, 2))),
     (80, 16384, 8)),
    (dict(bits_k=3, bits_v=3, group_k=64, group_v=32, smooth_keys=False), (3, 333, 5)),
    (dict(bits_k=3, bits_v=2, group_k=32, group_v=64, axis_k=1, axis_v=0, stages=((4, 4),), chunk_bytes=1024),
     (2, 77, 3)),
    (dict(bits_k=4, bits_v=4, group_k=64, group_v=64, stages=((1, 8), (4, 1))), (1, 0, 8)),
    # format v2: token delta; per-(layer, head) widths (both axes); both
    (dict(bits_k=4, bits_v=4, group_k=128, group_v=128, hadamard=True, token_delta=True,
          stages=((1, 8), (2, 8), (3, 1), (4, 2))), (4, 300, 8)),
    (dict(bits_k=4, bits_v=4, group_k=64, group_v=32, bits_map_k=[[2, 3, 4, 8]] * 3, bits_map_v=[[8, 8, 2, 2]] * 3,
          stages=((1, 8), (4, 2)), chunk_bytes=4096), (3, 200, 4)),
    (dict(bits_k=4, bits_v=4, group_k=32, group_v=64, smooth_keys=False, axis_k=1, axis_v=0,
          bits_map_k=[[2, 8]] * 5, token_delta=True), (5, 129, 2)),
]


@pytest.mark.parametrize("kw,geom", CASES)
def test_plan_layout_equals_oracle_layout(lib, oracle, kw, geom):
    L, T, H = geom
    prof = kvc.make_profile(**kw)
    shape = kvc.make_shape(L, T, H, 128, kvc.BF16)
    plan = kvc.Plan(prof, shape)
    okw = dict(kw)
    lay = oracle.layout(oracle.make_profile(**okw), oracle.make_shape(L, T, H, 128, 2))
    assert plan.payload_bytes == lay.payload_bytes
    assert plan.max_stream_bytes == lay.max_stream_bytes
    assert plan.n_chunks == lay.n_chunks
    assert plan.header_bytes == lay.header_bytes
    for i in range(8):
        assert plan.section(i) == (lay.off[i], lay.size[i])
    assert plan.workspace_bytes >= 256 + 8 * plan.n_chunks + (plan.payload_bytes if kw.get("stages") else 0)
    plan.close()


@pytest.mark.parametrize("bad,status", [
    (dict(bits_k=5), kvc.KVC_ERR_INVALID_ARG),
    (dict(group_v=16), kvc.KVC_ERR_INVALID_ARG),
    (dict(axis_k=2), kvc.KVC_ERR_INVALID_ARG),
    (dict(stages=((4, 2), (1, 8))), kvc.KVC_ERR_INVALID_ARG),   # RZE must be last
    (dict(stages=((2, 4),)), kvc.KVC_ERR_INVALID_ARG),          # BIT takes 8 only
    (dict(stages=((1, 3),)), kvc.KVC_ERR_INVALID_ARG),
    (dict(stages=((1, 8),), chunk_bytes=1000), kvc.KVC_ERR_INVALID_ARG),
])
def test_plan_rejects_bad_profiles(lib, bad, status):
    kw = dict(bits_k=4, bits_v=4, group_k=64, group_v=64)
    kw.update(bad)
    with pytest.raises(kvc.KvcError) as e:
        kvc.Plan(kvc.make_profile(**kw), kvc.make_shape(1, 16, 1, 128, kvc.BF16))
    assert e.value.status == status


def test_plan_accepts_the_v1_profile_struct(lib, oracle):
    """A caller built against the 40-byte profile (before the format-v2 fields) gets
    the same plan as one passing the full struct with the v2 fields unset."""
    full = kvc.make_profile(bits_k=3, bits_v=4, group_k=64, group_v=32, hadamard=True, stages=((1, 8), (4, 2)))
    v1 = kvc.make_profile(bits_k=3, bits_v=4, group_k=64, group_v=32, hadamard=True, stages=((1, 8), (4, 2)))
    v1.struct_size = kvc.PROFILE_V1_SIZE
    v1.token_delta = 1            # beyond the v1 size: must be ignored
    shape = kvc.make_shape(2, 100, 3, 128, kvc.BF16)
    a, b = kvc.Plan(full, shape), kvc.Plan(v1, shape)
    assert (a.payload_bytes, a.header_bytes, a.max_stream_bytes) == (b.payload_bytes, b.header_bytes,
                                                                     b.max_stream_bytes)
    assert b.section(6) == (b.payload_bytes, 0)
    bad = kvc.make_profile()
    bad.struct_size = 44
    with pytest.raises(kvc.KvcError) as e:
        kvc.Plan(bad, shape)
    assert e.value.status == kvc.KVC_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,geom,status", [
    (dict(bits_map_k=[[2, 5]]), (1, 16, 2), kvc.KVC_ERR_INVALID_ARG),            # width 5
    (dict(bits_map_v=[[4] * 8] * 257), (257, 16, 8), kvc.KVC_ERR_INVALID_ARG),  # too many layers anyway
    (dict(bits_map_k=[[4] * 64] * 33), (33, 16, 64), kvc.KVC_ERR_UNSUPPORTED),  # > 2048 map entries
])
def test_plan_rejects_bad_v2_profiles(lib, kw, geom, status):
    L, T, H = geom
    with pytest.raises(kvc.KvcError) as e:
        kvc.Plan(kvc.make_profile(**kw), kvc.make_shape(L, T, H, 128, kvc.BF16))
    assert e.value.status == status


def test_plan_rejects_bad_shapes(lib):
    prof = kvc.make_profile()
    for shape, status in [(kvc.make_shape(1, 16, 1, 64, kvc.BF16), kvc.KVC_ERR_UNSUPPORTED),
                          (kvc.make_shape(1, 16, 1, 128, 7), kvc.KVC_ERR_INVALID_ARG),
                          (kvc.make_shape(1, 16, 0, 128, kvc.BF16), kvc.KVC_ERR_INVALID_ARG),
                          (kvc.make_shape(300, 16, 1, 128, kvc.BF16), kvc.KVC_ERR_INVALID_ARG),
                          (kvc.make_shape(1, 16, 2, 128, kvc.BF16, token_stride=100), kvc.KVC_ERR_INVALID_ARG),
                          (kvc.make_shape(1, 16, 2, 128, kvc.BF16, page_size=12, num_pages=4, page_stride=12 * 512),
                           kvc.KVC_ERR_INVALID_ARG),
                          (kvc.make_shape(256, 2 ** 31 - 1, 8, 128, kvc.BF16), kvc.KVC_ERR_UNSUPPORTED)]:
        with pytest.raises(kvc.KvcError) as e:
            kvc.Plan(prof, shape)
        assert e.value.status == status


def test_entry_points_reject_bad_arguments_before_launching(lib):
    plan = kvc.Plan(kvc.make_profile(stages=((1, 8), (4, 1))), kvc.make_shape(1, 64, 2, 128, kvc.BF16))
    kv = kvc.KVRef([16], [32])
    with pytest.raises(kvc.KvcError) as e:   # stream capacity below the worst case
        kvc.kvc_encode(plan, kv, 4096, plan.max_stream_bytes - 1, 8192, plan.workspace_bytes)
    assert e.value.status == kvc.KVC_ERR_CAPACITY
    with pytest.raises(kvc.KvcError) as e:   # workspace too small
        kvc.kvc_encode(plan, kv, 4096, plan.max_stream_bytes, 8192, plan.workspace_bytes - 1)
    assert e.value.status == kvc.KVC_ERR_CAPACITY
    with pytest.raises(kvc.KvcError) as e:   # misaligned stream pointer
        kvc.kvc_encode(plan, kv, 4097, plan.max_stream_bytes, 8192, plan.workspace_bytes)
    assert e.value.status == kvc.KVC_ERR_INVALID_ARG
    with pytest.raises(kvc.KvcError) as e:   # misaligned layer pointer
        kvc.kvc_encode(plan, kvc.KVRef([17], [32]), 4096, plan.max_stream_bytes, 8192, plan.workspace_bytes)
    assert e.value.status == kvc.KVC_ERR_INVALID_ARG
    with pytest.raises(kvc.KvcError) as e:   # block table without a page size
        kvc.kvc_encode(plan, kvc.KVRef([16], [32], 64), 4096, plan.max_stream_bytes, 8192, plan.workspace_bytes)
    assert e.value.status == kvc.KVC_ERR_INVALID_ARG
    assert plan.launches == 0
    assert kvc.status_str(kvc.KVC_ERR_CORRUPT) == "corrupt stream"

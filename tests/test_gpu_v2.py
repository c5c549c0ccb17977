"""GPU (sm_103a) versus oracle for the format-v2 profile features, through the C ABI:

* per-(layer, head) code widths ("KVServe" §5.1 layer- and head-wise mixed
  precision): key tiles take their head's width per tile, value rows run in
  (layer, head, token) order; token counts that are not multiples of 16 make a
  warp's rows straddle two heads of different widths;
* the token-delta transformer ("KVServe" §5.1 Delta, after CacheGen): anchors are
  the first token of every 128-token block, for K (key tile) and V (rows).

Streams, payloads and reconstructions must equal the oracle's byte for byte, as
for format v1 (tests/test_gpu_parity.py)."""
import numpy as np
import pytest

from kv_cache_compression_encode_gb300 import kvc
from tests import parity_util as U
from tests.test_gpu_parity import FULL, LC, _run_full

pytestmark = pytest.mark.gpu


def _map(L, H, seed):
    rng = np.random.default_rng(seed)
    m = rng.choice([2, 3, 4, 8], size=(L, H))
    m[0, 0], m[-1, -1] = 2, 8
    return m.astype(np.uint8)


@pytest.mark.parametrize("had", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("bits,group", [(2, 32), (3, 64), (4, 128), (8, 64)])
def test_token_delta(had, dtype, bits, group):
    prof = dict(smooth_keys=True, hadamard=had, bits_k=bits, bits_v=bits, group_k=group, group_v=group,
                stages=FULL, chunk_bytes=4096, token_delta=True)
    _run_full(U.Case(L=2, T=300, H=3, dtype=dtype, dist="llama", seed=bits + group, profile=prof))


@pytest.mark.parametrize("smooth", [False, True])
def test_token_delta_axes_and_paging(smooth):
    for axis_k, axis_v in ((0, 1), (0, 0), (1, 1)):
        prof = dict(smooth_keys=smooth, hadamard=True, bits_k=4, bits_v=3, group_k=64, group_v=32, axis_k=axis_k,
                    axis_v=axis_v, stages=LC, chunk_bytes=2048, token_delta=True)
        _run_full(U.Case(L=2, T=200, H=2, dtype="bf16", dist="llama_sink", seed=7, profile=prof))
    prof = dict(smooth_keys=smooth, hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128, stages=LC,
                chunk_bytes=4096, token_delta=True)
    _run_full(U.Case(L=2, T=1000, H=8, dtype="bf16", dist="llama", seed=5, page_size=16, profile=prof))


@pytest.mark.parametrize("T", [1, 15, 129, 300])
@pytest.mark.parametrize("had", [False, True])
def test_mixed_widths(T, had):
    L, H = 3, 5
    prof = dict(smooth_keys=True, hadamard=had, bits_k=4, bits_v=4, group_k=64, group_v=32,
                bits_map_k=_map(L, H, T), bits_map_v=_map(L, H, T + 1), stages=FULL, chunk_bytes=2048)
    _run_full(U.Case(L=L, T=T, H=H, dtype="bf16", dist="llama", seed=T, profile=prof))


@pytest.mark.parametrize("axes,smooth", [((0, 0), False), ((1, 1), False), ((0, 1), False), ((1, 1), True),
                                         ((1, 0), True)])
def test_mixed_widths_axes_with_delta(axes, smooth):
    """Smoothed keys grouped over channels take the generic tile kernels."""
    L, H = 2, 4
    prof = dict(smooth_keys=smooth, hadamard=True, bits_k=4, bits_v=4, group_k=32, group_v=64, axis_k=axes[0],
                axis_v=axes[1], bits_map_k=_map(L, H, 3), bits_map_v=_map(L, H, 4), stages=LC, chunk_bytes=1024,
                token_delta=True)
    _run_full(U.Case(L=L, T=333, H=H, dtype="f16", dist="gauss_outlier", seed=9, profile=prof))


def test_mixed_widths_only_one_tensor_mapped_paged():
    L, H = 2, 8
    prof = dict(smooth_keys=True, hadamard=True, bits_k=3, bits_v=4, group_k=128, group_v=128,
                bits_map_v=_map(L, H, 8), stages=LC, chunk_bytes=4096)
    _run_full(U.Case(L=L, T=700, H=H, dtype="bf16", dist="llama", seed=12, page_size=16, profile=prof))


def test_stream_with_another_width_map_is_rejected():
    import torch

    from kv_cache_compression_encode_gb300.codec import Codec
    L, H = 2, 4
    m = _map(L, H, 1)
    prof = dict(smooth_keys=True, bits_k=4, bits_v=4, group_k=64, group_v=64, bits_map_k=m, bits_map_v=m,
                stages=LC, chunk_bytes=2048)
    case = U.Case(L=L, T=256, H=H, profile=prof, seed=2).materialize()
    codec = Codec(kvc.make_profile(**prof), case.kvc_shape())
    sg = codec.encode(case.k, case.v)
    st, nbytes, _ = codec.query()
    assert st == kvc.KVC_OK
    m2 = m.copy()
    m2[1, 2] = 8 if m2[1, 2] != 8 else 2
    other = Codec(kvc.make_profile(**dict(prof, bits_map_k=m2)), case.kvc_shape())
    ok, ov = case.empty_like_kv(fill=0x1234)
    other.decode(sg, nbytes, ok, ov)
    st, _, flags = other.query()
    assert st == kvc.KVC_ERR_CORRUPT and flags & kvc.FLAG_CORRUPT
    for t in ok + ov:
        assert bool((t.view(torch.int16) == 0x1234).all())


@pytest.mark.parametrize("delta", [False, True])
def test_tile_kernels_mixed_widths_ragged(delta):
    L, H = 3, 3
    prof = dict(smooth_keys=True, hadamard=False, bits_k=4, bits_v=4, group_k=64, group_v=32, axis_k=1, axis_v=1,
                bits_map_k=_map(L, H, 21), bits_map_v=_map(L, H, 22), stages=FULL, chunk_bytes=1024,
                token_delta=delta)
    _run_full(U.Case(L=L, T=201, H=H, dtype="bf16", dist="llama_sink", seed=13, profile=prof))

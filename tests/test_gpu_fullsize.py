"""Full-size parity: the five workloads at their real sizes, in the configuration
the benchmark times (default 16 KiB chunks, all layers in one call).

* tiny, llama8b, llama8b_32k, llama70b, and the format-v2 variants of llama8b
  (head-wise mixed widths; token delta): the whole stream and the whole
  reconstruction equal the oracle's, byte for byte.
* paged8b_128k (48 profiles, 17 GB of KV each): every run is encoded on the GPU
  through the paged gather; the payload slices of two sampled layers per profile
  equal the oracle's (run on those layers through the same block table), the
  GPU lossless round trip returns the payload, and four profiles (2, 3 and 8
  bits; groups 32, 64 and 128) are compared on the whole stream; one profile is
  decoded at full size and scattered through the block table, and sampled layers
  equal the oracle's reconstruction.
"""
import os

import numpy as np
import pytest
import torch

from kv_cache_compression_encode_gb300 import kvc, synth
from kv_cache_compression_encode_gb300.codec import Codec
from kv_cache_compression_encode_gb300.workloads import PROFILES, V2_PROFILES, WORKLOADS, paged_sweep
from oracle import oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _threads():
    O.set_threads(len(os.sched_getaffinity(0)))


def _dt(w):
    return (kvc.BF16, 2) if w.dtype == "bf16" else (kvc.F16, 1)


def _bits(tensors):
    return [synth.to_bits_numpy(t) for t in tensors]


@pytest.mark.parametrize("name", ["tiny", "llama8b", "llama8b_32k", "llama70b", "llama8b_mixhq", "llama8b_delta"])
def test_workload_stream_and_reconstruction(name):
    # the format-v2 variants run on the Llama-8B workload
    w = WORKLOADS[name if name in WORKLOADS else "llama8b"]
    prof = PROFILES[name] if name in PROFILES else V2_PROFILES[name]
    dk, do = _dt(w)
    k, v = [], []
    for l in range(w.layers):
        a, b = synth.layer_kv(w.dist, l, w.tokens, w.kv_heads, w.head_dim, w.dtype, w.seed, "cuda")
        k.append(a.contiguous())
        v.append(b.contiguous())
    codec = Codec(kvc.make_profile(**prof), kvc.make_shape(w.layers, w.tokens, w.kv_heads, w.head_dim, dk))
    sg = codec.encode(k, v)
    st, nbytes, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    hk, hv = _bits(k), _bits(v)
    oprof, oshape = O.make_profile(**prof), O.make_shape(w.layers, w.tokens, w.kv_heads, w.head_dim, do)
    so, fo = O.encode(oprof, oshape, hk, hv)
    assert fo == 0 and nbytes == so.size
    got = sg[:nbytes].cpu().numpy()
    assert np.array_equal(got, so), f"first differing byte {np.flatnonzero(got != so)[:4]}"
    del got
    # decode on the GPU; the oracle decodes its own stream
    ok = [torch.empty_like(x) for x in k]
    ov = [torch.empty_like(x) for x in v]
    codec.decode(sg, nbytes, ok, ov)
    st, _, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    del k, v, sg
    rk = [np.empty_like(a) for a in hk]
    rv = [np.empty_like(a) for a in hv]
    assert O.decode(oprof, oshape, so, rk, rv) == 0
    for l in range(w.layers):
        assert np.array_equal(synth.to_bits_numpy(ok[l]), rk[l]), f"K layer {l}"
        assert np.array_equal(synth.to_bits_numpy(ov[l]), rv[l]), f"V layer {l}"


@pytest.fixture(scope="module")
def paged_kv():
    w = WORKLOADS["paged8b_128k"]
    P = w.page_size
    n_pages = w.tokens // P
    bt = synth.block_table(w.tokens, P, w.seed)
    k, v = [], []
    for l in range(w.layers):
        a, b = synth.paged_layer_kv(w.dist, l, w.tokens, P, w.kv_heads, w.head_dim, w.dtype, w.seed, "cuda")
        k.append(a.contiguous())
        v.append(b.contiguous())
    torch.cuda.synchronize()
    yield w, k, v, bt, n_pages
    del k, v
    torch.cuda.empty_cache()


SWEEP = paged_sweep()
# whole streams against the oracle: 2-, 3- and 8-bit, groups of 32, 64 and 128, Hadamard on and off
FULL_STREAM = {"b2g32_lc", "b8g128h_lc", "b3g64h_lc", "b3g32_lc"}


@pytest.mark.parametrize("idx", range(len(SWEEP)), ids=[n for n, _ in SWEEP])
def test_paged_sweep(paged_kv, idx):
    name, prof = SWEEP[idx]
    w, k, v, bt, n_pages = paged_kv
    P = w.page_size
    shape = kvc.make_shape(w.layers, w.tokens, w.kv_heads, w.head_dim, kvc.BF16, page_size=P, num_pages=n_pages,
                           page_stride=P * w.kv_heads * w.head_dim * 2)
    codec = Codec(kvc.make_profile(**prof), shape)
    btd = bt.cuda()
    Qg = codec.quantize(k, v, btd)
    st, _, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    # two sampled layers (different for every profile) against the oracle on those layers
    layers = [(3 * idx) % w.layers, (3 * idx + 17) % w.layers]
    oprof = O.make_profile(**prof)
    oshape = O.make_shape(len(layers), w.tokens, w.kv_heads, w.head_dim, 2, page_size=P,
                          page_stride=P * w.kv_heads * w.head_dim * 2)
    Qo, fo = O.quantize(oprof, oshape, [synth.to_bits_numpy(k[l]) for l in layers],
                        [synth.to_bits_numpy(v[l]) for l in layers], bt.numpy())
    assert fo == 0
    lay_o = O.layout(oprof, oshape)
    for sec in range(6):
        off_g, size_g = codec.plan.section(sec)
        per = size_g // w.layers
        assert per * len(layers) == lay_o.size[sec]
        for j, l in enumerate(layers):
            g = Qg[off_g + l * per: off_g + (l + 1) * per].cpu().numpy()
            o = Qo[lay_o.off[sec] + j * per: lay_o.off[sec] + (j + 1) * per]
            assert np.array_equal(g, o), (name, sec, l)
    if prof["stages"]:
        sg = codec.lossless_encode(Qg)
        st, nbytes, flags = codec.query()
        assert st == kvc.KVC_OK and flags == 0
        back = codec.lossless_decode(sg, nbytes)
        st, _, flags = codec.query()
        assert st == kvc.KVC_OK and flags == 0
        assert torch.equal(back[:codec.plan.payload_bytes], Qg[:codec.plan.payload_bytes])
        if name in FULL_STREAM:
            full_shape = O.make_shape(w.layers, w.tokens, w.kv_heads, w.head_dim, 2, page_size=P,
                                      page_stride=P * w.kv_heads * w.head_dim * 2)
            so, fo = O.encode(oprof, full_shape, [synth.to_bits_numpy(x) for x in k],
                              [synth.to_bits_numpy(x) for x in v], bt.numpy())
            assert fo == 0 and so.size == nbytes
            assert np.array_equal(sg[:nbytes].cpu().numpy(), so)


@pytest.mark.parametrize("name", ["b4g128h_lc", "b3g64_lc"])
def test_paged_decode_scatter_full_size(paged_kv, name):
    """Full-size decode through the 131072-token block table: every page the table
    maps is written, and two sampled layers equal the oracle's reconstruction of
    the same payload through the same table."""
    prof = dict(SWEEP)[name]
    w, k, v, bt, n_pages = paged_kv
    P = w.page_size
    shape = kvc.make_shape(w.layers, w.tokens, w.kv_heads, w.head_dim, kvc.BF16, page_size=P, num_pages=n_pages,
                           page_stride=P * w.kv_heads * w.head_dim * 2)
    codec = Codec(kvc.make_profile(**prof), shape)
    btd = bt.cuda()
    sg = codec.encode(k, v, btd)
    st, nbytes, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    ok = [torch.full_like(x, 0).view(torch.int16).fill_(0x7E7E).view(x.dtype) for x in k]
    ov = [torch.full_like(x, 0).view(torch.int16).fill_(0x7E7E).view(x.dtype) for x in v]
    codec.decode(sg, nbytes, ok, ov, btd)
    st, _, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    del sg
    layers = [5, 26]
    oprof = O.make_profile(**prof)
    oshape = O.make_shape(len(layers), w.tokens, w.kv_heads, w.head_dim, 2, page_size=P,
                          page_stride=P * w.kv_heads * w.head_dim * 2)
    Qo, fo = O.quantize(oprof, oshape, [synth.to_bits_numpy(k[l]) for l in layers],
                        [synth.to_bits_numpy(v[l]) for l in layers], bt.numpy())
    assert fo == 0
    rk = [np.zeros_like(synth.to_bits_numpy(k[l])) for l in layers]
    rv = [np.zeros_like(synth.to_bits_numpy(v[l])) for l in layers]
    O.dequantize(oprof, oshape, Qo, rk, rv, bt.numpy())
    for j, l in enumerate(layers):
        assert np.array_equal(synth.to_bits_numpy(ok[l]), rk[j]), f"K layer {l}"
        assert np.array_equal(synth.to_bits_numpy(ov[l]), rv[j]), f"V layer {l}"
    # the table is a permutation of every page: no canary may survive anywhere
    for t in ok + ov:
        assert not bool((t.view(torch.int16) == 0x7E7E).all(dim=-1).any())

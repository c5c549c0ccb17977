"""Lossless stage pipeline on the GPU versus the oracle, on payloads of controlled
compressibility (the quantized payload of Gaussian KV is nearly incompressible,
so these cases make every chunk path run: raw, compressed, all-zero, mixed).

The payload is drawn with numpy and handed to both sides; the GPU stream must
equal the oracle's byte for byte, and decoding either stream on the GPU must
return the payload."""
import numpy as np
import pytest
import torch

from kv_cache_compression_encode_gb300 import kvc
from kv_cache_compression_encode_gb300.codec import Codec
from oracle import oracle as O

pytestmark = pytest.mark.gpu

PIPES = {
    "lc": ((1, 8), (2, 8), (4, 2)),
    "full": ((1, 8), (2, 8), (3, 1), (4, 2)),
    "shuffle_zero": ((1, 8), (4, 1)),
    "tupl_delta_rze2": ((1, 8), (3, 1), (4, 2)),
    "bit_rze1": ((1, 8), (2, 8), (4, 1)),
    "generic_delta2": ((3, 2), (4, 2)),
    "generic_t4": ((1, 4), (2, 8), (4, 4)),
    "generic_t2": ((1, 2), (3, 4), (4, 1)),
}


def _payload(kind, n, rng):
    if kind == "zeros":
        return np.zeros(n, np.uint8)
    if kind == "random":
        return rng.integers(0, 256, n, dtype=np.uint8)
    if kind == "sparse_bytes":
        return np.where(rng.random(n) < 0.07, rng.integers(1, 256, n), 0).astype(np.uint8)
    if kind == "sparse_words":
        w = np.where(rng.random(n // 2) < 0.2, rng.integers(1, 65536, n // 2), 0).astype(np.uint16)
        return np.concatenate([w.view(np.uint8), np.zeros(n - 2 * (n // 2), np.uint8)])
    if kind == "low_nibbles":  # codes that use only a few values (2-bit-like payload)
        c = np.clip(np.round(rng.standard_normal(n) * 0.6 + 1.5), 0, 3).astype(np.uint8)
        return (c | (c << 2) | (np.roll(c, 1) << 4)).astype(np.uint8)
    if kind == "mixed":  # alternating compressible and incompressible regions
        out = rng.integers(0, 256, n, dtype=np.uint8)
        blk = 3000
        for s in range(0, n, 2 * blk):
            out[s:s + blk] = np.where(rng.random(min(blk, n - s)) < 0.05, 9, 0)
        return out
    raise ValueError(kind)


def _plan_for(stages, chunk, tokens):
    prof = dict(smooth_keys=True, bits_k=4, bits_v=4, group_k=64, group_v=64, stages=stages, chunk_bytes=chunk)
    shape_k = kvc.make_shape(1, tokens, 4, 128, kvc.BF16)
    return prof, Codec(kvc.make_profile(**prof), shape_k), O.make_shape(1, tokens, 4, 128, 2)


@pytest.mark.parametrize("pipe", list(PIPES))
@pytest.mark.parametrize("chunk,tokens", [(512, 96), (1024, 300), (4096, 700), (16384, 1000), (16384, 1024),
                                          (768, 200), (65536, 900)])
def test_lossless_matches_oracle(pipe, chunk, tokens):
    stages = PIPES[pipe]
    prof, codec, oshape = _plan_for(stages, chunk, tokens)
    oprof = O.make_profile(**prof)
    n = codec.plan.payload_bytes
    rng = np.random.default_rng(chunk + tokens)
    for kind in ("zeros", "random", "sparse_bytes", "sparse_words", "low_nibbles", "mixed"):
        Q = _payload(kind, n, rng)
        so = O.lossless_encode(oprof, oshape, Q)
        dQ = torch.from_numpy(Q).cuda()
        sg = codec.lossless_encode(dQ)
        st, nbytes, flags = codec.query()
        assert st == kvc.KVC_OK and flags == 0, (kind, st, flags)
        got = sg[:nbytes].cpu().numpy()
        assert nbytes == so.size and np.array_equal(got, so), \
            (pipe, chunk, kind, nbytes, so.size, np.flatnonzero(got[:min(nbytes, so.size)] != so[:min(nbytes, so.size)])[:5])
        for stream in (sg, torch.from_numpy(so).cuda()):
            back = codec.lossless_decode(stream, nbytes)
            st, _, flags = codec.query()
            assert st == kvc.KVC_OK and flags == 0, (kind, st, flags)
            assert np.array_equal(back[:n].cpu().numpy(), Q), (pipe, chunk, kind)

"""Helpers that run one case through the CUDA library (via the C ABI) and through
the oracle on the same seeded bytes, and compare them.

Bars: quantized payload bytes, the lossless stream and the stream size are
bit-exact; reconstructed K/V are within 1e-3 relative or one quantization step
of the oracle's reconstruction (and expected to be bit-exact, checked apart)."""
from __future__ import annotations

import os
from dataclasses import dataclass, field

import numpy as np
import torch

from kv_cache_compression_encode_gb300 import kvc, synth
from kv_cache_compression_encode_gb300.codec import Codec
from oracle import oracle as O

DT = {"f16": (kvc.F16, 1), "bf16": (kvc.BF16, 2)}


@dataclass
class Case:
    L: int
    T: int
    H: int
    dtype: str = "bf16"
    dist: str = "llama"
    seed: int = 1
    page_size: int = 0
    profile: dict = field(default_factory=dict)
    gen_device: str = "cpu"
    k: list = None          # per-layer CUDA tensors ([T,H,D] or [pages,P,H,D])
    v: list = None
    block_table: torch.Tensor = None
    n_pages: int = 0

    def materialize(self):
        D = 128
        if self.page_size:
            self.n_pages = max(1, -(-self.T // self.page_size))
            bt = synth.block_table(self.n_pages * self.page_size, self.page_size, self.seed)
            self.block_table = bt.cuda()
            pairs = [synth.paged_layer_kv(self.dist, l, self.T, self.page_size, self.H, D, self.dtype, self.seed,
                                          self.gen_device) for l in range(self.L)]
        else:
            pairs = [synth.layer_kv(self.dist, l, self.T, self.H, D, self.dtype, self.seed, self.gen_device)
                     for l in range(self.L)]
        self.k = [p[0].cuda().contiguous() for p in pairs]
        self.v = [p[1].cuda().contiguous() for p in pairs]
        return self

    def kvc_shape(self):
        dt = DT[self.dtype][0]
        if self.page_size:
            return kvc.make_shape(self.L, self.T, self.H, 128, dt, page_size=self.page_size, num_pages=self.n_pages,
                                  page_stride=self.page_size * self.H * 128 * 2)
        return kvc.make_shape(self.L, self.T, self.H, 128, dt)

    def oracle_shape(self):
        dt = DT[self.dtype][1]
        if self.page_size:
            return O.make_shape(self.L, self.T, self.H, 128, dt, page_size=self.page_size,
                                page_stride=self.page_size * self.H * 128 * 2)
        return O.make_shape(self.L, self.T, self.H, 128, dt)

    def host_bits(self, tensors):
        return [synth.to_bits_numpy(t) for t in tensors]

    def bt_host(self):
        return None if self.block_table is None else self.block_table.cpu().numpy()

    def empty_like_kv(self, fill=0x7E7E):
        # a canary pattern so that rows the decoder fails to write show up
        mk = lambda t: torch.full_like(t, 0).view(torch.int16).fill_(fill).view(t.dtype)  # noqa: E731
        return [mk(t) for t in self.k], [mk(t) for t in self.v]


def kvc_profile(kw):
    return kvc.make_profile(**kw)


def oracle_profile(kw):
    return O.make_profile(**kw)


def to_np(t: torch.Tensor, n: int | None = None) -> np.ndarray:
    a = t.detach().cpu().numpy().view(np.uint8)
    return a if n is None else a[:n]


def set_oracle_threads():
    O.set_threads(len(os.sched_getaffinity(0)))


def quantize_both(case: Case):
    codec = Codec(kvc_profile(case.profile), case.kvc_shape())
    Qg = codec.quantize(case.k, case.v, case.block_table)
    st, _, flags_g = codec.query()
    Qo, flags_o = O.quantize(oracle_profile(case.profile), case.oracle_shape(), case.host_bits(case.k),
                             case.host_bits(case.v), case.bt_host())
    return codec, to_np(Qg, codec.plan.payload_bytes), Qo, flags_g, flags_o


def encode_both(case: Case):
    codec = Codec(kvc_profile(case.profile), case.kvc_shape())
    sg = codec.encode(case.k, case.v, case.block_table)
    st, nbytes, flags_g = codec.query()
    so, flags_o = O.encode(oracle_profile(case.profile), case.oracle_shape(), case.host_bits(case.k),
                           case.host_bits(case.v), case.bt_host())
    return codec, sg, nbytes, to_np(sg, nbytes), so, flags_g, flags_o


def bits_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    a = np.asarray(a, np.uint16)
    if dtype == "f16":
        return a.view(np.float16).astype(np.float64)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_recon_close(gpu_bits, ora_bits, dtype, step_bound):
    """|gpu - oracle| <= max(1e-3 |oracle|, step) elementwise (step = the case's
    largest quantization step in the original domain)."""
    g, o = bits_to_f64(gpu_bits, dtype), bits_to_f64(ora_bits, dtype)
    tol = np.maximum(1e-3 * np.abs(o), step_bound)
    bad = ~(np.abs(g - o) <= tol)
    assert not bad.any(), f"{int(bad.sum())} elements outside tolerance; max diff {np.nanmax(np.abs(g - o))}"

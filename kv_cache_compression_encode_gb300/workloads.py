"""The benchmark workloads: KV shapes, input distributions and compression profiles.

Plain data, no arithmetic.  Profiles are given as keyword dictionaries that both
the library binding (``kvc.Profile``) and the oracle (``oracle.make_profile``)
accept.  Stage lists are (kind, parameter) pairs with kinds TUPL = 1, BIT = 2,
DELTA = 3, RZE = 4; the page's searched pipeline TUPL8_1 -> BIT_8 -> RZE_2
("Beyond Compression Ratio: High-Throughput KV Compression for Disaggregated LLM
Serving", §4.2) is ``LC_PIPELINE``.
"""
from __future__ import annotations

from dataclasses import dataclass

TUPL, BIT, DELTA, RZE = 1, 2, 3, 4
LC_PIPELINE = ((TUPL, 8), (BIT, 8), (RZE, 2))
SHUFFLE_ZERO = ((TUPL, 8), (RZE, 1))
FULL_PIPELINE = ((TUPL, 8), (BIT, 8), (DELTA, 1), (RZE, 2))
HADAMARD_SEED = 0x4B5643_5EED


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    tokens: int
    kv_heads: int
    head_dim: int
    dtype: str          # "f16" or "bf16"
    dist: str           # distribution name in synth.py
    seed: int
    page_size: int = 0  # 0 = contiguous [tokens][heads][head_dim] per layer

    @property
    def raw_bytes(self) -> int:
        """Uncompressed K+V bytes of all layers."""
        return 2 * self.layers * self.tokens * self.kv_heads * self.head_dim * 2


WORKLOADS = {
    "tiny": Workload("tiny", 1, 256, 8, 128, "f16", "gauss_outlier", 1234),
    "llama8b": Workload("llama8b", 32, 4096, 8, 128, "bf16", "llama", 1235),
    "llama8b_32k": Workload("llama8b_32k", 32, 32768, 8, 128, "bf16", "llama_sink", 1236),
    "llama70b": Workload("llama70b", 80, 16384, 8, 128, "bf16", "llama", 1237),
    "paged8b_128k": Workload("paged8b_128k", 32, 131072, 8, 128, "bf16", "llama", 1238, page_size=16),
}


def profile_kwargs(smooth_keys=True, hadamard=False, bits_k=4, bits_v=4, group_k=64, group_v=64,
                   stages=(), chunk_bytes=16384, axis_k=0, axis_v=1, seed=HADAMARD_SEED, **v2):
    """v2: optional token_delta, bits_map_k, bits_map_v (format-v2 profile fields)."""
    return dict(smooth_keys=smooth_keys, hadamard=hadamard, bits_k=bits_k, bits_v=bits_v, group_k=group_k,
                group_v=group_v, axis_k=axis_k, axis_v=axis_v, stages=tuple(stages), chunk_bytes=chunk_bytes,
                seed=seed, **v2)


def mixhq_map(layers, kv_heads, retrieval=(0, 5), hi=8, lo=2):
    """A head-wise width map in the manner of MixHQ ("KVServe" §5.1): the heads listed
    as retrieval heads keep `hi` bits in every layer, the streaming heads get `lo`.
    Which heads are retrieval heads is the caller's labelling (a fixed synthetic
    choice here; scoring heads needs a model)."""
    return [[hi if h in retrieval else lo for h in range(kv_heads)] for _ in range(layers)]


PROFILES = {
    # one layer, 4-bit, group 64, byte shuffle + zero elimination
    "tiny": profile_kwargs(True, False, 4, 4, 64, 64, SHUFFLE_ZERO),
    # Hadamard on head_dim, 4-bit group 128, full lossless pipeline (shuffle, bit shuffle, delta, zero elim.)
    "llama8b": profile_kwargs(True, True, 4, 4, 128, 128, FULL_PIPELINE),
    # aggressive: 2-bit group 32 keys per-channel and values per-token, no Hadamard
    "llama8b_32k": profile_kwargs(True, False, 2, 2, 32, 32, LC_PIPELINE),
    # Hadamard + 8-bit group 128; the decode side is the headline
    "llama70b": profile_kwargs(True, True, 8, 8, 128, 128, LC_PIPELINE),
}

# Format-v2 variants of the Llama-8B workload: head-wise mixed precision (two
# retrieval heads of eight at 8 bits, the rest at 2, for K and V) and the token
# delta on top of the llama8b profile.
V2_PROFILES = {
    "llama8b_mixhq": profile_kwargs(True, True, 4, 4, 128, 128, LC_PIPELINE, bits_map_k=mixhq_map(32, 8),
                                    bits_map_v=mixhq_map(32, 8)),
    "llama8b_delta": profile_kwargs(True, True, 4, 4, 128, 128, FULL_PIPELINE, token_delta=True),
}


def paged_sweep():
    """The 48 profiles of the paged sweep: bits x group x Hadamard x lossless on/off."""
    out = []
    for bits in (2, 3, 4, 8):
        for g in (32, 64, 128):
            for had in (False, True):
                for lossless in (False, True):
                    name = f"b{bits}g{g}{'h' if had else ''}{'_lc' if lossless else ''}"
                    out.append((name, profile_kwargs(True, had, bits, bits, g, g,
                                                     LC_PIPELINE if lossless else ())))
    return out

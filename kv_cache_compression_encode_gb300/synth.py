"""Seeded synthetic KV tensors for the benchmark workloads.

This module only draws random numbers with the shapes and distributions of the
workloads; it holds none of the compression arithmetic.  Both the CUDA path and
the CPU oracle consume the exact bytes it produces (tensors drawn on the GPU are
copied to the host for the oracle).

Stand-in data: the pages measure on Llama-3.1-8B / Qwen2.5-7B KV caches of
LongBench requests ("Beyond Compression Ratio: High-Throughput KV Compression for
Disaggregated LLM Serving", §5 Experimental setup).  Those models and datasets are
not used; tensors with the same shapes and a comparable per-channel structure
stand in for them.

Distributions (per workload):
  * "gauss_outlier" -- V ~ N(0,1); K ~ N(0,1) with 4 channels per head (seeded
    choice) scaled x20.
  * "llama"  -- K[l,t,h,c] = mu[l,h,c] + sd[l,h,c] * N(0,1) with
    sd ~ LogNormal(0, 1) and mu ~ N(0, 2^2); V ~ N(0,1).
  * "llama_sink" -- "llama" plus a seeded 5% of token indices (shared by all
    layers and heads) whose K and V rows are scaled x50.
"""
from __future__ import annotations

import torch

_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def _gen(device, seed: int, layer: int, salt: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + layer * 7919 + salt) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def sink_tokens(tokens: int, seed: int, frac: float = 0.05) -> torch.Tensor:
    """Sorted indices of the attention-sink tokens (CPU, int64)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 31 + 17)
    n = max(1, int(round(frac * tokens)))
    return torch.sort(torch.randperm(tokens, generator=g)[:n]).values


def block_table(tokens: int, page_size: int, seed: int) -> torch.Tensor:
    """A seeded random permutation of the physical pages (int32, CPU)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 131 + 7)
    n_pages = (tokens + page_size - 1) // page_size
    return torch.randperm(n_pages, generator=g).to(torch.int32)


def layer_kv(dist: str, layer: int, tokens: int, kv_heads: int, head_dim: int, dtype: str,
             seed: int, device="cpu"):
    """K and V of one layer as [tokens, kv_heads, head_dim] tensors of `dtype`."""
    T, H, D = tokens, kv_heads, head_dim
    dt = _DTYPES[dtype]
    g = _gen(device, seed, layer, 1)
    if dist == "gauss_outlier":
        k = torch.randn(T, H, D, generator=g, device=device, dtype=torch.float32)
        v = torch.randn(T, H, D, generator=g, device=device, dtype=torch.float32)
        gc = torch.Generator(device="cpu")
        gc.manual_seed(seed * 977 + layer)
        for h in range(H):
            ch = torch.randperm(D, generator=gc)[:4].to(device)
            k[:, h, ch] *= 20.0
        return k.to(dt), v.to(dt)
    if dist in ("llama", "llama_sink"):
        mu = torch.randn(H, D, generator=g, device=device, dtype=torch.float32) * 2.0
        sd = torch.exp(torch.randn(H, D, generator=g, device=device, dtype=torch.float32))
        k = torch.randn(T, H, D, generator=g, device=device, dtype=torch.float32)
        k.mul_(sd).add_(mu)
        v = torch.randn(T, H, D, generator=g, device=device, dtype=torch.float32)
        if dist == "llama_sink":
            idx = sink_tokens(T, seed).to(device)
            k[idx] *= 50.0
            v[idx] *= 50.0
        return k.to(dt), v.to(dt)
    raise ValueError(f"unknown distribution {dist!r}")


def paged_layer_kv(dist: str, layer: int, tokens: int, page_size: int, kv_heads: int, head_dim: int,
                   dtype: str, seed: int, device="cpu"):
    """K and V of one layer as physical pages [n_pages, page_size, kv_heads, head_dim].

    Tokens are i.i.d. given the per-channel parameters, so drawing the physical
    pages directly has the same distribution as scattering logical pages."""
    n_pages = (tokens + page_size - 1) // page_size
    k, v = layer_kv(dist, layer, n_pages * page_size, kv_heads, head_dim, dtype, seed, device)
    return (k.view(n_pages, page_size, kv_heads, head_dim), v.view(n_pages, page_size, kv_heads, head_dim))


def to_bits_numpy(t: torch.Tensor):
    """Element bits of a half-precision tensor as a host numpy uint16 array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")

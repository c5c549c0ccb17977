"""Benefit condition of a compression profile from measured numbers.

"KVServe: Service-Aware KV Cache Compression for Communication-Efficient
Disaggregated LLM Serving", §3.1: a profile p is characterised by its compression
ratio cr_p = V / V_p and its effective (de)compression throughput s_p, the
harmonic mean of the encode and decode throughputs, so that encoding plus
decoding V bytes takes V / s_p.  §6.1, Eq. (5): moving the compressed KV instead
of the raw KV shortens the segment exactly when the link bandwidth B is below
B*_p = (1 - 1 / cr_p) s_p.

Host arithmetic only (no device work); throughputs in any one unit (bytes/s or
GB/s), the results in the same unit.
"""
from __future__ import annotations


def effective_throughput(enc: float, dec: float) -> float:
    """s_p: encode and decode of V bytes take V / enc + V / dec = V / s_p."""
    if enc <= 0 or dec <= 0:
        raise ValueError("throughputs must be positive")
    return enc * dec / (enc + dec)


def break_even_bandwidth(cr: float, s_p: float) -> float:
    """B*_p = (1 - 1 / cr_p) s_p: compression pays off on links slower than this."""
    if cr <= 0 or s_p <= 0:
        raise ValueError("compression ratio and throughput must be positive")
    return (1.0 - 1.0 / cr) * s_p


def segment_time(v_bytes: float, bandwidth: float, cr: float | None = None, s_p: float | None = None) -> float:
    """Transfer part of the segment time (Eq. (1) without T_model): V / B raw, or
    V / s_p + V / (B cr_p) with profile p."""
    if cr is None:
        return v_bytes / bandwidth
    return v_bytes / s_p + v_bytes / (bandwidth * cr)

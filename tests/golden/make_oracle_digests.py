"""Writes tests/golden/oracle_digests.json: SHA-256 digests of the oracle's stream
and reconstruction for small seeded cases of each workload profile.

Calls only the oracle.  Inputs are drawn with numpy's PCG64 as integers and turned
into element bits without floating-point library code, so every machine draws the
same bytes; a digest mismatch on another machine means the oracle's arithmetic
differs there.  Run:  python -m tests.golden.make_oracle_digests
"""
import hashlib
import json
import os

import numpy as np

from oracle import oracle as O

CASES = [
    # name, (L, T, H, D, dtype), profile kwargs
    ("tiny", (1, 256, 8, 128, 1), dict(smooth_keys=True, hadamard=False, bits_k=4, bits_v=4, group_k=64, group_v=64,
                                       stages=((1, 8), (4, 1)))),
    ("llama8b_small", (2, 300, 2, 128, 2), dict(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=128,
                                                group_v=128, stages=((1, 8), (2, 8), (3, 1), (4, 2)), chunk_bytes=4096)),
    ("aggressive_small", (2, 200, 2, 128, 2), dict(smooth_keys=True, hadamard=False, bits_k=2, bits_v=2, group_k=32,
                                                   group_v=32, stages=((1, 8), (2, 8), (4, 2)), chunk_bytes=2048)),
    ("b8_hadamard_small", (1, 160, 2, 128, 2), dict(smooth_keys=True, hadamard=True, bits_k=8, bits_v=8, group_k=128,
                                                    group_v=128, stages=((1, 8), (2, 8), (4, 2)))),
    ("b3_axes_swapped", (1, 97, 2, 128, 1), dict(smooth_keys=True, hadamard=True, bits_k=3, bits_v=3, group_k=32,
                                                 group_v=64, axis_k=1, axis_v=0, stages=((3, 2), (4, 2)))),
]


def _elements(n, dtype, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    sign = rng.integers(0, 2, n, dtype=np.uint16)
    if dtype == 1:   # binary16: exponents 9..19 (about 2^-6 .. 2^4)
        ex = rng.integers(9, 20, n, dtype=np.uint16)
        man = rng.integers(0, 1024, n, dtype=np.uint16)
        return (sign << 15) | (ex << 10) | man
    ex = rng.integers(120, 132, n, dtype=np.uint16)  # bfloat16: about 2^-7 .. 2^4
    man = rng.integers(0, 128, n, dtype=np.uint16)
    return (sign << 15) | (ex << 7) | man


def digest_cases():
    out = {}
    for i, (name, (L, T, H, D, dt), kw) in enumerate(CASES):
        shape = O.make_shape(L, T, H, D, dt)
        prof = O.make_profile(seed=0x5EED + i, **kw)
        n = L * T * H * D
        k = _elements(n, dt, 100 + i).reshape(L, T, H, D)
        v = _elements(n, dt, 200 + i).reshape(L, T, H, D)
        stream, flags = O.encode(prof, shape, k, v)
        ok, ov = np.zeros_like(k), np.zeros_like(v)
        dflags = O.decode(prof, shape, stream, ok, ov)
        h = hashlib.sha256()
        h.update(ok.tobytes())
        h.update(ov.tobytes())
        out[name] = {"flags": flags | dflags, "stream_bytes": int(stream.size),
                     "stream_sha256": hashlib.sha256(stream.tobytes()).hexdigest(), "kv_sha256": h.hexdigest()}
    return out


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_digests.json")
    with open(path, "w") as f:
        json.dump({"source": "written by tests/golden/make_oracle_digests.py from the oracle only",
                   "digests": digest_cases()}, f, indent=1)
    print("wrote", path)

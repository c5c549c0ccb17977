"""Python access to the plain C oracle of the KV-cache compression path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package smoke check
and by the CPU-baseline leg of ``bench.py``; never by the product library.

The oracle (``kvc_oracle.c``) restates, step by step, what the pages define:
  * "KVServe: Service-Aware KV Cache Compression for Communication-Efficient
    Disaggregated LLM Serving", §5.1 (pipeline BS = C(Q(T(X))), Hadamard
    transformer, KIVI quantizer) and §7.3 (2-bit KIVI metadata ceiling);
  * "Beyond Compression Ratio: High-Throughput KV Compression for Disaggregated
    LLM Serving" (FastKVComp), §4.1 (fused transform + quantization and the
    reconstruction path) and §4.2 (TUPL / BIT / RZE lossless pipeline).
Format-v1 readings (where the pages are silent) are marked READING in the C file.

Parity status: every function exported here is pinned by ``tests/test_oracle_*``
against closed forms, brute force, library routines or hand-worked examples.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvc_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkvc_oracle.so")
_lock = threading.Lock()
_lib = None

FLAG_RANGE = 1
FLAG_NONFINITE = 2
FLAG_CORRUPT = 4
FLAG_CAPACITY = 8

ST_TUPL, ST_BIT, ST_DELTA, ST_RZE = 1, 2, 3, 4
AXIS_OVER_TOKENS, AXIS_OVER_CHANNELS = 0, 1
F16, BF16 = 1, 2
HEADER_BYTES = 64
SMOOTH_BLOCK = 128


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (scalar C11, no contraction, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fexcess-precision=standard",
               "-fno-strict-aliasing", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Shape(C.Structure):
    _fields_ = [("layers", C.c_uint32), ("tokens", C.c_uint32), ("kv_heads", C.c_uint32),
                ("head_dim", C.c_uint32), ("dtype", C.c_uint32), ("page_size", C.c_uint32),
                ("token_stride", C.c_uint64), ("page_stride", C.c_uint64)]


class Profile(C.Structure):
    _fields_ = [("smooth_keys", C.c_uint32), ("hadamard", C.c_uint32),
                ("bits_k", C.c_uint32), ("bits_v", C.c_uint32), ("group_k", C.c_uint32),
                ("group_v", C.c_uint32), ("axis_k", C.c_uint32), ("axis_v", C.c_uint32),
                ("n_stages", C.c_uint32), ("stage_kind", C.c_uint32 * 4), ("stage_param", C.c_uint32 * 4),
                ("chunk_bytes", C.c_uint32), ("seed", C.c_uint64), ("token_delta", C.c_uint32),
                ("pad_", C.c_uint32), ("bits_map_k", C.c_void_p), ("bits_map_v", C.c_void_p)]


class Layout(C.Structure):
    _fields_ = [("off", C.c_uint64 * 8), ("size", C.c_uint64 * 8), ("payload_bytes", C.c_uint64),
                ("n_chunks", C.c_uint64), ("data_start", C.c_uint64), ("max_stream_bytes", C.c_uint64),
                ("header_bytes", C.c_uint64)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = C.CDLL(path)
            u8p, u16p, f32p = C.POINTER(C.c_uint8), C.POINTER(C.c_uint16), C.POINTER(C.c_float)
            vpp = C.POINTER(C.c_void_p)
            sig = {
                "kvo_f16_to_f32": (C.c_float, [C.c_uint16]),
                "kvo_f32_to_f16": (C.c_uint16, [C.c_float, C.c_int]),
                "kvo_bf16_to_f32": (C.c_float, [C.c_uint16]),
                "kvo_f32_to_bf16": (C.c_uint16, [C.c_float]),
                "kvo_splitmix64_output": (C.c_uint64, [C.c_uint64, C.c_uint32]),
                "kvo_signs": (None, [C.c_uint64, C.c_uint32, f32p]),
                "kvo_fwht": (None, [f32p, C.c_uint32]),
                "kvo_hadamard_scale": (C.c_float, [C.c_uint32]),
                "kvo_hadamard_forward": (None, [f32p, f32p, C.c_uint32]),
                "kvo_hadamard_inverse": (None, [f32p, f32p, C.c_uint32]),
                "kvo_ceil_log2": (C.c_int, [C.c_float]),
                "kvo_quantize_group": (None, [f32p, C.c_uint32, C.c_uint32, u16p, u16p, u8p,
                                              C.POINTER(C.c_uint32)]),
                "kvo_pack": (None, [u8p, C.c_uint32, C.c_uint32, u8p]),
                "kvo_unpack": (None, [u8p, C.c_uint32, C.c_uint32, u8p]),
                "kvo_layout_of": (C.c_int, [C.POINTER(Profile), C.POINTER(Shape), C.POINTER(Layout)]),
                "kvo_quantize": (C.c_uint32, [C.POINTER(Profile), C.POINTER(Shape), vpp, vpp, C.c_void_p, u8p]),
                "kvo_dequantize": (None, [C.POINTER(Profile), C.POINTER(Shape), u8p, vpp, vpp, C.c_void_p]),
                "kvo_stage_encode": (C.c_size_t, [C.c_uint32, C.c_uint32, u8p, C.c_size_t, u8p]),
                "kvo_tupl_decode": (C.c_size_t, [u8p, C.c_size_t, C.c_uint32, u8p]),
                "kvo_bit_decode": (C.c_size_t, [u8p, C.c_size_t, u8p]),
                "kvo_delta_decode": (C.c_size_t, [u8p, C.c_size_t, C.c_uint32, u8p]),
                "kvo_rze_decode": (C.c_int, [u8p, C.c_size_t, C.c_size_t, C.c_uint32, u8p]),
                "kvo_chunk_encode": (C.c_size_t, [C.POINTER(Profile), u8p, C.c_size_t, u8p, C.POINTER(C.c_int)]),
                "kvo_chunk_decode": (C.c_int, [C.POINTER(Profile), u8p, C.c_size_t, C.c_int, C.c_size_t, u8p]),
                "kvo_write_header": (None, [C.POINTER(Profile), C.POINTER(Shape), C.POINTER(Layout), u8p]),
                "kvo_lossless_encode": (C.c_uint64, [C.POINTER(Profile), C.POINTER(Layout), u8p, u8p]),
                "kvo_lossless_decode": (C.c_uint32, [C.POINTER(Profile), C.POINTER(Shape), u8p, C.c_uint64, u8p]),
                "kvo_encode": (C.c_uint32, [C.POINTER(Profile), C.POINTER(Shape), vpp, vpp, C.c_void_p, u8p,
                                            C.c_uint64, C.POINTER(C.c_uint64)]),
                "kvo_decode": (C.c_uint32, [C.POINTER(Profile), C.POINTER(Shape), u8p, C.c_uint64, vpp, vpp,
                                            C.c_void_p]),
                "kvo_set_threads": (C.c_int, [C.c_int]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.POINTER(ctype))


def set_threads(n: int) -> int:
    """Number of OpenMP threads the oracle uses (n <= 0 keeps the current value)."""
    return lib().kvo_set_threads(int(n))


# ----------------------------------------------------------------------------
# Profiles and shapes
# ----------------------------------------------------------------------------
def make_profile(*, smooth_keys=True, hadamard=False, bits_k=4, bits_v=4, group_k=64, group_v=64,
                 axis_k=AXIS_OVER_TOKENS, axis_v=AXIS_OVER_CHANNELS, stages=(), chunk_bytes=16384,
                 seed=0x5EED, token_delta=False, bits_map_k=None, bits_map_v=None) -> Profile:
    """bits_map_k / bits_map_v: optional [layers][kv_heads] code widths (format v2);
    token_delta: the anchor-token delta transformer (format v2)."""
    p = Profile()
    p.token_delta = int(bool(token_delta))
    p._maps = []  # keeps the width maps alive as long as the profile
    for name, m in (("bits_map_k", bits_map_k), ("bits_map_v", bits_map_v)):
        if m is not None:
            arr = np.ascontiguousarray(np.asarray(m, dtype=np.uint8).reshape(-1))
            p._maps.append(arr)
            setattr(p, name, arr.ctypes.data)
    p.smooth_keys, p.hadamard = int(bool(smooth_keys)), int(bool(hadamard))
    p.bits_k, p.bits_v, p.group_k, p.group_v = bits_k, bits_v, group_k, group_v
    p.axis_k, p.axis_v = axis_k, axis_v
    p.n_stages = len(stages)
    for i, (k, prm) in enumerate(stages):
        p.stage_kind[i], p.stage_param[i] = k, prm
    p.chunk_bytes = chunk_bytes
    p.seed = seed
    return p


def make_shape(layers, tokens, kv_heads, head_dim, dtype, page_size=0, token_stride=None, page_stride=0) -> Shape:
    s = Shape()
    s.layers, s.tokens, s.kv_heads, s.head_dim, s.dtype = layers, tokens, kv_heads, head_dim, dtype
    s.page_size = page_size
    s.token_stride = token_stride if token_stride is not None else kv_heads * head_dim * 2
    s.page_stride = page_stride
    return s


def layout(profile: Profile, shape: Shape) -> Layout:
    lay = Layout()
    lib().kvo_layout_of(C.byref(profile), C.byref(shape), C.byref(lay))
    return lay


def _bases(arrs):
    """Array of host base pointers, one per layer (keeps the arrays alive via the caller)."""
    return (C.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _layers(x):
    """Accept a [L][...] array or a list of per-layer arrays of uint16 element bits."""
    if isinstance(x, np.ndarray):
        x = [np.ascontiguousarray(x[i]) for i in range(x.shape[0])]
    out = []
    for a in x:
        assert a.dtype == np.uint16 and a.flags["C_CONTIGUOUS"]
        out.append(a)
    return out


# ----------------------------------------------------------------------------
# Whole-path entry points
# ----------------------------------------------------------------------------
def quantize(profile, shape, k, v, block_table=None):
    """Payload Q (uint8) and status flags."""
    kl, vl = _layers(k), _layers(v)
    lay = layout(profile, shape)
    Q = np.zeros(max(lay.payload_bytes, 1), np.uint8)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    kb, vb = _bases(kl), _bases(vl)
    flags = lib().kvo_quantize(C.byref(profile), C.byref(shape), kb, vb,
                               None if bt is None else bt.ctypes.data, _ptr(Q, C.c_uint8))
    return Q[:lay.payload_bytes], int(flags)


def dequantize(profile, shape, Q, out_k, out_v, block_table=None):
    """Write reconstructed element bits into out_k / out_v (per-layer uint16 arrays)."""
    kl, vl = _layers(out_k), _layers(out_v)
    Qc = np.ascontiguousarray(Q, dtype=np.uint8)
    if Qc.size == 0:
        Qc = np.zeros(1, np.uint8)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    lib().kvo_dequantize(C.byref(profile), C.byref(shape), _ptr(Qc, C.c_uint8), _bases(kl), _bases(vl),
                         None if bt is None else bt.ctypes.data)
    return kl, vl


def encode(profile, shape, k, v, block_table=None):
    """Full encode; returns (stream bytes as uint8 array, flags)."""
    kl, vl = _layers(k), _layers(v)
    lay = layout(profile, shape)
    cap = lay.max_stream_bytes
    out = np.zeros(cap, np.uint8)
    nbytes = C.c_uint64(0)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    flags = lib().kvo_encode(C.byref(profile), C.byref(shape), _bases(kl), _bases(vl),
                             None if bt is None else bt.ctypes.data, _ptr(out, C.c_uint8), C.c_uint64(cap),
                             C.byref(nbytes))
    return out[:nbytes.value], int(flags)


def decode(profile, shape, stream, out_k, out_v, block_table=None):
    """Full decode into out_k / out_v; returns flags (FLAG_CORRUPT leaves them untouched)."""
    kl, vl = _layers(out_k), _layers(out_v)
    s = np.ascontiguousarray(stream, dtype=np.uint8)
    n = s.size
    if n == 0:
        s = np.zeros(1, np.uint8)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    return int(lib().kvo_decode(C.byref(profile), C.byref(shape), _ptr(s, C.c_uint8), C.c_uint64(n),
                                _bases(kl), _bases(vl), None if bt is None else bt.ctypes.data))


def lossless_encode(profile, shape, Q):
    """Header + lossless stream of a given payload Q (uint8 array)."""
    lay = layout(profile, shape)
    assert Q.size == lay.payload_bytes
    out = np.zeros(max(lay.max_stream_bytes, HEADER_BYTES), np.uint8)
    Qc = np.ascontiguousarray(Q, dtype=np.uint8) if Q.size else np.zeros(1, np.uint8)
    lib().kvo_write_header(C.byref(profile), C.byref(shape), C.byref(lay), _ptr(out, C.c_uint8))
    n = lib().kvo_lossless_encode(C.byref(profile), C.byref(lay), _ptr(Qc, C.c_uint8), _ptr(out, C.c_uint8))
    return out[:n]


def lossless_decode(profile, shape, stream):
    lay = layout(profile, shape)
    Q = np.zeros(max(lay.payload_bytes, 1), np.uint8)
    s = np.ascontiguousarray(stream, dtype=np.uint8)
    n = s.size
    if n == 0:
        s = np.zeros(1, np.uint8)
    flags = lib().kvo_lossless_decode(C.byref(profile), C.byref(shape), _ptr(s, C.c_uint8), C.c_uint64(n),
                                      _ptr(Q, C.c_uint8))
    return Q[:lay.payload_bytes], int(flags)


# ----------------------------------------------------------------------------
# Single-step entry points (for pins)
# ----------------------------------------------------------------------------
def f16_to_f32(h: int) -> float:
    return lib().kvo_f16_to_f32(h)


def f32_to_f16(x: float, mode: int = 0) -> int:
    """mode 0 nearest-even, 1 toward -inf, 2 toward +inf."""
    return lib().kvo_f32_to_f16(C.c_float(x), mode)


def bf16_to_f32(b: int) -> float:
    return lib().kvo_bf16_to_f32(b)


def f32_to_bf16(x: float) -> int:
    return lib().kvo_f32_to_bf16(C.c_float(x))


def splitmix64_output(seed: int, j: int) -> int:
    return lib().kvo_splitmix64_output(C.c_uint64(seed), j)


def signs(seed: int, D: int) -> np.ndarray:
    out = np.zeros(D, np.float32)
    lib().kvo_signs(C.c_uint64(seed), D, _ptr(out, C.c_float))
    return out


def fwht(v: np.ndarray) -> np.ndarray:
    x = np.array(v, dtype=np.float32, copy=True)
    lib().kvo_fwht(_ptr(x, C.c_float), x.size)
    return x


def hadamard_scale(D: int) -> float:
    return lib().kvo_hadamard_scale(D)


def hadamard_forward(v: np.ndarray, sigma: np.ndarray) -> np.ndarray:
    x = np.array(v, dtype=np.float32, copy=True)
    s = np.ascontiguousarray(sigma, dtype=np.float32)
    lib().kvo_hadamard_forward(_ptr(x, C.c_float), _ptr(s, C.c_float), x.size)
    return x


def hadamard_inverse(v: np.ndarray, sigma: np.ndarray) -> np.ndarray:
    x = np.array(v, dtype=np.float32, copy=True)
    s = np.ascontiguousarray(sigma, dtype=np.float32)
    lib().kvo_hadamard_inverse(_ptr(x, C.c_float), _ptr(s, C.c_float), x.size)
    return x


def ceil_log2(r: float) -> int:
    return lib().kvo_ceil_log2(C.c_float(r))


def quantize_group(y: np.ndarray, bits: int):
    """Returns (scale_bits, zero_bits, codes uint8[n], flags)."""
    y32 = np.ascontiguousarray(y, dtype=np.float32)
    s, z, f = C.c_uint16(), C.c_uint16(), C.c_uint32(0)
    codes = np.zeros(y32.size, np.uint8)
    lib().kvo_quantize_group(_ptr(y32, C.c_float), y32.size, bits, C.byref(s), C.byref(z),
                             _ptr(codes, C.c_uint8), C.byref(f))
    return s.value, z.value, codes, f.value


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros((c.size * bits + 7) // 8, np.uint8)
    lib().kvo_pack(_ptr(c, C.c_uint8), c.size, bits, _ptr(out, C.c_uint8))
    return out


def unpack(data: np.ndarray, n: int, bits: int) -> np.ndarray:
    d = np.ascontiguousarray(data, dtype=np.uint8)
    out = np.zeros(n, np.uint8)
    lib().kvo_unpack(_ptr(d, C.c_uint8), n, bits, _ptr(out, C.c_uint8))
    return out


def stage_encode(kind: int, param: int, data: np.ndarray) -> np.ndarray:
    d = np.ascontiguousarray(data, dtype=np.uint8)
    n = d.size
    src = d if n else np.zeros(1, np.uint8)
    out = np.zeros(2 * n + 64, np.uint8)
    m = lib().kvo_stage_encode(kind, param, _ptr(src, C.c_uint8), n, _ptr(out, C.c_uint8))
    return out[:m]


def stage_decode(kind: int, param: int, data: np.ndarray, n: int):
    """Inverse of one stage; returns the n raw bytes, or None when inconsistent (RZE)."""
    d = np.ascontiguousarray(data, dtype=np.uint8)
    src = d if d.size else np.zeros(1, np.uint8)
    out = np.zeros(max(n, 1), np.uint8)
    if kind == ST_TUPL:
        lib().kvo_tupl_decode(_ptr(src, C.c_uint8), n, param, _ptr(out, C.c_uint8))
    elif kind == ST_BIT:
        lib().kvo_bit_decode(_ptr(src, C.c_uint8), n, _ptr(out, C.c_uint8))
    elif kind == ST_DELTA:
        lib().kvo_delta_decode(_ptr(src, C.c_uint8), n, param, _ptr(out, C.c_uint8))
    elif kind == ST_RZE:
        if lib().kvo_rze_decode(_ptr(src, C.c_uint8), d.size, n, param, _ptr(out, C.c_uint8)) != 0:
            return None
    return out[:n]


def chunk_encode(profile, data: np.ndarray):
    """(stored bytes, raw flag) of one chunk."""
    d = np.ascontiguousarray(data, dtype=np.uint8)
    n = d.size
    src = d if n else np.zeros(1, np.uint8)
    out = np.zeros(max(2 * n + 64, 1), np.uint8)
    raw = C.c_int(0)
    m = lib().kvo_chunk_encode(C.byref(profile), _ptr(src, C.c_uint8), n, _ptr(out, C.c_uint8), C.byref(raw))
    return out[:m], bool(raw.value)


def chunk_decode(profile, stored: np.ndarray, raw: bool, n: int):
    d = np.ascontiguousarray(stored, dtype=np.uint8)
    src = d if d.size else np.zeros(1, np.uint8)
    out = np.zeros(max(n, 1), np.uint8)
    rc = lib().kvo_chunk_decode(C.byref(profile), _ptr(src, C.c_uint8), d.size, int(raw), n, _ptr(out, C.c_uint8))
    return None if rc != 0 else out[:n]

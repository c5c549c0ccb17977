"""Thin Python binding of the C ABI in include/kvc.h (argument marshalling only).

Every step of the compression path runs in the CUDA library libkvc.so; this
module mirrors its structs with ctypes, exposes its entry points under the same
names, and turns torch tensors into the device pointers the ABI takes.  There is
no fallback: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

from . import build as _build

KVC_OK, KVC_ERR_INVALID_ARG, KVC_ERR_UNSUPPORTED, KVC_ERR_CAPACITY = 0, 1, 2, 3
KVC_ERR_CORRUPT, KVC_ERR_RANGE, KVC_ERR_NONFINITE, KVC_ERR_TIMEOUT, KVC_ERR_CUDA = 4, 5, 6, 7, 8
FLAG_RANGE, FLAG_NONFINITE, FLAG_CORRUPT, FLAG_CAPACITY, FLAG_TIMEOUT, FLAG_BAD_PAGE = 1, 2, 4, 8, 16, 32
F16, BF16 = 1, 2
AXIS_OVER_TOKENS, AXIS_OVER_CHANNELS = 0, 1
ST_TUPL, ST_BIT, ST_DELTA, ST_RZE = 1, 2, 3, 4
MAX_STAGES, MAX_LAYERS, HEADER_BYTES = 4, 256, 64
PROFILE_V1_SIZE, MAX_MAP_ENTRIES = 40, 2048

EXPORTS = ["kvc_plan", "kvc_plan_destroy", "kvc_workspace_bytes", "kvc_max_stream_bytes", "kvc_payload_bytes",
           "kvc_section", "kvc_num_chunks", "kvc_encode", "kvc_decode", "kvc_quantize", "kvc_lossless_encode",
           "kvc_lossless_decode", "kvc_dequantize", "kvc_query", "kvc_status_str", "kvc_launch_count",
           "kvc_timing_enable", "kvc_timing_read", "kvc_debug_lookback", "kvc_lossless_encode_noalloc",
           "kvc_header_bytes", "kvc_debug_generic_stages", "kvc_debug_quotient_check", "kvc_fuse_value_chunks",
           "kvc_decode_codes_in_place"]


class KvcError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} ({status})" if what else status_str(status))


class Stage(C.Structure):
    _fields_ = [("kind", C.c_uint8), ("param", C.c_uint8)]


class Profile(C.Structure):
    _fields_ = [("struct_size", C.c_uint32), ("smooth_keys", C.c_uint8), ("hadamard", C.c_uint8),
                ("bits_k", C.c_uint8), ("bits_v", C.c_uint8), ("group_k", C.c_uint16), ("group_v", C.c_uint16),
                ("axis_k", C.c_uint8), ("axis_v", C.c_uint8), ("n_stages", C.c_uint8), ("reserved0", C.c_uint8),
                ("stages", Stage * MAX_STAGES), ("chunk_bytes", C.c_uint32), ("reserved1", C.c_uint32),
                ("hadamard_seed", C.c_uint64), ("token_delta", C.c_uint8), ("reserved2", C.c_uint8 * 7),
                ("bits_map_k", C.c_void_p), ("bits_map_v", C.c_void_p)]


class Shape(C.Structure):
    _fields_ = [("struct_size", C.c_uint32), ("layers", C.c_uint32), ("tokens", C.c_uint32),
                ("kv_heads", C.c_uint32), ("head_dim", C.c_uint32), ("dtype", C.c_uint32),
                ("page_size", C.c_uint32), ("num_pages", C.c_uint32), ("token_stride", C.c_uint64),
                ("page_stride", C.c_uint64)]


class KV(C.Structure):
    _fields_ = [("k_layers", C.POINTER(C.c_void_p)), ("v_layers", C.POINTER(C.c_void_p)),
                ("block_table", C.c_void_p)]


class Timing(C.Structure):
    _fields_ = [("kernel", C.c_char_p), ("ms", C.c_float)]


assert C.sizeof(Profile) == 64 and C.sizeof(Shape) == 48 and C.sizeof(KV) == 24

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libkvc.so (building it with nvcc if it is missing); raises if impossible."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"libkvc.so not built ({path}); run kv_cache_compression_encode_gb300.build")
            _build.build()
        L = C.CDLL(path)
        P, vp, sz, u64, u32 = C.c_void_p, C.c_void_p, C.c_size_t, C.c_uint64, C.c_uint32
        st = C.c_int
        sigs = {
            "kvc_plan": (st, [C.POINTER(Profile), C.POINTER(Shape), C.POINTER(P)]),
            "kvc_plan_destroy": (None, [P]),
            "kvc_workspace_bytes": (sz, [P]),
            "kvc_max_stream_bytes": (sz, [P]),
            "kvc_payload_bytes": (sz, [P]),
            "kvc_section": (st, [P, C.c_int, C.POINTER(u64), C.POINTER(u64)]),
            "kvc_num_chunks": (u64, [P]),
            "kvc_encode": (st, [P, C.POINTER(KV), vp, sz, vp, sz, vp, vp]),
            "kvc_decode": (st, [P, vp, sz, C.POINTER(KV), vp, sz, vp]),
            "kvc_quantize": (st, [P, C.POINTER(KV), vp, vp, sz, vp]),
            "kvc_lossless_encode": (st, [P, vp, vp, sz, vp, sz, vp, vp]),
            "kvc_lossless_decode": (st, [P, vp, sz, vp, vp, sz, vp]),
            "kvc_dequantize": (st, [P, vp, C.POINTER(KV), vp, sz, vp]),
            "kvc_query": (st, [vp, vp, C.POINTER(u64), C.POINTER(u32)]),
            "kvc_status_str": (C.c_char_p, [C.c_int]),
            "kvc_launch_count": (u64, [P]),
            "kvc_timing_enable": (st, [P, C.c_int, C.c_int]),
            "kvc_timing_read": (C.c_int, [P, C.POINTER(Timing), C.c_int]),
            "kvc_debug_lookback": (st, [P, C.c_int64, C.c_uint32]),
            "kvc_lossless_encode_noalloc": (st, [P, vp, vp, sz, vp, vp, vp]),
            "kvc_header_bytes": (sz, [P]),
            "kvc_debug_generic_stages": (st, [P, C.c_int]),
            "kvc_fuse_value_chunks": (st, [P, C.c_int]),
            "kvc_decode_codes_in_place": (st, [P, C.c_int]),
            "kvc_debug_quotient_check": (st, [C.c_uint32, C.c_uint32, C.POINTER(C.c_ulonglong), vp]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def status_str(status: int) -> str:
    try:
        return load().kvc_status_str(status).decode()
    except Exception:  # noqa: BLE001 - only for error messages
        return f"status {status}"


def _check(status: int, what: str):
    if status != KVC_OK:
        raise KvcError(status, what)


# ----------------------------------------------------------------------------
# structs
# ----------------------------------------------------------------------------
def make_profile(*, smooth_keys=True, hadamard=False, bits_k=4, bits_v=4, group_k=64, group_v=64,
                 axis_k=AXIS_OVER_TOKENS, axis_v=AXIS_OVER_CHANNELS, stages=(), chunk_bytes=16384,
                 seed=0x5EED, token_delta=False, bits_map_k=None, bits_map_v=None) -> Profile:
    """bits_map_k / bits_map_v: optional [layers][kv_heads] code widths (kept alive by
    the returned profile, copied by kvc_plan); token_delta: the anchor-token delta."""
    p = Profile()
    p.struct_size = C.sizeof(Profile)
    p.token_delta = int(bool(token_delta))
    p._maps = []
    for name, m in (("bits_map_k", bits_map_k), ("bits_map_v", bits_map_v)):
        if m is not None:
            arr = (C.c_uint8 * len(_flat(m)))(*_flat(m))
            p._maps.append(arr)
            setattr(p, name, C.cast(arr, C.c_void_p).value)
    p.smooth_keys, p.hadamard = int(bool(smooth_keys)), int(bool(hadamard))
    p.bits_k, p.bits_v, p.group_k, p.group_v = bits_k, bits_v, group_k, group_v
    p.axis_k, p.axis_v = axis_k, axis_v
    p.n_stages = len(stages)
    for i, (k, prm) in enumerate(stages):
        p.stages[i].kind, p.stages[i].param = k, prm
    p.chunk_bytes = chunk_bytes
    p.hadamard_seed = seed
    return p


def _flat(m):
    out = []
    for row in m:
        if hasattr(row, "__iter__"):
            out.extend(int(x) for x in row)
        else:
            out.append(int(row))
    return out


def make_shape(layers, tokens, kv_heads, head_dim, dtype, page_size=0, num_pages=0, token_stride=0,
               page_stride=0) -> Shape:
    s = Shape()
    s.struct_size = C.sizeof(Shape)
    s.layers, s.tokens, s.kv_heads, s.head_dim, s.dtype = layers, tokens, kv_heads, head_dim, dtype
    s.page_size, s.num_pages = page_size, num_pages
    s.token_stride, s.page_stride = token_stride, page_stride
    return s


class KVRef:
    """A kvc_kv struct plus the host pointer arrays it refers to (kept alive here)."""

    def __init__(self, k_ptrs, v_ptrs, block_table_ptr=0, keep=()):
        self._k = (C.c_void_p * max(1, len(k_ptrs)))(*k_ptrs)
        self._v = (C.c_void_p * max(1, len(v_ptrs)))(*v_ptrs)
        self._keep = keep
        self.struct = KV(C.cast(self._k, C.POINTER(C.c_void_p)), C.cast(self._v, C.POINTER(C.c_void_p)),
                         block_table_ptr or None)

    @classmethod
    def from_tensors(cls, k_layers, v_layers, block_table=None):
        """k_layers / v_layers: per-layer CUDA tensors (or one tensor indexed by layer)."""
        ks = [k_layers[i] for i in range(len(k_layers))]
        vs = [v_layers[i] for i in range(len(v_layers))]
        for t in ks + vs:
            if not t.is_cuda:
                raise ValueError("KV tensors must live in CUDA device memory")
        bt = 0
        if block_table is not None:
            if not block_table.is_cuda or block_table.dtype.itemsize != 4:
                raise ValueError("block_table must be an int32 CUDA tensor")
            bt = block_table.data_ptr()
        return cls([t.data_ptr() for t in ks], [t.data_ptr() for t in vs], bt, keep=(ks, vs, block_table))


class Plan:
    """Owns a kvc_plan_t*."""

    def __init__(self, profile: Profile, shape: Shape):
        self.lib = load()
        self.profile, self.shape = profile, shape
        h = C.c_void_p()
        _check(self.lib.kvc_plan(C.byref(profile), C.byref(shape), C.byref(h)), "kvc_plan")
        self.handle = h

    def close(self):
        if self.handle:
            self.lib.kvc_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass

    @property
    def workspace_bytes(self) -> int:
        return self.lib.kvc_workspace_bytes(self.handle)

    @property
    def max_stream_bytes(self) -> int:
        return self.lib.kvc_max_stream_bytes(self.handle)

    @property
    def payload_bytes(self) -> int:
        return self.lib.kvc_payload_bytes(self.handle)

    @property
    def n_chunks(self) -> int:
        return self.lib.kvc_num_chunks(self.handle)

    @property
    def header_bytes(self) -> int:
        return self.lib.kvc_header_bytes(self.handle)

    @property
    def launches(self) -> int:
        return self.lib.kvc_launch_count(self.handle)

    def section(self, i: int):
        off, size = C.c_uint64(), C.c_uint64()
        _check(self.lib.kvc_section(self.handle, i, C.byref(off), C.byref(size)), "kvc_section")
        return off.value, size.value


# ----------------------------------------------------------------------------
# entry points (same names as the C ABI; pointers are ints, streams are
# cudaStream_t handles as ints, e.g. torch.cuda.current_stream().cuda_stream)
# ----------------------------------------------------------------------------
def kvc_plan(profile: Profile, shape: Shape) -> Plan:
    return Plan(profile, shape)


def kvc_encode(plan: Plan, kv: KVRef, d_stream: int, stream_cap: int, d_workspace: int, workspace_bytes: int,
               d_stream_bytes: int = 0, stream: int = 0):
    _check(plan.lib.kvc_encode(plan.handle, C.byref(kv.struct), d_stream, stream_cap, d_workspace, workspace_bytes,
                               d_stream_bytes or None, stream or None), "kvc_encode")


def kvc_decode(plan: Plan, d_stream: int, stream_bytes: int, kv: KVRef, d_workspace: int, workspace_bytes: int,
               stream: int = 0):
    _check(plan.lib.kvc_decode(plan.handle, d_stream, stream_bytes, C.byref(kv.struct), d_workspace,
                               workspace_bytes, stream or None), "kvc_decode")


def kvc_quantize(plan: Plan, kv: KVRef, d_payload: int, d_workspace: int, workspace_bytes: int, stream: int = 0):
    _check(plan.lib.kvc_quantize(plan.handle, C.byref(kv.struct), d_payload, d_workspace, workspace_bytes,
                                 stream or None), "kvc_quantize")


def kvc_lossless_encode(plan: Plan, d_payload: int, d_stream: int, stream_cap: int, d_workspace: int,
                        workspace_bytes: int, d_stream_bytes: int = 0, stream: int = 0):
    _check(plan.lib.kvc_lossless_encode(plan.handle, d_payload or None, d_stream, stream_cap, d_workspace,
                                        workspace_bytes, d_stream_bytes or None, stream or None),
           "kvc_lossless_encode")


def kvc_lossless_decode(plan: Plan, d_stream: int, stream_bytes: int, d_payload: int, d_workspace: int,
                        workspace_bytes: int, stream: int = 0):
    _check(plan.lib.kvc_lossless_decode(plan.handle, d_stream, stream_bytes, d_payload or None, d_workspace,
                                        workspace_bytes, stream or None), "kvc_lossless_decode")


def kvc_dequantize(plan: Plan, d_payload: int, kv: KVRef, d_workspace: int, workspace_bytes: int, stream: int = 0):
    _check(plan.lib.kvc_dequantize(plan.handle, d_payload or None, C.byref(kv.struct), d_workspace,
                                   workspace_bytes, stream or None), "kvc_dequantize")


def kvc_query(d_workspace: int, stream: int = 0):
    """Returns (status, stream_bytes, flags) after synchronizing `stream`."""
    nbytes, flags = C.c_uint64(0), C.c_uint32(0)
    st = load().kvc_query(d_workspace, stream or None, C.byref(nbytes), C.byref(flags))
    return st, nbytes.value, flags.value


def kvc_timing_enable(plan: Plan, enable: bool, capacity: int = 4096):
    _check(plan.lib.kvc_timing_enable(plan.handle, int(enable), capacity), "kvc_timing_enable")


def kvc_timing_read(plan: Plan, max_records: int = 4096):
    arr = (Timing * max_records)()
    n = plan.lib.kvc_timing_read(plan.handle, arr, max_records)
    return [(arr[i].kernel.decode(), arr[i].ms) for i in range(n)]


def kvc_fuse_value_chunks(plan: Plan, enable: bool):
    """kvc_encode with the value encoder writing its whole code chunks into the stream."""
    _check(plan.lib.kvc_fuse_value_chunks(plan.handle, int(bool(enable))), "kvc_fuse_value_chunks")


def kvc_decode_codes_in_place(plan: Plan, enable: bool):
    """kvc_decode with the dequantizers reading stored code chunks from the stream (the default)."""
    _check(plan.lib.kvc_decode_codes_in_place(plan.handle, int(bool(enable))), "kvc_decode_codes_in_place")


def kvc_debug_generic_stages(plan: Plan, enable: bool):
    _check(plan.lib.kvc_debug_generic_stages(plan.handle, int(bool(enable))), "kvc_debug_generic_stages")


def kvc_debug_quotient_check(seed: int = 0, rounds: int = 1, stream: int = 0):
    """Returns the six counts: code quotients differing for t >= 1e-30, codes
    differing, dividends tested; scale quotients differing for w >= 1e-30, binary16
    scales differing, patterns tested."""
    out = (C.c_ulonglong * 6)()
    _check(load().kvc_debug_quotient_check(seed, rounds, out, stream or None), "kvc_debug_quotient_check")
    return tuple(int(x) for x in out)


def kvc_debug_lookback(plan: Plan, ticket: int, poll_limit: int = 0):
    _check(plan.lib.kvc_debug_lookback(plan.handle, ticket, poll_limit), "kvc_debug_lookback")


def kvc_lossless_encode_noalloc(plan: Plan, d_payload: int, d_stream: int, stream_cap: int, d_stream_bytes: int,
                                d_status: int = 0, stream: int = 0):
    """Lossless encode whose scratch is the library's own device array (no workspace,
    nothing allocated); the size goes to the device u64 at d_stream_bytes and the
    status bits to the device u32 at d_status."""
    _check(plan.lib.kvc_lossless_encode_noalloc(plan.handle, d_payload or None, d_stream, stream_cap, d_stream_bytes,
                                                d_status or None, stream or None), "kvc_lossless_encode_noalloc")

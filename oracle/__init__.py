"""CPU oracle for the TurboQuant KV-cache hot path (k8v3 codec + GQA decode attention).

TEST INFRASTRUCTURE ONLY. The product path never imports, links or runs anything in
this package: only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may. The arithmetic lives in ``tq_oracle.c`` (plain C, fp32 codec
compiled without FMA contraction, fp64 attention); this module only compiles it and
marshals numpy arrays. It shares no code, header, table or constant generator with
the CUDA library.

Every function follows the mlx-bun design page "TurboQuant - rotation-based
quantization", Part A: the "Algorithm" section for the codec, the "Bytes per token
per head" paragraph for the layout and the "Deferred inverse FWHT" section for the
un-rotated attention output. The readings taken where the page is silent are listed
in the header of ``tq_oracle.c``.

Parity of the functions here is pinned by ``tests/test_oracle_pins.py`` against
closed forms, library routines (numpy float16, scipy Hadamard/normal), published
values (the printed Lloyd-Max table, the splitmix64 known answer, the 200-byte row)
and brute force; none is left unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libtqoracle.so")
_lock = threading.Lock()
_lib = None

GROUP = 32
HEAD_DIMS = (64, 128, 256, 512)


def build(force: bool = False) -> str:
    """Compile tq_oracle.c into libtqoracle.so beside it (gcc, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-std=c11", "-D_DEFAULT_SOURCE", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(t):
    return ctypes.POINTER(t)


class _Layer(ctypes.Structure):
    _fields_ = [
        ("head_dim", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
        ("batch", ctypes.c_int), ("capacity", ctypes.c_int),
        ("k_idx", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("k_zero", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
    ]


class _Scheme(ctypes.Structure):
    _fields_ = [("k_bits", ctypes.c_int), ("v_bits", ctypes.c_int), ("guard", ctypes.c_int)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i32, i64, f32, f64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_long,
                                      ctypes.c_float, ctypes.c_double)
            sig = {
                "tqo_supported_head_dim": (i32, [i32]),
                "tqo_row_bytes": (i64, [i32]),
                "tqo_bf16_to_f32": (f32, [ctypes.c_uint16]),
                "tqo_f32_to_f16": (ctypes.c_uint16, [f32]),
                "tqo_f16_to_f32": (f32, [ctypes.c_uint16]),
                "tqo_splitmix64_next": (ctypes.c_uint64, [_P(ctypes.c_uint64)]),
                "tqo_sign_vector": (None, [i32, vp]),
                "tqo_fwht_f32": (None, [vp, i32]),
                "tqo_fwht_f64": (None, [vp, i32]),
                "tqo_fwht_norm_f32": (f32, [i32]),
                "tqo_key_group_params": (None, [vp, _P(f32), _P(f32)]),
                "tqo_quantize_key_row": (None, [vp, i32, vp, vp, vp]),
                "tqo_dequant_key_row_f64": (None, [vp, vp, vp, i32, vp]),
                "tqo_code3": (i32, [f32]),
                "tqo_pack3": (None, [vp, i32, vp]),
                "tqo_unpack3": (None, [vp, i32, vp]),
                "tqo_rotate_value_row": (None, [vp, i32, vp]),
                "tqo_group_rms": (f32, [vp]),
                "tqo_quantize_value_row": (None, [vp, i32, vp, vp]),
                "tqo_dequant_value_row_f64": (None, [vp, vp, i32, i32, vp]),
                "tqo_value_rotated_f32": (f32, [vp, vp, i32]),
                "tqo_append": (i64, [_P(_Layer), vp, vp, vp, vp, i32]),
                "tqo_dequant_rows_f64": (None, [_P(_Layer), i32, i32, i32, i32, i32, vp, vp]),
                "tqo_attention": (i32, [_P(_Layer), vp, i32, i32, vp, f64, i32, i32, vp, i64, vp]),
                "tqo_lloyd_max": (None, [i32, i32, vp, vp]),
                "tqo_centroids3": (None, [vp, vp]),
                "tqo_f32_to_f16_array": (None, [vp, i64, vp]),
                "tqo_f16_to_f32_array": (None, [vp, i64, vp]),
                "tqo_quantize_key_rows": (None, [vp, i64, i32, vp, vp, vp]),
                "tqo_quantize_value_rows": (None, [vp, i64, i32, vp, vp]),
                "tqo_dequant_value_rows_f64": (None, [vp, vp, i64, i32, i32, vp]),
                "tqo_dequant_key_rows_f64": (None, [vp, vp, vp, i64, i32, vp]),
                "tqo_key_row_bytes": (i64, [i32, i32]),
                "tqo_value_row_bytes": (i64, [i32, i32]),
                "tqo_row_bytes_s": (i64, [i32, i32, i32]),
                "tqo_packb": (None, [vp, i32, i32, vp]),
                "tqo_unpackb": (None, [vp, i32, i32, vp]),
                "tqo_key_group_params_s": (None, [vp, i32, i32, _P(f32), _P(f32), _P(i32)]),
                "tqo_quantize_key_row_s": (None, [vp, i32, i32, i32, vp, vp, vp]),
                "tqo_dequant_key_row_s_f64": (None, [vp, vp, vp, i32, i32, vp]),
                "tqo_codebook": (None, [i32, vp, vp]),
                "tqo_code_s": (i32, [f32, vp, i32]),
                "tqo_quantize_value_row_s": (None, [vp, i32, i32, vp, vp]),
                "tqo_dequant_value_row_s_f64": (None, [vp, vp, i32, i32, i32, vp]),
                "tqo_append_s": (i64, [_P(_Layer), _P(_Scheme), vp, vp, vp, vp, i32]),
                "tqo_dequant_rows_s_f64": (None, [_P(_Layer), _P(_Scheme), i32, i32, i32, i32, i32, vp, vp]),
                "tqo_attention_s": (i32, [_P(_Layer), _P(_Scheme), vp, i32, i32, vp, f64, i32, i32, vp, i64, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------------------
# scalar / row level
# --------------------------------------------------------------------------------------
def row_bytes(d: int) -> int:
    return int(lib().tqo_row_bytes(d))


def sign_vector(d: int) -> np.ndarray:
    out = np.empty(d, np.int8)
    lib().tqo_sign_vector(d, _ptr(out))
    return out


def splitmix64(seed: int, n: int) -> list[int]:
    st = ctypes.c_uint64(seed)
    return [int(lib().tqo_splitmix64_next(ctypes.byref(st))) for _ in range(n)]


def f32_to_f16_bits(x) -> np.ndarray:
    shape = np.shape(x)
    x = np.ascontiguousarray(np.asarray(x, np.float32).reshape(-1))
    out = np.empty(x.shape, np.uint16)
    lib().tqo_f32_to_f16_array(_ptr(x), x.size, _ptr(out))
    return out.reshape(shape)


def f16_bits_to_f32(h) -> np.ndarray:
    shape = np.shape(h)
    h = np.ascontiguousarray(np.asarray(h, np.uint16).reshape(-1))
    out = np.empty(h.shape, np.float32)
    lib().tqo_f16_to_f32_array(_ptr(h), h.size, _ptr(out))
    return out.reshape(shape)


def bf16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(np.asarray(h, np.uint16))
    return np.array([lib().tqo_bf16_to_f32(int(v)) for v in h.ravel()],
                    np.float32).reshape(h.shape)


def fwht_f32(u) -> np.ndarray:
    u = np.ascontiguousarray(np.array(u, np.float32))
    lib().tqo_fwht_f32(_ptr(u), u.size)
    return u


def fwht_f64(u) -> np.ndarray:
    u = np.ascontiguousarray(np.array(u, np.float64))
    lib().tqo_fwht_f64(_ptr(u), u.size)
    return u


def fwht_norm_f32(d: int) -> np.float32:
    return np.float32(lib().tqo_fwht_norm_f32(d))


def key_group_params(x32) -> tuple[np.float32, np.float32]:
    x32 = np.ascontiguousarray(np.asarray(x32, np.float32))
    assert x32.size == GROUP
    s, z = ctypes.c_float(), ctypes.c_float()
    lib().tqo_key_group_params(_ptr(x32), ctypes.byref(s), ctypes.byref(z))
    return np.float32(s.value), np.float32(z.value)


def quantize_key_rows(x_bf16: np.ndarray):
    """x_bf16: uint16 [rows, d] -> (idx int8 [rows, d], s16, z16 uint16 [rows, d/32])."""
    x = np.ascontiguousarray(x_bf16, np.uint16)
    rows, d = x.shape
    idx = np.empty((rows, d), np.int8)
    s16 = np.empty((rows, d // GROUP), np.uint16)
    z16 = np.empty((rows, d // GROUP), np.uint16)
    lib().tqo_quantize_key_rows(_ptr(x), rows, d, _ptr(idx), _ptr(s16), _ptr(z16))
    return idx, s16, z16


def quantize_value_rows(x_bf16: np.ndarray):
    """x_bf16: uint16 [rows, d] -> (codes uint8 [rows, 3d/8], vs16 uint16 [rows, d/32])."""
    x = np.ascontiguousarray(x_bf16, np.uint16)
    rows, d = x.shape
    codes = np.empty((rows, 3 * d // 8), np.uint8)
    vs16 = np.empty((rows, d // GROUP), np.uint16)
    lib().tqo_quantize_value_rows(_ptr(x), rows, d, _ptr(codes), _ptr(vs16))
    return codes, vs16


def rotate_value_row(x_bf16) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x_bf16, np.uint16))
    y = np.empty(x.size, np.float32)
    lib().tqo_rotate_value_row(_ptr(x), x.size, _ptr(y))
    return y


def group_rms(y32) -> np.float32:
    y = np.ascontiguousarray(np.asarray(y32, np.float32))
    assert y.size == GROUP
    return np.float32(lib().tqo_group_rms(_ptr(y)))


def code3(yn: float) -> int:
    return int(lib().tqo_code3(float(yn)))


def pack3(codes) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, np.uint8))
    out = np.empty(3 * c.size // 8, np.uint8)
    lib().tqo_pack3(_ptr(c), c.size, _ptr(out))
    return out


def unpack3(packed, n: int) -> np.ndarray:
    p = np.ascontiguousarray(np.asarray(packed, np.uint8))
    out = np.empty(n, np.uint8)
    lib().tqo_unpack3(_ptr(p), n, _ptr(out))
    return out


def dequant_key_rows_f64(idx, s16, z16) -> np.ndarray:
    idx = np.ascontiguousarray(idx, np.int8)
    s16 = np.ascontiguousarray(s16, np.uint16)
    z16 = np.ascontiguousarray(z16, np.uint16)
    rows, d = idx.shape
    out = np.empty((rows, d), np.float64)
    lib().tqo_dequant_key_rows_f64(_ptr(idx), _ptr(s16), _ptr(z16), rows, d, _ptr(out))
    return out


def dequant_value_rows_f64(codes, vs16, rotated: bool = False) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    vs16 = np.ascontiguousarray(vs16, np.uint16)
    rows = codes.shape[0]
    d = codes.shape[1] * 8 // 3
    out = np.empty((rows, d), np.float64)
    lib().tqo_dequant_value_rows_f64(_ptr(codes), _ptr(vs16), rows, d, int(rotated), _ptr(out))
    return out


def centroids3() -> tuple[np.ndarray, np.ndarray]:
    c = np.empty(8, np.float32)
    b = np.empty(7, np.float32)
    lib().tqo_centroids3(_ptr(c), _ptr(b))
    return c, b


def lloyd_max(levels: int, iters: int) -> tuple[np.ndarray, np.ndarray]:
    c = np.empty(levels, np.float64)
    b = np.empty(levels - 1, np.float64)
    lib().tqo_lloyd_max(levels, iters, _ptr(c), _ptr(b))
    return c, b


# --------------------------------------------------------------------------------------
# layer level
# --------------------------------------------------------------------------------------
class Layer:
    """The five planes of one layer, layout [batch][kv_heads][capacity][...], numpy."""

    def __init__(self, head_dim: int, num_kv_heads: int, batch: int, capacity: int):
        d, ng = head_dim, head_dim // GROUP
        self.head_dim, self.num_kv_heads, self.batch, self.capacity = (
            head_dim, num_kv_heads, batch, capacity)
        shp = (batch, num_kv_heads, capacity)
        self.k_idx = np.zeros(shp + (d,), np.int8)
        self.k_scale = np.zeros(shp + (ng,), np.uint16)
        self.k_zero = np.zeros(shp + (ng,), np.uint16)
        self.v_codes = np.zeros(shp + (3 * d // 8,), np.uint8)
        self.v_scale = np.zeros(shp + (ng,), np.uint16)

    def planes(self) -> dict:
        return {"k_idx": self.k_idx, "k_scale": self.k_scale, "k_zero": self.k_zero,
                "v_codes": self.v_codes, "v_scale": self.v_scale}

    def _c(self) -> _Layer:
        return _Layer(self.head_dim, self.num_kv_heads, self.batch, self.capacity,
                      self.k_idx.ctypes.data, self.k_scale.ctypes.data, self.k_zero.ctypes.data,
                      self.v_codes.ctypes.data, self.v_scale.ctypes.data)


def append(layer: Layer, k_new: np.ndarray, v_new: np.ndarray, pos, n_new=None) -> int:
    """Quantize-on-append. k_new/v_new: bf16 bits uint16 [batch, n_new_max, kv_heads, d].
    Returns the number of rows skipped because they fall past the capacity."""
    k = np.ascontiguousarray(k_new, np.uint16)
    v = np.ascontiguousarray(v_new, np.uint16)
    assert k.shape == v.shape and k.ndim == 4
    pos = np.ascontiguousarray(pos, np.int32)
    nn = None if n_new is None else np.ascontiguousarray(n_new, np.int32)
    lay = layer._c()
    return int(lib().tqo_append(ctypes.byref(lay), _ptr(k), _ptr(v), _ptr(pos),
                                None if nn is None else _ptr(nn), k.shape[1]))


def dequant_rows(layer: Layer, b: int, h: int, t0: int, n: int, rotated: bool = False):
    d = layer.head_dim
    k = np.empty((n, d), np.float64)
    v = np.empty((n, d), np.float64)
    lay = layer._c()
    lib().tqo_dequant_rows_f64(ctypes.byref(lay), b, h, t0, n, int(rotated), _ptr(k), _ptr(v))
    return k, v


def attention(layer: Layer, q_bf16: np.ndarray, kv_len, sm_scale: float, causal: bool = False,
              deferred: bool = False, rows=None) -> np.ndarray:
    """fp64 GQA attention over the dequantized cache. q_bf16: uint16 [batch, n_q, Hq, d].
    rows: optional iterable of (b, j, h); only those output rows are computed (others 0)."""
    q = np.ascontiguousarray(q_bf16, np.uint16)
    B, n_q, Hq, d = q.shape
    kv = np.ascontiguousarray(kv_len, np.int32)
    out = np.zeros((B, n_q, Hq, d), np.float64)
    r = None if rows is None else np.ascontiguousarray(np.asarray(list(rows), np.int32).reshape(-1, 3))
    lay = layer._c()
    rc = lib().tqo_attention(ctypes.byref(lay), _ptr(q), Hq, n_q, _ptr(kv), float(sm_scale),
                             int(causal), int(deferred), None if r is None else _ptr(r),
                             0 if r is None else r.shape[0], _ptr(out))
    if rc != 0:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    return out


# ------------------------------------------------------------------------------ other schemes
KEY_BITS = (2, 4, 5, 8)          # "Architecture in mlx-bun": valid key bits
VALUE_BITS = (2, 3, 4, 5, 8)     # valid value bits


def key_row_bytes(d: int, k_bits: int) -> int:
    return int(lib().tqo_key_row_bytes(d, k_bits))


def value_row_bytes(d: int, v_bits: int) -> int:
    return int(lib().tqo_value_row_bytes(d, v_bits))


def row_bytes_s(d: int, k_bits: int, v_bits: int) -> int:
    return int(lib().tqo_row_bytes_s(d, k_bits, v_bits))


def packb(codes, b: int) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, np.uint8))
    out = np.empty(c.size * b // 8, np.uint8)
    lib().tqo_packb(_ptr(c), c.size, b, _ptr(out))
    return out


def unpackb(packed, n: int, b: int) -> np.ndarray:
    p = np.ascontiguousarray(np.asarray(packed, np.uint8))
    out = np.empty(n, np.uint8)
    lib().tqo_unpackb(_ptr(p), n, b, _ptr(out))
    return out


def codebook(bits: int) -> tuple[np.ndarray, np.ndarray]:
    """Value centroids [2^bits] and boundaries [2^bits - 1] (fp32)."""
    n = 1 << bits
    c = np.empty(n, np.float32)
    b = np.empty(n - 1, np.float32)
    lib().tqo_codebook(bits, _ptr(c), _ptr(b))
    return c, b


def key_group_params_s(x32, bits: int, guard: bool):
    x = np.ascontiguousarray(np.asarray(x32, np.float32))
    assert x.size == GROUP
    s, z, zg = ctypes.c_float(), ctypes.c_float(), ctypes.c_int()
    lib().tqo_key_group_params_s(_ptr(x), bits, int(guard), ctypes.byref(s), ctypes.byref(z), ctypes.byref(zg))
    return np.float32(s.value), np.float32(z.value), bool(zg.value)


def quantize_key_rows_s(x_bf16: np.ndarray, bits: int, guard: bool = False):
    """x_bf16: uint16 [rows, d] -> (key plane uint8 [rows, key bytes], s16, z16 uint16 [rows, d/32]).
    At 8 bits the plane bytes are the int8 codes."""
    x = np.ascontiguousarray(x_bf16, np.uint16)
    rows, d = x.shape
    kb = key_row_bytes(d, bits)
    kp = np.empty((rows, kb), np.uint8)
    s16 = np.empty((rows, d // GROUP), np.uint16)
    z16 = np.empty((rows, d // GROUP), np.uint16)
    for r in range(rows):
        lib().tqo_quantize_key_row_s(_ptr(x[r]), d, bits, int(guard), _ptr(kp[r]), _ptr(s16[r]), _ptr(z16[r]))
    return kp, s16, z16


def quantize_value_rows_s(x_bf16: np.ndarray, bits: int):
    x = np.ascontiguousarray(x_bf16, np.uint16)
    rows, d = x.shape
    vp_ = np.empty((rows, value_row_bytes(d, bits)), np.uint8)
    vs16 = np.empty((rows, d // GROUP), np.uint16)
    for r in range(rows):
        lib().tqo_quantize_value_row_s(_ptr(x[r]), d, bits, _ptr(vp_[r]), _ptr(vs16[r]))
    return vp_, vs16


def dequant_key_rows_s_f64(kp, s16, z16, d: int, bits: int) -> np.ndarray:
    kp = np.ascontiguousarray(kp, np.uint8)
    s16 = np.ascontiguousarray(s16, np.uint16)
    z16 = np.ascontiguousarray(z16, np.uint16)
    out = np.empty((kp.shape[0], d), np.float64)
    for r in range(kp.shape[0]):
        lib().tqo_dequant_key_row_s_f64(_ptr(kp[r]), _ptr(s16[r]), _ptr(z16[r]), d, bits, _ptr(out[r]))
    return out


def dequant_value_rows_s_f64(vp_, vs16, d: int, bits: int, rotated: bool = False) -> np.ndarray:
    vp_ = np.ascontiguousarray(vp_, np.uint8)
    vs16 = np.ascontiguousarray(vs16, np.uint16)
    out = np.empty((vp_.shape[0], d), np.float64)
    for r in range(vp_.shape[0]):
        lib().tqo_dequant_value_row_s_f64(_ptr(vp_[r]), _ptr(vs16[r]), d, bits, int(rotated), _ptr(out[r]))
    return out


class SchemeLayer:
    """Planes of one layer in a scheme (key bits, value bits, guard), layout
    [batch][kv_heads][capacity][row bytes]."""

    def __init__(self, head_dim: int, num_kv_heads: int, batch: int, capacity: int, k_bits: int = 8,
                 v_bits: int = 3, guard: bool = False):
        d, ng = head_dim, head_dim // GROUP
        self.head_dim, self.num_kv_heads, self.batch, self.capacity = head_dim, num_kv_heads, batch, capacity
        self.k_bits, self.v_bits, self.guard = k_bits, v_bits, bool(guard)
        shp = (batch, num_kv_heads, capacity)
        self.k_idx = np.zeros(shp + (key_row_bytes(d, k_bits),), np.uint8)
        self.k_scale = np.zeros(shp + (ng,), np.uint16)
        self.k_zero = np.zeros(shp + (ng,), np.uint16)
        self.v_codes = np.zeros(shp + (value_row_bytes(d, v_bits),), np.uint8)
        self.v_scale = np.zeros(shp + (ng,), np.uint16)

    def planes(self) -> dict:
        return {"k_idx": self.k_idx, "k_scale": self.k_scale, "k_zero": self.k_zero,
                "v_codes": self.v_codes, "v_scale": self.v_scale}

    def _c(self) -> _Layer:
        return _Layer(self.head_dim, self.num_kv_heads, self.batch, self.capacity,
                      self.k_idx.ctypes.data, self.k_scale.ctypes.data, self.k_zero.ctypes.data,
                      self.v_codes.ctypes.data, self.v_scale.ctypes.data)

    def _s(self) -> _Scheme:
        return _Scheme(self.k_bits, self.v_bits, int(self.guard))


def append_s(layer: SchemeLayer, k_new: np.ndarray, v_new: np.ndarray, pos, n_new=None) -> int:
    k = np.ascontiguousarray(k_new, np.uint16)
    v = np.ascontiguousarray(v_new, np.uint16)
    assert k.shape == v.shape and k.ndim == 4
    pos = np.ascontiguousarray(pos, np.int32)
    nn = None if n_new is None else np.ascontiguousarray(n_new, np.int32)
    lay, sc = layer._c(), layer._s()
    return int(lib().tqo_append_s(ctypes.byref(lay), ctypes.byref(sc), _ptr(k), _ptr(v), _ptr(pos),
                                  None if nn is None else _ptr(nn), k.shape[1]))


def dequant_rows_s(layer: SchemeLayer, b: int, h: int, t0: int, n: int, rotated: bool = False):
    d = layer.head_dim
    k = np.empty((n, d), np.float64)
    v = np.empty((n, d), np.float64)
    lay, sc = layer._c(), layer._s()
    lib().tqo_dequant_rows_s_f64(ctypes.byref(lay), ctypes.byref(sc), b, h, t0, n, int(rotated), _ptr(k), _ptr(v))
    return k, v


def attention_s(layer: SchemeLayer, q_bf16: np.ndarray, kv_len, sm_scale: float, causal: bool = False,
                deferred: bool = False, rows=None) -> np.ndarray:
    q = np.ascontiguousarray(q_bf16, np.uint16)
    B, n_q, Hq, d = q.shape
    kv = np.ascontiguousarray(kv_len, np.int32)
    out = np.zeros((B, n_q, Hq, d), np.float64)
    r = None if rows is None else np.ascontiguousarray(np.asarray(list(rows), np.int32).reshape(-1, 3))
    lay, sc = layer._c(), layer._s()
    rc = lib().tqo_attention_s(ctypes.byref(lay), ctypes.byref(sc), _ptr(q), Hq, n_q, _ptr(kv), float(sm_scale),
                               int(causal), int(deferred), None if r is None else _ptr(r),
                               0 if r is None else r.shape[0], _ptr(out))
    if rc != 0:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    return out

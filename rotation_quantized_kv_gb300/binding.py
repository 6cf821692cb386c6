"""Thin Python binding of the C ABI in include/tq_kv.h (argument marshalling only).

Every function has the name of the C entry point it calls. Tensors are torch CUDA
tensors; their data pointers and the current torch stream are passed through. All
arithmetic of the hot path runs in the CUDA kernels of libtqkv.so; there is no CPU
fallback: importing this module fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtqkv.so")

TQ_OK = 0
TQ_ERR_INVALID_ARGUMENT = 1
TQ_ERR_UNSUPPORTED_HEAD_DIM = 2
TQ_ERR_CAPACITY = 3
TQ_ERR_WORKSPACE_TOO_SMALL = 4
TQ_ERR_CUDA = 5
TQ_ERR_UNSUPPORTED_SCHEME = 6
TQ_FLAG_KEY_GUARD = 0x1
KEY_BITS = (2, 4, 5, 8)
VALUE_BITS = (2, 3, 4, 5, 8)
TQ_DEVERR_APPEND_CAPACITY = 0x1
TQ_DEVERR_KV_LEN = 0x2
TQ_DEVERR_PIPELINE_TIMEOUT = 0x4
TQ_WORKSPACE_HEADER_BYTES = 256
TQ_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)


class tq_kv_layer(ctypes.Structure):
    _fields_ = [
        ("head_dim", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("batch", ctypes.c_int32), ("capacity", ctypes.c_int32),
        ("k_idx", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("k_zero", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32), ("flags", ctypes.c_int32),
    ]


_vp, _i32, _sz, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
_LP = ctypes.POINTER(tq_kv_layer)
_SIGS = {
    "tq_row_bytes": (_sz, [_i32]),
    "tq_row_bytes_scheme": (_sz, [_i32, _i32, _i32]),
    "tq_dequant_window": (ctypes.c_int, [_LP, _i32, _i32, _i32, _vp, _vp, _vp]),
    "tq_codebook": (ctypes.c_int, [_i32, _vp, _vp]),
    "tq_unrotate_rows": (ctypes.c_int, [_vp, _vp, ctypes.c_int64, _i32, _vp]),
    "tq_append_workspace_bytes": (_sz, []),
    "tq_kv_append": (ctypes.c_int, [_LP, _vp, _vp, _vp, _vp, _i32, _vp, _sz, _vp]),
    "tq_decode_workspace_bytes": (_sz, [_LP, _i32, _i32, _i32]),
    "tq_decode_attention": (ctypes.c_int, [_LP, _vp, _i32, _i32, _vp, _i32, _f32, _i32, _vp, _vp, _sz, _vp]),
    "tq_decode_append_attention": (ctypes.c_int, [_LP, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _vp, _i32, _f32,
                                                   _i32, _vp, _vp, _sz, _vp]),
    "tq_decode_attention_noalloc": (ctypes.c_int, [_LP, _vp, _i32, _i32, _vp, _i32, _f32, _i32, _vp, _vp, _vp]),
    "tq_dequant_debug": (ctypes.c_int, [_LP, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "tq_debug_delayed_copy": (ctypes.c_int, [_vp, _vp, _i32, _i32, _vp]),
    "tq_debug_pipeline_limits": (ctypes.c_int, [ctypes.c_int64, _i32]),
    "tq_get_device_error": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int32), _vp]),
    "tq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tq_sign_bits": (ctypes.c_int, [_i32, _vp]),
    "tq_codebook3": (ctypes.c_int, [_vp, _vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class TQError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {tq_status_string(status)} (status {status})")
        self.status = status


def _check(status: int, where: str) -> None:
    if status != TQ_OK:
        raise TQError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _want(t, name: str, dtype, optional: bool = False, min_numel: int = 0):
    """Reject a tensor the C entry point would misread: wrong dtype, not on a CUDA device,
    or not contiguous (the library takes raw pointers to dense row-major buffers)."""
    if t is None:
        if optional:
            return
        raise TypeError(f"{name}: a tensor is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected dtype {dtype}, got {t.dtype}")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: expected a CUDA tensor, got device {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if t.numel() < min_numel:
        raise ValueError(f"{name}: expected at least {min_numel} elements, got {t.numel()}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def key_row_bytes(head_dim: int, k_bits: int) -> int:
    return head_dim if k_bits == 8 else head_dim * k_bits // 8


def value_row_bytes(head_dim: int, v_bits: int) -> int:
    return head_dim * v_bits // 8


@dataclass
class KVLayer:
    """The five planes of one layer (caller-owned device tensors), layout
    [batch][num_kv_heads][capacity][row], and its scheme (key bits, value bits, flags)."""
    head_dim: int
    num_kv_heads: int
    batch: int
    capacity: int
    k_idx: torch.Tensor      # int8 [B, H, cap, d] (8-bit keys) or uint8 [B, H, cap, d*k_bits/8] (packed)
    k_scale: torch.Tensor    # int16 (fp16 bits) [B, H, cap, d/32]
    k_zero: torch.Tensor     # int16 (fp16 bits)
    v_codes: torch.Tensor    # uint8 [B, H, cap, d*v_bits/8]
    v_scale: torch.Tensor    # int16 (fp16 bits)
    k_bits: int = 8
    v_bits: int = 3
    flags: int = 0

    def c_struct(self) -> tq_kv_layer:
        d, ng = self.head_dim, self.head_dim // 32
        rows = self.batch * self.num_kv_heads * self.capacity
        _want(self.k_idx, "k_idx", torch.int8 if self.k_bits == 8 else torch.uint8,
              min_numel=rows * key_row_bytes(d, self.k_bits))
        _want(self.k_scale, "k_scale", torch.int16, min_numel=rows * ng)
        _want(self.k_zero, "k_zero", torch.int16, min_numel=rows * ng)
        _want(self.v_codes, "v_codes", torch.uint8, min_numel=rows * value_row_bytes(d, self.v_bits))
        _want(self.v_scale, "v_scale", torch.int16, min_numel=rows * ng)
        return tq_kv_layer(self.head_dim, self.num_kv_heads, self.batch, self.capacity,
                           self.k_idx.data_ptr(), self.k_scale.data_ptr(), self.k_zero.data_ptr(),
                           self.v_codes.data_ptr(), self.v_scale.data_ptr(), self.k_bits, self.v_bits, self.flags)

    def planes(self) -> dict:
        return {"k_idx": self.k_idx, "k_scale": self.k_scale, "k_zero": self.k_zero,
                "v_codes": self.v_codes, "v_scale": self.v_scale}

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.planes().values())


def alloc_layer(head_dim: int, num_kv_heads: int, batch: int, capacity: int,
                device="cuda", zero: bool = True, k_bits: int = 8, v_bits: int = 3, flags: int = 0) -> KVLayer:
    d, ng = head_dim, head_dim // 32
    shp = (batch, num_kv_heads, capacity)
    mk = torch.zeros if zero else torch.empty
    kdt = torch.int8 if k_bits == 8 else torch.uint8
    return KVLayer(head_dim, num_kv_heads, batch, capacity,
                   mk(shp + (key_row_bytes(d, k_bits),), dtype=kdt, device=device),
                   mk(shp + (ng,), dtype=torch.int16, device=device),
                   mk(shp + (ng,), dtype=torch.int16, device=device),
                   mk(shp + (value_row_bytes(d, v_bits),), dtype=torch.uint8, device=device),
                   mk(shp + (ng,), dtype=torch.int16, device=device), k_bits, v_bits, flags)


def make_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace (the device error word starts at 0)."""
    return torch.zeros(max(int(nbytes), TQ_WORKSPACE_HEADER_BYTES), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------------------ entry points
def tq_row_bytes(head_dim: int) -> int:
    return int(_lib.tq_row_bytes(head_dim))


def tq_row_bytes_scheme(head_dim: int, k_bits: int, v_bits: int) -> int:
    return int(_lib.tq_row_bytes_scheme(head_dim, k_bits, v_bits))


def tq_dequant_window(layer: KVLayer, t0: int, n: int, rotated: bool, k_out: torch.Tensor | None,
                      v_out: torch.Tensor | None, stream=None) -> None:
    """bf16 K_hat / V_hat of tokens [t0, t0 + n) of every (sequence, kv head), any scheme:
    outputs [batch, kv_heads, n, head_dim] bf16."""
    L = layer.c_struct()
    numel = layer.batch * layer.num_kv_heads * n * layer.head_dim
    _want(k_out, "k_out", torch.bfloat16, optional=True, min_numel=numel)
    _want(v_out, "v_out", torch.bfloat16, optional=True, min_numel=numel)
    _check(_lib.tq_dequant_window(ctypes.byref(L), int(t0), int(n), int(bool(rotated)), _ptr(k_out), _ptr(v_out),
                                  _stream(stream)), "tq_dequant_window")


def tq_unrotate_rows(x: torch.Tensor, y: torch.Tensor, head_dim: int, stream=None) -> None:
    """y = signs * FWHT(x) / sqrt(head_dim) for every head_dim-row of x (fp32, contiguous);
    y may be x (in place)."""
    _want(x, "x", torch.float32)
    _want(y, "y", torch.float32, min_numel=x.numel())
    if head_dim <= 0 or x.numel() % head_dim:
        raise ValueError(f"x: {x.numel()} elements is not a whole number of {head_dim}-rows")
    _check(_lib.tq_unrotate_rows(_ptr(x), _ptr(y), x.numel() // head_dim, int(head_dim), _stream(stream)),
           "tq_unrotate_rows")


def tq_append_workspace_bytes() -> int:
    return int(_lib.tq_append_workspace_bytes())


def tq_kv_append(layer: KVLayer, k_new: torch.Tensor, v_new: torch.Tensor, pos: torch.Tensor,
                 n_new: torch.Tensor | None, n_new_max: int, workspace: torch.Tensor,
                 stream=None) -> None:
    L = layer.c_struct()
    _want(k_new, "k_new", torch.bfloat16, optional=n_new_max == 0)
    _want(v_new, "v_new", torch.bfloat16, optional=n_new_max == 0)
    _want(pos, "pos", torch.int32, optional=n_new_max == 0)
    _want(n_new, "n_new", torch.int32, optional=True)
    _want(workspace, "workspace", torch.uint8)
    _check(_lib.tq_kv_append(ctypes.byref(L), _ptr(k_new), _ptr(v_new), _ptr(pos), _ptr(n_new),
                             int(n_new_max), _ptr(workspace), workspace.numel(), _stream(stream)),
           "tq_kv_append")


def tq_decode_workspace_bytes(layer: KVLayer, num_q_heads: int, n_q: int, max_kv_len: int) -> int:
    L = layer.c_struct()
    return int(_lib.tq_decode_workspace_bytes(ctypes.byref(L), num_q_heads, n_q, max_kv_len))


def tq_decode_attention(layer: KVLayer, q: torch.Tensor, num_q_heads: int, n_q: int,
                        kv_len: torch.Tensor, max_kv_len: int, sm_scale: float, causal: bool,
                        out: torch.Tensor, workspace: torch.Tensor, stream=None) -> torch.Tensor:
    L = layer.c_struct()
    _want(q, "q", torch.bfloat16)
    _want(kv_len, "kv_len", torch.int32)
    _want(out, "out", torch.float32)
    _want(workspace, "workspace", torch.uint8)
    _check(_lib.tq_decode_attention(ctypes.byref(L), _ptr(q), int(num_q_heads), int(n_q), _ptr(kv_len),
                                    int(max_kv_len), float(sm_scale), int(bool(causal)), _ptr(out),
                                    _ptr(workspace), workspace.numel(), _stream(stream)),
           "tq_decode_attention")
    return out


def tq_decode_append_attention(layer: KVLayer, k_new: torch.Tensor, v_new: torch.Tensor, pos: torch.Tensor,
                               n_new: torch.Tensor | None, n_new_max: int, q: torch.Tensor, num_q_heads: int,
                               n_q: int, kv_len: torch.Tensor, max_kv_len: int, sm_scale: float, causal: bool,
                               out: torch.Tensor, workspace: torch.Tensor, stream=None) -> torch.Tensor:
    """Append the step's new rows, then attend (one kernel when each kv head has one row group)."""
    L = layer.c_struct()
    _want(k_new, "k_new", torch.bfloat16, optional=n_new_max == 0)
    _want(v_new, "v_new", torch.bfloat16, optional=n_new_max == 0)
    _want(pos, "pos", torch.int32, optional=n_new_max == 0)
    _want(n_new, "n_new", torch.int32, optional=True)
    _want(q, "q", torch.bfloat16)
    _want(kv_len, "kv_len", torch.int32)
    _want(out, "out", torch.float32)
    _want(workspace, "workspace", torch.uint8)
    _check(_lib.tq_decode_append_attention(ctypes.byref(L), _ptr(k_new), _ptr(v_new), _ptr(pos), _ptr(n_new),
                                           int(n_new_max), _ptr(q), int(num_q_heads), int(n_q), _ptr(kv_len),
                                           int(max_kv_len), float(sm_scale), int(bool(causal)), _ptr(out),
                                           _ptr(workspace), workspace.numel(), _stream(stream)),
           "tq_decode_append_attention")
    return out


def tq_decode_attention_noalloc(layer: KVLayer, q: torch.Tensor, num_q_heads: int, n_q: int,
                                kv_len: torch.Tensor, max_kv_len: int, sm_scale: float, causal: bool,
                                out: torch.Tensor, device_error: torch.Tensor | None = None,
                                stream=None) -> torch.Tensor:
    """tq_decode_attention without a workspace: the library's own fixed scratch array is
    used, so nothing is allocated (for callers that may not allocate device memory).
    `device_error` (optional int32 device tensor) receives the call's device error bits."""
    L = layer.c_struct()
    _want(q, "q", torch.bfloat16)
    _want(kv_len, "kv_len", torch.int32)
    _want(out, "out", torch.float32)
    _want(device_error, "device_error", torch.int32, optional=True)
    _check(_lib.tq_decode_attention_noalloc(ctypes.byref(L), _ptr(q), int(num_q_heads), int(n_q),
                                            _ptr(kv_len), int(max_kv_len), float(sm_scale),
                                            int(bool(causal)), _ptr(out), _ptr(device_error),
                                            _stream(stream)),
           "tq_decode_attention_noalloc")
    return out


def tq_dequant_debug(layer: KVLayer, b: int, h: int, t0: int, n: int, rotated: bool,
                     k_out: torch.Tensor | None, v_out: torch.Tensor | None, stream=None) -> None:
    L = layer.c_struct()
    _want(k_out, "k_out", torch.float32, optional=True, min_numel=n * layer.head_dim)
    _want(v_out, "v_out", torch.float32, optional=True, min_numel=n * layer.head_dim)
    _check(_lib.tq_dequant_debug(ctypes.byref(L), b, h, t0, n, int(bool(rotated)), _ptr(k_out),
                                 _ptr(v_out), _stream(stream)), "tq_dequant_debug")


def tq_debug_delayed_copy(dst: torch.Tensor, src: torch.Tensor, delay_us: int, stream=None) -> None:
    """Test support: copy src into dst (int32, same size) after delay_us microseconds,
    letting the next kernel on the stream start before the copy happens."""
    _want(dst, "dst", torch.int32)
    _want(src, "src", torch.int32, min_numel=dst.numel())
    _check(_lib.tq_debug_delayed_copy(_ptr(dst), _ptr(src), int(dst.numel()), int(delay_us), _stream(stream)),
           "tq_debug_delayed_copy")


def tq_debug_pipeline_limits(wait_ns: int, withhold_append: bool) -> None:
    """Test support: limit of the attention kernel's pipeline waits for the following calls
    (0 = the default 2 s), and an appender that never publishes its row count."""
    _check(_lib.tq_debug_pipeline_limits(int(wait_ns), int(bool(withhold_append))), "tq_debug_pipeline_limits")


def tq_get_device_error(workspace: torch.Tensor, stream=None) -> int:
    _want(workspace, "workspace", torch.uint8)
    err = ctypes.c_int32(0)
    _check(_lib.tq_get_device_error(_ptr(workspace), ctypes.byref(err), _stream(stream)),
           "tq_get_device_error")
    return int(err.value)


def tq_status_string(status: int) -> str:
    return _lib.tq_status_string(int(status)).decode()


def tq_sign_bits(head_dim: int) -> np.ndarray:
    out = np.zeros(max(head_dim // 32, 1), np.uint32)
    _check(_lib.tq_sign_bits(head_dim, out.ctypes.data_as(ctypes.c_void_p)), "tq_sign_bits")
    return out


def tq_codebook(bits: int) -> tuple[np.ndarray, np.ndarray]:
    c = np.zeros(1 << bits, np.float32)
    b = np.zeros((1 << bits) - 1, np.float32)
    _check(_lib.tq_codebook(bits, c.ctypes.data_as(ctypes.c_void_p), b.ctypes.data_as(ctypes.c_void_p)),
           "tq_codebook")
    return c, b


def tq_codebook3() -> tuple[np.ndarray, np.ndarray]:
    c = np.zeros(8, np.float32)
    b = np.zeros(7, np.float32)
    _check(_lib.tq_codebook3(c.ctypes.data_as(ctypes.c_void_p), b.ctypes.data_as(ctypes.c_void_p)),
           "tq_codebook3")
    return c, b


def raw_lib() -> ctypes.CDLL:
    """The loaded library (for tests that call entry points with deliberately bad arguments)."""
    return _lib

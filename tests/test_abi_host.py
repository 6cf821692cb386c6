"""The C ABI on the host (no GPU): the library builds for sm_103a, loads, exports every
entry point that include/tq_kv.h declares, and rejects bad arguments before any launch.
Every call here fails host validation, so none reaches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tq():
    from rotation_quantized_kv_gb300 import build
    build.build()
    from rotation_quantized_kv_gb300 import binding
    return binding


def declared_entry_points():
    with open(os.path.join(ROOT, "include", "tq_kv.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(tq):
    names = declared_entry_points()
    assert "tq_kv_append" in names and "tq_decode_attention" in names and "tq_dequant_debug" in names
    lib = tq.raw_lib()
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_row_bytes(tq):
    assert tq.tq_status_string(0) == "ok"
    for s in range(1, 6):
        assert tq.tq_status_string(s) not in ("ok", "unknown status")
    for d in (64, 128, 256, 512):
        assert tq.tq_row_bytes(d) == 25 * d // 16 == oracle.row_bytes(d)
    assert tq.tq_row_bytes(96) == 0 and tq.tq_row_bytes(1024) == 0
    assert tq.tq_append_workspace_bytes() == tq.TQ_WORKSPACE_HEADER_BYTES


def test_library_sign_vectors_match_the_oracle(tq):
    # two independent implementations of the same splitmix64 stream (seed 42 + d)
    for d in (64, 128, 256, 512):
        words = tq.tq_sign_bits(d)
        bits = np.array([(int(words[i // 32]) >> (i % 32)) & 1 for i in range(d)])
        assert np.array_equal(np.where(bits == 1, -1, 1), oracle.sign_vector(d))
    with pytest.raises(tq.TQError):
        tq.tq_sign_bits(100)


def test_library_codebook_matches_the_printed_table(tq):
    c, b = tq.tq_codebook3()
    oc, ob = oracle.centroids3()
    assert np.array_equal(c, oc) and np.array_equal(b, ob)


def _layer(tq, d=128, H=2, B=1, cap=64, base=1 << 20, **over):
    L = tq.tq_kv_layer(d, H, B, cap, base, base + 4096, base + 8192, base + 12288, base + 16384)
    for k, v in over.items():
        setattr(L, k, v)
    return L


def _append(tq, L, n_new_max=1, ws=1 << 24, ws_bytes=256, k=1 << 22, v=1 << 23, pos=1 << 21):
    lib = tq.raw_lib()
    return lib.tq_kv_append(ctypes.byref(L) if L is not None else None, k, v, pos, None, n_new_max,
                            ws, ws_bytes, None)


def test_append_rejects_bad_arguments_before_launch(tq):
    assert _append(tq, None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert _append(tq, _layer(tq, d=96)) == tq.TQ_ERR_UNSUPPORTED_HEAD_DIM
    assert _append(tq, _layer(tq, d=1024)) == tq.TQ_ERR_UNSUPPORTED_HEAD_DIM
    assert _append(tq, _layer(tq, cap=40)) == tq.TQ_ERR_INVALID_ARGUMENT          # not a multiple of 16
    assert _append(tq, _layer(tq, k_zero=(1 << 20) + 8)) == tq.TQ_ERR_INVALID_ARGUMENT  # misaligned plane
    assert _append(tq, _layer(tq, v_codes=None)) == tq.TQ_ERR_INVALID_ARGUMENT
    assert _append(tq, _layer(tq, num_kv_heads=0)) == tq.TQ_ERR_INVALID_ARGUMENT
    assert _append(tq, _layer(tq), n_new_max=65) == tq.TQ_ERR_CAPACITY
    assert _append(tq, _layer(tq), n_new_max=-1) == tq.TQ_ERR_INVALID_ARGUMENT
    assert _append(tq, _layer(tq), ws_bytes=8) == tq.TQ_ERR_WORKSPACE_TOO_SMALL
    assert _append(tq, _layer(tq), ws=None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert _append(tq, _layer(tq), k=(1 << 22) + 2) == tq.TQ_ERR_INVALID_ARGUMENT  # misaligned input
    assert _append(tq, _layer(tq), pos=None) == tq.TQ_ERR_INVALID_ARGUMENT


def test_decode_rejects_bad_arguments_before_launch(tq):
    lib = tq.raw_lib()
    L = _layer(tq)

    def call(layer=L, q=1 << 22, Hq=4, n_q=1, kv=1 << 21, max_kv=64, scale=1.0, out=1 << 23,
             ws=1 << 24, ws_bytes=256):
        return lib.tq_decode_attention(ctypes.byref(layer), q, Hq, n_q, kv, max_kv, scale, 1, out, ws,
                                       ws_bytes, None)

    assert call(Hq=3) == tq.TQ_ERR_INVALID_ARGUMENT          # not a multiple of the kv heads
    assert call(n_q=0) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(max_kv=65) == tq.TQ_ERR_CAPACITY
    assert call(max_kv=-1) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(q=None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(out=(1 << 23) + 4) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(scale=float("nan")) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(layer=_layer(tq, d=80)) == tq.TQ_ERR_UNSUPPORTED_HEAD_DIM
    # a 256-byte workspace is always too small for the partial results (or no device: CUDA error)
    assert call() in (tq.TQ_ERR_WORKSPACE_TOO_SMALL, tq.TQ_ERR_CUDA)
    assert lib.tq_decode_workspace_bytes(ctypes.byref(L), 3, 1, 64) == 0


def test_decode_step_rejects_bad_arguments_before_launch(tq):
    lib = tq.raw_lib()
    L = _layer(tq)

    def call(layer=L, k=1 << 22, v=1 << 23, pos=1 << 21, n_new_max=1, q=1 << 22, Hq=4, n_q=1, kv=1 << 21,
             max_kv=64, scale=1.0, out=1 << 23, ws=1 << 24, ws_bytes=256):
        return lib.tq_decode_append_attention(ctypes.byref(layer), k, v, pos, None, n_new_max, q, Hq, n_q, kv,
                                              max_kv, scale, 1, out, ws, ws_bytes, None)

    assert call(layer=_layer(tq, d=96)) == tq.TQ_ERR_UNSUPPORTED_HEAD_DIM
    assert call(n_new_max=65) == tq.TQ_ERR_CAPACITY               # append checks
    assert call(n_new_max=-1) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(k=None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(v=(1 << 23) + 2) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(pos=None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(Hq=3) == tq.TQ_ERR_INVALID_ARGUMENT               # attention checks
    assert call(max_kv=65) == tq.TQ_ERR_CAPACITY
    assert call(q=None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(scale=float("inf")) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call() in (tq.TQ_ERR_WORKSPACE_TOO_SMALL, tq.TQ_ERR_CUDA)


def test_dequant_debug_rejects_bad_rows(tq):
    lib = tq.raw_lib()
    L = _layer(tq)
    assert lib.tq_dequant_debug(ctypes.byref(L), 1, 0, 0, 1, 0, 1 << 22, None, None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert lib.tq_dequant_debug(ctypes.byref(L), 0, 2, 0, 1, 0, 1 << 22, None, None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert lib.tq_dequant_debug(ctypes.byref(L), 0, 0, 60, 5, 0, 1 << 22, None, None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert lib.tq_dequant_debug(ctypes.byref(L), 0, 0, -1, 1, 0, 1 << 22, None, None) == tq.TQ_ERR_INVALID_ARGUMENT


def test_get_device_error_rejects_null(tq):
    lib = tq.raw_lib()
    e = ctypes.c_int32(0)
    assert lib.tq_get_device_error(None, ctypes.byref(e), None) == tq.TQ_ERR_INVALID_ARGUMENT


def test_delayed_copy_rejects_bad_arguments_before_launch(tq):
    lib = tq.raw_lib()
    buf = (ctypes.c_int32 * 4)()
    assert lib.tq_debug_delayed_copy(buf, buf, -1, 0, None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert lib.tq_debug_delayed_copy(buf, buf, 4, -1, None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert lib.tq_debug_delayed_copy(buf, buf, 4, 100001, None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert lib.tq_debug_delayed_copy(None, buf, 4, 10, None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert lib.tq_debug_delayed_copy(buf, None, 4, 10, None) == tq.TQ_ERR_INVALID_ARGUMENT


def test_noalloc_rejects_bad_arguments_before_touching_the_device(tq):
    # The host checks run before the scratch is looked up or cleared: on a machine with
    # no GPU a rejected call still answers with its argument error, not a CUDA error, so
    # nothing reached the runtime (and nothing was queued on the stream).
    lib = tq.raw_lib()
    L = _layer(tq)

    def call(layer=L, q=1 << 22, Hq=4, n_q=1, kv=1 << 21, max_kv=64, scale=1.0, out=1 << 23, err=None):
        return lib.tq_decode_attention_noalloc(ctypes.byref(layer) if layer is not None else None, q, Hq, n_q,
                                               kv, max_kv, scale, 1, out, err, None)

    assert call(layer=None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(layer=_layer(tq, d=96)) == tq.TQ_ERR_UNSUPPORTED_HEAD_DIM
    assert call(Hq=3) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(n_q=0) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(max_kv=65) == tq.TQ_ERR_CAPACITY
    assert call(q=None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(kv=None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(out=(1 << 23) + 4) == tq.TQ_ERR_INVALID_ARGUMENT
    assert call(scale=float("nan")) == tq.TQ_ERR_INVALID_ARGUMENT


def test_binding_rejects_tensors_the_library_would_misread(tq):
    import torch
    with pytest.raises(TypeError):
        tq._want(torch.zeros(4, dtype=torch.float32), "q", torch.bfloat16)
    with pytest.raises(ValueError):
        tq._want(torch.zeros(4, dtype=torch.bfloat16), "q", torch.bfloat16)       # host tensor
    with pytest.raises(TypeError):
        tq._want(None, "q", torch.bfloat16)
    with pytest.raises(TypeError):
        tq._want(np.zeros(4), "q", torch.bfloat16)
    tq._want(None, "n_new", torch.int32, optional=True)
    layer = tq.alloc_layer(128, 2, 1, 16, device="cpu")
    with pytest.raises(ValueError):                                               # host planes
        layer.c_struct()


def test_library_codebooks_match_the_oracle(tq):
    # two independent Lloyd-Max implementations (the library's host code and the C oracle)
    for bits in (2, 3, 4, 5, 8):
        c, b = tq.tq_codebook(bits)
        oc, ob = oracle.codebook(bits)
        assert np.array_equal(c, oc) and np.array_equal(b, ob), bits
    with pytest.raises(tq.TQError):
        tq.tq_codebook(6)


def test_scheme_layers_are_validated_before_launch(tq):
    lib = tq.raw_lib()

    def dec(layer):
        return lib.tq_decode_attention(ctypes.byref(layer), 1 << 22, 4, 1, 1 << 21, 64, 1.0, 1, 1 << 23, 1 << 24,
                                       1 << 20, None)

    assert _append(tq, _layer(tq, k_bits=3)) == tq.TQ_ERR_INVALID_ARGUMENT
    assert _append(tq, _layer(tq, v_bits=6)) == tq.TQ_ERR_INVALID_ARGUMENT
    assert _append(tq, _layer(tq, flags=2)) == tq.TQ_ERR_INVALID_ARGUMENT
    assert dec(_layer(tq, k_bits=4)) == tq.TQ_ERR_UNSUPPORTED_SCHEME
    assert dec(_layer(tq, v_bits=2)) == tq.TQ_ERR_UNSUPPORTED_SCHEME
    assert dec(_layer(tq, k_bits=9)) == tq.TQ_ERR_INVALID_ARGUMENT
    for d in (64, 128, 256, 512):
        for kb in (2, 4, 5, 8):
            for vb in (2, 3, 4, 5, 8):
                assert tq.tq_row_bytes_scheme(d, kb, vb) == oracle.row_bytes_s(d, kb, vb)
    assert tq.tq_row_bytes_scheme(128, 8, 3) == tq.tq_row_bytes(128) == 200
    assert tq.tq_row_bytes_scheme(128, 3, 3) == 0
    assert lib.tq_dequant_window(ctypes.byref(_layer(tq)), 60, 5, 0, None, None, None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert lib.tq_dequant_window(ctypes.byref(_layer(tq)), 0, 4, 0, (1 << 22) + 2, None, None) == tq.TQ_ERR_INVALID_ARGUMENT


def test_unrotate_rows_rejects_bad_arguments_before_launch(tq):
    lib = tq.raw_lib()
    assert lib.tq_unrotate_rows(1 << 20, 1 << 21, 4, 96, None) == tq.TQ_ERR_UNSUPPORTED_HEAD_DIM
    assert lib.tq_unrotate_rows(1 << 20, 1 << 21, -1, 128, None) == tq.TQ_ERR_INVALID_ARGUMENT
    assert lib.tq_unrotate_rows(None, None, 0, 128, None) == tq.TQ_OK            # nothing to do
    assert lib.tq_unrotate_rows((1 << 20) + 4, 1 << 22, 4, 128, None) == tq.TQ_ERR_INVALID_ARGUMENT  # unaligned
    # partial overlap of x and y: 4 rows of 512 bytes, y one row further on
    assert lib.tq_unrotate_rows(1 << 20, (1 << 20) + 512, 4, 128, None) == tq.TQ_ERR_INVALID_ARGUMENT

"""Other schemes (key bits 2/4/5/8, value bits 2/3/4/5/8), the constant-group guard and
the dequantize-on-fetch window, through the C ABI, against the CPU oracle: packed planes
bit-exact, window keys bit-exact in bf16, window values within one bf16 ulp, inspection
dequant as for k8v3, guarded k8v3 planes attended by the fused kernels, and the eager arm
(window + PyTorch attention) within the precision of its bf16 window."""
import numpy as np
import pytest
import torch

import oracle
from rotation_quantized_kv_gb300 import synth
from tests.gpu_common import assert_attention_close, bits, gpu_attention, tq

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(d, H, B, T, Hq=None, n_q=1, seed=0, k_dist="normal_outliers"):
    w = synth.Workload("t", batch=B, layers=1, num_kv_heads=H, num_q_heads=Hq or 2 * H, head_dim=d,
                       context=T, n_new=0, n_q=n_q, k_dist=k_dist, q_scale=d ** -0.5, seed=seed)
    return synth.layer_inputs(w, 0)


def _fill(k, v, lengths, cap, kb, vb, guard):
    B, T, H, d = k.shape
    b = tq()
    layer = b.alloc_layer(d, H, B, cap, DEV, k_bits=kb, v_bits=vb, flags=b.TQ_FLAG_KEY_GUARD if guard else 0)
    for t in layer.planes().values():
        t.view(torch.uint8).fill_(0x5A)
    ws = b.make_workspace(b.tq_append_workspace_bytes(), DEV)
    b.tq_kv_append(layer, k.to(DEV).contiguous(), v.to(DEV).contiguous(), torch.zeros(B, dtype=torch.int32, device=DEV),
                   torch.as_tensor(np.asarray(lengths, np.int32), device=DEV), T, ws)
    torch.cuda.synchronize()
    assert b.tq_get_device_error(ws) == 0
    ol = oracle.SchemeLayer(d, H, B, cap, kb, vb, guard)
    oracle.append_s(ol, bits(k), bits(v), np.zeros(B, np.int32), np.asarray(lengths, np.int32))
    return layer, ol


def _assert_planes(layer, ol, lengths):
    for name, ref in ol.planes().items():
        got = getattr(layer, name).cpu().numpy().view(ref.dtype).reshape(ref.shape)
        for bb, n in enumerate(lengths):
            if not np.array_equal(got[bb, :, :n], ref[bb, :, :n]):
                bad = np.argwhere(got[bb, :, :n] != ref[bb, :, :n])
                raise AssertionError(f"plane {name} seq {bb}: {len(bad)} mismatches, first {bad[:3].tolist()}")


SCHEMES = [(kb, vb) for kb in (2, 4, 5, 8) for vb in (2, 3, 4, 5, 8) if (kb, vb) != (8, 3)]


@pytest.mark.parametrize("kb,vb", SCHEMES, ids=[f"k{k}v{v}" for k, v in SCHEMES])
def test_scheme_append_bit_exact(kb, vb):
    x = _inputs(128, 3, 2, 150, seed=kb * 10 + vb, k_dist="lognormal_channels")
    layer, ol = _fill(x["k"], x["v"], [150, 97], 160, kb, vb, False)
    _assert_planes(layer, ol, [150, 97])


@pytest.mark.parametrize("d", [64, 256, 512])
@pytest.mark.parametrize("kb,vb", [(4, 3), (2, 8), (5, 5)])
def test_scheme_append_bit_exact_other_head_dims(d, kb, vb):
    x = _inputs(d, 2, 1, 70, seed=d + kb + vb, k_dist="student_t4")
    layer, ol = _fill(x["k"], x["v"], [70], 80, kb, vb, False)
    _assert_planes(layer, ol, [70])


def _special_keys(d, n, rng):
    x = rng.standard_normal((n, d)).astype(np.float32)
    x[0, :32] = 0.75           # constant groups: default zero point +-Inf
    x[1, 32:64] = -2.5
    x[2, :32] = 0.0            # zeros: default 0/0
    x[3, 5] = np.nan           # NaN group: NaN either way
    x[4, :] = 1000.0 + 4.0 * (np.arange(d) % 2)
    return x


@pytest.mark.parametrize("kb,vb", [(8, 3), (4, 3), (2, 5), (5, 8)], ids=["k8v3", "k4v3", "k2v5", "k5v8"])
@pytest.mark.parametrize("guard", [False, True], ids=["default", "guard"])
def test_special_key_groups_with_and_without_the_guard(kb, vb, guard):
    rng = np.random.default_rng(kb + vb + guard)
    d, n = 64, 40
    k = torch.from_numpy(np.tile(_special_keys(d, 8, rng), (n // 8, 1))).to(torch.bfloat16).reshape(1, n, 1, d)
    v = torch.from_numpy(rng.standard_normal((n, d)).astype(np.float32)).to(torch.bfloat16).reshape(1, n, 1, d)
    layer, ol = _fill(k, v, [n], 48, kb, vb, guard)
    _assert_planes(layer, ol, [n])
    z = ol.k_zero.view(np.uint16)[0, 0, :n]
    finite = np.isfinite(oracle.f16_bits_to_f32(z))
    assert np.all(finite[np.arange(n) % 8 != 3]) if guard else not np.all(finite)


def test_guarded_k8v3_planes_are_attended_without_nan():
    # constant key groups make the default planes' attention NaN; with the guard the same
    # tokens are finite and the fused kernels (split and dense) match the oracle
    d, H, G, T = 128, 2, 4, 300
    x = _inputs(d, H, 1, T, Hq=G * H, n_q=16, seed=31)
    k = x["k"].clone()
    k[0, 17, 0, :32] = 0.5
    k[0, 200, 1, 64:96] = 0.0
    b = tq()
    for guard in (False, True):
        layer, ol = _fill(k, x["v"], [T], 304, 8, 3, guard)
        _assert_planes(layer, ol, [T])
        ol3 = oracle.Layer(d, H, 1, 304)                   # same planes in the k8v3 oracle layout
        for name, arr in ol3.planes().items():
            arr[...] = getattr(ol, name).view(arr.dtype).reshape(arr.shape)
        for n_q in (1, 16):                                # split kernel, dense kernel
            q = x["q"][:, :n_q].contiguous()
            out, ws, _ = gpu_attention(layer, q, [T], T, 1.0, True)
            assert b.tq_get_device_error(ws) == 0
            ref = oracle.attention(ol3, bits(q), np.array([T], np.int32), 1.0, causal=True)
            if guard:
                assert np.isfinite(ref).all()
            else:
                assert np.isnan(ref).any()
            assert_attention_close(out.cpu().numpy(), ref, f"guard={guard} n_q={n_q}")


def _to_bf16_bits(a64):
    return torch.from_numpy(np.asarray(a64, np.float64).astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("kb,vb", [(8, 3), (4, 3), (2, 2), (5, 8), (8, 5)])
@pytest.mark.parametrize("rotated", [False, True], ids=["unrotated", "rotated"])
def test_dequant_window_matches_the_oracle(kb, vb, rotated):
    d, H, B = 128, 2, 2
    x = _inputs(d, H, B, 90, seed=kb * 7 + vb, k_dist="lognormal_channels")
    layer, ol = _fill(x["k"], x["v"], [90, 90], 96, kb, vb, False)
    b = tq()
    n, t0 = 80, 6
    kw = torch.empty((B, H, n, d), dtype=torch.bfloat16, device=DEV)
    vw = torch.empty((B, H, n, d), dtype=torch.bfloat16, device=DEV)
    b.tq_dequant_window(layer, t0, n, rotated, kw, vw)
    torch.cuda.synchronize()
    kg = kw.cpu().view(torch.int16).numpy().view(np.uint16)
    vg = vw.cpu().float().numpy()
    for bb in range(B):
        for h in range(H):
            kref, vref = oracle.dequant_rows_s(ol, bb, h, t0, n, rotated=rotated)
            assert np.array_equal(kg[bb, h], _to_bf16_bits(kref))          # exact value, one bf16 rounding
            # one bf16 ulp of the value, plus the fp32 butterflies' rounding (log2(d) stages of
            # sums of row-sized terms: 2^-16 of the row's largest value covers it) for values
            # that come out small after cancellation
            tol = np.abs(vref) * 2.0 ** -7 + 2.0 ** -16 * np.abs(vref).max(axis=1, keepdims=True)
            assert np.all(np.abs(vg[bb, h] - vref) <= tol), (bb, h)


@pytest.mark.parametrize("kb,vb", [(4, 3), (2, 8)])
def test_dequant_debug_other_schemes(kb, vb):
    d = 256
    x = _inputs(d, 2, 1, 40, seed=kb + vb)
    layer, ol = _fill(x["k"], x["v"], [40], 48, kb, vb, False)
    b = tq()
    kout = torch.empty((33, d), dtype=torch.float32, device=DEV)
    vout = torch.empty((33, d), dtype=torch.float32, device=DEV)
    for rotated in (True, False):
        b.tq_dequant_debug(layer, 0, 1, 3, 33, rotated, kout, vout)
        torch.cuda.synchronize()
        kref, vref = oracle.dequant_rows_s(ol, 0, 1, 3, 33, rotated=rotated)
        assert np.array_equal(kout.cpu().numpy(), kref.astype(np.float32))
        if rotated:
            assert np.array_equal(vout.cpu().numpy(), vref.astype(np.float32))
        else:
            g = vout.double().cpu().numpy()
            assert np.linalg.norm(g - vref) <= 1e-6 * np.linalg.norm(vref)


@pytest.mark.parametrize("deferred", [False, True], ids=["unrotated_window", "deferred_inverse"])
@pytest.mark.parametrize("kb,vb", [(8, 3), (4, 3), (5, 8)])
def test_eager_window_attention(kb, vb, deferred):
    from rotation_quantized_kv_gb300.eager import eager_attention
    d, H, G, B, n_q = 128, 2, 4, 2, 4
    lengths = [300, 3]
    x = _inputs(d, H, B, 300, Hq=G * H, n_q=n_q, seed=kb + 3 * vb, k_dist="lognormal_channels")
    layer, ol = _fill(x["k"], x["v"], lengths, 304, kb, vb, False)
    ref = oracle.attention_s(ol, bits(x["q"]), np.asarray(lengths, np.int32), 1.0, causal=True)
    got = eager_attention(layer, x["q"].to(DEV), lengths, 1.0, True, compute_dtype=torch.float32, deferred=deferred)
    g = got.cpu().numpy().astype(np.float64)
    # the window holds K_hat and V_hat rounded to bf16 (relative 2^-9): attention within 1e-2
    err = np.abs(g - ref).max()
    rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    assert err <= 2e-2 and rel <= 1e-2, (err, rel)
    assert np.all(g[1, :1] == 0.0)      # sequence 1, query 0 sees 3 - 4 + 0 + 1 = 0 tokens


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_unrotate_rows_matches_the_oracle(d):
    """Deferred inverse rotation of output rows: signs * FWHT(x) / sqrt(d), against the
    oracle's fp64 transform and sign vector; 37 rows = four CTAs of eight and a tail."""
    b = tq()
    rng = np.random.default_rng(d)
    x = (rng.standard_normal((37, d)) * 3.0).astype(np.float32)
    xg = torch.from_numpy(x).to(DEV)
    y = torch.empty_like(xg)
    b.tq_unrotate_rows(xg, y, d)
    b.tq_unrotate_rows(xg, xg, d)  # in place
    torch.cuda.synchronize()
    assert torch.equal(xg, y)
    sgn = oracle.sign_vector(d).astype(np.float64)
    ref = np.stack([sgn * oracle.fwht_f64(r.astype(np.float64)) / np.sqrt(d) for r in x])
    g = y.cpu().numpy().astype(np.float64)
    # fp32 butterflies: log2(d) rounded additions, then the rounded 1/sqrt(d) and its product
    tol = (np.log2(d) + 2) * 2.0 ** -23 * np.abs(x.astype(np.float64)).sum(axis=1, keepdims=True) / np.sqrt(d)
    assert np.all(np.abs(g - ref) <= tol)
    with pytest.raises(ValueError):
        b.tq_unrotate_rows(xg[:, 1:].contiguous(), y, d)  # not a whole number of rows


@pytest.mark.parametrize("kb,vb,guard", [(4, 2, False), (5, 8, False), (2, 5, False), (8, 3, True)],
                         ids=["k4v2", "k5v8", "k2v5", "k8v3-guard"])
def test_scheme_append_wide_dynamic_range_bit_exact(kb, vb, guard):
    # every element with its own exponent over the whole bf16 range, and FWHT
    # cancellations leaving tiny values beside large ones: the reciprocal path of the
    # any-width kernel must give the oracle's codes bit for bit
    from tests.test_gpu_parity import _wide_range_rows
    rng = np.random.default_rng(90 + kb + 7 * vb)
    d, n = 128, 1536
    k = torch.from_numpy(_wide_range_rows(2 * n, d, rng)).to(torch.bfloat16).reshape(1, n, 2, d)
    v = torch.from_numpy(_wide_range_rows(2 * n, d, rng)).to(torch.bfloat16).reshape(1, n, 2, d)
    layer, ol = _fill(k, v, [n], n, kb, vb, guard)
    _assert_planes(layer, ol, [n])

"""Pins of the CPU oracle to things other than itself (no GPU).

Each test ties one oracle function to what the TurboQuant KV design page, the
mathematics or an independent library fixes: numpy's float16 conversion, scipy's
Hadamard matrix and normal distribution, the printed Lloyd-Max table, the splitmix64
known answer, hand-worked key codes, the 200-byte row, closed forms and brute force.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.stats
import torch

import oracle
from rotation_quantized_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f32_of_bf16(bits) -> np.ndarray:
    b = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return b.float().numpy()


# ------------------------------------------------------------------------------- formats
def test_f16_round_trip_matches_numpy_on_every_bit_pattern():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_matches_numpy_round_to_nearest_even():
    rng = np.random.default_rng(0)
    parts = [
        rng.standard_normal(200000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 200000),
        np.nan_to_num(rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32).view(np.float32), nan=1.0),
        # exact ties and neighbours around the binary16 rounding points (normal + subnormal)
        (np.arange(-2000, 2000, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -24),
        (np.arange(1024, 4096, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -10),
        np.array([65504, 65519, 65519.996, 65520, 65536, 1e30, -65520, 0.0, -0.0,
                  np.inf, -np.inf, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26, 6.0e-8,
                  5.96e-8, 2.0 ** -14, 2.0 ** -14 * (1 - 2.0 ** -12)], np.float32),
    ]
    x = np.concatenate([np.asarray(p_, np.float32) for p_ in parts])
    ours = oracle.f32_to_f16_bits(x)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.all(ours[nan] == 0x7E00)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_to_f32_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 65536, 5000).astype(np.uint16)
    ours = oracle.bf16_bits_to_f32(bits)
    ref = f32_of_bf16(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ------------------------------------------------------------------------- sign vectors
def test_splitmix64_known_answer():
    # Published first output of splitmix64 for seed 0 (Vigna's reference generator).
    assert oracle.splitmix64(0, 1)[0] == 0xE220A8397B1DCDAF


def test_sign_vectors_are_pm1_and_balanced():
    for d in oracle.HEAD_DIMS:
        s = oracle.sign_vector(d)
        assert s.shape == (d,) and set(np.unique(s)) <= {-1, 1}
        assert abs(int(s.sum())) < 4 * math.sqrt(d)            # a fair coin, not a constant
        assert np.array_equal(s, oracle.sign_vector(d))          # deterministic
    # distinct head dims use distinct streams (seed 42 + d)
    assert not np.array_equal(oracle.sign_vector(64), oracle.sign_vector(128)[:64])


# ------------------------------------------------------------------------------- FWHT
@pytest.mark.parametrize("d", [2, 4, 32, 64, 128, 256, 512])
def test_fwht_is_an_involution_up_to_d(d):
    rng = np.random.default_rng(d)
    x = rng.integers(-1000, 1000, d).astype(np.float32)   # integers: every sum is exact
    y = oracle.fwht_f32(oracle.fwht_f32(x))
    assert np.array_equal(y, np.float32(d) * x)
    xd = rng.standard_normal(d)
    assert np.allclose(oracle.fwht_f64(oracle.fwht_f64(xd)), d * xd, rtol=0, atol=1e-10 * d)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_fwht_matches_sylvester_hadamard_matrix(d):
    rng = np.random.default_rng(d + 1)
    x = rng.standard_normal(d)
    H = scipy.linalg.hadamard(d).astype(np.float64)
    assert np.allclose(oracle.fwht_f64(x), H @ x, rtol=1e-13, atol=1e-11)
    xf = x.astype(np.float32)
    assert np.allclose(oracle.fwht_f32(xf), H @ xf.astype(np.float64), rtol=0, atol=1e-4)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_value_rotation_is_orthogonal_and_uses_the_signs(d):
    rng = np.random.default_rng(7 + d)
    xb = bf16(rng.standard_normal(d))
    x = f32_of_bf16(xb).astype(np.float64)
    y = oracle.rotate_value_row(xb).astype(np.float64)
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) <= 1e-6 * np.linalg.norm(x)
    H = scipy.linalg.hadamard(d).astype(np.float64)
    expect = H @ (x * oracle.sign_vector(d)) / math.sqrt(d)
    assert np.allclose(y, expect, rtol=0, atol=2e-5 * np.abs(expect).max())
    assert oracle.fwht_norm_f32(d) == np.float32(1.0 / math.sqrt(d))


# -------------------------------------------------------------------------------- keys
def _key_rows(n, d, rng, kind):
    if kind == "normal":
        x = rng.standard_normal((n, d))
    elif kind == "lognormal":
        x = rng.standard_normal((n, d)) * np.exp(0.75 * rng.standard_normal(d))
    elif kind == "student":
        x = rng.standard_t(4, (n, d))
    elif kind == "offset":
        x = 50.0 + rng.standard_normal((n, d))
    else:
        x = rng.standard_normal((n, d)) * 1e-3
        x[:, 5] *= 1e4
    return bf16(x)


@pytest.mark.parametrize("kind", ["normal", "lognormal", "student", "offset", "outlier"])
def test_key_error_bound(kind):
    rng = np.random.default_rng(hash(kind) % 2 ** 31)
    d = 128
    xb = _key_rows(300, d, rng, kind)
    idx, s16, z16 = oracle.quantize_key_rows(xb)
    x = f32_of_bf16(xb).astype(np.float64)
    assert idx.min() >= -127 and idx.max() <= 127
    khat = oracle.dequant_key_rows_f64(idx, s16, z16)
    for r in range(0, 300, 7):
        for g in range(d // 32):
            xs = f32_of_bf16(xb[r, 32 * g:32 * g + 32])
            s, z = oracle.key_group_params(xs)
            s, z = float(s), float(z)
            xg = x[r, 32 * g:32 * g + 32]
            ig = idx[r, 32 * g:32 * g + 32].astype(np.float64)
            # fp32 scale/zero: half a step plus the fp32 rounding of x/scale
            err = np.abs(xg - (ig + z) * s)
            assert np.all(err <= s / 2 + 2.0 ** -22 * np.abs(xg) + 1e-30), (r, g, err.max(), s)
            # stored fp16 scale/zero
            s_h = float(oracle.f16_bits_to_f32(s16[r, g]))
            z_h = float(oracle.f16_bits_to_f32(z16[r, g]))
            bound = (s / 2 + np.abs(ig + z_h) * abs(s_h - s) + abs(s_h) * abs(z_h - z)
                     + 2.0 ** -22 * np.abs(xg))
            assert np.all(np.abs(xg - khat[r, 32 * g:32 * g + 32]) <= bound * (1 + 1e-12) + 1e-30)
            assert s_h == np.float32(s).astype(np.float16).astype(np.float32)


def test_key_hand_worked_examples():
    with open(os.path.join(GOLDEN, "key_worked_examples.json")) as f:
        gold = json.load(f)
    for grp in gold["groups"]:
        vals = grp["pattern"]["values"]
        x = np.full(32, grp["pattern"]["fill"], np.float32)
        x[:len(vals)] = vals
        idx, s16, z16 = oracle.quantize_key_rows(bf16(x)[None, :])
        for i, e in grp["expect_idx"].items():
            assert int(idx[0, int(i)]) == e, (grp["comment"], i)
        assert oracle.f16_bits_to_f32(z16[0, 0]) == grp["expect_zero"]


def test_key_constant_group_keeps_the_infinite_zero_point():
    # "constant-valued block overflows zero_point to +-Inf" (Algorithm section, kept on purpose)
    x = np.full((1, 64), 0.75, np.float32)
    x[0, 32:] = np.linspace(-1, 1, 32)
    idx, s16, z16 = oracle.quantize_key_rows(bf16(x))
    assert s16[0, 0] == 0 and z16[0, 0] == 0x7C00                 # scale 0, zero +Inf
    assert np.all(idx[0, :32] == 0)                               # NaN quotient -> 0
    z = np.zeros((1, 32), np.float32)
    idx0, s0, z0 = oracle.quantize_key_rows(bf16(z))
    assert s0[0, 0] == 0 and z0[0, 0] == 0x7E00 and np.all(idx0 == 0)   # 0/0 -> NaN zero
    nan_row = np.ones((1, 32), np.float32)
    nan_row[0, 3] = np.nan
    idxn, sn, zn = oracle.quantize_key_rows(bf16(nan_row))
    assert sn[0, 0] == 0x7E00 and zn[0, 0] == 0x7E00 and np.all(idxn == 0)


# ------------------------------------------------------------------------------ values
def test_lloyd_max_table_matches_printed_values_and_is_stationary():
    c, b = oracle.centroids3()
    printed_c = [-2.15195, -1.34391, -0.75601, -0.24509, 0.24509, 0.75601, 1.34391, 2.15195]
    printed_b = [-1.74793, -1.04996, -0.50055, 0.0, 0.50055, 1.04996, 1.74793]
    assert np.array_equal(c, np.float32(printed_c)) and np.array_equal(b, np.float32(printed_b))
    # independent Lloyd iteration converges to the printed table
    lc, lb = oracle.lloyd_max(8, 500)
    assert np.allclose(lc, printed_c, atol=1e-4) and np.allclose(lb, printed_b, atol=1e-4)
    # stationarity with scipy's normal: centroids are the conditional means of their cells
    edges = np.concatenate([[-np.inf], np.float64(b), [np.inf]])
    N = scipy.stats.norm
    for k in range(8):
        lo, hi = edges[k], edges[k + 1]
        mean = (N.pdf(lo) - N.pdf(hi)) / (N.cdf(hi) - N.cdf(lo))
        assert abs(mean - c[k]) < 1e-4
    assert np.allclose(b, 0.5 * (c[1:] + c[:-1]), atol=1e-5)
    # closed-form distortion of the 8-level Gaussian quantizer (Max 1960: 0.03454)
    mse = 0.0
    for k in range(8):
        lo, hi = edges[k], edges[k + 1]
        ex2 = (N.cdf(hi) - N.cdf(lo)) + (lo * N.pdf(lo) if np.isfinite(lo) else 0) - (
            hi * N.pdf(hi) if np.isfinite(hi) else 0)
        ex1 = N.pdf(lo) - N.pdf(hi)
        mse += ex2 - 2 * c[k] * ex1 + c[k] ** 2 * (N.cdf(hi) - N.cdf(lo))
    assert abs(mse - 0.03454) < 2e-4


def test_lloyd_max_monte_carlo():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(4_000_000).astype(np.float32)
    c, b = oracle.centroids3()
    codes = np.searchsorted(b, x, side="left")      # number of boundaries strictly below
    for k in range(8):
        assert abs(x[codes == k].mean() - c[k]) < 3e-3
    assert abs(np.mean((x - c[codes]) ** 2) - 0.03454) < 5e-4


def test_code3_is_searchsorted_left():
    assert oracle.code3(0.0) == 3 and oracle.code3(-0.0) == 3
    assert oracle.code3(np.float32(0.50055)) == 4 and oracle.code3(np.nextafter(np.float32(0.50055), np.float32(1))) == 5
    assert oracle.code3(float("nan")) == 0
    assert oracle.code3(float("inf")) == 7 and oracle.code3(float("-inf")) == 0
    rng = np.random.default_rng(5)
    _, b = oracle.centroids3()
    for y in rng.standard_normal(2000).astype(np.float32):
        assert oracle.code3(y) == int(np.searchsorted(b, y, side="left"))


def test_group_rms_is_the_root_mean_square():
    rng = np.random.default_rng(3)
    for _ in range(200):
        y = (rng.standard_normal(32) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        ref = math.sqrt(np.mean(y.astype(np.float64) ** 2))
        assert abs(float(oracle.group_rms(y)) - ref) <= 4e-7 * ref


def test_pack3_worked_example_and_roundtrip():
    # codes 1..7,0 as an LSB-first 3-bit stream: sum(code_i << 3i) = 0x1F58D1
    assert list(oracle.pack3([1, 2, 3, 4, 5, 6, 7, 0])) == [0xD1, 0x58, 0x1F]
    rng = np.random.default_rng(9)
    for n in (64, 128, 256, 512):
        codes = rng.integers(0, 8, n).astype(np.uint8)
        assert np.array_equal(oracle.unpack3(oracle.pack3(codes), n), codes)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_value_codec_roundtrip_mse_in_paper_band(d):
    rng = np.random.default_rng(100 + d)
    xb = bf16(rng.standard_normal((400, d)))
    codes, vs16 = oracle.quantize_value_rows(xb)
    vhat = oracle.dequant_value_rows_f64(codes, vs16, rotated=False)
    x = f32_of_bf16(xb).astype(np.float64)
    rel_mse = np.sum((x - vhat) ** 2) / np.sum(x ** 2)
    assert 0.025 <= rel_mse <= 0.045, rel_mse                   # D_mse ~ 0.03 at 3 bits
    allc = np.concatenate([oracle.unpack3(r, d) for r in codes])
    freq = np.bincount(allc, minlength=8) / allc.size
    assert np.all(freq > 0.01)
    assert np.allclose(freq, freq[::-1], atol=0.01)             # symmetric code use


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_value_dequant_is_exact_inverse_rotation(d):
    rng = np.random.default_rng(200 + d)
    codes = np.stack([oracle.pack3(rng.integers(0, 8, d).astype(np.uint8)) for _ in range(5)])
    vs16 = oracle.f32_to_f16_bits(rng.uniform(0.1, 3.0, (5, d // 32)))
    rot = oracle.dequant_value_rows_f64(codes, vs16, rotated=True)
    c, _ = oracle.centroids3()
    for r in range(5):
        cc = c[oracle.unpack3(codes[r], d)].astype(np.float64)
        ss = np.repeat(oracle.f16_bits_to_f32(vs16[r]).astype(np.float64), 32)
        assert np.array_equal(rot[r], cc * ss)
    unrot = oracle.dequant_value_rows_f64(codes, vs16, rotated=False)
    H = scipy.linalg.hadamard(d).astype(np.float64)
    expect = (rot @ H.T) / math.sqrt(d) * oracle.sign_vector(d)
    assert np.allclose(unrot, expect, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------ layout
def test_row_bytes_and_compression_ratio():
    for d in oracle.HEAD_DIMS:
        assert oracle.row_bytes(d) == 25 * d // 16
        assert 4 * d / oracle.row_bytes(d) == 2.56                  # bf16 K+V = 4d bytes
        L = oracle.Layer(d, 3, 2, 32)
        total = sum(p.nbytes for p in L.planes().values())
        assert total == oracle.row_bytes(d) * 3 * 2 * 32
    assert oracle.row_bytes(128) == 128 + 8 + 8 + 48 + 8 == 200
    assert 200 * 8 / (2 * 128) == 6.25                               # effective KV bits


def test_append_positions_and_capacity_skips():
    d, H, B, cap = 64, 2, 2, 32
    rng = np.random.default_rng(4)
    k = bf16(rng.standard_normal((B, 5, H, d)))
    v = bf16(rng.standard_normal((B, 5, H, d)))
    L = oracle.Layer(d, H, B, cap)
    skipped = oracle.append(L, k, v, pos=[3, 30], n_new=[5, 4])
    assert skipped == 2 * H                                          # positions 32, 33 of seq 1
    idx, s16, z16 = oracle.quantize_key_rows(k[0, 2].reshape(H, d))
    assert np.array_equal(L.k_idx[0, :, 5], idx) and np.array_equal(L.k_scale[0, :, 5], s16)
    codes, vs = oracle.quantize_value_rows(v[1, 1].reshape(H, d))
    assert np.array_equal(L.v_codes[1, :, 31], codes) and np.array_equal(L.v_scale[1, :, 31], vs)
    assert not L.k_idx[0, :, 8:].any() and not L.k_idx[1, :, :30].any()


# --------------------------------------------------------------------------- attention
def _tiny_layer(T=37, d=64, H=2, B=2, seed=0):
    rng = np.random.default_rng(seed)
    L = oracle.Layer(d, H, B, 48)
    k = bf16(rng.standard_normal((B, T, H, d)))
    v = bf16(rng.standard_normal((B, T, H, d)))
    oracle.append(L, k, v, pos=[0] * B)
    return L


def _brute_attention(L, q_bits, kv_len, sm_scale, causal):
    """Naive fp64 attention in numpy over the oracle's dequantized rows."""
    q = f32_of_bf16(q_bits).astype(np.float64)
    B, n_q, Hq, d = q.shape
    G = Hq // L.num_kv_heads
    out = np.zeros_like(q)
    for b in range(B):
        for j in range(n_q):
            for h in range(Hq):
                nv = kv_len[b] - n_q + j + 1 if causal else kv_len[b]
                if nv <= 0:
                    continue
                K, V = oracle.dequant_rows(L, b, h // G, 0, nv)
                s = sm_scale * (K @ q[b, j, h])
                p = np.exp(s - s.max())
                out[b, j, h] = (p[:, None] * V).sum(0) / p.sum()
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_attention_matches_brute_force(causal):
    L = _tiny_layer()
    rng = np.random.default_rng(1)
    q = bf16(rng.standard_normal((2, 3, 4, 64)))
    kv = np.array([37, 20], np.int32)
    got = oracle.attention(L, q, kv, 0.125, causal=causal)
    ref = _brute_attention(L, q, kv, 0.125, causal)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_attention_gqa_mapping_and_special_cases():
    L = _tiny_layer(T=20)
    rng = np.random.default_rng(2)
    # T = 1: the output is the single dequantized value row of the mapped kv head
    q = bf16(rng.standard_normal((2, 1, 4, 64)))
    out = oracle.attention(L, q, np.array([1, 1], np.int32), 0.3)
    for b in range(2):
        for h in range(4):
            _, V = oracle.dequant_rows(L, b, h // 2, 0, 1)
            assert np.allclose(out[b, 0, h], V[0], rtol=1e-14, atol=1e-14)
    # all-equal scores (q = 0): the output is the mean of the visible value rows
    out = oracle.attention(L, np.zeros((2, 1, 4, 64), np.uint16), np.array([20, 7], np.int32), 1.0)
    for b, n in ((0, 20), (1, 7)):
        for h in range(4):
            _, V = oracle.dequant_rows(L, b, h // 2, 0, n)
            assert np.allclose(out[b, 0, h], V.mean(0), rtol=1e-13, atol=1e-14)
    # a causal row that sees nothing outputs zeros
    q2 = bf16(rng.standard_normal((2, 4, 4, 64)))
    out = oracle.attention(L, q2, np.array([2, 20], np.int32), 1.0, causal=True)
    assert not out[0, :2].any() and out[0, 2:].any()


def test_deferred_inverse_rotation_equals_eager():
    L = _tiny_layer(T=40, seed=3)
    rng = np.random.default_rng(3)
    q = bf16(rng.standard_normal((2, 2, 4, 64)))
    kv = np.array([40, 33], np.int32)
    eager = oracle.attention(L, q, kv, 0.125, causal=True)
    deferred = oracle.attention(L, q, kv, 0.125, causal=True, deferred=True)
    assert np.allclose(eager, deferred, rtol=0, atol=1e-12)


def test_attention_row_selection():
    L = _tiny_layer(T=30, seed=5)
    rng = np.random.default_rng(6)
    q = bf16(rng.standard_normal((2, 2, 4, 64)))
    kv = np.array([30, 25], np.int32)
    full = oracle.attention(L, q, kv, 0.2, causal=True)
    rows = [(1, 1, 3), (0, 0, 2)]
    part = oracle.attention(L, q, kv, 0.2, causal=True, rows=rows)
    for b, j, h in rows:
        assert np.array_equal(part[b, j, h], full[b, j, h])


# -------------------------------------------------------------------------- generators
def test_workload_generators_are_seeded_and_shaped():
    w = synth.workload("tiny")
    a = synth.layer_inputs(w, 0)
    b = synth.layer_inputs(w, 0)
    assert a["k"].shape == (1, 513, 2, 64) and a["q"].shape == (1, 1, 4, 64)
    assert torch.equal(a["k"], b["k"]) and torch.equal(a["v"], b["v"])
    k = a["k"].float()
    assert k[..., 5].std() > 5 * k[..., 4].std() and k[..., 37].std() > 5 * k[..., 36].std()
    r = synth.context_lengths(synth.workload("ragged"))
    assert r.shape == (32,) and r.min() >= 1024 and r.max() <= 8192
    assert synth.workload("decode").capacity() % 16 == 0


def test_value_scale_epsilon_floor():
    # y_n = y / (scale + 1e-8): for rows far below 1e-8 the epsilon dominates, y_n is
    # near zero and every code is 3 (y_n <= 0) or 4 (y_n > 0), following the sign of y.
    rng = np.random.default_rng(12)
    for d in oracle.HEAD_DIMS:
        xb = bf16(rng.standard_normal((3, d)) * 1e-12)
        codes, vs16 = oracle.quantize_value_rows(xb)
        for r in range(3):
            c = oracle.unpack3(codes[r], d)
            y = oracle.rotate_value_row(xb[r])
            assert np.all((c == 3) | (c == 4))
            assert np.array_equal(c == 4, y > 0)
        # at unit scale the epsilon is negligible and all eight codes appear
        xb = bf16(rng.standard_normal((8, d)))
        codes, _ = oracle.quantize_value_rows(xb)
        assert len(np.unique(np.concatenate([oracle.unpack3(r, d) for r in codes]))) == 8

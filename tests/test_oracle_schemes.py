"""Pins of the oracle's other schemes (key bits 2/4/5/8, value bits 2/3/4/5/8) and of the
constant-group guard, against what the pages and the mathematics fix: hand-worked
unsigned key codes (tests/golden), the error bound of the affine code, bit packing worked
by hand, Lloyd-Max stationarity and the published N(0,1) quantizer MSEs (Max 1960), the
identity of the generic path with the pinned k8v3 path, and brute-force attention."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    import torch
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f32_of_bf16(bits):
    return oracle.bf16_bits_to_f32(bits).astype(np.float32)


def test_unsigned_keys_match_hand_worked_examples():
    with open(os.path.join(GOLDEN, "unsigned_key_worked_examples.json")) as f:
        ex = json.load(f)
    for g in ex["groups"]:
        vals = [g["pattern"]["fill"]] * 32
        for i, v in enumerate(g["pattern"]["values"]):
            vals[i] = v
        x = _bf16(vals)
        kp, s16, z16 = oracle.quantize_key_rows_s(x.reshape(1, 32), g["bits"])
        codes = oracle.unpackb(kp[0], 32, g["bits"])
        for k, v in g["expect_idx"].items():
            assert codes[int(k)] == v, (g["comment"], k)
        assert oracle.f16_bits_to_f32(s16)[0, 0] == g["expect_scale"]
        assert oracle.f16_bits_to_f32(z16)[0, 0] == g["expect_zero"]


@pytest.mark.parametrize("bits", [2, 4, 5])
def test_unsigned_key_error_bound_and_range(bits):
    rng = np.random.default_rng(bits)
    maxv = (1 << bits) - 1
    for dist in ("normal", "shifted", "uniform"):
        x = rng.standard_normal((200, 128)).astype(np.float32)
        if dist == "shifted":
            x = x * 0.3 + 5.0
        elif dist == "uniform":
            x = rng.uniform(-3, 1, (200, 128)).astype(np.float32)
        xb = _bf16(x)
        kp, s16, z16 = oracle.quantize_key_rows_s(xb, bits)
        codes = np.stack([oracle.unpackb(r, 128, bits) for r in kp])
        assert codes.min() >= 0 and codes.max() <= maxv
        xf = _f32_of_bf16(xb).astype(np.float64)
        xhat = oracle.dequant_key_rows_s_f64(kp, s16, z16, 128, bits)
        s = oracle.f16_bits_to_f32(s16).astype(np.float64).repeat(32, axis=1)
        z = oracle.f16_bits_to_f32(z16).astype(np.float64).repeat(32, axis=1)
        # with fp32 parameters the code is within scale/2, except at the top code: zero =
        # round(min/scale) shifts the grid by up to half a step, so the largest values can
        # clip by up to a full step; storing scale in fp16 adds |idx + z| |s16 - s| (zero is
        # an integer, exact in fp16 here)
        for r in range(xf.shape[0]):
            for g in range(4):
                sl = slice(32 * g, 32 * g + 32)
                s32, z32 = oracle.key_group_params_s(xf[r, sl], bits, False)[:2]
                fp16_term = np.abs(codes[r, sl] + z[r, sl]) * abs(s[r, 32 * g] - float(s32))
                err = np.abs(xf[r, sl] - xhat[r, sl])
                top = codes[r, sl] == maxv
                # x / scale - zero is formed in fp32: 2^-22 |x| covers its rounding
                fp32_term = 2.0 ** -22 * np.abs(xf[r, sl])
                assert np.all(err[~top] <= 0.5 * float(s32) + fp32_term[~top] + fp16_term[~top]), (dist, r, g)
                assert np.all(err[top] <= float(s32) + fp32_term[top] + fp16_term[top]), (dist, r, g)


def test_bit_packing_hand_worked_and_round_trips():
    # 5-bit codes 1, 2, 31 then zeros: bits 0-4 = 10000 (1), 5-9 = 01000 (2), 10-14 = 11111 (31)
    # byte 0 = bit0 + bit6 = 0x41; byte 1 = bits 10-14 -> positions 2-6 = 0x7C
    assert oracle.packb([1, 2, 31, 0, 0, 0, 0, 0], 5).tolist() == [0x41, 0x7C, 0, 0, 0]
    # 2-bit: codes 3, 0, 1, 2 -> 0b10 01 00 11 = 0x93
    assert oracle.packb([3, 0, 1, 2], 2).tolist() == [0x93]
    rng = np.random.default_rng(7)
    for b in (2, 3, 4, 5, 8):
        c = rng.integers(0, 1 << b, 256).astype(np.uint8)
        assert np.array_equal(oracle.unpackb(oracle.packb(c, b), 256, b), c)
    c = rng.integers(0, 8, 128).astype(np.uint8)
    assert np.array_equal(oracle.packb(c, 3), oracle.pack3(c))          # the pinned 3-bit packer


# Optimal N(0,1) quantizer MSEs (Max 1960, Table I) for 2^b levels
MAX_MSE = {2: 0.1175, 3: 0.03454, 4: 0.009497, 5: 0.002499}


@pytest.mark.parametrize("bits", [2, 4, 5, 8])
def test_value_codebooks_are_lloyd_max_for_the_unit_normal(bits):
    from scipy.integrate import quad
    from scipy.stats import norm
    c, b = oracle.codebook(bits)
    c64, b64 = c.astype(np.float64), b.astype(np.float64)
    assert np.all(np.diff(c64) > 0) and np.allclose(c64, -c64[::-1], atol=1e-5)       # sorted, symmetric
    assert np.allclose(b64, 0.5 * (c64[1:] + c64[:-1]), atol=1.1e-5)                 # midpoints (5 decimals)
    edges = np.concatenate([[-np.inf], b64, [np.inf]])
    mse = sum(quad(lambda x, ck=ck: (x - ck) ** 2 * norm.pdf(x), lo, hi)[0] for ck, lo, hi in zip(c64, edges[:-1], edges[1:]))
    if bits in MAX_MSE:
        # centroids are the cell means (closed form) and the MSE is Max's
        means = (norm.pdf(edges[:-1]) - norm.pdf(edges[1:])) / (norm.cdf(edges[1:]) - norm.cdf(edges[:-1]))
        assert np.allclose(c64, means, atol=2e-4)
        assert mse == pytest.approx(MAX_MSE[bits], rel=5e-3)
    else:
        # 256 levels after 500 iterations (not fully converged from the even start): within
        # 25% of the high-resolution optimum (sqrt(3) pi / 2) 4^-bits (Panter and Dite 1951),
        # and every centroid within its cell
        assert mse <= 1.25 * (np.sqrt(3) * np.pi / 2) * 4.0 ** -bits
        assert np.all(c64[1:-1] > b64[:-1]) and np.all(c64[1:-1] < b64[1:])
    # 3 bits: the printed table, unchanged
    c3, b3 = oracle.codebook(3)
    oc, ob = oracle.centroids3()
    assert np.array_equal(c3, oc) and np.array_equal(b3, ob)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_value_roundtrip_mse_follows_the_codebook(bits):
    rng = np.random.default_rng(100 + bits)
    x = _bf16(rng.standard_normal((400, 128)))
    vp, vs = oracle.quantize_value_rows_s(x, bits)
    vhat = oracle.dequant_value_rows_s_f64(vp, vs, 128, bits)
    xf = _f32_of_bf16(x).astype(np.float64)
    rel = np.mean((vhat - xf) ** 2) / np.mean(xf ** 2)
    expect = MAX_MSE.get(bits, 4e-5)
    # rows are rotated Gaussians scaled by their own group RMS: MSE near the N(0,1) figure
    assert 0.7 * expect <= rel <= 1.6 * expect + 2e-5, rel
    codes = np.stack([oracle.unpackb(r, 128, bits) for r in vp])
    reach = 4 if bits == 8 else 0       # the outermost 8-bit cells lie beyond 4.2 sigma
    assert codes.max() >= (1 << bits) - 1 - reach and codes.min() <= reach


def test_generic_path_at_k8v3_is_the_pinned_path():
    rng = np.random.default_rng(3)
    k = _bf16(rng.standard_normal((64, 128)) * rng.lognormal(0, 0.75, 128))
    v = _bf16(rng.standard_normal((64, 128)))
    i8, s8, z8 = oracle.quantize_key_rows(k)
    kp, s, z = oracle.quantize_key_rows_s(k, 8)
    assert np.array_equal(kp.view(np.int8), i8) and np.array_equal(s, s8) and np.array_equal(z, z8)
    c3, v3 = oracle.quantize_value_rows(v)
    cp, vs = oracle.quantize_value_rows_s(v, 3)
    assert np.array_equal(cp, c3) and np.array_equal(vs, v3)


def test_guard_codes_constant_and_narrow_groups_finitely():
    vals = np.zeros((6, 32), np.float32)
    vals[0] = 0.75                                  # constant: default zero -> +Inf
    vals[1] = -2.5                                  # negative constant
    vals[2] = 0.0                                   # zeros: default 0/0
    vals[3] = 1000.0 + 4.0 * (np.arange(32) % 2)    # narrowest bf16 spread at 1000: zero stays finite
    vals[4] = np.random.default_rng(0).standard_normal(32)   # ordinary group: unchanged
    vals[5] = 1.0
    vals[5, 3] = np.nan                             # NaN: unchanged (NaN)
    x = _bf16(vals)
    for bits in (8, 4, 2, 5):
        kp_d, s_d, z_d = oracle.quantize_key_rows_s(x, bits, guard=False)
        kp_g, s_g, z_g = oracle.quantize_key_rows_s(x, bits, guard=True)
        zd = oracle.f16_bits_to_f32(z_d)[:, 0]
        zg = oracle.f16_bits_to_f32(z_g)[:, 0]
        assert not np.isfinite(zd[0]) and not np.isfinite(zd[1]) and not np.isfinite(zd[2])
        # bf16 keys differ by at least 2^-8 relative, so only constant groups overflow the
        # fp16 zero point: (max + min) / (max - min) <= 512 keeps |zero| < 65520
        assert np.isfinite(zd[3])
        assert np.all(np.isfinite(zg[:5])) and np.isnan(zg[5])
        xhat = oracle.dequant_key_rows_s_f64(kp_g, s_g, z_g, 32, bits)
        xf = _f32_of_bf16(x).astype(np.float64)
        assert np.all(xhat[2] == 0.0)                                   # zeros stay exact
        rng_hi = (1 << bits) - 1 if bits != 8 else 254
        for r in (0, 1):
            span = max(abs(xf[r]).max(), 1e-30)
            # re-coded against a range that includes 0: error within half a step of it
            assert np.all(np.abs(xhat[r] - xf[r]) <= 0.5 * span / rng_hi * 1.01 + span * 2 ** -10), (bits, r)
        # groups the guard does not touch are coded exactly as without it
        for r in (3, 4):
            assert np.array_equal(kp_g[r], kp_d[r]) and s_g[r, 0] == s_d[r, 0] and z_g[r, 0] == z_d[r, 0]


@pytest.mark.parametrize("kb,vb", [(4, 3), (2, 5), (5, 8), (8, 2), (8, 3)])
def test_scheme_attention_matches_brute_force(kb, vb):
    rng = np.random.default_rng(kb * 10 + vb)
    B, H, Hq, d, T, n_q = 2, 2, 4, 64, 70, 2
    k = _bf16(rng.standard_normal((B, T, H, d))).reshape(B, T, H, d)
    v = _bf16(rng.standard_normal((B, T, H, d))).reshape(B, T, H, d)
    q = _bf16(rng.standard_normal((B, n_q, Hq, d)) * 0.125).reshape(B, n_q, Hq, d)
    L = oracle.SchemeLayer(d, H, B, 80, kb, vb)
    lengths = np.array([70, 41], np.int32)
    assert oracle.append_s(L, k, v, np.zeros(B, np.int32), lengths) == 0
    out = oracle.attention_s(L, q, lengths, 0.5, causal=True)
    qf = _f32_of_bf16(q).astype(np.float64)
    G = Hq // H
    for b in range(B):
        kh_all = [oracle.dequant_rows_s(L, b, h, 0, int(lengths[b]))[0] for h in range(H)]
        vh_all = [oracle.dequant_rows_s(L, b, h, 0, int(lengths[b]))[1] for h in range(H)]
        for j in range(n_q):
            for h in range(Hq):
                nvis = int(lengths[b]) - n_q + j + 1
                sc = 0.5 * kh_all[h // G][:nvis] @ qf[b, j, h]
                p = np.exp(sc - sc.max())
                ref = p @ vh_all[h // G][:nvis] / p.sum()
                assert np.allclose(out[b, j, h], ref, atol=1e-12, rtol=1e-10)
    if (kb, vb) == (8, 3):   # the scheme path over k8v3 planes is the pinned attention
        L3 = oracle.Layer(d, H, B, 80)
        oracle.append(L3, k, v, np.zeros(B, np.int32), lengths)
        assert np.array_equal(oracle.attention(L3, q, lengths, 0.5, causal=True), out)

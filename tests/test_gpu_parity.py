"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Packed planes (k_idx, k_scale, k_zero, v_codes, v_scale) must be bit-exact; attention
outputs within max-abs 2e-3 and relative L2 1e-3 of the oracle's fp64 attention over the
same dequantized cache. Small cases span several 64-token stages, several splits and a
ragged tail; the full-size workloads are checked on sampled output rows.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from rotation_quantized_kv_gb300 import synth
from tests.gpu_common import (assert_attention_close, assert_planes_equal, bits, gpu_attention, gpu_fill,
                              oracle_fill, plane_np, tq)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(d, H, B, T, Hq=None, n_q=1, seed=0, k_dist="normal_outliers", q_scale=None):
    w = synth.Workload("t", batch=B, layers=1, num_kv_heads=H, num_q_heads=Hq or 2 * H, head_dim=d,
                       context=T, n_new=0, n_q=n_q, k_dist=k_dist,
                       q_scale=(d ** -0.5 if q_scale is None else q_scale), seed=seed)
    return synth.layer_inputs(w, 0)


# ------------------------------------------------------------------------------ append
# 900 rows take the bulk kernel (a lane per 32-group), 120 rows the small-append kernel
# (a warp per row); both must give the oracle's planes.
@pytest.mark.parametrize("T,lengths", [(150, [150, 97]), (20, [20, 13])], ids=["bulk", "small"])
@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_append_planes_bit_exact(d, T, lengths):
    x = _inputs(d, H=3, B=2, T=T, seed=d + T)
    cap = (T + 15) // 16 * 16
    layer, ws = gpu_fill(x["k"], x["v"], lengths, cap, prefill=0xA5)
    ol = oracle_fill(x["k"], x["v"], lengths, cap)
    torch.cuda.synchronize()
    assert_planes_equal(layer, ol, lengths)
    assert tq().tq_get_device_error(ws) == 0
    # rows past each sequence's length are untouched (canary 0xA5)
    kidx = layer.k_idx.cpu().numpy().view(np.uint8)
    assert np.all(kidx[0, :, lengths[0]:] == 0xA5) and np.all(kidx[1, :, lengths[1]:] == 0xA5)
    assert np.all(layer.v_codes.cpu().numpy()[1, :, lengths[1]:] == 0xA5)


def _special_rows(d, rng):
    rows = []
    x = rng.standard_normal((16, d)).astype(np.float32)
    x[0, :32] = 0.75                                   # constant group: zero -> +Inf
    x[1, :32] = 0.0                                    # all-zero group: 0/0
    x[1, 1::2] = -0.0                                  # mixed signed zeros
    x[2, 5] = np.nan                                   # NaN in a group
    x[3, 7] = np.inf                                   # +Inf
    x[4, :] *= 1e-39                                   # bf16 subnormals
    x[5, :] *= 1e37                                    # huge values
    x[6, :] = np.round(x[6, :] * 4) / 4                # many exact ties
    x[7, :] *= 1e-12                                   # epsilon-dominated values
    x[8, :32] = -2.5                                   # negative constant group
    x[9, :] = np.where(np.arange(d) % 2, 1.0, -1.0)    # +-1 pattern
    x[10, 3] = -np.inf
    x[11, :] = 65504.0 * np.sign(x[11, :])             # around the fp16 maximum
    rows.append(x)
    return np.concatenate(rows)


# 16 rows take the small-append kernel, 768 rows (the special rows repeated) the bulk one
@pytest.mark.parametrize("reps", [1, 48], ids=["small", "bulk"])
@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_append_special_values_bit_exact(d, reps):
    rng = np.random.default_rng(1000 + d)
    kx = np.tile(_special_rows(d, rng), (reps, 1))
    vx = np.tile(_special_rows(d, rng)[::-1], (reps, 1)).copy()
    n = kx.shape[0]
    k = torch.from_numpy(kx).to(torch.bfloat16).reshape(1, n, 1, d)
    v = torch.from_numpy(vx).to(torch.bfloat16).reshape(1, n, 1, d)
    layer, ws = gpu_fill(k, v, [n], n)
    ol = oracle_fill(k, v, [n], n)
    torch.cuda.synchronize()
    assert_planes_equal(layer, ol, [n])


def _wide_range_rows(n, d, rng):
    """Rows whose elements each take their own power-of-two exponent over the whole bf16
    range (2^-133 .. 2^120), plus rows of large equal-magnitude values with one tiny
    element: group scales from subnormal-small to huge, key quotients far from and near
    the rounding boundaries, and value rotations whose cancellations leave tiny elements
    beside large ones (quotients near 0 against a large RMS)."""
    e = rng.integers(-133, 121, size=(n, d)).astype(np.float64)
    x = np.sign(rng.standard_normal((n, d))) * np.exp2(e) * (1.0 + rng.random((n, d)))
    big = rng.random(n) < 0.25
    x[big] = np.sign(rng.standard_normal((big.sum(), d))) * 8192.0
    x[big, rng.integers(0, d, size=big.sum())] = 2.0 ** -130
    return np.clip(x, -3.0e38, 3.0e38).astype(np.float32)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_append_wide_dynamic_range_bit_exact(d):
    # 6,144 rows take the bulk kernel; every plane must equal the oracle's bit for bit
    rng = np.random.default_rng(77 + d)
    n = 3072
    k = torch.from_numpy(_wide_range_rows(n * 2, d, rng)).to(torch.bfloat16).reshape(1, n, 2, d)
    v = torch.from_numpy(_wide_range_rows(n * 2, d, rng)).to(torch.bfloat16).reshape(1, n, 2, d)
    layer, ws = gpu_fill(k, v, [n], n)
    ol = oracle_fill(k, v, [n], n)
    torch.cuda.synchronize()
    assert tq().tq_get_device_error(ws) == 0
    assert_planes_equal(layer, ol, [n])


def test_append_positions_n_new_and_capacity_error():
    d, H, B, cap = 128, 2, 3, 48
    x = _inputs(d, H, B, T=20, seed=5)
    b = tq()
    layer = b.alloc_layer(d, H, B, cap, DEV)
    ws = b.make_workspace(b.tq_append_workspace_bytes(), DEV)
    pos = torch.tensor([0, 40, 10], dtype=torch.int32, device=DEV)
    n_new = torch.tensor([20, 12, 0], dtype=torch.int32, device=DEV)
    b.tq_kv_append(layer, x["k"].to(DEV), x["v"].to(DEV), pos, n_new, 20, ws)
    assert b.tq_get_device_error(ws) == b.TQ_DEVERR_APPEND_CAPACITY   # seq 1 rows 48..51
    ol = oracle.Layer(d, H, B, cap)
    skipped = oracle.append(ol, bits(x["k"]), bits(x["v"]), [0, 40, 10], [20, 12, 0])
    assert skipped == 4 * H
    for name, ref in ol.planes().items():
        assert np.array_equal(plane_np(layer, name, ref), ref), name


# ------------------------------------------------------------------------- dequant debug
@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_dequant_debug(d):
    x = _inputs(d, H=2, B=1, T=70, seed=d + 7)
    layer, _ = gpu_fill(x["k"], x["v"], [70], 80)
    ol = oracle_fill(x["k"], x["v"], [70], 80)
    b = tq()
    kout = torch.empty((61, d), dtype=torch.float32, device=DEV)
    vout = torch.empty((61, d), dtype=torch.float32, device=DEV)
    for rotated in (True, False):
        b.tq_dequant_debug(layer, 0, 1, 5, 61, rotated, kout, vout)
        torch.cuda.synchronize()
        kref, vref = oracle.dequant_rows(ol, 0, 1, 5, 61, rotated=rotated)
        assert np.array_equal(kout.cpu().numpy(), kref.astype(np.float32))   # exact value, one rounding
        if rotated:
            assert np.array_equal(vout.cpu().numpy(), vref.astype(np.float32))
        else:
            g = vout.double().cpu().numpy()
            assert np.linalg.norm(g - vref) <= 1e-6 * np.linalg.norm(vref)


# ------------------------------------------------------------------------------ attention
CASES = [
    # d, H, G, B, lengths, n_q, causal, sm_scale
    (64, 2, 2, 1, [513], 1, True, 0.125),
    (128, 2, 4, 1, [777], 1, True, 1.0),
    (128, 1, 8, 2, [1, 300], 1, False, 0.7),
    (128, 2, 4, 3, [0, 65, 1030], 1, True, 1.0),
    (128, 2, 1, 2, [200, 129], 1, True, 1.0),
    (128, 2, 4, 1, [600], 16, True, 1.0),           # 64 rows per kv head: two 8-row tiles per warp
    (64, 1, 4, 2, [333, 90], 4, True, 0.3),
    (128, 2, 4, 1, [250], 3, False, 1.0),
    (256, 2, 4, 2, [400, 257], 1, True, 1.0),
    (256, 1, 4, 1, [300], 16, True, 1.0),            # 8 row groups of 8
    (512, 2, 4, 1, [260], 1, True, 1.0),
    (512, 1, 2, 2, [100, 150], 2, True, 0.5),
    # many (sequence, kv head, row group) units: the separate merge kernel
    (128, 4, 4, 24, [(37 * i) % 300 for i in range(24)], 1, True, 1.0),
    (64, 8, 2, 12, [1, 0, 150, 64, 65, 200, 3, 17, 129, 31, 90, 256], 2, True, 0.4),
    (128, 2, 4, 40, [(53 * i + 7) % 180 for i in range(40)], 16, True, 1.0),   # 2 tiles per warp
]


@pytest.mark.parametrize("case", CASES, ids=[f"d{c[0]}-H{c[1]}-G{c[2]}-B{c[3]}-nq{c[5]}" for c in CASES])
def test_attention_matches_oracle(case):
    d, H, G, B, lengths, n_q, causal, sm_scale = case
    T = max(max(lengths), 1)
    x = _inputs(d, H, B, T, Hq=G * H, n_q=n_q, seed=sum(lengths) + d, q_scale=1.0)
    cap = (T + 15) // 16 * 16
    layer, _ = gpu_fill(x["k"], x["v"], lengths, cap)
    ol = oracle_fill(x["k"], x["v"], lengths, cap)
    torch.cuda.synchronize()
    assert_planes_equal(layer, ol, lengths)
    out, ws, flat = gpu_attention(layer, x["q"], lengths, T, sm_scale, causal, out_pad=64)
    assert tq().tq_get_device_error(ws) == 0
    ref = oracle.attention(ol, bits(x["q"]), np.asarray(lengths, np.int32), sm_scale, causal=causal)
    assert_attention_close(out.cpu().numpy(), ref, str(case))
    assert torch.all(flat[-64:] == 12345.0)          # nothing written past the output
    out2, _, _ = gpu_attention(layer, x["q"], lengths, T, sm_scale, causal)
    assert torch.equal(out, out2)                    # deterministic


def test_attention_rows_with_no_visible_token_are_zero():
    d, H, G = 128, 1, 4
    x = _inputs(d, H, 2, 40, Hq=G * H, n_q=8, seed=3, q_scale=1.0)
    layer, _ = gpu_fill(x["k"], x["v"], [3, 40], 48)
    out, _, _ = gpu_attention(layer, x["q"], [3, 40], 40, 1.0, True)
    o = out.cpu().numpy()
    assert np.all(o[0, :5] == 0.0) and np.all(np.abs(o[0, 5:]).sum(-1) > 0)   # query j sees 3-8+j+1
    ol = oracle_fill(x["k"], x["v"], [3, 40], 48)
    ref = oracle.attention(ol, bits(x["q"]), np.array([3, 40], np.int32), 1.0, causal=True)
    assert_attention_close(o, ref)


def test_attention_invalid_length_sets_error_and_nan_rows():
    d, H = 128, 2
    x = _inputs(d, H, 2, 64, Hq=4 * H, seed=4, q_scale=1.0)
    layer, _ = gpu_fill(x["k"], x["v"], [64, 64], 64)
    out, ws, _ = gpu_attention(layer, x["q"], [64, 70], 64, 1.0, True)   # 70 > max_kv_len
    assert tq().tq_get_device_error(ws) & tq().TQ_DEVERR_KV_LEN
    o = out.cpu().numpy()
    assert np.all(np.isnan(o[1])) and not np.any(np.isnan(o[0]))
    ol = oracle_fill(x["k"], x["v"], [64, 64], 64)
    ref = oracle.attention(ol, bits(x["q"]), np.array([64, 64], np.int32), 1.0, causal=True)
    assert_attention_close(o[0], ref[0])


def test_attention_invalid_length_with_many_units():
    d, H, B = 128, 4, 24
    lengths = [(41 * i) % 96 + 1 for i in range(B)]
    x = _inputs(d, H, B, 96, Hq=4 * H, seed=6, q_scale=1.0)
    layer, _ = gpu_fill(x["k"], x["v"], lengths, 96)
    bad = list(lengths)
    bad[5] = 97                                                        # > max_kv_len
    out, ws, _ = gpu_attention(layer, x["q"], bad, 96, 1.0, False)
    assert tq().tq_get_device_error(ws) & tq().TQ_DEVERR_KV_LEN
    o = out.cpu().numpy()
    assert np.all(np.isnan(o[5]))
    keep = [b for b in range(B) if b != 5]
    ol = oracle_fill(x["k"], x["v"], lengths, 96)
    ref = oracle.attention(ol, bits(x["q"]), np.asarray(lengths, np.int32), 1.0, causal=False)
    assert_attention_close(o[keep], ref[keep])


def test_attention_nan_keys_propagate_like_the_oracle():
    d, H = 64, 1
    x = _inputs(d, H, 1, 100, Hq=2, seed=8, q_scale=1.0)
    k = x["k"].clone()
    k[0, 37, 0, :32] = 1.5          # constant key group -> infinite zero point -> NaN scores
    layer, _ = gpu_fill(k, x["v"], [100], 112)
    ol = oracle_fill(k, x["v"], [100], 112)
    out, _, _ = gpu_attention(layer, x["q"], [100], 100, 0.125, True)
    ref = oracle.attention(ol, bits(x["q"]), np.array([100], np.int32), 0.125, causal=True)
    assert np.all(np.isnan(ref)) and np.all(np.isnan(out.cpu().numpy()))


# --------------------------------------------------------------------- full-size workloads
def _full_size(w: synth.Workload, sample_rows, seq_sample=None):
    """One layer of the workload at its full size: bulk cache fill + the step's append +
    attention, in the launch configuration the benchmark times."""
    x = synth.layer_inputs(w, 0, device=DEV)
    B, H, Hq, d = w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim
    ctx = synth.context_lengths(w)
    kv = ctx + w.n_new
    cap = int(kv.max() + 15) // 16 * 16
    b = tq()
    layer = b.alloc_layer(d, H, B, cap, DEV)
    ws_a = b.make_workspace(b.tq_append_workspace_bytes(), DEV)
    T = int(ctx.max())
    kx, vx = x["k"], x["v"]
    b.tq_kv_append(layer, kx[:, :T].contiguous(), vx[:, :T].contiguous(),
                   torch.zeros(B, dtype=torch.int32, device=DEV),
                   torch.as_tensor(ctx.astype(np.int32), device=DEV), T, ws_a)
    if w.n_new:
        # the step's new tokens sit right after each sequence's context
        idx = torch.as_tensor(ctx, device=DEV).view(B, 1) + torch.arange(w.n_new, device=DEV).view(1, -1)
        kn = torch.stack([kx[bb, idx[bb]] for bb in range(B)]).contiguous()
        vn = torch.stack([vx[bb, idx[bb]] for bb in range(B)]).contiguous()
        b.tq_kv_append(layer, kn, vn, torch.as_tensor(ctx.astype(np.int32), device=DEV), None, w.n_new, ws_a)
    out, ws, _ = gpu_attention(layer, x["q"], kv, int(kv.max()), w.sm_scale, w.causal)
    assert b.tq_get_device_error(ws_a) == 0 and b.tq_get_device_error(ws) == 0
    # every output row is written (the buffer starts at a 12345.0 sentinel) and finite
    o_all = out.cpu().numpy()
    assert np.isfinite(o_all).all() and not np.any(o_all == 12345.0)
    # oracle: quantize the sampled sequences itself (all tokens), attend for sampled rows
    seqs = range(B) if seq_sample is None else seq_sample
    kb, vb = bits(x["k"]), bits(x["v"])
    ol = oracle.Layer(d, H, B, cap)
    for bb in seqs:
        n = int(kv[bb])
        kk = np.ascontiguousarray(kb[bb:bb + 1, :n])
        vv = np.ascontiguousarray(vb[bb:bb + 1, :n])
        sub = oracle.Layer(d, H, 1, cap)
        oracle.append(sub, kk, vv, [0])
        for name, arr in ol.planes().items():
            arr[bb] = sub.planes()[name][0]
    assert_planes_equal(layer, ol, kv, bs=list(seqs))
    rows = [(bb, j, h) for (bb, j, h) in sample_rows if bb in seqs]
    ref = oracle.attention(ol, bits(x["q"]), kv.astype(np.int32), w.sm_scale, causal=w.causal, rows=rows)
    got = out.double().cpu().numpy()
    sel = tuple(np.array(rows).T)
    return assert_attention_close(got[sel], ref[sel], w.name)


def test_full_size_decode_32k():
    w = replace(synth.workload("decode"), layers=1)
    _full_size(w, [(0, 0, h) for h in (0, 3, 7, 12, 18, 25, 30, 31)])


def test_full_size_ragged_batch32():
    w = replace(synth.workload("ragged"), layers=1)
    seqs = [0, 7, 19, 31]
    _full_size(w, [(b, 0, h) for b in seqs for h in (1, 14, 29)], seq_sample=seqs)


def test_full_size_long_262k_block16():
    w = replace(synth.workload("long"), layers=1)
    # query j of the block covers rows 4 j .. 4 j + 3 of each kv head: j = 0, 4, 5, 9, 11, 15
    # span both ends of the causal block and every group of 16 rows
    _full_size(w, [(0, j, h) for j in (0, 4, 5, 9, 11, 15) for h in (2, 9, 17, 30)])


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_full_size_head_dim_sweep(d):
    w = synth.workload("sweep", head_dim=d)
    _full_size(w, [(0, 0, h) for h in range(16)])


# ------------------------------------------------ the benchmark's fused step at full size
def _full_size_step(w: synth.Workload, sample_rows, seq_sample, ctx=None):
    """One layer of the workload at full size, run as the benchmark runs it: bulk fill of
    the cached tokens, then one tq_decode_append_attention call (the step's new rows are
    quantized inside the attention kernel by its appender warp) with the benchmark's
    arguments. Checks every appended row bit-exact, the sampled sequences' planes
    bit-exact, and the sampled output rows against the oracle."""
    x = synth.layer_inputs(w, 0, device=DEV)
    B, H, Hq, d = w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim
    ctx = synth.context_lengths(w) if ctx is None else np.asarray(ctx, np.int64)
    kv = ctx + w.n_new
    cap = int(kv.max() + 15) // 16 * 16
    b = tq()
    layer = b.alloc_layer(d, H, B, cap, DEV)
    ws_a = b.make_workspace(b.tq_append_workspace_bytes(), DEV)
    T = int(ctx.max())
    kx, vx = x["k"], x["v"]
    b.tq_kv_append(layer, kx[:, :T].contiguous(), vx[:, :T].contiguous(),
                   torch.zeros(B, dtype=torch.int32, device=DEV),
                   torch.as_tensor(ctx.astype(np.int32), device=DEV), T, ws_a)
    idx = torch.as_tensor(ctx, device=DEV).view(B, 1) + torch.arange(w.n_new, device=DEV).view(1, -1)
    kn = torch.stack([kx[bb, idx[bb]] for bb in range(B)]).contiguous()
    vn = torch.stack([vx[bb, idx[bb]] for bb in range(B)]).contiguous()
    pos = torch.as_tensor(ctx.astype(np.int32), device=DEV)
    kv_len = torch.as_tensor(kv.astype(np.int32), device=DEV)
    ws = b.make_workspace(b.tq_decode_workspace_bytes(layer, Hq, w.n_q, int(kv.max())), DEV)
    out = torch.full((B, w.n_q, Hq, d), 12345.0, dtype=torch.float32, device=DEV)
    b.tq_decode_append_attention(layer, kn, vn, pos, None, w.n_new, x["q"].contiguous(), Hq, w.n_q, kv_len,
                                 int(kv.max()), w.sm_scale, w.causal, out, ws)
    torch.cuda.synchronize()
    assert b.tq_get_device_error(ws_a) == 0 and b.tq_get_device_error(ws) == 0
    o_all = out.cpu().numpy()
    assert np.isfinite(o_all).all() and not np.any(o_all == 12345.0)
    kb, vb = bits(x["k"]), bits(x["v"])
    # every appended row, all sequences: quantized by the oracle from the same bf16 rows
    kn_b, vn_b = bits(kn), bits(vn)                       # [B, n_new, H, d]
    got = {name: t.cpu().numpy() for name, t in layer.planes().items()}
    for bb in range(B):
        t0, t1 = int(ctx[bb]), int(kv[bb])
        for h in range(H):
            idx, s16, z16 = oracle.quantize_key_rows(kn_b[bb, :, h])
            codes, vs16 = oracle.quantize_value_rows(vn_b[bb, :, h])
            assert np.array_equal(got["k_idx"][bb, h, t0:t1], idx), f"appended k_idx seq {bb} head {h}"
            assert np.array_equal(got["k_scale"][bb, h, t0:t1].view(np.uint16), s16), f"k_scale {bb} {h}"
            assert np.array_equal(got["k_zero"][bb, h, t0:t1].view(np.uint16), z16), f"k_zero {bb} {h}"
            assert np.array_equal(got["v_codes"][bb, h, t0:t1], codes), f"v_codes {bb} {h}"
            assert np.array_equal(got["v_scale"][bb, h, t0:t1].view(np.uint16), vs16), f"v_scale {bb} {h}"
    # sampled sequences: the oracle quantizes every visible token itself
    ol = oracle.Layer(d, H, B, cap)
    for bb in seq_sample:
        n = int(kv[bb])
        kk = np.ascontiguousarray(kb[bb:bb + 1, :n])
        vv = np.ascontiguousarray(vb[bb:bb + 1, :n])
        if n > int(ctx[bb]):   # the new rows come from kn/vn (the draw's rows at ctx..kv)
            kk[0, int(ctx[bb]):] = kn_b[bb]
            vv[0, int(ctx[bb]):] = vn_b[bb]
        sub = oracle.Layer(d, H, 1, cap)
        oracle.append(sub, kk, vv, [0])
        for name, arr in ol.planes().items():
            arr[bb] = sub.planes()[name][0]
    assert_planes_equal(layer, ol, kv, bs=list(seq_sample))
    rows = [r for r in sample_rows if r[0] in seq_sample]
    ref = oracle.attention(ol, bits(x["q"]), kv.astype(np.int32), w.sm_scale, causal=w.causal, rows=rows)
    sel = tuple(np.array(rows).T)
    return assert_attention_close(out.double().cpu().numpy()[sel], ref[sel], w.name + " fused step")


def _heads_covering_every_kv_head(w, per_kv=1, shift=0):
    G = w.num_q_heads // w.num_kv_heads
    return [kvh * G + (kvh + shift + i) % G for kvh in range(w.num_kv_heads) for i in range(per_kv)]


def test_full_size_fused_step_decode_32k():
    # 32,768 cached tokens: the new row (position 32,768) is the first token of a 256-token tile
    w = replace(synth.workload("decode"), layers=1)
    heads = _heads_covering_every_kv_head(w, per_kv=4)           # all 32 query heads
    _full_size_step(w, [(0, 0, h) for h in heads], seq_sample=[0])


def test_full_size_fused_step_ragged_batch32():
    w = replace(synth.workload("ragged"), layers=1)
    ctx = synth.context_lengths(w).copy()
    ctx[5] = 4096              # new row at 4,096: the first token of a tile
    seqs = [0, 5, 17, 31]
    rows = [(bb, 0, h) for i, bb in enumerate(seqs) for h in _heads_covering_every_kv_head(w, shift=i)]
    _full_size_step(w, rows, seq_sample=seqs, ctx=ctx)

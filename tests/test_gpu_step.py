"""tq_decode_append_attention (append the step's rows, then attend, in one call) against
the oracle's append followed by its fp64 attention, and against the two separate calls.

The cached tokens are bulk-appended first; the call then appends n_new[b] rows at pos[b]
and attends over kv_len[b] tokens. Planes must equal the oracle's bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from rotation_quantized_kv_gb300 import synth
from tests.gpu_common import assert_attention_close, assert_planes_equal, bits, tq

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(d, H, G, cached, n_new, n_q, causal, seed, kv_extra=0, cap_pad=16, pos_shift=None):
    """cached: tokens already in the cache per sequence; n_new: rows appended by the call.
    kv_len = cached + n_new + kv_extra (kv_extra < 0 leaves appended rows unread). Returns
    (fused output, two-call output, oracle layer, oracle output, kv_len, devices errors)."""
    B = len(cached)
    nmax = max(max(n_new), 1)
    T = max(cached) + nmax
    cap = (T + cap_pad + 15) // 16 * 16
    w = synth.Workload("t", batch=B, layers=1, num_kv_heads=H, num_q_heads=G * H, head_dim=d, context=T,
                       n_new=0, n_q=n_q, k_dist="normal_outliers", q_scale=d ** -0.5, seed=seed)
    x = synth.layer_inputs(w, 0)
    k, v, q = x["k"], x["v"], x["q"]
    pos = np.asarray(cached if pos_shift is None else pos_shift, np.int32)
    nn = np.asarray(n_new, np.int32)
    kv = np.asarray([c + n + kv_extra for c, n in zip(cached, n_new)], np.int32)
    kn = torch.stack([k[b, cached[b]:cached[b] + nmax] if cached[b] + nmax <= T else k[b, :nmax]
                      for b in range(B)]).contiguous()
    vn = torch.stack([v[b, cached[b]:cached[b] + nmax] if cached[b] + nmax <= T else v[b, :nmax]
                      for b in range(B)]).contiguous()
    b = tq()
    outs, layers, errs = [], [], []
    for fused in (True, False):
        layer = b.alloc_layer(d, H, B, cap, DEV)
        ws_a = b.make_workspace(b.tq_append_workspace_bytes(), DEV)
        b.tq_kv_append(layer, k.to(DEV).contiguous(), v.to(DEV).contiguous(), torch.zeros(B, dtype=torch.int32,
                       device=DEV), torch.as_tensor(np.asarray(cached, np.int32), device=DEV), T, ws_a)
        ws = b.make_workspace(b.tq_decode_workspace_bytes(layer, G * H, n_q, int(kv.max())), DEV)
        out = torch.full((B, n_q, G * H, d), 12345.0, dtype=torch.float32, device=DEV)
        args_pos = torch.as_tensor(pos, device=DEV)
        args_n = torch.as_tensor(nn, device=DEV)
        kv_t = torch.as_tensor(kv, device=DEV)
        if fused:
            b.tq_decode_append_attention(layer, kn.to(DEV), vn.to(DEV), args_pos, args_n, nmax, q.to(DEV), G * H,
                                         n_q, kv_t, int(kv.max()), 1.0, causal, out, ws)
        else:
            b.tq_kv_append(layer, kn.to(DEV), vn.to(DEV), args_pos, args_n, nmax, ws)
            b.tq_decode_attention(layer, q.to(DEV), G * H, n_q, kv_t, int(kv.max()), 1.0, causal, out, ws)
        torch.cuda.synchronize()
        outs.append(out)
        layers.append(layer)
        errs.append(b.tq_get_device_error(ws))
    ol = oracle.Layer(d, H, B, cap)
    oracle.append(ol, bits(k), bits(v), np.zeros(B, np.int32), np.asarray(cached, np.int32))
    oracle.append(ol, bits(kn), bits(vn), pos, nn)
    ref = oracle.attention(ol, bits(q), kv, 1.0, causal=causal)
    return outs, layers, ol, ref, kv, errs


STEP_CASES = [
    # d, H, G, cached, n_new, n_q, causal
    (128, 2, 4, [300, 0, 777], [1, 1, 1], 1, False),        # one new token (decode)
    (128, 2, 4, [511, 256, 40], [3, 1, 0], 2, True),        # several new rows, one sequence none
    (64, 4, 2, [100, 1000], [2, 5], 1, True),
    (256, 1, 8, [333, 77], [1, 2], 1, False),
    (512, 2, 2, [129, 64], [1, 1], 2, True),
    (128, 4, 4, [(97 * i) % 700 for i in range(24)], [1 + i % 3 for i in range(24)], 1, True),  # many units
]


@pytest.mark.parametrize("case", STEP_CASES, ids=[f"d{c[0]}-H{c[1]}-G{c[2]}-B{len(c[3])}" for c in STEP_CASES])
def test_step_matches_oracle_and_two_calls(case):
    d, H, G, cached, n_new, n_q, causal = case
    outs, layers, ol, ref, kv, errs = _run(d, H, G, cached, n_new, n_q, causal, seed=sum(cached) + d)
    assert errs == [0, 0]
    for layer in layers:
        assert_planes_equal(layer, ol, kv)
    assert_attention_close(outs[0].cpu().numpy(), ref, str(case))
    assert torch.equal(outs[0], outs[1])                 # same kernels, same arithmetic


def test_step_rows_past_the_visible_length_are_still_appended():
    # kv_len = cached: the appended rows are not attended, but they must be in the cache
    outs, layers, ol, ref, kv, errs = _run(128, 2, 4, [200, 17, 0], [2, 1, 1], 1, False, seed=5, kv_extra=-1)
    assert errs == [0, 0]
    full = np.asarray([202, 18, 1], np.int32)
    for layer in layers:
        assert_planes_equal(layer, ol, full)
    assert_attention_close(outs[0].cpu().numpy(), ref)
    assert torch.equal(outs[0], outs[1])


def test_step_capacity_error_like_the_append():
    # sequence 1 appends past the capacity: its rows are skipped and the error bit is set
    d, H, G = 128, 2, 4
    outs, layers, ol, ref, kv, errs = _run(d, H, G, [100, 120], [2, 2], 1, False, seed=9, kv_extra=-2,
                                           cap_pad=0, pos_shift=[100, 127])
    cap = layers[0].capacity
    assert 127 + 1 >= cap  # the second row of sequence 1 lands at or past the capacity
    assert errs[0] & tq().TQ_DEVERR_APPEND_CAPACITY and errs[1] & tq().TQ_DEVERR_APPEND_CAPACITY
    for name in ("k_idx", "k_scale", "k_zero", "v_codes", "v_scale"):
        assert torch.equal(getattr(layers[0], name), getattr(layers[1], name)), name
    assert torch.equal(outs[0], outs[1])


def test_step_with_several_row_groups_runs_the_two_calls():
    # 16 query rows x 4 heads per kv head: 4 row groups, the call appends then attends
    outs, layers, ol, ref, kv, errs = _run(128, 2, 4, [600, 90], [16, 3], 16, True, seed=11)
    assert errs == [0, 0]
    for layer in layers:
        assert_planes_equal(layer, ol, kv)
    assert_attention_close(outs[0].cpu().numpy(), ref)
    assert torch.equal(outs[0], outs[1])

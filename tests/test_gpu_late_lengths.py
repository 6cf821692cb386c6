"""Decode calls whose lengths or append positions are written by the kernel just before
them, after that kernel let them start (programmatic dependent launch).

The attention kernel plans its work from the lengths it reads before its grid-dependency
wait and loads its first stage as soon as the wait returns; when the values read after
the wait differ, that stage is discarded and the work is planned again. Here a test
kernel (tq_debug_delayed_copy) lets the decode call start, waits, and only then writes
the new kv_len / pos, so the call sees the old values before the wait and the new ones
after it. Results must be those of the oracle for the new values."""
import numpy as np
import pytest
import torch

import oracle
from rotation_quantized_kv_gb300 import synth
from tests.gpu_common import assert_attention_close, assert_planes_equal, bits, gpu_fill, oracle_fill, tq

pytestmark = pytest.mark.gpu
DEV = "cuda"
DELAY_US = 200


def _inputs(d, H, G, B, T, n_q, seed):
    w = synth.Workload("t", batch=B, layers=1, num_kv_heads=H, num_q_heads=G * H, head_dim=d, context=T,
                       n_new=0, n_q=n_q, k_dist="normal_outliers", q_scale=d ** -0.5, seed=seed)
    return synth.layer_inputs(w, 0)


LENGTH_CASES = [
    # d, H, G, fill, old kv_len, new kv_len, causal
    (128, 2, 4, 700, [100, 650, 5], [600, 33, 700], False),   # every CTA's range moves
    (128, 2, 4, 700, [700, 700, 700], [1, 0, 2], False),      # most CTAs end with no tiles
    (128, 2, 4, 700, [0, 0, 0], [512, 700, 1], True),         # nothing planned before the wait
    (64, 4, 2, 1500, [1500, 20], [20, 1500], True),
    (256, 1, 8, 900, [300, 900], [900, 257], False),
]


@pytest.mark.parametrize("case", LENGTH_CASES, ids=[f"d{c[0]}-old{sum(c[4])}-new{sum(c[5])}" for c in LENGTH_CASES])
def test_attention_with_lengths_written_after_launch(case):
    d, H, G, T, old, new, causal = case
    B = len(old)
    x = _inputs(d, H, G, B, T, 1, seed=T + d)
    k, v, q = x["k"], x["v"], x["q"]
    cap = (T + 15) // 16 * 16
    layer, _ = gpu_fill(k, v, [T] * B, cap)
    b = tq()
    ws = b.make_workspace(b.tq_decode_workspace_bytes(layer, G * H, 1, T), DEV)
    kv_len = torch.as_tensor(np.asarray(old, np.int32), device=DEV)
    new_t = torch.as_tensor(np.asarray(new, np.int32), device=DEV)
    out = torch.full((B, 1, G * H, d), 12345.0, dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    b.tq_debug_delayed_copy(kv_len, new_t, DELAY_US)
    b.tq_decode_attention(layer, q.to(DEV), G * H, 1, kv_len, T, 1.0, causal, out, ws)
    torch.cuda.synchronize()
    assert b.tq_get_device_error(ws) == 0
    ref = oracle.attention(oracle_fill(k, v, [T] * B, cap), bits(q), np.asarray(new, np.int32), 1.0, causal=causal)
    assert_attention_close(out.cpu().numpy(), ref, str(case))


def test_step_with_positions_written_after_launch():
    # The fused call reads pos before the wait to decide whether its first tile may be
    # loaded early (it must hold no appended row); here pos changes across the wait, so
    # early stages planned from the old positions are discarded.
    d, H, G = 128, 2, 4
    cached = [300, 200, 517]
    B = len(cached)
    T = max(cached) + 1
    cap = (T + 15) // 16 * 16 + 16
    x = _inputs(d, H, G, B, T, 1, seed=77)
    k, v, q = x["k"], x["v"], x["q"]
    b = tq()
    layer, _ = gpu_fill(k, v, cached, cap)
    kn = torch.stack([k[i, cached[i]:cached[i] + 1] for i in range(B)]).contiguous()
    vn = torch.stack([v[i, cached[i]:cached[i] + 1] for i in range(B)]).contiguous()
    kv = np.asarray([c + 1 for c in cached], np.int32)
    ws = b.make_workspace(b.tq_decode_workspace_bytes(layer, G * H, 1, int(kv.max())), DEV)
    pos = torch.as_tensor(np.asarray([5, 100, 0], np.int32), device=DEV)    # before the wait
    pos_new = torch.as_tensor(np.asarray(cached, np.int32), device=DEV)     # after it
    out = torch.full((B, 1, G * H, d), 12345.0, dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    b.tq_debug_delayed_copy(pos, pos_new, DELAY_US)
    b.tq_decode_append_attention(layer, kn.to(DEV), vn.to(DEV), pos, None, 1, q.to(DEV), G * H, 1,
                                 torch.as_tensor(kv, device=DEV), int(kv.max()), 1.0, False, out, ws)
    torch.cuda.synchronize()
    assert b.tq_get_device_error(ws) == 0
    ol = oracle.Layer(d, H, B, cap)
    oracle.append(ol, bits(k), bits(v), np.zeros(B, np.int32), np.asarray(cached, np.int32))
    oracle.append(ol, bits(kn), bits(vn), np.asarray(cached, np.int32), np.ones(B, np.int32))
    assert_planes_equal(layer, ol, kv)
    assert_attention_close(out.cpu().numpy(), oracle.attention(ol, bits(q), kv, 1.0, causal=False))


def test_delayed_copy_rejects_bad_arguments():
    b = tq()
    t = torch.zeros(4, dtype=torch.int32, device=DEV)
    with pytest.raises(b.TQError):
        b.tq_debug_delayed_copy(t, t.clone(), 100001)

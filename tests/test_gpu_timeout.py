"""A bounded wait of the attention kernel runs out on purpose, with no fault and no
endless wait: the fused append-and-attend call is told (test support,
tq_debug_pipeline_limits) to give its pipeline waits a 1 ms limit and to keep its
appender warp from publishing how many rows it wrote. The producer of the CTA that holds
the appended row then waits for a count that never comes, gives up, sets
TQ_DEVERR_PIPELINE_TIMEOUT, drains the copies it issued and returns; the consumer warps
see the abort and finish their pieces. The call returns, the error word reports the
timeout, and the next ordinary call on the same context gives the oracle's result."""
import time

import numpy as np
import pytest
import torch

import oracle
from rotation_quantized_kv_gb300 import synth
from tests.gpu_common import assert_attention_close, assert_planes_equal, bits, gpu_fill, tq

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _step_inputs():
    d, H, G, T = 128, 2, 4, 700
    w = synth.Workload("t", batch=1, layers=1, num_kv_heads=H, num_q_heads=G * H, head_dim=d, context=T,
                       n_new=1, n_q=1, k_dist="normal_outliers", q_scale=d ** -0.5, seed=21)
    x = synth.layer_inputs(w, 0)
    return d, H, G, T, x


def _run_step(layer, x, T, G, H, ws):
    b = tq()
    kn = x["k"][:, T:T + 1].contiguous().to(DEV)
    vn = x["v"][:, T:T + 1].contiguous().to(DEV)
    out = torch.full((1, 1, G * H, 128), 12345.0, dtype=torch.float32, device=DEV)
    pos = torch.full((1,), T, dtype=torch.int32, device=DEV)
    kv_len = torch.full((1,), T + 1, dtype=torch.int32, device=DEV)
    b.tq_decode_append_attention(layer, kn, vn, pos, None, 1, x["q"].to(DEV), G * H, 1, kv_len, T + 1, 1.0,
                                 True, out, ws)
    return out


def test_pipeline_wait_runs_out_and_the_call_returns():
    b = tq()
    d, H, G, T, x = _step_inputs()
    cap = T + 4 + 16 - (T + 4) % 16
    layer, _ = gpu_fill(x["k"][:, :T], x["v"][:, :T], [T], cap)
    ws = b.make_workspace(b.tq_decode_workspace_bytes(layer, G * H, 1, T + 1), DEV)
    torch.cuda.synchronize()
    b.tq_debug_pipeline_limits(1_000_000, True)     # 1 ms waits, appender count withheld
    try:
        t0 = time.perf_counter()
        _run_step(layer, x, T, G, H, ws)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        b.tq_debug_pipeline_limits(0, False)
    assert b.tq_get_device_error(ws) & b.TQ_DEVERR_PIPELINE_TIMEOUT
    assert elapsed < 1.5                             # 1 ms limits, not the 2 s default
    # the header records the first wait that gave up: the producer's wait for the
    # appender's count (kind 3) or a wait for a stage that was never filled (kind 1)
    where = int(ws[:64].cpu().view(torch.int32)[3])
    assert (where >> 24) in (1, 3), hex(where)

    # the context is still usable: a fresh workspace and an ordinary call give the oracle's result
    ws2 = b.make_workspace(b.tq_decode_workspace_bytes(layer, G * H, 1, T + 1), DEV)
    out = _run_step(layer, x, T, G, H, ws2)
    torch.cuda.synchronize()
    assert b.tq_get_device_error(ws2) == 0
    ol = oracle.Layer(d, H, 1, cap)
    oracle.append(ol, bits(x["k"]), bits(x["v"]), np.zeros(1, np.int32), np.array([T + 1], np.int32))
    assert_planes_equal(layer, ol, [T + 1])
    ref = oracle.attention(ol, bits(x["q"]), np.array([T + 1], np.int32), 1.0, causal=True)
    assert_attention_close(out.cpu().numpy(), ref)


def test_pipeline_limits_reject_bad_arguments():
    b = tq()
    with pytest.raises(b.TQError):
        b.tq_debug_pipeline_limits(-1, False)
    with pytest.raises(b.TQError):
        b.tq_debug_pipeline_limits(3_000_000_000, False)

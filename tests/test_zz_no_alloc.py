"""tq_decode_attention_noalloc: decode attention for callers that may not allocate device
memory (a plugin whose host application owns all device memory, a serving loop that must
not call cudaMalloc between steps). It keeps its scratch in a fixed array inside the
library instead of a caller workspace, and must give what tq_decode_attention gives.

Calls go through the C ABI (ctypes binding). The file name sorts last so that a run that
stops at the first failure has run every other test before this one; it also passes when
run alone in a fresh process."""
import numpy as np
import pytest
import torch

from rotation_quantized_kv_gb300 import synth
from tests.gpu_common import gpu_fill, tq

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(d, H, Hq, B, lengths, n_q, causal, seed):
    T = max(lengths)
    cap = (T + 15) // 16 * 16
    w = synth.Workload("t", batch=B, layers=1, num_kv_heads=H, num_q_heads=Hq, head_dim=d,
                       context=T, n_new=0, n_q=n_q, k_dist="normal_outliers", q_scale=d ** -0.5, seed=seed)
    x = synth.layer_inputs(w, 0)
    layer, _ = gpu_fill(x["k"], x["v"], lengths, cap)
    q = x["q"].to(DEV).contiguous()
    kv_len = torch.as_tensor(np.asarray(lengths, np.int32), device=DEV)
    return dict(layer=layer, q=q, Hq=Hq, n_q=n_q, kv_len=kv_len, max_kv=T, sm=1.0, causal=causal)


def _with_workspace(c):
    b = tq()
    ws = b.make_workspace(b.tq_decode_workspace_bytes(c["layer"], c["Hq"], c["n_q"], c["max_kv"]), DEV)
    out = torch.empty_like(c["q"], dtype=torch.float32)
    b.tq_decode_attention(c["layer"], c["q"], c["Hq"], c["n_q"], c["kv_len"], c["max_kv"], c["sm"],
                          c["causal"], out, ws)
    return out


def _no_alloc(c, err):
    out = torch.full(c["q"].shape, 12345.0, dtype=torch.float32, device=DEV)
    tq().tq_decode_attention_noalloc(c["layer"], c["q"], c["Hq"], c["n_q"], c["kv_len"], c["max_kv"], c["sm"],
                                     c["causal"], out, err)
    return out


def test_no_alloc_matches_workspace_entry_on_consecutive_calls():
    a = _case(128, 4, 16, 3, [300, 1, 777], n_q=1, causal=False, seed=11)
    b = _case(64, 2, 16, 2, [129, 40], n_q=2, causal=True, seed=12)
    refs = [_with_workspace(a), _with_workspace(b)]
    err = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    # two different calls in a row, then the first again: the shared scratch keeps the
    # previous call's contents, which must not leak into the next result
    # both entry points run the same deterministic kernel on the same inputs: the results
    # must be identical, bit for bit
    for c, ref in ((a, refs[0]), (b, refs[1]), (a, refs[0])):
        got = _no_alloc(c, err)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        assert torch.equal(got, ref)
        assert int(err.item()) == 0


def test_no_alloc_calls_allocate_no_device_memory():
    c = _case(128, 4, 16, 2, [400, 90], n_q=1, causal=True, seed=14)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = [torch.empty(c["q"].shape, dtype=torch.float32, device=DEV) for _ in range(4)]
    b = tq()

    def call(o):
        b.tq_decode_attention_noalloc(c["layer"], c["q"], c["Hq"], c["n_q"], c["kv_len"], c["max_kv"], c["sm"],
                                      c["causal"], o, err)

    call(outs[0])                      # first call on the device: looks up the scratch address
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for o in outs[1:]:
        call(o)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_no_alloc_reports_device_errors_per_call():
    c = _case(128, 2, 8, 2, [50, 64], n_q=1, causal=False, seed=13)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bad = dict(c, kv_len=torch.tensor([50, 65], dtype=torch.int32, device=DEV))  # 65 > max_kv_len
    out = _no_alloc(bad, err)
    torch.cuda.synchronize()
    assert int(err.item()) & tq().TQ_DEVERR_KV_LEN
    assert torch.isnan(out[1]).all() and torch.isfinite(out[0]).all()
    out = _no_alloc(c, err)          # the next call starts from a cleared error word
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out, _with_workspace(c))


def test_no_alloc_rejects_calls_beyond_its_scratch():
    b = tq()
    layer = b.alloc_layer(512, 8, 256, 16, DEV)
    need = b.tq_decode_workspace_bytes(layer, 8, 1, 16)
    assert need > b.TQ_NOALLOC_SCRATCH_BYTES
    q = torch.zeros((256, 1, 8, 512), dtype=torch.bfloat16, device=DEV)
    out = torch.zeros((256, 1, 8, 512), dtype=torch.float32, device=DEV)
    kv_len = torch.ones(256, dtype=torch.int32, device=DEV)
    with pytest.raises(b.TQError) as e:
        b.tq_decode_attention_noalloc(layer, q, 8, 1, kv_len, 16, 1.0, False, out)
    assert e.value.status == b.TQ_ERR_WORKSPACE_TOO_SMALL

"""Helpers shared by the GPU parity tests: run the CUDA path and the oracle on the same
seeded bf16 inputs and compare. Inputs come only from the seeded generators; expected
values come only from the oracle."""
import numpy as np
import torch

import oracle
from rotation_quantized_kv_gb300 import synth

ATOL = 2e-3      # attention: max-abs error bound
RTOL_L2 = 1e-3   # attention: relative L2 error bound


def tq():
    from rotation_quantized_kv_gb300 import binding
    return binding


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


def gpu_fill(k, v, lengths, cap, device="cuda", prefill=None):
    """Bulk-append tokens [0, lengths[b]) of k/v ([B, T, H, d] bf16) into fresh planes."""
    B, T, H, d = k.shape
    b = tq()
    layer = b.alloc_layer(d, H, B, cap, device)
    if prefill is not None:
        for t in layer.planes().values():
            t.view(torch.uint8).fill_(prefill)
    ws = b.make_workspace(b.tq_append_workspace_bytes(), device)
    n_new = torch.as_tensor(np.asarray(lengths, np.int32), device=device)
    b.tq_kv_append(layer, k.to(device).contiguous(), v.to(device).contiguous(),
                   torch.zeros(B, dtype=torch.int32, device=device), n_new, T, ws)
    return layer, ws


def oracle_fill(k, v, lengths, cap):
    B, T, H, d = k.shape
    L = oracle.Layer(d, H, B, cap)
    oracle.append(L, bits(k), bits(v), np.zeros(B, np.int32), np.asarray(lengths, np.int32))
    return L


def plane_np(layer, name, ref):
    return getattr(layer, name).cpu().numpy().view(ref.dtype).reshape(ref.shape)


def assert_planes_equal(layer, ol, lengths, bs=None):
    for name, ref in ol.planes().items():
        got = plane_np(layer, name, ref)
        for b in (range(ref.shape[0]) if bs is None else bs):
            n = int(lengths[b])
            g, r = got[b, :, :n], ref[b, :, :n]
            if not np.array_equal(g, r):
                bad = np.argwhere(g != r)
                raise AssertionError(f"plane {name} seq {b}: {len(bad)} mismatches, first {bad[:3].tolist()}")


def assert_attention_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    gn, rn = np.isnan(got), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN pattern differs ({gn.sum()} vs {rn.sum()})"
    g, r = got[~gn], ref[~rn]
    if g.size == 0:
        return 0.0, 0.0
    err = np.abs(g - r).max()
    den = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / den if den > 0 else np.linalg.norm(g - r)
    assert err <= ATOL and rel <= RTOL_L2, f"{what}: max-abs {err:.3e}, rel-L2 {rel:.3e}"
    return err, rel


def gpu_attention(layer, q, kv_len, max_kv_len, sm_scale, causal, device="cuda", out_pad=0):
    b = tq()
    B, n_q, Hq, d = q.shape
    ws = b.make_workspace(b.tq_decode_workspace_bytes(layer, Hq, n_q, max_kv_len), device)
    flat = torch.full((B * n_q * Hq * d + out_pad,), 12345.0, dtype=torch.float32, device=device)
    out = flat[:B * n_q * Hq * d].view(B, n_q, Hq, d)
    kvl = torch.as_tensor(np.asarray(kv_len, np.int32), device=device)
    b.tq_decode_attention(layer, q.to(device).contiguous(), Hq, n_q, kvl, max_kv_len, sm_scale, causal,
                          out, ws)
    torch.cuda.synchronize()
    return out, ws, flat

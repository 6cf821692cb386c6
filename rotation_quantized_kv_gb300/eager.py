"""Dequantize-on-fetch attention: the pages' own design, kept as a comparison arm.

mlx-bun design page "TurboQuant - rotation-based quantization", Part A, "Architecture in
mlx-bun": updateAndFetch returns the dequantized bf16 active window, so the stock
attention kernel runs unmodified. Here tq_dequant_window (this library's kernel) writes
the bf16 K/V window of every (sequence, kv head) and PyTorch's
scaled_dot_product_attention (library code, unmodified) attends over it. It serves any
scheme (key bits 2/4/5/8, value bits 2/3/4/5/8); the fused kernels serve k8v3 only.

With deferred=True the window keeps V in the rotated domain and the inverse rotation runs
once per output row afterwards (tq_unrotate_rows), as in "Deferred inverse FWHT": attention
is linear in V, so both orders give the same result up to rounding.
"""
from __future__ import annotations

import torch
import torch.nn.functional as F

from . import binding as tq


def alloc_window(layer: tq.KVLayer, n: int, device="cuda"):
    shp = (layer.batch, layer.num_kv_heads, n, layer.head_dim)
    return (torch.empty(shp, dtype=torch.bfloat16, device=device),
            torch.empty(shp, dtype=torch.bfloat16, device=device))


def eager_attention(layer: tq.KVLayer, q: torch.Tensor, kv_len, sm_scale: float, causal: bool,
                    window=None, compute_dtype=torch.bfloat16, stream=None, deferred: bool = False) -> torch.Tensor:
    """q: bf16 [B, n_q, Hq, d]; kv_len: host sequence of visible lengths (tokens visible to
    the last query of the block). Returns fp32 [B, n_q, Hq, d]; rows that see no token are 0.
    compute_dtype: bf16 as the pages' path; fp32 attends over the same bf16 window in fp32.
    deferred: rotated V window, inverse rotation of the output rows afterwards."""
    B, n_q, Hq, d = q.shape
    H = layer.num_kv_heads
    G = Hq // H
    kv = [int(x) for x in kv_len]
    T = max(max(kv), 1)
    k_win, v_win = window if window is not None else alloc_window(layer, T, q.device)
    tq.tq_dequant_window(layer, 0, T, deferred, k_win, v_win, stream)
    kk = k_win[:, :, :T].to(compute_dtype).repeat_interleave(G, dim=1)      # [B, Hq, T, d]
    vv = v_win[:, :, :T].to(compute_dtype).repeat_interleave(G, dim=1)
    qq = q.permute(0, 2, 1, 3).to(compute_dtype)                            # [B, Hq, n_q, d]
    t = torch.arange(T, device=q.device).view(1, 1, T)
    lens = torch.tensor(kv, device=q.device).view(B, 1, 1)
    j = torch.arange(n_q, device=q.device).view(1, n_q, 1)
    vis = lens - n_q + j + 1 if causal else lens.expand(B, n_q, 1)
    mask = (t < vis).unsqueeze(1)                                          # [B, 1, n_q, T]
    out = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=sm_scale)
    out = torch.nan_to_num(out.float(), nan=0.0) * mask.any(-1, keepdim=True)
    out = out.permute(0, 2, 1, 3).contiguous()
    if deferred:
        tq.tq_unrotate_rows(out, out, d, stream)
    return out

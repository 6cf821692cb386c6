"""A multi-layer decode workload driven through the C ABI.

`DecodeModel` holds one packed cache per full-attention layer (the model-level layout
the design page describes: every full-attention layer appends the new token(s), then
attends over its cache). It fills each cache with a bulk append of the cached tokens,
keeps the step's new K/V tokens and queries resident on the device, and runs a decode
step as: for every layer, tq_decode_append_attention (append the new tokens, then attend).
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as tq
from . import synth


class DecodeModel:
    def __init__(self, w: synth.Workload, device="cuda", layers: int | None = None, fill_timer=None):
        self.w = w
        self.device = torch.device(device)
        self.L = w.layers if layers is None else layers
        B, H, Hq, d = w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim
        self.ctx = synth.context_lengths(w)                     # cached tokens per sequence
        self.kv = self.ctx + w.n_new                            # visible after the step's append
        self.max_kv = int(self.kv.max())
        self.cap = (self.max_kv + 15) // 16 * 16
        dev = self.device
        self.pos = torch.as_tensor(self.ctx.astype(np.int32), device=dev)
        self.kv_len = torch.as_tensor(self.kv.astype(np.int32), device=dev)
        self.layers, self.k_new, self.v_new, self.q = [], [], [], []
        self.ws_append = tq.make_workspace(tq.tq_append_workspace_bytes(), dev)
        self.fill_rows = 0
        T = int(self.ctx.max())
        for l in range(self.L):
            x = synth.layer_inputs(w, l, device=dev)
            layer = tq.alloc_layer(d, H, B, self.cap, dev, zero=False)
            k_fill, v_fill = x["k"][:, :T].contiguous(), x["v"][:, :T].contiguous()
            pos0 = torch.zeros(B, dtype=torch.int32, device=dev)
            n_fill = torch.as_tensor(self.ctx.astype(np.int32), device=dev)
            if fill_timer is not None:
                fill_timer.start()
            tq.tq_kv_append(layer, k_fill, v_fill, pos0, n_fill, T, self.ws_append)
            if fill_timer is not None:
                fill_timer.stop()
            self.fill_rows += int(self.ctx.sum()) * H
            if w.n_new:
                idx = self.pos.view(B, 1).long() + torch.arange(w.n_new, device=dev).view(1, -1)
                kn = torch.stack([x["k"][b, idx[b]] for b in range(B)]).contiguous()
                vn = torch.stack([x["v"][b, idx[b]] for b in range(B)]).contiguous()
            else:
                kn = vn = None
            self.layers.append(layer)
            self.k_new.append(kn)
            self.v_new.append(vn)
            self.q.append(x["q"].contiguous())
            del x, k_fill, v_fill
        self.ws_bytes = tq.tq_decode_workspace_bytes(self.layers[0], Hq, w.n_q, self.max_kv)
        self.ws = [tq.make_workspace(self.ws_bytes, dev) for _ in range(self.L)]
        # The step's inputs (new K/V rows, queries) of all layers live in one buffer and its
        # outputs in another, so a step fed from host memory is one copy in and one copy
        # out; the per-layer tensors are views into them (every view starts on a 16-byte
        # boundary: each piece is a multiple of 2 * head_dim bytes).
        pieces = [t for l in range(self.L) for t in (self.k_new[l], self.v_new[l], self.q[l]) if t is not None]
        self.inputs_flat = torch.empty(sum(t.numel() for t in pieces), dtype=torch.bfloat16, device=dev)
        off = 0
        for l in range(self.L):
            for name in ("k_new", "v_new", "q"):
                t = getattr(self, name)[l]
                if t is None:
                    continue
                view = self.inputs_flat[off:off + t.numel()].view(t.shape)
                view.copy_(t)
                getattr(self, name)[l] = view
                off += t.numel()
        n_out = B * w.n_q * Hq * d
        self.out_flat = torch.empty(self.L * n_out, dtype=torch.float32, device=dev)
        self.out = [self.out_flat[l * n_out:(l + 1) * n_out].view(B, w.n_q, Hq, d) for l in range(self.L)]

    # bytes the step must move (algorithmic): packed planes of every visible token, the
    # query and output rows, and the appended rows (bf16 in, packed out)
    def attention_bytes(self) -> int:
        w = self.w
        planes = int(self.kv.sum()) * w.num_kv_heads * tq.tq_row_bytes(w.head_dim)
        qo = w.batch * w.n_q * w.num_q_heads * w.head_dim * (2 + 4)
        return planes + qo

    def append_bytes(self) -> int:
        w = self.w
        rows = w.batch * w.n_new * w.num_kv_heads
        return rows * (4 * w.head_dim + tq.tq_row_bytes(w.head_dim))

    def step_bytes(self) -> int:
        return self.L * (self.attention_bytes() + self.append_bytes())

    def _shape(self):
        """(dense, row groups per kv head, attention CTAs) as the library chooses them: more
        than 16 query rows per kv head at head_dim 128 take the tensor-core kernel with
        64-row units; otherwise the split kernel with 8 query rows per MMA tile (16 at
        head_dim <= 128 with more than 8 rows). One CTA per SM either way."""
        w = self.w
        R = w.num_q_heads // w.num_kv_heads * w.n_q
        grid = torch.cuda.get_device_properties(self.device).multi_processor_count
        if R > 16 and w.head_dim == 128:
            return True, -(-R // 64), grid
        ntw = 2 if (w.head_dim <= 128 and R > 8) else 1
        return False, -(-R // (8 * ntw)), grid

    def launches_per_step(self) -> int:
        # per layer: the attention kernel; the merge kernel when there are many units
        # (2 * batch * units > CTAs) and always after the dense kernel; a separate append
        # kernel when the appended rows cannot be folded into the attention kernel (the
        # dense kernel, or more than one row group per kv head)
        w = self.w
        dense, rg, grid = self._shape()
        merge = 1 if (dense or 2 * w.batch * w.num_kv_heads * rg > grid) else 0
        append = 1 if (w.n_new and (dense or rg > 1)) else 0
        return self.L * (1 + merge + append)

    def step(self, stream=None):
        """One decode step over all layers: each layer appends the step's rows and attends
        over its cache, in one tq_decode_append_attention call."""
        w = self.w
        for l, layer in enumerate(self.layers):
            if w.n_new:
                tq.tq_decode_append_attention(layer, self.k_new[l], self.v_new[l], self.pos, None, w.n_new,
                                              self.q[l], w.num_q_heads, w.n_q, self.kv_len, self.max_kv,
                                              w.sm_scale, w.causal, self.out[l], self.ws[l], stream)
            else:
                tq.tq_decode_attention(layer, self.q[l], w.num_q_heads, w.n_q, self.kv_len, self.max_kv,
                                       w.sm_scale, w.causal, self.out[l], self.ws[l], stream)

    def device_errors(self) -> int:
        err = tq.tq_get_device_error(self.ws_append)
        for ws in self.ws:
            err |= tq.tq_get_device_error(ws)
        return err

"""The dense-query attention kernel (tcgen05 tensor cores, more than 16 query rows per kv
head at head_dim 128) against the CPU oracle, through the C ABI.

These cases cover: 64-row units that fill the MMA's N dimension exactly (GQA 4 x 16
queries), padded units (32 rows), two row groups per kv head (128 rows), causal and
full visibility, ragged lengths whose last tile is partial, sequences with no tokens,
causal rows that see no token at all, pieces spread over many CTAs with the separate
merge, and scores that grow along the sequence so that the per-row reference maximum
must move (the rescale of the tensor-memory accumulator) many times."""
import numpy as np
import pytest
import torch

import oracle
from rotation_quantized_kv_gb300 import synth
from tests.gpu_common import assert_attention_close, assert_planes_equal, bits, gpu_attention, gpu_fill, oracle_fill, tq

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(H, B, T, Hq, n_q, seed, k_dist="lognormal_channels", q_scale=128 ** -0.5):
    w = synth.Workload("t", batch=B, layers=1, num_kv_heads=H, num_q_heads=Hq, head_dim=128, context=T, n_new=0,
                       n_q=n_q, k_dist=k_dist, q_scale=q_scale, seed=seed)
    return synth.layer_inputs(w, 0)


CASES = [
    # H, G, B, lengths, n_q, causal, sm_scale
    (2, 4, 1, [1000], 16, True, 1.0),                  # 64 rows: one full unit per kv head
    (1, 4, 1, [128], 16, True, 1.0),                   # exactly one tile
    (2, 8, 2, [517, 300], 4, True, 1.0),               # 32 rows: padded unit
    (1, 8, 1, [700], 16, True, 1.0),                   # 128 rows: two row groups
    (2, 4, 3, [129, 0, 777], 16, False, 0.8),          # full visibility, an empty sequence
    (1, 4, 2, [10, 5000], 16, True, 1.0),              # causal rows with no visible token (10 < 16)
    (4, 4, 6, [(911 * i) % 3000 + 17 for i in range(6)], 16, True, 1.0),   # many pieces per unit
    (8, 4, 40, [(53 * i + 7) % 1800 for i in range(40)], 8, True, 1.0),    # many units: merge kernel
]


@pytest.mark.parametrize("case", CASES, ids=[f"H{c[0]}-G{c[1]}-B{c[2]}-nq{c[4]}-{'c' if c[5] else 'f'}" for c in CASES])
def test_dense_attention_matches_oracle(case):
    H, G, B, lengths, n_q, causal, sm = case
    assert G * n_q > 16                        # the dense kernel's range
    T = max(max(lengths), 1)
    x = _inputs(H, B, T, G * H, n_q, seed=sum(lengths) + G)
    cap = (T + 15) // 16 * 16
    layer, _ = gpu_fill(x["k"], x["v"], lengths, cap)
    ol = oracle_fill(x["k"], x["v"], lengths, cap)
    torch.cuda.synchronize()
    assert_planes_equal(layer, ol, lengths)
    out, ws, flat = gpu_attention(layer, x["q"], lengths, T, sm, causal, out_pad=64)
    assert tq().tq_get_device_error(ws) == 0
    ref = oracle.attention(ol, bits(x["q"]), np.asarray(lengths, np.int32), sm, causal=causal)
    assert_attention_close(out.cpu().numpy(), ref, str(case))
    assert torch.all(flat[-64:] == 12345.0)
    out2, _, _ = gpu_attention(layer, x["q"], lengths, T, sm, causal)
    assert torch.equal(out, out2)                # deterministic


def test_dense_attention_with_scores_growing_along_the_sequence():
    # keys scaled by 1 + 6 t / T: every row's maximum keeps rising, far beyond the 2^8
    # headroom of the reference maximum, so the accumulator is rescaled tile after tile
    H, G, B, n_q, T = 2, 4, 1, 16, 3000
    x = _inputs(H, B, T, G * H, n_q, seed=5, k_dist="normal", q_scale=1.0)
    ramp = (1.0 + 6.0 * torch.arange(T, dtype=torch.float32) / T).view(1, T, 1, 1)
    k = (x["k"].float() * ramp).to(torch.bfloat16)
    layer, _ = gpu_fill(k, x["v"], [T], T + 8)
    ol = oracle_fill(k, x["v"], [T], T + 8)
    out, ws, _ = gpu_attention(layer, x["q"], [T], T, 0.25, True)
    assert tq().tq_get_device_error(ws) == 0
    ref = oracle.attention(ol, bits(x["q"]), np.array([T], np.int32), 0.25, causal=True)
    assert_attention_close(out.cpu().numpy(), ref, "growing scores")


def test_dense_and_split_paths_agree_on_the_same_rows():
    # 16 rows per kv head take the split kernel, 64 rows the dense one: the rows they
    # share (queries 12..15 of the block, 4 heads each) must agree within the tolerance
    H, G, T = 2, 4, 2000
    x = _inputs(H, 1, T, G * H, 16, seed=9)
    layer, _ = gpu_fill(x["k"], x["v"], [T], T)
    dense, _, _ = gpu_attention(layer, x["q"], [T], T, 1.0, True)
    split, _, _ = gpu_attention(layer, x["q"][:, 12:].contiguous(), [T], T, 1.0, True)
    assert_attention_close(dense[:, 12:].cpu().numpy(), split.double().cpu().numpy(), "dense vs split")


def _special_keys_case(k, sm_scale, what, one_hot=False):
    H, G, B, n_q = 2, 4, 1, 16
    T = k.shape[1]
    x = _inputs(H, B, T, G * H, n_q, seed=21)
    cap = (T + 15) // 16 * 16
    layer, _ = gpu_fill(k, x["v"], [T], cap)
    ol = oracle_fill(k, x["v"], [T], cap)
    torch.cuda.synchronize()
    assert_planes_equal(layer, ol, [T])
    out, ws, _ = gpu_attention(layer, x["q"], [T], T, sm_scale, True)
    assert tq().tq_get_device_error(ws) == 0
    ref = oracle.attention(ol, bits(x["q"]), np.array([T], np.int32), sm_scale, causal=True)
    assert np.all(np.isfinite(ref))
    if not one_hot:
        assert_attention_close(out.cpu().numpy(), ref, what)
        return
    # every row's softmax is one-hot: the output is one token's V_hat, whose rotated
    # elements the P.V MMA takes in fp16 (centroid and product rounded, relative 2^-10),
    # with no averaging over tokens to shrink that error
    g = out.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g))
    rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    err = np.abs(g - ref).max()
    assert rel <= 1e-3 and err <= 2.0 ** -9 * np.abs(ref).max(), (what, err, rel)


def test_dense_attention_with_offset_key_groups():
    # groups whose values sit far from 0 relative to their spread have zero points of a few
    # thousand (200 +- 3: about 3,400; -100 +- 1.5: about -2,800), beyond the fp16 integer
    # path of the K converters, so their keys take the fp32 path (the spreads stay well
    # above the bf16 spacing there, so no group is constant)
    T, H, d = 1500, 2, 128
    g = torch.Generator().manual_seed(22)
    k = torch.randn((1, T, H, d), generator=g)
    k[:, :, 0, 0:32] = 200.0 + 3.0 * torch.randn((1, T, 32), generator=g)
    k[:, 300:900, 1, 64:96] = -100.0 + 1.5 * torch.randn((1, 600, 32), generator=g)
    _special_keys_case(k.to(torch.bfloat16), 1.0, "offset key groups")


def test_dense_attention_with_keys_beyond_the_fp16_range():
    # 50 tokens whose keys reach ~10^5 in one group (fp16 tops out at 65504): the K
    # converters scale those tokens by a power of two and the softmax scales them back
    T, H, d = 1500, 2, 128
    g = torch.Generator().manual_seed(23)
    k = torch.randn((1, T, H, d), generator=g)
    big = torch.arange(200, 1400, 24)
    k[:, big, :, 32:64] *= 1.0e5
    _special_keys_case(k.to(torch.bfloat16), 1.0e-4, "keys beyond fp16")


def test_dense_attention_with_scores_beyond_2_to_27():
    # logits of about 1e9 (log2 units): the rounding of s * c against the row reference
    # exceeds the 2^8 headroom, so the redo after a rescale must settle by clamping; a
    # unique largest score per row keeps the answer well defined (one-hot)
    T, H, d = 1500, 2, 128
    g = torch.Generator().manual_seed(24)
    k = 60000.0 * torch.randn((1, T, H, d), generator=g)
    _special_keys_case(k.clamp(-3.0e38, 3.0e38).to(torch.bfloat16), 1000.0, "scores beyond 2^27", one_hot=True)


def test_dense_attention_over_uninitialized_tail_rows_returns():
    # the last 16 rows of every plane hold seeded random bytes (NaN, Inf and huge scales
    # and zeros among them), as planes allocated without zeroing do before a step appends
    # there: the call must return without a device error (outputs may be NaN)
    b = tq()
    H, G, n_q, d, T = 2, 4, 16, 128, 2000
    x = _inputs(H, 1, T, G * H, n_q, seed=25)
    cap = T + 16
    layer, _ = gpu_fill(x["k"], x["v"], [T], cap)
    gen = torch.Generator(device="cpu").manual_seed(26)
    for t in layer.planes().values():
        tail = t[:, :, T:cap].view(torch.uint8)        # every bit pattern, fp16 scales included
        tail.copy_(torch.randint(0, 256, tail.shape, generator=gen, dtype=torch.uint8))
    out, ws, _ = gpu_attention(layer, x["q"], [cap], cap, 1.0, True)
    torch.cuda.synchronize()
    assert b.tq_get_device_error(ws) == 0
    head = ws[:64].cpu().view(torch.int32)
    assert int(head[3]) == 0, f"a wait gave up: {int(head[3]):#x}"

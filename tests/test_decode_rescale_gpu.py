"""Decode and prefill with scores that grow along the keys, against the fp64
oracle.

Every kernel keeps a lazy running maximum: the reference is raised,
and the accumulated output rescaled, only when a tile's maximum exceeds it by
more than a factor 2^8.  With N(0,1) inputs that almost never happens after
the first tile, so the ordinary parity tests barely reach the rescale code.
Here the key rows are multiplied by a ramp growing from 1 to 40 along the
sequence (scores up to about 180 in base-2 units), so that the tile maxima
keep rising through every split's share of the keys and the rescale runs many
times (at 3000 keys, 7 heads of one KV head: 37 rises past 2^8 with one
split, 125 with three), in the fp32 and bf16 kernels, the paged kernel, the
4-bit kernel (the ramp applied before quantization) and the stacked-layers
launch, and the prefill kernel's work units.  A falling ramp (40 down to 1)
checks the opposite extreme: the first tile holds the maximum and later
probabilities underflow towards zero.  Split counts are forced too, including
one split (the whole sequence in one CTA).
Bounds of tests/parity.py.
"""

import numpy as np
import pytest
import torch

import oracle
import parity
from gqa_attention_kv_decode_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def f64(t):
    return t.detach().double().cpu().numpy()


def ramp(S, rising=True):
    r = 1.0 + 39.0 * torch.arange(S, dtype=torch.float32) / max(S - 1, 1)
    return (r if rising else r.flip(0)).view(1, 1, S, 1).to(DEV)


def ramped_qkv(B, Hq, Hkv, D, S, dtype, layer, rising=True):
    q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, S, torch.float32, layer=layer, device=DEV)
    k = k * ramp(S, rising)
    return q.to(dtype), k.to(dtype), v.to(dtype)


@pytest.mark.parametrize("splits", [0, 1, 3], ids=["planned", "one_split", "three_splits"])
@pytest.mark.parametrize("rising", [True, False], ids=["rising", "falling"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_decode_ramped_scores(dtype, D, rising, splits):
    B, Hq, Hkv, S = 2, 28, 4, 3000
    lens = [3000, 1777]
    q, k, v = ramped_qkv(B, Hq, Hkv, D, S, dtype, layer=D + int(rising), rising=rising)
    inputs.poison_tail(k, lens)
    inputs.poison_tail(v, lens)
    with binding.plan_override(decode_splits=splits):
        o = binding.decode(q, k, v, kv_lens=torch.tensor(lens, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    got = f64(o)
    kind = parity.kind_of(dtype)
    for b, L in enumerate(lens):
        ref = oracle.attention(f64(q[b:b + 1]), f64(k[b:b + 1, :, :L]), f64(v[b:b + 1, :, :L]),
                               scale=D ** -0.5)["o"]
        parity.check(got[b:b + 1], ref, kind, f"request {b}")


@pytest.mark.parametrize("rising", [True, False], ids=["rising", "falling"])
def test_paged_decode_ramped_scores(rising):
    B, Hq, Hkv, D, S, bs = 3, 32, 8, 128, 2000, 64
    lens = [2000, 1500, 64]
    q, k, v = ramped_qkv(B, Hq, Hkv, D, S, torch.bfloat16, layer=31, rising=rising)
    kp, vp, table = inputs.paged_pool(k, v, lens, bs, seed=5)
    ref = oracle.attention_paged(f64(q), f64(kp), f64(vp), table.cpu().numpy(), lens, bs, scale=D ** -0.5)["o"]
    o = binding.decode_paged(q, kp, vp, table, torch.tensor(lens, dtype=torch.int32, device=DEV), S)
    torch.cuda.synchronize()
    parity.check(f64(o), ref, "bf16")


@pytest.mark.parametrize("splits", [0, 1], ids=["planned", "one_split"])
@pytest.mark.parametrize("rising", [True, False], ids=["rising", "falling"])
@pytest.mark.parametrize("D", [64, 128])
def test_q4_decode_ramped_scores(D, rising, splits):
    """The ramp is applied to K before quantization, so the scales (and the
    scores) grow along the cache; the oracle attends over the same codes."""
    B, Hq, Hkv, S = 2, 32, 8, 2048
    lens = [2048, 999]
    _, k, v = ramped_qkv(B, Hq, Hkv, D, S, torch.bfloat16, layer=41, rising=rising)
    q = inputs.randn((B, Hq, 1, D), inputs.tensor_seed(41, 0), torch.bfloat16, DEV)
    kc, ks, kb = (torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in oracle.quantize_q4(k.float().cpu().numpy()))
    vc, vs, vb = (torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in oracle.quantize_q4(v.float().cpu().numpy()))
    for t in (ks, kb, vs, vb):
        inputs.poison_tail(t, lens)
    with binding.plan_override(decode_splits=splits):
        o = binding.decode_q4(q, kc, ks, kb, vc, vs, vb, kv_lens=torch.tensor(lens, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    ref = oracle.attention_q4(q.float().cpu().numpy(), kc.cpu().numpy(), ks.cpu().numpy(), kb.cpu().numpy(),
                              vc.cpu().numpy(), vs.cpu().numpy(), vb.cpu().numpy(), kv_lens=lens,
                              scale=D ** -0.5)["o"]
    parity.check(o.float().cpu().numpy(), ref, "q4")


def test_stacked_layers_ramped_scores():
    """Four layers in one launch, rising and falling ramps alternating."""
    NL, B, Hq, Hkv, D, S = 4, 1, 28, 4, 128, 4096
    per = [ramped_qkv(B, Hq, Hkv, D, S, torch.float32, layer=50 + l, rising=l % 2 == 0) for l in range(NL)]
    q, k, v = (torch.stack([x[i] for x in per]).contiguous() for i in range(3))
    ws = torch.zeros(binding.gqa_attn_decode_layers_workspace_size(NL, B, Hq, Hkv, D, S, binding.GQA_F32),
                     dtype=torch.uint8, device=DEV)
    o = torch.empty_like(q)
    binding.gqa_attn_decode_layers(q, k, v, o, None, D ** -0.5, ws)
    torch.cuda.synchronize()
    for l in range(NL):
        ref = oracle.attention(f64(q[l]), f64(k[l]), f64(v[l]), scale=D ** -0.5)["o"]
        parity.check(f64(o[l]), ref, "f32", f"layer {l}")


@pytest.mark.parametrize("unit", ["planned", "pairs", "single_tiles", "kv_split_2", "kv_split_4"])
@pytest.mark.parametrize("rising", [True, False], ids=["rising", "falling"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("q_len,kv_len", [(1000, 1000), (300, 2000)], ids=["square", "chunk"])
def test_prefill_ramped_scores(q_len, kv_len, D, rising, unit):
    """Prefill under the same ramp (1 to 40 along the keys, or 40 to 1): the
    lazy reference of every work-unit kind (pairs, single tiles whose odd
    slot starts with no visible key, KV shares merged across a cluster)."""
    Hq, Hkv = 14, 2
    q = inputs.randn((1, Hq, q_len, D), inputs.tensor_seed(61, 0), torch.float32, DEV)
    _, k, v = inputs.qkv(1, Hq, Hkv, D, 1, kv_len, torch.float32, layer=61, device=DEV)
    k = k * ramp(kv_len, rising)
    q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    override = {"planned": {}, "pairs": {"prefill_interleave_from": 1 << 20},
                "single_tiles": {"prefill_interleave_from": 0}, "kv_split_2": {"prefill_kv_split": 2},
                "kv_split_4": {"prefill_kv_split": 4}}[unit]
    with binding.plan_override(**override):
        o = binding.prefill(q, k, v, causal=True)
    torch.cuda.synchronize()
    ref = oracle.attention(f64(q), f64(k), f64(v), scale=D ** -0.5, causal=True)["o"]
    parity.check(f64(o), ref, "bf16")

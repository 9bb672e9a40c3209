"""Requests much shorter than the call's max_kv_len, against the fp64 oracle.

The split plan is sized for max_kv_len.  A request of L keys uses
min(n_split, ceil(L / chunk)) splits, and in a one-wave plan the chunk is two
tiles, so a short request spreads over all of its splits instead of leaving
most of its CTAs idle (a capacity-sized max_kv_len with short requests is what
a CUDA graph replayed over many decode steps sees).  Each case puts one short
request (1 key up to a few thousand, on both sides of the one- and two-tile
boundaries) beside a full-length one, so that the spread and the full plan run
in the same launch: the fp32 and bf16 kernels, the 4-bit kernel, the paged
kernel and the 4-bit cache with a residual window.  Rows past each length are
NaN, so a read past L fails.  Bounds of tests/parity.py.
"""

import numpy as np
import pytest
import torch

import oracle
import parity
from gqa_attention_kv_decode_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
S = 16384
SHORT = [1, 63, 64, 65, 129, 700, 5000]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def f64(t):
    return t.detach().double().cpu().numpy()


@pytest.mark.parametrize("L", SHORT)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_decode_short_beside_long(dtype, D, L):
    Hq, Hkv = 28, 4
    lens = [L, S]
    q, k, v = inputs.qkv(2, Hq, Hkv, D, 1, S, dtype, layer=200 + L % 97, device=DEV)
    inputs.poison_tail(k, lens)
    inputs.poison_tail(v, lens)
    assert binding.gqa_attn_decode_num_splits(2, Hq, Hkv, D, S, binding._dtype_code(q)) > 1
    o = binding.decode(q, k, v, kv_lens=torch.tensor(lens, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    got = f64(o)
    for b, n in enumerate(lens):
        ref = oracle.attention(f64(q[b:b + 1]), f64(k[b:b + 1, :, :n]), f64(v[b:b + 1, :, :n]),
                               scale=D ** -0.5)["o"]
        parity.check(got[b:b + 1], ref, parity.kind_of(dtype), f"request {b} ({n} keys)")


@pytest.mark.parametrize("L", SHORT)
def test_decode_one_short_request_with_capacity_max(L):
    """One request, max_kv_len the cache's capacity (32,768) and L keys."""
    Hq, Hkv, D, cap = 28, 4, 128, 32768
    q, k, v = inputs.qkv(1, Hq, Hkv, D, 1, cap, torch.float32, layer=300 + L % 89, device=DEV)
    inputs.poison_tail(k, [L])
    inputs.poison_tail(v, [L])
    o = binding.decode(q, k, v, kv_lens=torch.tensor([L], dtype=torch.int32, device=DEV), max_kv_len=cap)
    torch.cuda.synchronize()
    ref = oracle.attention(f64(q), f64(k[:, :, :L]), f64(v[:, :, :L]), scale=D ** -0.5)["o"]
    parity.check(f64(o), ref, "f32")


@pytest.mark.parametrize("L", SHORT)
def test_q4_short_beside_long(L):
    B, Hq, Hkv, D = 2, 32, 8, 128
    lens = [L, S]
    kc, ks, kb, vc, vs, vb = inputs.q4_cache(B, Hkv, D, S, layer=400 + L % 83, device=DEV)
    for t in (ks, kb, vs, vb):
        inputs.poison_tail(t, lens)
    q = inputs.randn((B, Hq, 1, D), inputs.tensor_seed(400 + L % 83, 0), torch.bfloat16, DEV)
    o = binding.decode_q4(q, kc, ks, kb, vc, vs, vb, kv_lens=torch.tensor(lens, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    ref = oracle.attention_q4(q.float().cpu().numpy(), kc.cpu().numpy(), ks.cpu().numpy(), kb.cpu().numpy(),
                              vc.cpu().numpy(), vs.cpu().numpy(), vb.cpu().numpy(), kv_lens=lens,
                              scale=D ** -0.5)["o"]
    parity.check(o.float().cpu().numpy(), ref, "q4")


@pytest.mark.parametrize("L", [1, 64, 65, 700, 5000])
def test_paged_short_beside_long(L):
    B, Hq, Hkv, D, bs = 2, 32, 8, 128, 64
    lens = [L, 8192]
    q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, 8192, torch.bfloat16, layer=500 + L % 79, device=DEV)
    kp, vp, table = inputs.paged_pool(k, v, lens, bs, seed=7)
    ref = oracle.attention_paged(f64(q), f64(kp), f64(vp), table.cpu().numpy(), lens, bs, scale=D ** -0.5)["o"]
    o = binding.decode_paged(q, kp, vp, table, torch.tensor(lens, dtype=torch.int32, device=DEV), 8192)
    torch.cuda.synchronize()
    parity.check(f64(o), ref, "bf16")


@pytest.mark.parametrize("L", [0, 1, 64, 65, 700, 5000])
def test_q4_residual_short_beside_long(L):
    """L quantized keys plus a 10-key window beside a full 4-bit cache with a
    50-key window: the window's partial sits in the slot after the splits the
    short request uses."""
    B, Hq, Hkv, D, R = 2, 32, 8, 128, 64
    n_quant, kv_lens = [L, S], [L + 10, S + 50]
    seed = 600 + L % 73
    cache = inputs.q4_cache(B, Hkv, D, S, layer=seed, device=DEV)
    for t in cache[1:3] + cache[4:6]:
        inputs.poison_tail(t, n_quant)
    kr = inputs.randn((B, Hkv, R, D), inputs.tensor_seed(seed, 5), torch.bfloat16, DEV)
    vr = inputs.randn((B, Hkv, R, D), inputs.tensor_seed(seed, 6), torch.bfloat16, DEV)
    inputs.poison_tail(kr, [a - b for a, b in zip(kv_lens, n_quant)])
    inputs.poison_tail(vr, [a - b for a, b in zip(kv_lens, n_quant)])
    q = inputs.randn((B, Hq, 1, D), inputs.tensor_seed(seed, 0), torch.bfloat16, DEV)
    o = binding.decode_q4_residual(q, *cache, kr, vr, torch.tensor(n_quant, dtype=torch.int32, device=DEV),
                                   torch.tensor(kv_lens, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    kc, ks, kb, vc, vs, vb = (t.cpu().numpy() for t in cache)
    ref = oracle.attention_q4_residual(q.float().cpu().numpy(), kc, ks, kb, vc, vs, vb, kr.float().cpu().numpy(),
                                       vr.float().cpu().numpy(), n_quant, kv_lens, scale=D ** -0.5)["o"]
    parity.check(o.float().cpu().numpy(), ref, "q4")

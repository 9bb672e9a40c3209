"""The decode kernels' lost-copy path, forced without faulting anything.

Every wait of a decode kernel on a tile copy gives up after a time limit; the
CTA then drains the copies it issued, writes no partials, sets
GQA_DEV_WAIT_TIMEOUT in the workspace status word and returns.  A real lost
copy cannot be produced safely, so gqa_attn_set_decode_wait_test makes the
first thread of every CTA wait, after issuing its first copies, on a barrier
that nothing arrives on (a bounded wait of 100 us here), which sends every
CTA down that path.  The test checks that the status word reports it, and
that the same context then computes a correct result (the GPU stays usable),
for the fp32 and bf16 kernels (both bf16 shapes), the paged, 4-bit and
stacked-layers launches.
"""

import contextlib

import numpy as np
import pytest
import torch

import oracle
import parity
from gqa_attention_kv_decode_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
STALL_NS = 100_000


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@contextlib.contextmanager
def lost_copies():
    binding.gqa_attn_set_decode_wait_test(STALL_NS)
    try:
        yield
    finally:
        binding.gqa_attn_set_decode_wait_test(0)


def f64(t):
    return t.detach().double().cpu().numpy()


def fresh_ws(n_bytes):
    return torch.zeros(n_bytes, dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("dtype,S,B", [(torch.float32, 3000, 2), (torch.bfloat16, 3000, 2),
                                       (torch.bfloat16, 16384, 1), (torch.float32, 32768, 1)],
                         ids=["f32", "bf16_4warp", "bf16_8warp", "f32_long"])
def test_decode_lost_copy_is_reported_and_the_context_survives(dtype, S, B):
    Hq, Hkv, D = 28, 4, 128
    q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, S, dtype, layer=101, device=DEV)
    n_ws = binding.gqa_attn_decode_workspace_size(B, Hq, Hkv, D, S, binding._dtype_code(q))
    o = torch.empty_like(q)
    ws = fresh_ws(n_ws)
    with lost_copies():
        binding.gqa_attn_decode(q, k, v, o, None, D ** -0.5, ws)
    status = binding.gqa_attn_read_device_status(ws)
    assert status & binding.GQA_DEV_WAIT_TIMEOUT
    ws = fresh_ws(n_ws)
    binding.gqa_attn_decode(q, k, v, o, None, D ** -0.5, ws)
    torch.cuda.synchronize()
    assert not binding.gqa_attn_read_device_status(ws) & binding.GQA_DEV_WAIT_TIMEOUT
    ref = oracle.attention(f64(q), f64(k), f64(v), scale=D ** -0.5)["o"]
    parity.check(f64(o), ref, parity.kind_of(dtype))


def test_paged_decode_lost_copy_is_reported():
    B, Hq, Hkv, D, S, bs = 2, 32, 8, 128, 1000, 64
    lens = [1000, 333]
    q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, S, torch.bfloat16, layer=102, device=DEV)
    kp, vp, table = inputs.paged_pool(k, v, lens, bs, seed=3)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    n_ws = binding.gqa_attn_decode_workspace_size(B, Hq, Hkv, D, S, binding.GQA_BF16)
    o = torch.empty_like(q)
    ws = fresh_ws(n_ws)
    with lost_copies():
        binding.gqa_attn_decode_paged(q, None, None, kp, vp, table, lens_t, o, D ** -0.5, ws, S)
    assert binding.gqa_attn_read_device_status(ws) & binding.GQA_DEV_WAIT_TIMEOUT
    ws = fresh_ws(n_ws)
    binding.gqa_attn_decode_paged(q, None, None, kp, vp, table, lens_t, o, D ** -0.5, ws, S)
    torch.cuda.synchronize()
    ref = oracle.attention_paged(f64(q), f64(kp), f64(vp), table.cpu().numpy(), lens, bs, scale=D ** -0.5)["o"]
    parity.check(f64(o), ref, "bf16")


def test_q4_decode_lost_copy_is_reported():
    B, Hq, Hkv, D, S = 2, 32, 8, 128, 2048
    cache = inputs.q4_cache(B, Hkv, D, S, layer=103, device=DEV)
    q = inputs.randn((B, Hq, 1, D), 104, torch.bfloat16, DEV)
    n_ws = binding.gqa_attn_decode_q4_workspace_size(B, Hq, Hkv, D, S)
    o = torch.empty_like(q)
    ws = fresh_ws(n_ws)
    with lost_copies():
        binding.gqa_attn_decode_q4(q, *cache, o, None, D ** -0.5, ws)
    assert binding.gqa_attn_read_device_status(ws) & binding.GQA_DEV_WAIT_TIMEOUT
    ws = fresh_ws(n_ws)
    binding.gqa_attn_decode_q4(q, *cache, o, None, D ** -0.5, ws)
    torch.cuda.synchronize()
    kc, ks, kb, vc, vs, vb = (t.cpu().numpy() for t in cache)
    ref = oracle.attention_q4(q.float().cpu().numpy(), kc, ks, kb, vc, vs, vb, scale=D ** -0.5)["o"]
    parity.check(o.float().cpu().numpy(), ref, "q4")


def test_stacked_layers_lost_copy_is_reported():
    NL, B, Hq, Hkv, D, S = 3, 1, 28, 4, 128, 2048
    q = inputs.randn((NL, B, Hq, 1, D), 105, torch.float32, DEV)
    k = inputs.randn((NL, B, Hkv, S, D), 106, torch.float32, DEV)
    v = inputs.randn((NL, B, Hkv, S, D), 107, torch.float32, DEV)
    n_ws = binding.gqa_attn_decode_layers_workspace_size(NL, B, Hq, Hkv, D, S, binding.GQA_F32)
    o = torch.empty_like(q)
    ws = fresh_ws(n_ws)
    with lost_copies():
        binding.gqa_attn_decode_layers(q, k, v, o, None, D ** -0.5, ws)
    assert binding.gqa_attn_read_device_status(ws) & binding.GQA_DEV_WAIT_TIMEOUT
    ws = fresh_ws(n_ws)
    binding.gqa_attn_decode_layers(q, k, v, o, None, D ** -0.5, ws)
    torch.cuda.synchronize()
    for l in range(NL):
        ref = oracle.attention(f64(q[l]), f64(k[l]), f64(v[l]), scale=D ** -0.5)["o"]
        parity.check(f64(o[l]), ref, "f32", f"layer {l}")


def test_wait_test_rejects_limits_past_one_second():
    with pytest.raises(binding.GqaAttnError) as e:
        binding.gqa_attn_set_decode_wait_test(2_000_000_000)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG

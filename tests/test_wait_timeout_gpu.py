"""The kernels' lost-copy path, forced without faulting anything.

Every wait of a kernel on a copy or a product gives up after a time limit;
the CTA then drains what it issued and returns: a decode CTA writes no
partials and sets GQA_DEV_WAIT_TIMEOUT in the workspace status word, a
prefill CTA writes its rows as NaN and sets it in the prefill status word.
A real lost copy cannot be produced safely, so gqa_attn_set_wait_test makes
the thread that issues a CTA's copies wait, after its first ones, on a
barrier that nothing arrives on (a bounded wait of 100 us here), which sends
every CTA down that path.  The tests check that the status word reports it
and that the same context then computes a correct result (the GPU stays
usable): the fp32 and bf16 decode kernels (both bf16 shapes), the paged,
4-bit and stacked-layers launches, and prefill at D = 64 and 128 in pairs,
single-tile units, KV splits over clusters and with per-request lengths.
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
    binding.gqa_attn_set_wait_test(STALL_NS)
    try:
        yield
    finally:
        binding.gqa_attn_set_wait_test(0)


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
        binding.gqa_attn_set_wait_test(2_000_000_000)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG


@pytest.mark.parametrize("case", ["pairs", "single_tiles", "kv_split", "varlen"])
@pytest.mark.parametrize("D", [64, 128])
def test_prefill_lost_copy_is_reported_and_the_context_survives(D, case):
    """Prefill's TMA thread stalls after its first copies: the CTA drains its
    products and copies, writes the rows that waited on it as NaN and flags
    the prefill status word; the next call on the same context is correct."""
    Hq, Hkv = 14, 2
    q_len, kv_len = (300, 2000) if case == "kv_split" else (1000, 1000)
    q = inputs.randn((2 if case == "varlen" else 1, Hq, q_len, D), 111, torch.bfloat16, DEV)
    k = inputs.randn((q.shape[0], Hkv, kv_len, D), 112, torch.bfloat16, DEV)
    v = inputs.randn((q.shape[0], Hkv, kv_len, D), 113, torch.bfloat16, DEV)
    override = {"pairs": {"prefill_interleave_from": 1 << 20}, "single_tiles": {"prefill_interleave_from": 0},
                "kv_split": {"prefill_kv_split": 4}, "varlen": {}}[case]
    lens = [1000, 700]

    def run():
        o = torch.full_like(q, 3.0)
        with binding.plan_override(**override):
            if case == "varlen":
                binding.gqa_attn_prefill_varlen(q, k, v, o, torch.tensor(lens, dtype=torch.int32, device=DEV),
                                                torch.tensor(lens, dtype=torch.int32, device=DEV), D ** -0.5)
            else:
                binding.gqa_attn_prefill(q, k, v, o, kv_len, D ** -0.5, True)
        torch.cuda.synchronize()
        return o

    binding.gqa_attn_clear_prefill_status()
    with lost_copies():
        o = run()
    assert binding.gqa_attn_read_prefill_status() & binding.GQA_DEV_WAIT_TIMEOUT
    rows = lens if case == "varlen" else [q_len]
    # The last query rows belong to the unit with the most KV tiles, more than
    # the stages hold, so its work waited on copies that were never issued:
    # those rows are NaN.  (A unit whose copies were all issued before the
    # stall may finish normally.)
    for b, n in enumerate(rows):
        assert torch.isnan(o[b, :, n - 1].float()).all(), "rows that waited on a lost copy are NaN"
    binding.gqa_attn_clear_prefill_status()
    o = run()
    assert not binding.gqa_attn_read_prefill_status() & binding.GQA_DEV_WAIT_TIMEOUT
    for b, n in enumerate(rows):
        kn = n if case == "varlen" else kv_len
        ref = oracle.attention(f64(q[b:b + 1, :, :n]), f64(k[b:b + 1, :, :kn]), f64(v[b:b + 1, :, :kn]),
                               scale=D ** -0.5, causal=True)["o"]
        parity.check(f64(o[b:b + 1, :, :n]), ref, "bf16", f"request {b}")

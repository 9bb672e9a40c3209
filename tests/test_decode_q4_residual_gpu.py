"""Decode over a 4-bit cache followed by a bf16 residual window, on the GPU,
against the fp64 oracle (bounds of tests/parity.py for 4-bit caches: max abs
error 2e-2 and 2^-5 of each row's largest reference value).

Scales and biases past n_quant and window rows past kv_len - n_quant are
NaN: a kernel that reads them fails.  The last test runs a decode loop that
appends each new token to the window and moves aged 64-token blocks into the
4-bit cache with the GPU quantizer, checking every step.
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
    return t.detach().float().cpu().numpy()


def make(B, Hq, Hkv, D, S_cap, R_cap, n_quant, kv_lens, seed):
    cache = inputs.q4_cache(B, Hkv, D, S_cap, layer=seed, device=DEV)
    for t in cache[1:3] + cache[4:6]:
        inputs.poison_tail(t, n_quant)
    kr = inputs.randn((B, Hkv, R_cap, D), inputs.tensor_seed(seed, 5), torch.bfloat16, DEV)
    vr = inputs.randn((B, Hkv, R_cap, D), inputs.tensor_seed(seed, 6), torch.bfloat16, DEV)
    inputs.poison_tail(kr, [L - n for L, n in zip(kv_lens, n_quant)])
    inputs.poison_tail(vr, [L - n for L, n in zip(kv_lens, n_quant)])
    q = inputs.randn((B, Hq, 1, D), inputs.tensor_seed(seed, 0), torch.bfloat16, DEV)
    return q, cache, kr, vr


def run_check(q, cache, kr, vr, n_quant, kv_lens, max_quant=None):
    D = q.shape[-1]
    nq_t = torch.tensor(n_quant, dtype=torch.int32, device=DEV)
    L_t = torch.tensor(kv_lens, dtype=torch.int32, device=DEV)
    o = binding.decode_q4_residual(q, *cache, kr, vr, nq_t, L_t, max_quant=max_quant)
    torch.cuda.synchronize()
    kc, ks, kb, vc, vs, vb = (t.cpu().numpy() for t in cache)
    ref = oracle.attention_q4_residual(f64(q), kc, ks, kb, vc, vs, vb, f64(kr), f64(vr), n_quant, kv_lens,
                                       scale=D ** -0.5)["o"]
    return parity.check(f64(o), ref, "q4")


CASES = [(128, 64), (64, 128), (128, 200)]


@pytest.mark.parametrize("D,R_cap", CASES, ids=[f"D{d}-R{r}" for d, r in CASES])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (14, 2), (28, 4)], ids=["32x8", "14x2", "28x4"])
def test_q4_residual_matches_oracle(D, R_cap, Hq, Hkv):
    S_cap = 1024
    n_quant = [1000, 0, 700, 333, 64, 0, 1024]
    kv_lens = [min(1000 + R_cap, 1000 + 64), 50, 700, 390, 65, 0, 1024 + R_cap]
    q, cache, kr, vr = make(len(n_quant), Hq, Hkv, D, S_cap, R_cap, n_quant, kv_lens, R_cap + D)
    run_check(q, cache, kr, vr, n_quant, kv_lens)


@pytest.mark.parametrize("splits", ["1", "4", "33"])
def test_q4_residual_forced_split_counts(splits):
    n_quant, kv_lens = [4096, 1500, 0], [4096 + 100, 1500, 77]
    q, cache, kr, vr = make(3, 32, 8, 128, 4096, 128, n_quant, kv_lens, 9)
    with binding.plan_override(decode_splits=int(splits)):
        run_check(q, cache, kr, vr, n_quant, kv_lens)


def test_q4_residual_empty_request_is_zero_and_flagged():
    n_quant, kv_lens = [0, 10], [0, 20]
    q, cache, kr, vr = make(2, 8, 8, 64, 64, 64, n_quant, kv_lens, 4)
    ws = torch.zeros(binding.gqa_attn_decode_q4_residual_workspace_size(2, 8, 8, 64, 64),
                     dtype=torch.uint8, device=DEV)
    o = torch.empty_like(q)
    binding.gqa_attn_decode_q4_residual(q, *cache, kr, vr, torch.tensor(n_quant, dtype=torch.int32, device=DEV),
                                        torch.tensor(kv_lens, dtype=torch.int32, device=DEV), o, 0.125, ws)
    assert binding.gqa_attn_read_device_status(ws) & binding.GQA_DEV_EMPTY_REQUEST
    assert (o[0] == 0).all()


def test_decode_loop_with_window_flushes():
    """200 decode steps: each appends its token to the window (capacity 128);
    a full window moves its oldest 64 rows into the 4-bit cache (GPU
    quantizer) and shifts.  Every step matches the oracle on the state."""
    B, Hq, Hkv, D, S_cap, R = 2, 32, 8, 128, 1024, 128
    cache = inputs.q4_cache(B, Hkv, D, S_cap, layer=21, device=DEV)
    kc, ks, kb, vc, vs, vb = cache
    kr = torch.zeros((B, Hkv, R, D), dtype=torch.bfloat16, device=DEV)
    vr = torch.zeros_like(kr)
    nq, nr = 512, 0  # 512 tokens already quantized, empty window
    ws = torch.zeros(binding.gqa_attn_decode_q4_residual_workspace_size(B, Hq, Hkv, D, S_cap),
                     dtype=torch.uint8, device=DEV)
    o = torch.empty((B, Hq, 1, D), dtype=torch.bfloat16, device=DEV)
    for step in range(200):
        if nr == R:  # flush the oldest 64 window rows
            binding.gqa_attn_quantize_q4(kr[:, :, :64].contiguous(), kc, ks, kb, dst_row0=nq)
            binding.gqa_attn_quantize_q4(vr[:, :, :64].contiguous(), vc, vs, vb, dst_row0=nq)
            kr[:, :, :R - 64] = kr[:, :, 64:].clone()
            vr[:, :, :R - 64] = vr[:, :, 64:].clone()
            nq, nr = nq + 64, nr - 64
        kr[:, :, nr] = inputs.randn((B, Hkv, D), inputs.tensor_seed(step, 7), torch.bfloat16, DEV)
        vr[:, :, nr] = inputs.randn((B, Hkv, D), inputs.tensor_seed(step, 8), torch.bfloat16, DEV)
        nr += 1
        q = inputs.randn((B, Hq, 1, D), inputs.tensor_seed(step, 9), torch.bfloat16, DEV)
        nq_t = torch.full((B,), nq, dtype=torch.int32, device=DEV)
        L_t = torch.full((B,), nq + nr, dtype=torch.int32, device=DEV)
        binding.gqa_attn_decode_q4_residual(q, kc, ks, kb, vc, vs, vb, kr, vr, nq_t, L_t, o, D ** -0.5, ws)
        if step % 25 == 0 or step == 199:
            torch.cuda.synchronize()
            ref = oracle.attention_q4_residual(f64(q), *(t.cpu().numpy() for t in (kc, ks, kb, vc, vs, vb)),
                                               f64(kr), f64(vr), [nq] * B, [nq + nr] * B, scale=D ** -0.5)["o"]
            parity.check(f64(o), ref, "q4", f"step {step}")
    assert nq > 512  # at least one flush happened

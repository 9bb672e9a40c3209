"""Seeded random shapes against the oracle: prefill (D = 64 and 128, causal
and full, chunks at an offset, every work-unit kind the planner can pick or
the override forces, and per-request lengths), decode (fp32 and bf16, ragged
lengths with empty requests) and 4-bit decode.  Bounds of tests/parity.py.  The shapes are drawn once from a fixed
seed, so a failure names a reproducible case.
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


def _heads(rng):
    hkv = int(rng.choice([1, 2, 4, 8]))
    return hkv * int(rng.choice([1, 2, 3, 5, 7, 8])), hkv


def _prefill_cases(n=24, seed=20261202):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        D = int(rng.choice([64, 128]))
        Hq, Hkv = _heads(rng)
        B = int(rng.integers(1, 3))
        kv_len = int(rng.integers(1, 1500))
        q_len = int(rng.integers(1, kv_len + 1)) if rng.random() < 0.5 else kv_len
        causal = bool(rng.random() < 0.75)
        unit = int(rng.choice([-1, -1, 0, 1, 1 << 20]))  # planner, every tile single, from pair 1, pairs only
        cases.append((i, B, Hq, Hkv, D, q_len, kv_len, causal, unit))
    return cases


@pytest.mark.parametrize("i,B,Hq,Hkv,D,q_len,kv_len,causal,unit", _prefill_cases())
def test_prefill_random_shape(i, B, Hq, Hkv, D, q_len, kv_len, causal, unit):
    s_cap = kv_len + int(i % 3) * 37
    q = inputs.randn((B, Hq, q_len, D), inputs.tensor_seed(100 + i, 0), torch.bfloat16, DEV)
    k = inputs.randn((B, Hkv, s_cap, D), inputs.tensor_seed(100 + i, 1), torch.bfloat16, DEV)
    v = inputs.randn((B, Hkv, s_cap, D), inputs.tensor_seed(100 + i, 2), torch.bfloat16, DEV)
    k[:, :, kv_len:] = float("nan")
    v[:, :, kv_len:] = float("nan")
    with binding.plan_override(prefill_interleave_from=unit):
        o = binding.prefill(q, k, v, kv_len=kv_len, causal=causal)
    torch.cuda.synchronize()
    ref = oracle.attention(f64(q), f64(k[:, :, :kv_len]), f64(v[:, :, :kv_len]), scale=D ** -0.5,
                           causal=causal)["o"]
    parity.check(f64(o), ref, "bf16", f"case {i}")


def _decode_cases(n=24, seed=20261203):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        D = int(rng.choice([64, 128]))
        Hq, Hkv = _heads(rng)
        B = int(rng.integers(1, 6))
        s_cap = int(rng.integers(1, 5000))
        dtype = "f32" if rng.random() < 0.5 else "bf16"
        lens = [int(x) for x in rng.integers(0, s_cap + 1, size=B)]
        if rng.random() < 0.3:
            lens = None  # every request at s_cap
        cases.append((i, B, Hq, Hkv, D, s_cap, dtype, lens))
    return cases


@pytest.mark.parametrize("i,B,Hq,Hkv,D,s_cap,dtype,lens", _decode_cases())
def test_decode_random_shape(i, B, Hq, Hkv, D, s_cap, dtype, lens):
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, s_cap, dt, layer=200 + i, device=DEV)
    kv_lens = None
    if lens is not None:
        inputs.poison_tail(k, lens)
        inputs.poison_tail(v, lens)
        kv_lens = torch.tensor(lens, dtype=torch.int32, device=DEV)
    o = binding.decode(q, k, v, kv_lens=kv_lens)
    torch.cuda.synchronize()
    got = f64(o)
    for b in range(B):
        L = s_cap if lens is None else lens[b]
        if L == 0:
            assert (got[b] == 0).all(), f"case {i}: request {b} has no keys"
            continue
        ref = oracle.attention(f64(q[b:b + 1]), f64(k[b:b + 1, :, :L]), f64(v[b:b + 1, :, :L]),
                               scale=D ** -0.5)["o"]
        parity.check(got[b:b + 1], ref, dtype, f"case {i} request {b}")


def _q4_cases(n=16, seed=20261204):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        D = int(rng.choice([64, 128]))
        Hq, Hkv = _heads(rng)
        B = int(rng.integers(1, 5))
        s_cap = 8 * int(rng.integers(1, 500))  # the 4-bit cache holds a multiple of 8 rows
        lens = [int(x) for x in rng.integers(0, s_cap + 1, size=B)]
        if rng.random() < 0.3:
            lens = None
        cases.append((i, B, Hq, Hkv, D, s_cap, lens))
    return cases


@pytest.mark.parametrize("i,B,Hq,Hkv,D,s_cap,lens", _q4_cases())
def test_q4_decode_random_shape(i, B, Hq, Hkv, D, s_cap, lens):
    """4-bit decode on random shapes; scales and biases past each request's
    length are NaN, and a request without keys returns zeros."""
    kc, ks, kb, vc, vs, vb = inputs.q4_cache(B, Hkv, D, s_cap, layer=300 + i, device=DEV)
    q = inputs.randn((B, Hq, 1, D), inputs.tensor_seed(300 + i, 0), torch.bfloat16, DEV)
    kv_lens = None
    if lens is not None:
        for t in (ks, kb, vs, vb):
            inputs.poison_tail(t, lens)
        kv_lens = torch.tensor(lens, dtype=torch.int32, device=DEV)
    o = binding.decode_q4(q, kc, ks, kb, vc, vs, vb, kv_lens=kv_lens)
    torch.cuda.synchronize()
    got = o.float().cpu().numpy()
    ref = oracle.attention_q4(q.float().cpu().numpy(), kc.cpu().numpy(), ks.cpu().numpy(), kb.cpu().numpy(),
                              vc.cpu().numpy(), vs.cpu().numpy(), vb.cpu().numpy(),
                              kv_lens=lens, scale=D ** -0.5)["o"]
    for b in range(B):
        if lens is not None and lens[b] == 0:
            assert (got[b] == 0).all(), f"case {i}: request {b} has no keys"
            continue
        parity.check(got[b:b + 1], ref[b:b + 1], "q4", f"case {i} request {b}")


def _varlen_cases(n=12, seed=20261205):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        D = int(rng.choice([64, 128]))
        Hq, Hkv = _heads(rng)
        B = int(rng.integers(1, 7))
        kv = [int(x) for x in rng.integers(0, 1200, size=B)]
        ql = [int(rng.integers(0, k + 1)) if rng.random() < 0.7 else k for k in kv]
        causal = bool(rng.random() < 0.75)
        cases.append((i, Hq, Hkv, D, ql, kv, causal))
    return cases


@pytest.mark.parametrize("i,Hq,Hkv,D,q_lens,kv_lens,causal", _varlen_cases())
def test_prefill_varlen_random_shape(i, Hq, Hkv, D, q_lens, kv_lens, causal):
    """Per-request query and key lengths (empty requests included), NaN past
    each request's rows; rows past a request's queries keep their sentinel."""
    B = len(q_lens)
    Tq_cap, S_cap = max(max(q_lens), 1), max(max(kv_lens), 1)
    q = inputs.randn((B, Hq, Tq_cap, D), inputs.tensor_seed(400 + i, 0), torch.bfloat16, DEV)
    k = inputs.randn((B, Hkv, S_cap, D), inputs.tensor_seed(400 + i, 1), torch.bfloat16, DEV)
    v = inputs.randn((B, Hkv, S_cap, D), inputs.tensor_seed(400 + i, 2), torch.bfloat16, DEV)
    inputs.poison_tail(q, q_lens)
    inputs.poison_tail(k, kv_lens)
    inputs.poison_tail(v, kv_lens)
    o = torch.full_like(q, 3.0)
    binding.gqa_attn_prefill_varlen(q, k, v, o, torch.tensor(q_lens, dtype=torch.int32, device=DEV),
                                    torch.tensor(kv_lens, dtype=torch.int32, device=DEV), D ** -0.5, causal=causal)
    torch.cuda.synchronize()
    got = f64(o)
    for b, (qn, kn) in enumerate(zip(q_lens, kv_lens)):
        assert (got[b, :, qn:] == 3.0).all(), f"case {i} request {b}: rows past q_len were written"
        if qn == 0:
            continue
        ref = oracle.attention(f64(q[b:b + 1, :, :qn]), f64(k[b:b + 1, :, :kn]), f64(v[b:b + 1, :, :kn]),
                               scale=D ** -0.5, causal=causal)["o"]
        parity.check(got[b:b + 1, :, :qn], ref, "bf16", f"case {i} request {b}")

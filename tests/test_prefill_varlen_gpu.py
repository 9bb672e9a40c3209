"""Varlen batched prefill (each request's own query chunk, aligned to the end
of its own keys) against the oracle, one request at a time.

K/V rows past a request's kv_len and Q rows past its q_len are NaN, and O is
pre-filled with a sentinel: the rows past q_len must keep it.  Bounds of
tests/parity.py (bf16: max abs error 2e-2, and 2^-6 of each row's largest
reference value).
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


def run_varlen(q_lens, kv_lens, Hq=14, Hkv=2, causal=True, seed=0, Tq_cap=None, S_cap=None):
    B = len(q_lens)
    Tq_cap = Tq_cap or max(max(q_lens), 1)
    S_cap = S_cap or max(max(kv_lens), 1)
    q = inputs.randn((B, Hq, Tq_cap, 64), inputs.tensor_seed(seed, 0), torch.bfloat16, DEV)
    k = inputs.randn((B, Hkv, S_cap, 64), inputs.tensor_seed(seed, 1), torch.bfloat16, DEV)
    v = inputs.randn((B, Hkv, S_cap, 64), inputs.tensor_seed(seed, 2), torch.bfloat16, DEV)
    inputs.poison_tail(q, q_lens)
    inputs.poison_tail(k, kv_lens)
    inputs.poison_tail(v, kv_lens)
    o = torch.full_like(q, 3.0)
    ql = torch.tensor(q_lens, dtype=torch.int32, device=DEV)
    kl = torch.tensor(kv_lens, dtype=torch.int32, device=DEV)
    binding.gqa_attn_prefill_varlen(q, k, v, o, ql, kl, 0.125, causal=causal)
    torch.cuda.synchronize()
    got = f64(o)
    for b, (qn, kn) in enumerate(zip(q_lens, kv_lens)):
        assert (got[b, :, qn:] == 3.0).all(), f"request {b}: rows past q_len were written"
        if qn == 0:
            continue
        ref = oracle.attention(f64(q[b:b + 1, :, :qn]), f64(k[b:b + 1, :, :kn]), f64(v[b:b + 1, :, :kn]),
                               scale=0.125, causal=causal)["o"]
        parity.check(got[b:b + 1, :, :qn], ref, "bf16", f"request {b}")


MIX = ([512, 1, 129, 300, 0, 257, 64], [4096, 300, 129, 2000, 50, 257, 200])


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_varlen_mix_matches_oracle(causal):
    run_varlen(*MIX, causal=causal, seed=1)


@pytest.mark.parametrize("ks", ["1", "2", "3", "4", "5"])
def test_varlen_under_forced_kv_splits(ks):
    with binding.plan_override(prefill_kv_split=int(ks)):
        run_varlen([200, 33, 512], [3000, 700, 512], seed=2)


@pytest.mark.parametrize("Hq,Hkv", [(14, 2), (8, 8), (16, 2)])
def test_varlen_head_mappings(Hq, Hkv):
    run_varlen([128, 7], [1000, 7], Hq=Hq, Hkv=Hkv, seed=3, Tq_cap=200, S_cap=1100)


def test_varlen_uniform_equals_plain_prefill():
    """Equal lengths for every request: the same as gqa_attn_prefill run with
    pairs of query tiles only (per-request lengths always use pairs; the
    plain call's planner may run long causal tiles as single-tile units,
    which sum the same products in another order)."""
    B, q_len, kv_len = 3, 300, 900
    q = inputs.randn((B, 14, q_len, 64), 7, torch.bfloat16, DEV)
    k = inputs.randn((B, 2, kv_len, 64), 8, torch.bfloat16, DEV)
    v = inputs.randn((B, 2, kv_len, 64), 9, torch.bfloat16, DEV)
    with binding.plan_override(prefill_interleave_from=1 << 20):
        o1 = binding.prefill(q, k, v, causal=True)
    o2 = torch.empty_like(q)
    lens = lambda n: torch.full((B,), n, dtype=torch.int32, device=DEV)
    binding.gqa_attn_prefill_varlen(q, k, v, o2, lens(q_len), lens(kv_len), 0.125)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_prefill_status_word_flags_clamped_lengths():
    """In-range lengths leave the prefill status word at 0; a key length past
    S_cap or a query length past the request's keys is clamped and flagged."""
    binding.gqa_attn_clear_prefill_status()
    run_varlen(*MIX, seed=4)
    assert binding.gqa_attn_read_prefill_status() == 0
    B, S_cap, Tq_cap = 3, 256, 128
    q = inputs.randn((B, 14, Tq_cap, 64), 11, torch.bfloat16, DEV)
    k = inputs.randn((B, 2, S_cap, 64), 12, torch.bfloat16, DEV)
    v = inputs.randn((B, 2, S_cap, 64), 13, torch.bfloat16, DEV)
    o = torch.full_like(q, 3.0)
    ql = torch.tensor([100, 128, 64], dtype=torch.int32, device=DEV)
    kl = torch.tensor([256, 999, 20], dtype=torch.int32, device=DEV)  # 999 > S_cap; 64 queries > 20 keys
    binding.gqa_attn_prefill_varlen(q, k, v, o, ql, kl, 0.125)
    status = binding.gqa_attn_read_prefill_status()
    assert status & binding.GQA_DEV_KVLEN_CLAMPED
    assert not status & binding.GQA_DEV_WAIT_TIMEOUT
    # the clamped requests computed what the clamped lengths define
    got = f64(o)
    for b, (qn, kn) in enumerate([(100, 256), (128, 256), (20, 20)]):
        ref = oracle.attention(f64(q[b:b + 1, :, :qn]), f64(k[b:b + 1, :, :kn]), f64(v[b:b + 1, :, :kn]),
                               scale=0.125, causal=True)["o"]
        parity.check(got[b:b + 1, :, :qn], ref, "bf16", f"request {b}")
    assert (got[2, :, 20:] == 3.0).all()
    binding.gqa_attn_clear_prefill_status()
    assert binding.gqa_attn_read_prefill_status() == 0

"""Causal / chunked prefill on the tcgen05 tensor cores against the oracle.

bf16 Q/K/V/O, fp32 accumulation; bounds (tests/parity.py) max abs error 2e-2
and, per output row, 2^-6 of its largest reference value.  The causal
mask is aligned to the end of the keys: with q_len < kv_len (a chunk), query
row i sees keys j <= i + kv_len - q_len.  For the 16,384-token case the
oracle checks every row of two query heads, 2048 rows at a time.
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


def case(B, Hq, Hkv, q_len, kv_len, s_cap=None, layer=0):
    s_cap = kv_len if s_cap is None else s_cap
    q, _, _ = inputs.qkv(B, Hq, Hkv, 64, q_len, 1, torch.bfloat16, layer=layer, device=DEV)
    _, k, v = inputs.qkv(B, Hq, Hkv, 64, 1, s_cap, torch.bfloat16, layer=layer, device=DEV)
    return q, k, v


def check_full(q, k, v, kv_len, causal):
    o = binding.prefill(q, k, v, kv_len=kv_len, causal=causal)
    torch.cuda.synchronize()
    ref = oracle.attention(f64(q), f64(k[:, :, :kv_len]), f64(v[:, :, :kv_len]),
                           scale=0.125, causal=causal)["o"]
    parity.check(f64(o), ref, "bf16")


@pytest.mark.parametrize("T", [1, 5, 127, 128, 129, 300, 513])
def test_causal_prefill_square(T):
    q, k, v = case(1, 14, 2, T, T, layer=T)
    check_full(q, k, v, T, True)


@pytest.mark.parametrize("q_len,kv_len", [(1, 77), (64, 200), (129, 1000), (100, 128), (3, 300)])
def test_chunked_prefill_aligned_to_end(q_len, kv_len):
    q, k, v = case(1, 14, 2, q_len, kv_len, layer=q_len + kv_len)
    check_full(q, k, v, kv_len, True)


@pytest.mark.parametrize("q_len,kv_len", [(128, 128), (70, 300), (256, 1000)])
def test_non_causal_prefill(q_len, kv_len):
    q, k, v = case(1, 14, 2, q_len, kv_len, layer=7)
    check_full(q, k, v, kv_len, False)


@pytest.mark.parametrize("B,Hq,Hkv", [(2, 8, 8), (2, 32, 8), (3, 6, 1)])
def test_prefill_head_ratios_and_batch(B, Hq, Hkv):
    q, k, v = case(B, Hq, Hkv, 200, 333, layer=B)
    check_full(q, k, v, 333, True)


def test_keys_past_kv_len_are_ignored():
    q, k, v = case(1, 14, 2, 100, 250, s_cap=300, layer=11)
    k[:, :, 250:] = float("nan")
    v[:, :, 250:] = float("nan")
    check_full(q, k, v, 250, True)
    check_full(q, k, v, 250, False)


@pytest.mark.parametrize("T", [513, 2049, 4097])
def test_config_causal_prefill_qwen05b(T):
    """B=1, Hq=14, Hkv=2, D=64, bf16, q_len = kv_len = T, causal."""
    q, k, v = case(1, 14, 2, T, T, layer=T % 13)
    check_full(q, k, v, T, True)


def test_config_chunked_prefill_512_at_3584():
    """A 512-query chunk at kv offset 3584 (kv_len 4096), queries end-aligned."""
    q, k, v = case(1, 14, 2, 512, 4096, layer=5)
    check_full(q, k, v, 4096, True)


def test_config_causal_prefill_16384_two_heads_every_row():
    """Every row of query heads 0 and 13 (KV heads 0 and 1).  Rows [r0, r1)
    of a causal prefill are a chunk of r1 - r0 queries aligned to the end of
    keys [0, r1), so the oracle runs in chunks of 2048 rows."""
    T = 16384
    q, k, v = case(1, 14, 2, T, T, layer=3)
    o = binding.prefill(q, k, v, causal=True)
    torch.cuda.synchronize()
    on = f64(o)
    for h in (0, 13):
        g = h // 7
        qh, kh, vh = f64(q[:, h:h + 1]), f64(k[:, g:g + 1]), f64(v[:, g:g + 1])
        for r0 in range(0, T, 2048):
            r1 = r0 + 2048
            ref = oracle.attention(qh[:, :, r0:r1], kh[:, :, :r1], vh[:, :, :r1], scale=0.125, causal=True)["o"]
            parity.check(on[:, h:h + 1, r0:r1], ref, "bf16", f"head {h} rows {r0}..{r1}")


@pytest.mark.parametrize("causal", [True, False])
def test_growing_scores_force_rescales(causal):
    """Keys whose norm grows along the sequence make later tiles' scores
    exceed the running maximum by far more than 2^8 (in base 2), in first and
    second halves of KV tiles alike, so every rescale path of the kernel runs."""
    T = 1000
    q, k, v = case(1, 14, 2, T, T, layer=21)
    ramp = (1.0 + 6.0 * torch.arange(T, device=DEV, dtype=torch.float32) / T).view(1, 1, T, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    check_full(q, k, v, T, causal)


@pytest.mark.parametrize("ks", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("q_len,kv_len,causal", [(1100, 1100, True), (200, 3000, True), (300, 2000, False),
                                                  (129, 300, True)])
def test_kv_split_over_cluster(ks, q_len, kv_len, causal):
    """The KV range of each query-tile pair split over a cluster of ks CTAs
    (forced through the tuning override), partials merged through
    distributed shared memory; shares may be empty when ks exceeds the
    pair's KV tiles (129 queries at 300 keys: 3 tiles)."""
    q, k, v = case(1, 14, 2, q_len, kv_len, layer=ks)
    with binding.plan_override(prefill_kv_split=ks):
        check_full(q, k, v, kv_len, causal)


@pytest.mark.parametrize("from_pair", [0, 1, 2])
@pytest.mark.parametrize("q_len,kv_len,causal", [(1, 1, True), (127, 127, True), (129, 129, True), (300, 300, True),
                                                  (513, 513, True), (1000, 1000, True), (100, 150, True),
                                                  (129, 1000, True), (300, 2000, False), (256, 256, False)])
def test_single_tile_units(from_pair, q_len, kv_len, causal):
    """Pairs from `from_pair` on run as single query tiles whose KV tiles the
    two softmax warpgroups take in turn (forced through the tuning
    override); chunks whose first rows see none of the odd KV tiles (100
    queries at 150 keys) and tiles with one KV tile (no odd tiles) included."""
    q, k, v = case(1, 14, 2, q_len, kv_len, layer=from_pair + 3)
    with binding.plan_override(prefill_interleave_from=from_pair):
        check_full(q, k, v, kv_len, causal)


@pytest.mark.parametrize("causal", [True, False])
def test_single_tile_units_rescale(causal):
    """Growing key norms force rescales in both slots of single-tile units."""
    T = 1000
    q, k, v = case(1, 14, 2, T, T, layer=22)
    ramp = (1.0 + 6.0 * torch.arange(T, device=DEV, dtype=torch.float32) / T).view(1, 1, T, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    with binding.plan_override(prefill_interleave_from=0):
        check_full(q, k, v, T, causal)


def test_single_tile_units_equal_pairs_bit_for_bit_where_slot_one_is_empty():
    """A tile with a single KV tile gives slot 1 nothing to do: its single-tile
    unit must then reproduce the pair result exactly (same products, same
    order, weight 1 for slot 0)."""
    q, k, v = case(1, 14, 2, 100, 100, layer=9)
    o_pair = binding.prefill(q, k, v)
    with binding.plan_override(prefill_interleave_from=0):
        o_single = binding.prefill(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o_pair, o_single)


@pytest.mark.parametrize("q_len,kv_len", [(300, 300), (512, 4096)])
def test_back_to_back_calls_read_the_previous_output(q_len, kv_len):
    """Launches wait for the grid before them (programmatic dependent launch):
    a second call whose queries are the first call's output, issued on the
    same stream with no synchronisation in between, must see that output
    complete.  (512 queries at 4096 keys takes the cluster-split path.)"""
    q, k, v = case(1, 14, 2, q_len, kv_len, layer=11)
    _, k2, v2 = case(1, 14, 2, q_len, kv_len, layer=12)
    o1 = binding.prefill(q, k, v)
    o2 = binding.prefill(o1, k2, v2)
    torch.cuda.synchronize()
    ref1 = oracle.attention(f64(q), f64(k), f64(v), scale=0.125, causal=True)["o"]
    parity.check(f64(o1), ref1, "bf16", "first call")
    ref2 = oracle.attention(f64(o1), f64(k2), f64(v2), scale=0.125, causal=True)["o"]
    parity.check(f64(o2), ref2, "bf16", "second call")

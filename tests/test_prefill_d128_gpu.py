"""Prefill at head dimension 128 against the oracle.

At D = 128 the kernel loads Q, K and V tiles as two 64-column boxes, runs
eight 16-deep slices per score product and two 64-column halves per P.V
product, and writes P over the first half of the S columns in tensor memory
(so the next score product of a tile waits for the P.V product before it).
The cases are those of the D = 64 tests at the 7B (28/4) and Qwen3-4B (32/8)
head geometries: ragged tails, chunks aligned to the end of the keys, full
attention, keys past kv_len poisoned with NaN, growing scores that force
every rescale, every cluster size of the KV split, per-request lengths and
back-to-back calls.  Bounds of tests/parity.py for bf16 (max abs error 2e-2,
and 2^-6 of each row's largest reference value).
"""

import pytest
import torch

import oracle
import parity
from gqa_attention_kv_decode_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128
SCALE = D ** -0.5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def f64(t):
    return t.detach().float().cpu().numpy()


def case(B, Hq, Hkv, q_len, kv_len, s_cap=None, layer=0):
    s_cap = kv_len if s_cap is None else s_cap
    q, _, _ = inputs.qkv(B, Hq, Hkv, D, q_len, 1, torch.bfloat16, layer=layer, device=DEV)
    _, k, v = inputs.qkv(B, Hq, Hkv, D, 1, s_cap, torch.bfloat16, layer=layer, device=DEV)
    return q, k, v


def check_full(q, k, v, kv_len, causal, heads=None):
    o = binding.prefill(q, k, v, kv_len=kv_len, causal=causal)
    torch.cuda.synchronize()
    n_rep = q.shape[1] // k.shape[1]
    for h in (range(q.shape[1]) if heads is None else heads):
        g = h // n_rep
        ref = oracle.attention(f64(q[:, h:h + 1]), f64(k[:, g:g + 1, :kv_len]), f64(v[:, g:g + 1, :kv_len]),
                               scale=SCALE, causal=causal)["o"]
        parity.check(f64(o[:, h:h + 1]), ref, "bf16", f"head {h}")


@pytest.mark.parametrize("T", [1, 5, 127, 128, 129, 300, 513])
def test_causal_prefill_square_7b_heads(T):
    q, k, v = case(1, 28, 4, T, T, layer=T)
    check_full(q, k, v, T, True)


@pytest.mark.parametrize("q_len,kv_len", [(1, 77), (64, 200), (129, 1000), (100, 128), (3, 300)])
def test_chunked_prefill_aligned_to_end(q_len, kv_len):
    q, k, v = case(1, 28, 4, q_len, kv_len, layer=q_len + kv_len)
    check_full(q, k, v, kv_len, True)


@pytest.mark.parametrize("q_len,kv_len", [(128, 128), (70, 300), (256, 1000)])
def test_non_causal_prefill(q_len, kv_len):
    q, k, v = case(1, 32, 8, q_len, kv_len, layer=7)
    check_full(q, k, v, kv_len, False)


@pytest.mark.parametrize("B,Hq,Hkv", [(2, 32, 8), (3, 6, 1), (2, 8, 8)])
def test_prefill_head_ratios_and_batch(B, Hq, Hkv):
    q, k, v = case(B, Hq, Hkv, 200, 333, layer=B)
    check_full(q, k, v, 333, True)


def test_keys_past_kv_len_are_ignored():
    q, k, v = case(1, 28, 4, 100, 250, s_cap=300, layer=11)
    k[:, :, 250:] = float("nan")
    v[:, :, 250:] = float("nan")
    check_full(q, k, v, 250, True)
    check_full(q, k, v, 250, False)


def test_causal_prefill_4097_7b_one_head_per_kv_head():
    """7B head geometry at 4,097 tokens: every row of query heads 0, 9, 18
    and 27 (KV heads 0 to 3)."""
    T = 4097
    q, k, v = case(1, 28, 4, T, T, layer=4)
    check_full(q, k, v, T, True, heads=(0, 9, 18, 27))


def test_causal_prefill_16384_7b_two_heads_every_row():
    """Every row of query heads 0 and 27 (KV heads 0 and 3).  Rows [r0, r1)
    of a causal prefill are a chunk of r1 - r0 queries aligned to the end of
    keys [0, r1), so the oracle runs in chunks of 2048 rows."""
    T = 16384
    q, k, v = case(1, 28, 4, T, T, layer=3)
    o = binding.prefill(q, k, v, causal=True)
    torch.cuda.synchronize()
    on = f64(o)
    for h in (0, 27):
        g = h // 7
        qh, kh, vh = f64(q[:, h:h + 1]), f64(k[:, g:g + 1]), f64(v[:, g:g + 1])
        for r0 in range(0, T, 2048):
            r1 = r0 + 2048
            ref = oracle.attention(qh[:, :, r0:r1], kh[:, :, :r1], vh[:, :, :r1], scale=SCALE, causal=True)["o"]
            parity.check(on[:, h:h + 1, r0:r1], ref, "bf16", f"head {h} rows {r0}..{r1}")


def test_chunked_prefill_512_at_3584_7b():
    q, k, v = case(1, 28, 4, 512, 4096, layer=5)
    check_full(q, k, v, 4096, True)


@pytest.mark.parametrize("causal", [True, False])
def test_growing_scores_force_rescales(causal):
    T = 1000
    q, k, v = case(1, 28, 4, T, T, layer=21)
    ramp = (1.0 + 6.0 * torch.arange(T, device=DEV, dtype=torch.float32) / T).view(1, 1, T, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    check_full(q, k, v, T, causal)


@pytest.mark.parametrize("ks", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("q_len,kv_len,causal", [(1100, 1100, True), (200, 3000, True), (300, 2000, False),
                                                  (129, 300, True)])
def test_kv_split_over_cluster(ks, q_len, kv_len, causal):
    """Cluster sizes 6 and 7 do not fit the exchange at D = 128 and run as 5."""
    q, k, v = case(1, 28, 4, q_len, kv_len, layer=ks)
    with binding.plan_override(prefill_kv_split=ks):
        check_full(q, k, v, kv_len, causal)


@pytest.mark.parametrize("from_pair", [0, 2])
@pytest.mark.parametrize("q_len,kv_len,causal", [(129, 129, True), (513, 513, True), (100, 150, True),
                                                  (300, 2000, False)])
def test_single_tile_units(from_pair, q_len, kv_len, causal):
    q, k, v = case(1, 28, 4, q_len, kv_len, layer=from_pair + 5)
    with binding.plan_override(prefill_interleave_from=from_pair):
        check_full(q, k, v, kv_len, causal)


def test_back_to_back_calls_read_the_previous_output():
    q, k, v = case(1, 28, 4, 512, 4096, layer=11)
    _, k2, v2 = case(1, 28, 4, 512, 4096, layer=12)
    o1 = binding.prefill(q, k, v)
    o2 = binding.prefill(o1, k2, v2)
    torch.cuda.synchronize()
    ref1 = oracle.attention(f64(q), f64(k), f64(v), scale=SCALE, causal=True)["o"]
    parity.check(f64(o1), ref1, "bf16", "first call")
    ref2 = oracle.attention(f64(o1), f64(k2), f64(v2), scale=SCALE, causal=True)["o"]
    parity.check(f64(o2), ref2, "bf16", "second call")


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_varlen_mix(causal):
    """Per-request lengths with NaN past each request's rows; O rows past a
    request's queries keep their sentinel."""
    q_lens, kv_lens = [512, 1, 129, 300, 0, 257], [4096, 300, 129, 2000, 50, 257]
    B, Hq, Hkv = len(q_lens), 28, 4
    Tq_cap, S_cap = max(q_lens), max(kv_lens)
    q = inputs.randn((B, Hq, Tq_cap, D), inputs.tensor_seed(31, 0), torch.bfloat16, DEV)
    k = inputs.randn((B, Hkv, S_cap, D), inputs.tensor_seed(31, 1), torch.bfloat16, DEV)
    v = inputs.randn((B, Hkv, S_cap, D), inputs.tensor_seed(31, 2), torch.bfloat16, DEV)
    inputs.poison_tail(q, q_lens)
    inputs.poison_tail(k, kv_lens)
    inputs.poison_tail(v, kv_lens)
    o = torch.full_like(q, 3.0)
    ql = torch.tensor(q_lens, dtype=torch.int32, device=DEV)
    kl = torch.tensor(kv_lens, dtype=torch.int32, device=DEV)
    binding.gqa_attn_prefill_varlen(q, k, v, o, ql, kl, SCALE, causal=causal)
    torch.cuda.synchronize()
    got = f64(o)
    for b, (qn, kn) in enumerate(zip(q_lens, kv_lens)):
        assert (got[b, :, qn:] == 3.0).all(), f"request {b}: rows past q_len were written"
        if qn == 0:
            continue
        ref = oracle.attention(f64(q[b:b + 1, :, :qn]), f64(k[b:b + 1, :, :kn]), f64(v[b:b + 1, :, :kn]),
                               scale=SCALE, causal=causal)["o"]
        parity.check(got[b:b + 1, :, :qn], ref, "bf16", f"request {b}")


def test_status_stays_clear():
    binding.gqa_attn_clear_prefill_status()
    q, k, v = case(1, 28, 4, 300, 300, layer=2)
    binding.prefill(q, k, v)
    assert binding.gqa_attn_read_prefill_status() == 0

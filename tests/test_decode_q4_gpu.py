"""4-bit group-affine decode on the GPU against the fp64 oracle.

The oracle dequantises the stored codes explicitly (x = code*scale + bias)
and attends; the kernel never materialises that copy.  Both read the same
codes, scales and biases, so the comparison is independent of how the cache
was quantized.  Bounds (tests/parity.py): max abs error 2e-2 (bf16 q and
output, fp32 accumulation) and, per output row, 2^-5 of the row's largest
reference value.  Scales and biases of rows past kv_len are NaN: a kernel that
reads them into the result fails.
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


def make_case(B, Hq, Hkv, D, S_cap, layer=0, poison_lens=None):
    kc, ks, kb, vc, vs, vb = inputs.q4_cache(B, Hkv, D, S_cap, layer=layer, device=DEV)
    q = inputs.randn((B, Hq, 1, D), inputs.tensor_seed(layer, 0), torch.bfloat16, DEV)
    if poison_lens is not None:
        for t in (ks, kb, vs, vb):
            inputs.poison_tail(t, poison_lens)
    return q, (kc, ks, kb, vc, vs, vb)


def oracle_o(q, cache, kv_lens, D):
    kc, ks, kb, vc, vs, vb = (t.cpu().numpy() for t in cache)
    return oracle.attention_q4(q.float().cpu().numpy(), kc, ks, kb, vc, vs, vb,
                               kv_lens=kv_lens, scale=D ** -0.5)["o"]


def run(q, cache, kv_lens=None, max_kv_len=None):
    lens_t = None if kv_lens is None else torch.tensor(kv_lens, dtype=torch.int32, device=DEV)
    o = binding.decode_q4(q, *cache, kv_lens=lens_t, max_kv_len=max_kv_len)
    torch.cuda.synchronize()
    return o


HEADS = [(32, 8), (14, 2), (8, 8), (16, 2), (12, 4), (24, 2)]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", HEADS, ids=[f"{a}x{b}" for a, b in HEADS])
@pytest.mark.parametrize("S", [8, 64, 200, 2048])
def test_q4_decode_matches_oracle(D, Hq, Hkv, S):
    q, cache = make_case(2, Hq, Hkv, D, S, layer=S % 97)
    o = run(q, cache)
    ref = oracle_o(q, cache, [S, S], D)
    parity.check(o.float().cpu().numpy(), ref, "q4")


def test_q4_ragged_with_poisoned_tails():
    kv_lens = [1, 64, 333, 1000, 65, 8]
    q, cache = make_case(len(kv_lens), 32, 8, 128, 1024, layer=4, poison_lens=kv_lens)
    o = run(q, cache, kv_lens=kv_lens, max_kv_len=1000)
    parity.check(o.float().cpu().numpy(), oracle_o(q, cache, kv_lens, 128), "q4")


@pytest.mark.parametrize("splits", ["1", "5", "64"])
def test_q4_forced_split_counts(splits):
    q, cache = make_case(2, 32, 8, 128, 4096, layer=9)
    with binding.plan_override(decode_splits=int(splits)):
        o = run(q, cache, kv_lens=[4096, 1500])
    parity.check(o.float().cpu().numpy(), oracle_o(q, cache, [4096, 1500], 128), "q4")


def test_q4_rejects_unaligned_capacity():
    q, cache = make_case(1, 32, 8, 128, 8)
    kc, ks, kb, vc, vs, vb = cache
    o = torch.empty_like(q)
    ws = binding.decode_q4_workspace(1, 32, 8, 128, 8)
    with pytest.raises(binding.GqaAttnError) as e:   # S_cap = 6 is not a multiple of 8
        binding.gqa_attn_decode_q4(q, kc[:, :, :6].contiguous(), ks[:, :, :6].contiguous(),
                                   kb[:, :, :6].contiguous(), vc[:, :, :6].contiguous(),
                                   vs[:, :, :6].contiguous(), vb[:, :, :6].contiguous(), o, None,
                                   0.1, ws)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG


@pytest.mark.parametrize("S", [64, 2048, 16384])
def test_config_qwen3_4b_q4_36_layers(S):
    """Hq=32, Hkv=8, D=128, B=4, q4 cache, 36 layer calls; all four requests
    of four sampled layers checked."""
    ws = binding.decode_q4_workspace(4, 32, 8, 128, S)
    rng = np.random.default_rng(S)
    check = sorted(set([0, 35] + list(rng.choice(36, 2, replace=False))))
    for l in range(36):
        q, cache = make_case(4, 32, 8, 128, S, layer=l)
        o = binding.decode_q4(q, *cache, workspace=ws)
        if l in check:
            torch.cuda.synchronize()
            ref = oracle_o(q, cache, [S] * 4, 128)
            parity.check(o.float().cpu().numpy(), ref, "q4", f"layer {l}")


@pytest.mark.parametrize("mag", [1e-3, 1e4, 1e6], ids=["small", "1e4", "1e6"])
def test_q4_query_range(mag):
    """q enters the score product as fp16, so a q with elements of 2^14 or
    more is scaled by 2^-e inside the kernel and the scores by 2^e after.
    Here q is multiplied by mag and the softmax scale divided by it, so the
    scores keep their usual size while q spans fp16's range and beyond (e = 2
    and 6 for 1e4 and 1e6; a small q takes no scaling)."""
    B, Hq, Hkv, D, S = 2, 32, 8, 128, 1000
    q, cache = make_case(B, Hq, Hkv, D, S, layer=71)
    q = (q.float() * mag).to(torch.bfloat16)
    lens_t = torch.tensor([S, 377], dtype=torch.int32, device=DEV)
    o = binding.decode_q4(q, *cache, kv_lens=lens_t, scale=D ** -0.5 / mag)
    torch.cuda.synchronize()
    kc, ks, kb, vc, vs, vb = (t.cpu().numpy() for t in cache)
    ref = oracle.attention_q4(q.float().cpu().numpy(), kc, ks, kb, vc, vs, vb, kv_lens=[S, 377],
                              scale=D ** -0.5 / mag)["o"]
    parity.check(o.float().cpu().numpy(), ref, "q4")

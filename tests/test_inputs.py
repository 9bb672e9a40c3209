"""The seeded input builders the GPU tests and the bench share (CPU only).

They hold no attention arithmetic, but every parity test trusts them: the
draws must be reproducible and distinct per layer and tensor, the NaN tails
must cover exactly the rows past each length, the paged pool must hold every
valid row where its block table says (each block used once, spare and tail
rows NaN), and the 4-bit cache they build must be the encoding the oracle
defines.
"""

import numpy as np
import pytest
import torch

import oracle
from gqa_attention_kv_decode_gb300 import inputs


def test_draws_are_reproducible_and_distinct():
    a = inputs.qkv(2, 4, 2, 64, 1, 50, torch.float32, layer=3)
    b = inputs.qkv(2, 4, 2, 64, 1, 50, torch.float32, layer=3)
    c = inputs.qkv(2, 4, 2, 64, 1, 50, torch.float32, layer=4)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    for x, y in zip(a, c):
        assert not torch.equal(x, y)
    q, k, v = a
    assert not torch.equal(k, v), "K and V come from different seeds"
    assert inputs.tensor_seed(3, 1) == inputs.BASE_SEED + 3001


def test_bf16_draws_are_the_rounded_fp32_draws():
    x32 = inputs.randn((3, 100), 77, torch.float32)
    x16 = inputs.randn((3, 100), 77, torch.bfloat16)
    assert torch.equal(x32.to(torch.bfloat16), x16)


def test_ragged_lengths_stay_in_range():
    for B, lo, hi, seed in ((1, 64, 8192, 1), (64, 64, 8192, 2), (16, 512, 8192, 3)):
        lens = inputs.ragged_kv_lens(B, lo, hi, seed)
        assert lens.dtype == np.int32 and lens.shape == (B,)
        assert (lens >= lo).all() and (lens <= hi).all()
        assert (lens == inputs.ragged_kv_lens(B, lo, hi, seed)).all()


def test_poison_tail_covers_exactly_the_rows_past_each_length():
    x = torch.zeros(3, 2, 10, 4)
    lens = [10, 3, 0]
    inputs.poison_tail(x, lens)
    for b, L in enumerate(lens):
        assert not torch.isnan(x[b, :, :L]).any()
        assert torch.isnan(x[b, :, L:]).all()


@pytest.mark.parametrize("block_size", [16, 64])
def test_paged_pool_places_every_valid_row_where_the_table_says(block_size):
    B, Hkv, S, D = 3, 2, 150, 8
    lens = [150, 37, 1]
    k = inputs.randn((B, Hkv, S, D), 5, torch.float32)
    v = inputs.randn((B, Hkv, S, D), 6, torch.float32)
    kp, vp, table = inputs.paged_pool(k, v, lens, block_size, seed=9)
    nb = -(-S // block_size)
    assert table.shape == (B, nb) and table.dtype == torch.int32
    ids = table.flatten().tolist()
    assert len(set(ids)) == len(ids), "each block belongs to one request once"
    assert all(0 <= i < kp.shape[0] for i in ids)
    for b, L in enumerate(lens):
        for j in range(S):
            blk, r = int(table[b, j // block_size]), j % block_size
            if j < L:
                assert torch.equal(kp[blk, :, r], k[b, :, j]) and torch.equal(vp[blk, :, r], v[b, :, j])
            else:
                assert torch.isnan(kp[blk, :, r]).all() and torch.isnan(vp[blk, :, r]).all()
    spare = sorted(set(range(kp.shape[0])) - set(ids))
    assert len(spare) == 3 and torch.isnan(kp[spare]).all()


def test_builder_encoding_is_the_oracle_encoding():
    """The 4-bit caches the GPU tests feed the kernels are the oracle's
    encoding of the same bf16 data: codes, scales and biases identical."""
    x = inputs.randn((2, 3, 70, 128), 11, torch.bfloat16)
    c, s, b = inputs.quantize_q4(x)
    oc, os_, ob = oracle.quantize_q4(x.float().numpy())
    assert np.array_equal(c.numpy(), oc)
    assert np.array_equal(s.numpy(), os_)
    assert np.array_equal(b.numpy(), ob)

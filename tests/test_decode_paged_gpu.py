"""Paged-cache decode (block table, optional fused append) on the GPU against
the fp64 oracle.

The pools hold every request's blocks in a seeded random order, spare blocks
and every row past kv_len are NaN, and the appended token's slot starts as
NaN: a kernel that reads a row it should not, or misses the append, fails.
Bounds as for contiguous decode (tests/parity.py: absolute and row-scaled); the
pool rows written by the append must equal the new token bit for bit.
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


def make(B, Hq, Hkv, D, S, kv_lens, dtype, block_size, seed, append):
    q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, S, dtype, layer=seed, device=DEV)
    kn = vn = None
    if append:
        kn = inputs.randn((B, Hkv, 1, D), inputs.tensor_seed(seed, 3), dtype, DEV)
        vn = inputs.randn((B, Hkv, 1, D), inputs.tensor_seed(seed, 4), dtype, DEV)
        # the slot of the new token holds garbage (NaN) before the call
        prior = [max(0, L - 1) for L in kv_lens]
    else:
        prior = kv_lens
    kp, vp, table = inputs.paged_pool(k, v, prior, block_size, seed)
    return q, kp, vp, table, kn, vn


def run_and_check(q, kp, vp, table, kn, vn, kv_lens, max_kv_len, block_size):
    D = q.shape[-1]
    ref = oracle.attention_paged(f64(q), f64(kp), f64(vp), table.cpu().numpy(), kv_lens, block_size,
                                 scale=D ** -0.5, k_new=None if kn is None else f64(kn),
                                 v_new=None if vn is None else f64(vn))
    lens_t = torch.tensor(kv_lens, dtype=torch.int32, device=DEV)
    o = binding.decode_paged(q, kp, vp, table, lens_t, max_kv_len, k_new=kn, v_new=vn)
    torch.cuda.synchronize()
    got = f64(o)
    err = parity.check(got, ref["o"], parity.kind_of(q.dtype))
    if kn is not None:  # the pools now hold the new tokens at row kv_len - 1
        for b, L in enumerate(kv_lens):
            if L == 0:
                continue
            blk = int(table[b, (L - 1) // block_size])
            r = (L - 1) % block_size
            assert torch.equal(kp[blk, :, r], kn[b, :, 0])
            assert torch.equal(vp[blk, :, r], vn[b, :, 0])
    return err


CASES = [(torch.float32, 128, 64), (torch.float32, 64, 128), (torch.bfloat16, 128, 64),
         (torch.bfloat16, 64, 64), (torch.bfloat16, 128, 256), (torch.float32, 128, 128)]


@pytest.mark.parametrize("dtype,D,block_size", CASES, ids=[f"{str(d)[6:]}-D{D}-bs{bs}" for d, D, bs in CASES])
@pytest.mark.parametrize("append", [False, True], ids=["read", "append"])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (28, 4), (14, 2), (8, 8)], ids=["32x8", "28x4", "14x2", "8x8"])
def test_paged_decode_matches_oracle(dtype, D, block_size, append, Hq, Hkv):
    S = 1000
    kv_lens = [1000, 1, block_size, block_size + 1, 333]
    q, kp, vp, table, kn, vn = make(len(kv_lens), Hq, Hkv, D, S, kv_lens, dtype, block_size, 7, append)
    run_and_check(q, kp, vp, table, kn, vn, kv_lens, S, block_size)


@pytest.mark.parametrize("splits", ["1", "3", "7", "40"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_paged_append_under_forced_split_counts(splits, dtype):
    """The CTA that owns the appended row depends on the split count."""
    kv_lens = [3000, 1500, 65, 64, 129]
    q, kp, vp, table, kn, vn = make(len(kv_lens), 28, 4, 128, 3000, kv_lens, dtype, 64, 11, True)
    with binding.plan_override(decode_splits=int(splits)):
        run_and_check(q, kp, vp, table, kn, vn, kv_lens, 3000, 64)


def test_paged_qwen3_4b_ragged_B16_bf16():
    """Qwen3-4B head geometry, 16 requests with lengths uniform in [64, 8192], append."""
    kv_lens = [int(x) for x in inputs.ragged_kv_lens(16, 64, 8192, 5)]
    q, kp, vp, table, kn, vn = make(16, 32, 8, 128, 8192, kv_lens, torch.bfloat16, 64, 5, True)
    run_and_check(q, kp, vp, table, kn, vn, kv_lens, 8192, 64)


def test_paged_bad_block_id_is_reported_and_stays_in_the_pool():
    kv_lens = [500, 700]
    q, kp, vp, table, kn, vn = make(2, 28, 4, 128, 700, kv_lens, torch.bfloat16, 64, 13, False)
    table[0, 3] = kp.shape[0] + 5  # request 0 points past the pool
    ws = binding.decode_workspace(2, 28, 4, 128, 700, binding.GQA_BF16, DEV)
    lens_t = torch.tensor(kv_lens, dtype=torch.int32, device=DEV)
    o = binding.decode_paged(q, kp, vp, table, lens_t, 700, workspace=ws)
    status = binding.gqa_attn_read_device_status(ws)
    assert status & binding.GQA_DEV_BAD_BLOCK
    ref = oracle.attention_paged(f64(q[1:]), f64(kp), f64(vp), table[1:].cpu().numpy(), kv_lens[1:], 64,
                                 scale=128 ** -0.5)
    parity.check(f64(o[1:]), ref["o"], "bf16", "the other request is intact")


def test_paged_rejects_unsupported_block_size():
    q, kp, vp, table, kn, vn = make(1, 8, 8, 64, 128, [128], torch.float32, 64, 3, False)
    lens_t = torch.tensor([128], dtype=torch.int32, device=DEV)
    with pytest.raises(binding.GqaAttnError) as e:  # fp32 with D = 64 needs a multiple of 128
        binding.decode_paged(q, kp, vp, table, lens_t, 128)
    assert e.value.status == binding.GQA_ERR_UNSUPPORTED

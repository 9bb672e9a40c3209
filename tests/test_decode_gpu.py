"""Split-KV decode on the GPU against the fp64 oracle, element by element.

Bounds (tests/parity.py): max abs error 1e-4 for fp32 Q/K/V/O and 2e-2 for
bf16 with fp32 accumulation, and per output row an error scaled to the
row's largest reference value (2^-16 fp32, 2^-6 bf16).  Lengths, head mapping and tails must be exact: rows past
kv_len are filled with NaN, so a kernel that reads them (instead of skipping
them) fails.
"""

import os

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


def run_decode(q, k, v, kv_lens=None, max_kv_len=None, scale=None):
    lens_t = None if kv_lens is None else torch.tensor(kv_lens, dtype=torch.int32, device=DEV)
    o = binding.decode(q, k, v, kv_lens=lens_t, scale=scale, max_kv_len=max_kv_len)
    torch.cuda.synchronize()
    return o


def check(q, k, v, o, kv_lens=None, scale=None):
    D = q.shape[-1]
    scale = D ** -0.5 if scale is None else scale
    ref = oracle.attention(f64(q), f64(k), f64(v), kv_lens=kv_lens, scale=scale)["o"]
    return parity.check(f64(o), ref, parity.kind_of(q.dtype))


HEADS = [(14, 2), (28, 4), (32, 8), (8, 8), (6, 3), (12, 4), (10, 2), (16, 2), (24, 2), (32, 2)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", HEADS, ids=[f"{a}x{b}" for a, b in HEADS])
@pytest.mark.parametrize("S", [1, 37, 128, 1000])
def test_decode_matches_oracle(dtype, D, Hq, Hkv, S):
    q, k, v = inputs.qkv(2, Hq, Hkv, D, 1, S, dtype, layer=S, device=DEV)
    o = run_decode(q, k, v)
    check(q, k, v, o)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_ragged_batch_with_poisoned_tails(dtype):
    kv_lens = [1, 64, 333, 700, 65, 129]
    B, Hq, Hkv, D, S_cap = len(kv_lens), 32, 8, 128, 768
    q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, S_cap, dtype, layer=3, device=DEV)
    inputs.poison_tail(k, kv_lens)
    inputs.poison_tail(v, kv_lens)
    o = run_decode(q, k, v, kv_lens=kv_lens, max_kv_len=700)
    check(q, k, v, o, kv_lens=kv_lens)


@pytest.mark.parametrize("splits", ["1", "3", "16", "1000"])
def test_forced_split_counts(splits):
    q, k, v = inputs.qkv(2, 28, 4, 128, 1, 1000, torch.float32, layer=5, device=DEV)
    with binding.plan_override(decode_splits=int(splits)):
        o = run_decode(q, k, v, kv_lens=[1000, 517])
    check(q, k, v, o, kv_lens=[1000, 517])


def test_same_call_twice_is_bit_identical():
    q, k, v = inputs.qkv(3, 28, 4, 128, 1, 3000, torch.bfloat16, layer=6, device=DEV)
    ws = binding.decode_workspace(3, 28, 4, 128, 3000, binding.GQA_BF16)
    a = binding.decode(q, k, v, workspace=ws)
    b = binding.decode(q, k, v, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert binding.gqa_attn_decode_num_splits(3, 28, 4, 128, 3000, binding.GQA_BF16) > 1


def test_empty_and_out_of_range_lengths_set_status():
    B, Hq, Hkv, D, S = 4, 8, 2, 64, 100
    q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, S, torch.float32, layer=7, device=DEV)
    ws = binding.decode_workspace(B, Hq, Hkv, D, S, binding.GQA_F32)
    lens = torch.tensor([0, 100, 150, -3], dtype=torch.int32, device=DEV)
    o = torch.full_like(q, 7.0)
    binding.gqa_attn_decode(q, k, v, o, lens, D ** -0.5, ws, max_kv_len=S)
    status = binding.gqa_attn_read_device_status(ws)
    assert status & binding.GQA_DEV_EMPTY_REQUEST
    assert status & binding.GQA_DEV_KVLEN_CLAMPED
    assert not status & binding.GQA_DEV_WAIT_TIMEOUT
    got = f64(o)
    assert (got[0] == 0).all() and (got[3] == 0).all()     # 0 and -3 -> empty
    ref = oracle.attention(f64(q), f64(k), f64(v), kv_lens=[0, 100, 100, 0], scale=D ** -0.5)["o"]
    parity.check(got, ref, "f32", "150 clamped to max_kv_len")
    binding.gqa_attn_clear_device_status(ws)
    assert binding.gqa_attn_read_device_status(ws) == 0


def test_host_pointers_are_rejected():
    q, k, v = inputs.qkv(1, 14, 2, 64, 1, 128, torch.float32)   # CPU tensors
    o = torch.empty_like(q)
    ws = binding.decode_workspace(1, 14, 2, 64, 128, binding.GQA_F32)
    with pytest.raises(binding.GqaAttnError) as e:
        binding.gqa_attn_decode(q, k, v, o, None, 0.125, ws)
    assert e.value.status == binding.GQA_ERR_NOT_DEVICE_PTR


def test_small_workspace_is_rejected():
    q, k, v = inputs.qkv(1, 14, 2, 64, 1, 128, torch.float32, device=DEV)
    o = torch.empty_like(q)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    with pytest.raises(binding.GqaAttnError) as e:
        binding.gqa_attn_decode(q, k, v, o, None, 0.125, ws)
    assert e.value.status == binding.GQA_ERR_WORKSPACE


def test_config_single_layer_qwen05b():
    """B=1, Hq=14, Hkv=2, D=64, kv_len=128, fp32, scale 1/8."""
    q, k, v = inputs.qkv(1, 14, 2, 64, 1, 128, torch.float32, device=DEV)
    o = run_decode(q, k, v, scale=0.125)
    check(q, k, v, o, scale=0.125)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("S", [128, 256, 512, 1024, 2048, 4096, 32768])
def test_config_qwen7b_28_layers(dtype, S):
    """28 layer calls on distinct buffers (the bench's launch configuration);
    layers 0 and 27 checked in full, the others on two sampled KV heads."""
    layers = []
    for l in range(28):
        layers.append(inputs.qkv(1, 28, 4, 128, 1, S, dtype, layer=l, device=DEV))
    ws = binding.decode_workspace(1, 28, 4, 128, S, binding._dtype_code(layers[0][0]))
    outs = [binding.decode(q, k, v, workspace=ws) for q, k, v in layers]
    torch.cuda.synchronize()
    rng = np.random.default_rng(S)
    for l in range(28):
        q, k, v = layers[l]
        if l in (0, 27):
            check(q, k, v, outs[l])
            continue
        for g in rng.choice(4, 2, replace=False):
            hs = slice(7 * g, 7 * g + 7)
            ref = oracle.attention(f64(q[:, hs]), f64(k[:, g:g + 1]), f64(v[:, g:g + 1]),
                                   scale=128 ** -0.5)["o"]
            parity.check(f64(outs[l][:, hs]), ref, parity.kind_of(dtype), f"layer {l} group {g}")


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16, 64])
def test_config_qwen3_4b_ragged_36_layers(B):
    """Hq=32, Hkv=8, D=128, bf16, lengths uniform in [64, 8192], 36 layers;
    every request of four sampled layers checked against the oracle."""
    kv_lens = inputs.ragged_kv_lens(B, 64, 8192, seed=inputs.BASE_SEED + B)
    lens_t = torch.from_numpy(kv_lens).to(DEV)
    ws = binding.decode_workspace(B, 32, 8, 128, 8192, binding.GQA_BF16)
    rng = np.random.default_rng(B)
    check_layers = sorted(set([0, 35] + list(rng.choice(36, 2, replace=False))))
    for l in range(36):
        q, k, v = inputs.qkv(B, 32, 8, 128, 1, 8192, torch.bfloat16, layer=l, device=DEV)
        o = binding.decode(q, k, v, kv_lens=lens_t, max_kv_len=8192, workspace=ws)
        if l not in check_layers:
            continue
        torch.cuda.synchronize()
        for b in range(B):
            L = int(kv_lens[b])
            ref = oracle.attention(f64(q[b:b + 1]), f64(k[b:b + 1, :, :L]), f64(v[b:b + 1, :, :L]),
                                   scale=128 ** -0.5)["o"]
            parity.check(f64(o[b:b + 1]), ref, "bf16", f"layer {l} request {b}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_back_to_back_calls_read_the_previous_output(dtype):
    """Each call waits for the grid before it (programmatic dependent launch;
    only an L2 prefetch of q runs earlier): a second call whose query is the
    first call's output, on the same stream with no synchronisation and a
    shared workspace, must see that output complete."""
    q, k, v = inputs.qkv(1, 28, 4, 128, 1, 4096, dtype, layer=21, device=DEV)
    _, k2, v2 = inputs.qkv(1, 28, 4, 128, 1, 4096, dtype, layer=22, device=DEV)
    ws = binding.decode_workspace(1, 28, 4, 128, 4096, binding._dtype_code(q), q.device)
    o1 = binding.decode(q, k, v, workspace=ws)
    o2 = binding.decode(o1, k2, v2, workspace=ws)
    torch.cuda.synchronize()
    ref2 = oracle.attention(f64(o1), f64(k2), f64(v2), scale=128 ** -0.5)["o"]
    parity.check(f64(o2), ref2, parity.kind_of(dtype))

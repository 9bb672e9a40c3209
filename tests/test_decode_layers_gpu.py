"""Cross-layer batched decode (one launch over n_layers stacked layers): bit
for bit equal to one gqa_attn_decode call per layer, and to the oracle
within the decode tolerances."""

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


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("NL,B,S,ragged", [(1, 2, 128, False), (3, 2, 1000, True), (28, 1, 300, False),
                                           (5, 3, 4096, True)])
def test_layers_equal_per_layer_calls(dtype, D, NL, B, S, ragged):
    Hq, Hkv = 28, 4
    q = inputs.randn((NL, B, Hq, 1, D), 31, dtype, DEV)
    k = inputs.randn((NL, B, Hkv, S, D), 32, dtype, DEV)
    v = inputs.randn((NL, B, Hkv, S, D), 33, dtype, DEV)
    lens = [S, max(1, S // 3), 7][:B] if ragged else None
    lens_t = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=DEV)
    dc = binding._dtype_code(q)
    ws = torch.zeros(binding.gqa_attn_decode_layers_workspace_size(NL, B, Hq, Hkv, D, S, dc), dtype=torch.uint8,
                     device=DEV)
    o = torch.empty_like(q)
    binding.gqa_attn_decode_layers(q, k, v, o, lens_t, D ** -0.5, ws)
    ws1 = binding.decode_workspace(B, Hq, Hkv, D, S, dc, DEV)
    for l in range(NL):
        o1 = torch.empty_like(q[l])
        binding.gqa_attn_decode(q[l], k[l], v[l], o1, lens_t, D ** -0.5, ws1)
        torch.cuda.synchronize()
        assert torch.equal(o[l], o1), f"layer {l}"
    l = NL - 1
    ref = oracle.attention(q[l].float().cpu().numpy(), k[l].float().cpu().numpy(), v[l].float().cpu().numpy(),
                           kv_lens=lens, scale=D ** -0.5)["o"]
    parity.check(o[l].float().cpu().numpy(), ref, parity.kind_of(dtype))


def test_layers_reject_too_many_rows():
    q = torch.empty((2, 1, 8, 1, 64), dtype=torch.float32, device=DEV)
    assert binding.gqa_attn_decode_layers_workspace_size(70000, 1, 8, 8, 64, 64, binding.GQA_F32) == 0

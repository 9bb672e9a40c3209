"""The allocation-free decode entry point against the workspace entry point.

gqa_attn_decode_noalloc serves callers that cannot allocate device memory:
it uses scratch compiled into the library instead of a caller workspace.
Here it is called through the C ABI directly and must agree with
gqa_attn_decode (same tolerance as the other decode tests) on two calls in a
row with different inputs, so that scratch left behind by the first call
cannot leak into the second.  This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

from gqa_attention_kv_decode_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _noalloc(q, k, v, o, lens, max_kv_len, scale):
    B, Hq, _, D = q.shape
    Hkv, S_cap = k.shape[1], k.shape[2]
    return binding.lib().gqa_attn_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lens.data_ptr()), B, Hq, Hkv, D, S_cap,
        max_kv_len, scale, binding._dtype_code(q),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(dtype):
    B, Hq, Hkv, D, S = 3, 28, 4, 128, 5000
    lens = torch.tensor([5000, 1777, 64], dtype=torch.int32, device="cuda")
    scale = D ** -0.5
    for layer in (11, 12):  # two calls in a row, different inputs
        q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, S, dtype, layer=layer, device="cuda")
        o_na = torch.full_like(q, float("nan"))
        assert _noalloc(q, k, v, o_na, lens, S, scale) == binding.GQA_OK
        o_ws = binding.decode(q, k, v, kv_lens=lens, scale=scale, max_kv_len=S)
        torch.cuda.synchronize()
        a, b = o_na.float().cpu().numpy(), o_ws.float().cpu().numpy()
        assert np.isfinite(a).all()
        assert np.abs(a - b).max() <= TOL[dtype]
    assert binding.gqa_attn_decode_num_splits(B, Hq, Hkv, D, S, binding._dtype_code(q)) > 1


def test_noalloc_rejects_problems_larger_than_its_scratch():
    # 4096 requests x 32 heads x 128 dims needs far more than 16 MiB of partials
    q = torch.zeros(1, dtype=torch.float32, device="cuda")
    rc = binding.lib().gqa_attn_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(q.data_ptr()), None, 4096, 32, 8, 128, 8192, 8192, 0.1, binding.GQA_F32, None)
    assert rc == binding.GQA_ERR_SCRATCH_LIMIT
    assert "16 MiB" in binding.gqa_attn_status_string(rc)

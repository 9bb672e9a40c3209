"""The allocation-free decode entry point against the workspace entry point.

gqa_attn_decode_noalloc serves callers that cannot allocate device memory:
it uses scratch compiled into the library instead of a caller workspace.
Here it is called through the C ABI directly.  It runs the same kernels with
the same split plan as gqa_attn_decode, so the outputs must be bit for bit
equal.  Two calls run in a row: the first is larger (more requests, more
split partials) than the second, which has short requests and an empty one,
so partials that the first call leaves in the scratch would show up in the
second's output if any were read.  This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

from gqa_attention_kv_decode_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _noalloc(q, k, v, o, lens, max_kv_len, scale):
    B, Hq, _, D = q.shape
    Hkv, S_cap = k.shape[1], k.shape[2]
    return binding.lib().gqa_attn_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), None if lens is None else ctypes.c_void_p(lens.data_ptr()), B, Hq, Hkv, D, S_cap,
        max_kv_len, scale, binding._dtype_code(q),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(dtype):
    Hq, Hkv, D = 28, 4, 128
    scale = D ** -0.5
    calls = [  # (layer, per-request lengths, max_kv_len): a large call, then a small one
        (11, [5000, 1777, 64], 5000),
        (12, [300, 0], 300),
    ]
    splits = []
    for layer, lens_list, S in calls:
        B = len(lens_list)
        lens = torch.tensor(lens_list, dtype=torch.int32, device="cuda")
        q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, S, dtype, layer=layer, device="cuda")
        o_na = torch.full_like(q, float("nan"))
        assert _noalloc(q, k, v, o_na, lens, S, scale) == binding.GQA_OK
        o_ws = binding.decode(q, k, v, kv_lens=lens, scale=scale, max_kv_len=S)
        torch.cuda.synchronize()
        assert torch.isfinite(o_na).all()
        assert torch.equal(o_na, o_ws)
        splits.append(binding.gqa_attn_decode_num_splits(B, Hq, Hkv, D, S, binding._dtype_code(q)))
    assert splits[0] > splits[1] > 1  # both calls use partials, the first more of them


def test_noalloc_reports_argument_errors_like_the_workspace_entry_point():
    q, k, v = inputs.qkv(1, 14, 2, 64, 1, 128, torch.float32, device="cuda")
    o = torch.empty_like(q)
    qh = q.cpu()
    assert _noalloc(q, k, v, o, None, 200, 0.125) == binding.GQA_ERR_INVALID_ARG  # max_kv_len > S_cap
    assert _noalloc(qh, k, v, o, None, 128, 0.125) == binding.GQA_ERR_NOT_DEVICE_PTR
    # too large for the scratch AND given a host pointer: the argument error wins
    big = binding.lib().gqa_attn_decode_noalloc(
        ctypes.c_void_p(qh.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), None, 4096, 32, 8, 128, 8192, 8192, 0.1, binding.GQA_F32, None)
    assert big == binding.GQA_ERR_NOT_DEVICE_PTR


def test_noalloc_rejects_problems_larger_than_its_scratch():
    # 4096 requests x 32 heads x 128 dims at 8192 keys needs far more than
    # 16 MiB of partials.  The pointers are valid device pointers, so the
    # argument checks pass and the size limit rejects the call before any
    # launch (the buffers are never read).
    B, Hq, Hkv, D, S = 4096, 32, 8, 128, 8192
    assert binding.gqa_attn_decode_workspace_size(B, Hq, Hkv, D, S, binding.GQA_F32) > 16 << 20
    t = torch.zeros(64, dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(t.data_ptr())
    rc = binding.lib().gqa_attn_decode_noalloc(p, p, p, p, None, B, Hq, Hkv, D, S, S, 0.1, binding.GQA_F32, None)
    assert rc == binding.GQA_ERR_SCRATCH_LIMIT
    assert "16 MiB" in binding.gqa_attn_status_string(rc)

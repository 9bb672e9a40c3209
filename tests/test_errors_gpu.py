"""Argument errors of every entry point: the status code include/gqa_attn.h
documents, and nothing written.

Host validation runs before any launch, so a rejected call must leave the
output untouched (it is filled with a sentinel first and compared after a
synchronize).  The cases are those the boundary lists: a head count that
does not divide, a query longer than the keys, a head dimension other than
64 or 128, a non-positive or non-finite scale, a host pointer where device
memory is required (the analogue of the pages' FusedAttentionNeedsMetal:
there is no CPU fallback), a dtype without a kernel and a missing workspace.
"""

import math

import pytest
import torch

from gqa_attention_kv_decode_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENTINEL = 3.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def expect(status, fn, out):
    """fn() raises GqaAttnError with `status`, and `out` keeps its sentinel."""
    with pytest.raises(binding.GqaAttnError) as e:
        fn()
    torch.cuda.synchronize()
    assert e.value.status == status, binding.gqa_attn_status_string(e.value.status)
    assert (out == SENTINEL).all(), "a rejected call wrote its output"


def bf16(shape, seed, device=DEV):
    return inputs.randn(shape, seed, torch.bfloat16, device)


# ---------------------------------------------------------------- prefill

def prefill_args(Hq=14, Hkv=2, D=64, q_len=100, S=200, dtype=torch.bfloat16, device=DEV):
    q = inputs.randn((1, Hq, q_len, D), 1, dtype, device)
    k = inputs.randn((1, Hkv, S, D), 2, dtype, device)
    v = inputs.randn((1, Hkv, S, D), 3, dtype, device)
    o = torch.full_like(q, SENTINEL, device=DEV)
    return q, k, v, o


@pytest.mark.parametrize("case,status", [
    ("heads_not_divisible", binding.GQA_ERR_INVALID_ARG),
    ("query_longer_than_keys", binding.GQA_ERR_INVALID_ARG),
    ("kv_len_past_capacity", binding.GQA_ERR_INVALID_ARG),
    ("head_dim_96", binding.GQA_ERR_INVALID_ARG),
    ("scale_zero", binding.GQA_ERR_INVALID_ARG),
    ("scale_negative", binding.GQA_ERR_INVALID_ARG),
    ("scale_nan", binding.GQA_ERR_INVALID_ARG),
    ("scale_inf", binding.GQA_ERR_INVALID_ARG),
    ("fp32", binding.GQA_ERR_UNSUPPORTED),
    ("host_q", binding.GQA_ERR_NOT_DEVICE_PTR),
])
def test_prefill_rejects(case, status):
    kw = {}
    kv_len, scale = 200, 0.125
    if case == "heads_not_divisible":
        kw = dict(Hq=14, Hkv=3)
    elif case == "query_longer_than_keys":
        kv_len = 99
    elif case == "kv_len_past_capacity":
        kv_len = 201
    elif case == "head_dim_96":
        kw = dict(D=96)
    elif case == "fp32":
        kw = dict(dtype=torch.float32)
    scale = {"scale_zero": 0.0, "scale_negative": -0.125, "scale_nan": math.nan,
             "scale_inf": math.inf}.get(case, scale)
    q, k, v, o = prefill_args(**kw)
    if case == "host_q":
        q = q.cpu()
    expect(status, lambda: binding.gqa_attn_prefill(q, k, v, o, kv_len, scale, True), o)


@pytest.mark.parametrize("case,status", [
    ("heads_not_divisible", binding.GQA_ERR_INVALID_ARG),
    ("head_dim_96", binding.GQA_ERR_INVALID_ARG),
    ("scale_nan", binding.GQA_ERR_INVALID_ARG),
    ("fp32", binding.GQA_ERR_UNSUPPORTED),
    ("host_lengths", binding.GQA_ERR_NOT_DEVICE_PTR),
])
def test_prefill_varlen_rejects(case, status):
    kw = dict(Hq=14, Hkv=3) if case == "heads_not_divisible" else dict(D=96) if case == "head_dim_96" else \
        dict(dtype=torch.float32) if case == "fp32" else {}
    q, k, v, o = prefill_args(**kw)
    ql = torch.tensor([100], dtype=torch.int32, device=DEV)
    kl = torch.tensor([200], dtype=torch.int32, device=DEV)
    if case == "host_lengths":
        ql = ql.cpu()
    scale = math.nan if case == "scale_nan" else 0.125
    expect(status, lambda: binding.gqa_attn_prefill_varlen(q, k, v, o, ql, kl, scale, True), o)


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("case,status", [
    ("heads_not_divisible", binding.GQA_ERR_INVALID_ARG),
    ("head_dim_96", binding.GQA_ERR_INVALID_ARG),
    ("max_kv_len_past_capacity", binding.GQA_ERR_INVALID_ARG),
    ("scale_inf", binding.GQA_ERR_INVALID_ARG),
    ("host_k", binding.GQA_ERR_NOT_DEVICE_PTR),
    ("no_workspace", binding.GQA_ERR_WORKSPACE),
])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_decode_rejects(case, status, dtype):
    Hq, Hkv, D, S = 14, 2, 64, 128
    if case == "heads_not_divisible":
        Hkv = 3
    if case == "head_dim_96":
        D = 96
    q = inputs.randn((1, Hq, 1, D), 1, dtype, DEV)
    k = inputs.randn((1, Hkv, S, D), 2, dtype, DEV)
    v = inputs.randn((1, Hkv, S, D), 3, dtype, DEV)
    o = torch.full_like(q, SENTINEL)
    if case == "host_k":
        k = k.cpu()
    max_kv_len = S + 1 if case == "max_kv_len_past_capacity" else S
    scale = math.inf if case == "scale_inf" else 0.125
    ws_bytes = binding.gqa_attn_decode_workspace_size(1, Hq, 2, 64, S, binding._dtype_code(q))
    ws = torch.zeros(0 if case == "no_workspace" else ws_bytes, dtype=torch.uint8, device=DEV)
    expect(status, lambda: binding.gqa_attn_decode(q, k, v, o, None, scale, ws, max_kv_len=max_kv_len), o)


@pytest.mark.parametrize("case,status", [
    ("head_dim_96", binding.GQA_ERR_INVALID_ARG),
    ("group_size_32", binding.GQA_ERR_INVALID_ARG),
    ("scale_zero", binding.GQA_ERR_INVALID_ARG),
    ("host_codes", binding.GQA_ERR_NOT_DEVICE_PTR),
    ("no_workspace", binding.GQA_ERR_WORKSPACE),
])
def test_decode_q4_rejects(case, status):
    B, Hq, Hkv, S = 1, 8, 2, 64
    D = 96 if case == "head_dim_96" else 128
    kc, ks, kb, vc, vs, vb = inputs.q4_cache(B, Hkv, 128, S, device=DEV)
    if case == "head_dim_96":  # codes and groups sized for D = 96 (one and a half groups)
        kc, vc = kc[..., :48].contiguous(), vc[..., :48].contiguous()
    q = bf16((B, Hq, 1, D), 1)
    o = torch.full_like(q, SENTINEL)
    if case == "host_codes":
        kc = kc.cpu()
    ws_bytes = binding.gqa_attn_decode_q4_workspace_size(B, Hq, Hkv, 128, S)
    ws = torch.zeros(0 if case == "no_workspace" else ws_bytes, dtype=torch.uint8, device=DEV)
    scale = 0.0 if case == "scale_zero" else 0.09
    group = 32 if case == "group_size_32" else 64
    expect(status, lambda: binding.gqa_attn_decode_q4(q, kc, ks, kb, vc, vs, vb, o, None, scale, ws,
                                                      group_size=group), o)


@pytest.mark.parametrize("case,status", [
    ("heads_not_divisible", binding.GQA_ERR_INVALID_ARG),
    ("head_dim_96", binding.GQA_ERR_INVALID_ARG),
    ("host_q", binding.GQA_ERR_NOT_DEVICE_PTR),
])
def test_decode_layers_rejects(case, status):
    NL, B, Hq, Hkv, D, S = 3, 1, 14, 2, 64, 128
    if case == "heads_not_divisible":
        Hkv = 3
    if case == "head_dim_96":
        D = 96
    q = inputs.randn((NL, B, Hq, 1, D), 1, torch.float32, DEV)
    k = inputs.randn((NL, B, Hkv, S, D), 2, torch.float32, DEV)
    v = inputs.randn((NL, B, Hkv, S, D), 3, torch.float32, DEV)
    o = torch.full_like(q, SENTINEL)
    if case == "host_q":
        q = q.cpu()
    ws = torch.zeros(binding.gqa_attn_decode_layers_workspace_size(NL, B, 14, 2, 64, S, binding.GQA_F32),
                     dtype=torch.uint8, device=DEV)
    expect(status, lambda: binding.gqa_attn_decode_layers(q, k, v, o, None, 0.125, ws), o)


@pytest.mark.parametrize("case,status", [
    ("group_size_32", binding.GQA_ERR_INVALID_ARG),
    ("scale_nan", binding.GQA_ERR_INVALID_ARG),
    ("host_window", binding.GQA_ERR_NOT_DEVICE_PTR),
    ("no_workspace", binding.GQA_ERR_WORKSPACE),
])
def test_decode_q4_residual_rejects(case, status):
    B, Hq, Hkv, D, S, R = 1, 8, 2, 128, 64, 64
    kc, ks, kb, vc, vs, vb = inputs.q4_cache(B, Hkv, D, S, device=DEV)
    kr, vr = bf16((B, Hkv, R, D), 5), bf16((B, Hkv, R, D), 6)
    if case == "host_window":
        kr = kr.cpu()
    q = bf16((B, Hq, 1, D), 1)
    o = torch.full_like(q, SENTINEL)
    nq = torch.tensor([S], dtype=torch.int32, device=DEV)
    L = torch.tensor([S + 10], dtype=torch.int32, device=DEV)
    ws_bytes = binding.gqa_attn_decode_q4_residual_workspace_size(B, Hq, Hkv, D, S)
    ws = torch.zeros(0 if case == "no_workspace" else ws_bytes, dtype=torch.uint8, device=DEV)
    scale = math.nan if case == "scale_nan" else 0.09
    group = 32 if case == "group_size_32" else 64
    expect(status, lambda: binding.gqa_attn_decode_q4_residual(q, kc, ks, kb, vc, vs, vb, kr, vr, nq, L, o, scale,
                                                               ws, group_size=group), o)

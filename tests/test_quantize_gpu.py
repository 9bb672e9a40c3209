"""The GPU 4-bit quantizer against the oracle's, bit for bit.

Codes are integers decided in fp32 and scale/bias are fp16 roundings, so the
comparison is exact (no tolerance): same codes, same scale and bias bits.
Rows of the cache outside the destination range must keep their contents.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import parity
from gqa_attention_kv_decode_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def empty_cache(B, Hkv, S_cap, D, fill=0xA5):
    codes = torch.full((B, Hkv, S_cap, D // 2), fill, dtype=torch.uint8, device=DEV)
    scale = torch.full((B, Hkv, S_cap, D // 64), 7.0, dtype=torch.float16, device=DEV)
    bias = torch.full((B, Hkv, S_cap, D // 64), -7.0, dtype=torch.float16, device=DEV)
    return codes, scale, bias


def _same_fp16_bits(got, want):
    """Equal fp16 bit patterns, except that a NaN matches any NaN (the
    quantizer fixes no NaN payload: numpy's division and CUDA's conversion
    write different quiet NaNs)."""
    g = got.cpu().numpy()
    gb, wb = g.view(np.int16), want.view(np.int16)
    gn, wn = np.isnan(g), np.isnan(want)
    np.testing.assert_array_equal(gn, wn)
    np.testing.assert_array_equal(np.where(gn, 0, gb), np.where(wn, 0, wb))


def check_rows(src, codes, scale, bias, dst_row0):
    n = src.shape[2]
    c, s, b = oracle.quantize_q4(src.float().cpu().numpy())
    np.testing.assert_array_equal(codes[:, :, dst_row0:dst_row0 + n].cpu().numpy(), c)
    _same_fp16_bits(scale[:, :, dst_row0:dst_row0 + n], s)
    _same_fp16_bits(bias[:, :, dst_row0:dst_row0 + n], b)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 7, 64, 1000])
@pytest.mark.parametrize("mag", [1.0, 1e-3, 300.0])
def test_quantizer_matches_oracle_bit_for_bit(D, S, mag):
    x = (inputs.randn((2, 8, S, D), 71 + S, torch.float32, DEV) * mag).to(torch.bfloat16)
    codes, scale, bias = empty_cache(2, 8, S + 5, D)
    binding.gqa_attn_quantize_q4(x, codes, scale, bias, dst_row0=3)
    torch.cuda.synchronize()
    check_rows(x, codes, scale, bias, 3)
    # rows outside [3, 3 + S) are untouched
    assert (codes[:, :, :3] == 0xA5).all() and (codes[:, :, 3 + S:] == 0xA5).all()
    assert (scale[:, :, :3] == 7.0).all() and (bias[:, :, 3 + S:] == -7.0).all()


def test_quantizer_hand_cases_on_the_gpu():
    with open(GOLDEN) as f:
        cases = json.load(f)["quantizer_cases"]
    x = torch.tensor([c["x"] for c in cases], dtype=torch.float32).to(torch.bfloat16).view(1, len(cases), 1, 64).to(DEV)
    codes, scale, bias = empty_cache(1, len(cases), 1, 64)
    binding.gqa_attn_quantize_q4(x, codes, scale, bias)
    torch.cuda.synchronize()
    for i, c in enumerate(cases):
        assert codes[0, i, 0].cpu().tolist() == c["codes"], c["name"]
        assert scale[0, i, 0].float().item() == c["scale"][0]
        assert bias[0, i, 0].float().item() == c["bias"][0]


def test_incremental_flush_equals_one_pass():
    """Quantizing a cache one aged block of 64 rows at a time (the decode-time
    flush) gives the same bytes as quantizing it in one call."""
    S, B, Hkv, D = 640, 4, 8, 128
    x = inputs.randn((B, Hkv, S, D), 81, torch.bfloat16, DEV)
    whole = empty_cache(B, Hkv, S, D)
    binding.gqa_attn_quantize_q4(x, *whole)
    parts = empty_cache(B, Hkv, S, D, fill=0x11)
    for r0 in range(0, S, 64):
        binding.gqa_attn_quantize_q4(x[:, :, r0:r0 + 64].contiguous(), *parts, dst_row0=r0)
    torch.cuda.synchronize()
    for a, b in zip(whole, parts):
        assert torch.equal(a, b)


def test_decode_over_the_gpu_quantized_cache():
    """q4 decode on a cache the GPU quantized matches the oracle on the oracle's codes."""
    B, Hq, Hkv, D, S = 4, 32, 8, 128, 2048
    k = inputs.randn((B, Hkv, S, D), 91, torch.bfloat16, DEV)
    v = inputs.randn((B, Hkv, S, D), 92, torch.bfloat16, DEV)
    q = inputs.randn((B, Hq, 1, D), 93, torch.bfloat16, DEV)
    kc, ks, kb = empty_cache(B, Hkv, S, D)
    vc, vs, vb = empty_cache(B, Hkv, S, D)
    binding.gqa_attn_quantize_q4(k, kc, ks, kb)
    binding.gqa_attn_quantize_q4(v, vc, vs, vb)
    o = binding.decode_q4(q, kc, ks, kb, vc, vs, vb)
    torch.cuda.synchronize()
    okc, oks, okb = oracle.quantize_q4(k.float().cpu().numpy())
    ovc, ovs, ovb = oracle.quantize_q4(v.float().cpu().numpy())
    ref = oracle.attention_q4(q.float().cpu().numpy(), okc, oks, okb, ovc, ovs, ovb, scale=D ** -0.5)["o"]
    parity.check(o.float().cpu().numpy(), ref, "q4")


def test_quantizer_rejects_bad_ranges():
    x = inputs.randn((1, 2, 8, 128), 5, torch.bfloat16, DEV)
    codes, scale, bias = empty_cache(1, 2, 8, 128)
    with pytest.raises(binding.GqaAttnError) as e:
        binding.gqa_attn_quantize_q4(x, codes, scale, bias, dst_row0=1)  # 1 + 8 rows > 8
    assert e.value.status == binding.GQA_ERR_INVALID_ARG


def test_quantizer_more_heads_than_one_grid_row():
    # 70,001 heads of 3 rows: the launch spreads heads over two grid dimensions
    # (65,535 per row), so the last heads sit in the second z slice
    heads, S, D = 70001, 3, 64
    x = inputs.randn((1, heads, S, D), 97, torch.float32, DEV).to(torch.bfloat16)
    codes, scale, bias = empty_cache(1, heads, S, D)
    binding.gqa_attn_quantize_q4(x, codes, scale, bias, dst_row0=0)
    torch.cuda.synchronize()
    check_rows(x, codes, scale, bias, 0)


def _tie_groups(n_groups, seed):
    """Groups whose quotients (x - bias) / scale sit on or next to half-integers.

    Per group: scale s with 3 significant bits (exact in fp16 and bf16), bias
    lo = -j s, maximum lo + 15 s, so that the group's own scale and bias are
    s and lo; then 40 values lo + (k + 1/2) s (exact ties), 10 bf16 neighbours
    of such ties and 12 values drawn inside [lo, lo + 15 s].
    """
    rng = np.random.default_rng(seed)
    out = np.empty((n_groups, 64), dtype=np.float32)
    for g in range(n_groups):
        s = np.float32((8 + rng.integers(0, 8)) * 2.0 ** int(rng.integers(-12, 7)) / 8)
        lo = np.float32(-int(rng.integers(0, 4)) * s)
        k = rng.integers(0, 15, 50).astype(np.float32)
        ties = lo + (k + np.float32(0.5)) * s
        vals = np.concatenate([[lo, lo + 15 * s], ties,
                               lo + rng.uniform(0, 15, 12).astype(np.float32) * s])
        vals = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
        bits = vals.view(torch.int16)
        bits[42:52] += torch.from_numpy(rng.choice([-1, 1], 10).astype(np.int16))  # bf16 neighbours
        vals = bits.view(torch.bfloat16).float().numpy()
        out[g] = np.clip(vals, lo, lo + 15 * s)[rng.permutation(64)]
    return out


def test_quantizer_ties_bit_for_bit():
    """Codes on and next to the round-half-even ties: the GPU's quotient must
    be the correctly rounded fp32 division, not the reciprocal product."""
    x = _tie_groups(2048, 123)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert torch.equal(xb.float(), torch.from_numpy(x))  # every value is exact in bf16
    src = xb.view(1, 2048, 1, 64).to(DEV)
    codes, scale, bias = empty_cache(1, 2048, 1, 64)
    binding.gqa_attn_quantize_q4(src, codes, scale, bias)
    torch.cuda.synchronize()
    check_rows(src, codes, scale, bias, 0)
    # the same groups quantized with the reciprocal product differ somewhere,
    # so this test separates the two readings
    c, s_ref, b_ref = oracle.quantize_q4(x)
    s32, b32 = s_ref.astype(np.float32), b_ref.astype(np.float32)
    alt = np.clip(np.rint((x - b32) * (np.float32(1.0) / s32)), 0, 15).astype(np.uint8)
    alt = alt[:, 0::2] | (alt[:, 1::2] << 4)
    assert (alt != c).any()


def _special_group(kind, rng):
    """64 values of one group of a given kind (float32, exact in bf16 after
    the caller's rounding).  Kinds 0, 12 and 13 are ordinary groups; the
    others reach the clamps and the special values of the quantizer."""
    x = rng.standard_normal(64).astype(np.float32)
    if kind == 1:
        x[rng.integers(64)] = np.nan                   # one NaN element: code 0, left out of min/max
    elif kind == 2:
        x[:] = np.nan                                  # all NaN: NaN scale and bias, codes 0
    elif kind == 3:
        x[rng.integers(64)] = np.inf                   # infinite maximum: infinite scale
    elif kind == 4:
        x[rng.integers(64)] = -np.inf                  # infinite minimum and bias
    elif kind == 5:
        x = np.float32(1e-4) * (1 + rng.integers(0, 8, 64).astype(np.float32) / 128)  # subnormal fp16 scale
    elif kind == 6:
        x = rng.uniform(0, 1, 64).astype(np.float32)
        x[rng.integers(64)] = np.float32(-1e-6)        # fp16(min) != min: some x - bias < 0
    elif kind == 7:
        x = x * np.float32(1e5)                        # |min| past the fp16 range: infinite bias
    elif kind == 8:
        x = rng.uniform(0, 2e6, 64).astype(np.float32)  # range / 15 past the fp16 range
    elif kind == 9:
        x[:] = np.float32(0.75)                        # constant: zero scale
    elif kind == 10:
        x = np.where(rng.random(64) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
    elif kind == 11:
        x[:] = np.nan
        x[rng.integers(64)] = np.float32(2.5)          # one finite value: zero scale
    elif kind == 12:
        x = x - np.float32(5.0)
    elif kind == 13:
        x = x * np.float32(1e-3)
    return x


@pytest.mark.parametrize("D", [64, 128])
def test_quantizer_special_groups_bit_for_bit(D):
    """Special groups (NaN elements, infinities, subnormal fp16 scales, a bias
    that is not the minimum, zero scales) spread over the first 64 rows, so
    that warps mix them with ordinary groups, and ordinary groups alone in
    the rows after them: both code paths of the kernel against the oracle."""
    rng = np.random.default_rng(2026 + D)
    G, S = D // 64, 160
    x = np.empty((S, D), dtype=np.float32)
    for r in range(S):
        for g in range(G):
            kind = (r * G + g) % 14 if r < 64 else int(rng.choice([0, 12, 13]))
            x[r, g * 64:(g + 1) * 64] = _special_group(kind, rng)
    xb = torch.from_numpy(x).to(torch.bfloat16).view(1, 1, S, D).to(DEV)
    codes, scale, bias = empty_cache(1, 1, S, D)
    binding.gqa_attn_quantize_q4(xb, codes, scale, bias)
    torch.cuda.synchronize()
    check_rows(xb, codes, scale, bias, 0)

"""The decode split planner, on the host (no GPU): the plans of the fp32 and
bf16 kernels (contiguous and paged caches) and of the 4-bit kernel for a
device of a given SM count, checked against the rule the kernels and the
merge follow.

A request of L keys uses n_used(L) = min(n_split, ceil(L / chunk)) splits
and deals its ceil(L / tile) tiles to them round-robin.  The properties:
a full-length request uses every planned split; every used split gets at
least one tile; n_used grows with L and never exceeds n_split; a short request
in a one-wave plan spreads over its splits (chunk of at most two tiles); a
split of a several-wave plan holds at most 1024 rows; and under the split
override a request's splits do not depend on the batch.
"""

import math

import pytest

from gqa_attention_kv_decode_gb300 import binding

KERNELS = [(binding.GQA_PLAN_DECODE, binding.GQA_F32), (binding.GQA_PLAN_DECODE, binding.GQA_BF16),
           (binding.GQA_PLAN_PAGED, binding.GQA_F32), (binding.GQA_PLAN_PAGED, binding.GQA_BF16),
           (binding.GQA_PLAN_Q4, binding.GQA_BF16)]
SHAPES = [(B, Hq, Hkv, D, S, variant, dt)
          for B in (1, 2, 4, 16, 64)
          for Hq, Hkv in ((28, 4), (32, 8), (14, 2))
          for D in (64, 128)
          for S in (64, 128, 2048, 8192, 32768)
          for variant, dt in KERNELS]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def n_used(L, n_split, chunk):
    return min(n_split, -(-L // chunk))


def lengths(S):
    return sorted({1, 2, S // 3, S // 2, max(1, S - 1), S} | set(range(1, min(S, 300) + 1, 7)))


@pytest.mark.parametrize("B,Hq,Hkv,D,S,variant,dt", SHAPES)
def test_plan_invariants(B, Hq, Hkv, D, S, variant, dt):
    n_split, chunk, tile = binding.gqa_attn_decode_plan_for(B, Hq, Hkv, D, S, dt, 152, variant)
    assert 1 <= n_split <= 1024 and tile in (16, 32, 64, 128) and chunk >= 1
    assert n_used(S, n_split, chunk) == n_split, "a full-length request uses every planned split"
    prev = 0
    for L in lengths(S):
        u = n_used(L, n_split, chunk)
        assert 1 <= u <= n_split and u >= prev
        prev = u
        tiles = -(-L // tile)
        assert u <= tiles, f"L={L}: {u} splits for {tiles} tiles leaves a split without a tile"
        # round-robin: split s takes tiles s, s + u, ...; together every tile once
        per = [len(range(s, tiles, u)) for s in range(u)]
        assert sum(per) == tiles and max(per) - min(per) <= 1
    spread = chunk * n_split < S
    if spread:
        assert chunk <= 2 * tile, "a one-wave plan spreads short requests (chunk of at most two tiles)"
    else:
        assert chunk <= max(1024, S) and (n_split == 1 or chunk <= 1024)


@pytest.mark.parametrize("dt", [binding.GQA_F32, binding.GQA_BF16])
def test_short_request_uses_more_splits_than_its_share(dt):
    """One-wave plan sized for 32,768 keys: a 2,048-key request takes far more
    splits than 2048 / (32768 / n_split)."""
    n_split, chunk, tile = binding.gqa_attn_decode_plan_for(1, 28, 4, 128, 32768, dt, 152)
    assert n_split > 1 and chunk * n_split < 32768
    assert n_used(2048, n_split, chunk) >= min(n_split, 2048 // (2 * tile))
    assert n_used(2048, n_split, chunk) > math.ceil(2048 / math.ceil(32768 / n_split))


def test_more_sms_never_fewer_splits():
    for dt in (binding.GQA_F32, binding.GQA_BF16):
        for B, S in ((1, 32768), (2, 8192), (4, 2048)):
            counts = [binding.gqa_attn_decode_plan_for(B, 32, 8, 128, S, dt, n)[0] for n in (8, 38, 76, 152, 304)]
            assert counts == sorted(counts), (dt, B, S, counts)


@pytest.mark.parametrize("splits", [3, 6, 40])
def test_override_makes_a_requests_splits_independent_of_the_batch(splits):
    with binding.plan_override(decode_splits=splits):
        plans = {B: binding.gqa_attn_decode_plan_for(B, 28, 4, 128, 3000, binding.GQA_BF16, 152) for B in (1, 4, 64)}
    assert len({p[0] for p in plans.values()}) == 1
    for L in (1, 64, 700, 1777, 3000):
        assert len({n_used(L, p[0], p[1]) for p in plans.values()}) == 1, L


@pytest.mark.parametrize("args,status", [
    ((1, 28, 3, 128, 100, 0, 152), binding.GQA_ERR_INVALID_ARG),   # heads do not divide
    ((1, 28, 4, 96, 100, 0, 152), binding.GQA_ERR_INVALID_ARG),    # head dimension
    ((1, 28, 4, 128, 0, 0, 152), binding.GQA_ERR_INVALID_ARG),     # no keys
    ((1, 28, 4, 128, 100, 0, 0), binding.GQA_ERR_INVALID_ARG),     # no SMs
    ((1, 28, 4, 128, 100, 7, 152), binding.GQA_ERR_UNSUPPORTED),   # dtype without a plain decode kernel
])
def test_plan_for_rejects(args, status):
    with pytest.raises(binding.GqaAttnError) as e:
        binding.gqa_attn_decode_plan_for(*args[:5], binding.GQA_F32 if args[5] == 0 else args[5], args[6])
    assert e.value.status == status


def test_plan_for_rejects_unknown_variants_and_fp32_queries_for_q4():
    with pytest.raises(binding.GqaAttnError) as e:
        binding.gqa_attn_decode_plan_for(1, 32, 8, 128, 100, binding.GQA_BF16, 152, 3)
    assert e.value.status == binding.GQA_ERR_INVALID_ARG
    with pytest.raises(binding.GqaAttnError) as e:
        binding.gqa_attn_decode_plan_for(1, 32, 8, 128, 100, binding.GQA_F32, 152, binding.GQA_PLAN_Q4)
    assert e.value.status == binding.GQA_ERR_UNSUPPORTED

"""The parity bounds of the GPU tests can fail at full size (CPU only).

Mistakes are planted in the oracle's own computation, at the headline decode
geometry (Qwen2.5-7B heads, one KV head group, 32,768 keys): a split of the
keys left out, and a log-sum-exp merge that forgets the per-split maxima.
Each planted result passes the bf16 absolute bound of 2e-2, which is why the
scaled bound exists, and fails the scaled bound.  A bf16-rounded copy of the
true result passes both.
"""

import numpy as np
import pytest
import torch

import oracle
import parity
from gqa_attention_kv_decode_gb300 import inputs

S, D, NREP, TILE, NSPLIT = 32768, 128, 7, 64, 38


@pytest.fixture(scope="module")
def group():
    q, k, v = inputs.qkv(1, NREP, 1, D, 1, S, torch.bfloat16, layer=3)
    q, k, v = (t.float().numpy() for t in (q, k, v))
    ref = oracle.attention(q, k, v, scale=D ** -0.5)
    return q, k, v, ref


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def test_rounded_truth_passes(group):
    q, k, v, ref = group
    parity.check(_bf16(ref["o"]), ref["o"], "bf16", "bf16-rounded oracle")


def test_dropped_split_fails_only_the_scaled_bound(group):
    q, k, v, ref = group
    # tiles are dealt round-robin to the splits: split 5 holds tiles 5, 43, 81, ...
    tile = np.arange(S) // TILE
    keep = tile % NSPLIT != 5
    bad = oracle.attention(q, k[:, :, keep], v[:, :, keep], scale=D ** -0.5)["o"]
    err = np.abs(_bf16(bad) - ref["o"]).max()
    assert err <= parity.ABS["bf16"]  # the absolute bound alone accepts it
    assert not parity.within(_bf16(bad), ref["o"], "bf16")


def test_merge_without_maxima_fails_only_the_scaled_bound(group):
    q, k, v, ref = group
    # two halves merged as if both had the same maximum: o = (l1 o1 + l2 o2)
    # / (l1 + l2) with each l taken relative to its own half's maximum
    h = S // 2
    a = oracle.attention(q, k[:, :, :h], v[:, :, :h], scale=D ** -0.5)
    b = oracle.attention(q, k[:, :, h:], v[:, :, h:], scale=D ** -0.5)
    s = D ** -0.5
    la = np.exp(a["lse"] - (s * q @ np.swapaxes(k[:, :, :h], -1, -2)).max(-1))
    lb = np.exp(b["lse"] - (s * q @ np.swapaxes(k[:, :, h:], -1, -2)).max(-1))
    bad = (la[..., None] * a["o"] + lb[..., None] * b["o"]) / (la + lb)[..., None]
    assert np.abs(_bf16(bad) - ref["o"]).max() <= parity.ABS["bf16"]
    assert not parity.within(_bf16(bad), ref["o"], "bf16")
    # the correct merge (weights exp(lse)) passes
    wa, wb = np.exp(a["lse"] - ref["lse"]), np.exp(b["lse"] - ref["lse"])
    good = wa[..., None] * a["o"] + wb[..., None] * b["o"]
    parity.check(_bf16(good), ref["o"], "bf16", "correct merge")

"""Seeded synthetic inputs shared by the tests, the oracle runs and the bench.

This module holds no attention arithmetic: it only draws tensors and builds
the 4-bit cache encoding that the decode kernels consume.  It imports torch
(for generators and device placement) and numpy, nothing else.

Recipe:
  * base seed 20261202; tensor ``t`` of layer ``l`` is drawn from
    ``torch.Generator(device).manual_seed(base + 1000 * l + t)`` with
    ``torch.randn`` in float32 and then rounded to the storage dtype (RNE);
    t = 0, 1, 2 for Q, K, V.  A CPU and a CUDA generator give different
    numbers for the same seed; every comparison feeds the same tensors (moved
    between devices) to both sides.
  * ragged lengths: ``numpy.random.default_rng(seed).integers(lo, hi + 1, B)``.
  * the 4-bit cache is built by quantizing bf16 N(0,1) data per group of 64
    elements along D (see ``quantize_q4``).
"""

from __future__ import annotations

import numpy as np
import torch

BASE_SEED = 20261202


def tensor_seed(layer: int, t: int, base: int = BASE_SEED) -> int:
    return base + 1000 * layer + t


def randn(shape, seed: int, dtype=torch.float32, device="cpu") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    return x.to(dtype)


def ragged_kv_lens(B: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Per-request lengths drawn uniformly from the integers lo..hi inclusive."""
    return np.random.default_rng(seed).integers(lo, hi + 1, B).astype(np.int32)


def qkv(B, Hq, Hkv, D, q_len, s_cap, dtype, layer=0, device="cpu", base=BASE_SEED):
    """Q [B,Hq,q_len,D], K and V [B,Hkv,s_cap,D], N(0,1), one layer's seeds."""
    q = randn((B, Hq, q_len, D), tensor_seed(layer, 0, base), dtype, device)
    k = randn((B, Hkv, s_cap, D), tensor_seed(layer, 1, base), dtype, device)
    v = randn((B, Hkv, s_cap, D), tensor_seed(layer, 2, base), dtype, device)
    return q, k, v


def poison_tail(x: torch.Tensor, kv_lens) -> torch.Tensor:
    """Fill rows >= kv_lens[b] of a [B, H, S, ...] cache with NaN (in place).

    A kernel that multiplies invalid rows by zero instead of skipping them
    turns these rows into NaN outputs.
    """
    for b, L in enumerate(kv_lens):
        x[b, :, int(L):] = float("nan")
    return x


def quantize_q4(x: torch.Tensor, group_size: int = 64):
    """Build a 4-bit group-affine cache from ``x`` [..., D].

    Per group of ``group_size`` consecutive elements along D (values widened
    to float32): scale = fp16((max - min) / 15), bias = fp16(min),
    code = clamp(round_half_even((x - bias) / scale), 0, 15), code 0 when the
    scale is 0.  Codes are packed two per byte: element 2t in the low nibble
    of byte t, element 2t+1 in the high nibble.

    Returns (codes uint8 [..., D/2], scale fp16 [..., D/G], bias fp16 [..., D/G]).
    """
    D = x.shape[-1]
    if D % group_size != 0 or D % 2 != 0:
        raise ValueError("D must be a multiple of the group size")
    xf = x.float().reshape(*x.shape[:-1], D // group_size, group_size)
    mn = xf.amin(dim=-1)
    mx = xf.amax(dim=-1)
    scale = ((mx - mn) / 15.0).to(torch.float16)
    bias = mn.to(torch.float16)
    s32 = scale.float().unsqueeze(-1)
    b32 = bias.float().unsqueeze(-1)
    safe = torch.where(s32 > 0, s32, torch.ones_like(s32))
    code = torch.round((xf - b32) / safe).clamp_(0, 15)
    code = torch.where(s32 > 0, code, torch.zeros_like(code))
    code = code.to(torch.uint8).reshape(*x.shape[:-1], D)
    packed = code[..., 0::2] | (code[..., 1::2] << 4)
    return packed.contiguous(), scale.contiguous(), bias.contiguous()


def q4_cache(B, Hkv, D, s_cap, layer=0, device="cpu", group_size=64, base=BASE_SEED):
    """One layer's quantized K and V caches, built from bf16 N(0,1) data."""
    k = randn((B, Hkv, s_cap, D), tensor_seed(layer, 1, base), torch.bfloat16, device)
    v = randn((B, Hkv, s_cap, D), tensor_seed(layer, 2, base), torch.bfloat16, device)
    kc, ks, kb = quantize_q4(k, group_size)
    vc, vs, vb = quantize_q4(v, group_size)
    return kc, ks, kb, vc, vs, vb


def paged_pool(k: torch.Tensor, v: torch.Tensor, kv_lens, block_size: int, seed: int, spare: int = 3,
               fill=float("nan")):
    """Scatter a dense cache [B, Hkv, S, D] into block pools.

    Returns (k_pool, v_pool, block_table): pools [num_blocks, Hkv, block_size,
    D] with the blocks of all requests in a seeded random order, ``spare``
    extra blocks and every row past kv_lens[b] set to ``fill``; block_table
    int32 [B, ceil(S / block_size)] (on the device of ``k``).  Key row j of
    request b is row j % block_size of block block_table[b, j // block_size].
    """
    B, hkv, S, D = k.shape
    nb = -(-S // block_size)
    n_pool = B * nb + spare
    order = np.random.default_rng(seed).permutation(n_pool)
    kp = torch.full((n_pool, hkv, block_size, D), fill, dtype=k.dtype, device=k.device)
    vp = torch.full_like(kp, fill)
    table = torch.zeros((B, nb), dtype=torch.int32)
    for b in range(B):
        L = int(kv_lens[b])
        for i in range(nb):
            blk = int(order[b * nb + i])
            table[b, i] = blk
            r0 = i * block_size
            n = max(0, min(block_size, L - r0))
            if n:
                kp[blk, :, :n] = k[b, :, r0:r0 + n]
                vp[blk, :, :n] = v[b, :, r0:r0 + n]
    return kp, vp, table.to(k.device)

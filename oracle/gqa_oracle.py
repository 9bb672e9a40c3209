"""Plain, slow fp64 oracle for grouped-query scaled-dot-product attention.

TEST INFRASTRUCTURE.  Nothing on the product path may import or call this
module; it exists so that the CUDA kernels can be compared, element by
element, with the textbook definition of the operation.

Every function takes numpy arrays (any float dtype; bf16 data is passed in as
its exact float32 widening) and computes in float64.  It follows the
unfused ("naive") attention the pages describe, one step per line:

  1. repeat_kv: copy each KV head to the n_rep = Hq / Hkv query heads that
     share it ("Fused attention makes a 4,096-token Qwen2 prefill on Metal
     4.5x faster", section "Cause and workaround", the naive path; and
     "2x Faster Qwen2 Decode on Metal in Candle", section "Why It Matters:
     7x KV Expansion on Every Decode Step", steps 1-2).
  2. scores = scale * Q K^T (a matmul).
  3. causal mask aligned to the END of the keys: query row i of a q_len-row
     block sees key j iff j <= i + (kv_len - q_len) ("Fused attention ...",
     "Cause and workaround", item 2).
  4. softmax over the visible keys.
  5. O = P V (a matmul).

Readings of points the pages leave open (each one is also listed in the
design notes):
  * head mapping: query head h reads KV head h // n_rep, the grouping that
    repeat_kv produces;
  * kv_len == 0 (no visible key): the output row is defined as zeros and its
    log-sum-exp as -inf;
  * the 4-bit cache stores element 2t of a row in the low nibble of byte t
    and element 2t+1 in the high nibble; x = code * scale + bias with one fp16
    scale and bias per group of ``group_size`` consecutive elements along D
    ("Batching Decode Attention Across Requests ...", VeloxQuant-MLX blog,
    sections "The setup" and "Part 4: the other half of the lever actually
    works": the fused kernel reads the group-affine codes, the baseline
    dequantises them and calls SDPA -- this module is that baseline);
  * the 4-bit quantizer (the pages say "group-affine", x = code*scale + bias,
    and give no quantizer): per group, scale = fp16((max - min) / 15),
    bias = fp16(min), code = clamp(round_half_even((x - bias) / scale), 0,
    15), code 0 when scale == 0.  The code inverts the dequantisation
    formula directly: one IEEE float32 subtraction and one correctly rounded
    float32 division per element (float32 is the precision the bf16 source
    and the fp16 scale and bias widen to exactly), then round half to even;
  * the residual window of a 4-bit cache (the pages: a production KIVI cache
    keeps the most recent tokens unquantized): key rows [0, n_quant[b]) of
    request b come from the 4-bit cache and rows [n_quant[b], kv_lens[b])
    from rows [0, kv_lens[b] - n_quant[b]) of the residual buffer, which is
    kept in the activation dtype (bf16 here);
  * a paged cache (the pages name paged attention but give no layout): a
    pool [num_blocks, Hkv, block_size, D] and an integer block table
    [B, max_blocks]; key row j of request b is row j % block_size of block
    block_table[b, j // block_size].  With an appended token, kv_lens counts
    it and its K/V go to row kv_lens[b] - 1 before attending.
"""

from __future__ import annotations

import warnings

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def repeat_kv(x, n_rep: int) -> np.ndarray:
    """Expand [B, Hkv, S, D] to [B, Hkv * n_rep, S, D] by copying heads.

    Query head h gets KV head h // n_rep (an explicit gather, i.e. the copy
    the fused kernels avoid).
    """
    x = _f64(x)
    hkv = x.shape[1]
    src = np.arange(hkv * n_rep) // n_rep
    return x[:, src].copy()


def visible_mask(q_len: int, kv_len: int, causal: bool) -> np.ndarray:
    """Boolean [q_len, kv_len] mask of visible keys.

    With ``causal`` the queries are aligned to the end of the keys: row i is
    query position kv_len - q_len + i, so it sees keys j <= i + kv_len - q_len.
    Without ``causal`` every key is visible.
    """
    i = np.arange(q_len)[:, None]
    j = np.arange(kv_len)[None, :]
    if not causal:
        return np.ones((q_len, kv_len), dtype=bool)
    return j <= i + (kv_len - q_len)


def attention(q, k, v, kv_lens=None, scale=None, causal=False, return_probs=False):
    """Grouped-query attention by its definition, in float64.

    q: [B, Hq, Tq, D]; k, v: [B, Hkv, S_cap, D] with Hq % Hkv == 0.
    kv_lens: per-request number of valid key rows (None: all S_cap rows).
    Only rows j < kv_lens[b] of K and V are read.
    Returns a dict with ``o`` [B, Hq, Tq, D], ``lse`` [B, Hq, Tq] (natural
    log of the softmax denominator, scores including the scale) and, when
    ``return_probs``, ``p``: a list over b of [Hq, Tq, kv_len_b] arrays.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    B, Hq, Tq, D = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("query heads must be a multiple of the KV heads")
    n_rep = Hq // Hkv
    s_cap = k.shape[2]
    if kv_lens is None:
        kv_lens = [s_cap] * B
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    scale = float(scale)

    k_rep = repeat_kv(k, n_rep)
    v_rep = repeat_kv(v, n_rep)

    o = np.zeros((B, Hq, Tq, D), dtype=np.float64)
    lse = np.full((B, Hq, Tq), -np.inf, dtype=np.float64)
    probs = []
    for b in range(B):
        L = int(kv_lens[b])
        if L > s_cap or L < 0:
            raise ValueError("kv_len out of range")
        if causal and 0 < L < Tq:
            raise ValueError("causal attention needs q_len <= kv_len")
        if L == 0:
            probs.append(np.zeros((Hq, Tq, 0)))
            continue
        kb = k_rep[b, :, :L, :]                                 # [Hq, L, D]
        vb = v_rep[b, :, :L, :]
        s = scale * np.matmul(q[b], np.swapaxes(kb, -1, -2))    # [Hq, Tq, L]
        mask = visible_mask(Tq, L, causal)
        s = np.where(mask[None], s, -np.inf)
        m = np.max(s, axis=-1, keepdims=True)
        e = np.exp(s - m)
        den = np.sum(e, axis=-1, keepdims=True)
        p = e / den
        o[b] = np.matmul(p, vb)
        lse[b] = (m + np.log(den))[..., 0]
        probs.append(p)
    out = {"o": o, "lse": lse}
    if return_probs:
        out["p"] = probs
    return out


def dequant_q4(codes, scale, bias, group_size: int = 64) -> np.ndarray:
    """Expand a packed 4-bit group-affine cache to float64.

    codes: uint8 [..., D/2]; element 2t is the low nibble of byte t and
    element 2t+1 the high nibble.  scale, bias: fp16 [..., D/group_size].
    Returns x[..., d] = code[d] * scale[d // group_size] + bias[d // group_size].
    """
    codes = np.asarray(codes, dtype=np.uint8)
    lo = (codes & 0x0F).astype(np.float64)
    hi = (codes >> 4).astype(np.float64)
    D = codes.shape[-1] * 2
    c = np.empty(codes.shape[:-1] + (D,), dtype=np.float64)
    c[..., 0::2] = lo
    c[..., 1::2] = hi
    sc = np.repeat(np.asarray(scale, dtype=np.float16).astype(np.float64), group_size, axis=-1)
    bi = np.repeat(np.asarray(bias, dtype=np.float16).astype(np.float64), group_size, axis=-1)
    if sc.shape[-1] != D:
        raise ValueError("D must be a multiple of group_size")
    return c * sc + bi


def attention_q4(q, k_codes, k_scale, k_bias, v_codes, v_scale, v_bias,
                 kv_lens=None, scale=None, group_size: int = 64, causal=False):
    """Attention over a 4-bit group-affine cache: dequantise, then attend."""
    k = dequant_q4(k_codes, k_scale, k_bias, group_size)
    v = dequant_q4(v_codes, v_scale, v_bias, group_size)
    return attention(q, k, v, kv_lens=kv_lens, scale=scale, causal=causal)


def paged_to_contiguous(pool, block_table, kv_lens, block_size: int) -> np.ndarray:
    """Gather a paged cache into a dense [B, Hkv, max(kv_lens), D] array.

    pool: [num_blocks, Hkv, block_size, D]; block_table: [B, max_blocks].
    Row j < kv_lens[b] of request b is pool[block_table[b, j // block_size],
    :, j % block_size]; rows past kv_lens[b] are zero (never read).
    """
    pool = _f64(pool)
    table = np.asarray(block_table, dtype=np.int64)
    B = table.shape[0]
    hkv, D = pool.shape[1], pool.shape[3]
    S = max(1, int(max(kv_lens)))
    out = np.zeros((B, hkv, S, D), dtype=np.float64)
    for b in range(B):
        for j in range(int(kv_lens[b])):
            out[b, :, j, :] = pool[table[b, j // block_size], :, j % block_size, :]
    return out


def append_paged(k_pool, v_pool, block_table, kv_lens, block_size: int, k_new, v_new):
    """Copies of the pools with the new token of every request written.

    k_new, v_new: [B, Hkv, 1, D]; the token of request b goes to position
    kv_lens[b] - 1, i.e. row (kv_lens[b] - 1) % block_size of block
    block_table[b, (kv_lens[b] - 1) // block_size].  Requests with
    kv_lens[b] == 0 write nothing.
    """
    kp = _f64(k_pool).copy()
    vp = _f64(v_pool).copy()
    table = np.asarray(block_table, dtype=np.int64)
    kn, vn = _f64(k_new), _f64(v_new)
    for b in range(table.shape[0]):
        pos = int(kv_lens[b]) - 1
        if pos < 0:
            continue
        blk = table[b, pos // block_size]
        kp[blk, :, pos % block_size, :] = kn[b, :, 0, :]
        vp[blk, :, pos % block_size, :] = vn[b, :, 0, :]
    return kp, vp


def attention_paged(q, k_pool, v_pool, block_table, kv_lens, block_size: int, scale=None,
                    k_new=None, v_new=None):
    """Decode attention over a paged cache: (append,) gather, then attend.

    Returns the dict of ``attention`` plus ``k_pool`` and ``v_pool`` (the
    pools after the append; the inputs are not modified).
    """
    kp, vp = _f64(k_pool), _f64(v_pool)
    if k_new is not None:
        kp, vp = append_paged(kp, vp, block_table, kv_lens, block_size, k_new, v_new)
    k = paged_to_contiguous(kp, block_table, kv_lens, block_size)
    v = paged_to_contiguous(vp, block_table, kv_lens, block_size)
    out = attention(q, k, v, kv_lens=kv_lens, scale=scale)
    out["k_pool"] = kp
    out["v_pool"] = vp
    return out


def quantize_q4(x, group_size: int = 64):
    """Group-affine 4-bit quantization of x [..., D] (float32 arithmetic).

    Per group of ``group_size`` consecutive elements along D: the minimum and
    maximum m, M (NaN elements left out); scale = fp16((M - m) / 15) and
    bias = fp16(m) (round to nearest); code = round-half-even((x - bias) /
    scale) with the subtraction and the division each one IEEE float32
    operation, clamped to [0, 15]; code 0 where the scale is 0 or the
    quotient is NaN.  Codes are packed two per byte, element 2t in the low
    nibble of byte t.  Returns (codes uint8 [..., D/2], scale fp16, bias fp16
    [..., D/group_size]).  ("Batching Decode Attention Across Requests ...",
    VeloxQuant-MLX blog, "Part 4": the format x = code * scale + bias, and a
    cache quantized incrementally, one newly aged group-aligned block per
    step.)
    """
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    if D % group_size != 0 or D % 2 != 0:
        raise ValueError("D must be a multiple of the group size")
    grp = x.reshape(x.shape[:-1] + (D // group_size, group_size))
    with np.errstate(all="ignore"), warnings.catch_warnings():
        warnings.simplefilter("ignore", RuntimeWarning)  # an all-NaN group has a NaN scale
        lo = np.nanmin(grp, axis=-1)
        hi = np.nanmax(grp, axis=-1)
        scale = ((hi - lo) / np.float32(15.0)).astype(np.float16)
        bias = lo.astype(np.float16)
        s32 = scale.astype(np.float32)[..., None]
        b32 = bias.astype(np.float32)[..., None]
        q = np.rint((grp - b32) / s32)
        q = np.where(np.isnan(q), np.float32(0), np.clip(q, 0, 15))
    q = np.where(s32 > 0, q, 0).astype(np.uint8).reshape(x.shape)
    packed = (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
    return packed, scale, bias


def attention_q4_residual(q, k_codes, k_scale, k_bias, v_codes, v_scale, v_bias, k_res, v_res,
                          n_quant, kv_lens, scale=None, group_size: int = 64):
    """Decode attention over a 4-bit cache followed by an unquantized window.

    Key row j < n_quant[b] of request b is the dequantised row j of the 4-bit
    cache; key row n_quant[b] + i (i < kv_lens[b] - n_quant[b]) is row i of
    k_res / v_res [B, Hkv, R_cap, D].  The rows are concatenated, then the
    attention definition applies.
    """
    kq = dequant_q4(k_codes, k_scale, k_bias, group_size)
    vq = dequant_q4(v_codes, v_scale, v_bias, group_size)
    kr, vr = _f64(k_res), _f64(v_res)
    B, hkv, _, D = kq.shape
    S = max(1, int(max(kv_lens)))
    k = np.zeros((B, hkv, S, D))
    v = np.zeros((B, hkv, S, D))
    for b in range(B):
        nq, L = int(n_quant[b]), int(kv_lens[b])
        if not 0 <= nq <= L:
            raise ValueError("need 0 <= n_quant <= kv_len")
        k[b, :, :nq] = kq[b, :, :nq]
        v[b, :, :nq] = vq[b, :, :nq]
        k[b, :, nq:L] = kr[b, :, :L - nq]
        v[b, :, nq:L] = vr[b, :, :L - nq]
    return attention(q, k, v, kv_lens=kv_lens, scale=scale)

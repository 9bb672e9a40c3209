"""Algorithmic byte and flop counts for the roofline figures.

These count what the operation must move or compute, not what a kernel
happens to move: padding rows past kv_len, split-KV partials and the
expanded copies the fused kernels avoid are all excluded.

  * decode (per request): Q + K + V + O, with K and V counted over the
    kv_len valid rows of the Hkv unexpanded heads.  At Qwen2.5-7B head
    geometry (4 KV heads, D = 128), 2,048 tokens and an fp32 cache the K+V
    part is 8 MiB per layer, the figure "2x Faster Qwen2 Decode on Metal in
    Candle" gives in "Why It Matters: 7x KV Expansion on Every Decode Step".
  * q4 decode (per request): codes (D/2 bytes per row) plus one fp16 scale
    and one fp16 bias per group of G elements, for K and V, plus bf16 Q and O.
  * prefill: 4 * D * Hq * (visible query/key pairs) flops (two matmuls of
    2 * D flops per pair).  The score matrix the unfused path materialises,
    Hq * T * T elements, is reported separately: 470 MB for 14 heads at
    T = 4,096 in bf16 ("Fused attention makes a 4,096-token Qwen2 prefill on
    Metal 4.5x faster", "Why it matters").
"""

from __future__ import annotations

ELEM_BYTES = {"f32": 4, "bf16": 2}


def decode_bytes(Hq, Hkv, D, kv_lens, elem_bytes):
    """Q + K + V + O bytes of one decode call over requests with kv_lens."""
    total = 0
    for L in kv_lens:
        total += 2 * Hq * D * elem_bytes            # q row in, o row out
        total += 2 * Hkv * int(L) * D * elem_bytes  # K and V valid rows
    return total


def decode_kv_bytes(Hkv, D, kv_len, elem_bytes):
    return 2 * Hkv * int(kv_len) * D * elem_bytes


def q4_row_bytes(D, group_size=64):
    """Bytes of one K or V row of one KV head in the 4-bit cache."""
    return D // 2 + 2 * 2 * (D // group_size)


def q4_decode_bytes(Hq, Hkv, D, kv_lens, group_size=64):
    total = 0
    for L in kv_lens:
        total += 2 * Hq * D * 2                       # bf16 q in, o out
        total += 2 * Hkv * int(L) * q4_row_bytes(D, group_size)
    return total


def prefill_visible_pairs(q_len, kv_len, causal=True):
    """Number of (query, key) pairs the causal, end-aligned mask keeps."""
    if not causal:
        return q_len * kv_len
    off = kv_len - q_len
    # query i sees keys 0 .. off + i, i.e. off + i + 1 of them
    return q_len * (off + 1) + q_len * (q_len - 1) // 2


def prefill_flops(Hq, D, q_len, kv_len, causal=True, batch=1):
    return 4 * D * Hq * prefill_visible_pairs(q_len, kv_len, causal) * batch


def score_matrix_bytes(Hq, q_len, kv_len, elem_bytes):
    """Bytes of the [Hq, q_len, kv_len] score matrix the unfused path writes."""
    return Hq * q_len * kv_len * elem_bytes


def quantize_bytes(rows: int, D: int, group_size: int = 64) -> int:
    """Bytes moved by 4-bit quantization of `rows` bf16 rows: each row is read
    (2*D bytes) and written as D/2 code bytes plus an fp16 scale and bias per
    group."""
    return rows * (2 * D + D // 2 + 4 * (D // group_size))

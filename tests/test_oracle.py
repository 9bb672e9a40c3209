"""Pins for the fp64 oracle: hand-derived cases, a library routine, closed
forms and invariants of attention.  CPU only.

Each check is chosen so that a plausible slip in the oracle (a dropped
scale, a transposed operand, a wrong head mapping, a top-left instead of
end-aligned mask, a swapped nibble order) fails at least one of them; the
tests at the bottom plant such slips in the oracle and confirm that.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import gqa_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --- hand-derived cases -------------------------------------------------------

@pytest.mark.parametrize("case", _cases()["cases"], ids=lambda c: c["name"])
def test_hand_cases(case):
    out = oracle.attention(np.array(case["q"]), np.array(case["k"]), np.array(case["v"]),
                           kv_lens=case["kv_lens"], scale=case["scale"], causal=case["causal"])
    np.testing.assert_allclose(out["o"], np.array(case["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["lse"], np.array(case["lse"]), rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", _cases()["q4_cases"], ids=lambda c: c["name"])
def test_hand_q4_dequant(case):
    x = oracle.dequant_q4(np.array(case["codes"], dtype=np.uint8),
                          np.array(case["scale"], dtype=np.float16),
                          np.array(case["bias"], dtype=np.float16),
                          group_size=case["group_size"])
    np.testing.assert_array_equal(x, np.array(case["x"]))


# --- library routine: torch float64 SDPA with an explicit end-aligned mask ----

@pytest.mark.parametrize("Hq,Hkv,Tq,L,causal", [
    (14, 2, 1, 37, False), (4, 4, 5, 9, True), (6, 2, 7, 19, True), (8, 1, 3, 3, True)])
def test_matches_torch_sdpa_f64(Hq, Hkv, Tq, L, causal):
    B, D = 2, 16
    q = _rand((B, Hq, Tq, D), 1)
    k = _rand((B, Hkv, L, D), 2)
    v = _rand((B, Hkv, L, D), 3)
    scale = 0.3
    got = oracle.attention(q, k, v, scale=scale, causal=causal)["o"]
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    n_rep = Hq // Hkv
    tk = torch.repeat_interleave(tk, n_rep, dim=1)
    tv = torch.repeat_interleave(tv, n_rep, dim=1)
    # torch's is_causal is aligned top-left; build the end-aligned mask by hand
    i = torch.arange(Tq)[:, None]
    j = torch.arange(L)[None, :]
    mask = (j <= i + (L - Tq)) if causal else torch.ones(Tq, L, dtype=torch.bool)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-12)


# --- invariants and closed forms ----------------------------------------------

def test_gqa_equals_mha_on_repeated_kv():
    q = _rand((2, 12, 3, 8), 4)
    k = _rand((2, 3, 10, 8), 5)
    v = _rand((2, 3, 10, 8), 6)
    a = oracle.attention(q, k, v, kv_lens=[10, 6], causal=True)["o"]
    b = oracle.attention(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1),
                         kv_lens=[10, 6], causal=True)["o"]
    np.testing.assert_array_equal(a, b)


def test_probability_rows_sum_to_one():
    q = _rand((2, 4, 6, 8), 7)
    k = _rand((2, 2, 12, 8), 8)
    v = _rand((2, 2, 12, 8), 9)
    out = oracle.attention(q, k, v, kv_lens=[12, 7], causal=True, return_probs=True)
    for p in out["p"]:
        np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
        assert (p >= 0).all()


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(10)
    k = np.repeat(rng.standard_normal((1, 1, 1, 8)), 9, axis=2)
    v = rng.standard_normal((1, 1, 9, 8))
    q = rng.standard_normal((1, 3, 1, 8))
    o = oracle.attention(q, k, v, kv_lens=[9])["o"]
    np.testing.assert_allclose(o[0, :, 0], np.broadcast_to(v[0, 0].mean(0), (3, 8)), atol=1e-12)


def test_zero_query_gives_mean_of_visible_values():
    v = _rand((1, 2, 11, 4), 11)
    k = _rand((1, 2, 11, 4), 12)
    q = np.zeros((1, 4, 1, 4))
    o = oracle.attention(q, k, v, kv_lens=[7])["o"]
    for h in range(4):
        np.testing.assert_allclose(o[0, h, 0], v[0, h // 2, :7].mean(0), atol=1e-12)


def test_single_visible_key_returns_that_row():
    v = _rand((1, 1, 5, 6), 13)
    k = _rand((1, 1, 5, 6), 14)
    q = _rand((1, 2, 1, 6), 15) * 50
    o = oracle.attention(q, k, v, kv_lens=[1])["o"]
    np.testing.assert_array_equal(o[0, :, 0], np.broadcast_to(v[0, 0, 0], (2, 6)))
    # causal prefill with q_len == kv_len: row 0 sees only key 0
    q2 = _rand((1, 2, 5, 6), 16)
    o2 = oracle.attention(q2, k, v, causal=True)["o"]
    np.testing.assert_array_equal(o2[0, :, 0], np.broadcast_to(v[0, 0, 0], (2, 6)))


def test_chunked_prefill_equals_rows_of_full_prefill():
    # the 512-query chunk at offset 3584 of 4096 keys, scaled down by 16
    T, chunk = 256, 32
    q = _rand((1, 4, T, 8), 17)
    k = _rand((1, 2, T, 8), 18)
    v = _rand((1, 2, T, 8), 19)
    full = oracle.attention(q, k, v, causal=True)["o"]
    part = oracle.attention(q[:, :, T - chunk:], k, v, causal=True)["o"]
    np.testing.assert_allclose(part, full[:, :, T - chunk:], rtol=0, atol=1e-12)


def test_key_permutation_leaves_decode_unchanged():
    q = _rand((1, 4, 1, 8), 20)
    k = _rand((1, 2, 13, 8), 21)
    v = _rand((1, 2, 13, 8), 22)
    perm = np.random.default_rng(23).permutation(13)
    a = oracle.attention(q, k, v)["o"]
    b = oracle.attention(q, k[:, :, perm], v[:, :, perm])["o"]
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_log_sum_exp_split_combine_equals_whole():
    """Combining two key halves with their log-sum-exp weights equals the whole.

    This is the identity a split-KV decode relies on: with lse_s the
    log-sum-exp of part s and o_s its normalised output,
    o = sum_s exp(lse_s - M) o_s / sum_s exp(lse_s - M), M = max_s lse_s.
    """
    q = _rand((1, 4, 1, 8), 24)
    k = _rand((1, 2, 20, 8), 25)
    v = _rand((1, 2, 20, 8), 26)
    whole = oracle.attention(q, k, v)
    a = oracle.attention(q, k[:, :, :7], v[:, :, :7])
    b = oracle.attention(q, k[:, :, 7:], v[:, :, 7:])
    M = np.maximum(a["lse"], b["lse"])
    wa = np.exp(a["lse"] - M)[..., None]
    wb = np.exp(b["lse"] - M)[..., None]
    o = (wa * a["o"] + wb * b["o"]) / (wa + wb)
    np.testing.assert_allclose(o, whole["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(M + np.log(wa + wb)[..., 0], whole["lse"], atol=1e-12)


def test_large_scale_selects_argmax_key():
    q = _rand((1, 1, 1, 8), 27)
    k = _rand((1, 1, 9, 8), 28)
    v = _rand((1, 1, 9, 8), 29)
    j = int(np.argmax(k[0, 0] @ q[0, 0, 0]))
    o = oracle.attention(q, k, v, scale=1e4)["o"]
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, j], atol=1e-9)


def test_empty_request_is_zero():
    q = _rand((2, 2, 1, 4), 30)
    k = _rand((2, 1, 3, 4), 31)
    v = _rand((2, 1, 3, 4), 32)
    out = oracle.attention(q, k, v, kv_lens=[0, 3])
    assert (out["o"][0] == 0).all()
    assert np.isneginf(out["lse"][0]).all()


def test_rows_past_kv_len_are_not_read():
    q = _rand((1, 2, 1, 4), 33)
    k = _rand((1, 1, 6, 4), 34)
    v = _rand((1, 1, 6, 4), 35)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 4:] = np.nan
    v2[:, :, 4:] = np.nan
    a = oracle.attention(q, k, v, kv_lens=[4])["o"]
    b = oracle.attention(q, k2, v2, kv_lens=[4])["o"]
    np.testing.assert_array_equal(a, b)


def test_brute_force_loops_tiny():
    """Scalar loops with math.exp on tiny random inputs (grouped, causal)."""
    B, Hq, Hkv, Tq, D = 1, 4, 2, 3, 3
    L = 5
    q = _rand((B, Hq, Tq, D), 36)
    k = _rand((B, Hkv, L, D), 37)
    v = _rand((B, Hkv, L, D), 38)
    scale = 0.7
    got = oracle.attention(q, k, v, scale=scale, causal=True)["o"]
    for h in range(Hq):
        g = h // (Hq // Hkv)
        for i in range(Tq):
            vis = [j for j in range(L) if j <= i + L - Tq]
            s = [scale * sum(q[0, h, i, d] * k[0, g, j, d] for d in range(D)) for j in vis]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            z = sum(e)
            for d in range(D):
                ref = sum(e[t] / z * v[0, g, j, d] for t, j in enumerate(vis))
                assert abs(got[0, h, i, d] - ref) < 1e-12


def test_q4_attention_equals_attention_on_dequantised_cache():
    rng = np.random.default_rng(39)
    B, Hq, Hkv, D, S, G = 2, 4, 2, 128, 9, 64
    kc = rng.integers(0, 256, (B, Hkv, S, D // 2), dtype=np.uint8)
    vc = rng.integers(0, 256, (B, Hkv, S, D // 2), dtype=np.uint8)
    ks = rng.uniform(0.1, 0.5, (B, Hkv, S, D // G)).astype(np.float16)
    kb = rng.uniform(-3, -1, (B, Hkv, S, D // G)).astype(np.float16)
    vs = rng.uniform(0.1, 0.5, (B, Hkv, S, D // G)).astype(np.float16)
    vb = rng.uniform(-3, -1, (B, Hkv, S, D // G)).astype(np.float16)
    q = rng.standard_normal((B, Hq, 1, D))

    def deq(c, s, b):   # element-wise loop form, independent of dequant_q4
        out = np.zeros(c.shape[:-1] + (D,))
        for idx in np.ndindex(*c.shape[:-1]):
            for d in range(D):
                byte = int(c[idx + (d // 2,)])
                code = (byte >> 4) if d % 2 else (byte & 15)
                out[idx + (d,)] = code * float(s[idx + (d // G,)]) + float(b[idx + (d // G,)])
        return out

    got = oracle.attention_q4(q, kc, ks, kb, vc, vs, vb, kv_lens=[9, 4])["o"]
    ref = oracle.attention(q, deq(kc, ks, kb), deq(vc, vs, vb), kv_lens=[9, 4])["o"]
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_quantizer_round_trip_error_is_half_a_step():
    """The input builder's codes dequantise to within scale/2 (+fp16 rounding)."""
    from gqa_attention_kv_decode_gb300 import inputs
    x = inputs.randn((2, 2, 17, 128), 40, torch.bfloat16)
    c, s, b = inputs.quantize_q4(x)
    deq = oracle.dequant_q4(c.numpy(), s.numpy(), b.numpy())
    err = np.abs(deq - x.float().numpy())
    step = np.repeat(s.float().numpy(), 64, axis=-1)
    assert (err <= step * 0.5 + 1e-2 * step + 2e-3).all()


# --- planted mistakes: each one must be caught by a pin above -----------------

def _golden_fails():
    try:
        for case in _cases()["cases"]:
            test_hand_cases(case)
    except AssertionError:
        return True
    return False


def test_pins_catch_wrong_head_mapping(monkeypatch):
    def bad_repeat(x, n_rep):
        x = np.asarray(x, dtype=np.float64)
        hkv = x.shape[1]
        return x[:, np.arange(hkv * n_rep) % hkv].copy()
    monkeypatch.setattr(gqa_oracle, "repeat_kv", bad_repeat)
    assert _golden_fails()


def test_pins_catch_top_left_causal_mask(monkeypatch):
    def bad_mask(q_len, kv_len, causal):
        i = np.arange(q_len)[:, None]
        j = np.arange(kv_len)[None, :]
        return (j <= i) if causal else np.ones((q_len, kv_len), dtype=bool)
    monkeypatch.setattr(gqa_oracle, "visible_mask", bad_mask)
    assert _golden_fails()


def test_pins_catch_dropped_scale(monkeypatch):
    real = gqa_oracle.attention

    def no_scale(q, k, v, kv_lens=None, scale=None, causal=False, return_probs=False):
        return real(q, k, v, kv_lens=kv_lens, scale=1.0, causal=causal, return_probs=return_probs)
    monkeypatch.setattr(oracle, "attention", no_scale)
    assert _golden_fails()


def test_pins_catch_swapped_nibbles(monkeypatch):
    case = _cases()["q4_cases"][0]
    codes = np.array(case["codes"], dtype=np.uint8)
    swapped = ((codes & 15) << 4) | (codes >> 4)
    x = oracle.dequant_q4(swapped, np.array(case["scale"], dtype=np.float16),
                          np.array(case["bias"], dtype=np.float16), group_size=case["group_size"])
    assert not np.array_equal(x, np.array(case["x"]))


# --- paged cache: a relabeling of rows, and the append -------------------------

@pytest.mark.parametrize("case", _cases()["paged_cases"], ids=lambda c: c["name"])
def test_hand_paged_cases(case):
    kn = np.array(case["k_new"]) if "k_new" in case else None
    vn = np.array(case["v_new"]) if "v_new" in case else None
    out = oracle.attention_paged(np.array(case["q"]), np.array(case["k_pool"]), np.array(case["v_pool"]),
                                 case["block_table"], case["kv_lens"], case["block_size"],
                                 scale=case["scale"], k_new=kn, v_new=vn)
    np.testing.assert_allclose(out["o"], np.array(case["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["lse"], np.array(case["lse"]), rtol=0, atol=1e-12)
    if "k_pool_after" in case:
        np.testing.assert_array_equal(out["k_pool"], np.array(case["k_pool_after"]))
        np.testing.assert_array_equal(out["v_pool"], np.array(case["v_pool_after"]))


def _paged_from_contiguous(k, v, kv_lens, block_size, seed):
    """Cut a contiguous cache into blocks, shuffle them into a larger pool
    (with unused blocks full of NaN) and build the block table."""
    B, hkv, S, D = k.shape
    nb = -(-S // block_size)
    n_pool = B * nb + 3
    rng = np.random.default_rng(seed)
    slots = rng.permutation(n_pool)
    kp = np.full((n_pool, hkv, block_size, D), np.nan)
    vp = np.full((n_pool, hkv, block_size, D), np.nan)
    table = np.zeros((B, nb), dtype=np.int32)
    for b in range(B):
        for i in range(nb):
            blk = slots[b * nb + i]
            table[b, i] = blk
            rows = slice(i * block_size, min(S, (i + 1) * block_size))
            n = rows.stop - rows.start
            kp[blk, :, :n] = k[b, :, rows]
            vp[blk, :, :n] = v[b, :, rows]
    return kp, vp, table


@pytest.mark.parametrize("block_size", [1, 4, 16])
def test_paged_attention_equals_contiguous(block_size):
    B, Hq, Hkv, S, D = 3, 6, 2, 37, 8
    q = _rand((B, Hq, 1, D), 41)
    k = _rand((B, Hkv, S, D), 42)
    v = _rand((B, Hkv, S, D), 43)
    kv_lens = [37, 1, 20]
    kp, vp, table = _paged_from_contiguous(k, v, kv_lens, block_size, 44)
    got = oracle.attention_paged(q, kp, vp, table, kv_lens, block_size)
    want = oracle.attention(q, k, v, kv_lens=kv_lens)
    np.testing.assert_allclose(got["o"], want["o"], rtol=0, atol=1e-12)
    dense = oracle.paged_to_contiguous(kp, table, kv_lens, block_size)
    for b, L in enumerate(kv_lens):
        np.testing.assert_array_equal(dense[b, :, :L], k[b, :, :L])


def test_paged_append_equals_contiguous_with_new_row():
    B, Hq, Hkv, S, D, bs = 2, 4, 2, 24, 8, 8
    q = _rand((B, Hq, 1, D), 51)
    k = _rand((B, Hkv, S, D), 52)
    v = _rand((B, Hkv, S, D), 53)
    kn = _rand((B, Hkv, 1, D), 54)
    vn = _rand((B, Hkv, 1, D), 55)
    kv_lens = [17, 8]  # the new tokens land in row 0 of a block and in the last row of one
    kp, vp, table = _paged_from_contiguous(k, v, kv_lens, bs, 56)
    got = oracle.attention_paged(q, kp, vp, table, kv_lens, bs, k_new=kn, v_new=vn)
    k2, v2 = k.copy(), v.copy()
    for b, L in enumerate(kv_lens):
        k2[b, :, L - 1] = kn[b, :, 0]
        v2[b, :, L - 1] = vn[b, :, 0]
    want = oracle.attention(q, k2, v2, kv_lens=kv_lens)
    np.testing.assert_allclose(got["o"], want["o"], rtol=0, atol=1e-12)
    # exactly the two slots changed in each pool
    changed = ~np.isclose(got["k_pool"], kp, equal_nan=True)
    assert changed.any(axis=(1, 3)).sum() == len(kv_lens)


def test_pins_catch_paged_row_index_slip(monkeypatch):
    def bad_gather(pool, block_table, kv_lens, block_size):
        pool = np.asarray(pool, dtype=np.float64)
        table = np.asarray(block_table, dtype=np.int64)
        out = np.zeros((table.shape[0], pool.shape[1], max(1, int(max(kv_lens))), pool.shape[3]))
        for b in range(table.shape[0]):
            for j in range(int(kv_lens[b])):  # block index and row swapped
                out[b, :, j, :] = pool[table[b, j % block_size], :, j // block_size, :]
        return out
    monkeypatch.setattr(gqa_oracle, "paged_to_contiguous", bad_gather)
    # (the hand cases select the same set of rows either way: only a larger
    # relabeling tells the two apart)
    with pytest.raises((AssertionError, IndexError)):
        test_paged_attention_equals_contiguous(4)


def test_pins_catch_append_off_by_one(monkeypatch):
    real = gqa_oracle.append_paged

    def late_append(k_pool, v_pool, block_table, kv_lens, block_size, k_new, v_new):
        return real(k_pool, v_pool, block_table, [int(x) + 1 for x in kv_lens], block_size, k_new, v_new)
    monkeypatch.setattr(gqa_oracle, "append_paged", late_append)
    with pytest.raises((AssertionError, IndexError)):
        test_paged_append_equals_contiguous_with_new_row()


# --- the 4-bit quantizer --------------------------------------------------------

@pytest.mark.parametrize("case", _cases()["quantizer_cases"], ids=lambda c: c["name"])
def test_hand_quantizer_cases(case):
    c, s, b = oracle.quantize_q4(np.array(case["x"], dtype=np.float32), case["group_size"])
    np.testing.assert_array_equal(c, np.array(case["codes"], dtype=np.uint8))
    np.testing.assert_array_equal(s.astype(np.float64), np.array(case["scale"]))
    np.testing.assert_array_equal(b.astype(np.float64), np.array(case["bias"]))


def test_quantizer_invariants():
    """Round trip within half a step; the group minimum gets code 0 and the
    maximum code 15; codes are monotone in x within a group."""
    x = torch.randn((3, 5, 256), generator=torch.Generator().manual_seed(61)).to(torch.bfloat16).float().numpy()
    c, s, b = oracle.quantize_q4(x)
    deq = oracle.dequant_q4(c, s, b)
    step = np.repeat(s.astype(np.float64), 64, axis=-1)
    assert (np.abs(deq - x) <= 0.5 * step + 1e-2 * step + 2e-3).all()
    codes = np.empty(x.shape, dtype=np.int64)
    codes[..., 0::2] = c & 15
    codes[..., 1::2] = c >> 4
    g = x.reshape(3, 5, 4, 64)
    cg = codes.reshape(3, 5, 4, 64)
    assert (np.take_along_axis(cg, g.argmin(-1)[..., None], -1) == 0).all()
    assert (np.take_along_axis(cg, g.argmax(-1)[..., None], -1) == 15).all()
    order = np.argsort(g, axis=-1, kind="stable")
    assert (np.diff(np.take_along_axis(cg, order, -1), axis=-1) >= 0).all()


def test_pins_catch_quantizer_slips(monkeypatch):
    real = np.rint
    monkeypatch.setattr(np, "rint", np.trunc)  # round toward zero instead of to nearest even
    with pytest.raises(AssertionError):
        for case in _cases()["quantizer_cases"]:
            test_hand_quantizer_cases(case)
    monkeypatch.setattr(np, "rint", real)
    case = _cases()["quantizer_cases"][0]
    c, _, _ = oracle.quantize_q4(np.array(case["x"], dtype=np.float32))
    swapped = ((c & 15) << 4) | (c >> 4)
    assert not np.array_equal(swapped, np.array(case["codes"], dtype=np.uint8))


def test_pin_separates_division_from_reciprocal():
    """A quantizer that multiplies by the fp32 reciprocal of the scale instead
    of dividing by it fails the 'division_ties_not_reciprocal' hand case."""
    case = next(c for c in _cases()["quantizer_cases"] if c["name"] == "division_ties_not_reciprocal")
    x = np.array(case["x"], dtype=np.float32)
    c, _, _ = oracle.quantize_q4(x)
    np.testing.assert_array_equal(c, np.array(case["codes"], dtype=np.uint8))
    # the same group, quotients formed with the reciprocal
    s = np.float32(case["scale"][0])
    alt = np.clip(np.rint(x * (np.float32(1.0) / s)), 0, 15).astype(np.uint8)
    alt_packed = alt[0::2] | (alt[1::2] << 4)
    assert not np.array_equal(alt_packed, np.array(case["codes"], dtype=np.uint8))
    assert alt_packed[:3].tolist() == [240, 215, 63]


# --- 4-bit cache with an unquantized residual window ------------------------------

@pytest.mark.parametrize("case", _cases()["residual_cases"], ids=lambda c: c["name"])
def test_hand_residual_cases(case):
    f16 = lambda a: np.array(a, dtype=np.float16)
    out = oracle.attention_q4_residual(
        np.array(case["q"]), np.array(case["k_codes"], dtype=np.uint8), f16(case["k_scale"]), f16(case["k_bias"]),
        np.array(case["v_codes"], dtype=np.uint8), f16(case["v_scale"]), f16(case["v_bias"]),
        np.array(case["k_res"]), np.array(case["v_res"]), case["n_quant"], case["kv_lens"], scale=case["scale"])
    np.testing.assert_allclose(out["o"], np.array(case["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["lse"], np.array(case["lse"]), rtol=0, atol=1e-12)


def _q4_and_residual(B, Hkv, S, R, D, seed):
    from gqa_attention_kv_decode_gb300 import inputs
    kc, ks, kb, vc, vs, vb = (t.numpy() for t in inputs.q4_cache(B, Hkv, D, S, layer=seed))
    kr = inputs.randn((B, Hkv, R, D), 900 + seed, torch.bfloat16).float().numpy()
    vr = inputs.randn((B, Hkv, R, D), 901 + seed, torch.bfloat16).float().numpy()
    return kc, ks, kb, vc, vs, vb, kr, vr


def test_residual_window_reduces_to_the_two_parts():
    """All keys quantized: the q4 oracle.  No key quantized: plain attention on
    the residual window."""
    B, Hq, Hkv, S, R, D = 2, 8, 2, 40, 16, 64
    kc, ks, kb, vc, vs, vb, kr, vr = _q4_and_residual(B, Hkv, S, R, D, 1)
    q = _rand((B, Hq, 1, D), 77)
    lens = [40, 9]
    got = oracle.attention_q4_residual(q, kc, ks, kb, vc, vs, vb, kr, vr, lens, lens)
    want = oracle.attention_q4(q, kc, ks, kb, vc, vs, vb, kv_lens=lens)
    np.testing.assert_allclose(got["o"], want["o"], rtol=0, atol=1e-12)
    lens = [16, 3]
    got = oracle.attention_q4_residual(q, kc, ks, kb, vc, vs, vb, kr, vr, [0, 0], lens)
    want = oracle.attention(q, kr, vr, kv_lens=lens)
    np.testing.assert_allclose(got["o"], want["o"], rtol=0, atol=1e-12)


def test_residual_flush_moves_a_block_without_changing_the_keys():
    """Flushing the oldest block of the window into the 4-bit cache (as
    dequantised values) leaves the attended key set, hence the output, the
    same: a row is either in the cache or in the window, never both."""
    B, Hq, Hkv, S, R, D = 1, 4, 1, 64, 32, 64
    kc, ks, kb, vc, vs, vb, kr, vr = _q4_and_residual(B, Hkv, S, R, D, 2)
    q = _rand((B, Hq, 1, D), 78)
    # window holds rows 20..43 of the sequence; then rows 20..35 move to the cache
    nq, L = 20, 44
    before = oracle.attention_q4_residual(q, kc, ks, kb, vc, vs, vb, kr, vr, [nq], [L])
    kc2, ks2, kb2, vc2, vs2, vb2 = (a.copy() for a in (kc, ks, kb, vc, vs, vb))
    kq, ksq, kbq = oracle.quantize_q4(kr[:, :, :16])
    vq, vsq, vbq = oracle.quantize_q4(vr[:, :, :16])
    kc2[:, :, nq:nq + 16], ks2[:, :, nq:nq + 16], kb2[:, :, nq:nq + 16] = kq, ksq, kbq
    vc2[:, :, nq:nq + 16], vs2[:, :, nq:nq + 16], vb2[:, :, nq:nq + 16] = vq, vsq, vbq
    kr2 = np.zeros_like(kr)
    vr2 = np.zeros_like(vr)
    kr2[:, :, :L - nq - 16] = kr[:, :, 16:L - nq]
    vr2[:, :, :L - nq - 16] = vr[:, :, 16:L - nq]
    after = oracle.attention_q4_residual(q, kc2, ks2, kb2, vc2, vs2, vb2, kr2, vr2, [nq + 16], [L])
    # the same keys, except that the flushed rows are now quantized: compare
    # against the window with those rows replaced by their dequantised values
    kr3, vr3 = kr.copy(), vr.copy()
    kr3[:, :, :16] = oracle.dequant_q4(kq, ksq, kbq)
    vr3[:, :, :16] = oracle.dequant_q4(vq, vsq, vbq)
    ref = oracle.attention_q4_residual(q, kc, ks, kb, vc, vs, vb, kr3, vr3, [nq], [L])
    np.testing.assert_allclose(after["o"], ref["o"], rtol=0, atol=1e-12)
    assert not np.allclose(after["o"], before["o"], atol=1e-9)  # quantizing changed the values


def test_pins_catch_residual_offset_slip(monkeypatch):
    real = gqa_oracle.attention_q4_residual

    def off_by_one(q, kc, ks, kb, vc, vs, vb, kr, vr, n_quant, kv_lens, scale=None, group_size=64):
        return real(q, kc, ks, kb, vc, vs, vb, kr, vr, [max(0, int(n) - 1) for n in n_quant], kv_lens,
                    scale=scale, group_size=group_size)
    monkeypatch.setattr(oracle, "attention_q4_residual", off_by_one)
    with pytest.raises(AssertionError):
        for case in _cases()["residual_cases"]:
            test_hand_residual_cases(case)

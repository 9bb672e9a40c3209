"""Writes stay inside their buffers, and requests do not see each other.

Canaries: the output and the workspace are views into larger buffers whose
guard regions before and after hold a known pattern; after the call every
guard byte must be unchanged (a stray store past O or past the workspace
fails).  Batch independence: with the split count fixed (the plan override),
a request's keys are cut into the same splits whatever else is in the
batch, so its output must be bit for bit the same alone as inside a batch of
requests with other lengths.  Seeded, distinct data per request and head, so
a swapped stride cannot pass.
"""

import pytest
import torch

from gqa_attention_kv_decode_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 64  # elements of O (>= 128 bytes, so the view stays 16-byte aligned)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def guarded_like(t, fill=7.0):
    """A buffer GUARD elements larger on each side; returns (buffer, view)."""
    buf = torch.full((t.numel() + 2 * GUARD,), fill, dtype=t.dtype, device=DEV)
    return buf, buf[GUARD:GUARD + t.numel()].view(t.shape)


def guarded_workspace(n_bytes):
    """Workspace view with 4 KiB guards of 0xA5 around it; the status word
    (the first 256 bytes) starts at zero."""
    buf = torch.full((n_bytes + 8192,), 0xA5, dtype=torch.uint8, device=DEV)
    ws = buf[4096:4096 + n_bytes]
    ws[:256] = 0
    return buf, ws


def check_guards(obuf, n_o, fill, wsbuf=None, n_ws=0):
    torch.cuda.synchronize()
    assert (obuf[:GUARD] == fill).all() and (obuf[GUARD + n_o:] == fill).all(), "a store left O"
    if wsbuf is not None:
        assert (wsbuf[:4096] == 0xA5).all() and (wsbuf[4096 + n_ws:] == 0xA5).all(), "a store left the workspace"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("S,splits", [(64, 0), (3000, 0), (3000, 1000)], ids=["short", "planned", "many_splits"])
def test_decode_canaries(dtype, S, splits):
    B, Hq, Hkv, D = 3, 28, 4, 128
    q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, S, dtype, layer=81, device=DEV)
    lens = torch.tensor([S, max(1, S // 3), 1], dtype=torch.int32, device=DEV)
    obuf, o = guarded_like(q)
    with binding.plan_override(decode_splits=splits):  # (the size follows the forced plan)
        n_ws = binding.gqa_attn_decode_workspace_size(B, Hq, Hkv, D, S, binding._dtype_code(q))
        wsbuf, ws = guarded_workspace(n_ws)
        binding.gqa_attn_decode(q, k, v, o, lens, D ** -0.5, ws)
    check_guards(obuf, o.numel(), 7.0, wsbuf, n_ws)
    assert torch.isfinite(o).all()


def test_q4_decode_canaries():
    B, Hq, Hkv, D, S = 2, 32, 8, 128, 2048
    kc, ks, kb, vc, vs, vb = inputs.q4_cache(B, Hkv, D, S, layer=82, device=DEV)
    q = inputs.randn((B, Hq, 1, D), 83, torch.bfloat16, DEV)
    lens = torch.tensor([S, 700], dtype=torch.int32, device=DEV)
    obuf, o = guarded_like(q)
    n_ws = binding.gqa_attn_decode_q4_workspace_size(B, Hq, Hkv, D, S)
    wsbuf, ws = guarded_workspace(n_ws)
    binding.gqa_attn_decode_q4(q, kc, ks, kb, vc, vs, vb, o, lens, D ** -0.5, ws)
    check_guards(obuf, o.numel(), 7.0, wsbuf, n_ws)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("q_len,kv_len,ks", [(1000, 1000, 0), (513, 513, 0), (300, 2000, 4)])
def test_prefill_canaries(D, q_len, kv_len, ks):
    q = inputs.randn((1, 14, q_len, D), 84, torch.bfloat16, DEV)
    k = inputs.randn((1, 2, kv_len, D), 85, torch.bfloat16, DEV)
    v = inputs.randn((1, 2, kv_len, D), 86, torch.bfloat16, DEV)
    obuf, o = guarded_like(q)
    with binding.plan_override(prefill_kv_split=ks):
        binding.gqa_attn_prefill(q, k, v, o, kv_len, D ** -0.5, True)
    check_guards(obuf, o.numel(), 7.0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_request_alone_equals_request_in_batch(dtype, D):
    """Four requests of different lengths decoded together and each alone,
    with the split count fixed: the outputs agree bit for bit."""
    Hq, Hkv, S = 28, 4, 3000
    lens = [3000, 1777, 64, 2500]
    B = len(lens)
    q, k, v = inputs.qkv(B, Hq, Hkv, D, 1, S, dtype, layer=90 + D, device=DEV)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    with binding.plan_override(decode_splits=6):
        together = binding.decode(q, k, v, kv_lens=lens_t, max_kv_len=S)
        alone = [binding.decode(q[b:b + 1].contiguous(), k[b:b + 1].contiguous(), v[b:b + 1].contiguous(),
                                kv_lens=lens_t[b:b + 1].contiguous(), max_kv_len=S) for b in range(B)]
    torch.cuda.synchronize()
    for b in range(B):
        assert torch.equal(together[b:b + 1], alone[b]), f"request {b}"


def test_q4_request_alone_equals_request_in_batch():
    Hq, Hkv, D, S = 32, 8, 128, 2048
    lens = [2048, 999, 64]
    B = len(lens)
    kc, ks, kb, vc, vs, vb = inputs.q4_cache(B, Hkv, D, S, layer=95, device=DEV)
    q = inputs.randn((B, Hq, 1, D), 96, torch.bfloat16, DEV)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    with binding.plan_override(decode_splits=5):
        together = binding.decode_q4(q, kc, ks, kb, vc, vs, vb, kv_lens=lens_t, max_kv_len=S)
        alone = [binding.decode_q4(q[b:b + 1].contiguous(), *(t[b:b + 1].contiguous() for t in (kc, ks, kb, vc, vs, vb)),
                                   kv_lens=lens_t[b:b + 1].contiguous(), max_kv_len=S) for b in range(B)]
    torch.cuda.synchronize()
    for b in range(B):
        assert torch.equal(together[b:b + 1], alone[b]), f"request {b}"

"""ctypes binding over libgqa_attn.so (include/gqa_attn.h).

The functions named like the C entry points take torch tensors, check that
they are dense (the C ABI cannot see strides), pass ``data_ptr()`` values,
sizes and the CUDA stream handle, and raise ``GqaAttnError`` on a non-zero
status.  Every step of the computation runs in the library's kernels; there
is no Python or CPU implementation behind these names.  If the library has
not been built, the first call raises instead of falling back to anything.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgqa_attn.so")

GQA_OK = 0
GQA_ERR_INVALID_ARG = -1
GQA_ERR_UNSUPPORTED = -2
GQA_ERR_NOT_DEVICE_PTR = -3
GQA_ERR_CUDA = -4
GQA_ERR_WORKSPACE = -5
GQA_ERR_SCRATCH_LIMIT = -6

GQA_F32 = 0
GQA_BF16 = 1

GQA_DEV_KVLEN_CLAMPED = 1
GQA_DEV_EMPTY_REQUEST = 2
GQA_DEV_WAIT_TIMEOUT = 4
GQA_DEV_BAD_BLOCK = 8

EXPORTED = (
    "gqa_attn_decode_workspace_size",
    "gqa_attn_decode",
    "gqa_attn_decode_noalloc",
    "gqa_attn_decode_paged",
    "gqa_attn_decode_layers_workspace_size",
    "gqa_attn_decode_layers",
    "gqa_attn_quantize_q4",
    "gqa_attn_decode_q4_residual_workspace_size",
    "gqa_attn_decode_q4_residual",
    "gqa_attn_decode_q4_workspace_size",
    "gqa_attn_decode_q4",
    "gqa_attn_prefill",
    "gqa_attn_prefill_varlen",
    "gqa_attn_status_string",
    "gqa_attn_read_device_status",
    "gqa_attn_clear_device_status",
    "gqa_attn_decode_num_splits",
    "gqa_attn_decode_plan_for",
    "gqa_attn_version",
    "gqa_attn_set_plan_override",
    "gqa_attn_set_prefill_interleave_override",
    "gqa_attn_set_wait_test",
    "gqa_attn_read_prefill_status",
    "gqa_attn_clear_prefill_status",
)

_lib = None


class GqaAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().gqa_attn_status_string(status).decode()
        super().__init__(f"{where}: {msg} ({status})")


def lib() -> ctypes.CDLL:
    """Loads libgqa_attn.so once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -m gqa_attention_kv_decode_gb300.build` "
            "(there is no CPU or Python fallback)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    L.gqa_attn_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
    L.gqa_attn_decode_workspace_size.restype = sz
    L.gqa_attn_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
    L.gqa_attn_decode.restype = i32
    L.gqa_attn_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp]
    L.gqa_attn_decode_noalloc.restype = i32
    L.gqa_attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                        i32, f32, i32, vp, sz, vp]
    L.gqa_attn_decode_paged.restype = i32
    L.gqa_attn_decode_layers_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    L.gqa_attn_decode_layers_workspace_size.restype = sz
    L.gqa_attn_decode_layers.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32, vp,
                                         sz, vp]
    L.gqa_attn_decode_layers.restype = i32
    i64 = ctypes.c_int64
    L.gqa_attn_quantize_q4.argtypes = [vp, i64, vp, vp, vp, i64, i64, i32, i32, i32, i32, vp]
    L.gqa_attn_quantize_q4.restype = i32
    L.gqa_attn_decode_q4_residual_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.gqa_attn_decode_q4_residual_workspace_size.restype = sz
    L.gqa_attn_decode_q4_residual.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                              i32, i32, i32, i32, i32, i32, i32, i32, f32, vp, sz, vp]
    L.gqa_attn_decode_q4_residual.restype = i32
    L.gqa_attn_decode_q4_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.gqa_attn_decode_q4_workspace_size.restype = sz
    L.gqa_attn_decode_q4.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                     i32, i32, i32, i32, i32, i32, i32, f32, vp, sz, vp]
    L.gqa_attn_decode_q4.restype = i32
    L.gqa_attn_prefill.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32, i32, vp]
    L.gqa_attn_prefill.restype = i32
    L.gqa_attn_prefill_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, i32, vp]
    L.gqa_attn_prefill_varlen.restype = i32
    L.gqa_attn_status_string.argtypes = [i32]
    L.gqa_attn_status_string.restype = ctypes.c_char_p
    L.gqa_attn_read_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    L.gqa_attn_read_device_status.restype = i32
    L.gqa_attn_clear_device_status.argtypes = [vp, vp]
    L.gqa_attn_clear_device_status.restype = i32
    L.gqa_attn_decode_num_splits.argtypes = [i32, i32, i32, i32, i32, i32]
    L.gqa_attn_decode_num_splits.restype = i32
    i32p = ctypes.POINTER(ctypes.c_int32)
    L.gqa_attn_decode_plan_for.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32p, i32p, i32p]
    L.gqa_attn_decode_plan_for.restype = i32
    L.gqa_attn_version.argtypes = []
    L.gqa_attn_version.restype = i32
    L.gqa_attn_set_plan_override.argtypes = [i32, i32]
    L.gqa_attn_set_plan_override.restype = i32
    L.gqa_attn_set_prefill_interleave_override.argtypes = [i32]
    L.gqa_attn_set_prefill_interleave_override.restype = i32
    L.gqa_attn_set_wait_test.argtypes = [ctypes.c_uint64]
    L.gqa_attn_set_wait_test.restype = i32
    L.gqa_attn_read_prefill_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
    L.gqa_attn_read_prefill_status.restype = i32
    L.gqa_attn_clear_prefill_status.argtypes = [vp]
    L.gqa_attn_clear_prefill_status.restype = i32
    _lib = L
    return L


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GQA_F32
    if t.dtype == torch.bfloat16:
        return GQA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: float32 or bfloat16")


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libgqa_attn must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(rc: int, where: str):
    if rc != GQA_OK:
        raise GqaAttnError(rc, where)


# --- entry points (same names as the C ABI) ----------------------------------

def gqa_attn_decode_workspace_size(B, Hq, Hkv, D, max_kv_len, dtype) -> int:
    return lib().gqa_attn_decode_workspace_size(B, Hq, Hkv, D, max_kv_len, dtype)


def gqa_attn_decode_num_splits(B, Hq, Hkv, D, max_kv_len, dtype) -> int:
    return lib().gqa_attn_decode_num_splits(B, Hq, Hkv, D, max_kv_len, dtype)


GQA_PLAN_DECODE, GQA_PLAN_PAGED, GQA_PLAN_Q4 = 0, 1, 2


def gqa_attn_decode_plan_for(B, Hq, Hkv, D, max_kv_len, dtype, num_sms, variant=GQA_PLAN_DECODE):
    """(n_split, chunk, tile) of a decode plan for a device of num_sms SMs."""
    n_split, chunk, tile = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    rc = lib().gqa_attn_decode_plan_for(B, Hq, Hkv, D, max_kv_len, dtype, variant, num_sms, ctypes.byref(n_split),
                                        ctypes.byref(chunk), ctypes.byref(tile))
    _check(rc, "gqa_attn_decode_plan_for")
    return n_split.value, chunk.value, tile.value


def gqa_attn_set_plan_override(decode_splits=0, prefill_kv_split=0) -> None:
    """Tuning and tests only: force the decode split count and the prefill
    KV-split cluster size (0 = the planner's choice)."""
    _check(lib().gqa_attn_set_plan_override(int(decode_splits), int(prefill_kv_split)),
           "gqa_attn_set_plan_override")


def gqa_attn_set_wait_test(stall_ns=0) -> None:
    """Tests only: later decode and prefill launches take the path of a copy
    that never lands (a wait of stall_ns on a barrier nothing arrives on), so
    they report GQA_DEV_WAIT_TIMEOUT; 0 turns it off."""
    _check(lib().gqa_attn_set_wait_test(int(stall_ns)), "gqa_attn_set_wait_test")


def gqa_attn_set_prefill_interleave_override(from_pair=-1) -> None:
    """Tuning and tests only: prefill pairs from index from_pair on run as
    single query tiles whose keys the two softmax warpgroups take in turn
    (0 = every tile; past the last pair = none; negative = the planner)."""
    _check(lib().gqa_attn_set_prefill_interleave_override(int(from_pair)),
           "gqa_attn_set_prefill_interleave_override")


@contextlib.contextmanager
def plan_override(decode_splits=0, prefill_kv_split=0, prefill_interleave_from=-1):
    """``with plan_override(...)``: the overrides for the block, then none."""
    gqa_attn_set_plan_override(decode_splits, prefill_kv_split)
    gqa_attn_set_prefill_interleave_override(prefill_interleave_from)
    try:
        yield
    finally:
        gqa_attn_set_plan_override(0, 0)
        gqa_attn_set_prefill_interleave_override(-1)


def gqa_attn_decode(q, k, v, o, kv_lens, scale, workspace, max_kv_len=None, stream=None):
    """q, o [B,Hq,1,D]; k, v [B,Hkv,S_cap,D]; kv_lens int32 [B] or None."""
    B, Hq, Tq, D = q.shape
    Hkv, S_cap = k.shape[1], k.shape[2]
    if Tq != 1:
        raise ValueError("decode takes one query row per request")
    if max_kv_len is None:
        max_kv_len = S_cap
    rc = lib().gqa_attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(kv_lens), B, Hq, Hkv, D,
                               S_cap, int(max_kv_len), float(scale), _dtype_code(q),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
    _check(rc, "gqa_attn_decode")


def gqa_attn_decode_noalloc(q, k, v, o, kv_lens, scale, max_kv_len=None, stream=None):
    """gqa_attn_decode without a workspace: the library's built-in scratch is
    used (for callers that cannot allocate; calls must not overlap on the GPU)."""
    B, Hq, Tq, D = q.shape
    Hkv, S_cap = k.shape[1], k.shape[2]
    if Tq != 1:
        raise ValueError("decode takes one query row per request")
    if max_kv_len is None:
        max_kv_len = S_cap
    rc = lib().gqa_attn_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(kv_lens), B, Hq, Hkv,
                                       D, S_cap, int(max_kv_len), float(scale), _dtype_code(q),
                                       _stream(stream))
    _check(rc, "gqa_attn_decode_noalloc")


def gqa_attn_decode_paged(q, k_new, v_new, k_pool, v_pool, block_table, kv_lens, o, scale, workspace,
                          max_kv_len, stream=None):
    """q, o [B,Hq,1,D]; k_pool, v_pool [num_blocks,Hkv,block_size,D] (modified
    when k_new, v_new [B,Hkv,1,D] are given: the new token goes to row
    kv_lens[b]-1); block_table int32 [B,max_blocks]; kv_lens int32 [B]."""
    B, Hq, Tq, D = q.shape
    num_blocks, Hkv, block_size = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    if Tq != 1:
        raise ValueError("decode takes one query row per request")
    if block_table.dtype != torch.int32 or kv_lens.dtype != torch.int32:
        raise TypeError("block_table and kv_lens are int32")
    rc = lib().gqa_attn_decode_paged(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                                     _ptr(block_table), _ptr(kv_lens), _ptr(o), B, Hq, Hkv, D,
                                     block_size, num_blocks, block_table.shape[1], int(max_kv_len),
                                     float(scale), _dtype_code(q), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "gqa_attn_decode_paged")


def gqa_attn_quantize_q4(src, codes, scale, bias, dst_row0=0, rows=None, group_size=64, stream=None):
    """src bf16 [B,Hkv,S_src,D]; codes uint8 [B,Hkv,S_cap,D/2]; scale, bias fp16
    [B,Hkv,S_cap,D/64]: rows [0, rows) of src go to rows [dst_row0, dst_row0 + rows)."""
    B, Hkv, S_src, D = src.shape
    if src.dtype != torch.bfloat16 or codes.dtype != torch.uint8:
        raise TypeError("bf16 source, uint8 codes")
    if scale.dtype != torch.float16 or bias.dtype != torch.float16:
        raise TypeError("fp16 scale and bias")
    rows = S_src if rows is None else int(rows)
    rc = lib().gqa_attn_quantize_q4(_ptr(src), S_src, _ptr(codes), _ptr(scale), _ptr(bias), codes.shape[2],
                                    int(dst_row0), B * Hkv, rows, D, int(group_size), _stream(stream))
    _check(rc, "gqa_attn_quantize_q4")


def gqa_attn_decode_layers_workspace_size(n_layers, B, Hq, Hkv, D, max_kv_len, dtype) -> int:
    return lib().gqa_attn_decode_layers_workspace_size(n_layers, B, Hq, Hkv, D, max_kv_len, dtype)


def gqa_attn_decode_layers(q, k, v, o, kv_lens, scale, workspace, max_kv_len=None, stream=None):
    """Layers stacked on a leading axis: q, o [NL,B,Hq,1,D]; k, v [NL,B,Hkv,S_cap,D];
    kv_lens int32 [B] shared by the layers, or None."""
    NL, B, Hq, Tq, D = q.shape
    Hkv, S_cap = k.shape[2], k.shape[3]
    if Tq != 1:
        raise ValueError("decode takes one query row per request")
    if max_kv_len is None:
        max_kv_len = S_cap
    rc = lib().gqa_attn_decode_layers(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(kv_lens), NL, B, Hq, Hkv, D,
                                      S_cap, int(max_kv_len), float(scale), _dtype_code(q), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "gqa_attn_decode_layers")


def gqa_attn_decode_q4_residual_workspace_size(B, Hq, Hkv, D, max_quant) -> int:
    return lib().gqa_attn_decode_q4_residual_workspace_size(B, Hq, Hkv, D, max_quant)


def gqa_attn_decode_q4_residual(q, k_codes, k_scale, k_bias, v_codes, v_scale, v_bias, k_res, v_res,
                                n_quant, kv_lens, o, scale, workspace, max_quant=None, group_size=64,
                                stream=None):
    """4-bit cache rows [0, n_quant[b]) then window rows (bf16 k_res, v_res
    [B,Hkv,R_cap,D]) up to kv_lens[b]; q, o bf16 [B,Hq,1,D]."""
    B, Hq, Tq, D = q.shape
    Hkv, S_cap = k_codes.shape[1], k_codes.shape[2]
    R_cap = k_res.shape[2]
    if q.dtype != torch.bfloat16 or k_res.dtype != torch.bfloat16:
        raise TypeError("bf16 q and window")
    max_quant = S_cap if max_quant is None else int(max_quant)
    rc = lib().gqa_attn_decode_q4_residual(_ptr(q), _ptr(k_codes), _ptr(k_scale), _ptr(k_bias),
                                           _ptr(v_codes), _ptr(v_scale), _ptr(v_bias), _ptr(k_res),
                                           _ptr(v_res), _ptr(n_quant), _ptr(kv_lens), _ptr(o), B, Hq, Hkv,
                                           D, S_cap, R_cap, max_quant, int(group_size), float(scale),
                                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream(stream))
    _check(rc, "gqa_attn_decode_q4_residual")


def gqa_attn_decode_q4_workspace_size(B, Hq, Hkv, D, max_kv_len) -> int:
    return lib().gqa_attn_decode_q4_workspace_size(B, Hq, Hkv, D, max_kv_len)


def gqa_attn_decode_q4(q, k_codes, k_scale, k_bias, v_codes, v_scale, v_bias, o, kv_lens, scale,
                       workspace, max_kv_len=None, group_size=64, stream=None):
    """q, o bf16 [B,Hq,1,D]; codes uint8 [B,Hkv,S_cap,D/2]; scale/bias fp16 [B,Hkv,S_cap,D/G]."""
    B, Hq, Tq, D = q.shape
    Hkv, S_cap = k_codes.shape[1], k_codes.shape[2]
    if q.dtype != torch.bfloat16 or o.dtype != torch.bfloat16:
        raise TypeError("q4 decode takes bf16 q and o")
    if max_kv_len is None:
        max_kv_len = S_cap
    rc = lib().gqa_attn_decode_q4(_ptr(q), _ptr(k_codes), _ptr(k_scale), _ptr(k_bias),
                                  _ptr(v_codes), _ptr(v_scale), _ptr(v_bias), _ptr(o),
                                  _ptr(kv_lens), B, Hq, Hkv, D, S_cap, int(max_kv_len),
                                  int(group_size), float(scale), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "gqa_attn_decode_q4")


def gqa_attn_prefill(q, k, v, o, kv_len, scale, causal=True, stream=None):
    """q, o [B,Hq,q_len,D]; k, v [B,Hkv,S_cap,D]; keys 0..kv_len-1 visible."""
    B, Hq, q_len, D = q.shape
    Hkv, S_cap = k.shape[1], k.shape[2]
    rc = lib().gqa_attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, D, q_len,
                                int(kv_len), S_cap, float(scale), 1 if causal else 0,
                                _dtype_code(q), _stream(stream))
    _check(rc, "gqa_attn_prefill")


def gqa_attn_prefill_varlen(q, k, v, o, q_lens, kv_lens, scale, causal=True, stream=None):
    """q, o [B,Hq,Tq_cap,D]; k, v [B,Hkv,S_cap,D]; q_lens, kv_lens int32 [B]:
    request b's q_lens[b] queries aligned to the end of its kv_lens[b] keys."""
    B, Hq, Tq_cap, D = q.shape
    Hkv, S_cap = k.shape[1], k.shape[2]
    if q_lens.dtype != torch.int32 or kv_lens.dtype != torch.int32:
        raise TypeError("q_lens and kv_lens are int32")
    rc = lib().gqa_attn_prefill_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(q_lens), _ptr(kv_lens), B, Hq,
                                       Hkv, D, Tq_cap, S_cap, float(scale), 1 if causal else 0, _dtype_code(q),
                                       _stream(stream))
    _check(rc, "gqa_attn_prefill_varlen")


def gqa_attn_status_string(status: int) -> str:
    return lib().gqa_attn_status_string(status).decode()


def gqa_attn_read_device_status(workspace, stream=None) -> int:
    out = ctypes.c_uint32(0)
    _check(lib().gqa_attn_read_device_status(_ptr(workspace), ctypes.byref(out), _stream(stream)),
           "gqa_attn_read_device_status")
    return out.value


def gqa_attn_clear_device_status(workspace, stream=None):
    _check(lib().gqa_attn_clear_device_status(_ptr(workspace), _stream(stream)),
           "gqa_attn_clear_device_status")


def gqa_attn_read_prefill_status(stream=None) -> int:
    out = ctypes.c_uint32(0)
    _check(lib().gqa_attn_read_prefill_status(ctypes.byref(out), _stream(stream)),
           "gqa_attn_read_prefill_status")
    return out.value


def gqa_attn_clear_prefill_status(stream=None):
    _check(lib().gqa_attn_clear_prefill_status(_stream(stream)), "gqa_attn_clear_prefill_status")


def gqa_attn_version() -> int:
    return lib().gqa_attn_version()


# --- conveniences: allocate outputs / workspaces with torch, then call -------

def decode_workspace(B, Hq, Hkv, D, max_kv_len, dtype, device="cuda") -> torch.Tensor:
    n = gqa_attn_decode_workspace_size(B, Hq, Hkv, D, max_kv_len, dtype)
    if n == 0:
        raise ValueError("invalid decode shape")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode_q4_workspace(B, Hq, Hkv, D, max_kv_len, device="cuda") -> torch.Tensor:
    n = gqa_attn_decode_q4_workspace_size(B, Hq, Hkv, D, max_kv_len)
    if n == 0:
        raise ValueError("invalid decode shape")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode(q, k, v, kv_lens=None, scale=None, max_kv_len=None, workspace=None, stream=None):
    B, Hq, _, D = q.shape
    Hkv, S_cap = k.shape[1], k.shape[2]
    max_kv_len = S_cap if max_kv_len is None else int(max_kv_len)
    if scale is None:
        scale = D ** -0.5
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, D, max_kv_len, _dtype_code(q), q.device)
    o = torch.empty_like(q)
    gqa_attn_decode(q, k, v, o, kv_lens, scale, workspace, max_kv_len, stream)
    return o


def decode_q4_residual(q, k_codes, k_scale, k_bias, v_codes, v_scale, v_bias, k_res, v_res, n_quant,
                       kv_lens, max_quant=None, scale=None, workspace=None, stream=None):
    B, Hq, _, D = q.shape
    Hkv, S_cap = k_codes.shape[1], k_codes.shape[2]
    max_quant = S_cap if max_quant is None else int(max_quant)
    if scale is None:
        scale = D ** -0.5
    if workspace is None:
        n = gqa_attn_decode_q4_residual_workspace_size(B, Hq, Hkv, D, max_quant)
        if n == 0:
            raise ValueError("invalid decode shape")
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    gqa_attn_decode_q4_residual(q, k_codes, k_scale, k_bias, v_codes, v_scale, v_bias, k_res, v_res,
                                n_quant, kv_lens, o, scale, workspace, max_quant, stream=stream)
    return o


def decode_paged(q, k_pool, v_pool, block_table, kv_lens, max_kv_len, k_new=None, v_new=None,
                 scale=None, workspace=None, stream=None):
    B, Hq, _, D = q.shape
    Hkv = k_pool.shape[1]
    if scale is None:
        scale = D ** -0.5
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, D, max_kv_len, _dtype_code(q), q.device)
    o = torch.empty_like(q)
    gqa_attn_decode_paged(q, k_new, v_new, k_pool, v_pool, block_table, kv_lens, o, scale, workspace,
                          max_kv_len, stream)
    return o


def decode_q4(q, k_codes, k_scale, k_bias, v_codes, v_scale, v_bias, kv_lens=None, scale=None,
              max_kv_len=None, workspace=None, stream=None):
    B, Hq, _, D = q.shape
    Hkv, S_cap = k_codes.shape[1], k_codes.shape[2]
    max_kv_len = S_cap if max_kv_len is None else int(max_kv_len)
    if scale is None:
        scale = D ** -0.5
    if workspace is None:
        workspace = decode_q4_workspace(B, Hq, Hkv, D, max_kv_len, q.device)
    o = torch.empty_like(q)
    gqa_attn_decode_q4(q, k_codes, k_scale, k_bias, v_codes, v_scale, v_bias, o, kv_lens, scale,
                       workspace, max_kv_len, stream=stream)
    return o


def prefill(q, k, v, kv_len=None, scale=None, causal=True, stream=None):
    D = q.shape[-1]
    kv_len = k.shape[2] if kv_len is None else int(kv_len)
    if scale is None:
        scale = D ** -0.5
    o = torch.empty_like(q)
    gqa_attn_prefill(q, k, v, o, kv_len, scale, causal, stream)
    return o

"""The C ABI without a GPU: the library loads, exports exactly what the
header declares, and rejects invalid shapes on the host before touching the
device."""

import ctypes
import os
import re
import subprocess

import pytest

import __graft_entry__
from gqa_attention_kv_decode_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "gqa_attn.h")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return binding.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GQA_ATTN_API\s+[\w\s\*]+?\b(gqa_attn_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("gqa_attn_decode", "gqa_attn_prefill", "gqa_attn_decode_q4"):
        assert n in names
    assert set(names) == set(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    gqa = {s for s in exported if s.startswith("gqa_attn_")}
    assert gqa == set(declared_symbols())


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        s = binding.gqa_attn_status_string(code)
        assert s.startswith("GQA_")
    assert binding.gqa_attn_version() >= 100


P = ctypes.c_void_p(16)  # never dereferenced: shape checks come first


@pytest.mark.parametrize("args", [
    dict(B=1, Hq=14, Hkv=3, D=64, S=128, L=128, scale=0.125),     # Hq % Hkv != 0
    dict(B=1, Hq=14, Hkv=2, D=96, S=128, L=128, scale=0.125),     # unsupported head size
    dict(B=1, Hq=14, Hkv=2, D=64, S=128, L=129, scale=0.125),     # max_kv_len > S_cap
    dict(B=1, Hq=14, Hkv=2, D=64, S=128, L=0, scale=0.125),       # max_kv_len < 1
    dict(B=0, Hq=14, Hkv=2, D=64, S=128, L=128, scale=0.125),     # no requests
    dict(B=1, Hq=14, Hkv=2, D=64, S=128, L=128, scale=float("nan")),
    dict(B=1, Hq=14, Hkv=2, D=64, S=128, L=128, scale=0.0),
])
def test_decode_rejects_bad_shapes_on_host(lib, args):
    rc = lib.gqa_attn_decode(P, P, P, P, None, args["B"], args["Hq"], args["Hkv"], args["D"],
                             args["S"], args["L"], args["scale"], 0, P, 1 << 20, None)
    assert rc == binding.GQA_ERR_INVALID_ARG


def test_decode_rejects_bad_dtype(lib):
    rc = lib.gqa_attn_decode(P, P, P, P, None, 1, 14, 2, 64, 128, 128, 0.125, 7, P, 1 << 20, None)
    assert rc == binding.GQA_ERR_INVALID_ARG


def test_q4_rejects_group_size(lib):
    rc = lib.gqa_attn_decode_q4(P, P, P, P, P, P, P, P, None, 1, 32, 8, 128, 64, 64, 32, 0.1,
                                P, 1 << 20, None)
    assert rc == binding.GQA_ERR_INVALID_ARG


@pytest.mark.parametrize("q_len,kv_len,S", [(5, 4, 8), (0, 4, 8), (4, 9, 8)])
def test_prefill_rejects_bad_lengths(lib, q_len, kv_len, S):
    rc = lib.gqa_attn_prefill(P, P, P, P, 1, 14, 2, 64, q_len, kv_len, S, 0.125, 1, 1, None)
    assert rc == binding.GQA_ERR_INVALID_ARG


def test_prefill_rejects_bad_causal_flag(lib):
    rc = lib.gqa_attn_prefill(P, P, P, P, 1, 14, 2, 64, 4, 4, 8, 0.125, 2, 1, None)
    assert rc == binding.GQA_ERR_INVALID_ARG


def test_workspace_size_is_zero_for_invalid_shapes(lib):
    assert binding.gqa_attn_decode_workspace_size(1, 14, 3, 64, 128, 0) == 0
    assert binding.gqa_attn_decode_workspace_size(1, 14, 2, 64, 128, 0) > 0


def test_plan_override_checks_its_arguments(lib):
    assert lib.gqa_attn_set_plan_override(-1, 0) == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_attn_set_plan_override(0, 9) == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_attn_set_plan_override(0, -2) == binding.GQA_ERR_INVALID_ARG
    assert lib.gqa_attn_set_plan_override(0, 0) == binding.GQA_OK


def test_prefill_interleave_override_accepts_any_value_and_resets(lib):
    for v in (0, 3, 1 << 20, -1, -7):
        assert lib.gqa_attn_set_prefill_interleave_override(v) == binding.GQA_OK
    with binding.plan_override(prefill_interleave_from=2):
        pass  # restores the planner's choice on exit


def test_plan_override_is_not_read_from_the_environment(lib, monkeypatch):
    """Only the explicit call changes a plan: the split count the planner
    reports does not move when a tuning-looking variable is set."""
    before = lib.gqa_attn_decode_workspace_size(1, 28, 4, 128, 32768, 0)
    monkeypatch.setenv("GQA_ATTN_SPLITS", "3")
    assert lib.gqa_attn_decode_workspace_size(1, 28, 4, 128, 32768, 0) == before


def test_read_prefill_status_rejects_a_null_output(lib):
    assert lib.gqa_attn_read_prefill_status(None, None) == binding.GQA_ERR_INVALID_ARG

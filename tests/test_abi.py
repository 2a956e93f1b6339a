"""The C ABI library builds for sm_103a, loads, exports every symbol that
include/moe.h declares, and rejects bad configurations on the host."""
import os
import re
import subprocess

import pytest

from sparse_moe_expert_02_gb300 import _lib as L
from sparse_moe_expert_02_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"^MOE_API\s+[\w\s\*]*?\b(moe_\w+)\(", text, re.M)))


def test_header_declarations_match_binding():
    decl = declared_symbols()
    assert len(decl) >= 19
    assert decl == sorted(L.SYMBOLS)


def test_header_flags_match_binding():
    """Every MOE_FLAG_* bit of the header has the same value in the binding,
    and no two flags share a bit."""
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    flags = {n: int(v, 16) for n, v in re.findall(r"^#define\s+(MOE_FLAG_\w+)\s+(0x[0-9a-fA-F]+)u", text, re.M)}
    assert len(flags) >= 8
    for n, v in flags.items():
        assert getattr(L, n) == v, n
        assert v & (v - 1) == 0, n
    assert len(set(flags.values())) == len(flags)


def test_library_exports_every_declared_symbol():
    path = B.build()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(moe_\w+)$", out, re.M))
    missing = [s for s in declared_symbols() if s not in exported]
    assert not missing, missing
    lib = L.lib()
    for s in declared_symbols():
        assert getattr(lib, s) is not None


def test_library_is_built_for_sm103a_only():
    flags = B.ARCH
    assert flags == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings_and_build_info():
    lib = L.lib()
    assert lib.moe_status_str(0) == b"ok"
    assert lib.moe_status_str(5) == b"device wait timed out"
    assert b"sm_103a" in lib.moe_build_info()


@pytest.mark.parametrize("bad,status", [
    (dict(E=0), L.MOE_ERR_UNSUPPORTED),
    (dict(E=2000), L.MOE_ERR_UNSUPPORTED),
    (dict(top_k=0), L.MOE_ERR_UNSUPPORTED),
    (dict(top_k=33, E=64), L.MOE_ERR_UNSUPPORTED),
    (dict(top_k=17, E=16), L.MOE_ERR_UNSUPPORTED),
    (dict(D=200), L.MOE_ERR_UNSUPPORTED),
    (dict(D=128, dtype=2), L.MOE_ERR_UNSUPPORTED),  # FP8: the down GEMM's units are 256 features wide
    (dict(I=100), L.MOE_ERR_UNSUPPORTED),
    (dict(T_max=0), L.MOE_ERR_UNSUPPORTED),
    (dict(T_max=(1 << 20) + 1), L.MOE_ERR_UNSUPPORTED),
    (dict(dtype=7), L.MOE_ERR_UNSUPPORTED),
    (dict(out_dtype=2), L.MOE_ERR_UNSUPPORTED),
])
def test_plan_rejects_bad_config_before_touching_a_device(bad, status):
    import ctypes
    cfg = dict(T_max=128, D=512, E=32, I=256, top_k=4, dtype=1, out_dtype=0, has_router_bias=0, flags=0,
               spin_limit_ns=0)
    cfg.update(bad)
    c = L.moe_config(**cfg)
    plan = ctypes.c_void_p(1)
    st = L.lib().moe_plan_create(ctypes.byref(c), 0, ctypes.byref(plan))
    assert st == status
    assert plan.value is None


def test_null_arguments_are_rejected():
    import ctypes
    lib = L.lib()
    assert lib.moe_plan_create(None, 0, None) == L.MOE_ERR_INVALID_ARG
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(None, 1, ctypes.byref(n)) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_forward(None, None, None, 1, None, None, None, None, 0, None) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_check(None, None, None) == L.MOE_ERR_INVALID_ARG

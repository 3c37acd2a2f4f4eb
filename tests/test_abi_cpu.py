"""The C-ABI library builds, loads and exports every symbol include/*.h
declares; host-side validation and the size helpers work without a GPU.

No compute call is made here: every call below fails validation (or finds no
device) on the host before anything is enqueued.
"""
import ctypes
import glob
import os
import re

import pytest

import routed_grouped_gemm_dispatch_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    moe.build()
    return moe.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(L):
    names = _declared_functions()
    assert {"moe_build_dispatch", "moe_fused_forward", "moe_num_blocks"} <= names
    for n in names:
        assert hasattr(L, n), n


def test_abi_version_and_strings(L):
    assert L.moe_abi_version() == 1
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, 12345):
        assert moe.status_string(code)


def test_num_blocks_closed_form(L):
    # ceil(pairs/128) + n_experts
    assert moe.num_blocks(0, 5) == 5
    assert moe.num_blocks(1, 5) == 6
    assert moe.num_blocks(128, 5) == 6
    assert moe.num_blocks(129, 5) == 7
    assert moe.num_blocks(131072, 256) == 1280
    assert moe.num_blocks(-1, 5) == -1


P = ctypes.c_void_p


def _fwd(L, **kw):
    a = dict(x=0x1000, rows=1280, H=256, g=0x2000, u=0x3000, d=0x4000, E=4, I=256,
             rw=0x5000, valid=100, s=0x6000, o=0x7000, p=0x8000, gi=0x9000, m=5,
             ul=0xA000, out=0xB000, st=None, stream=None)
    a.update(kw)
    return L.moe_fused_forward(a["x"], a["rows"], a["H"], a["g"], a["u"], a["d"], a["E"], a["I"],
                               a["rw"], a["valid"], a["s"], a["o"], a["p"], a["gi"], a["m"],
                               a["ul"], a["out"], a["st"], a["stream"])


def test_forward_host_validation(L):
    assert _fwd(L, x=None) == -1            # MOE_ERR_NULL
    assert _fwd(L, out=None) == -1
    assert _fwd(L, H=200) == -2             # not a multiple of 128
    assert _fwd(L, I=0) == -2
    assert _fwd(L, rows=5 * 128 - 1) == -2  # fewer rows than blocks
    assert _fwd(L, E=0) == -7
    assert _fwd(L, E=5000) == -7
    assert _fwd(L, m=20000, rows=20000 * 128) == -7
    assert _fwd(L, x=0x1008) == -3          # misaligned
    assert _fwd(L, ul=0xA004) == -3


def test_dispatch_host_validation(L):
    args = dict(ids=0x1000, T=10, k=2, E=4, bt=128, s=0x2000, o=0x3000, p=0x4000, g=0x5000, m=5)

    def call(**kw):
        a = {**args, **kw}
        return L.moe_build_dispatch(a["ids"], a["T"], a["k"], a["E"], a["bt"], a["s"], a["o"],
                                    a["p"], a["g"], a["m"], None, None)
    assert call(bt=64) == -4
    assert call(m=6) == -2                  # num_blocks_m must be ceil(20/128) + 4 = 5
    assert call(E=0) == -7
    assert call(E=2000, m=1 + 2000) == -7
    assert call(k=0) == -2
    assert call(s=None) == -1
    assert call(ids=None) == -1


def test_binding_limits_match_header():
    import re
    import routed_grouped_gemm_dispatch_gb300 as moe
    text = open(os.path.join(ROOT, "include", "moe_gb300.h")).read()
    defs = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define (MOE_\w+)\s+(\d+)\b", text)}
    assert defs["MOE_BLOCK_TOKEN"] == moe.BLOCK_TOKEN
    assert defs["MOE_MAX_EXPERTS"] == moe.MAX_EXPERTS
    assert defs["MOE_MAX_BLOCKS"] == moe.MAX_BLOCKS
    assert defs["MOE_ROUTER_MAX_EXPERTS"] == moe.ROUTER_MAX_EXPERTS
    assert defs["MOE_ROUTER_MAX_TOPK"] == moe.ROUTER_MAX_TOPK
    bits = {m.group(1): int(m.group(2), 16) for m in re.finditer(r"#define (MOE_DEV_\w+)\s+0x([0-9a-fA-F]+)", text)}
    assert bits == {"MOE_DEV_BAD_EXPERT_ID": moe.MOE_DEV_BAD_EXPERT_ID, "MOE_DEV_BAD_TABLE": moe.MOE_DEV_BAD_TABLE,
                    "MOE_DEV_TIMEOUT": moe.MOE_DEV_TIMEOUT, "MOE_DEV_DEBUG_CHECK": moe.MOE_DEV_DEBUG_CHECK}

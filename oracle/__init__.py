"""CPU oracle for the routed fused-MoE expert GEMM — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The product
library never loads it and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (plain C, compiled with gcc, no
fast-math and no FMA contraction so that x86 and Arm give the same bits).  This
module only builds that library and marshals numpy arrays into it.

Pages followed (title, section):
  * "Fused MoE GEMM 提交说明" — §算子来源, §实现要点, §完整算子代码
  * "moe_dispatch_contract.py" (TileLang tutorial ch. 18) — docstring, build_contract
  * "MetaX-TileLang工具链" — §1.9, §1.12.1, §2.4 (also the router: logits,
    softmax, top-k)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

BLOCK_TOKEN = 128  # the pages' block_token and padding_M

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = f64
        lib.oracle_half_from_double.argtypes = [f64]
        lib.oracle_half_from_double.restype = ctypes.c_uint16
        lib.oracle_halves_to_doubles.argtypes = [P, i64, P]
        lib.oracle_doubles_to_halves.argtypes = [P, i64, P]
        lib.oracle_num_blocks.argtypes = [i64, i32, i32]
        lib.oracle_num_blocks.restype = i64
        lib.oracle_build_dispatch.argtypes = [P, i64, i32, i32, i32, i32, P, P, P, P, i64]
        lib.oracle_build_dispatch.restype = ctypes.c_int
        lib.oracle_pair_padded_rows.argtypes = [P, i64, i32, P, P]
        lib.oracle_pair_padded_rows.restype = ctypes.c_int
        lib.oracle_fused_forward.argtypes = [P, i64, i32, P, P, P, i32, i32, P,
                                             P, P, P, P, i64, i32, P, P, i32, i32]
        lib.oracle_fused_forward.restype = ctypes.c_int
        lib.oracle_forward_rows.argtypes = [P, i64, i32, P, P, P, i32, i32, P,
                                            P, P, P, P, i64, i32, P, i64, P, P, P, i32, i32]
        lib.oracle_forward_rows.restype = ctypes.c_int
        lib.oracle_pack.argtypes = [P, i64, i32, i32, P, P, P, P, P, P, i64, P]
        lib.oracle_pack.restype = ctypes.c_int
        lib.oracle_combine.argtypes = [P, i64, i32, P, i64, i32, P]
        lib.oracle_combine.restype = ctypes.c_int
        lib.oracle_router.argtypes = [P, i64, i32, P, i32, i32, P, P, i32]
        lib.oracle_router.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _bits16(a) -> np.ndarray:
    """fp16 array (or its uint16 bit pattern) as a contiguous uint16 view."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError(f"expected float16/uint16 bits, got {a.dtype}")


# --------------------------------------------------------------------------
# fp16 by definition
# --------------------------------------------------------------------------

def half_bits_to_double(bits) -> np.ndarray:
    bits = _c(np.asarray(bits, dtype=np.uint16), np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_halves_to_doubles(_ptr(bits), bits.size, _ptr(out))
    return out


def double_to_half_bits(values) -> np.ndarray:
    v = _c(np.asarray(values, dtype=np.float64), np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_doubles_to_halves(_ptr(v), v.size, _ptr(out))
    return out


# --------------------------------------------------------------------------
# dispatch tables
# --------------------------------------------------------------------------

def num_blocks(pairs: int, n_experts: int, block_token: int = BLOCK_TOKEN) -> int:
    return int(_load().oracle_num_blocks(int(pairs), int(n_experts), int(block_token)))


def build_dispatch(topk_ids, n_experts: int, block_token: int = BLOCK_TOKEN,
                   padding_m: int | None = None) -> dict:
    """The four tables for ``topk_ids`` [T, k] (int32)."""
    ids = _c(np.asarray(topk_ids), np.int32)
    if ids.ndim != 2:
        raise ValueError("topk_ids must be [tokens, top_k]")
    T, k = ids.shape
    E = int(n_experts)
    pm = block_token if padding_m is None else padding_m
    m = num_blocks(T * k, E, block_token)
    sizes = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    padded = np.zeros(E + 1, np.int32)
    gidx = np.zeros(m, np.int32)
    rc = _load().oracle_build_dispatch(_ptr(ids), T, k, E, pm, block_token, _ptr(sizes),
                                       _ptr(offsets), _ptr(padded), _ptr(gidx), m)
    if rc != 0:
        raise ValueError("oracle_build_dispatch rejected its input")
    return {"group_sizes": sizes, "group_offsets": offsets,
            "group_padded_offsets": padded, "group_idx_for_bx": gidx,
            "num_blocks_m": m}


def pair_padded_rows(topk_ids, n_experts: int, group_padded_offsets) -> np.ndarray:
    ids = _c(np.asarray(topk_ids), np.int32)
    padded = _c(np.asarray(group_padded_offsets), np.int32)
    rows = np.full(ids.size, -1, np.int32)
    rc = _load().oracle_pair_padded_rows(_ptr(ids), ids.size, int(n_experts), _ptr(padded),
                                         _ptr(rows))
    if rc != 0:
        raise ValueError("expert id out of range")
    return rows.reshape(ids.shape)


# --------------------------------------------------------------------------
# forward
# --------------------------------------------------------------------------

def _fwd_common(x, gate_w, up_w, down_w, rw, tables):
    x = _bits16(x)
    g = _bits16(gate_w)
    u = _bits16(up_w)
    d = _bits16(down_w)
    rw = _c(np.asarray(rw), np.float32)
    E, I, H = g.shape
    if x.shape[1] != H or u.shape != g.shape or d.shape != (E, H, I):
        raise ValueError("shape mismatch")
    t = {k: _c(np.asarray(tables[k]), np.int32) for k in
         ("group_sizes", "group_offsets", "group_padded_offsets", "group_idx_for_bx")}
    return x, g, u, d, rw, t, E, I, H


def fused_forward(x, gate_w, up_w, down_w, routed_expert_weights, tables,
                  up_logits=None, out=None, acc_f64: bool = False,
                  n_threads: int = 0, block_token: int = BLOCK_TOKEN):
    """Full forward.  ``up_logits``/``out`` (uint16 bits) are updated in place
    on valid rows only; if None they are created filled with zeros."""
    x, g, u, d, rw, t, E, I, H = _fwd_common(x, gate_w, up_w, down_w,
                                            routed_expert_weights, tables)
    rows = x.shape[0]
    if up_logits is None:
        up_logits = np.zeros((rows, I), np.uint16)
    if out is None:
        out = np.zeros((rows, H), np.uint16)
    up_logits = _bits16(up_logits)
    out = _bits16(out)
    m = t["group_idx_for_bx"].size
    rc = _load().oracle_fused_forward(
        _ptr(x), rows, H, _ptr(g), _ptr(u), _ptr(d), E, I, _ptr(rw),
        _ptr(t["group_sizes"]), _ptr(t["group_offsets"]), _ptr(t["group_padded_offsets"]),
        _ptr(t["group_idx_for_bx"]), m, block_token, _ptr(up_logits), _ptr(out),
        int(acc_f64), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_fused_forward rejected its input")
    return up_logits, out


def forward_rows(x, gate_w, up_w, down_w, routed_expert_weights, tables, rows,
                 acc_f64: bool = False, n_threads: int = 0,
                 block_token: int = BLOCK_TOKEN):
    """Forward for selected padded rows; returns (up [n, I], out [n, H], valid [n])."""
    x, g, u, d, rw, t, E, I, H = _fwd_common(x, gate_w, up_w, down_w,
                                            routed_expert_weights, tables)
    rl = _c(np.asarray(rows, dtype=np.int64), np.int64)
    n = rl.size
    up = np.zeros((n, I), np.uint16)
    out = np.zeros((n, H), np.uint16)
    valid = np.zeros(n, np.int32)
    m = t["group_idx_for_bx"].size
    rc = _load().oracle_forward_rows(
        _ptr(x), x.shape[0], H, _ptr(g), _ptr(u), _ptr(d), E, I, _ptr(rw),
        _ptr(t["group_sizes"]), _ptr(t["group_offsets"]), _ptr(t["group_padded_offsets"]),
        _ptr(t["group_idx_for_bx"]), m, block_token, _ptr(rl), n, _ptr(up), _ptr(out),
        _ptr(valid), int(acc_f64), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_forward_rows rejected its input")
    return up, out, valid.astype(bool)


# --------------------------------------------------------------------------
# harness steps around the path
# --------------------------------------------------------------------------

def pack(x_tokens, topk_ids, topk_weights, pair_rows, tables, rows_total: int,
         pad_bits: int = 0x7E00):
    """Grouped, padded x [rows_total, H] (padding rows = ``pad_bits``) and the
    routed weights in compact order."""
    xt = _bits16(x_tokens)
    ids = _c(np.asarray(topk_ids), np.int32)
    tw = _c(np.asarray(topk_weights), np.float32)
    pr = _c(np.asarray(pair_rows), np.int32)
    T, k = ids.shape
    H = xt.shape[1]
    offsets = _c(np.asarray(tables["group_offsets"]), np.int32)
    padded = _c(np.asarray(tables["group_padded_offsets"]), np.int32)
    x_packed = np.full((rows_total, H), pad_bits, np.uint16)
    rw = np.zeros(T * k, np.float32)
    rc = _load().oracle_pack(_ptr(xt), T, k, H, _ptr(ids), _ptr(tw), _ptr(pr),
                             _ptr(offsets), _ptr(padded), _ptr(x_packed), rows_total,
                             _ptr(rw))
    if rc != 0:
        raise ValueError("oracle_pack rejected its input")
    return x_packed, rw


def combine(out, pair_rows, n_tokens: int, top_k: int):
    o = _bits16(out)
    pr = _c(np.asarray(pair_rows), np.int32)
    H = o.shape[1]
    y = np.zeros((n_tokens, H), np.uint16)
    rc = _load().oracle_combine(_ptr(o), o.shape[0], H, _ptr(pr), n_tokens, top_k, _ptr(y))
    if rc != 0:
        raise ValueError("oracle_combine rejected its input")
    return y


def router(x_tokens, router_w, top_k: int, n_threads: int = 0):
    """topk_ids int32 [T, k] and topk_weights fp32 [T, k] ("MetaX-TileLang工具链"
    §2.4: logits -> softmax -> top-k)."""
    x = _bits16(x_tokens)
    w = _bits16(router_w)
    T, H = x.shape
    E, H2 = w.shape
    if H2 != H:
        raise ValueError("router weight shape mismatch")
    ids = np.zeros((T, top_k), np.int32)
    wts = np.zeros((T, top_k), np.float32)
    rc = _load().oracle_router(_ptr(x), T, H, _ptr(w), E, int(top_k), _ptr(ids), _ptr(wts), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_router rejected its input")
    return ids, wts

"""Python binding of the routed fused-MoE expert GEMM library (GB300, sm_103a).

Argument marshalling only: every step runs in the CUDA library
``_build/libmoe_gb300.so`` through its C ABI (``include/moe_gb300.h``).
PyTorch provides device memory and the current stream.  There is no CPU or
PyTorch fallback: if the library is missing or the device is not an sm_103
part, every call raises.

Calls (names follow "Fused MoE GEMM 提交说明", §提交文件 / §完整算子代码, and
"moe_dispatch_contract.py"):

  build_dispatch(topk_ids, n_experts)           -> dict of the four int32 tables
  fused_forward(stacked_expert_tokens, gate_w, up_w, down_w,
                routed_expert_weights, group_sizes, group_offsets,
                group_padded_offsets, group_idx_for_bx, up_logits, out)
  run_kernel(...)                               the page's signature (no up_logits;
                                                a cached workspace is used)
  pack_routed(topk_ids, topk_weights, x_tokens, tables)  -> grouped, padded inputs
  combine_routed(out, pair_rows)                -> token-major sum of the expert rows
  router_topk(x_tokens, router_w, top_k)        -> topk_ids, topk_weights
"""
from __future__ import annotations

import ctypes
import os
import threading

BLOCK_TOKEN = 128
MAX_EXPERTS = 1024          # MOE_MAX_EXPERTS
MAX_BLOCKS = 16384          # MOE_MAX_BLOCKS
ROUTER_MAX_EXPERTS = 256    # MOE_ROUTER_MAX_EXPERTS
ROUTER_MAX_TOPK = 16        # MOE_ROUTER_MAX_TOPK

_PKG = os.path.dirname(os.path.abspath(__file__))
# MOE_GB300_DEBUG=1 in the environment selects the MOE_DEBUG build (kernels
# that also check their own indices and report MOE_DEV_DEBUG_CHECK).
LIB_PATH = os.path.join(_PKG, "_build", "libmoe_gb300_debug.so" if os.environ.get("MOE_GB300_DEBUG") == "1"
                        else "libmoe_gb300.so")

MOE_OK = 0
MOE_DEV_BAD_EXPERT_ID = 0x1
MOE_DEV_BAD_TABLE = 0x2
MOE_DEV_TIMEOUT = 0x4
MOE_DEV_DEBUG_CHECK = 0x8
MOE_RUN_PHASE1 = 0x1
MOE_RUN_PHASE2 = 0x2
MOE_NO_PDL = 0x4
MOE_TEST_DROP_SIGNAL = 0x100

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    """A call of the C ABI returned a MOE_ERR_* status."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def build(force: bool = False, debug: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a); debug=True builds the
    MOE_DEBUG variant."""
    from . import _build
    return _build.build(force=force, debug=debug)


def lib():
    """The loaded C library; raises if it has not been built."""
    global _lib
    L = _lib
    if L is not None:
        return L
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built ({LIB_PATH}); call build() first")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.moe_abi_version.argtypes = []
        L.moe_abi_version.restype = i32
        L.moe_status_string.argtypes = [i32]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_num_blocks.argtypes = [i64, i32, i32]
        L.moe_num_blocks.restype = i64
        L.moe_build_dispatch.argtypes = [P, i64, i32, i32, i32, P, P, P, P, i64, P, P]
        L.moe_build_dispatch.restype = i32
        L.moe_fused_forward.argtypes = [P, i64, i32, P, P, P, i32, i32, P, i64,
                                        P, P, P, P, i64, P, P, P, P]
        L.moe_fused_forward.restype = i32
        L.moe_fused_forward_ex.argtypes = L.moe_fused_forward.argtypes + [ctypes.c_uint32]
        L.moe_fused_forward_ex.restype = i32
        L.moe_fused_forward_static_workspace.argtypes = [P, i64, i32, P, P, P, i32, i32, P, i64,
                                                         P, P, P, P, i64, P, P, P]
        L.moe_fused_forward_static_workspace.restype = i32
        L.moe_pack_workspace_bytes.argtypes = [i64, i32]
        L.moe_pack_workspace_bytes.restype = i64
        L.moe_pack_routed.argtypes = [P, P, i64, i32, i32, P, i32, P, P, i64, P, P, P, P,
                                      ctypes.c_size_t, P, P]
        L.moe_pack_routed.restype = i32
        L.moe_combine_routed.argtypes = [P, i64, i32, P, i64, i32, P, P]
        L.moe_combine_routed.restype = i32
        L.moe_router_topk.argtypes = [P, i64, i32, P, i32, i32, P, P, P, P]
        L.moe_router_topk.restype = i32
        L.moe_single_launch_workspace_bytes.argtypes = [i64]
        L.moe_single_launch_workspace_bytes.restype = i64
        L.moe_fused_forward_single_launch.argtypes = [P, i64, i32, P, P, P, i32, i32, P, i64,
                                                      P, P, P, P, i64, P, P, P, ctypes.c_size_t, P, P]
        L.moe_fused_forward_single_launch.restype = i32
        _lib = L
        return L


def single_launch_workspace_bytes(num_blocks_m: int) -> int:
    return int(lib().moe_single_launch_workspace_bytes(int(num_blocks_m)))


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def num_blocks(pairs: int, n_experts: int, block_token: int = BLOCK_TOKEN) -> int:
    return int(lib().moe_num_blocks(int(pairs), int(n_experts), int(block_token)))


def _stream(stream):
    import torch
    if stream is None:
        # the current stream's handle without building a Stream object (the
        # call Triton uses too); the public query where it does not exist
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dev(t, name, dtype, ndim=None):
    import torch
    # the common case in one expression; the checks below name what is wrong
    if (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype is dtype and (ndim is None or t.dim() == ndim)
            and t.is_contiguous()):
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def build_dispatch(topk_ids, n_experts: int, block_token: int = BLOCK_TOKEN,
                   status=None, stream=None, out=None) -> dict:
    """The four dispatch tables for ``topk_ids`` [T, k] int32 (device).

    ``out`` may supply preallocated tables (same keys as the result)."""
    import torch
    ids = _dev(topk_ids, "topk_ids", torch.int32, 2)
    T, k = ids.shape
    E = int(n_experts)
    m = num_blocks(T * k, E, block_token)
    if out is None:
        dev = ids.device
        out = {
            "group_sizes": torch.empty(E, dtype=torch.int32, device=dev),
            "group_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
            "group_padded_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
            "group_idx_for_bx": torch.empty(max(m, 0), dtype=torch.int32, device=dev),
        }
    st = lib().moe_build_dispatch(
        _ptr(ids), T, k, E, int(block_token), _ptr(out["group_sizes"]), _ptr(out["group_offsets"]),
        _ptr(out["group_padded_offsets"]), _ptr(out["group_idx_for_bx"]), m,
        _ptr(status), _stream(stream))
    _check(st, "moe_build_dispatch")
    return out


def fused_forward(stacked_expert_tokens, gate_w, up_w, down_w, routed_expert_weights,
                  group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx,
                  up_logits, out, status=None, stream=None,
                  flags: int = MOE_RUN_PHASE1 | MOE_RUN_PHASE2, single_launch_workspace=None):
    """Phase 1 + phase 2 on the current stream; writes ``up_logits`` and ``out``
    in place on valid rows only.  ``flags`` selects phases (MOE_RUN_PHASE1 /
    MOE_RUN_PHASE2, optionally MOE_NO_PDL).  With ``single_launch_workspace``
    (a device tensor of at least single_launch_workspace_bytes() bytes) both
    phases run in one persistent launch."""
    import torch
    x = _dev(stacked_expert_tokens, "stacked_expert_tokens", torch.float16, 2)
    g = _dev(gate_w, "gate_w", torch.float16, 3)
    u = _dev(up_w, "up_w", torch.float16, 3)
    d = _dev(down_w, "down_w", torch.float16, 3)
    rw = _dev(routed_expert_weights, "routed_expert_weights", torch.float32, 1)
    sizes = _dev(group_sizes, "group_sizes", torch.int32, 1)
    offs = _dev(group_offsets, "group_offsets", torch.int32, 1)
    padded = _dev(group_padded_offsets, "group_padded_offsets", torch.int32, 1)
    gidx = _dev(group_idx_for_bx, "group_idx_for_bx", torch.int32, 1)
    ul = _dev(up_logits, "up_logits", torch.float16, 2)
    o = _dev(out, "out", torch.float16, 2)
    rows, H = x.shape
    E, I, H2 = g.shape
    if H2 != H or tuple(u.shape) != (E, I, H) or tuple(d.shape) != (E, H, I):
        raise ValueError("weight shapes do not match [E, I, H] / [E, H, I]")
    if tuple(ul.shape) != (rows, I) or tuple(o.shape) != (rows, H):
        raise ValueError("up_logits / out shapes do not match the padded rows")
    if sizes.numel() != E or offs.numel() < E or padded.numel() < E:
        raise ValueError("table lengths do not match n_experts")
    args = (_ptr(x), rows, H, _ptr(g), _ptr(u), _ptr(d), E, I, _ptr(rw), rw.numel(),
            _ptr(sizes), _ptr(offs), _ptr(padded), _ptr(gidx), gidx.numel(),
            _ptr(ul), _ptr(o), _ptr(status), _stream(stream))
    if single_launch_workspace is not None:
        ws = single_launch_workspace
        _check(lib().moe_fused_forward_single_launch(*args[:17], _ptr(ws), ws.numel() * ws.element_size(),
                                                     *args[17:]), "moe_fused_forward_single_launch")
    elif flags == (MOE_RUN_PHASE1 | MOE_RUN_PHASE2):
        _check(lib().moe_fused_forward(*args), "moe_fused_forward")
    else:
        _check(lib().moe_fused_forward_ex(*args, int(flags)), "moe_fused_forward_ex")
    return o


def fused_forward_static_workspace(stacked_expert_tokens, gate_w, up_w, down_w,
                                   routed_expert_weights, group_sizes, group_offsets,
                                   group_padded_offsets, group_idx_for_bx, out,
                                   status=None, stream=None):
    """The fused forward without an up_logits argument, for callers that
    cannot allocate device memory: the workspace is the library's fixed
    64 MiB array (total_padded_tokens * intermediate * 2 bytes at most).
    Calls share that array, so calls that overlap on the GPU race."""
    import torch
    x = _dev(stacked_expert_tokens, "stacked_expert_tokens", torch.float16, 2)
    g = _dev(gate_w, "gate_w", torch.float16, 3)
    u = _dev(up_w, "up_w", torch.float16, 3)
    d = _dev(down_w, "down_w", torch.float16, 3)
    rw = _dev(routed_expert_weights, "routed_expert_weights", torch.float32, 1)
    tabs = [_dev(t, n, torch.int32, 1) for t, n in
            ((group_sizes, "group_sizes"), (group_offsets, "group_offsets"),
             (group_padded_offsets, "group_padded_offsets"), (group_idx_for_bx, "group_idx_for_bx"))]
    o = _dev(out, "out", torch.float16, 2)
    rows, H = x.shape
    E, I, _ = g.shape
    if tuple(o.shape) != (rows, H):
        raise ValueError("out shape does not match the padded rows")
    st = lib().moe_fused_forward_static_workspace(
        _ptr(x), rows, H, _ptr(g), _ptr(u), _ptr(d), E, I, _ptr(rw), rw.numel(),
        *[_ptr(t) for t in tabs], tabs[3].numel(), _ptr(o), _ptr(status), _stream(stream))
    _check(st, "moe_fused_forward_static_workspace")
    return o


def pack_routed(topk_ids, topk_weights, x_tokens, tables, rows_total: int | None = None,
                stacked=None, routed_weights=None, pair_rows=None, workspace=None,
                status=None, stream=None) -> dict:
    """Grouped, padded activations, compact routed weights and every pair's
    padded row, from token-major inputs (all device tensors).  Preallocated
    outputs may be passed; padding rows of ``stacked`` are left untouched
    (a new ``stacked`` is filled with fp16 NaN there)."""
    import torch
    ids = _dev(topk_ids, "topk_ids", torch.int32, 2)
    T, k = ids.shape
    E = tables["group_sizes"].numel()
    x = _dev(x_tokens, "x_tokens", torch.float16, 2) if x_tokens is not None else None
    tw = _dev(topk_weights, "topk_weights", torch.float32, 2) if topk_weights is not None else None
    H = x.shape[1] if x is not None else 128
    if rows_total is None:
        rows_total = tables["group_idx_for_bx"].numel() * BLOCK_TOKEN
    dev = ids.device
    if stacked is None and x is not None:
        stacked = torch.full((rows_total, H), float("nan"), dtype=torch.float16, device=dev)
    if routed_weights is None and tw is not None:
        routed_weights = torch.empty(T * k, dtype=torch.float32, device=dev)
    if pair_rows is None:
        pair_rows = torch.empty((T, k), dtype=torch.int32, device=dev)
    need = int(lib().moe_pack_workspace_bytes(T * k, E))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = lib().moe_pack_routed(
        _ptr(ids), _ptr(tw), T, k, E, _ptr(x), H, _ptr(tables["group_offsets"]),
        _ptr(tables["group_padded_offsets"]), rows_total, _ptr(stacked), _ptr(routed_weights),
        _ptr(pair_rows), _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    _check(st, "moe_pack_routed")
    return {"stacked_expert_tokens": stacked, "routed_expert_weights": routed_weights,
            "pair_padded_rows": pair_rows}


def combine_routed(out, pair_rows, y=None, stream=None):
    """y[t] = fp16(sum_j out[pair_rows[t, j]]) with an fp32 sum in j order."""
    import torch
    o = _dev(out, "out", torch.float16, 2)
    pr = _dev(pair_rows, "pair_rows", torch.int32, 2)
    T, k = pr.shape
    if y is None:
        y = torch.empty((T, o.shape[1]), dtype=torch.float16, device=o.device)
    st = lib().moe_combine_routed(_ptr(o), o.shape[0], o.shape[1], _ptr(pr), T, k, _ptr(y),
                                  _stream(stream))
    _check(st, "moe_combine_routed")
    return y


def router_topk(x_tokens, router_w, top_k: int, topk_ids=None, topk_weights=None,
                status=None, stream=None):
    """Router logits (x·W_gᵀ), softmax over all experts, top-k: returns
    (topk_ids int32 [T, k], topk_weights fp32 [T, k])."""
    import torch
    x = _dev(x_tokens, "x_tokens", torch.float16, 2)
    w = _dev(router_w, "router_w", torch.float16, 2)
    T, H = x.shape
    E = w.shape[0]
    if w.shape[1] != H:
        raise ValueError("router_w must be [n_experts, hidden]")
    if topk_ids is None:
        topk_ids = torch.empty((T, top_k), dtype=torch.int32, device=x.device)
    if topk_weights is None:
        topk_weights = torch.empty((T, top_k), dtype=torch.float32, device=x.device)
    st = lib().moe_router_topk(_ptr(x), T, H, _ptr(w), E, int(top_k), _ptr(topk_ids),
                               _ptr(topk_weights), _ptr(status), _stream(stream))
    _check(st, "moe_router_topk")
    return topk_ids, topk_weights


_WORKSPACE = {}


def run_kernel(stacked_expert_tokens, gate_w, up_w, down_w, routed_expert_weights,
               group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx, out):
    """The page's submission signature: ``up_logits`` comes from a per-device,
    per-shape workspace cache (allocated once by PyTorch); ``out`` is written in
    place; no synchronisation, no new tensor."""
    import torch
    key = (stacked_expert_tokens.device.index, int(stacked_expert_tokens.shape[0]),
           int(gate_w.shape[1]))
    ws = _WORKSPACE.get(key)
    if ws is None:
        ws = torch.empty((key[1], key[2]), dtype=torch.float16, device=stacked_expert_tokens.device)
        _WORKSPACE[key] = ws
    fused_forward(stacked_expert_tokens, gate_w, up_w, down_w, routed_expert_weights,
                  group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx, ws, out)

"""ctypes binding of libmoe.so (the C ABI in include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. Tensors are torch CUDA tensors (used as plain device memory). The
functions take the same names and arguments as the C entry points and raise
``MoeError`` on a non-zero status. There is no fallback: if the library cannot
be loaded, every call fails loudly.

Inside ``with debug_library():`` the same functions call libmoe_debug.so,
the build whose kernels also check their own derived indices (see
``debug_take``).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import re
import threading

from . import _build

MOE_F32, MOE_BF16 = 0, 1
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_STATUS",
                6: "MOE_ERR_TIMEOUT"}
DEV_BAD_EXPERT_ID, DEV_CAP_OVERFLOW, DEV_TIMEOUT, DEV_BAD_SEGMENT = 0x1, 0x2, 0x4, 0x8


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        self.cuda_error = lib().moe_last_cuda_error() if status == 4 else 0
        why = f", CUDA error {self.cuda_error}" if self.cuda_error else ""
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({strerror(status)}{why})")


class MoeConfig(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("hidden_size", ctypes.c_int), ("intermediate_size", ctypes.c_int),
                ("renormalize", ctypes.c_int), ("use_grouped_topk", ctypes.c_int),
                ("num_expert_group", ctypes.c_int), ("topk_group", ctypes.c_int),
                ("routed_scaling_factor", ctypes.c_float),
                ("num_shared_experts", ctypes.c_int),
                ("shared_intermediate_size", ctypes.c_int),
                ("ep_size", ctypes.c_int), ("ep_rank", ctypes.c_int),
                ("act_dtype", ctypes.c_int), ("router_dtype", ctypes.c_int),
                ("scoring_func", ctypes.c_int), ("bias_mode", ctypes.c_int),
                ("max_replicas", ctypes.c_int), ("num_redundant_experts", ctypes.c_int)]


class WorkspaceOffsets(ctypes.Structure):
    _fields_ = [("status", ctypes.c_size_t), ("topk_ids", ctypes.c_size_t),
                ("topk_w", ctypes.c_size_t), ("counts", ctypes.c_size_t),
                ("offsets", ctypes.c_size_t), ("sorted_ids", ctypes.c_size_t),
                ("inv_pos", ctypes.c_size_t), ("total", ctypes.c_size_t),
                ("cap", ctypes.c_int), ("block_m", ctypes.c_int)]


class DebugRecord(ctypes.Structure):
    _fields_ = [("count", ctypes.c_uint32), ("site", ctypes.c_uint32),
                ("index", ctypes.c_int64), ("bound", ctypes.c_int64)]


DEBUG_FILES = {1: "moe_api.cu", 2: "kernels_gemm.cu", 3: "kernels_gemm_pair.cu",
               4: "kernels_mlp_fused.cu", 5: "kernels_route.cu", 6: "kernels_align.cu"}


class Plan(ctypes.Structure):
    _fields_ = [("kernels", ctypes.c_int), ("fused_route", ctypes.c_int),
                ("router_tensor_cores", ctypes.c_int),
                ("router_partials", ctypes.c_int), ("align_kernels", ctypes.c_int),
                ("tile_rows", ctypes.c_int), ("gemm1_k_split", ctypes.c_int),
                ("cta_pairs", ctypes.c_int), ("fused_mlp", ctypes.c_int),
                ("gemm2_overlap", ctypes.c_int), ("combine_ring", ctypes.c_int)]


def make_config(num_experts, top_k, hidden_size, intermediate_size, renormalize=True,
                num_expert_group=0, topk_group=0, routed_scaling_factor=1.0,
                num_shared_experts=0, shared_intermediate_size=0, ep_size=1, ep_rank=0,
                act_dtype="bf16", router_dtype="bf16", scoring="softmax",
                bias_mode="logit", max_replicas=0, num_redundant_experts=0) -> MoeConfig:
    dt = {"bf16": MOE_BF16, "f32": MOE_F32}
    sc = {"softmax": 0, "sigmoid": 1}
    bm = {"logit": 0, "select": 1}
    return MoeConfig(num_experts, top_k, hidden_size, intermediate_size, int(bool(renormalize)),
                     int(num_expert_group > 0), num_expert_group, topk_group,
                     float(routed_scaling_factor), num_shared_experts,
                     shared_intermediate_size, ep_size, ep_rank, dt[act_dtype],
                     dt[router_dtype], sc[scoring], bm[bias_mode], max_replicas,
                     num_redundant_experts)


_libs: dict[bool, ctypes.CDLL] = {}  # debug build? -> loaded library
_use_debug = False
_lock = threading.Lock()
_VP, _SZ, _I = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
_CFG = ctypes.POINTER(MoeConfig)

_SIGS = {
    "moe_strerror": (ctypes.c_char_p, [_I]),
    "moe_validate_config": (_I, [_CFG]),
    "moe_align_cap": (_SZ, [_CFG, _I, _I]),
    "moe_route_workspace_size": (_SZ, [_CFG, _I]),
    "moe_route": (_I, [_CFG, _I, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "moe_align_workspace_size": (_SZ, [_CFG, _I]),
    "moe_align_permute": (_I, [_CFG, _I, _VP, _VP, _I, _VP, _VP, _VP, _VP, _I, _VP, _SZ, _VP]),
    "moe_align_permute_noalloc": (_I, [_CFG, _I, _VP, _VP, _I, _VP, _VP, _VP, _VP, _I, _VP]),
    "moe_grouped_mlp_workspace_size": (_SZ, [_CFG, _I, _I]),
    "moe_grouped_mlp": (_I, [_CFG, _I, _VP, _VP, _VP, _VP, _I, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "moe_combine": (_I, [_CFG, _I, _VP, _I, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "moe_workspace_size": (_SZ, [_CFG, _I]),
    "moe_workspace_layout": (_I, [_CFG, _I, ctypes.POINTER(WorkspaceOffsets)]),
    "moe_forward": (_I, [_CFG, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "moe_forward_timed": (_I, [_CFG, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                               _SZ, _VP, ctypes.POINTER(ctypes.c_void_p),
                               ctypes.POINTER(ctypes.c_int)]),
    "moe_get_status": (_I, [_VP, _VP, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_last_cuda_error": (_I, []),
    "moe_set_wait_limit_ns": (_I, [ctypes.c_uint64]),
    "moe_forward_plan": (_I, [_CFG, _I, ctypes.POINTER(Plan)]),
    "moe_ep_dispatch_workspace_size": (_SZ, [_CFG, _I]),
    "moe_ep_dispatch": (_I, [_CFG, _I] + [_VP] * 12 + [_SZ, _VP]),
    "moe_ep_expert_compute_workspace_size": (_SZ, [_CFG, _I]),
    "moe_ep_expert_compute": (_I, [_CFG, _I] + [_VP] * 7 + [_SZ, _VP]),
    "moe_ep_combine": (_I, [_CFG, _I] + [_VP] * 5 + [_SZ, _VP]),
    "moe_debug_build": (_I, []),
    "moe_debug_take": (_I, [ctypes.POINTER(DebugRecord)]),
    "moe_debug_selftest": (_I, [_VP]),
}


def header_functions() -> list[str]:
    """Names of the functions declared in include/moe.h."""
    with open(os.path.join(_build.INCLUDE, "moe.h")) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def lib(build: bool = True, debug: bool | None = None) -> ctypes.CDLL:
    """Load libmoe.so, or libmoe_debug.so inside ``debug_library()`` (or with
    debug=True), building it in place first if missing or stale."""
    dbg = _use_debug if debug is None else debug
    with _lock:
        L = _libs.get(dbg)
        if L is None:
            path = _build.lib_path(dbg)
            if build:
                _build.build(debug=dbg)
            if not os.path.exists(path):
                raise RuntimeError(f"{os.path.basename(path)} is not built; "
                                   "call __graft_entry__.build()")
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _libs[dbg] = L
    return L


@contextlib.contextmanager
def debug_library():
    """Route every call of this module to libmoe_debug.so for the duration
    (one thread at a time; not reentrant across threads)."""
    global _use_debug
    old = _use_debug
    _use_debug = True
    try:
        yield lib()
    finally:
        _use_debug = old


def strerror(status: int) -> str:
    return lib().moe_strerror(status).decode()


def _p(t):
    """Device pointer of a tensor (None -> NULL); integers pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libmoe takes device tensors; got one on " + str(t.device))
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmoe must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(fn, rc):
    if rc != 0:
        raise MoeError(fn, rc)


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def validate_config(cfg: MoeConfig) -> int:
    return lib().moe_validate_config(ctypes.byref(cfg))


def align_cap(cfg, T, block_m) -> int:
    return lib().moe_align_cap(ctypes.byref(cfg), T, block_m)


def route_workspace_size(cfg, T) -> int:
    return lib().moe_route_workspace_size(ctypes.byref(cfg), T)


def align_workspace_size(cfg, T) -> int:
    return lib().moe_align_workspace_size(ctypes.byref(cfg), T)


def grouped_mlp_workspace_size(cfg, T, cap) -> int:
    return lib().moe_grouped_mlp_workspace_size(ctypes.byref(cfg), T, cap)


def workspace_size(cfg, T) -> int:
    return lib().moe_workspace_size(ctypes.byref(cfg), T)


def workspace_layout(cfg, T) -> WorkspaceOffsets:
    out = WorkspaceOffsets()
    _check("moe_workspace_layout", lib().moe_workspace_layout(ctypes.byref(cfg), T,
                                                             ctypes.byref(out)))
    return out


def forward_plan(cfg, T) -> Plan:
    out = Plan()
    _check("moe_forward_plan", lib().moe_forward_plan(ctypes.byref(cfg), T, ctypes.byref(out)))
    return out


def ep_dispatch_workspace_size(cfg, T) -> int:
    return lib().moe_ep_dispatch_workspace_size(ctypes.byref(cfg), T)


def moe_ep_dispatch(cfg, T, x, topk_ids, topk_w, send_counts, send_offsets, send_pos, send_x,
                    send_ids, send_w, send_tok, ws, stream=None, phys_map=None):
    _check("moe_ep_dispatch", lib().moe_ep_dispatch(
        ctypes.byref(cfg), T, _p(x), _p(topk_ids), _p(topk_w), _p(phys_map), _p(send_counts),
        _p(send_offsets), _p(send_pos), _p(send_x), _p(send_ids), _p(send_w), _p(send_tok),
        _p(ws), _nbytes(ws), _stream(stream)))


def ep_expert_compute_workspace_size(cfg, R) -> int:
    return lib().moe_ep_expert_compute_workspace_size(ctypes.byref(cfg), R)


def moe_ep_expert_compute(cfg, R, recv_x, recv_ids, recv_w, w13, w2, y, ws, stream=None):
    _check("moe_ep_expert_compute", lib().moe_ep_expert_compute(
        ctypes.byref(cfg), R, _p(recv_x), _p(recv_ids), _p(recv_w), _p(w13), _p(w2), _p(y),
        _p(ws), _nbytes(ws), _stream(stream)))


def moe_ep_combine(cfg, T, ret, send_pos, shared_out, out, ws=None, stream=None):
    _check("moe_ep_combine", lib().moe_ep_combine(
        ctypes.byref(cfg), T, _p(ret), _p(send_pos), _p(shared_out), _p(out), _p(ws),
        _nbytes(ws), _stream(stream)))


def moe_route(cfg, T, x, router_w, router_bias, topk_ids, topk_w, ws, stream=None):
    _check("moe_route", lib().moe_route(ctypes.byref(cfg), T, _p(x), _p(router_w),
                                        _p(router_bias), _p(topk_ids), _p(topk_w), _p(ws),
                                        _nbytes(ws), _stream(stream)))


def moe_align_permute(cfg, T, topk_ids, expert_map, block_m, counts, offsets, sorted_ids,
                      inv_pos, cap, ws, stream=None):
    _check("moe_align_permute", lib().moe_align_permute(
        ctypes.byref(cfg), T, _p(topk_ids), _p(expert_map), block_m, _p(counts), _p(offsets),
        _p(sorted_ids), _p(inv_pos), cap, _p(ws), _nbytes(ws), _stream(stream)))


def moe_align_permute_noalloc(cfg, T, topk_ids, expert_map, block_m, counts, offsets,
                              sorted_ids, inv_pos, cap, stream=None):
    """moe_align_permute with its scratch in the library's static device array
    (for callers that cannot allocate a workspace)."""
    _check("moe_align_permute_noalloc", lib().moe_align_permute_noalloc(
        ctypes.byref(cfg), T, _p(topk_ids), _p(expert_map), block_m, _p(counts), _p(offsets),
        _p(sorted_ids), _p(inv_pos), cap, _stream(stream)))


def moe_grouped_mlp(cfg, T, x, sorted_ids, counts, offsets, cap, w13, w2, y_perm, ws,
                    stream=None):
    _check("moe_grouped_mlp", lib().moe_grouped_mlp(
        ctypes.byref(cfg), T, _p(x), _p(sorted_ids), _p(counts), _p(offsets), cap, _p(w13),
        _p(w2), _p(y_perm), _p(ws), _nbytes(ws), _stream(stream)))


def moe_combine(cfg, T, y_perm, cap, inv_pos, topk_w, shared_out, out, ws=None, stream=None):
    _check("moe_combine", lib().moe_combine(
        ctypes.byref(cfg), T, _p(y_perm), cap, _p(inv_pos), _p(topk_w), _p(shared_out),
        _p(out), _p(ws), _nbytes(ws), _stream(stream)))


def moe_forward(cfg, T, x, router_w, router_bias, w13, w2, shared_w13, shared_w2, expert_map,
                out, ws, stream=None):
    _check("moe_forward", lib().moe_forward(
        ctypes.byref(cfg), T, _p(x), _p(router_w), _p(router_bias), _p(w13), _p(w2),
        _p(shared_w13), _p(shared_w2), _p(expert_map), _p(out), _p(ws), _nbytes(ws),
        _stream(stream)))


def moe_forward_timed(cfg, T, x, router_w, router_bias, w13, w2, shared_w13, shared_w2,
                      expert_map, out, ws, events, stream=None) -> int:
    """moe_forward that records 8 torch.cuda.Event objects (or None) at the
    stage boundaries on the stream; returns the number of kernels launched."""
    handles = (ctypes.c_void_p * 8)()
    for i, ev in enumerate(events):
        handles[i] = None if ev is None else ev.cuda_event
    n = ctypes.c_int(0)
    _check("moe_forward_timed", lib().moe_forward_timed(
        ctypes.byref(cfg), T, _p(x), _p(router_w), _p(router_bias), _p(w13), _p(w2),
        _p(shared_w13), _p(shared_w2), _p(expert_map), _p(out), _p(ws), _nbytes(ws),
        _stream(stream), handles, ctypes.byref(n)))
    return n.value


def moe_get_status(ws, stream=None) -> tuple[int, int]:
    """(status code, raw MOE_DEV_* flags); synchronises the stream."""
    flags = ctypes.c_uint32(0)
    rc = lib().moe_get_status(_p(ws), _stream(stream), ctypes.byref(flags))
    return rc, flags.value


def debug_build() -> bool:
    """True when the active library is libmoe_debug.so."""
    return bool(lib().moe_debug_build())


def debug_take() -> DebugRecord:
    """Synchronise the device, then read and clear the debug build's record
    of failed bounds checks (count, and site / index / bound of the first)."""
    rec = DebugRecord()
    _check("moe_debug_take", lib().moe_debug_take(ctypes.byref(rec)))
    return rec


def debug_site(site: int) -> str:
    """'file:line' of a record's site."""
    return f"{DEBUG_FILES.get(site >> 16, site >> 16)}:{site & 0xffff}"


def debug_selftest(stream=None) -> None:
    """Enqueue the debug build's one failing check (index 5, bound 4)."""
    _check("moe_debug_selftest", lib().moe_debug_selftest(_stream(stream)))


def set_wait_limit_ns(ns: int) -> None:
    """Time limit of the kernels' pipeline waits on the current device, in ns
    (0 restores the default of 1 s)."""
    _check("moe_set_wait_limit_ns", lib().moe_set_wait_limit_ns(int(ns)))

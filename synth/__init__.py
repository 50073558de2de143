"""Seeded synthetic inputs for MoE layer workloads.

This module holds the input generator and the workload shapes. It holds none
of the MoE method's arithmetic. The generator is the counter-based normal
sampler defined in ``synth/gen.c`` (SplitMix64 mixing plus Box-Muller), built
here as a small host library. Every tensor is addressed by
``(seed, tensor_id, row, attempt)``, so any slice can be drawn on its own: one
expert's weights, one EP shard, or one redrawn token row.

Workload shapes follow the layers the source pages discuss: the Mixtral-style
MixtralMoE block (SGLang issue "Expert parallelism support"), the Qwen3-MoE
and DeepSeek-V2 style FusedMoE configurations (vLLM ``MoEMixin.recursive_replace``
reading ``num_experts_per_tok``, ``moe_intermediate_size``, ``n_group``,
``topk_group``, ``routed_scaling_factor``, ``n_shared_experts``), and an
expert-parallel local shard (``ep_fused_moe_patch.py``, ``_ep_init``).
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "_gen.so")
_lock = threading.Lock()
_lib = None

# tensor ids of the counter-based streams
X, ROUTER_W, ROUTER_B, W13, W2, SHARED_W13, SHARED_W2 = 1, 2, 3, 4, 5, 6, 7


def build(force: bool = False) -> str:
    """Compile the generator library in place (host C, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.synth_normal_rows.restype = ctypes.c_int
            lib.synth_normal_rows.argtypes = [
                ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p]
            lib.synth_bf16_to_f32.restype = None
            lib.synth_bf16_to_f32.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int64]
            lib.synth_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return _load().synth_num_threads()


def draw(seed, tensor_id, row0, nrows, ncols, std, bf16, attempts=None,
         out=None):
    """Rows [row0, row0+nrows) as float32 (values exactly bf16 when bf16)."""
    lib = _load()
    if out is None:
        out = np.empty((nrows, ncols), dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous
    assert out.size == nrows * ncols
    att = None
    if attempts is not None:
        attempts = np.ascontiguousarray(attempts, dtype=np.int32)
        assert attempts.shape == (nrows,)
        att = attempts.ctypes.data
    rc = lib.synth_normal_rows(seed, tensor_id, row0, nrows, ncols, att,
                               float(std), int(bool(bf16)), out.ctypes.data,
                               None)
    if rc != 0:
        raise ValueError("synth_normal_rows: bad arguments")
    return out


def draw_bf16_bits(seed, tensor_id, row0, nrows, ncols, std, attempts=None,
                   out_ptr=None):
    """Same values as ``draw(..., bf16=True)``, as raw bf16 bit patterns.

    With ``out_ptr`` (an address of nrows*ncols uint16, e.g. a pinned torch
    buffer) the bits are written there and None is returned.
    """
    lib = _load()
    res = None
    if out_ptr is None:
        res = np.empty((nrows, ncols), dtype=np.uint16)
        out_ptr = res.ctypes.data
    att = None
    if attempts is not None:
        attempts = np.ascontiguousarray(attempts, dtype=np.int32)
        assert attempts.shape == (nrows,)
        att = attempts.ctypes.data
    rc = lib.synth_normal_rows(seed, tensor_id, row0, nrows, ncols, att,
                               float(std), 1, None, out_ptr)
    if rc != 0:
        raise ValueError("synth_normal_rows: bad arguments")
    return res


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _load().synth_bf16_to_f32(bits.ctypes.data, out.ctypes.data, bits.size)
    return out


class BF16Experts:
    """Expert-indexed view of bf16 bit patterns [E, R, C] that widens one
    expert to float32 on access (a host copy at half the memory)."""

    def __init__(self, bits: np.ndarray):
        self.bits = bits
        self.shape = bits.shape

    def __getitem__(self, e):
        return bf16_bits_to_f32(self.bits[e])


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and input distribution of one synthetic MoE layer."""
    name: str
    T: int                      # tokens
    H: int                      # hidden_size
    I: int                      # (moe_)intermediate_size
    E: int                      # global num_experts
    K: int                      # top_k
    renormalize: bool = True
    n_group: int = 0            # num_expert_group (0 = plain top-k)
    topk_group: int = 0
    rsf: float = 1.0            # routed_scaling_factor
    n_shared: int = 0           # shared experts
    I_shared: int = 0           # intermediate size of each shared expert
    ep_size: int = 1
    ep_rank: int = 0
    act: str = "bf16"           # "bf16" or "f32": x, expert weights, output
    router: str = "bf16"        # "bf16" or "f32": router weight storage
    router_bias: bool = False   # per-expert bias b ~ N(0, 1) (role: bias_mode)
    bias_mode: str = "logit"    # "logit": b skews the logits; "select": b corrects
                                # the scores for the top-k choice only
    scoring: str = "softmax"    # "softmax" or "sigmoid" routing scores
    x_std: float = 1.0

    @property
    def E_local(self) -> int:
        return self.E // self.ep_size

    @property
    def grouped(self) -> bool:
        return self.n_group > 0

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def std(self, tensor_id: int) -> float:
        """Std of each tensor: x as configured, weights 1/sqrt(fan_in)."""
        return {X: self.x_std,
                ROUTER_W: 1.0 / math.sqrt(self.H),
                ROUTER_B: 1.0,
                W13: 1.0 / math.sqrt(self.H),
                W2: 1.0 / math.sqrt(self.I),
                SHARED_W13: 1.0 / math.sqrt(self.H),
                SHARED_W2: 1.0 / math.sqrt(max(self.I_shared, 1))}[tensor_id]

    def flops(self, assignments: int) -> int:
        """Algorithmic FLOPs: router GEMM + routed MLPs + shared MLPs."""
        return (2 * self.T * self.H * self.E + 6 * self.H * self.I * assignments
                + 6 * self.H * self.I_shared * self.n_shared * self.T)


# The five layer workloads (T is the default token count; decode has 3).
TINY = Workload("tiny", T=64, H=128, I=256, E=8, K=2, act="f32", router="f32",
                x_std=1.0 / math.sqrt(128))
MIXTRAL = Workload("mixtral_prefill", T=4096, H=4096, I=14336, E=8, K=2,
                   router="f32")
QWEN_DECODE = Workload("qwen3_decode", T=64, H=2048, I=512, E=256, K=8,
                       router_bias=True)
DEEPSEEK = Workload("deepseek_v2_prefill", T=2048, H=5120, I=1536, E=160, K=6,
                    renormalize=False, n_group=8, topk_group=3, rsf=16.0,
                    n_shared=2, I_shared=1536)
EP_SHARD = Workload("ep_shard", T=8192, H=2048, I=512, E=256, K=8, ep_size=4,
                    ep_rank=1)

WORKLOADS = {w.name: w for w in (TINY, MIXTRAL, QWEN_DECODE, DEEPSEEK, EP_SHARD)}
DECODE_TOKENS = (1, 8, 64)


def draw_tensor(wl: Workload, tensor_id: int, seed: int = 0, attempts=None,
                local: bool = True) -> np.ndarray:
    """Draw one tensor of a workload as float32 host values.

    Expert tensors are drawn by global flat row, so the local shard of rank r
    equals rows of the global tensor (``local=False`` gives the global one).
    """
    bf = wl.act == "bf16"
    e0, ne = (wl.ep_rank * wl.E_local, wl.E_local) if local else (0, wl.E)
    if tensor_id == X:
        return draw(seed, X, 0, wl.T, wl.H, wl.std(X), bf, attempts)
    if tensor_id == ROUTER_W:
        return draw(seed, ROUTER_W, 0, wl.E, wl.H, wl.std(ROUTER_W),
                    wl.router == "bf16")
    if tensor_id == ROUTER_B:
        return draw(seed, ROUTER_B, 0, 1, wl.E, 1.0, False).reshape(wl.E)
    if tensor_id == W13:
        a = draw(seed, W13, e0 * 2 * wl.I, ne * 2 * wl.I, wl.H, wl.std(W13), bf)
        return a.reshape(ne, 2 * wl.I, wl.H)
    if tensor_id == W2:
        a = draw(seed, W2, e0 * wl.H, ne * wl.H, wl.I, wl.std(W2), bf)
        return a.reshape(ne, wl.H, wl.I)
    if tensor_id == SHARED_W13:
        a = draw(seed, SHARED_W13, 0, wl.n_shared * 2 * wl.I_shared, wl.H,
                 wl.std(SHARED_W13), bf)
        return a.reshape(wl.n_shared, 2 * wl.I_shared, wl.H)
    if tensor_id == SHARED_W2:
        a = draw(seed, SHARED_W2, 0, wl.n_shared * wl.H, wl.I_shared,
                 wl.std(SHARED_W2), bf)
        return a.reshape(wl.n_shared, wl.H, wl.I_shared)
    raise ValueError(tensor_id)


def layer_inputs(wl: Workload, seed: int = 0, attempts=None,
                 local: bool = True) -> dict:
    """All host inputs of one layer as float32 arrays (bf16-exact for bf16)."""
    d = {"x": draw_tensor(wl, X, seed, attempts),
         "router_w": draw_tensor(wl, ROUTER_W, seed),
         "router_b": draw_tensor(wl, ROUTER_B, seed) if wl.router_bias else None,
         "w13": draw_tensor(wl, W13, seed, local=local),
         "w2": draw_tensor(wl, W2, seed, local=local),
         "shared_w13": None, "shared_w2": None}
    if wl.n_shared:
        d["shared_w13"] = draw_tensor(wl, SHARED_W13, seed)
        d["shared_w2"] = draw_tensor(wl, SHARED_W2, seed)
    return d

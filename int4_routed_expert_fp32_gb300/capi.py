"""ctypes binding of ``libmoe.so`` (declared in ``include/moe.h``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Output tensors and workspaces are allocated with torch (device
memory) and passed as raw pointers; calls are enqueued on torch's current CUDA
stream.  Importing this module fails loudly when the library is missing -- there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p
from typing import Dict, Optional

import torch

from .build import LIB_PATH

MOE_OK = 0
MOE_ERR_INVALID = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_TIMEOUT = -5


class MoeError(RuntimeError):
    def __init__(self, name: str, code: int):
        super().__init__(f"{name} returned {code} ({status_string(code)})")
        self.code = code


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", c_int32), ("H", c_int32), ("E", c_int32), ("k", c_int32), ("I", c_int32),
                ("L", c_int32), ("act_bits", c_int32), ("renorm", c_int32), ("eps", c_float),
                ("I_shared", c_int32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in (
        "router_w", "router_bias", "gate_packed", "gate_scale", "up_packed", "up_scale",
        "down_packed", "down_scale", "lat_down", "lat_norm", "lat_up", "shared_gate", "shared_up",
        "shared_down")]


# name -> (restype, argtypes); mirrors include/moe.h
SIGNATURES = {
    "moe_route_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_route": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                          c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_dispatch_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_dispatch": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p,
                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_size_t, c_void_p]),
    "moe_dispatch_pairs": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                   c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_dispatch_noalloc": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p]),
    "moe_expert_ffn_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "moe_expert_ffn": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                               c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                               c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_expert_ffn_pairs_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "moe_expert_ffn_pairs": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_int4_linear_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_int4_linear": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_quantize_rows": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_quantize_int4": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_shared_expert_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_shared_expert": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                  c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_combine": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]),
    "moe_linear_bf16": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]),
    "moe_rmsnorm": (c_int, [c_void_p, c_void_p, c_int, c_int, c_float, c_void_p, c_void_p]),
    "moe_workspace_size": (c_size_t, [POINTER(MoeConfig)]),
    "moe_layer_forward": (c_int, [POINTER(MoeConfig), POINTER(MoeWeights), c_void_p, c_void_p,
                                  c_void_p, c_size_t, c_void_p]),
    "moe_layer_forward_host": (c_int, [POINTER(MoeConfig), POINTER(MoeWeights), c_void_p, c_void_p,
                                       c_void_p, c_size_t, c_void_p]),
    "moe_check_error": (c_int, [c_void_p]),
    "moe_wait_selftest": (c_int, [c_int64, c_void_p]),
    "moe_status_string": (ctypes.c_char_p, [c_int]),
    "moe_version": (ctypes.c_char_p, []),
    "moe_launch_count": (ctypes.c_uint64, []),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.moe_status_string(code).decode()


def launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(lib.moe_launch_count())


def _check(name: str, rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(name, rc)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else c_void_p(t.data_ptr())


def _stream():
    return c_void_p(torch.cuda.current_stream().cuda_stream)


def _ws(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _dev(t: torch.Tensor, dtype=None) -> None:
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"expected {dtype}, got {t.dtype}")


# ------------------------------------------------------------------ stages

def route(x: torch.Tensor, w_router: torch.Tensor, bias: torch.Tensor, k: int, renorm: bool = True):
    """topk_idx int32 [T, k], topk_w fp32 [T, k] for bf16 x [T, H]."""
    _dev(x, torch.bfloat16); _dev(w_router, torch.float32); _dev(bias, torch.float32)
    T, H = x.shape
    E = w_router.shape[0]
    idx = torch.empty(T, k, dtype=torch.int32, device=x.device)
    w = torch.empty(T, k, dtype=torch.float32, device=x.device)
    ws = _ws(lib.moe_route_workspace_size(T, H, E), x.device)
    _check("moe_route", lib.moe_route(_p(x), _p(w_router), _p(bias), T, H, E, k, int(renorm),
                                      _p(idx), _p(w), _p(ws), ws.numel(), _stream()))
    return idx, w


def _dispatch_out(T: int, k: int, D: int, E: int, act_bits: int, pairs: bool, dev):
    R = T * k
    xdt = torch.int8 if act_bits == 8 else (torch.float16 if pairs else torch.bfloat16)
    return {
        "counts": torch.empty(E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "row_token": torch.empty(R, dtype=torch.int32, device=dev),
        "row_slot": torch.empty(R, dtype=torch.int32, device=dev),
        "inv_row": torch.empty(R, dtype=torch.int32, device=dev),
        "x_sorted": torch.empty(R, D, dtype=xdt, device=dev),
        "x_scale": torch.empty(R, dtype=torch.float32, device=dev) if act_bits == 8 else None,
    }


def dispatch(topk_idx: torch.Tensor, x: torch.Tensor, E: int, act_bits: int = 16,
             pairs: bool = False) -> Dict[str, torch.Tensor]:
    """Counts, offsets, the stable expert-major permutation and the gathered
    rows (pairs=True: moe_dispatch_pairs, rows in the expert kernels' pair
    order, fp16 or int8)."""
    _dev(topk_idx, torch.int32); _dev(x, torch.bfloat16)
    T, k = topk_idx.shape
    D = x.shape[1]
    dev = x.device
    out = _dispatch_out(T, k, D, E, act_bits, pairs, dev)
    ws = _ws(lib.moe_dispatch_workspace_size(T, E, k), dev)
    name = "moe_dispatch_pairs" if pairs else "moe_dispatch"
    _check(name, getattr(lib, name)(
        _p(topk_idx), _p(x), T, D, E, k, act_bits, _p(out["counts"]), _p(out["offsets"]),
        _p(out["row_token"]), _p(out["row_slot"]), _p(out["inv_row"]), _p(out["x_sorted"]),
        _p(out["x_scale"]), _p(ws), ws.numel(), _stream()))
    return out


def dispatch_noalloc(topk_idx: torch.Tensor, x: torch.Tensor, E: int,
                     act_bits: int = 16) -> Dict[str, torch.Tensor]:
    """moe_dispatch without a workspace: the library's fixed device scratch is
    used instead (for callers that cannot allocate device memory; calls must
    not overlap on the GPU)."""
    _dev(topk_idx, torch.int32); _dev(x, torch.bfloat16)
    T, k = topk_idx.shape
    D = x.shape[1]
    dev = x.device
    out = _dispatch_out(T, k, D, E, act_bits, False, dev)
    _check("moe_dispatch_noalloc", lib.moe_dispatch_noalloc(
        _p(topk_idx), _p(x), T, D, E, k, act_bits, _p(out["counts"]), _p(out["offsets"]),
        _p(out["row_token"]), _p(out["row_slot"]), _p(out["inv_row"]), _p(out["x_sorted"]),
        _p(out["x_scale"]), _stream()))
    return out


def expert_ffn(x_sorted: torch.Tensor, x_scale: Optional[torch.Tensor], offsets: torch.Tensor,
               experts: Dict[str, torch.Tensor], act_bits: int = 16,
               pairs: bool = False) -> torch.Tensor:
    """y_sorted bf16 [rows, D] = down(SiLU(gate(x)) * up(x)) per expert segment
    (pairs=True: moe_expert_ffn_pairs on rows from dispatch(..., pairs=True))."""
    _dev(x_sorted); _dev(offsets, torch.int32)
    rows, D = x_sorted.shape
    E, I = experts["gate_packed"].shape[0], experts["gate_packed"].shape[1]
    y = torch.empty(rows, D, dtype=torch.bfloat16, device=x_sorted.device)
    name = "moe_expert_ffn_pairs" if pairs else "moe_expert_ffn"
    ws = _ws(getattr(lib, name + "_workspace_size")(E, D, I, rows, act_bits), x_sorted.device)
    _check(name, getattr(lib, name)(
        _p(x_sorted), _p(x_scale), _p(offsets), E, D, I, rows,
        _p(experts["gate_packed"]), _p(experts["gate_scale"]), _p(experts["up_packed"]),
        _p(experts["up_scale"]), _p(experts["down_packed"]), _p(experts["down_scale"]), act_bits,
        _p(y), _p(ws), ws.numel(), _stream()))
    return y


def int4_linear(x: torch.Tensor, x_scale: Optional[torch.Tensor], offsets: torch.Tensor,
                w_packed: torch.Tensor, w_scale: torch.Tensor, act_bits: int = 16) -> torch.Tensor:
    """fp32 [rows, N] = x W_e^T per expert segment (one grouped PackedInt4Linear)."""
    _dev(x); _dev(offsets, torch.int32); _dev(w_packed, torch.int32)
    rows, K = x.shape
    E, N = w_packed.shape[0], w_packed.shape[1]
    out = torch.empty(rows, N, dtype=torch.float32, device=x.device)
    ws = _ws(lib.moe_int4_linear_workspace_size(E, K, rows), x.device)
    _check("moe_int4_linear", lib.moe_int4_linear(
        _p(x), _p(x_scale), _p(offsets), E, K, N, rows, _p(w_packed), _p(w_scale), act_bits,
        _p(out), _p(ws), ws.numel(), _stream()))
    return out


def quantize_rows(v: torch.Tensor):
    """Per-row int8 quantisation: (q int8 [R, C], scale fp32 [R])."""
    _dev(v, torch.bfloat16)
    R, C = v.shape
    q = torch.empty(R, C, dtype=torch.int8, device=v.device)
    s = torch.empty(R, dtype=torch.float32, device=v.device)
    _check("moe_quantize_rows", lib.moe_quantize_rows(_p(v), R, C, _p(q), _p(s), _stream()))
    return q, s


def quantize_int4(w: torch.Tensor):
    """bf16 weight [..., N, K] -> (packed int32 [..., N, K/8], bf16 scale [..., N, K/32])."""
    _dev(w, torch.bfloat16)
    K = w.shape[-1]
    rows = w.numel() // K if K else 0
    packed = torch.empty(*w.shape[:-1], K // 8, dtype=torch.int32, device=w.device)
    scale = torch.empty(*w.shape[:-1], K // 32, dtype=torch.bfloat16, device=w.device)
    _check("moe_quantize_int4", lib.moe_quantize_int4(_p(w), rows, K, _p(packed), _p(scale),
                                                      _stream()))
    return packed, scale


def shared_expert(x: torch.Tensor, gate_w: torch.Tensor, up_w: torch.Tensor,
                  down_w: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """out (+)= down(SiLU(gate x) * up x) with bf16 weights; a new output when
    ``out`` is None, else added to it in place."""
    for t in (x, gate_w, up_w, down_w):
        _dev(t, torch.bfloat16)
    T, H = x.shape
    I = gate_w.shape[0]
    acc = out is not None
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    ws = _ws(lib.moe_shared_expert_workspace_size(T, H, I), x.device)
    _check("moe_shared_expert", lib.moe_shared_expert(
        _p(x), T, H, I, _p(gate_w), _p(up_w), _p(down_w), int(acc), _p(out), _p(ws), ws.numel(),
        _stream()))
    return out


def combine(y_sorted: torch.Tensor, inv_row: torch.Tensor, topk_w: torch.Tensor) -> torch.Tensor:
    _dev(y_sorted, torch.bfloat16); _dev(inv_row, torch.int32); _dev(topk_w, torch.float32)
    T, k = topk_w.shape
    D = y_sorted.shape[1]
    out = torch.empty(T, D, dtype=torch.bfloat16, device=y_sorted.device)
    _check("moe_combine", lib.moe_combine(_p(y_sorted), _p(inv_row), _p(topk_w), T, D, k, _p(out),
                                          _stream()))
    return out


def linear_bf16(x: torch.Tensor, w: torch.Tensor) -> torch.Tensor:
    _dev(x, torch.bfloat16); _dev(w, torch.bfloat16)
    M, K = x.shape
    N = w.shape[0]
    y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _check("moe_linear_bf16", lib.moe_linear_bf16(_p(x), _p(w), M, N, K, _p(y), _stream()))
    return y


def rmsnorm(x: torch.Tensor, gain: torch.Tensor, eps: float) -> torch.Tensor:
    _dev(x, torch.bfloat16); _dev(gain, torch.bfloat16)
    M, N = x.shape
    y = torch.empty_like(x)
    _check("moe_rmsnorm", lib.moe_rmsnorm(_p(x), _p(gain), M, N, float(eps), _p(y), _stream()))
    return y


def check_error() -> int:
    """Synchronise the current stream and return (and clear) the device status word."""
    return lib.moe_check_error(_stream())


def wait_selftest(limit_ns: int) -> None:
    _check("moe_wait_selftest", lib.moe_wait_selftest(int(limit_ns), _stream()))


# ------------------------------------------------------------------ layer

class MoeLayer:
    """One routed int4 MoE layer: configuration, device weights and a workspace."""

    def __init__(self, T: int, H: int, E: int, k: int, I: int, weights: Dict[str, torch.Tensor],
                 L: int = 0, act_bits: int = 16, renorm: bool = True, eps: float = 1e-6,
                 I_shared: int = 0):
        self.cfg = MoeConfig(T, H, E, k, I, L, act_bits, int(renorm), eps, I_shared)
        self.weights = weights
        self.device = weights["router_w"].device
        for name, t in weights.items():
            if t is not None:
                _dev(t)
        self.wstruct = MoeWeights(*[_p(weights.get(n)) for n, _ in MoeWeights._fields_])
        self.ws = _ws(lib.moe_workspace_size(ctypes.byref(self.cfg)), self.device)

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        _dev(x, torch.bfloat16)
        if out is None:
            out = torch.empty_like(x)
        _check("moe_layer_forward", lib.moe_layer_forward(
            ctypes.byref(self.cfg), ctypes.byref(self.wstruct), _p(x), _p(out), _p(self.ws),
            self.ws.numel(), _stream()))
        return out

    def forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor) -> None:
        """x_host / out_host: CPU bf16 [T, H] (pinned for asynchronous copies)."""
        if x_host.is_cuda or out_host.is_cuda:
            raise ValueError("forward_host takes host tensors")
        _check("moe_layer_forward_host", lib.moe_layer_forward_host(
            ctypes.byref(self.cfg), ctypes.byref(self.wstruct), _p(x_host), _p(out_host),
            _p(self.ws), self.ws.numel(), _stream()))
